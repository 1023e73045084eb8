"""The CPU oracle on all host cores, for parity checks of full-size workloads.

Test infrastructure, like the oracle itself.  Worker processes are started
with "spawn" (safe after the parent has initialised CUDA); the parent puts
the inputs and the outputs in shared memory, and each worker runs the oracle
on a range of rows and writes its rows of the outputs in place.  Every block
is independent in all three calls, so splitting by rows changes no result.
"""

from __future__ import annotations

import atexit
import concurrent.futures as cf
import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np

_POOL = None


def cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def pool() -> cf.ProcessPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = cf.ProcessPoolExecutor(max_workers=cores(), mp_context=mp.get_context("spawn"))
        atexit.register(_POOL.shutdown)
    return _POOL


class Shared:
    """Named arrays, each in a shared-memory segment of its own."""

    def __init__(self):
        self.segs, self.spec = [], {}

    def put(self, name: str, a: np.ndarray) -> np.ndarray:
        a = np.ascontiguousarray(a)
        return self._alloc(name, a.shape, a.dtype, a)

    def empty(self, name: str, shape, dtype) -> np.ndarray:
        return self._alloc(name, tuple(shape), np.dtype(dtype), None)

    def _alloc(self, name, shape, dtype, src):
        nbytes = max(1, int(np.prod(shape)) * dtype.itemsize)
        seg = shared_memory.SharedMemory(create=True, size=nbytes)
        self.segs.append(seg)
        view = np.ndarray(shape, dtype=dtype, buffer=seg.buf)
        if src is not None:
            view[...] = src
        self.spec[name] = (seg.name, shape, dtype.str)
        return view

    def close(self):
        for seg in self.segs:
            seg.close()
            seg.unlink()
        self.segs = []


def _attach(spec):
    segs, arrays = [], {}
    for name, (seg_name, shape, dt) in spec.items():
        seg = shared_memory.SharedMemory(name=seg_name)
        segs.append(seg)
        arrays[name] = np.ndarray(shape, dtype=np.dtype(dt), buffer=seg.buf)
    return segs, arrays


def _task(args):
    import oracle

    kind, spec, r0, r1, block = args
    segs, A = _attach(spec)
    try:
        if kind == "compress":  # x [P, rows, d] -> codes [P, rows, d], alpha / scale [P, rows, d / block]
            for p in range(A["x"].shape[0]):
                c, a, s = oracle.compress(A["x"][p, r0:r1].copy(), block)
                A["codes"][p, r0:r1] = c
                A["alpha"][p, r0:r1] = a
                A["scale"][p, r0:r1] = s
        elif kind == "compress_f64":  # y float64 [rows, d] -> codes [rows, d], alpha / scale [rows, d / block]
            c, a, s = oracle.compress_f64(A["y"][r0:r1].copy(), block)
            A["rcodes"][r0:r1] = c
            A["ralpha"][r0:r1] = a
            A["rscale"][r0:r1] = s
        elif kind == "reduce":  # shards [P, rows, d] + scalars -> one compressed [rows, d]
            P = A["codes"].shape[0]
            c, a, s = oracle.reduce_shards([A["codes"][p, r0:r1].copy() for p in range(P)],
                                           [A["alpha"][p, r0:r1].copy() for p in range(P)],
                                           [A["scale"][p, r0:r1].copy() for p in range(P)], block)
            A["rcodes"][r0:r1] = c
            A["ralpha"][r0:r1] = a
            A["rscale"][r0:r1] = s
        elif kind == "agoq_accumulate":  # rows = blocks of flat buffers, in place
            b0, b1 = r0 * block, r1 * block
            c, sc = oracle.agoq_accumulate(A["acodes"][b0:b1].copy(), A["ascale"][r0:r1].copy(),
                                           A["grad"][b0:b1].copy(), block)
            A["acodes"][b0:b1] = c
            A["ascale"][r0:r1] = sc
        elif kind == "agoq_reduce":  # shards [P, n] + multipliers [P, n / block] -> [n], [n / block]
            b0, b1 = r0 * block, r1 * block
            P = A["pcodes"].shape[0]
            c, sc = oracle.agoq_reduce([A["pcodes"][p, b0:b1].copy() for p in range(P)],
                                       [A["pscale"][p, r0:r1].copy() for p in range(P)], block)
            A["acodes"][b0:b1] = c
            A["ascale"][r0:r1] = sc
        else:  # decompress [rows, d] -> float64 [rows, d]
            A["out"][r0:r1] = oracle.decompress(A["rcodes"][r0:r1].copy(), A["ralpha"][r0:r1].copy(),
                                                A["rscale"][r0:r1].copy(), block)
    finally:
        del A
        for seg in segs:
            seg.close()
    return r1 - r0


def _run(kind: str, sh: Shared, rows: int, block: int):
    step = max(1, -(-rows // (4 * cores())))
    tasks = [(kind, sh.spec, r, min(rows, r + step), block) for r in range(0, rows, step)]
    assert sum(pool().map(_task, tasks)) == rows


# Shared memory is a tmpfs of limited size: large inputs go through in
# pieces of at most this many bytes of shared arrays.
PIECE_BYTES = 256 << 20


def _pieces(rows: int, bytes_per_row: int):
    step = max(1, PIECE_BYTES // max(1, bytes_per_row))
    return [(r, min(rows, r + step)) for r in range(0, rows, step)]


def compress(bits: np.ndarray, block: int):
    """bf16 bits [P, rows, d] -> oracle (codes [P, rows, d], alpha, scale [P, rows, d / block])."""
    P, rows, d = bits.shape
    codes = np.empty((P, rows, d), np.uint8)
    alpha = np.empty((P, rows, d // block), np.float32)
    scale = np.empty((P, rows, d // block), np.float32)
    for p in range(P):
        for r0, r1 in _pieces(rows, 3 * d + 8 * (d // block)):
            sh = Shared()
            try:
                sh.put("x", bits[p:p + 1, r0:r1])
                c = sh.empty("codes", (1, r1 - r0, d), np.uint8)
                a = sh.empty("alpha", (1, r1 - r0, d // block), np.float32)
                s = sh.empty("scale", (1, r1 - r0, d // block), np.float32)
                _run("compress", sh, r1 - r0, block)
                codes[p, r0:r1], alpha[p, r0:r1], scale[p, r0:r1] = c[0], a[0], s[0]
            finally:
                sh.close()
    return codes, alpha, scale


def compress_f64(y: np.ndarray, block: int):
    """float64 [rows, d] -> the oracle's (codes [rows, d], alpha, scale [rows, d / block])."""
    rows, d = y.shape
    nbr = d // block
    out = (np.empty((rows, d), np.uint8), np.empty((rows, nbr), np.float32), np.empty((rows, nbr), np.float32))
    for r0, r1 in _pieces(rows, 9 * d + 8 * nbr):
        sh = Shared()
        try:
            sh.put("y", y[r0:r1])
            c = sh.empty("rcodes", (r1 - r0, d), np.uint8)
            a = sh.empty("ralpha", (r1 - r0, nbr), np.float32)
            s = sh.empty("rscale", (r1 - r0, nbr), np.float32)
            _run("compress_f64", sh, r1 - r0, block)
            out[0][r0:r1], out[1][r0:r1], out[2][r0:r1] = c, a, s
        finally:
            sh.close()
    return out


def reduce_shards(codes: np.ndarray, alpha: np.ndarray, scale: np.ndarray, block: int):
    """P compressed shards (codes [P, rows, d], scalars [P, rows * d / block])
    -> the oracle's compressed sum (codes [rows, d], alpha, scale [rows, d / block])."""
    P, rows, d = codes.shape
    nbr = d // block
    alpha, scale = alpha.reshape(P, rows, nbr), scale.reshape(P, rows, nbr)
    out = (np.empty((rows, d), np.uint8), np.empty((rows, nbr), np.float32), np.empty((rows, nbr), np.float32))
    for r0, r1 in _pieces(rows, (P + 1) * (d + 8 * nbr)):
        sh = Shared()
        try:
            sh.put("codes", codes[:, r0:r1])
            sh.put("alpha", alpha[:, r0:r1])
            sh.put("scale", scale[:, r0:r1])
            c = sh.empty("rcodes", (r1 - r0, d), np.uint8)
            a = sh.empty("ralpha", (r1 - r0, nbr), np.float32)
            s = sh.empty("rscale", (r1 - r0, nbr), np.float32)
            _run("reduce", sh, r1 - r0, block)
            out[0][r0:r1], out[1][r0:r1], out[2][r0:r1] = c, a, s
        finally:
            sh.close()
    return out


def decompress(codes: np.ndarray, alpha: np.ndarray, scale: np.ndarray, block: int) -> np.ndarray:
    """codes [rows, d] + scalars -> the oracle's float64 reconstruction [rows, d]."""
    rows, d = codes.shape
    nbr = d // block
    alpha, scale = alpha.reshape(rows, nbr), scale.reshape(rows, nbr)
    out = np.empty((rows, d), np.float64)
    for r0, r1 in _pieces(rows, 9 * d + 8 * nbr):
        sh = Shared()
        try:
            sh.put("rcodes", codes[r0:r1])
            sh.put("ralpha", alpha[r0:r1])
            sh.put("rscale", scale[r0:r1])
            o = sh.empty("out", (r1 - r0, d), np.float64)
            _run("decompress", sh, r1 - r0, block)
            out[r0:r1] = o
        finally:
            sh.close()
    return out


def agoq_accumulate(codes: np.ndarray, scale: np.ndarray, grad_bf16: np.ndarray, block: int = 128):
    """One AGoQ accumulation step of the flat buffer: the oracle's new (codes, scale)."""
    codes, scale, grad = codes.reshape(-1), scale.reshape(-1), grad_bf16.reshape(-1)
    nb = codes.size // block
    oc, os_ = np.empty_like(codes), np.empty_like(scale)
    for b0, b1 in _pieces(nb, 3 * block + 4):
        sh = Shared()
        try:
            c = sh.put("acodes", codes[b0 * block:b1 * block])
            s = sh.put("ascale", scale[b0:b1])
            sh.put("grad", grad[b0 * block:b1 * block])
            _run("agoq_accumulate", sh, b1 - b0, block)
            oc[b0 * block:b1 * block], os_[b0:b1] = c, s
        finally:
            sh.close()
    return oc, os_


def agoq_reduce(codes: np.ndarray, scale: np.ndarray, block: int = 128):
    """The AGoQ reduce of P flat shards (codes [P, n], multipliers [P, n / block])."""
    P, n = codes.shape
    scale = scale.reshape(P, -1)
    nb = n // block
    oc, os_ = np.empty(n, np.uint8), np.empty(nb, np.float32)
    for b0, b1 in _pieces(nb, (P + 1) * (block + 4)):
        sh = Shared()
        try:
            sh.put("pcodes", codes[:, b0 * block:b1 * block])
            sh.put("pscale", scale[:, b0:b1])
            c = sh.empty("acodes", ((b1 - b0) * block,), np.uint8)
            s = sh.empty("ascale", (b1 - b0,), np.float32)
            _run("agoq_reduce", sh, b1 - b0, block)
            oc[b0 * block:b1 * block], os_[b0:b1] = c, s
        finally:
            sh.close()
    return oc, os_
