"""C-ABI checks that need no GPU: the library builds, loads and exports every
function include/taco.h declares, and argument validation rejects bad calls
before any CUDA call is made (the pointers below are never dereferenced)."""

import ctypes
import os
import re

import pytest

from fp8_communication_compression_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "taco.h")

OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3
A = 1 << 20  # a fake, 16-byte aligned "device address"; never dereferenced


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)) - {"if"})


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_header_declares_the_calls_of_the_boundary():
    names = declared_functions()
    for n in ("taco_compress", "taco_decompress", "taco_reduce_shards", "agoq_fp8_accumulate",
              "agoq_reduce_shards", "taco_status_string", "taco_abi_version", "taco_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_abi_version_and_status_strings(lib):
    assert lib.taco_abi_version() == 1
    for s in range(5):
        assert lib.taco_status_string(s)
    assert lib.taco_status_string(99) == b"unknown status"
    assert lib.taco_block_supported(128) and lib.taco_block_supported(256)
    assert not lib.taco_block_supported(64) and not lib.taco_block_supported(100)


def compress(lib, x=A, rows=4, d=256, block=128, e=1.0, eps=1e-12, codes=A * 4, alpha=A * 8,
             scale=A * 12):
    return lib.taco_compress(x, rows, d, block, e, eps, codes, alpha, scale, None)


def test_compress_validation(lib):
    assert compress(lib, block=100) == UNSUPPORTED
    assert compress(lib, block=64) == UNSUPPORTED
    assert compress(lib, d=200) == INVALID
    assert compress(lib, rows=-1) == INVALID
    assert compress(lib, d=0) == INVALID
    assert compress(lib, e=0.0) == INVALID
    assert compress(lib, eps=-1.0) == INVALID
    assert compress(lib, e=float("inf")) == INVALID
    assert compress(lib, eps=float("nan")) == INVALID
    assert compress(lib, rows=0) == OK  # empty input: no launch
    # the size limit: 2^31 - 256 rows of 128 elements; one more is rejected
    assert compress(lib, rows=(1 << 31) - 255, d=128) == UNSUPPORTED
    assert compress(lib, rows=1 << 40, d=1 << 30) == INVALID  # rows * d overflows
    assert compress(lib, x=0) == INVALID
    assert compress(lib, codes=0) == INVALID
    assert compress(lib, x=A + 8) == MISALIGNED
    assert compress(lib, codes=A * 4 + 4) == MISALIGNED
    assert compress(lib, alpha=A * 8 + 2) == MISALIGNED
    assert compress(lib, codes=A + 16) == INVALID  # codes overlap the input
    assert compress(lib, scale=A * 8 + 4) == INVALID  # scale overlaps alpha
    assert compress(lib, rows=1 << 40, d=1 << 30) == INVALID  # rows * d overflows


def test_decompress_validation(lib):
    f = lambda **k: lib.taco_decompress(k.get("codes", A), k.get("alpha", A * 4), k.get("scale", A * 8),
                                        k.get("rows", 4), k.get("d", 256), k.get("block", 128),
                                        k.get("out", A * 12), k.get("bf16", 0), None)
    assert f(block=512) == UNSUPPORTED
    assert f(rows=0) == OK
    assert f(out=0) == INVALID
    assert f(out=A * 12 + 8) == MISALIGNED
    assert f(out=A) == INVALID  # output overlaps the codes


def test_reduce_validation(lib):
    def f(P=2, rows=4, d=256, block=128, codes=None, out_codes=A * 64, e=1.0):
        c = codes if codes is not None else [A * (1 + p) for p in range(P)]
        cp, k1 = _lib.ptr_array(c)
        ap, k2 = _lib.ptr_array([A * (20 + p) for p in range(P)])
        sp, k3 = _lib.ptr_array([A * (40 + p) for p in range(P)])
        return lib.taco_reduce_shards(P, cp, ap, sp, rows, d, block, e, 1e-12, out_codes, A * 80,
                                      A * 90, None)
    assert f(P=0) == UNSUPPORTED
    assert f(P=17) == UNSUPPORTED
    assert f(block=64) == UNSUPPORTED
    assert f(rows=0) == OK
    assert f(e=-1.0) == INVALID
    assert f(codes=[A, 0]) == INVALID
    assert f(codes=[A, A + 8]) == MISALIGNED
    assert f(out_codes=A) == INVALID  # output overlaps shard 0


def test_agoq_validation(lib):
    acc = lambda n=1024, block=128, c=A, s=A * 4, g=A * 8: lib.agoq_fp8_accumulate(c, s, g, n, block, None)
    assert acc(block=64) == UNSUPPORTED
    assert acc(n=1000) == INVALID
    assert acc(n=-128) == INVALID
    assert acc(n=0) == OK
    assert acc(g=A * 8 + 2) == MISALIGNED
    assert acc(g=A + 512) == INVALID  # grad overlaps codes
    cp, k1 = _lib.ptr_array([A, A * 2])
    sp, k2 = _lib.ptr_array([A * 3, A * 4])
    red = lambda P=2, n=1024, oc=A * 10, os_=A * 12: lib.agoq_reduce_shards(P, cp, sp, n, 128, oc, os_, None)
    assert red(P=0) == UNSUPPORTED
    assert red(n=0) == OK
    assert red(oc=A * 10 + 1) == MISALIGNED
    assert red(oc=A) == INVALID


def test_device_error_rejects_null(lib):
    assert lib.taco_device_error(None, 0) == INVALID


def test_reduce_decompress_validation(lib):
    def f(P=2, rows=4, d=256, block=128, out=A * 100, out_codes=A * 64, bf16=0):
        cp, k1 = _lib.ptr_array([A * (1 + p) for p in range(P)])
        ap, k2 = _lib.ptr_array([A * (20 + p) for p in range(P)])
        sp, k3 = _lib.ptr_array([A * (40 + p) for p in range(P)])
        return lib.taco_reduce_decompress(P, cp, ap, sp, rows, d, block, 1.0, 1e-12, out_codes, A * 80,
                                          A * 90, out, bf16, None)
    assert f(P=17) == UNSUPPORTED
    assert f(block=512) == UNSUPPORTED
    assert f(rows=0) == OK
    assert f(out=0) == INVALID
    assert f(out=A * 100 + 4) == MISALIGNED
    assert f(out=A * 64) == INVALID  # reconstruction overlaps the output codes
    assert f(out=A * 2) == INVALID  # reconstruction overlaps shard 1


def test_laaq_validation(lib):
    q = lambda n=1024, block=128, bits=4, x=A, p=A * 4, s=A * 8: lib.agoq_laaq_quantize(x, n, block, bits, p, s, None)
    assert q(bits=3) == UNSUPPORTED
    assert q(bits=7) == UNSUPPORTED
    assert q(block=16) == UNSUPPORTED
    assert q(n=1000) == INVALID
    assert q(n=0) == OK
    assert q(p=A * 4 + 8) == MISALIGNED
    assert q(p=A + 64) == INVALID  # packed codes overlap the input
    d = lambda n=1024, out=A * 16, bf=1: lib.agoq_laaq_dequantize(A * 4, A * 8, n, 128, 4, out, bf, None)
    assert d(out=0) == INVALID
    assert d(out=A * 16 + 2) == MISALIGNED
    assert d(out=A * 4) == INVALID  # output overlaps the packed codes
    assert d(n=0) == OK


def test_laaq_recompute_validation(lib):
    s = lambda n=1024, block=128, bits=4, out=A * 16, bf=1: lib.agoq_laaq_dequantize_silu(
        A * 4, A * 8, n, block, bits, out, bf, None)
    assert s(bits=3) == UNSUPPORTED and s(block=16) == UNSUPPORTED
    assert s(n=1000) == INVALID and s(n=-128) == INVALID
    assert s(n=0) == OK
    assert s(out=0) == INVALID and s(out=A * 16 + 8) == MISALIGNED
    assert s(out=A * 4) == INVALID  # output over the packed codes
    r = lambda rows=8, d=256, block=128, bits=4, g=A * 32, eps=1e-6, out=A * 16, bf=0: \
        lib.agoq_laaq_dequantize_rmsnorm(A * 4, A * 8, rows, d, block, bits, g, eps, out, bf, None)
    assert r(bits=7) == UNSUPPORTED and r(block=512) == UNSUPPORTED
    assert r(d=192) == INVALID                     # rows of 192 hold 1.5 blocks of 128
    assert r(rows=-1) == INVALID and r(eps=-1.0) == INVALID and r(eps=float("nan")) == INVALID
    assert r(eps=float("inf")) == INVALID
    assert r(rows=0) == OK and r(d=0) == OK
    assert r(g=0) == INVALID and r(g=A * 32 + 4) == MISALIGNED
    assert r(g=A * 16 + 64) == INVALID             # gamma inside the output
    assert r(out=A * 8) == INVALID                 # output over the multipliers


def test_e4m3_encode_validation(lib):
    f = lambda n=1024, x=A, c=A * 8: lib.taco_e4m3_encode(x, n, c, None)
    assert f(n=-1) == INVALID
    assert f(n=0) == OK
    assert f(x=0) == INVALID
    assert f(c=0) == INVALID
    assert f(x=A + 4) == MISALIGNED
    assert f(c=A * 8 + 8) == MISALIGNED
    assert f(c=A + 1024) == INVALID  # codes overlap the input


def test_host_pipeline_validation(lib):
    h, ws = ctypes.c_void_p(), ctypes.c_uint64()
    c = lambda P=4, rows=64, d=1024, block=128, chunks=4: lib.taco_host_pipeline_create(
        P, rows, d, block, chunks, 0, ctypes.byref(h), ctypes.byref(ws))
    assert c(P=0) == UNSUPPORTED
    assert c(P=17) == UNSUPPORTED
    assert c(block=64) == UNSUPPORTED
    assert c(d=1000) == INVALID
    assert c(rows=0) == INVALID
    assert c(chunks=0) == INVALID
    assert c(chunks=65) == INVALID
    assert h.value is None
    assert lib.taco_host_pipeline_create(4, 64, 1024, 128, 4, 0, None, ctypes.byref(ws)) == INVALID
    assert lib.taco_host_pipeline_run(None, A, A, A, 1.0, 1e-12, None) == INVALID
    assert lib.taco_host_pipeline_destroy(None) == INVALID


def gemm_compress(lib, a=A, b=A * 64, M=256, N=512, K=128, block=128, e=1.0, eps=1e-12, codes=A * 128,
                  alpha=A * 192, scale=A * 200, y=None, ws=None, ws_bytes=0):
    return lib.taco_gemm_compress(a, b, M, N, K, block, e, eps, codes, alpha, scale, y, ws, ws_bytes, None)


def test_gemm_compress_validation(lib):
    # shapes the tile grid does not cover, and block sizes other than 128
    assert gemm_compress(lib, block=256) == UNSUPPORTED
    assert gemm_compress(lib, M=100) == UNSUPPORTED
    assert gemm_compress(lib, N=320) == UNSUPPORTED
    assert gemm_compress(lib, K=96) == UNSUPPORTED
    assert gemm_compress(lib, M=128 * 65536) == UNSUPPORTED
    assert gemm_compress(lib, M=-1) == INVALID
    assert gemm_compress(lib, e=0.0) == INVALID
    assert gemm_compress(lib, eps=float("nan")) == INVALID
    # nothing to do
    assert gemm_compress(lib, M=0) == OK and gemm_compress(lib, N=0) == OK
    # pointers
    assert gemm_compress(lib, a=None) == INVALID
    assert gemm_compress(lib, scale=None) == INVALID
    assert gemm_compress(lib, a=A + 8) == MISALIGNED
    assert gemm_compress(lib, y=A * 300 + 4) == MISALIGNED
    assert gemm_compress(lib, alpha=A * 192 + 2) == MISALIGNED
    # outputs overlapping each other or the operands
    assert gemm_compress(lib, codes=A) == INVALID
    assert gemm_compress(lib, alpha=A * 128 + 16) == INVALID
    assert gemm_compress(lib, y=A * 64) == INVALID
    # the split tail's workspace: 256-byte aligned, apart from every other buffer
    assert gemm_compress(lib, ws=A * 400 + 128, ws_bytes=1 << 20) == MISALIGNED
    assert gemm_compress(lib, ws=A * 128 + 256, ws_bytes=1 << 20) == INVALID  # over the codes
    assert gemm_compress(lib, ws=A * 63, ws_bytes=2 << 20) == INVALID         # over both operands


def test_agoq_gemm_laaq_quantize_validation(lib):
    f = lambda **k: lib.agoq_gemm_laaq_quantize(k.get("a", A), k.get("b", A * 64), k.get("M", 256),
                                                k.get("N", 512), k.get("K", 128), k.get("block", 128),
                                                k.get("bits", 4), k.get("packed", A * 128), k.get("scale", A * 200),
                                                k.get("y", None), k.get("ws", None), k.get("ws_bytes", 0), None)
    assert f(bits=3) == UNSUPPORTED and f(bits=7) == UNSUPPORTED and f(bits=16) == UNSUPPORTED
    assert f(block=64) == UNSUPPORTED
    assert f(M=100) == UNSUPPORTED and f(N=192) == UNSUPPORTED and f(K=32) == UNSUPPORTED
    assert f(M=-1) == INVALID
    assert f(M=0) == OK and f(N=0) == OK
    assert f(packed=None) == INVALID and f(scale=None) == INVALID
    assert f(packed=A * 128 + 8) == MISALIGNED
    # the packed stream is M N bits / 8 bytes: 64 KB at 4 bits, 128 KB at 8
    assert f(scale=A * 128 + 65532, bits=4) == INVALID       # multipliers inside the stream
    assert f(scale=A * 128 + 65536 + 4096, bits=8) == INVALID
    assert f(y=A * 64) == INVALID                              # output over an operand
    assert f(ws=A * 400 + 16, ws_bytes=4096) == MISALIGNED


def test_gemm_workspace_bytes_validation(lib):
    v = ctypes.c_uint64(7)
    assert lib.taco_gemm_workspace_bytes(256, 512, 128, None) == INVALID
    assert lib.taco_gemm_workspace_bytes(-1, 512, 128, ctypes.byref(v)) == INVALID
    assert lib.taco_gemm_workspace_bytes(100, 512, 128, ctypes.byref(v)) == UNSUPPORTED
    assert lib.taco_gemm_workspace_bytes(256, 512, 96, ctypes.byref(v)) == UNSUPPORTED
    assert lib.taco_gemm_workspace_bytes(0, 512, 128, ctypes.byref(v)) == OK and v.value == 0


def test_agoq_gemm_accumulate_validation(lib):
    f = lambda **k: lib.agoq_gemm_accumulate(k.get("a", A), k.get("b", A * 64), k.get("M", 256), k.get("N", 512),
                                             k.get("K", 128), k.get("block", 128), k.get("codes", A * 128),
                                             k.get("scale", A * 200), k.get("y", None), k.get("ws", None),
                                             k.get("ws_bytes", 0), None)
    assert f(block=256) == UNSUPPORTED
    assert f(M=100) == UNSUPPORTED and f(N=192) == UNSUPPORTED and f(K=32) == UNSUPPORTED
    assert f(M=-1) == INVALID
    assert f(M=0) == OK
    assert f(codes=None) == INVALID and f(scale=None) == INVALID
    assert f(codes=A * 128 + 8) == MISALIGNED
    assert f(scale=A * 128 + 64) == INVALID  # multipliers inside the codes
    assert f(y=A * 64) == INVALID            # output over an operand
    assert f(ws=A * 400 + 16, ws_bytes=4096) == MISALIGNED
    assert f(ws=A * 200 - 256, ws_bytes=4096) == INVALID  # workspace over the multipliers
