"""CPU oracle for the TACO ASH+DS codec and the AGoQ FP8 gradient paths.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
benchmark's CPU-baseline / reference leg may import this package.  The
product library never calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``taco_oracle.c`` (plain scalar C, double
precision); this module compiles it with gcc when needed and wraps it with
numpy arrays.  See the C file's header for the page sections each function
follows and for the readings taken where the pages are silent.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "taco_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

QMAX = 448.0


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode.argtypes = [f32]
            lib.oracle_fwht.restype = None
            lib.oracle_fwht.argtypes = [P, i32]
            lib.oracle_compress.argtypes = [P, i64, i64, i32, f32, f32, P, P, P]
            lib.oracle_compress_f64.argtypes = [P, i64, i64, i32, f32, f32, P, P, P]
            lib.oracle_decompress.argtypes = [P, P, P, i64, i64, i32, P]
            lib.oracle_reduce_shards.argtypes = [i32, P, P, P, i64, i64, i32, f32, f32, P, P, P]
            lib.oracle_agoq_accumulate.argtypes = [P, P, P, i64, i32]
            lib.oracle_agoq_reduce.argtypes = [i32, P, P, i64, i32, P, P]
            lib.oracle_agoq_accumulate_f32.argtypes = [P, P, P, i64, i32]
            lib.oracle_int8_roundtrip.argtypes = [P, i64, i64, i32, P]
            lib.oracle_compress_int8.argtypes = [P, i64, i64, i32, f32, f32, P, P, P]
            lib.oracle_decompress_int8.argtypes = [P, P, P, i64, i64, i32, P]
            lib.oracle_laaq_quantize.argtypes = [P, i64, i32, i32, P, P]
            lib.oracle_laaq_dequantize.argtypes = [P, P, i64, i32, i32, P]
            lib.oracle_laaq_quantize_f32.argtypes = [P, i64, i32, i32, P, P]
            lib.oracle_laaq_dequantize_silu.argtypes = [P, P, i64, i32, i32, P]
            lib.oracle_laaq_dequantize_rmsnorm.argtypes = [P, P, i64, i64, i32, i32, P, ctypes.c_double, P]
            for f in ("oracle_compress", "oracle_compress_f64", "oracle_decompress",
                      "oracle_reduce_shards", "oracle_agoq_accumulate", "oracle_agoq_reduce",
                      "oracle_agoq_accumulate_f32",
                      "oracle_int8_roundtrip", "oracle_compress_int8", "oracle_decompress_int8",
                      "oracle_laaq_quantize", "oracle_laaq_dequantize", "oracle_laaq_quantize_f32",
                      "oracle_laaq_dequantize_silu", "oracle_laaq_dequantize_rmsnorm"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int):
    if rc != 0:
        raise ValueError("oracle: invalid shape or argument")


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


# ------------------------------------------------------------------ E4M3 --

def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(int(code) & 0xFF)


def e4m3_decode_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    lib = _load()
    v = np.asarray(v, dtype=np.float32).reshape(-1)
    return np.array([lib.oracle_e4m3_encode(float(x)) for x in v], dtype=np.uint8)


def fwht(v: np.ndarray) -> np.ndarray:
    """Unnormalised Sylvester-order Walsh-Hadamard transform of each row."""
    out = np.array(v, dtype=np.float64, copy=True, order="C")
    n = out.shape[-1]
    flat = out.reshape(-1, n)
    lib = _load()
    for r in range(flat.shape[0]):
        lib.oracle_fwht(flat[r].ctypes.data_as(ctypes.c_void_p), n)
    return out


# ------------------------------------------------------------ TACO codec --

def compress(x_bf16: np.ndarray, block: int, e_target: float = 1.0, eps: float = 1e-12):
    """bf16 bits [rows, d] -> (codes uint8 [rows, d], alpha f32 [rows, d/block], scale f32)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, d = x.shape
    codes = np.empty((rows, d), dtype=np.uint8)
    alpha = np.empty((rows, d // block), dtype=np.float32)
    scale = np.empty((rows, d // block), dtype=np.float32)
    _check(_load().oracle_compress(_ptr(x), rows, d, block, e_target, eps, _ptr(codes),
                                   _ptr(alpha), _ptr(scale)))
    return codes, alpha, scale


def compress_f64(x: np.ndarray, block: int, e_target: float = 1.0, eps: float = 1e-12):
    x = np.ascontiguousarray(x, dtype=np.float64)
    rows, d = x.shape
    codes = np.empty((rows, d), dtype=np.uint8)
    alpha = np.empty((rows, d // block), dtype=np.float32)
    scale = np.empty((rows, d // block), dtype=np.float32)
    _check(_load().oracle_compress_f64(_ptr(x), rows, d, block, e_target, eps, _ptr(codes),
                                       _ptr(alpha), _ptr(scale)))
    return codes, alpha, scale


def decompress(codes: np.ndarray, alpha: np.ndarray, scale: np.ndarray, block: int) -> np.ndarray:
    """-> float64 reconstruction [rows, d]."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    a = np.ascontiguousarray(alpha, dtype=np.float32)
    s = np.ascontiguousarray(scale, dtype=np.float32)
    rows, d = c.shape
    assert a.size == rows * d // block and s.size == a.size
    out = np.empty((rows, d), dtype=np.float64)
    _check(_load().oracle_decompress(_ptr(c), _ptr(a), _ptr(s), rows, d, block, _ptr(out)))
    return out


def reduce_shards(codes, alphas, scales, block: int, e_target: float = 1.0, eps: float = 1e-12):
    """P compressed shards (lists) -> compressed sum (codes, alpha, scale)."""
    cs = [np.ascontiguousarray(c, dtype=np.uint8) for c in codes]
    As = [np.ascontiguousarray(a, dtype=np.float32) for a in alphas]
    Ss = [np.ascontiguousarray(s, dtype=np.float32) for s in scales]
    rows, d = cs[0].shape
    for c, a, s in zip(cs, As, Ss):
        assert c.shape == (rows, d) and a.size == rows * d // block and s.size == a.size
    out_c = np.empty((rows, d), dtype=np.uint8)
    out_a = np.empty((rows, d // block), dtype=np.float32)
    out_s = np.empty((rows, d // block), dtype=np.float32)
    _check(_load().oracle_reduce_shards(len(cs), _ptr_array(cs), _ptr_array(As), _ptr_array(Ss),
                                        rows, d, block, e_target, eps, _ptr(out_c), _ptr(out_a),
                                        _ptr(out_s)))
    return out_c, out_a, out_s


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gemm_bt(a_bf16: np.ndarray, b_bf16: np.ndarray) -> np.ndarray:
    """Y = A B^T in float64 for bf16 A [M, K] and B [N, K] (the GEMM whose
    output the fused kernel compresses; AGoQ 2.C).  Every product of two
    bf16 values is exact in float64; the sums are numpy's float64 matrix
    product (a library primitive)."""
    return bf16_to_f64(a_bf16) @ bf16_to_f64(b_bf16).T


def gemm_compress(a_bf16: np.ndarray, b_bf16: np.ndarray, block: int = 128, e_target: float = 1.0,
                  eps: float = 1e-12):
    """The fused GEMM + compress, as two plain steps: Y = A B^T in float64,
    then the TACO compressor on Y's blocks (compress_f64)."""
    return compress_f64(gemm_bt(a_bf16, b_bf16), block, e_target, eps)


# ------------------------------------------------------------------ AGoQ --

def agoq_accumulate(codes: np.ndarray, scale: np.ndarray, grad_bf16: np.ndarray, block: int = 128):
    """Returns the new (codes, scale); the inputs are not modified."""
    c = np.array(codes, dtype=np.uint8, copy=True).reshape(-1)
    s = np.array(scale, dtype=np.float32, copy=True).reshape(-1)
    g = np.ascontiguousarray(grad_bf16, dtype=np.uint16).reshape(-1)
    assert g.size == c.size and s.size == c.size // block
    _check(_load().oracle_agoq_accumulate(_ptr(c), _ptr(s), _ptr(g), c.size, block))
    return c, s


def agoq_accumulate_f32(codes: np.ndarray, scale: np.ndarray, grad_f32: np.ndarray, block: int = 128):
    """The accumulation step with an fp32 gradient (the GEMM-fused form,
    AGoQ 2.C); returns the new (codes, scale), the inputs unmodified."""
    c = np.array(codes, dtype=np.uint8, copy=True).reshape(-1)
    s = np.array(scale, dtype=np.float32, copy=True).reshape(-1)
    g = np.ascontiguousarray(grad_f32, dtype=np.float32).reshape(-1)
    assert g.size == c.size and s.size == c.size // block
    _check(_load().oracle_agoq_accumulate_f32(_ptr(c), _ptr(s), _ptr(g), c.size, block))
    return c, s


def gemm_agoq_accumulate(a_bf16: np.ndarray, b_bf16: np.ndarray, codes: np.ndarray, scale: np.ndarray,
                         block: int = 128):
    """The fused weight-gradient GEMM + FP8 accumulation, as two plain steps:
    Y = A B^T in float64, rounded to fp32, then the FP32 accumulation step."""
    return agoq_accumulate_f32(codes, scale, gemm_bt(a_bf16, b_bf16).astype(np.float32), block)


def agoq_reduce(codes, scales, block: int = 128):
    cs = [np.ascontiguousarray(c, dtype=np.uint8).reshape(-1) for c in codes]
    ss = [np.ascontiguousarray(s, dtype=np.float32).reshape(-1) for s in scales]
    n = cs[0].size
    out_c = np.empty(n, dtype=np.uint8)
    out_s = np.empty(n // block, dtype=np.float32)
    _check(_load().oracle_agoq_reduce(len(cs), _ptr_array(cs), _ptr_array(ss), n, block,
                                      _ptr(out_c), _ptr(out_s)))
    return out_c, out_s


def agoq_dequantise(codes: np.ndarray, scale: np.ndarray, block: int = 128) -> np.ndarray:
    """decode(code) * m per block, as float64 (the stored AGoQ scale m is the
    dequantisation multiplier max|g| / 448)."""
    table = e4m3_decode_table()
    c = np.asarray(codes, dtype=np.uint8).reshape(-1, block)
    return (table[c] * np.asarray(scale, dtype=np.float64).reshape(-1, 1)).reshape(-1)


# --------------------------------------------------------- INT8 baseline --

def int8_roundtrip(x_bf16: np.ndarray, block: int) -> np.ndarray:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, d = x.shape
    out = np.empty((rows, d), dtype=np.float64)
    _check(_load().oracle_int8_roundtrip(_ptr(x), rows, d, block, _ptr(out)))
    return out


# ------------------------------------------------------ INT8 ASH + DS ----

def compress_int8(x_bf16: np.ndarray, block: int, e_target: float = 1.0, eps: float = 1e-12):
    """ASH + DS with INT8 codes: (codes int8 [rows, d], alpha, scale)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, d = x.shape
    codes = np.empty((rows, d), dtype=np.int8)
    alpha = np.empty((rows, d // block), dtype=np.float32)
    scale = np.empty((rows, d // block), dtype=np.float32)
    _check(_load().oracle_compress_int8(_ptr(x), rows, d, block, e_target, eps, _ptr(codes),
                                        _ptr(alpha), _ptr(scale)))
    return codes, alpha, scale


def decompress_int8(codes: np.ndarray, alpha: np.ndarray, scale: np.ndarray, block: int) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.int8)
    a = np.ascontiguousarray(alpha, dtype=np.float32)
    s = np.ascontiguousarray(scale, dtype=np.float32)
    rows, d = c.shape
    out = np.empty((rows, d), dtype=np.float64)
    _check(_load().oracle_decompress_int8(_ptr(c), _ptr(a), _ptr(s), rows, d, block, _ptr(out)))
    return out


# ------------------------------------------------------------------ LAAQ --

def laaq_quantize(x_bf16: np.ndarray, block: int = 128, bits: int = 4):
    """bf16 bits [n] -> (packed uint8 [n * bits / 8], scale fp32 [n / block])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(-1)
    packed = np.zeros(x.size * bits // 8, dtype=np.uint8)
    scale = np.empty(x.size // block, dtype=np.float32)
    _check(_load().oracle_laaq_quantize(_ptr(x), x.size, block, bits, _ptr(packed), _ptr(scale)))
    return packed, scale


def laaq_quantize_f32(x_f32: np.ndarray, block: int = 128, bits: int = 4):
    """The quantisation of fp32 values (the GEMM-fused form, AGoQ 2.C):
    fp32 [n] -> (packed uint8 [n * bits / 8], scale fp32 [n / block])."""
    x = np.ascontiguousarray(x_f32, dtype=np.float32).reshape(-1)
    packed = np.zeros(x.size * bits // 8, dtype=np.uint8)
    scale = np.empty(x.size // block, dtype=np.float32)
    _check(_load().oracle_laaq_quantize_f32(_ptr(x), x.size, block, bits, _ptr(packed), _ptr(scale)))
    return packed, scale


def gemm_laaq_quantize(a_bf16: np.ndarray, b_bf16: np.ndarray, block: int = 128, bits: int = 4):
    """The GEMM with LAAQ quantisation of its output, as two plain steps:
    Y = A B^T in float64, rounded to fp32, then the fp32 quantisation."""
    return laaq_quantize_f32(gemm_bt(a_bf16, b_bf16).astype(np.float32), block, bits)


def laaq_dequantize(packed: np.ndarray, scale: np.ndarray, n: int, block: int = 128, bits: int = 4):
    p = np.ascontiguousarray(packed, dtype=np.uint8).reshape(-1)
    s = np.ascontiguousarray(scale, dtype=np.float32).reshape(-1)
    out = np.empty(n, dtype=np.float32)
    _check(_load().oracle_laaq_dequantize(_ptr(p), _ptr(s), n, block, bits, _ptr(out)))
    return out


def laaq_dequantize_silu(packed: np.ndarray, scale: np.ndarray, n: int, block: int = 128, bits: int = 4):
    """SiLU recomputed from the stored quantised input (AGoQ 2.A): float64 [n]."""
    p = np.ascontiguousarray(packed, dtype=np.uint8).reshape(-1)
    s = np.ascontiguousarray(scale, dtype=np.float32).reshape(-1)
    out = np.empty(n, dtype=np.float64)
    _check(_load().oracle_laaq_dequantize_silu(_ptr(p), _ptr(s), n, block, bits, _ptr(out)))
    return out


def laaq_dequantize_rmsnorm(packed: np.ndarray, scale: np.ndarray, rows: int, d: int, gamma: np.ndarray,
                            eps: float = 1e-6, block: int = 128, bits: int = 4):
    """RMSNorm of each row of d values recomputed from the stored quantised
    input (AGoQ 2.A): float64 [rows, d]."""
    p = np.ascontiguousarray(packed, dtype=np.uint8).reshape(-1)
    s = np.ascontiguousarray(scale, dtype=np.float32).reshape(-1)
    g = np.ascontiguousarray(gamma, dtype=np.float32).reshape(-1)
    assert g.size == d
    out = np.empty(rows * d, dtype=np.float64)
    _check(_load().oracle_laaq_dequantize_rmsnorm(_ptr(p), _ptr(s), rows, d, block, bits, _ptr(g), eps, _ptr(out)))
    return out.reshape(rows, d)
