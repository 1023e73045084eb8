"""Python binding of the C ABI, with the same names.

Argument marshalling only: tensors are checked for device, dtype and
contiguity, outputs are allocated with torch when the caller passes none,
and the raw device pointers plus the current CUDA stream are handed to
libtaco.so.  Every step of the codec runs in the library's kernels.
"""

from __future__ import annotations

import ctypes
from typing import Sequence

import torch

from . import _lib

E_TARGET = 1.0
EPS = 1e-12


def _stream_handle(stream: torch.cuda.Stream | None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtypes, numel: int | None = None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")


_BF16 = (torch.bfloat16, torch.int16, torch.uint16)
_U8 = (torch.uint8, torch.float8_e4m3fn)


def _shape2(x: torch.Tensor):
    if x.dim() < 1:
        raise ValueError("tensor must have at least one dimension")
    d = x.shape[-1]
    return x.numel() // d if d else 0, d


def taco_compress(x: torch.Tensor, block: int = 128, e_target: float = E_TARGET, eps: float = EPS,
                  codes: torch.Tensor | None = None, alpha: torch.Tensor | None = None,
                  scale: torch.Tensor | None = None, stream=None):
    """bf16 [..., d] -> (codes uint8 [..., d], alpha fp32 [nb], scale fp32 [nb])."""
    _need(x, "x", _BF16)
    rows, d = _shape2(x)
    nb = rows * d // block if block else 0
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if alpha is None:
        alpha = torch.empty(nb, dtype=torch.float32, device=x.device)
    if scale is None:
        scale = torch.empty(nb, dtype=torch.float32, device=x.device)
    _need(codes, "codes", _U8, x.numel())
    _need(alpha, "alpha", (torch.float32,))
    _need(scale, "scale", (torch.float32,))
    st = _lib.load().taco_compress(x.data_ptr(), rows, d, block, e_target, eps, codes.data_ptr(),
                                   alpha.data_ptr(), scale.data_ptr(), _stream_handle(stream))
    _lib.check("taco_compress", st)
    return codes, alpha, scale


def taco_decompress(codes: torch.Tensor, alpha: torch.Tensor, scale: torch.Tensor, block: int = 128,
                    out_dtype: torch.dtype = torch.float32, out: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """(codes [..., d], alpha, scale) -> reconstruction [..., d] in fp32 or bf16."""
    _need(codes, "codes", _U8)
    _need(alpha, "alpha", (torch.float32,))
    _need(scale, "scale", (torch.float32,))
    rows, d = _shape2(codes)
    if out is None:
        out = torch.empty(codes.shape, dtype=out_dtype, device=codes.device)
    _need(out, "out", (torch.float32, torch.bfloat16), codes.numel())
    st = _lib.load().taco_decompress(codes.data_ptr(), alpha.data_ptr(), scale.data_ptr(), rows, d,
                                     block, out.data_ptr(), int(out.dtype == torch.bfloat16),
                                     _stream_handle(stream))
    _lib.check("taco_decompress", st)
    return out


def taco_compress_int8(x: torch.Tensor, block: int = 128, e_target: float = E_TARGET,
                       eps: float = EPS, codes: torch.Tensor | None = None,
                       alpha: torch.Tensor | None = None, scale: torch.Tensor | None = None,
                       stream=None):
    """ASH + DS with INT8 codes: bf16 [..., d] -> (codes int8, alpha, scale)."""
    _need(x, "x", _BF16)
    rows, d = _shape2(x)
    nb = rows * d // block if block else 0
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    if alpha is None:
        alpha = torch.empty(nb, dtype=torch.float32, device=x.device)
    if scale is None:
        scale = torch.empty(nb, dtype=torch.float32, device=x.device)
    _need(codes, "codes", (torch.int8,), x.numel())
    _need(alpha, "alpha", (torch.float32,))
    _need(scale, "scale", (torch.float32,))
    st = _lib.load().taco_compress_int8(x.data_ptr(), rows, d, block, e_target, eps, codes.data_ptr(),
                                        alpha.data_ptr(), scale.data_ptr(), _stream_handle(stream))
    _lib.check("taco_compress_int8", st)
    return codes, alpha, scale


def taco_decompress_int8(codes: torch.Tensor, alpha: torch.Tensor, scale: torch.Tensor,
                         block: int = 128, out_dtype: torch.dtype = torch.float32,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _need(codes, "codes", (torch.int8,))
    _need(alpha, "alpha", (torch.float32,))
    _need(scale, "scale", (torch.float32,))
    rows, d = _shape2(codes)
    if out is None:
        out = torch.empty(codes.shape, dtype=out_dtype, device=codes.device)
    _need(out, "out", (torch.float32, torch.bfloat16), codes.numel())
    st = _lib.load().taco_decompress_int8(codes.data_ptr(), alpha.data_ptr(), scale.data_ptr(), rows,
                                          d, block, out.data_ptr(), int(out.dtype == torch.bfloat16),
                                          _stream_handle(stream))
    _lib.check("taco_decompress_int8", st)
    return out


def taco_reduce_shards(codes: Sequence[torch.Tensor], alpha: Sequence[torch.Tensor],
                       scale: Sequence[torch.Tensor], block: int = 128, e_target: float = E_TARGET,
                       eps: float = EPS, out_codes: torch.Tensor | None = None,
                       out_alpha: torch.Tensor | None = None, out_scale: torch.Tensor | None = None,
                       stream=None):
    """Compressed sum of P compressed shards (two-shot local reduce)."""
    P = len(codes)
    if not (len(alpha) == P and len(scale) == P) or P == 0:
        raise ValueError("codes, alpha and scale must be non-empty lists of equal length")
    for p in range(P):
        _need(codes[p], f"codes[{p}]", _U8, codes[0].numel())
        _need(alpha[p], f"alpha[{p}]", (torch.float32,))
        _need(scale[p], f"scale[{p}]", (torch.float32,))
    rows, d = _shape2(codes[0])
    dev = codes[0].device
    if out_codes is None:
        out_codes = torch.empty(codes[0].shape, dtype=torch.uint8, device=dev)
    if out_alpha is None:
        out_alpha = torch.empty_like(alpha[0])
    if out_scale is None:
        out_scale = torch.empty_like(scale[0])
    cp, _k1 = _lib.ptr_array([c.data_ptr() for c in codes])
    ap, _k2 = _lib.ptr_array([a.data_ptr() for a in alpha])
    sp, _k3 = _lib.ptr_array([s.data_ptr() for s in scale])
    st = _lib.load().taco_reduce_shards(P, cp, ap, sp, rows, d, block, e_target, eps,
                                        out_codes.data_ptr(), out_alpha.data_ptr(),
                                        out_scale.data_ptr(), _stream_handle(stream))
    _lib.check("taco_reduce_shards", st)
    return out_codes, out_alpha, out_scale


def taco_reduce_decompress(codes: Sequence[torch.Tensor], alpha: Sequence[torch.Tensor],
                           scale: Sequence[torch.Tensor], block: int = 128, e_target: float = E_TARGET,
                           eps: float = EPS, out_codes: torch.Tensor | None = None,
                           out_alpha: torch.Tensor | None = None, out_scale: torch.Tensor | None = None,
                           out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float32,
                           stream=None):
    """Compressed sum of P compressed shards and its reconstruction, in one call
    (the shard-reduce and decompress kernels back to back)."""
    P = len(codes)
    if not (len(alpha) == P and len(scale) == P) or P == 0:
        raise ValueError("codes, alpha and scale must be non-empty lists of equal length")
    for p in range(P):
        _need(codes[p], f"codes[{p}]", _U8, codes[0].numel())
        _need(alpha[p], f"alpha[{p}]", (torch.float32,))
        _need(scale[p], f"scale[{p}]", (torch.float32,))
    rows, d = _shape2(codes[0])
    dev = codes[0].device
    if out_codes is None:
        out_codes = torch.empty(codes[0].shape, dtype=torch.uint8, device=dev)
    if out_alpha is None:
        out_alpha = torch.empty_like(alpha[0])
    if out_scale is None:
        out_scale = torch.empty_like(scale[0])
    if out is None:
        out = torch.empty(codes[0].shape, dtype=out_dtype, device=dev)
    _need(out, "out", (torch.float32, torch.bfloat16), codes[0].numel())
    cp, _k1 = _lib.ptr_array([c.data_ptr() for c in codes])
    ap, _k2 = _lib.ptr_array([a.data_ptr() for a in alpha])
    sp, _k3 = _lib.ptr_array([s.data_ptr() for s in scale])
    st = _lib.load().taco_reduce_decompress(P, cp, ap, sp, rows, d, block, e_target, eps,
                                            out_codes.data_ptr(), out_alpha.data_ptr(),
                                            out_scale.data_ptr(), out.data_ptr(),
                                            int(out.dtype == torch.bfloat16), _stream_handle(stream))
    _lib.check("taco_reduce_decompress", st)
    return out_codes, out_alpha, out_scale, out


def agoq_fp8_accumulate(main_codes: torch.Tensor, main_scale: torch.Tensor, grad: torch.Tensor,
                        block: int = 128, stream=None):
    """In place: main <- requantise(dequantise(main) + grad)."""
    _need(main_codes, "main_codes", _U8)
    _need(main_scale, "main_scale", (torch.float32,))
    _need(grad, "grad", _BF16, main_codes.numel())
    st = _lib.load().agoq_fp8_accumulate(main_codes.data_ptr(), main_scale.data_ptr(), grad.data_ptr(),
                                         main_codes.numel(), block, _stream_handle(stream))
    _lib.check("agoq_fp8_accumulate", st)
    return main_codes, main_scale


def agoq_reduce_shards(codes: Sequence[torch.Tensor], scale: Sequence[torch.Tensor], block: int = 128,
                       out_codes: torch.Tensor | None = None, out_scale: torch.Tensor | None = None,
                       stream=None):
    P = len(codes)
    if len(scale) != P or P == 0:
        raise ValueError("codes and scale must be non-empty lists of equal length")
    n = codes[0].numel()
    for p in range(P):
        _need(codes[p], f"codes[{p}]", _U8, n)
        _need(scale[p], f"scale[{p}]", (torch.float32,))
    if out_codes is None:
        out_codes = torch.empty(n, dtype=torch.uint8, device=codes[0].device)
    if out_scale is None:
        out_scale = torch.empty(n // block, dtype=torch.float32, device=codes[0].device)
    cp, _k1 = _lib.ptr_array([c.data_ptr() for c in codes])
    sp, _k2 = _lib.ptr_array([s.data_ptr() for s in scale])
    st = _lib.load().agoq_reduce_shards(P, cp, sp, n, block, out_codes.data_ptr(), out_scale.data_ptr(),
                                        _stream_handle(stream))
    _lib.check("agoq_reduce_shards", st)
    return out_codes, out_scale


def agoq_laaq_quantize(x: torch.Tensor, block: int = 128, bits: int = 4,
                       packed: torch.Tensor | None = None, scale: torch.Tensor | None = None,
                       stream=None):
    """bf16 activations -> (packed b-bit codes uint8 [n*bits/8], fp32 scale [n/block])."""
    _need(x, "x", _BF16)
    n = x.numel()
    if packed is None:
        packed = torch.empty(n * bits // 8, dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(n // block, dtype=torch.float32, device=x.device)
    _need(packed, "packed", (torch.uint8,), n * bits // 8)
    _need(scale, "scale", (torch.float32,))
    st = _lib.load().agoq_laaq_quantize(x.data_ptr(), n, block, bits, packed.data_ptr(),
                                        scale.data_ptr(), _stream_handle(stream))
    _lib.check("agoq_laaq_quantize", st)
    return packed, scale


def agoq_laaq_dequantize(packed: torch.Tensor, scale: torch.Tensor, n: int, block: int = 128,
                         bits: int = 4, out_dtype: torch.dtype = torch.bfloat16,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _need(packed, "packed", (torch.uint8,), n * bits // 8)
    _need(scale, "scale", (torch.float32,))
    if out is None:
        out = torch.empty(n, dtype=out_dtype, device=packed.device)
    _need(out, "out", (torch.float32, torch.bfloat16), n)
    st = _lib.load().agoq_laaq_dequantize(packed.data_ptr(), scale.data_ptr(), n, block, bits,
                                          out.data_ptr(), int(out.dtype == torch.bfloat16),
                                          _stream_handle(stream))
    _lib.check("agoq_laaq_dequantize", st)
    return out


def agoq_laaq_dequantize_silu(packed: torch.Tensor, scale: torch.Tensor, n: int, block: int = 128,
                              bits: int = 4, out_dtype: torch.dtype = torch.bfloat16,
                              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """SiLU recomputed from the stored quantised input: x_hat / (1 + exp(-x_hat))
    of the dequantised values, fp32 or bf16 [n] (AGoQ 2.A)."""
    _need(packed, "packed", (torch.uint8,), n * bits // 8)
    _need(scale, "scale", (torch.float32,))
    if out is None:
        out = torch.empty(n, dtype=out_dtype, device=packed.device)
    _need(out, "out", (torch.float32, torch.bfloat16), n)
    st = _lib.load().agoq_laaq_dequantize_silu(packed.data_ptr(), scale.data_ptr(), n, block, bits,
                                               out.data_ptr(), int(out.dtype == torch.bfloat16),
                                               _stream_handle(stream))
    _lib.check("agoq_laaq_dequantize_silu", st)
    return out


def agoq_laaq_dequantize_rmsnorm(packed: torch.Tensor, scale: torch.Tensor, rows: int, d: int,
                                 gamma: torch.Tensor, eps: float = 1e-6, block: int = 128, bits: int = 4,
                                 out_dtype: torch.dtype = torch.bfloat16, out: torch.Tensor | None = None,
                                 stream=None) -> torch.Tensor:
    """RMSNorm of each row of d values recomputed from the stored quantised
    input: x_hat / sqrt(mean(x_hat^2) + eps) * gamma, fp32 or bf16 [rows, d]
    (AGoQ 2.A)."""
    _need(packed, "packed", (torch.uint8,), rows * d * bits // 8)
    _need(scale, "scale", (torch.float32,))
    _need(gamma, "gamma", (torch.float32,), d)
    if out is None:
        out = torch.empty((rows, d), dtype=out_dtype, device=packed.device)
    _need(out, "out", (torch.float32, torch.bfloat16), rows * d)
    st = _lib.load().agoq_laaq_dequantize_rmsnorm(packed.data_ptr(), scale.data_ptr(), rows, d, block, bits,
                                                  gamma.data_ptr(), eps, out.data_ptr(),
                                                  int(out.dtype == torch.bfloat16), _stream_handle(stream))
    _lib.check("agoq_laaq_dequantize_rmsnorm", st)
    return out


def taco_e4m3_encode(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fp32 [n] -> E4M3FN codes uint8 [n] (round to nearest even, saturating at +-448)."""
    _need(x, "x", (torch.float32,))
    n = x.numel()
    if out is None:
        out = torch.empty(n, dtype=torch.uint8, device=x.device)
    _need(out, "out", (torch.uint8,), n)
    st = _lib.load().taco_e4m3_encode(x.data_ptr(), n, out.data_ptr(), _stream_handle(stream))
    _lib.check("taco_e4m3_encode", st)
    return out


_gemm_workspaces: dict = {}
_gemm_workspaces_replaced: list = []  # kept alive: a captured CUDA graph may still use them


def gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    """Bytes of workspace the GEMM's split tail takes for an M x N x K
    product on the current device (0: no split for this shape)."""
    v = ctypes.c_uint64(0)
    _lib.check("taco_gemm_workspace_bytes", _lib.load().taco_gemm_workspace_bytes(M, N, K, ctypes.byref(v)))
    return int(v.value)


def _gemm_workspace(device: torch.device, M: int, N: int, K: int, workspace: torch.Tensor | None):
    """(pointer, bytes) of the split tail's workspace: the caller's, or the
    one kept per device, grown when a shape needs more.  A new one is zeroed
    and synchronised, so it cannot be made during a CUDA graph capture (call
    once outside the capture first); one it replaces stays allocated, since
    a captured graph may still use it.  The kept one is shared by every
    stream of the device: GEMM calls that may run at the same time on
    different streams pass their own ``workspace``."""
    if workspace is not None:
        _need(workspace, "workspace", _U8)
        return workspace.data_ptr(), workspace.numel()
    need = gemm_workspace_bytes(M, N, K)
    if need == 0:
        return None, 0
    ws = _gemm_workspaces.get(device.index)
    if ws is None or ws.numel() < need:
        if torch.cuda.is_current_stream_capturing():
            raise RuntimeError("the GEMM's split-tail workspace must be made outside a CUDA graph capture: "
                               "call once with this shape before capturing, or pass workspace=")
        if ws is not None:
            _gemm_workspaces_replaced.append(ws)
        ws = torch.zeros(need, dtype=torch.uint8, device=device)
        torch.cuda.synchronize(device)
        _gemm_workspaces[device.index] = ws
    return ws.data_ptr(), ws.numel()


def _gemm_operands(a, b):
    _need(a, "a", _BF16)
    _need(b, "b", _BF16)
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[1]:
        raise ValueError("a must be [M, K] and b [N, K]")
    return a.shape[0], b.shape[0], a.shape[1]


def taco_gemm_compress(a: torch.Tensor, b: torch.Tensor, block: int = 128, e_target: float = E_TARGET,
                       eps: float = EPS, codes: torch.Tensor | None = None, alpha: torch.Tensor | None = None,
                       scale: torch.Tensor | None = None, y_out: torch.Tensor | None = None, stream=None,
                       split_tail: bool = True, workspace: torch.Tensor | None = None):
    """Y = a @ b.T on the tensor cores (a bf16 [M, K], b bf16 [N, K]), leaving
    the kernel compressed: (codes uint8 [M, N], alpha, scale fp32 [M * N / 128]).
    ``y_out`` (fp32 [M, N]), if given, also receives the uncompressed Y.
    ``split_tail`` lets the tiles of a partial last round of SMs be split
    along K, through ``workspace`` (uint8, zeroed before its first use, at
    least gemm_workspace_bytes(M, N, K) bytes) or, if that is None, a
    workspace kept per device."""
    M, N, K = _gemm_operands(a, b)
    nb = M * N // block if block else 0
    if codes is None:
        codes = torch.empty((M, N), dtype=torch.uint8, device=a.device)
    if alpha is None:
        alpha = torch.empty(nb, dtype=torch.float32, device=a.device)
    if scale is None:
        scale = torch.empty(nb, dtype=torch.float32, device=a.device)
    _need(codes, "codes", _U8, M * N)
    _need(alpha, "alpha", (torch.float32,), nb)
    _need(scale, "scale", (torch.float32,), nb)
    if y_out is not None:
        _need(y_out, "y_out", (torch.float32,), M * N)
    ws, ws_bytes = _gemm_workspace(a.device, M, N, K, workspace) if split_tail and M and N else (None, 0)
    st = _lib.load().taco_gemm_compress(a.data_ptr(), b.data_ptr(), M, N, K, block, e_target, eps,
                                        codes.data_ptr(), alpha.data_ptr(), scale.data_ptr(),
                                        y_out.data_ptr() if y_out is not None else None, ws, ws_bytes,
                                        _stream_handle(stream))
    _lib.check("taco_gemm_compress", st)
    return codes, alpha, scale


def agoq_gemm_accumulate(a: torch.Tensor, b: torch.Tensor, main_codes: torch.Tensor, main_scale: torch.Tensor,
                         block: int = 128, y_out: torch.Tensor | None = None, stream=None, split_tail: bool = True,
                         workspace: torch.Tensor | None = None):
    """In place: main <- requantise(dequantise(main) + a @ b.T), the GEMM
    (a bf16 [M, K], b bf16 [N, K]) on the tensor cores and the FP8
    accumulation in its epilogue.  main_codes uint8 [M, N], main_scale fp32
    [M * N / 128].  ``y_out`` (fp32 [M, N]), if given, also receives a @ b.T.
    ``split_tail`` and ``workspace`` as for taco_gemm_compress."""
    M, N, K = _gemm_operands(a, b)
    _need(main_codes, "main_codes", _U8, M * N)
    _need(main_scale, "main_scale", (torch.float32,), M * N // block if block else 0)
    if y_out is not None:
        _need(y_out, "y_out", (torch.float32,), M * N)
    ws, ws_bytes = _gemm_workspace(a.device, M, N, K, workspace) if split_tail and M and N else (None, 0)
    st = _lib.load().agoq_gemm_accumulate(a.data_ptr(), b.data_ptr(), M, N, K, block, main_codes.data_ptr(),
                                          main_scale.data_ptr(), y_out.data_ptr() if y_out is not None else None,
                                          ws, ws_bytes, _stream_handle(stream))
    _lib.check("agoq_gemm_accumulate", st)
    return main_codes, main_scale


def agoq_gemm_laaq_quantize(a: torch.Tensor, b: torch.Tensor, bits: int = 4, block: int = 128,
                            packed: torch.Tensor | None = None, scale: torch.Tensor | None = None,
                            y_out: torch.Tensor | None = None, stream=None, split_tail: bool = True,
                            workspace: torch.Tensor | None = None):
    """Y = a @ b.T on the tensor cores (a bf16 [M, K], b bf16 [N, K]),
    leaving the kernel as LAAQ codes: (packed uint8 [M * N * bits / 8],
    scale fp32 [M * N / 128]), readable by agoq_laaq_dequantize.  ``y_out``
    (fp32 [M, N]), if given, also receives Y; ``split_tail`` and
    ``workspace`` as for taco_gemm_compress."""
    M, N, K = _gemm_operands(a, b)
    nb = M * N // block if block else 0
    if packed is None:
        packed = torch.empty(M * N * bits // 8, dtype=torch.uint8, device=a.device)
    if scale is None:
        scale = torch.empty(nb, dtype=torch.float32, device=a.device)
    _need(packed, "packed", _U8, M * N * bits // 8)
    _need(scale, "scale", (torch.float32,), nb)
    if y_out is not None:
        _need(y_out, "y_out", (torch.float32,), M * N)
    ws, ws_bytes = _gemm_workspace(a.device, M, N, K, workspace) if split_tail and M and N else (None, 0)
    st = _lib.load().agoq_gemm_laaq_quantize(a.data_ptr(), b.data_ptr(), M, N, K, block, bits, packed.data_ptr(),
                                             scale.data_ptr(), y_out.data_ptr() if y_out is not None else None,
                                             ws, ws_bytes, _stream_handle(stream))
    _lib.check("agoq_gemm_laaq_quantize", st)
    return packed, scale


def taco_device_error(clear: bool = True) -> int:
    v = ctypes.c_uint32(0)
    _lib.check("taco_device_error", _lib.load().taco_device_error(ctypes.byref(v), int(clear)))
    return int(v.value)


class TwoShotLocal:
    """The two-shot AllReduce's on-GPU path for P shards of [rows, d]:
    compress all shards in one call, reduce them, decompress the result
    (two launches, or one ``taco_reduce_decompress`` call with ``fused=True``,
    which runs the same two kernels).  Buffers are allocated once; ``run`` only launches."""

    def __init__(self, P: int, rows: int, d: int, block: int = 128, device="cuda",
                 e_target: float = E_TARGET, eps: float = EPS, out_dtype=torch.float32,
                 fused: bool = False):
        self.P, self.rows, self.d, self.block = P, rows, d, block
        self.fused = fused
        self.e_target, self.eps = e_target, eps
        nb = rows * d // block
        self.codes = torch.empty((P, rows, d), dtype=torch.uint8, device=device)
        self.alpha = torch.empty((P, nb), dtype=torch.float32, device=device)
        self.scale = torch.empty((P, nb), dtype=torch.float32, device=device)
        self.r_codes = torch.empty((rows, d), dtype=torch.uint8, device=device)
        self.r_alpha = torch.empty(nb, dtype=torch.float32, device=device)
        self.r_scale = torch.empty(nb, dtype=torch.float32, device=device)
        self.out = torch.empty((rows, d), dtype=out_dtype, device=device)
        self._shard_codes = list(self.codes)
        self._shard_alpha = list(self.alpha)
        self._shard_scale = list(self.scale)

    def bytes_per_step(self) -> dict:
        """Algorithmic bytes each launch must move (reads + writes)."""
        n = self.rows * self.d
        nb = n // self.block
        comp = self.P * (2 * n + n + 8 * nb)
        red_in = self.P * (n + 8 * nb)
        red_out = n + 8 * nb
        dec_out = n * self.out.element_size()
        if self.fused:
            return {"compress": comp, "reduce_decompress": red_in + red_out + dec_out}
        return {"compress": comp, "reduce": red_in + red_out, "decompress": red_out + dec_out}

    def reduce_decompress(self, stream=None):
        return taco_reduce_decompress(self._shard_codes, self._shard_alpha, self._shard_scale,
                                      self.block, self.e_target, self.eps, self.r_codes, self.r_alpha,
                                      self.r_scale, self.out, stream=stream)

    def compress(self, x: torch.Tensor, stream=None):
        return taco_compress(x, self.block, self.e_target, self.eps, self.codes, self.alpha,
                             self.scale, stream=stream)

    def reduce(self, stream=None):
        return taco_reduce_shards(self._shard_codes, self._shard_alpha, self._shard_scale, self.block,
                                  self.e_target, self.eps, self.r_codes, self.r_alpha, self.r_scale,
                                  stream=stream)

    def decompress(self, stream=None) -> torch.Tensor:
        return taco_decompress(self.r_codes, self.r_alpha, self.r_scale, self.block, out=self.out,
                               stream=stream)

    def launches(self):
        """The step's launches, in order, as (name, callable taking x)."""
        if self.fused:
            return [("compress", self.compress), ("reduce_decompress", lambda x: self.reduce_decompress())]
        return [("compress", self.compress), ("reduce", lambda x: self.reduce()),
                ("decompress", lambda x: self.decompress())]

    def run(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        """x: bf16 [P, rows, d] on the device -> fp32/bf16 [rows, d]."""
        self.compress(x, stream)
        if self.fused:
            self.reduce_decompress(stream)
            return self.out
        self.reduce(stream)
        return self.decompress(stream)

    def run_host(self, x_host: torch.Tensor, out_host: torch.Tensor, x_dev: torch.Tensor,
                 stream=None) -> torch.Tensor:
        """Host-buffer variant: copies the pinned bf16 input [P, rows, d] to
        ``x_dev``, runs the path, and copies the result into the pinned
        ``out_host``, all asynchronously on the stream."""
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            x_dev.copy_(x_host, non_blocking=True)
            self.run(x_dev, s)
            out_host.copy_(self.out, non_blocking=True)
        return out_host


class HostPipeline:
    """The two-shot local path between pinned HOST buffers, overlapped: a
    handle on the library's native host pipeline (taco_host_pipeline_*).

    The rows are split into ``chunks`` chunks (the last may be shorter).
    For each chunk, one 2-D copy gathers its rows of all P shards to the
    device, compress, reduce and decompress run on a second stream, and the
    result is copied back on a third, so copies in, kernels and copies out
    of different chunks overlap.  Consecutive runs overlap chunk by chunk.
    The first run is ordered after the work queued on the current stream;
    every run makes the current stream wait for its result, which equals
    ``TwoShotLocal.run`` on the same data.  The device workspace is
    allocated once here (torch), the streams and events by the library."""

    def __init__(self, P: int, rows: int, d: int, block: int = 128, chunks: int = 4, device="cuda",
                 e_target: float = E_TARGET, eps: float = EPS, out_dtype=torch.float32):
        self.P, self.rows, self.d, self.block = P, rows, d, block
        self.e_target, self.eps, self.out_dtype = e_target, eps, out_dtype
        c = max(1, min(chunks, rows))
        self.R = -(-rows // c)
        self.C = -(-rows // self.R)
        self._h = None
        lib = _lib.load()
        h, ws = ctypes.c_void_p(), ctypes.c_uint64()
        with torch.cuda.device(torch.device(device)):
            st = lib.taco_host_pipeline_create(P, rows, d, block, chunks, int(out_dtype == torch.bfloat16),
                                               ctypes.byref(h), ctypes.byref(ws))
            _lib.check("taco_host_pipeline_create", st)
            self._h = h
            self.workspace = torch.empty(ws.value, dtype=torch.uint8, device=device)

    def run(self, x_host: torch.Tensor, out_host: torch.Tensor, stream=None) -> torch.Tensor:
        """x_host: pinned bf16 [P, rows, d]; out_host: pinned [rows, d] of out_dtype."""
        for t, name, dt, shape in ((x_host, "x_host", torch.bfloat16, (self.P, self.rows, self.d)),
                                   (out_host, "out_host", self.out_dtype, (self.rows, self.d))):
            if t.device.type != "cpu" or t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous host tensor {dt} {shape}")
        st = _lib.load().taco_host_pipeline_run(self._h, x_host.data_ptr(), out_host.data_ptr(),
                                                self.workspace.data_ptr(), self.e_target, self.eps,
                                                _stream_handle(stream))
        _lib.check("taco_host_pipeline_run", st)
        return out_host

    def __del__(self):
        if getattr(self, "_h", None) is not None and _lib is not None:
            try:
                _lib.load().taco_host_pipeline_destroy(self._h)
            except Exception:
                pass
            self._h = None