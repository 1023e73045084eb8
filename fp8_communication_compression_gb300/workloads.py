"""Seeded synthetic inputs for the TACO / AGoQ codec paths.

This module holds data generation only: it draws random numbers and rounds
them to bf16.  It holds none of the codec's arithmetic, so both the CUDA path
and the CPU oracle can be fed from it.

Distributions follow the data property described on the TACO page (section 1,
"data distribution"): tensor-parallel intermediate tensors are dense around
zero with a long tail.  The recipe per element is

  * with probability 0.9:  N(0, (1e-3)^2)
  * with probability 0.1:  0.05 * Student-t(nu = 3)
  * then an independent 0.1 % of positions are overwritten with +-U(2, 8).

Optional structure on top of that (GPT-shaped activations):

  * per-channel scale: column j of a [rows, d] tensor is multiplied by
    exp(U(ln 1e-3, 0)) (log-uniform in [1e-3, 1]), drawn once per tensor;
  * row spikes: each element independently with probability 1e-4 becomes
    +-100 x the row's RMS (RMS taken before spikes).

AGoQ micro-batch gradients (AGoQ page, section 2.B, QuanGrad) are
N(0, (1e-4)^2) with 0.05 % of positions multiplied by 1000.

Every array is generated in fixed-size chunks, each chunk from its own
PCG64 stream keyed by (seed, stream id, chunk index), so a tensor's first
elements do not depend on its total size and huge buffers can be produced
chunk by chunk.  float64 draws are rounded to fp32 and then to bf16 with
round-to-nearest-even on the bit pattern.
"""

from __future__ import annotations

import numpy as np

CHUNK = 1 << 22

_MIX = 0
_SCALES = 1
_SPIKES = 2
_GRAD = 3


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(list(key)))


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    # finite inputs only: the sum stays below 2^32
    b = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _mixture_chunk(seed: int, chunk: int, n: int) -> np.ndarray:
    g = _rng(seed, _MIX, chunk)
    x = g.standard_normal(n) * 1e-3
    heavy = np.flatnonzero(g.random(n) >= 0.9)
    x[heavy] = 0.05 * g.standard_t(3.0, heavy.size)
    out = np.flatnonzero(g.random(n) < 1e-3)
    sign = np.where(g.random(out.size) < 0.5, -1.0, 1.0)
    x[out] = sign * g.uniform(2.0, 8.0, out.size)
    return x


def mixture(seed: int, count: int) -> np.ndarray:
    """float64 draws of the near-zero / Student-t / outlier mixture."""
    x = np.empty(count, dtype=np.float64)
    for c, lo in enumerate(range(0, count, CHUNK)):
        hi = min(count, lo + CHUNK)
        x[lo:hi] = _mixture_chunk(seed, c, hi - lo)
    return x


def tp_activation(seed: int, rows: int, d: int, *, channel_scale: bool = False,
                  spikes: bool = False, zero_blocks: tuple = (), block: int = 128) -> np.ndarray:
    """bf16 bit pattern array [rows, d] shaped like a TP intermediate tensor.

    ``zero_blocks`` lists flat block indices (blocks are contiguous ``block``
    elements of the row-major tensor) that are forced to exactly zero.
    """
    x = mixture(seed, rows * d).reshape(rows, d)
    if channel_scale:
        g = _rng(seed, _SCALES)
        x *= np.exp(g.uniform(np.log(1e-3), 0.0, d))[None, :]
    if spikes:
        rms = np.sqrt(np.mean(x * x, axis=1))
        for r0 in range(0, rows, max(1, CHUNK // d)):
            r1 = min(rows, r0 + max(1, CHUNK // d))
            g = _rng(seed, _SPIKES, r0)
            sub = x[r0:r1]
            hit = g.random(sub.shape) < 1e-4
            sign = np.where(g.random(sub.shape) < 0.5, -1.0, 1.0)
            sub[hit] = (sign * 100.0 * rms[r0:r1, None])[hit]
    flat = x.reshape(-1)
    for b in zero_blocks:
        flat[b * block:(b + 1) * block] = 0.0
    return f32_to_bf16_bits(x.astype(np.float32))


def agoq_grad(seed: int, count: int) -> np.ndarray:
    """bf16 bits of one AGoQ micro-batch gradient of ``count`` elements."""
    out = np.empty(count, dtype=np.uint16)
    for c, lo in enumerate(range(0, count, CHUNK)):
        hi = min(count, lo + CHUNK)
        g = _rng(seed, _GRAD, c)
        v = g.standard_normal(hi - lo, dtype=np.float32) * np.float32(1e-4)
        hit = g.random(hi - lo, dtype=np.float32) < np.float32(5e-4)
        v[hit] *= np.float32(1000.0)
        out[lo:hi] = f32_to_bf16_bits(v)
    return out


# ---------------------------------------------------------------------------
# The five workloads.  Sizes are those of GPT-2.7B / 6.7B / 13B tensor-parallel
# activations and of an AGoQ gradient buffer; see the module docstring for the
# distributions.

E_TARGET = 1.0
EPS = 1e-12

WORKLOADS = {
    "tiny_64x1024_n128": dict(rows=64, d=1024, block=128, shards=2, seeds=(0, 1),
                              channel_scale=False, spikes=False, zero_first_last=True),
    "gpt2.7b_4096x2560_n128": dict(rows=4096, d=2560, block=128, shards=1, seeds=(0,),
                                   channel_scale=True, spikes=False, zero_first_last=False),
    "gpt6.7b_p4x8192x4096_n128": dict(rows=8192, d=4096, block=128, shards=4, seeds=(0, 1, 2, 3),
                                      channel_scale=True, spikes=False, zero_first_last=False),
    "gpt13b_p8x8192x5120_n256": dict(rows=8192, d=5120, block=256, shards=8,
                                     seeds=tuple(range(8)), channel_scale=True, spikes=True,
                                     zero_first_last=False),
}

AGOQ = dict(name="agoq_2p28_n128", n_main=1 << 28, block=128, micro_batches=4,
            grad_seeds=(100, 101, 102, 103), reduce_P=8, n_shard=1 << 25,
            shard_seeds=tuple(range(200, 208)))


def shard_input(name: str, shard: int, rows: int | None = None) -> np.ndarray:
    """bf16 bits [rows, d] of shard ``shard`` of workload ``name``.

    ``rows`` may shrink the tensor (the first ``rows`` rows of the same draw
    are not reproduced exactly for channel-scaled tensors; use it for small
    cases only).
    """
    w = WORKLOADS[name]
    r = w["rows"] if rows is None else rows
    nb = r * w["d"] // w["block"]
    zb = (0, nb - 1) if w["zero_first_last"] else ()
    return tp_activation(w["seeds"][shard], r, w["d"], channel_scale=w["channel_scale"],
                         spikes=w["spikes"], zero_blocks=zb, block=w["block"])


def agoq_shard_grad(shard: int, step: int, count: int) -> np.ndarray:
    """Micro-batch ``step`` gradient of AGoQ reduce shard ``shard``."""
    return agoq_grad(AGOQ["shard_seeds"][shard] * 16 + step, count)
