"""GPU parity: the sm_103a kernels, called through the C ABI, against the CPU
oracle on the same seeded inputs.

Small and ragged cases are compared element by element.  The full-size
GPT-shaped workloads (launched exactly as the benchmark launches them) are
and the full-size AGoQ buffers are compared on every block, with the oracle
run over all host cores.
"""

import math

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
from fp8_communication_compression_gb300 import api
from fp8_communication_compression_gb300 import workloads as W

import oracle_pool
from parity import (assert_codes_match, assert_recon_match, assert_scalars_match, gather_blocks,
                    gather_scalars, sample_blocks, to_dev_bf16, to_host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def no_watchdog_flags():
    api.taco_device_error(clear=True)
    yield
    assert api.taco_device_error(clear=True) == 0


def check_compress(bits: np.ndarray, block: int, e_target=1.0, eps=1e-12):
    x = to_dev_bf16(bits)
    c, a, s = api.taco_compress(x, block, e_target, eps)
    rc, ra, rs = oracle.compress(bits, block, e_target, eps)
    stats = assert_codes_match(to_host(c), rc)
    assert_scalars_match(to_host(a), ra, "alpha")
    assert_scalars_match(to_host(s), rs, "scale")
    return (c, a, s), stats


def check_decompress(c, a, s, block):
    out = api.taco_decompress(c, a, s, block)
    ref = oracle.decompress(to_host(c), to_host(a), to_host(s), block)
    assert_recon_match(to_host(out), ref.reshape(-1), block)
    outb = api.taco_decompress(c, a, s, block, out_dtype=torch.bfloat16)
    g = to_host(outb.float()).astype(np.float64).reshape(-1)
    r = ref.reshape(-1)
    # bf16 output: round-to-nearest of a value within 1e-6 of the oracle's
    assert np.all(np.abs(g - r) <= 2.0 ** -8 * np.abs(r) * (1 + 1e-5) + 1e-6 * np.abs(r).max())
    return out


# ------------------------------------------------------------ tiny case --

def test_tiny_round_trip_and_p2_reduce():
    name, n = "tiny_64x1024_n128", 128
    shards = []
    for p in range(2):
        bits = W.shard_input(name, p)
        (c, a, s), _ = check_compress(bits, n)
        check_decompress(c, a, s, n)
        shards.append((c, a, s))
    cs, as_, ss = zip(*shards)
    oc, oa, os_ = api.taco_reduce_shards(list(cs), list(as_), list(ss), n)
    rc, ra, rs = oracle.reduce_shards([to_host(c) for c in cs], [to_host(a) for a in as_],
                                      [to_host(s) for s in ss], n)
    assert_codes_match(to_host(oc), rc, "reduced codes")
    assert_scalars_match(to_host(oa), ra, "reduced alpha")
    assert_scalars_match(to_host(os_), rs, "reduced scale")
    check_decompress(oc, oa, os_, n)


# ------------------------------------------------- ragged / multi-tile --

@pytest.mark.parametrize("rows,d,block", [
    (1, 128, 128), (37, 384, 128), (1000, 256, 128), (1, 256, 256), (33, 512, 256),
    (500, 1024, 256), (2048, 4096, 128), (16384, 1024, 128), (8192, 2048, 256)])
def test_codec_shapes(rows, d, block):
    bits = W.tp_activation(rows * 7 + d, rows, d, channel_scale=True, block=block)
    (c, a, s), _ = check_compress(bits, block)
    check_decompress(c, a, s, block)


@pytest.mark.parametrize("e_target,eps", [(4.0, 1e-12), (0.25, 1e-6), (1.0, 1e-30)])
def test_codec_other_parameters(e_target, eps):
    bits = W.tp_activation(5, 64, 1024, channel_scale=True)
    (c, a, s), _ = check_compress(bits, 128, e_target, eps)
    check_decompress(c, a, s, 128)


def edge_blocks(n: int) -> np.ndarray:
    H = scipy.linalg.hadamard(n).astype(np.float32)
    rng = np.random.default_rng(3)
    blocks = [
        np.zeros(n),                                   # zero block
        -np.zeros(n),                                  # negative zeros
        np.eye(n)[5] * 1.0,                            # one-hot
        -np.eye(n)[n - 1] * 0.015625,                  # one-hot, small
        H[3] * 0.5,                                    # a Hadamard row
        np.full(n, 2.0),                               # constant
        np.where(np.arange(n) % 2, -1.0, 1.0) * 3.0,   # alternating signs
        rng.standard_normal(n) * 1e-39,                # bf16 subnormals
        rng.standard_normal(n) * 1e-30,                # tiny normals
        rng.standard_normal(n) * 1e15,                 # large
        np.concatenate([[1e4], rng.standard_normal(n - 1) * 1e-20]),  # one outlier
        rng.standard_normal(n) * 448.0,
        rng.standard_t(3, n) * 0.05,
    ]
    return np.stack(blocks).astype(np.float32)


@pytest.mark.parametrize("block", [128, 256])
def test_codec_edge_blocks(block):
    x = edge_blocks(block)
    bits = W.f32_to_bf16_bits(x)
    (c, a, s), _ = check_compress(bits, block)
    codes = to_host(c).reshape(-1, block)
    assert np.all((codes[0] & 0x7F) == 0) and np.all((codes[1] & 0x7F) == 0)
    assert to_host(s)[0] == 1.0 and to_host(s)[1] == 1.0
    out = check_decompress(c, a, s, block)
    assert np.all(to_host(out).reshape(-1, block)[:2] == 0.0)


# ------------------------------------------------------ INT8 ASH + DS --

@pytest.mark.parametrize("rows,d,block", [(64, 1024, 128), (37, 384, 128), (33, 512, 256),
                                          (4096, 2048, 128), (2048, 2560, 256)])
def test_int8_codec(rows, d, block):
    bits = W.tp_activation(rows + 3 * d, rows, d, channel_scale=True, zero_blocks=(1,), block=block)
    c, a, s = api.taco_compress_int8(to_dev_bf16(bits), block)
    rc, ra, rs = oracle.compress_int8(bits, block)
    g = to_host(c).astype(np.int32).reshape(-1)
    r = rc.astype(np.int32).reshape(-1)
    assert np.abs(g).max() <= 127 and np.abs(g - r).max() <= 1 and np.mean(g == r) >= 0.9999
    assert_scalars_match(to_host(a), ra, "alpha")
    assert_scalars_match(to_host(s), rs, "scale")
    out = api.taco_decompress_int8(c, a, s, block)
    ref = oracle.decompress_int8(to_host(c), to_host(a), to_host(s), block)
    assert_recon_match(to_host(out), ref.reshape(-1), block)
    outb = api.taco_decompress_int8(c, a, s, block, out_dtype=torch.bfloat16)
    gb = to_host(outb.float()).astype(np.float64).reshape(-1)
    assert np.all(np.abs(gb - ref.reshape(-1)) <= 2.0 ** -8 * np.abs(ref.reshape(-1)) * (1 + 1e-5)
                  + 1e-6 * np.abs(ref).max())


def test_int8_codec_edge_blocks():
    for block in (128, 256):
        bits = W.f32_to_bf16_bits(edge_blocks(block))
        c, a, s = api.taco_compress_int8(to_dev_bf16(bits), block)
        rc, ra, rs = oracle.compress_int8(bits, block)
        g = to_host(c).astype(np.int32).reshape(-1)
        assert np.abs(g - rc.astype(np.int32).reshape(-1)).max() <= 1
        assert_scalars_match(to_host(a), ra, "alpha")
        assert_scalars_match(to_host(s), rs, "scale")
        out = api.taco_decompress_int8(c, a, s, block)
        assert np.all(to_host(out).reshape(-1, block)[:2] == 0.0)


# ---------------------------------------------------------------- reduce --

@pytest.mark.parametrize("P,block", [(1, 128), (2, 256), (3, 128), (4, 128), (8, 256), (16, 128)])
def test_reduce_shard_counts(P, block):
    rows, d = 96, 1024
    shards = [api.taco_compress(to_dev_bf16(W.tp_activation(100 + p, rows, d, channel_scale=True,
                                                           block=block)), block) for p in range(P)]
    cs, as_, ss = zip(*shards)
    oc, oa, os_ = api.taco_reduce_shards(list(cs), list(as_), list(ss), block)
    rc, ra, rs = oracle.reduce_shards([to_host(c) for c in cs], [to_host(a) for a in as_],
                                      [to_host(s) for s in ss], block)
    assert_codes_match(to_host(oc), rc, "reduced codes")
    assert_scalars_match(to_host(oa), ra, "reduced alpha")
    assert_scalars_match(to_host(os_), rs, "reduced scale")


@pytest.mark.parametrize("P,block", [(4, 128), (8, 256)])
def test_reduce_is_invariant_to_shard_order(P, block):
    """Any order of the shards reduces to the same compressed sum, within
    the parity bar: the FP32 sum runs in shard order, so a permutation may
    change the last bit of a sum, hence at most one code step."""
    rows, d = 128, 1024
    shards = [api.taco_compress(to_dev_bf16(W.tp_activation(140 + p, rows, d, channel_scale=True,
                                                           block=block)), block) for p in range(P)]
    cs, as_, ss = (list(t) for t in zip(*shards))
    ref = [to_host(t) for t in api.taco_reduce_shards(cs, as_, ss, block)]
    for perm in (list(range(P))[::-1], [(3 * i + 1) % P for i in range(P)]):
        got = api.taco_reduce_shards([cs[i] for i in perm], [as_[i] for i in perm], [ss[i] for i in perm], block)
        assert_codes_match(to_host(got[0]), ref[0], "permuted codes")
        assert_scalars_match(to_host(got[1]), ref[1], "permuted alpha")
        assert_scalars_match(to_host(got[2]), ref[2], "permuted scale")


@pytest.mark.parametrize("P,block", [(1, 128), (3, 128), (4, 256)])
def test_reduce_with_16_byte_aligned_shards_equals_32_byte_aligned(P, block):
    """The reduce loads each shard's codes with one 32-byte load when every
    shard is 32-byte aligned, with two 16-byte loads otherwise: the same
    arithmetic on the same values, so the results are bit-identical.  The
    shards are copied to 16-byte (not 32-byte) aligned views, and against
    the oracle the reduce is checked on the misaligned path too."""
    rows, d = 96, 1024
    shards = [api.taco_compress(to_dev_bf16(W.tp_activation(160 + p, rows, d, channel_scale=True, block=block)),
                                block) for p in range(P)]
    cs, as_, ss = (list(t) for t in zip(*shards))
    ref = api.taco_reduce_shards(cs, as_, ss, block)
    n = rows * d
    buf = torch.empty(P * n + 64, dtype=torch.uint8, device="cuda")
    base = (32 - buf.data_ptr() % 32) % 32 + 16  # 16 bytes past a 32-byte boundary
    mis = [buf[base + p * n: base + (p + 1) * n].view(rows, d) for p in range(P)]
    for p in range(P):
        assert mis[p].data_ptr() % 32 == 16
        mis[p].copy_(cs[p])
    got = api.taco_reduce_shards(mis, as_, ss, block)
    for g, r in zip(got, ref):
        assert torch.equal(g.view(torch.uint8) if g.dtype == torch.uint8 else g.view(torch.int32),
                           r.view(torch.uint8) if r.dtype == torch.uint8 else r.view(torch.int32))
    rc, ra, rs = oracle.reduce_shards([to_host(c) for c in cs], [to_host(a) for a in as_],
                                      [to_host(s) for s in ss], block)
    assert_codes_match(to_host(got[0]), rc, "reduced codes, 16-byte aligned shards")
    assert_scalars_match(to_host(got[1]), ra, "reduced alpha, 16-byte aligned shards")


def test_reduce_shard_and_negation_gives_zero_blocks():
    block = 128
    c, a, s = api.taco_compress(to_dev_bf16(W.tp_activation(9, 32, 512, block=block)), block)
    neg = c ^ 0x80
    oc, oa, os_ = api.taco_reduce_shards([c, neg], [a, a], [s, s], block)
    assert torch.all((oc & 0x7F) == 0) and torch.all(os_ == 1.0)
    assert torch.all(oa == np.float32(math.sqrt(1.0 / np.float64(np.float32(1e-12)))))


@pytest.mark.parametrize("P,block,rows,d", [(1, 128, 40, 512), (2, 128, 96, 1024), (3, 256, 33, 512),
                                         (4, 128, 300, 1024), (8, 256, 64, 1280), (16, 128, 17, 384),
                                         (4, 256, 1000, 2048)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fused_reduce_decompress_equals_the_two_calls(P, block, rows, d, out_dtype):
    shards = [api.taco_compress(to_dev_bf16(W.tp_activation(200 + p, rows, d, channel_scale=True,
                                                           block=block)), block) for p in range(P)]
    cs, as_, ss = map(list, zip(*shards))
    rc, ra, rs = api.taco_reduce_shards(cs, as_, ss, block)
    ref_out = api.taco_decompress(rc, ra, rs, block, out_dtype=out_dtype)
    fc, fa, fs, fout = api.taco_reduce_decompress(cs, as_, ss, block, out_dtype=out_dtype)
    assert torch.equal(fc, rc) and torch.equal(fa, ra) and torch.equal(fs, rs)
    assert torch.equal(fout.view(torch.int32 if out_dtype == torch.float32 else torch.int16),
                       ref_out.view(torch.int32 if out_dtype == torch.float32 else torch.int16))
    oc, oa, os_ = oracle.reduce_shards([to_host(c) for c in cs], [to_host(a) for a in as_],
                                       [to_host(s) for s in ss], block)
    assert_codes_match(to_host(fc), oc, "fused codes")
    assert_scalars_match(to_host(fa), oa, "fused alpha")
    assert_scalars_match(to_host(fs), os_, "fused scale")
    if out_dtype == torch.float32:
        ref = oracle.decompress(to_host(fc), to_host(fa), to_host(fs), block)
        assert_recon_match(to_host(fout), ref.reshape(-1), block)


# ------------------------------------------------------------------ AGoQ --

@pytest.mark.parametrize("block", [128, 256])
def test_agoq_accumulate_steps(block):
    n = 1 << 16
    codes = torch.zeros(n, dtype=torch.uint8, device="cuda")
    scale = torch.ones(n // block, dtype=torch.float32, device="cuda")
    for k in range(4):
        g = W.agoq_grad(100 + k, n)
        prev_c, prev_s = to_host(codes).copy(), to_host(scale).copy()
        api.agoq_fp8_accumulate(codes, scale, to_dev_bf16(g), block)
        rc, rs = oracle.agoq_accumulate(prev_c, prev_s, g, block)
        # AGoQ arithmetic is fully specified in FP32: bit-identical results
        assert_codes_match(to_host(codes), rc, f"step {k} codes", exact=True)
        assert_scalars_match(to_host(scale), rs, f"step {k} scale", exact=True)


def test_agoq_zero_gradient_keeps_zero_buffer():
    n = 4096
    codes = torch.zeros(n, dtype=torch.uint8, device="cuda")
    scale = torch.ones(n // 128, dtype=torch.float32, device="cuda")
    api.agoq_fp8_accumulate(codes, scale, torch.zeros(n, dtype=torch.bfloat16, device="cuda"))
    assert torch.all(codes == 0) and torch.all(scale == 1.0)


@pytest.mark.parametrize("P,block", [(1, 128), (2, 128), (8, 128), (16, 256)])
def test_agoq_reduce(P, block):
    n = 1 << 15
    shards = []
    for p in range(P):
        c = torch.zeros(n, dtype=torch.uint8, device="cuda")
        s = torch.ones(n // block, dtype=torch.float32, device="cuda")
        api.agoq_fp8_accumulate(c, s, to_dev_bf16(W.agoq_grad(300 + p, n)), block)
        shards.append((c, s))
    cs, ss = zip(*shards)
    oc, os_ = api.agoq_reduce_shards(list(cs), list(ss), block)
    rc, rs = oracle.agoq_reduce([to_host(c) for c in cs], [to_host(s) for s in ss], block)
    assert_codes_match(to_host(oc), rc, exact=True)
    assert_scalars_match(to_host(os_), rs, "scale", exact=True)


def test_agoq_reduce_shard_and_negation_gives_zero():
    n = 1 << 13
    c = torch.zeros(n, dtype=torch.uint8, device="cuda")
    s = torch.ones(n // 128, dtype=torch.float32, device="cuda")
    api.agoq_fp8_accumulate(c, s, to_dev_bf16(W.agoq_grad(11, n)))
    oc, os_ = api.agoq_reduce_shards([c, c ^ 0x80], [s, s])
    assert torch.all((oc & 0x7F) == 0) and torch.all(os_ == 1.0)


# ------------------------------------------------------------------ LAAQ --

@pytest.mark.parametrize("bits", [4, 5, 6, 8])
@pytest.mark.parametrize("block", [32, 64, 128, 256])
def test_laaq_codec_is_bit_identical_to_the_oracle(bits, block):
    n = 96 * 1024 + 3 * 256  # several grid strides and a ragged tail of blocks
    x = W.tp_activation(500 + bits, n // 256, 256, channel_scale=True, zero_blocks=(2,), block=block)
    packed, scale = api.agoq_laaq_quantize(to_dev_bf16(x).reshape(-1), block, bits)
    rp, rs = oracle.laaq_quantize(x, block, bits)
    assert np.array_equal(to_host(packed), rp)
    assert np.array_equal(to_host(scale), rs)
    out32 = api.agoq_laaq_dequantize(packed, scale, n, block, bits, out_dtype=torch.float32)
    ref = oracle.laaq_dequantize(rp, rs, n, block, bits)
    assert np.array_equal(to_host(out32), ref)
    out16 = api.agoq_laaq_dequantize(packed, scale, n, block, bits, out_dtype=torch.bfloat16)
    assert np.array_equal(to_host(out16.view(torch.int16)).view(np.uint16), W.f32_to_bf16_bits(ref))


@pytest.mark.parametrize("bits,block", [(4, 128), (5, 64), (6, 32), (8, 256)])
def test_laaq_quantize_of_an_input_16_but_not_32_byte_aligned(bits, block):
    """The quantizer takes 32-byte loads when the input is 32-byte aligned
    and 16-byte loads otherwise: an input 16 bytes past a 32-byte boundary
    gives the same codes as the oracle too."""
    n = 40 * 1024 + 256
    x = W.tp_activation(540 + bits, n // 256, 256, channel_scale=True, zero_blocks=(1,), block=block)
    buf = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")
    xs = buf[8:]
    assert xs.data_ptr() % 32 == 16
    xs.copy_(to_dev_bf16(x).reshape(-1))
    packed, scale = api.agoq_laaq_quantize(xs, block, bits)
    rp, rs = oracle.laaq_quantize(x, block, bits)
    assert np.array_equal(to_host(packed), rp)
    assert np.array_equal(to_host(scale), rs)


# SiLU and RMSNorm recomputed from the stored quantised input (AGoQ 2.A).
# The GPU computes in fp32 (expf within 2 units in the last place, IEEE
# division and square root; the RMSNorm sum of squares compensated), the
# oracle in double on the same dequantised values, so the bar is the
# reconstruction bar, 1e-6 relative per element; bf16 outputs within 2^-8
# relative (half a bf16 step plus the fp32 error).
RECOMPUTE_RTOL = 1e-6
BF16_RTOL = 2.0 ** -8


def _stored_on_gpu(x_bits, block, bits):
    packed, scale = api.agoq_laaq_quantize(to_dev_bf16(x_bits).reshape(-1), block, bits)
    rp, rs = oracle.laaq_quantize(x_bits, block, bits)
    assert np.array_equal(to_host(packed), rp) and np.array_equal(to_host(scale), rs)
    return packed, scale, rp, rs


def _assert_close(got, ref, rtol, what):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bad = err > rtol * np.abs(ref) + 1e-30
    assert not bad.any(), f"{what}: {int(bad.sum())} values off, worst {float((err / np.maximum(np.abs(ref), 1e-300)).max()):.3g}"


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
@pytest.mark.parametrize("block", [32, 128, 256])
def test_laaq_silu_recompute_matches_the_oracle(bits, block):
    n = 96 * 1024 + 3 * 256
    x = W.tp_activation(560 + bits, n // 256, 256, channel_scale=True, zero_blocks=(2,), block=block)
    packed, scale, rp, rs = _stored_on_gpu(x, block, bits)
    ref = oracle.laaq_dequantize_silu(rp, rs, n, block, bits)
    out32 = api.agoq_laaq_dequantize_silu(packed, scale, n, block, bits, out_dtype=torch.float32)
    _assert_close(to_host(out32), ref, RECOMPUTE_RTOL, f"silu fp32, {bits} bits, block {block}")
    out16 = api.agoq_laaq_dequantize_silu(packed, scale, n, block, bits, out_dtype=torch.bfloat16)
    _assert_close(to_host(out16.float()), ref, BF16_RTOL, f"silu bf16, {bits} bits, block {block}")


def test_laaq_silu_recompute_over_the_whole_range():
    """Inputs spread over [-120, 120]: SiLU's saturation on both sides, and
    values below -88 where exp(-x) overflows fp32 (the result is then -0,
    within 1e-30 of the exact value)."""
    n = 64 * 1024
    v = np.random.default_rng(7).uniform(-120.0, 120.0, n).astype(np.float32)
    x = W.f32_to_bf16_bits(v)
    packed, scale, rp, rs = _stored_on_gpu(x, 128, 8)
    ref = oracle.laaq_dequantize_silu(rp, rs, n, 128, 8)
    out = api.agoq_laaq_dequantize_silu(packed, scale, n, 128, 8, out_dtype=torch.float32)
    _assert_close(to_host(out), ref, RECOMPUTE_RTOL, "silu over [-120, 120]")


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
@pytest.mark.parametrize("block,d", [(128, 4096), (32, 96), (256, 5120), (64, 1088)])
def test_laaq_rmsnorm_recompute_matches_the_oracle(bits, block, d):
    """37 rows (not a multiple of the 8 warps of a CTA), row lengths from 96
    to 5120, rows that are all zero."""
    rows = 37
    x = W.tp_activation(580 + bits, rows, d, channel_scale=True, zero_blocks=(3,), block=block)
    x[5] = 0
    packed, scale, rp, rs = _stored_on_gpu(x, block, bits)
    g = (1.0 + 0.5 * np.sin(np.arange(d))).astype(np.float32)
    ref = oracle.laaq_dequantize_rmsnorm(rp, rs, rows, d, g, 1e-6, block, bits)
    gd = torch.from_numpy(g).cuda()
    out32 = api.agoq_laaq_dequantize_rmsnorm(packed, scale, rows, d, gd, 1e-6, block, bits,
                                             out_dtype=torch.float32)
    _assert_close(to_host(out32), ref, RECOMPUTE_RTOL, f"rmsnorm fp32, {bits} bits, block {block}, d {d}")
    assert np.all(to_host(out32)[5] == 0)
    out16 = api.agoq_laaq_dequantize_rmsnorm(packed, scale, rows, d, gd, 1e-6, block, bits,
                                             out_dtype=torch.bfloat16)
    _assert_close(to_host(out16.float()), ref, BF16_RTOL, f"rmsnorm bf16, {bits} bits")


def test_laaq_recompute_full_size_4_bits():
    """A GPT-6.7B-sized activation [8192, 4096] stored in 4 bits: SiLU and
    RMSNorm recomputed, every element against the oracle."""
    rows, d = 8192, 4096
    x = W.tp_activation(599, rows, d, channel_scale=True, block=128)
    packed, scale, rp, rs = _stored_on_gpu(x, 128, 4)
    out = api.agoq_laaq_dequantize_silu(packed, scale, rows * d, 128, 4, out_dtype=torch.float32)
    _assert_close(to_host(out), oracle.laaq_dequantize_silu(rp, rs, rows * d, 128, 4), RECOMPUTE_RTOL,
                  "silu full size")
    g = np.ones(d, np.float32)
    out = api.agoq_laaq_dequantize_rmsnorm(packed, scale, rows, d, torch.from_numpy(g).cuda(), 1e-6, 128, 4,
                                           out_dtype=torch.float32)
    _assert_close(to_host(out), oracle.laaq_dequantize_rmsnorm(rp, rs, rows, d, g, 1e-6, 128, 4),
                  RECOMPUTE_RTOL, "rmsnorm full size")


@pytest.mark.parametrize("bits,block", [(4, 128), (5, 32), (6, 256), (8, 64)])
def test_laaq_codec_many_slots_per_lane(bits, block):
    """8.4 M elements: more lanes than one grid holds, so each lane takes
    several grid-stride slots per loop trip, and the last trip is ragged
    (some of its slots past the end)."""
    rows, d = 2051, 4096
    n = rows * d
    x = W.tp_activation(520 + bits, rows, d, channel_scale=True, zero_blocks=(5,), block=block)
    packed, scale = api.agoq_laaq_quantize(to_dev_bf16(x).reshape(-1), block, bits)
    rp, rs = oracle.laaq_quantize(x, block, bits)
    assert np.array_equal(to_host(packed), rp)
    assert np.array_equal(to_host(scale), rs)
    out16 = api.agoq_laaq_dequantize(packed, scale, n, block, bits, out_dtype=torch.bfloat16)
    ref = oracle.laaq_dequantize(rp, rs, n, block, bits)
    assert np.array_equal(to_host(out16.view(torch.int16)).view(np.uint16), W.f32_to_bf16_bits(ref))


# ------------------------------------------------------ E4M3 encoder --

def oracle_e4m3_thresholds() -> np.ndarray:
    """T[m] (m = 1 .. 126): the bit pattern of the smallest non-negative fp32
    value that the oracle's encoder maps to a magnitude code >= m.  Found by
    bisection over the bit patterns of non-negative floats, whose order is
    the order of their values; the nearest-value encoder is monotone in the
    value, so one threshold per code describes it on all 2^31 patterns."""
    T = np.zeros(127, dtype=np.int64)
    start = 0
    for m in range(1, 127):
        lo, hi = start, 0x7F800000  # +Inf saturates to magnitude 126
        while lo < hi:
            mid = (lo + hi) // 2
            v = float(np.array([mid], dtype=np.uint32).view(np.float32)[0])
            if (oracle.e4m3_encode(v) & 0x7F) >= m:
                hi = mid
            else:
                lo = mid + 1
        T[m] = start = lo
    return T


def test_e4m3_encoder_matches_the_oracle_on_every_fp32_pattern():
    """All 2^32 fp32 bit patterns through taco_e4m3_encode (the conversion the
    codec kernels use), against the oracle's encoder: its per-code thresholds
    for every non-NaN pattern, and NaN codes for NaN patterns."""
    T = torch.tensor(oracle_e4m3_thresholds(), dtype=torch.int64, device="cuda")
    chunk = 1 << 28
    for c in range(1 << 4):
        bits = torch.arange(c * chunk, (c + 1) * chunk, dtype=torch.int64, device="cuda")
        x = torch.where(bits >= 1 << 31, bits - (1 << 32), bits).to(torch.int32).view(torch.float32)
        codes = api.taco_e4m3_encode(x).to(torch.int64)
        mag = bits & 0x7FFFFFFF
        nan = mag > 0x7F800000
        expect = ((bits >> 31) << 7) | (torch.bucketize(mag, T, right=True) - 1)
        assert torch.equal(codes[~nan], expect[~nan]), f"chunk {c}"
        assert torch.all((codes[nan] & 0x7F) == 0x7F), f"chunk {c}: NaN"
        del bits, x, codes, mag, nan, expect


def test_e4m3_encoder_direct_oracle_sample_and_ragged_tail():
    """A direct check of the thresholds above: random bit patterns and the
    format's special values, encoded one by one by the oracle, with a length
    that leaves a ragged tail of 3 values."""
    g = np.random.default_rng(7)
    bits = g.integers(0, 1 << 32, size=20003, dtype=np.uint64).astype(np.uint32)
    special = np.array([0.0, -0.0, 448.0, -448.0, 464.0, 480.0, 1e30, np.inf, -np.inf, 2.0 ** -9,
                        2.0 ** -10, 2.0 ** -10 * 1.0000001, 0.5 * (416 + 448), -0.5 * (416 + 448)],
                       dtype=np.float32).view(np.uint32)
    bits[:special.size] = special
    v = bits.view(np.float32)
    v = v[~np.isnan(v)]
    v = np.ascontiguousarray(v[:len(v) - len(v) % 8 - 5])  # n % 8 == 3
    got = to_host(api.taco_e4m3_encode(torch.from_numpy(v).cuda()))
    assert np.array_equal(got, oracle.e4m3_encode_array(v))


# ----------------------------------------------- full-size workloads --

def assert_code_properties(codes: torch.Tensor, x_bits_dev: torch.Tensor | None, block: int):
    mag = (codes.reshape(-1, block) & 0x7F)
    assert not torch.any(mag == 0x7F), "NaN code"
    if x_bits_dev is not None:
        nonzero = (x_bits_dev.reshape(-1, block).view(torch.int16) & 0x7FFF).ne(0).any(dim=1)
        assert torch.all(mag.amax(dim=1)[nonzero] == 0x7E), "a non-zero block misses +-448"


@pytest.mark.parametrize("name", ["gpt2.7b_4096x2560_n128", "gpt6.7b_p4x8192x4096_n128",
                                  "gpt13b_p8x8192x5120_n256"])
def test_full_size_two_shot_local_path(name):
    """Every block of every shard, at full size, against the oracle run over
    all host cores: the compress of each shard, the reduce of the GPU's own
    compressed shards, and the decompress of the GPU's reduced codes."""
    w = W.WORKLOADS[name]
    P, rows, d, block = w["shards"], w["rows"], w["d"], w["block"]
    bits = np.stack([W.shard_input(name, p) for p in range(P)])
    x = to_dev_bf16(bits).reshape(P, rows, d)
    path = api.TwoShotLocal(P, rows, d, block)  # the benchmark's path
    out = path.run(x)
    if P > 1:  # the one-call reduce + decompress gives the same bits
        fpath = api.TwoShotLocal(P, rows, d, block, fused=True)
        fpath.codes.copy_(path.codes)
        fpath.alpha.copy_(path.alpha)
        fpath.scale.copy_(path.scale)
        fout = fpath.reduce_decompress()[3]
        assert torch.equal(fout.view(torch.int32), out.view(torch.int32))
        assert torch.equal(fpath.r_codes, path.r_codes)
        del fpath, fout
    torch.cuda.synchronize()
    assert_code_properties(path.codes, x, block)
    assert_code_properties(path.r_codes, None, block)
    del x
    codes, alpha, scale = to_host(path.codes), to_host(path.alpha), to_host(path.scale)
    # compress: every block of every shard
    rc, ra, rs = oracle_pool.compress(bits, block)
    del bits
    assert_codes_match(codes, rc, f"codes of all {P} shards")
    assert_scalars_match(alpha, ra, "alpha")
    assert_scalars_match(scale, rs, "scale")
    del rc, ra, rs
    if P > 1:
        # reduce of the GPU's own compressed shards, every block
        rc, ra, rs = oracle_pool.reduce_shards(codes, alpha, scale, block)
        assert_codes_match(to_host(path.r_codes), rc, "reduced codes")
        assert_scalars_match(to_host(path.r_alpha), ra, "reduced alpha")
        assert_scalars_match(to_host(path.r_scale), rs, "reduced scale")
        src = (to_host(path.r_codes), to_host(path.r_alpha), to_host(path.r_scale))
    else:
        src = (codes[0], alpha[0], scale[0])
        out = api.taco_decompress(path.codes[0], path.alpha[0], path.scale[0], block)
    # decompress of the (reduced) codes, every block
    ref = oracle_pool.decompress(*src, block)
    assert_recon_match(to_host(out), ref, block)


@pytest.mark.parametrize("P,rows,d,block,chunks", [(4, 512, 1024, 128, 8), (2, 96, 512, 256, 3),
                                                 (3, 100, 384, 128, 7)])
def test_host_pipeline_equals_device_path(P, rows, d, block, chunks):
    bits = np.stack([W.tp_activation(400 + p, rows, d, channel_scale=True, block=block) for p in range(P)])
    x = to_dev_bf16(bits).reshape(P, rows, d)
    ref = api.TwoShotLocal(P, rows, d, block).run(x).clone()
    pipe = api.HostPipeline(P, rows, d, block, chunks=chunks)
    h_in = torch.empty((P, rows, d), dtype=torch.bfloat16, pin_memory=True)
    h_in.view(torch.int16).copy_(torch.from_numpy(bits.view(np.int16)))
    h_out = torch.empty((rows, d), dtype=torch.float32, pin_memory=True)
    for _ in range(2):
        pipe.run(h_in, h_out)
        torch.cuda.synchronize()
        assert torch.equal(h_out.view(torch.int32), ref.cpu().view(torch.int32))


def test_host_pipeline_back_to_back_runs_and_bf16_output():
    """Runs on two inputs, alternated without synchronising, so that every
    run reuses the chunk workspace of the previous one while it may still be
    copying out; and the bf16-output pipeline."""
    P, rows, d, block = 4, 384, 2048, 128
    ins, refs = [], []
    for k in range(2):
        bits = np.stack([W.tp_activation(450 + 10 * k + p, rows, d, channel_scale=True, block=block)
                         for p in range(P)])
        x = to_dev_bf16(bits).reshape(P, rows, d)
        refs.append(api.TwoShotLocal(P, rows, d, block).run(x).cpu())
        h = torch.empty((P, rows, d), dtype=torch.bfloat16, pin_memory=True)
        h.view(torch.int16).copy_(torch.from_numpy(bits.view(np.int16)))
        ins.append(h)
    outs = [torch.empty((rows, d), dtype=torch.float32, pin_memory=True) for _ in range(2)]
    pipe = api.HostPipeline(P, rows, d, block, chunks=5)
    for _ in range(3):
        for k in range(2):
            pipe.run(ins[k], outs[k])
    torch.cuda.synchronize()
    for k in range(2):
        assert torch.equal(outs[k].view(torch.int32), refs[k].view(torch.int32))
    pb = api.HostPipeline(P, rows, d, block, chunks=3, out_dtype=torch.bfloat16)
    ob = torch.empty((rows, d), dtype=torch.bfloat16, pin_memory=True)
    pb.run(ins[0], ob)
    torch.cuda.synchronize()
    assert torch.equal(ob.view(torch.int16), refs[0].to(torch.bfloat16).view(torch.int16))


def test_two_paths_on_two_streams_at_once_match_sequential_runs():
    """The kernels keep no state between launches (only the watchdog flags),
    so two paths running concurrently on two streams give what they give
    one after the other."""
    P, rows, d, block = 4, 1024, 2048, 128
    xs = [to_dev_bf16(np.stack([W.tp_activation(470 + 10 * k + p, rows, d, channel_scale=True, block=block)
                                for p in range(P)])).reshape(P, rows, d) for k in range(2)]
    paths = [api.TwoShotLocal(P, rows, d, block) for _ in range(2)]
    refs = [paths[k].run(xs[k]).clone() for k in range(2)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(2)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(4):
        for k in range(2):
            paths[k].run(xs[k], stream=streams[k])
    torch.cuda.synchronize()
    for k in range(2):
        assert torch.equal(paths[k].out.view(torch.int32), refs[k].view(torch.int32))


def test_full_size_agoq_accumulate_and_reduce():
    """Every block of the 2^28-element buffer after each of the four
    accumulation steps, and every block of the P = 8 reduce of 2^25-element
    shards, against the oracle run over all host cores (bit-exact)."""
    a = W.AGOQ
    block, n = a["block"], a["n_main"]
    nb = n // block
    codes = torch.zeros(n, dtype=torch.uint8, device="cuda")
    scale = torch.ones(nb, dtype=torch.float32, device="cuda")
    for k, seed in enumerate(a["grad_seeds"]):
        g = W.agoq_grad(seed, n)
        prev_c, prev_s = to_host(codes), to_host(scale)
        api.agoq_fp8_accumulate(codes, scale, to_dev_bf16(g), block)
        rc, rs = oracle_pool.agoq_accumulate(prev_c, prev_s, g, block)
        assert_codes_match(to_host(codes), rc, f"step {k}", exact=True)
        assert_scalars_match(to_host(scale), rs, f"step {k} scale", exact=True)
        del g, prev_c, prev_s, rc, rs
    assert_code_properties(codes, None, block)
    del codes, scale
    ns = a["n_shard"]
    shards = []
    for p in range(a["reduce_P"]):
        c = torch.zeros(ns, dtype=torch.uint8, device="cuda")
        s = torch.ones(ns // block, dtype=torch.float32, device="cuda")
        for k in range(a["micro_batches"]):
            api.agoq_fp8_accumulate(c, s, to_dev_bf16(W.agoq_shard_grad(p, k, ns)), block)
        shards.append((c, s))
    cs, ss = zip(*shards)
    oc, os_ = api.agoq_reduce_shards(list(cs), list(ss), block)
    rc, rs = oracle_pool.agoq_reduce(np.stack([to_host(c) for c in cs]), np.stack([to_host(s) for s in ss]),
                                     block)
    assert_codes_match(to_host(oc), rc, "agoq reduce", exact=True)
    assert_scalars_match(to_host(os_), rs, "agoq reduce scale", exact=True)
