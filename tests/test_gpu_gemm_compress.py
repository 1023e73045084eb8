"""GPU parity of taco_gemm_compress: the tensor-core GEMM with the compressor
fused into its epilogue (AGoQ 2.C applied to the TACO compressor).

Two separate checks, so that the GEMM's rounding and the compressor's do
not blur each other:
  * the uncompressed Y the kernel accumulated (its optional fp32 output)
    against the oracle's float64 product, within an fp32-accumulation bound
    of (K/16 + 2) * 2^-22 * sum_k |a_k b_k| per element (each 16-deep MMA
    step and each accumulation rounds at most a few units in the last place
    of fp32, truncation allowed), and against cuBLAS (torch.matmul) within
    twice that;
  * the codes and scalars against the oracle's compressor run on that same
    fp32 Y: the codec's parity bar (codes >= 99.99 % bit-identical and never
    more than 1 E4M3 ULP apart, alpha and s within 1e-6 relative), since
    both sides take the code decisions from the same fp32 values.
The call without the optional output gives the same codes bit for bit.

Shapes whose tiles do not fill whole rounds of SMs, with K long enough for
pieces of 2048 or more, take the split tail (the last round's tiles cut
along K, their fp32 partial sums added in piece order through a workspace);
they are checked with and without it.  The split
changes the order of Y's fp32 additions, so the two Y differ in the last
places, each within the bound.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import oracle_pool
from fp8_communication_compression_gb300 import _lib, api
from fp8_communication_compression_gb300 import workloads as W

from parity import assert_codes_match, assert_recon_match, assert_scalars_match, to_dev_bf16, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def no_watchdog_flags():
    api.taco_device_error(clear=True)
    yield
    assert api.taco_device_error(clear=True) == 0


def operands(M, N, K, seed):
    """A: a TP activation (near-zero mixture, per-channel scales); B: weights
    N(0, 0.02^2), both rounded to bf16."""
    a = W.tp_activation(700 + seed, M, K, channel_scale=True)
    b = W.f32_to_bf16_bits(np.random.default_rng(800 + seed).normal(0.0, 0.02, (N, K)).astype(np.float32))
    return a, b


def sentinel_outputs(M, N):
    """Outputs filled with values the kernel never writes (code 0x7F, NaN
    scalars and Y), so that a block left unwritten fails the checks."""
    nb = M * N // 128
    return (torch.full((M, N), 0x7F, dtype=torch.uint8, device="cuda"),
            torch.full((nb,), float("nan"), device="cuda"), torch.full((nb,), float("nan"), device="cuda"))


def check_gemm_compress(M, N, K, seed=0, split_tail=True):
    a, b = operands(M, N, K, seed)
    ad, bd = to_dev_bf16(a), to_dev_bf16(b)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    c, al, sc = sentinel_outputs(M, N)
    c2, al2, sc2 = sentinel_outputs(M, N)
    api.taco_gemm_compress(ad, bd, codes=c, alpha=al, scale=sc, y_out=y, split_tail=split_tail)
    api.taco_gemm_compress(ad, bd, codes=c2, alpha=al2, scale=sc2, split_tail=split_tail)
    torch.cuda.synchronize()
    # the optional output changes nothing
    assert torch.equal(c, c2) and torch.equal(al, al2) and torch.equal(sc, sc2)
    # GEMM: against the float64 product, within the accumulation bound
    yg = to_host(y).astype(np.float64)
    ref = oracle.gemm_bt(a, b)
    mag = np.abs(oracle.bf16_to_f64(a)) @ np.abs(oracle.bf16_to_f64(b)).T
    bound = (K / 16 + 2) * 2.0 ** -22 * mag
    err = np.abs(yg - ref)
    assert np.all(err <= bound), f"GEMM error {float((err / np.maximum(bound, 1e-300)).max()):.2f} x the bound"
    cub = to_host(torch.matmul(ad.float(), bd.float().T)).astype(np.float64)
    assert np.all(np.abs(yg - cub) <= 2 * bound)
    # compressor: against the oracle on the same fp32 values
    rc, ra, rs = oracle.compress_f64(yg, 128)
    assert_codes_match(to_host(c), rc, "gemm codes")
    assert_scalars_match(to_host(al), ra, "gemm alpha")
    assert_scalars_match(to_host(sc), rs, "gemm scale")
    # and the codes decompress to the oracle's reconstruction of them
    out = api.taco_decompress(c, al, sc, 128)
    assert_recon_match(to_host(out), oracle.decompress(to_host(c), to_host(al), to_host(sc), 128), 128)
    return yg, ref


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 320), (384, 768, 1024), (128, 256, 4096),
                                   (256, 384, 128), (128, 128, 192)])
def test_gemm_compress_small_shapes(M, N, K):
    """Shapes that take 256-wide and 128-wide tiles (N = 384 and 128 only the
    latter), one to a few tiles."""
    check_gemm_compress(M, N, K)


@pytest.mark.parametrize("M,N,K", [(2048, 4096, 512), (4096, 4096, 128), (8192, 2048, 64)])
def test_gemm_compress_many_tiles_per_sm(M, N, K):
    """More tiles than SMs: the persistent CTAs take several tiles each
    (256, 512 and 512 tiles), so both tensor-memory accumulators are used and
    reused, and a tile's epilogue runs while the next tile's MMAs do."""
    check_gemm_compress(M, N, K, seed=3)


def expected_workspace(M, N, K, sms):
    """The split-tail rule of taco_gemm_workspace_bytes, restated: the tiles
    of the partial last round (all tiles when fewer than the SMs) split into
    the S in 2..4 dividing K / 64, into pieces of at least 32 k-blocks, that
    lowers ceil(rem S / sms) / S by at least 1/8 of a round the most."""
    bn = 256 if N % 256 == 0 else 128
    t, kb = (M // 128) * (N // bn), K // 64
    rem = t % sms if t >= sms else t
    best, split = (1.0 if rem else 0.0), 1
    for s in (2, 3, 4):
        if kb % s == 0 and kb // s >= 32:
            cost = -(-rem * s // sms) / s
            if cost <= best - 0.125:
                best, split = cost, s
    if split == 1:
        return 0
    return -(-16 * sms // 256) * 256 + rem * split * 128 * bn * 4


@pytest.mark.parametrize("M,N,K", [(384, 768, 1024), (128, 256, 4096), (256, 384, 128), (128, 128, 6144),
                                   (384, 768, 4096), (2048, 4096, 8192), (2048, 4096, 512), (4096, 4096, 128),
                                   (8192, 4096, 4096), (4096, 4096, 8192), (256, 512, 8192), (384, 640, 4096)])
def test_gemm_workspace_bytes_follows_the_split_rule(M, N, K):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert api.gemm_workspace_bytes(M, N, K) == expected_workspace(M, N, K, sms)


@pytest.mark.parametrize("M,N,K", [(384, 768, 4096), (128, 128, 6144), (2048, 4096, 8192)])
def test_gemm_compress_with_and_without_the_split_tail(M, N, K):
    """Shapes that take a split tail (S = 2, 3 and 4; 9, 1 and 104 tail
    tiles), computed without it and with it: both pass the same checks."""
    assert api.gemm_workspace_bytes(M, N, K) > 0
    check_gemm_compress(M, N, K, seed=4, split_tail=False)
    check_gemm_compress(M, N, K, seed=4, split_tail=True)


def test_gemm_compress_with_a_workspace_too_small_takes_no_split():
    """A workspace smaller than taco_gemm_workspace_bytes() is not used: the
    result is the unsplit kernel's, bit for bit."""
    M, N, K = 384, 768, 4096
    a, b = operands(M, N, K, 6)
    ad, bd = to_dev_bf16(a), to_dev_bf16(b)
    ref = api.taco_gemm_compress(ad, bd, split_tail=False)
    need = api.gemm_workspace_bytes(M, N, K)
    ws = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    c, al, sc = sentinel_outputs(M, N)
    st = _lib.load().taco_gemm_compress(ad.data_ptr(), bd.data_ptr(), M, N, K, 128, api.E_TARGET, api.EPS,
                                        c.data_ptr(), al.data_ptr(), sc.data_ptr(), None, ws.data_ptr(), need - 256,
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(c, ref[0]) and torch.equal(al, ref[1]) and torch.equal(sc, ref[2])
    assert bool(torch.all(ws == 0))  # untouched


def test_one_workspace_serves_shapes_in_any_order():
    """Calls of different shapes, one after another on the workspace kept per
    device, give the same bits as each shape on a fresh zeroed workspace of
    its own: a call leaves nothing behind that another shape would read."""
    shapes = [(2048, 4096, 8192), (384, 768, 4096), (128, 128, 6144), (2048, 4096, 8192), (384, 768, 4096)]
    ops = {s: tuple(to_dev_bf16(x) for x in operands(*s, 11)) for s in set(shapes)}
    fresh = {}
    for s in set(shapes):
        ws = torch.zeros(api.gemm_workspace_bytes(*s), dtype=torch.uint8, device="cuda")
        fresh[s] = api.taco_gemm_compress(*ops[s], workspace=ws)
    for s in shapes:
        c, al, sc = sentinel_outputs(s[0], s[1])
        api.taco_gemm_compress(*ops[s], codes=c, alpha=al, scale=sc)
        torch.cuda.synchronize()
        assert torch.equal(c, fresh[s][0]) and torch.equal(al, fresh[s][1]) and torch.equal(sc, fresh[s][2]), s


def test_gemm_compress_zero_rows_give_zero_blocks():
    """Rows of A that are all zero make rows of Y that are all zero: their
    blocks take the zero-block rule (codes +0, s = 1, alpha = sqrt(E/eps))."""
    M, N, K = 256, 256, 128
    a, b = operands(M, N, K, 5)
    a[7] = 0
    a[200] = 0
    c, al, sc = api.taco_gemm_compress(to_dev_bf16(a), to_dev_bf16(b))
    c, al, sc = to_host(c), to_host(al).reshape(M, -1), to_host(sc).reshape(M, -1)
    for r in (7, 200):
        assert np.all(c[r] == 0) and np.all(sc[r] == 1.0)
        assert np.allclose(al[r], np.float32(np.sqrt(1.0 / 1e-12)), rtol=1e-6)


def test_gemm_compress_full_size_gpt67b_down_projection():
    """The GPT-6.7B row-parallel MLP down-projection at TP = 4: [8192 tokens,
    4096] x [4096, 4096]^T, every block; the codes against the oracle's
    compressor on the kernel's own fp32 Y, Y against cuBLAS."""
    M, N, K = 8192, 4096, 4096
    a, b = operands(M, N, K, 9)
    ad, bd = to_dev_bf16(a), to_dev_bf16(b)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    c, al, sc = api.taco_gemm_compress(ad, bd, y_out=y)
    cub = torch.matmul(ad.float(), bd.float().T)
    mag = torch.matmul(ad.float().abs(), bd.float().abs().T)
    bound = 2 * (K / 16 + 2) * 2.0 ** -22 * mag
    assert bool(torch.all((y - cub).abs() <= bound))
    del cub, mag, bound
    rc, ra, rs = oracle_pool.compress_f64(to_host(y).astype(np.float64), 128)
    assert_codes_match(to_host(c), rc, "gemm codes, full size")
    assert_scalars_match(to_host(al), ra, "gemm alpha, full size")
    assert_scalars_match(to_host(sc), rs, "gemm scale, full size")


# ---------------------------------------------- AGoQ accumulate epilogue --

def grad_operands(M, N, K, seed):
    """A = dY^T: micro-batch output gradients N(0, (1e-4)^2) with 0.05 %
    outliers x1000 (the AGoQ gradient recipe); B = X^T: TP activations; both
    bf16 and K-major (K = the tokens)."""
    a = W.agoq_grad(900 + seed, M * K).reshape(M, K)
    b = W.tp_activation(950 + seed, N, K, channel_scale=True)
    return a, b


def check_agoq_gemm(M, N, K, steps=2, seed=0, split_tail=True):
    """agoq_gemm_accumulate over several micro-batches from the zero gradient:
    after every step the main gradient's codes and multipliers equal, bit for
    bit, the oracle's FP32 accumulation of the kernel's own fp32 G (the AGoQ
    arithmetic is a fixed FP32 sequence); G is checked against the float64
    product within the accumulation bound; the call without the optional
    output gives the same bits."""
    codes = torch.zeros((M, N), dtype=torch.uint8, device="cuda")
    scale = torch.ones(M * N // 128, dtype=torch.float32, device="cuda")
    rc, rs = np.zeros(M * N, np.uint8), np.ones(M * N // 128, np.float32)
    for step in range(steps):
        a, b = grad_operands(M, N, K, seed + 7 * step)
        ad, bd = to_dev_bf16(a), to_dev_bf16(b)
        c2, s2 = codes.clone(), scale.clone()
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        api.agoq_gemm_accumulate(ad, bd, codes, scale, y_out=y, split_tail=split_tail)
        api.agoq_gemm_accumulate(ad, bd, c2, s2, split_tail=split_tail)
        torch.cuda.synchronize()
        assert torch.equal(codes, c2) and torch.equal(scale, s2)
        yg = to_host(y)
        ref = oracle.gemm_bt(a, b)
        mag = np.abs(oracle.bf16_to_f64(a)) @ np.abs(oracle.bf16_to_f64(b)).T
        assert np.all(np.abs(yg.astype(np.float64) - ref) <= (K / 16 + 2) * 2.0 ** -22 * mag)
        rc, rs = oracle.agoq_accumulate_f32(rc, rs, yg, 128)
        assert_codes_match(to_host(codes), rc, f"main gradient codes, step {step}", exact=True)
        assert_scalars_match(to_host(scale), rs, f"main gradient multipliers, step {step}", exact=True)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 320), (2048, 4096, 512), (384, 640, 128)])
def test_agoq_gemm_accumulate_small_shapes(M, N, K):
    check_agoq_gemm(M, N, K)


@pytest.mark.parametrize("M,N,K", [(384, 640, 4096), (256, 512, 8192)])
def test_agoq_gemm_accumulate_with_and_without_the_split_tail(M, N, K):
    """Shapes that take a split tail (S = 2 with 128-wide tiles, S = 4 with
    256-wide ones), without it and with it."""
    assert api.gemm_workspace_bytes(M, N, K) > 0
    check_agoq_gemm(M, N, K, seed=2, split_tail=False)
    check_agoq_gemm(M, N, K, seed=2, split_tail=True)


def test_agoq_gemm_accumulate_full_size_weight_gradient():
    """A GPT-6.7B-shaped weight gradient, dW [4096, 4096] = dY^T X over 8192
    tokens, accumulated over two micro-batches: every block bit-exact."""
    check_agoq_gemm(4096, 4096, 8192, steps=2, seed=3)


# ------------------------------------------ LAAQ quantisation epilogue --

def check_laaq_gemm(M, N, K, bits, seed=0, split_tail=True):
    """agoq_gemm_laaq_quantize: the packed codes and multipliers equal, bit
    for bit, the oracle's fp32 quantisation of the kernel's own fp32 Y (the
    quantisation is a fixed FP32 sequence); Y is checked against the float64
    product within the accumulation bound; the call without the optional
    output gives the same bits; the library's dequantizer reads the stream
    back as the oracle's does."""
    a, b = operands(M, N, K, seed)
    ad, bd = to_dev_bf16(a), to_dev_bf16(b)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    p = torch.full((M * N * bits // 8,), 0xA5, dtype=torch.uint8, device="cuda")
    s = torch.full((M * N // 128,), float("nan"), dtype=torch.float32, device="cuda")
    api.agoq_gemm_laaq_quantize(ad, bd, bits, packed=p, scale=s, y_out=y, split_tail=split_tail)
    p2, s2 = api.agoq_gemm_laaq_quantize(ad, bd, bits, split_tail=split_tail)
    torch.cuda.synchronize()
    assert torch.equal(p, p2) and torch.equal(s, s2)
    yg = to_host(y)
    ref = oracle.gemm_bt(a, b)
    mag = np.abs(oracle.bf16_to_f64(a)) @ np.abs(oracle.bf16_to_f64(b)).T
    assert np.all(np.abs(yg.astype(np.float64) - ref) <= (K / 16 + 2) * 2.0 ** -22 * mag)
    rp, rs = oracle.laaq_quantize_f32(yg, 128, bits)
    assert np.array_equal(to_host(p), rp), f"packed codes differ at {bits} bits"
    assert np.array_equal(to_host(s), rs), f"multipliers differ at {bits} bits"
    out = api.agoq_laaq_dequantize(p, s, M * N, 128, bits, out_dtype=torch.float32)
    assert np.array_equal(to_host(out), oracle.laaq_dequantize(rp, rs, M * N, 128, bits))


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 384, 128), (2048, 4096, 512), (384, 768, 4096),
                                   (128, 128, 6144)])
def test_gemm_laaq_quantize_shapes(M, N, K, bits):
    """One tile (256 and 128 wide), several tiles per SM, and split tails of 2
    and 3 pieces, at every width."""
    check_laaq_gemm(M, N, K, bits, seed=bits)


@pytest.mark.parametrize("bits", [4, 6])
def test_gemm_laaq_quantize_without_the_split_tail(bits):
    check_laaq_gemm(384, 768, 4096, bits, seed=20 + bits, split_tail=False)


def test_gemm_laaq_quantize_full_size_4_bits():
    """A GPT-6.7B-sized activation, [8192 tokens, 4096] = X W^T with W [4096,
    4096], stored in 4 bits: every block bit-exact against the oracle's
    quantisation of the kernel's own fp32 Y."""
    M, N, K = 8192, 4096, 4096
    a, b = operands(M, N, K, 31)
    ad, bd = to_dev_bf16(a), to_dev_bf16(b)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    p, s = api.agoq_gemm_laaq_quantize(ad, bd, 4, y_out=y)
    cub = torch.matmul(ad.float(), bd.float().T)
    mag = torch.matmul(ad.float().abs(), bd.float().abs().T)
    assert bool(torch.all((y - cub).abs() <= 2 * (K / 16 + 2) * 2.0 ** -22 * mag))
    del cub, mag
    rp, rs = oracle.laaq_quantize_f32(to_host(y), 128, 4)
    assert np.array_equal(to_host(p), rp) and np.array_equal(to_host(s), rs)
