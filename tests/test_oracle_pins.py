"""Pins for the CPU oracle: facts that do not come from the oracle itself.

Each test checks one oracle function against something fixed independently:
hand-worked examples from the page definitions (tests/golden), torch's
float8_e4m3fn conversion, scipy's Sylvester Hadamard matrix, closed forms,
invariants and the E4M3 rounding error bound.  Everything here runs on CPU.
"""

import json
import math
import os
import struct

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
from fp8_communication_compression_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits_to_f32(h: str) -> float:
    return struct.unpack("<f", struct.pack("<I", int(h, 16)))[0]


def f32(v):
    return np.float32(v)


def bf16(values) -> np.ndarray:
    return W.f32_to_bf16_bits(np.asarray(values, dtype=np.float32))


def torch_e4m3_decode_table() -> np.ndarray:
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def torch_e4m3_encode(v32: np.ndarray) -> np.ndarray:
    """torch's RNE fp32 -> float8_e4m3fn, with the saturation at 448 applied first
    (torch maps |v| > 464 to NaN; the saturating format keeps them at 448)."""
    v = np.clip(np.asarray(v32, dtype=np.float32), -448.0, 448.0)
    neg0 = np.signbit(np.asarray(v32, dtype=np.float32))
    v = np.where(neg0 & (v == 0), np.float32(-0.0), v)
    return torch.from_numpy(v.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    a = a.astype(np.int32)
    b = b.astype(np.int32)
    ma, mb = a & 0x7F, b & 0x7F
    sa = np.where(ma == 0, 0, a >> 7)
    sb = np.where(mb == 0, 0, b >> 7)
    sia = np.where(sa == 1, -ma, ma)
    sib = np.where(sb == 1, -mb, mb)
    return np.abs(sia - sib)


# ------------------------------------------------------------------ E4M3 ---

def test_e4m3_decode_matches_torch_for_all_256_codes():
    mine = oracle.e4m3_decode_table()
    ref = torch_e4m3_decode_table()
    nan = np.isnan(ref)
    assert list(np.flatnonzero(nan)) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))


def test_e4m3_known_values_from_the_format_definition():
    g = json.load(open(os.path.join(GOLDEN, "e4m3_known.json")))
    for e in g["decode"]:
        v = oracle.e4m3_decode(e["code"])
        assert v == e["value"] and math.copysign(1, v) == math.copysign(1, e["value"]), e
    for c in g["nan_codes"]:
        assert math.isnan(oracle.e4m3_decode(c))
    for e in g["encode"]:
        assert oracle.e4m3_encode(e["value"]) == e["code"], e


def test_e4m3_encode_matches_torch_on_midpoints_and_neighbours():
    table = torch_e4m3_decode_table()[:127]
    mids = (table[:-1] + table[1:]) / 2
    pts = np.concatenate([table, mids]).astype(np.float32)
    probe = [pts, np.nextafter(pts, np.float32(np.inf)), np.nextafter(pts, np.float32(-np.inf))]
    rng = np.random.default_rng(7)
    probe.append(rng.uniform(-448, 448, 20000).astype(np.float32))
    probe.append((rng.standard_normal(20000) * 0.01).astype(np.float32))
    probe.append(np.array([448.0, 449.0, 463.9, 464.0, 470.0, 1e20, 3e38, -0.0, 0.0, 1e-30,
                           -1e-30, -448.5], dtype=np.float32))
    v = np.concatenate([p.reshape(-1) for p in probe]).astype(np.float32)
    v = np.concatenate([v, -v])
    mine = oracle.e4m3_encode_array(v)
    ref = torch_e4m3_encode(v)
    assert np.array_equal(mine, ref)


def test_e4m3_encode_never_emits_nan_and_inverts_decode():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c
    for v in (1e38, -1e38, 500.0, -500.0):
        assert oracle.e4m3_encode(v) & 0x7F == 0x7E


# ------------------------------------------------------------- Hadamard ---

@pytest.mark.parametrize("n", [2, 4, 8, 16, 32, 64, 128, 256, 512, 1024])
def test_fwht_equals_scipy_sylvester_matrix(n):
    H = scipy.linalg.hadamard(n).astype(np.float64)
    assert np.array_equal(oracle.fwht(np.eye(n)), H.T)
    rng = np.random.default_rng(n)
    x = rng.standard_normal((3, n))
    assert np.allclose(oracle.fwht(x), x @ H.T, rtol=0, atol=1e-10 * n)


@pytest.mark.parametrize("n", [2, 8, 128, 1024])
def test_normalised_hadamard_is_orthogonal_and_involutive(n):
    c = 1.0 / math.sqrt(n)
    Hn = c * oracle.fwht(np.eye(n))
    assert np.allclose(Hn @ Hn, np.eye(n), atol=1e-12)
    rng = np.random.default_rng(1)
    x = rng.standard_normal(n)
    y = c * oracle.fwht(x)
    assert math.isclose(np.dot(y, y), np.dot(x, x), rel_tol=1e-12)
    assert np.allclose(c * oracle.fwht(y), x, atol=1e-12)


# ------------------------------------------------- hand-worked examples ---

def test_hand_worked_examples():
    g = json.load(open(os.path.join(GOLDEN, "hand_examples.json")))
    for ex in g["examples"]:
        n = ex["block"]
        x = bf16(ex["x"]).reshape(1, n)
        codes, alpha, scale = oracle.compress(x, n, g["e_target"], g["eps"])
        assert codes.reshape(-1).tolist() == ex["codes"], ex["name"]
        assert alpha.reshape(-1)[0] == f32(bits_to_f32(ex["alpha_bits"])), ex["name"]
        assert scale.reshape(-1)[0] == f32(bits_to_f32(ex["scale_bits"])), ex["name"]
        xhat = oracle.decompress(codes, alpha, scale, n).reshape(-1)
        assert np.allclose(xhat, ex["xhat"], rtol=1e-6, atol=1e-12), ex["name"]


# -------------------------------------------- independent re-derivation ---

def independent_compress(x_bf16, n, e_target=1.0, eps=1e-12):
    """The compress steps with library routines (scipy H, torch E4M3)."""
    x = W.bf16_bits_to_f32(x_bf16).astype(np.float64).reshape(-1, n)
    H = scipy.linalg.hadamard(n).astype(np.float64)
    m = np.mean(x * x, axis=1)
    alpha = np.sqrt(e_target / (m + np.float64(np.float32(eps)))).astype(np.float32)
    y = (alpha.astype(np.float64)[:, None] * x) @ H.T / math.sqrt(n)
    M = np.abs(y).max(axis=1)
    with np.errstate(divide="ignore"):
        s = np.where(M == 0, 1.0, 448.0 / np.where(M == 0, 1.0, M)).astype(np.float32)
    v = (y * s.astype(np.float64)[:, None]).astype(np.float32)
    return torch_e4m3_encode(v).reshape(-1, n), alpha, s, y


@pytest.mark.parametrize("n", [32, 64, 128, 256, 512])
def test_compress_matches_library_rederivation(n):
    x = W.tp_activation(3, 16, 2048, channel_scale=True, zero_blocks=(0, 5), block=n)
    codes, alpha, scale = oracle.compress(x, n)
    c2, a2, s2, _ = independent_compress(x, n)
    assert np.array_equal(alpha.reshape(-1), a2)
    assert np.max(np.abs(scale.reshape(-1).astype(np.float64) / s2 - 1)) <= 2 ** -23
    same = codes.reshape(-1, n) == c2
    assert same.mean() >= 0.9999 and ulp_distance(codes.reshape(-1), c2.reshape(-1)).max() <= 1


@pytest.mark.parametrize("n", [64, 128, 256])
def test_decompress_matches_library_rederivation(n):
    x = W.tp_activation(4, 8, 1024, block=n)
    codes, alpha, scale = oracle.compress(x, n)
    H = scipy.linalg.hadamard(n).astype(np.float64)
    q = torch_e4m3_decode_table()[codes.reshape(-1, n)] / scale.reshape(-1, 1).astype(np.float64)
    ref = (q @ H.T) / math.sqrt(n) / alpha.reshape(-1, 1).astype(np.float64)
    got = oracle.decompress(codes, alpha, scale, n).reshape(-1, n)
    scale_blk = np.abs(ref).max(axis=1, keepdims=True)
    assert np.all(np.abs(got - ref) <= 1e-12 * scale_blk)


# ------------------------------------------------------------ invariants ---

@pytest.mark.parametrize("e_target", [1.0, 4.0, 0.25])
def test_ash_normalises_block_energy_to_target(e_target):
    n = 128
    x = W.tp_activation(5, 32, 1024, channel_scale=True, block=n)
    _, alpha, _ = oracle.compress(x, n, e_target=e_target)
    xf = W.bf16_bits_to_f32(x).astype(np.float64).reshape(-1, n)
    m = np.mean(xf * xf, axis=1)
    energy = np.mean((alpha.reshape(-1, 1).astype(np.float64) * xf) ** 2, axis=1)
    expect = e_target * m / (m + np.float64(np.float32(1e-12)))
    assert np.allclose(energy, expect, rtol=2e-7)


def test_ds_keeps_codes_inside_qmax_and_hits_it_in_every_nonzero_block():
    n = 128
    x = W.shard_input("tiny_64x1024_n128", 0)
    codes, alpha, scale = oracle.compress(x, n)
    c = codes.reshape(-1, n)
    assert not np.any((c & 0x7F) == 0x7F)
    mag = c & 0x7F
    assert mag.max() <= 0x7E
    nonzero = np.any(W.bf16_bits_to_f32(x).reshape(-1, n) != 0, axis=1)
    assert np.all(mag.max(axis=1)[nonzero] == 0x7E)
    assert np.all(mag[~nonzero] == 0) and np.all(scale.reshape(-1)[~nonzero] == 1.0)


def test_zero_block_edge_case():
    n = 128
    x = np.zeros((2, 256), dtype=np.uint16)
    codes, alpha, scale = oracle.compress(x, n, e_target=1.0, eps=1e-12)
    assert np.all(codes == 0) and np.all(scale == 1.0)
    assert np.all(alpha == np.float32(math.sqrt(1.0 / np.float64(np.float32(1e-12)))))
    assert np.all(oracle.decompress(codes, alpha, scale, n) == 0.0)


# --------------------------------------------------- closed-form trips ---

@pytest.mark.parametrize("n", [128, 256])
def test_one_hot_block_codes_are_all_qmax_and_round_trip(n):
    H = scipy.linalg.hadamard(n)
    for j, v in [(0, 1.0), (7, -3.5), (n - 1, 0.015625)]:
        xv = np.zeros(n, dtype=np.float32)
        xv[j] = v
        x = bf16(xv).reshape(1, n)
        codes, alpha, scale = oracle.compress(x, n)
        sign = (v * H[:, j]) < 0
        assert np.array_equal(codes.reshape(-1), np.where(sign, 0xFE, 0x7E).astype(np.uint8))
        xhat = oracle.decompress(codes, alpha, scale, n).reshape(-1)
        assert np.allclose(xhat, xv, rtol=0, atol=1e-6 * abs(v))


@pytest.mark.parametrize("n", [128, 256])
def test_hadamard_row_block_compresses_to_one_code(n):
    H = scipy.linalg.hadamard(n)
    for r, v in [(3, 0.5), (n // 2 + 1, -2.0)]:
        xv = (v * H[r]).astype(np.float32)
        codes, alpha, scale = oracle.compress(bf16(xv).reshape(1, n), n)
        expect = np.zeros(n, dtype=np.uint8)
        expect[r] = 0x7E if v > 0 else 0xFE
        assert np.array_equal(codes.reshape(-1), expect)
        xhat = oracle.decompress(codes, alpha, scale, n).reshape(-1)
        assert np.allclose(xhat, xv, rtol=1e-6, atol=0)


def test_exact_round_trip_for_inputs_already_representable():
    n = 128
    H = scipy.linalg.hadamard(n)
    table = torch_e4m3_decode_table()
    # second magnitudes t for which 448 +- t is exact in bf16 (8 significant bits)
    mags = [t for t in table[1:127]
            if all(W.bf16_bits_to_f32(bf16([448.0 + sg * t]))[0] == 448.0 + sg * t for sg in (1, -1))]
    assert len(mags) >= 10
    rng = np.random.default_rng(11)
    for trial in range(20):
        v = np.zeros(n)
        pos = rng.choice(n, 2, replace=False)
        v[pos[0]] = 448.0 * rng.choice([-1, 1])
        v[pos[1]] = mags[rng.integers(0, len(mags))] * rng.choice([-1, 1])
        xv = (H @ v).astype(np.float32)
        x = bf16(xv)
        assert np.array_equal(W.bf16_bits_to_f32(x), xv)  # H v is exact in bf16 here
        codes, alpha, scale = oracle.compress(x.reshape(1, n), n)
        assert np.array_equal(table[codes.reshape(-1)], v)
        xhat = oracle.decompress(codes, alpha, scale, n).reshape(-1)
        assert np.allclose(xhat, xv, rtol=1e-6, atol=0)


@pytest.mark.parametrize("n", [128, 256])
def test_reconstruction_within_e4m3_rounding_bound(n):
    x = W.tp_activation(9, 32, 2048, channel_scale=True, block=n)
    codes, alpha, scale = oracle.compress(x, n)
    _, _, _, y = independent_compress(x, n)
    s = scale.reshape(-1, 1).astype(np.float64)
    q = torch_e4m3_decode_table()[codes.reshape(-1, n)]
    ys = y * s
    # E4M3 round-to-nearest: half a spacing, 2^-4 relative for normals,
    # 2^-10 absolute in the subnormal range (plus fp32 rounding of y*s)
    bound = np.maximum(np.abs(ys) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(q - ys) <= bound)
    xf = W.bf16_bits_to_f32(x).astype(np.float64).reshape(-1, n)
    xhat = oracle.decompress(codes, alpha, scale, n).reshape(-1, n)
    a = alpha.reshape(-1, 1).astype(np.float64)
    err = np.sqrt(np.sum((xhat - xf) ** 2, axis=1))
    lim = np.sqrt(np.sum(bound ** 2, axis=1)) / (a[:, 0] * s[:, 0])
    assert np.all(err <= lim * (1 + 1e-9) + 1e-300)


def test_int8_zero_collapse_and_fp8_codec_keeps_small_values():
    """TACO sections 2.A and 3: uniform INT8 maps the dense near-zero values to
    the same integer (zero), the ASH+DS FP8 codec does not.  (The global
    relative L2 error is reported, not asserted: it is dominated by the
    outliers, where uniform INT8 is accurate.)"""
    n = 128
    x = W.shard_input("tiny_64x1024_n128", 0)
    xf = W.bf16_bits_to_f32(x).astype(np.float64)
    codes, alpha, scale = oracle.compress(x, n)
    taco = oracle.decompress(codes, alpha, scale, n)
    int8 = oracle.int8_roundtrip(x, n)
    small = (xf != 0) & (np.abs(xf) < 1e-2)
    assert np.mean(int8[small] == 0) > 0.3
    assert np.mean(taco[small] == 0) < 0.05


def test_int8_baseline_closed_forms():
    n = 128
    xv = np.zeros(n, dtype=np.float32)
    xv[:4] = [127.0, -64.0, 1.0, 0.0]
    out = oracle.int8_roundtrip(bf16(xv).reshape(1, n), n).reshape(-1)
    assert np.array_equal(out, xv.astype(np.float64))
    x = W.tp_activation(2, 4, 512, block=n)
    out = oracle.int8_roundtrip(x, n).reshape(-1, n)
    xf = W.bf16_bits_to_f32(x).astype(np.float64).reshape(-1, n)
    amax = np.abs(xf).max(axis=1, keepdims=True)
    assert np.all(np.abs(out - xf) <= amax / 254 * (1 + 1e-12))


# ---------------------------------------------------------------- reduce ---

def _shards(P, rows=16, d=1024, n=128):
    xs = [W.tp_activation(20 + p, rows, d, channel_scale=True, block=n) for p in range(P)]
    return [oracle.compress(x, n) for x in xs]


def test_reduce_of_one_shard_is_decompress_then_compress():
    n = 128
    (c, a, s), = _shards(1)
    rc, ra, rs = oracle.reduce_shards([c], [a], [s], n)
    dc, da, ds = oracle.compress_f64(oracle.decompress(c, a, s, n), n)
    assert np.array_equal(rc, dc) and np.array_equal(ra, da) and np.array_equal(rs, ds)


def test_reduce_is_invariant_to_shard_order():
    n = 128
    sh = _shards(4)
    r1 = oracle.reduce_shards(*zip(*sh), n)
    r2 = oracle.reduce_shards(*zip(*sh[::-1]), n)
    assert (r1[0] == r2[0]).mean() >= 0.9999
    assert ulp_distance(r1[0].reshape(-1), r2[0].reshape(-1)).max() <= 1
    assert np.allclose(r1[1], r2[1], rtol=1e-6) and np.allclose(r1[2], r2[2], rtol=1e-6)


def test_reduce_of_shard_and_its_negation_is_the_zero_block():
    n = 128
    (c, a, s), = _shards(1)
    rc, ra, rs = oracle.reduce_shards([c, c ^ 0x80], [a, a], [s, s], n)
    assert np.all(rc == 0) and np.all(rs == 1.0)
    assert np.all(ra == np.float32(math.sqrt(1.0 / np.float64(np.float32(1e-12)))))


def test_reduce_of_two_one_hot_shards_doubles_the_block():
    n = 128
    xv = np.zeros(n, dtype=np.float32)
    xv[5] = 0.75
    c, a, s = oracle.compress(bf16(xv).reshape(1, n), n)
    rc, ra, rs = oracle.reduce_shards([c, c], [a, a], [s, s], n)
    assert np.allclose(oracle.decompress(rc, ra, rs, n).reshape(-1), 2 * xv, rtol=0, atol=1e-6)


def test_reduce_matches_library_rederivation():
    n = 128
    sh = _shards(3)
    H = scipy.linalg.hadamard(n).astype(np.float64)
    table = torch_e4m3_decode_table()
    S = 0
    for c, a, s in sh:
        q = table[c.reshape(-1, n)] / s.reshape(-1, 1).astype(np.float64)
        S = S + (q @ H.T) / math.sqrt(n) / a.reshape(-1, 1).astype(np.float64)
    m = np.mean(S * S, axis=1)
    alpha = np.sqrt(1.0 / (m + np.float64(np.float32(1e-12)))).astype(np.float32)
    y = (alpha.astype(np.float64)[:, None] * S) @ H.T / math.sqrt(n)
    scale = (448.0 / np.abs(y).max(axis=1)).astype(np.float32)
    codes = torch_e4m3_encode((y * scale.astype(np.float64)[:, None]).astype(np.float32))
    rc, ra, rs = oracle.reduce_shards(*zip(*sh), n)
    assert np.max(np.abs(ra.reshape(-1).astype(np.float64) / alpha - 1)) <= 2 ** -23
    assert np.max(np.abs(rs.reshape(-1).astype(np.float64) / scale - 1)) <= 2 ** -23
    assert (rc.reshape(-1) == codes.reshape(-1)).mean() >= 0.9999


# ------------------------------------------------------------------ AGoQ ---
# The AGoQ page fixes FP32 for the dequantised values and the local sum; the
# stored per-block scale is the dequantisation multiplier m = max|g| / 448 and
# codes are E4M3(g * q) with q = 448 / max|g|.  The re-derivations below use
# numpy float32 arithmetic and torch's float8 conversion.

def f32_requantise(g32: np.ndarray):
    amax = np.abs(g32).max(axis=1)
    with np.errstate(divide="ignore"):
        q = np.where(amax > 0, np.float32(448.0) / np.where(amax > 0, amax, 1), 1).astype(np.float32)
        m = np.where(amax > 0, amax / np.float32(448.0), 1).astype(np.float32)
    codes = torch_e4m3_encode((g32 * q[:, None]).astype(np.float32))
    return codes.reshape(-1), m


def test_agoq_first_step_from_zero_is_absmax_quantisation():
    n = 1 << 14
    g = W.agoq_grad(100, n)
    c, s = oracle.agoq_accumulate(np.zeros(n, np.uint8), np.ones(n // 128, np.float32), g)
    gf = W.bf16_bits_to_f32(g).reshape(-1, 128)
    c_ref, m_ref = f32_requantise(gf)
    assert np.array_equal(s, m_ref)
    assert np.array_equal(c, c_ref)


def test_agoq_accumulate_matches_float32_rederivation():
    n = 1 << 14
    table = torch_e4m3_decode_table().astype(np.float32)
    c = np.zeros(n, np.uint8)
    s = np.ones(n // 128, np.float32)
    for k in range(4):
        g = W.bf16_bits_to_f32(W.agoq_grad(100 + k, n)).reshape(-1, 128)
        deq = (table[c].reshape(-1, 128) * s[:, None]).astype(np.float32)
        c_ref, m_ref = f32_requantise((deq + g).astype(np.float32))
        c, s = oracle.agoq_accumulate(c, s, W.agoq_grad(100 + k, n))
        assert np.array_equal(s, m_ref) and np.array_equal(c, c_ref)


def test_agoq_accumulate_tracks_the_exact_sum_within_rounding():
    n = 1 << 14
    c = np.zeros(n, np.uint8)
    s = np.ones(n // 128, np.float32)
    exact = np.zeros(n)
    for k in range(4):
        g = W.agoq_grad(100 + k, n)
        exact += W.bf16_bits_to_f32(g)
        c, s = oracle.agoq_accumulate(c, s, g)
        got = oracle.agoq_dequantise(c, s)
        amax = np.abs(exact.reshape(-1, 128)).max(axis=1, keepdims=True)
        # each requantisation adds at most half an E4M3 spacing per element
        # (2^-4 relative, or 2^-10 / q in the subnormal range)
        lim = (k + 1) * np.maximum(np.abs(exact.reshape(-1, 128)) * 2 ** -4 * 1.1,
                                   2 ** -10 * amax / 448 * 1.1) + (k + 1) * amax * 2 ** -4
        assert np.all(np.abs(got.reshape(-1, 128) - exact.reshape(-1, 128)) <= lim)


def test_agoq_reduce_of_two_identical_shards_doubles_the_scale():
    n = 1 << 12
    g = W.agoq_grad(7, n)
    c, s = oracle.agoq_accumulate(np.zeros(n, np.uint8), np.ones(n // 128, np.float32), g)
    rc, rs = oracle.agoq_reduce([c, c], [s, s])
    # equal codes; a -0 code may come back as +0 (the sum of zeros starts at +0)
    zero = (c & 0x7F) == 0
    assert np.array_equal(rc[~zero], c[~zero]) and np.all(rc[zero] & 0x7F == 0)
    assert np.array_equal(rs, s * np.float32(2))


def test_agoq_reduce_is_an_fp32_sum_of_dequantised_shards():
    n = 1 << 12
    shards = []
    for p in range(3):
        shards.append(oracle.agoq_accumulate(np.zeros(n, np.uint8), np.ones(n // 128, np.float32),
                                             W.agoq_grad(50 + p, n)))
    table = torch_e4m3_decode_table().astype(np.float32)
    S = None
    for c, s in shards:
        x = (table[c].reshape(-1, 128) * s[:, None]).astype(np.float32)
        S = x if S is None else (S + x).astype(np.float32)
    c_ref, m_ref = f32_requantise(S)
    rc, rs = oracle.agoq_reduce(*zip(*shards))
    assert np.array_equal(rs, m_ref) and np.array_equal(rc, c_ref)
    # and the FP32 sum is within rounding of the exact sum
    parts = [oracle.agoq_dequantise(c, s) for c, s in shards]
    exact = sum(parts)
    # P - 1 rounded adds plus one rounded product per shard
    bound = len(parts) * 2.0 ** -24 * sum(np.abs(p) for p in parts) * (1 + 1e-9)
    assert np.all(np.abs(S.reshape(-1) - exact) <= bound)


def test_agoq_reduce_of_shard_and_negation_is_zero():
    n = 1 << 12
    c, s = oracle.agoq_accumulate(np.zeros(n, np.uint8), np.ones(n // 128, np.float32),
                                  W.agoq_grad(8, n))
    rc, rs = oracle.agoq_reduce([c, c ^ 0x80], [s, s])
    assert np.all(rc & 0x7F == 0) and np.all(rs == 1.0)


# ------------------------------------------------------ INT8 ASH + DS ---
# TACO section 5: the same pipeline with INT8 codes (Q_max = 127).

def test_int8_codec_matches_library_rederivation():
    n = 128
    x = W.tp_activation(12, 16, 1024, channel_scale=True, zero_blocks=(3,), block=n)
    codes, alpha, scale = oracle.compress_int8(x, n)
    xf = W.bf16_bits_to_f32(x).astype(np.float64).reshape(-1, n)
    H = scipy.linalg.hadamard(n).astype(np.float64)
    m = np.mean(xf * xf, axis=1)
    a = np.sqrt(1.0 / (m + np.float64(np.float32(1e-12)))).astype(np.float32)
    y = (a.astype(np.float64)[:, None] * xf) @ H.T / math.sqrt(n)
    M = np.abs(y).max(axis=1)
    s = np.where(M > 0, 127.0 / np.where(M > 0, M, 1), 1.0).astype(np.float32)
    ref = np.clip(np.rint((y * s.astype(np.float64)[:, None]).astype(np.float32)), -127, 127)
    assert np.array_equal(alpha.reshape(-1), a)
    assert np.max(np.abs(scale.reshape(-1).astype(np.float64) / s - 1)) <= 2 ** -23
    assert np.mean(codes.reshape(-1, n) == ref) >= 0.9999
    assert np.max(np.abs(codes.reshape(-1, n).astype(int) - ref)) <= 1


def test_int8_codec_closed_forms():
    n = 128
    H = scipy.linalg.hadamard(n)
    xv = np.zeros(n, dtype=np.float32)
    xv[9] = -0.5
    c, a, s = oracle.compress_int8(bf16(xv).reshape(1, n), n)
    assert np.array_equal(c.reshape(-1), np.where(-H[:, 9] < 0, -127, 127))
    assert np.allclose(oracle.decompress_int8(c, a, s, n).reshape(-1), xv, atol=1e-7)
    row = (2.0 * H[5]).astype(np.float32)
    c, a, s = oracle.compress_int8(bf16(row).reshape(1, n), n)
    expect = np.zeros(n, dtype=np.int8)
    expect[5] = 127
    assert np.array_equal(c.reshape(-1), expect)
    c, a, s = oracle.compress_int8(np.zeros((1, n), np.uint16), n)
    assert np.all(c == 0) and s[0, 0] == 1.0 and np.all(oracle.decompress_int8(c, a, s, n) == 0)


def test_int8_codec_error_within_half_a_step():
    n = 256
    x = W.tp_activation(13, 8, 1024, channel_scale=True, block=n)
    codes, alpha, scale = oracle.compress_int8(x, n)
    xf = W.bf16_bits_to_f32(x).astype(np.float64).reshape(-1, n)
    xhat = oracle.decompress_int8(codes, alpha, scale, n).reshape(-1, n)
    # |code - y s| <= 1/2 per element and the transform is orthonormal
    lim = 0.5 * math.sqrt(n) / (alpha.reshape(-1).astype(np.float64) * scale.reshape(-1))
    assert np.all(np.sqrt(np.sum((xhat - xf) ** 2, axis=1)) <= lim * (1 + 1e-6))
    assert np.abs(codes).max() == 127


def test_int8_ash_avoids_the_zero_collapse_of_plain_int8():
    """TACO sections 2.A and 5: plain per-block INT8 maps most of the dense
    near-zero values to 0; with the ASH rotation in front they survive."""
    n = 128
    x = W.shard_input("tiny_64x1024_n128", 0)
    xf = W.bf16_bits_to_f32(x).astype(np.float64)
    small = (xf != 0) & (np.abs(xf) < 1e-2)
    c, a, s = oracle.compress_int8(x, n)
    ash = oracle.decompress_int8(c, a, s, n)
    plain = oracle.int8_roundtrip(x, n)
    assert np.mean(plain[small] == 0) > 0.3
    assert np.mean(ash[small] == 0) < 0.05


# ------------------------------------------------------------------ LAAQ ---
# AGoQ section 2.A: block-wise 4-bit activation codes (5, 6, 8 bits under the
# pipeline-stage compensation), read as symmetric absmax integers packed into
# a little-endian bit stream, in FP32 arithmetic.

def test_laaq_hand_worked_examples():
    g = json.load(open(os.path.join(GOLDEN, "laaq_examples.json")))
    for ex in g["examples"]:
        x = bf16(ex["x"])
        packed, scale = oracle.laaq_quantize(x, ex["block"], ex["bits"])
        assert packed.tolist() == ex["packed"], ex["name"]
        assert scale[0] == np.float32(ex["scale"]), ex["name"]
        out = oracle.laaq_dequantize(packed, scale, x.size, ex["block"], ex["bits"])
        assert np.array_equal(out, (np.array(ex["codes"], np.float32) * scale[0]).astype(np.float32))


def laaq_rederive(x_bf16, block, bits):
    xf = W.bf16_bits_to_f32(x_bf16).reshape(-1, block)
    qmax = np.float32(2 ** (bits - 1) - 1)
    amax = np.abs(xf).max(axis=1)
    with np.errstate(divide="ignore"):
        q = np.where(amax > 0, qmax / np.where(amax > 0, amax, 1), 1).astype(np.float32)
        m = np.where(amax > 0, amax / qmax, 1).astype(np.float32)
    codes = np.clip(np.rint((xf * q[:, None]).astype(np.float32)), -qmax, qmax).astype(np.int64)
    u = (codes & ((1 << bits) - 1)).reshape(-1)
    bitarr = ((u[:, None] >> np.arange(bits)) & 1).astype(np.uint8).reshape(-1)
    return np.packbits(bitarr, bitorder="little"), m, codes


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
@pytest.mark.parametrize("block", [32, 128, 256])
def test_laaq_matches_library_rederivation(bits, block):
    x = W.tp_activation(30 + bits, 16, 1024, channel_scale=True, zero_blocks=(1,), block=block)
    packed, scale = oracle.laaq_quantize(x, block, bits)
    ref_packed, ref_m, codes = laaq_rederive(x, block, bits)
    assert np.array_equal(packed, ref_packed)
    assert np.array_equal(scale, ref_m)
    out = oracle.laaq_dequantize(packed, scale, x.size, block, bits)
    assert np.array_equal(out, (codes.astype(np.float32) * ref_m[:, None]).astype(np.float32).reshape(-1))


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_laaq_error_within_half_a_step_and_uses_the_full_range(bits):
    block = 64
    x = W.tp_activation(40 + bits, 8, 2048, block=block)
    packed, scale = oracle.laaq_quantize(x, block, bits)
    out = oracle.laaq_dequantize(packed, scale, x.size, block, bits).reshape(-1, block)
    xf = W.bf16_bits_to_f32(x).astype(np.float64).reshape(-1, block)
    step = scale.astype(np.float64)[:, None]
    amax = np.abs(xf).max(axis=1, keepdims=True)
    # half a step, plus the fp32 roundings of q, x*q, m and code*m (each at
    # most 2^-24 relative to values no larger than amax)
    assert np.all(np.abs(out - xf) <= 0.5 * step + 4 * 2.0 ** -24 * amax * 2)
    qmax = 2 ** (bits - 1) - 1
    nz = np.any(xf != 0, axis=1)
    assert np.all(np.abs(np.rint(out / step)).max(axis=1)[nz] == qmax)


# ------------------------------------------- GEMM feeding the compressor --

def test_gemm_bt_matches_exactly_rounded_dot_products():
    """AGoQ 2.C fuses the compressor into the GEMM that produces the tensor:
    the oracle's GEMM is numpy's float64 product of the exact bf16 values.
    Pinned against dot products summed with math.fsum (exactly rounded) on a
    small case, including a K that is not a power of two."""
    import math

    from fp8_communication_compression_gb300 import workloads as W

    a = W.tp_activation(11, 5, 37)
    b = W.f32_to_bf16_bits(np.random.default_rng(3).normal(0, 0.02, (7, 37)).astype(np.float32))
    y = oracle.gemm_bt(a, b)
    af, bf = oracle.bf16_to_f64(a), oracle.bf16_to_f64(b)
    for i in range(5):
        for j in range(7):
            terms = [af[i, k] * bf[j, k] for k in range(37)]
            exact = math.fsum(terms)
            assert abs(y[i, j] - exact) <= 1e-15 * math.fsum(abs(t) for t in terms)
    # a transposed operand would not even have the right shape; a swapped
    # pair of operands would give Y^T
    assert y.shape == (5, 7)


def test_gemm_compress_is_compress_of_the_product():
    """The fused path's oracle on a case where Y is known in closed form: with
    A = I (the first N columns of an identity, in bf16) Y = B exactly, so
    the codes equal those of compressing B itself."""
    from fp8_communication_compression_gb300 import workloads as W

    n = 128

    b = W.tp_activation(12, 256, n)          # [N = 256, K = 128]
    a = np.zeros((n, n), dtype=np.uint16)    # [M = 128, K = 128] identity in bf16 (1.0 = 0x3F80)
    a[np.arange(n), np.arange(n)] = 0x3F80
    c, al, sc = oracle.gemm_compress(a, b, n)
    # Y = A B^T = B^T [128, 256]: compress the transpose of B directly
    rc, ra, rs = oracle.compress_f64(oracle.bf16_to_f64(b).T.copy(), n)
    assert np.array_equal(c, rc) and np.array_equal(al, ra) and np.array_equal(sc, rs)


def test_agoq_accumulate_f32_equals_the_bf16_step_on_bf16_representable_gradients():
    """The fp32-gradient accumulation (the GEMM-fused form, AGoQ 2.C) runs the
    same FP32 sequence as the bf16 one: on gradients that are bf16 values it
    gives the same codes and scales, step after step."""
    from fp8_communication_compression_gb300 import workloads as W

    n = 128 * 40
    c, s = np.zeros(n, np.uint8), np.ones(n // 128, np.float32)
    cf, sf = c.copy(), s.copy()
    for step in range(3):
        g = W.agoq_grad(500 + step, n)
        c, s = oracle.agoq_accumulate(c, s, g, 128)
        cf, sf = oracle.agoq_accumulate_f32(cf, sf, oracle.bf16_to_f64(g).astype(np.float32), 128)
        assert np.array_equal(c, cf) and np.array_equal(s, sf)


def test_agoq_accumulate_f32_first_step_is_absmax_quantisation():
    """From the zero buffer (codes 0, multiplier 1) one step is plain
    per-block absmax FP8 quantisation of the gradient: the multiplier is
    max|g| / 448 and the codes are E4M3(g * 448 / max|g|)."""
    rng = np.random.default_rng(4)
    g = (rng.standard_normal(256) * 1e-3).astype(np.float32)
    g[:128] *= 1000.0
    c, s = oracle.agoq_accumulate_f32(np.zeros(256, np.uint8), np.ones(2, np.float32), g, 128)
    for b in range(2):
        blk = g[128 * b:128 * (b + 1)]
        amax = np.float32(np.abs(blk).max())
        assert s[b] == np.float32(amax / np.float32(448.0))
        q = np.float32(448.0) / amax
        want = oracle.e4m3_encode_array((blk * q).astype(np.float32))
        assert np.array_equal(c[128 * b:128 * (b + 1)], want)


# ------------------------------- LAAQ quantisation fused into the GEMM --
# AGoQ 2.C: the activation quantisation runs in the epilogue of the GEMM that
# produces the activation, on its fp32 result.

@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_laaq_quantize_f32_equals_the_bf16_quantize_on_bf16_values(bits):
    """The fp32-input quantisation runs the same FP32 sequence as the bf16
    one: on values that are bf16 values it gives the same stream and
    multipliers."""
    for block in (32, 128, 256):
        x = W.tp_activation(60 + bits, 8, 1024, channel_scale=True, zero_blocks=(3,), block=block)
        p16, s16 = oracle.laaq_quantize(x, block, bits)
        p32, s32 = oracle.laaq_quantize_f32(W.bf16_bits_to_f32(x), block, bits)
        assert np.array_equal(p16, p32) and np.array_equal(s16, s32)


def test_laaq_quantize_f32_hand_worked_ties_and_non_bf16_values():
    """One 32-element block at 4 bits with max|x| = 7, so q = 7 / 7 = 1 and
    the multiplier is 1: the codes are the values rounded to the nearest
    integer, ties to even.  2.4999998 and 2.5000002 (the fp32 neighbours of
    2.5, no bf16 value) go to 2 and 3; -3.5 and 4.5 to -4 and 4; -0.5 to 0;
    1.5 to 2.  Element i takes bits 4i .. 4i + 3 (two's complement), so byte
    j holds element 2j in its low nibble and 2j + 1 in its high one."""
    f = lambda bits: np.array([bits], np.uint32).view(np.float32)[0]
    x = np.zeros(32, np.float32)
    x[:9] = [7.0, -7.0, f(0x401FFFFF), f(0x40200001), -3.5, 4.5, 0.5, -0.5, 1.5]
    assert x[2] == np.float32(2.4999998) and x[3] == np.float32(2.5000002)
    packed, scale = oracle.laaq_quantize_f32(x, 32, 4)
    # codes 7, -7, 2, 3, -4, 4, 0, 0, 2, 0 ... -> nibbles 7, 9, 2, 3, C, 4, 0, 0, 2, 0 ...
    assert packed.tolist() == [0x97, 0x32, 0x4C, 0x00, 0x02] + [0] * 11
    assert scale.tolist() == [1.0]


def test_gemm_laaq_quantize_is_quantize_of_the_product():
    """The fused path's oracle on a case where Y is known in closed form: with
    A = I in bf16, Y = B^T exactly, so the stream and multipliers equal
    those of quantising B^T's bf16 values."""
    n = 128
    b = W.tp_activation(13, 256, n)           # [N = 256, K = 128]
    a = np.zeros((n, n), dtype=np.uint16)     # [M = 128, K = 128] identity (1.0 = 0x3F80)
    a[np.arange(n), np.arange(n)] = 0x3F80
    for bits in (4, 5, 6, 8):
        p, s = oracle.gemm_laaq_quantize(a, b, 128, bits)
        rp, rs = oracle.laaq_quantize(np.ascontiguousarray(b.T), 128, bits)
        assert np.array_equal(p, rp) and np.array_equal(s, rs)


# ------------------------- RMSNorm / SiLU recomputed from the stored input --
# AGoQ 2.A: for RMSNorm and SiLU, only the quantised input is stored and the
# operator's output is recomputed from it in the backward pass.

def _stored(seed, rows, d, bits, block=128):
    x = W.tp_activation(seed, rows, d, channel_scale=True, zero_blocks=(2,), block=block)
    packed, scale = oracle.laaq_quantize(x, block, bits)
    xhat = oracle.laaq_dequantize(packed, scale, rows * d, block, bits).astype(np.float64)
    return x, packed, scale, xhat


@pytest.mark.parametrize("bits", [4, 8])
def test_silu_recompute_odd_part_is_the_input(bits):
    """SiLU(x) - SiLU(-x) = x (x sigma(x) + x sigma(-x) = x): the recompute of
    the negated stream (codes -c with the same multipliers, what quantising
    -x gives) subtracted from the recompute of the stream is the dequantised
    input itself, to rounding."""
    rows, d = 16, 1024
    x, packed, scale, xhat = _stored(91, rows, d, bits)
    neg_packed, neg_scale = oracle.laaq_quantize(x ^ np.uint16(0x8000), 128, bits)
    assert np.array_equal(neg_scale, scale)
    s_pos = oracle.laaq_dequantize_silu(packed, scale, rows * d, 128, bits)
    s_neg = oracle.laaq_dequantize_silu(neg_packed, neg_scale, rows * d, 128, bits)
    assert np.allclose(s_pos - s_neg, xhat, rtol=1e-14, atol=1e-300)


def test_silu_recompute_equals_the_tanh_form():
    """x sigma(x) = (x / 2) (1 + tanh(x / 2)), evaluated with numpy's tanh on
    the dequantised input; zeros stay zeros."""
    rows, d = 8, 512
    _, packed, scale, xhat = _stored(92, rows, d, 5)
    s = oracle.laaq_dequantize_silu(packed, scale, rows * d, 128, 5)
    want = 0.5 * xhat * (1.0 + np.tanh(0.5 * xhat))
    assert np.allclose(s, want, rtol=1e-13, atol=0)
    assert np.all(s[xhat == 0] == 0)


@pytest.mark.parametrize("bits", [4, 6])
def test_rmsnorm_recompute_invariants(bits):
    """Per row: y_i / (xhat_i g_i) is one constant r > 0, and mean(y^2 / g^2)
    = r^2 mean(xhat^2) = mean(xhat^2) / (mean(xhat^2) + eps), so with the
    row's mean square m: r = 1 / sqrt(m + eps).  A transposed index, a sum in
    place of the mean or a dropped eps breaks one of these."""
    rows, d, eps = 12, 1024, 1e-6
    _, packed, scale, xhat = _stored(93 + bits, rows, d, bits)
    xhat = xhat.reshape(rows, d)
    g = (1.0 + 0.5 * np.sin(np.arange(d))).astype(np.float32)
    y = oracle.laaq_dequantize_rmsnorm(packed, scale, rows, d, g, eps, 128, bits)
    gd = g.astype(np.float64)
    for r in range(rows):
        nz = xhat[r] != 0
        ratio = y[r][nz] / (xhat[r][nz] * gd[nz])
        assert np.allclose(ratio, ratio[0], rtol=1e-13) and ratio[0] > 0
        m = float(np.mean(xhat[r] ** 2))
        assert abs(ratio[0] - 1.0 / math.sqrt(m + eps)) <= 1e-12 * ratio[0]
        assert np.all(y[r][~nz] == 0)


def test_rmsnorm_recompute_hand_worked_row():
    """One row of 128 values, every code 7 at 4 bits with multiplier 0.5 (x =
    3.5 everywhere, stored as amax 3.5): mean(x^2) = 12.25, so with eps = 0
    y = 3.5 / 3.5 * g = g exactly."""
    x = np.full(128, 0x4060, dtype=np.uint16)  # bf16 3.5
    packed, scale = oracle.laaq_quantize(x, 128, 4)
    assert scale.tolist() == [0.5] and packed.tolist() == [0x77] * 64
    g = np.linspace(-2, 2, 128).astype(np.float32)
    y = oracle.laaq_dequantize_rmsnorm(packed, scale, 1, 128, g, 0.0, 128, 4)
    assert np.array_equal(y[0], g.astype(np.float64))
