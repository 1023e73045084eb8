"""The multi-process oracle used by the full-size parity tests gives the
single-process oracle's results bit for bit (every block is independent, so
splitting the rows over worker processes changes nothing)."""

import numpy as np

import oracle
import oracle_pool
from fp8_communication_compression_gb300 import workloads as W


import pytest


@pytest.mark.parametrize("piece_bytes", [None, 50_000])
def test_pool_matches_the_oracle_called_directly(piece_bytes, monkeypatch):
    if piece_bytes:  # many sequential pieces, each split over the workers
        monkeypatch.setattr(oracle_pool, "PIECE_BYTES", piece_bytes)
    P, rows, d, block = 3, 37, 512, 256
    bits = np.stack([W.tp_activation(90 + p, rows, d, channel_scale=True, spikes=True, block=block)
                     for p in range(P)])
    c, a, s = oracle_pool.compress(bits, block)
    for p in range(P):
        rc, ra, rs = oracle.compress(bits[p], block)
        assert np.array_equal(c[p], rc) and np.array_equal(a[p], ra) and np.array_equal(s[p], rs)
    pc, pa, ps = oracle_pool.reduce_shards(c, a.reshape(P, -1), s.reshape(P, -1), block)
    rc, ra, rs = oracle.reduce_shards(list(c), list(a), list(s), block)
    assert np.array_equal(pc, rc) and np.array_equal(pa, ra) and np.array_equal(ps, rs)
    out = oracle_pool.decompress(pc, pa, ps, block)
    assert np.array_equal(out, oracle.decompress(rc, ra, rs, block))
    fc, fa, fs = oracle_pool.compress_f64(out, block)
    gc, ga, gs = oracle.compress_f64(out, block)
    assert np.array_equal(fc, gc) and np.array_equal(fa, ga) and np.array_equal(fs, gs)


@pytest.mark.parametrize("piece_bytes", [None, 5_000])
def test_pool_matches_the_agoq_oracle_called_directly(piece_bytes, monkeypatch):
    if piece_bytes:
        monkeypatch.setattr(oracle_pool, "PIECE_BYTES", piece_bytes)
    n, block, P = 128 * 45, 128, 3
    c, s = np.zeros(n, np.uint8), np.ones(n // block, np.float32)
    for step in range(2):
        g = W.agoq_grad(300 + step, n)
        pc, ps = oracle_pool.agoq_accumulate(c, s, g, block)
        c, s = oracle.agoq_accumulate(c, s, g, block)
        assert np.array_equal(pc, c) and np.array_equal(ps, s)
    cs = np.stack([oracle.agoq_accumulate(np.zeros(n, np.uint8), np.ones(n // block, np.float32),
                                          W.agoq_grad(310 + p, n), block)[0] for p in range(P)])
    ss = np.stack([oracle.agoq_accumulate(np.zeros(n, np.uint8), np.ones(n // block, np.float32),
                                          W.agoq_grad(310 + p, n), block)[1] for p in range(P)])
    pc, ps = oracle_pool.agoq_reduce(cs, ss, block)
    rc, rs = oracle.agoq_reduce(list(cs), list(ss), block)
    assert np.array_equal(pc, rc) and np.array_equal(ps, rs)
