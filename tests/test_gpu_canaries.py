"""Out-of-bounds write checks: every output of every entry point is placed
between two 4 KB guard regions filled with a byte pattern, on ragged sizes
(row counts that leave partial warp tiles, shard counts that are not powers
of two, element counts with a tail), and after the launch the guards must
be untouched and the inputs unchanged."""

import numpy as np
import pytest
import torch

from fp8_communication_compression_gb300 import api
from fp8_communication_compression_gb300 import workloads as W

from parity import to_dev_bf16

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A device buffer of `nbytes` between two guard regions."""

    def __init__(self, nbytes: int, device="cuda", pin=False):
        kw = dict(dtype=torch.uint8)
        if device == "cpu":
            self.buf = torch.full((2 * GUARD + nbytes,), PATTERN, pin_memory=pin, **kw)
        else:
            self.buf = torch.full((2 * GUARD + nbytes,), PATTERN, device=device, **kw)
        self.nbytes = nbytes

    def view(self, dtype, shape):
        return self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        return bool(torch.all(self.buf[:GUARD] == PATTERN) and torch.all(self.buf[GUARD + self.nbytes:] == PATTERN))


def guarded(dtype, shape, device="cuda", pin=False):
    n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
    g = Guarded(n, device, pin)
    return g, g.view(dtype, shape)


def activation(seed, rows, d, block):
    return to_dev_bf16(W.tp_activation(seed, rows, d, channel_scale=True, zero_blocks=(1,), block=block))


@pytest.fixture(autouse=True)
def no_watchdog_flags():
    api.taco_device_error(clear=True)
    yield
    assert api.taco_device_error(clear=True) == 0


@pytest.mark.parametrize("block,rows,d", [(128, 37, 1024), (256, 38, 768), (128, 1, 128)])
def test_codec_writes_stay_inside_their_outputs(block, rows, d):
    x = activation(1, rows, d, block).reshape(rows, d)
    x0 = x.clone()
    nb = rows * d // block
    for int8 in (False, True):
        cdt = torch.int8 if int8 else torch.uint8
        gc, c = guarded(cdt, (rows, d))
        ga, a = guarded(torch.float32, (nb,))
        gs, s = guarded(torch.float32, (nb,))
        (api.taco_compress_int8 if int8 else api.taco_compress)(x, block, codes=c, alpha=a, scale=s)
        assert gc.intact() and ga.intact() and gs.intact()
        c0, a0, s0 = c.clone(), a.clone(), s.clone()
        for dt in (torch.float32, torch.bfloat16):
            go, o = guarded(dt, (rows, d))
            (api.taco_decompress_int8 if int8 else api.taco_decompress)(c, a, s, block, out=o)
            assert go.intact()
        assert torch.equal(c, c0) and torch.equal(a, a0) and torch.equal(s, s0)
    assert torch.equal(x, x0)


@pytest.mark.parametrize("P,block,rows,d", [(3, 128, 37, 1024), (5, 256, 38, 512), (16, 128, 33, 256)])
def test_reduce_writes_stay_inside_their_outputs(P, block, rows, d):
    nb = rows * d // block
    shards = [api.taco_compress(activation(10 + p, rows, d, block).reshape(rows, d), block) for p in range(P)]
    codes = [s[0] for s in shards]
    alpha = [s[1] for s in shards]
    scale = [s[2] for s in shards]
    before = [t.clone() for t in codes + alpha + scale]
    gc, oc = guarded(torch.uint8, (rows, d))
    ga, oa = guarded(torch.float32, (nb,))
    gs, os_ = guarded(torch.float32, (nb,))
    api.taco_reduce_shards(codes, alpha, scale, block, out_codes=oc, out_alpha=oa, out_scale=os_)
    assert gc.intact() and ga.intact() and gs.intact()
    for dt in (torch.float32, torch.bfloat16):
        gc, oc = guarded(torch.uint8, (rows, d))
        ga, oa = guarded(torch.float32, (nb,))
        gs, os_ = guarded(torch.float32, (nb,))
        go, o = guarded(dt, (rows, d))
        api.taco_reduce_decompress(codes, alpha, scale, block, out_codes=oc, out_alpha=oa, out_scale=os_, out=o)
        assert gc.intact() and ga.intact() and gs.intact() and go.intact()
    assert all(torch.equal(t, b) for t, b in zip(codes + alpha + scale, before))


@pytest.mark.parametrize("P,n,block", [(3, 37 * 1024, 128), (8, 96 * 256, 256)])
def test_agoq_writes_stay_inside_their_buffers(P, n, block):
    g = to_dev_bf16(W.agoq_grad(31, n))
    g0 = g.clone()
    gc, c = guarded(torch.uint8, (n,))
    gs, s = guarded(torch.float32, (n // block,))
    c.zero_()
    s.fill_(1.0)
    api.agoq_fp8_accumulate(c, s, g, block)
    assert gc.intact() and gs.intact() and torch.equal(g, g0)
    codes = [c.clone() for _ in range(P)]
    scales = [s.clone() for _ in range(P)]
    goc, oc = guarded(torch.uint8, (n,))
    gos, os_ = guarded(torch.float32, (n // block,))
    api.agoq_reduce_shards(codes, scales, block, out_codes=oc, out_scale=os_)
    assert goc.intact() and gos.intact()
    assert all(torch.equal(t, c) for t in codes) and all(torch.equal(t, s) for t in scales)


@pytest.mark.parametrize("bits,block", [(4, 128), (5, 32), (6, 64), (8, 256)])
def test_laaq_writes_stay_inside_their_outputs(bits, block):
    n = 37 * 1024 + 3 * 256
    x = activation(40, n // 256, 256, block).reshape(-1)
    x0 = x.clone()
    gp, packed = guarded(torch.uint8, (n * bits // 8,))
    gs, scale = guarded(torch.float32, (n // block,))
    api.agoq_laaq_quantize(x, block, bits, packed, scale)
    assert gp.intact() and gs.intact() and torch.equal(x, x0)
    for dt in (torch.float32, torch.bfloat16):
        go, o = guarded(dt, (n,))
        api.agoq_laaq_dequantize(packed, scale, n, block, bits, out=o)
        assert go.intact()


@pytest.mark.parametrize("n", [1, 7, 8, 1003, 65536 + 5])
def test_e4m3_encode_writes_stay_inside_its_output(n):
    x = torch.randn(n, device="cuda") * 100
    x0 = x.clone()
    gc, c = guarded(torch.uint8, (n,))
    api.taco_e4m3_encode(x, out=c)
    assert gc.intact() and torch.equal(x, x0)


def test_host_pipeline_writes_stay_inside_the_host_output():
    P, rows, d, block = 3, 101, 1024, 128
    bits = np.stack([W.tp_activation(60 + p, rows, d, channel_scale=True, block=block) for p in range(P)])
    h_in = torch.empty((P, rows, d), dtype=torch.bfloat16, pin_memory=True)
    h_in.view(torch.int16).copy_(torch.from_numpy(bits.view(np.int16)))
    h0 = h_in.clone()
    gh, h_out = guarded(torch.float32, (rows, d), device="cpu", pin=True)
    pipe = api.HostPipeline(P, rows, d, block, chunks=6)
    for _ in range(2):
        pipe.run(h_in, h_out)
    assert gh.intact() and torch.equal(h_in.view(torch.int16), h0.view(torch.int16))


def gemm_operands(M, N, K, seed):
    a = to_dev_bf16(W.tp_activation(seed, M, K, channel_scale=True))
    b = to_dev_bf16(W.f32_to_bf16_bits(np.random.default_rng(seed + 1).normal(0.0, 0.02, (N, K))
                                       .astype(np.float32)))
    return a, b


def guarded_workspace(M, N, K):
    """The split tail's workspace between guards (zeroed inside), or None."""
    nb = api.gemm_workspace_bytes(M, N, K)
    if nb == 0:
        return None, None
    g, ws = guarded(torch.uint8, (nb,))
    ws.zero_()
    return g, ws


# (384, 768, 4096): 9 tiles split into 2 pieces; (256, 384, 128): 128-wide
# tiles, no split; (2048, 4096, 512): several tiles per SM
@pytest.mark.parametrize("M,N,K", [(384, 768, 4096), (256, 384, 128), (2048, 4096, 512)])
def test_gemm_compress_writes_stay_inside_their_outputs(M, N, K):
    a, b = gemm_operands(M, N, K, 60)
    a0, b0 = a.clone(), b.clone()
    gc, c = guarded(torch.uint8, (M, N))
    ga, al = guarded(torch.float32, (M * N // 128,))
    gs, sc = guarded(torch.float32, (M * N // 128,))
    gy, y = guarded(torch.float32, (M, N))
    gw, ws = guarded_workspace(M, N, K)
    api.taco_gemm_compress(a, b, codes=c, alpha=al, scale=sc, y_out=y, workspace=ws)
    assert gc.intact() and ga.intact() and gs.intact() and gy.intact() and (gw is None or gw.intact())
    assert torch.equal(a, a0) and torch.equal(b, b0)


@pytest.mark.parametrize("M,N,K", [(384, 640, 4096), (2048, 4096, 512)])
def test_agoq_gemm_accumulate_writes_stay_inside_their_buffers(M, N, K):
    a, b = gemm_operands(M, N, K, 70)
    a0, b0 = a.clone(), b.clone()
    gc, c = guarded(torch.uint8, (M, N))
    gs, sc = guarded(torch.float32, (M * N // 128,))
    c.zero_()
    sc.fill_(1.0)
    gw, ws = guarded_workspace(M, N, K)
    api.agoq_gemm_accumulate(a, b, c, sc, workspace=ws)
    assert gc.intact() and gs.intact() and (gw is None or gw.intact())
    assert torch.equal(a, a0) and torch.equal(b, b0)


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
@pytest.mark.parametrize("M,N,K", [(384, 768, 4096), (256, 384, 128)])
def test_gemm_laaq_quantize_writes_stay_inside_their_outputs(M, N, K, bits):
    a, b = gemm_operands(M, N, K, 80 + bits)
    a0, b0 = a.clone(), b.clone()
    gp, p = guarded(torch.uint8, (M * N * bits // 8,))
    gs, sc = guarded(torch.float32, (M * N // 128,))
    gw, ws = guarded_workspace(M, N, K)
    api.agoq_gemm_laaq_quantize(a, b, bits, packed=p, scale=sc, workspace=ws)
    assert gp.intact() and gs.intact() and (gw is None or gw.intact())
    assert torch.equal(a, a0) and torch.equal(b, b0)


@pytest.mark.parametrize("bits,block,rows,d", [(4, 128, 37, 512), (5, 32, 9, 96), (6, 256, 5, 768), (8, 128, 7, 2048)])
def test_laaq_recompute_writes_stay_inside_their_outputs(bits, block, rows, d):
    n = rows * d
    x = activation(41, rows, d, block).reshape(-1)
    packed, scale = api.agoq_laaq_quantize(x, block, bits)
    p0, s0 = packed.clone(), scale.clone()
    g = torch.linspace(0.5, 1.5, d, device="cuda")
    for dt in (torch.float32, torch.bfloat16):
        go, o = guarded(dt, (n,))
        api.agoq_laaq_dequantize_silu(packed, scale, n, block, bits, out=o)
        assert go.intact()
        go, o = guarded(dt, (rows, d))
        api.agoq_laaq_dequantize_rmsnorm(packed, scale, rows, d, g, 1e-6, block, bits, out=o)
        assert go.intact()
    assert torch.equal(packed, p0) and torch.equal(scale, s0)
