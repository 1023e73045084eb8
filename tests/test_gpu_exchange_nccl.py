"""The two-shot exchange on the GPU through NCCL, in a group of one rank.

One process, one GPU: the collectives copy the rank's own pieces and no
kernel waits on another rank.  This runs the exchange's CUDA path end to end
(the library's kernels on the pieces, NCCL collectives on device buffers,
the ordering of asynchronous collectives against the current stream) and
checks it against the one-GPU path: with one rank the sum is the rank's own
tensor compressed, reduced as one shard and decompressed, and since every
block is independent the result is bit-identical however the rows are cut
into pieces.  The exchange's bookkeeping across several ranks is tested on
CPU ranks (test_exchange_gloo.py).
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

from fp8_communication_compression_gb300 import api, exchange
from fp8_communication_compression_gb300 import workloads as W

from parity import to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nccl_group():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=torch.device("cuda", 0))
    yield
    dist.destroy_process_group()


@pytest.mark.parametrize("rows,d,block,stages", [(512, 1024, 128, 1), (512, 1024, 128, 4), (300, 512, 256, 3)])
def test_exchange_on_one_rank_equals_the_local_path(nccl_group, rows, d, block, stages):
    x = to_dev_bf16(W.tp_activation(77, rows, d, channel_scale=True, block=block))
    ar = exchange.TwoShotAllReduce(rows, d, block, stages=stages)
    out = ar.run(x).clone()
    ref = api.TwoShotLocal(1, rows, d, block).run(x.view(1, rows, d))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
    # a second call on the same buffers gives the same bits
    assert torch.equal(ar.run(x).view(torch.int32), ref.view(torch.int32))


def test_agoq_exchange_on_one_rank_equals_the_local_reduce(nccl_group):
    n, block = 128 * 1000, 128
    ar = exchange.AgoqAllReduce(n, block)
    g = to_dev_bf16(W.agoq_grad(5, n))
    api.agoq_fp8_accumulate(ar.codes, ar.scale, g, block)
    c, s = ar.run()
    rc, rs = api.agoq_reduce_shards([ar.codes], [ar.scale], block)
    torch.cuda.synchronize()
    assert torch.equal(c, rc) and torch.equal(s, rs)


@pytest.mark.parametrize("rows,d,K,stages", [(512, 1024, 256, 1), (1024, 512, 512, 4)])
def test_gemm_exchange_on_one_rank_equals_the_local_path(nccl_group, rows, d, K, stages):
    """run_gemm: the row-parallel layer's partial sum Y = A W^T leaves the
    GEMM compressed, piece by piece, into the send buffer.  With one rank the
    result is the same pieces' taco_gemm_compress, reduced as one shard and
    decompressed, bit for bit (the same shapes take the same tile plan)."""
    a = to_dev_bf16(W.tp_activation(81, rows, K, channel_scale=True))
    w = to_dev_bf16(W.f32_to_bf16_bits(np.random.default_rng(82).normal(0.0, 0.02, (d, K)).astype(np.float32)))
    ar = exchange.TwoShotAllReduce(rows, d, 128, stages=stages)
    out = ar.run_gemm(a, w).clone()
    Rs, nbr = rows // stages, d // 128
    codes = torch.empty((rows, d), dtype=torch.uint8, device="cuda")
    alpha = torch.empty(rows * nbr, dtype=torch.float32, device="cuda")
    scale = torch.empty_like(alpha)
    for k in range(stages):
        r0, r1 = k * Rs, (k + 1) * Rs
        api.taco_gemm_compress(a[r0:r1], w, codes=codes[r0:r1], alpha=alpha[r0 * nbr:r1 * nbr],
                               scale=scale[r0 * nbr:r1 * nbr])
    rc, ra, rs = api.taco_reduce_shards([codes], [alpha], [scale], 128)
    ref = api.taco_decompress(rc, ra, rs, 128)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32))


def test_agoq_exchange_of_gradients_accumulated_by_the_gemm(nccl_group):
    """The AGoQ path end to end on one rank: two micro-batches' weight
    gradients accumulated by the GEMM with the FP8 accumulation in its
    epilogue, straight into the exchange's send buffer (AgoqAllReduce.codes
    and .scale viewed as the [M, N] gradient), then the All-to-All, FP32
    reduce and All-Gather.  With one rank the result is the reduce of that
    buffer, bit for bit."""
    M, N, K = 256, 512, 256
    ar = exchange.AgoqAllReduce(M * N, 128)
    for step in range(2):
        a = to_dev_bf16(W.agoq_grad(40 + step, M * K).reshape(M, K))
        b = to_dev_bf16(W.tp_activation(50 + step, N, K, channel_scale=True))
        api.agoq_gemm_accumulate(a, b, ar.codes.view(M, N), ar.scale)
    c, s = ar.run()
    rc, rs = api.agoq_reduce_shards([ar.codes], [ar.scale], 128)
    torch.cuda.synchronize()
    assert torch.equal(c, rc) and torch.equal(s, rs)
    assert int((rc != 0).sum()) > 0
