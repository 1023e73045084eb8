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
