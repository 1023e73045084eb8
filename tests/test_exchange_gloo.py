"""The two-shot exchange on CPU ranks (gloo, world sizes 2 and 3).

TACO (gist.science summary of arXiv 2604.24088), 2.B.3: ReduceScatter +
AllGather with the tensor compressed in between; AGoQ (gist.science summary
of arXiv 2605.00539), 2.B: All-to-All of FP8 shards, local FP32 sum,
All-Gather.  These tests check the exchange's bookkeeping: how the rows or
blocks are cut into chunks, the padding of a ragged last chunk, and the order
in which the received chunks reach the reduce.  The three local steps are
the oracle's here, passed in through ``ops`` (test infrastructure: on GPUs
the library's kernels run them).  The exchange only moves bytes and every
block is independent, so every rank's result must equal, bit for bit, the
oracle's reduce of all ranks' full tensors in rank order.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from fp8_communication_compression_gb300 import exchange
from fp8_communication_compression_gb300 import workloads as W


class OracleOps:
    """The local steps of the exchange on the CPU oracle (numpy)."""

    @staticmethod
    def compress(x, codes, alpha, scale, block, e_target, eps):
        bits = x.contiguous().view(torch.int16).numpy().view(np.uint16)
        c, a, s = oracle.compress(bits, block, e_target, eps)
        codes.copy_(torch.from_numpy(c))
        alpha.copy_(torch.from_numpy(a.reshape(-1)))
        scale.copy_(torch.from_numpy(s.reshape(-1)))

    @staticmethod
    def gemm_compress(a, w, codes, alpha, scale, block, e_target, eps):
        ab = a.contiguous().view(torch.int16).numpy().view(np.uint16)
        wb = w.contiguous().view(torch.int16).numpy().view(np.uint16)
        c, al, sc = oracle.gemm_compress(ab, wb, block, e_target, eps)
        codes.copy_(torch.from_numpy(c.reshape(codes.shape)))
        alpha.copy_(torch.from_numpy(al.reshape(-1)))
        scale.copy_(torch.from_numpy(sc.reshape(-1)))

    @staticmethod
    def reduce(codes, alpha, scale, block, e_target, eps, out_codes, out_alpha, out_scale):
        c, a, s = oracle.reduce_shards([t.numpy() for t in codes], [t.numpy() for t in alpha],
                                       [t.numpy() for t in scale], block, e_target, eps)
        out_codes.copy_(torch.from_numpy(c))
        out_alpha.copy_(torch.from_numpy(a.reshape(-1)))
        out_scale.copy_(torch.from_numpy(s.reshape(-1)))

    @staticmethod
    def decompress(codes, alpha, scale, block, out):
        out.copy_(torch.from_numpy(oracle.decompress(codes.numpy(), alpha.numpy(), scale.numpy(), block)
                                   .astype(np.float32)))

    @staticmethod
    def agoq_reduce(codes, scale, block, out_codes, out_scale):
        c, s = oracle.agoq_reduce([t.numpy() for t in codes], [t.numpy() for t in scale], block)
        out_codes.copy_(torch.from_numpy(c))
        out_scale.copy_(torch.from_numpy(s))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _taco_input(rank, rows, d, block):
    return W.tp_activation(50 + rank, rows, d, channel_scale=True, block=block)


GEMM_K = 64


def _gemm_operands(rank, rows, d):
    """Rank r's slice of a row-parallel layer: its activations [rows, K] and
    its slice of the weight [d, K], bf16."""
    a = W.tp_activation(80 + rank, rows, GEMM_K, channel_scale=True)
    w = W.f32_to_bf16_bits(np.random.default_rng(90 + rank).normal(0.0, 0.05, (d, GEMM_K)).astype(np.float32))
    return a, w


def _agoq_buffer(rank, n, block):
    c, s = np.zeros(n, np.uint8), np.ones(n // block, np.float32)
    for step in range(2):
        c, s = oracle.agoq_accumulate(c, s, W.agoq_grad(70 + 10 * rank + step, n), block)
    return c, s


def _worker(rank, world, port, case, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        kind, a, b, block, stages = case
        if kind == "gemm":
            rows, d = a, b
            xa, xw = _gemm_operands(rank, rows, d)
            ar = exchange.TwoShotAllReduce(rows, d, block, device="cpu", ops=OracleOps, stages=stages)
            ta = torch.from_numpy(xa.view(np.int16)).view(torch.bfloat16)
            tw = torch.from_numpy(xw.view(np.int16)).view(torch.bfloat16)
            q.put((rank, ar.run_gemm(ta, tw).clone().numpy(), ar.R, None))
        elif kind == "taco":
            rows, d = a, b
            x = torch.from_numpy(_taco_input(rank, rows, d, block).view(np.int16)).view(torch.bfloat16)
            ar = exchange.TwoShotAllReduce(rows, d, block, device="cpu", ops=OracleOps, stages=stages)
            out = ar.run(x).clone().numpy()
            sent = ar.bytes_exchanged()
            q.put((rank, out, ar.R, sent))
        else:
            n = a
            c, s = _agoq_buffer(rank, n, block)
            ar = exchange.AgoqAllReduce(n, block, device="cpu", ops=OracleOps)
            ar.codes.copy_(torch.from_numpy(c))
            ar.scale.copy_(torch.from_numpy(s))
            rc, rs = ar.run()
            q.put((rank, (rc.clone().numpy(), rs.clone().numpy()), ar.Cb, None))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(world, case):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, case, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return sorted(out, key=lambda o: o[0])


@pytest.mark.parametrize("world,rows,d,block,stages", [(2, 64, 512, 128, 1), (3, 50, 512, 256, 1),
                                                       (2, 64, 512, 128, 4), (3, 50, 256, 128, 3)])
def test_two_shot_exchange_equals_the_reduce_of_all_ranks(world, rows, d, block, stages):
    """stages > 1 is the overlapped exchange: pieces of every chunk travel
    in turn with asynchronous collectives (the 3-rank, 3-stage case has
    pieces that are partly and wholly padding)."""
    res = _run(world, ("taco", rows, d, block, stages))
    comp = [oracle.compress(_taco_input(r, rows, d, block), block) for r in range(world)]
    rc, ra, rs = oracle.reduce_shards(*zip(*comp), block)
    ref = oracle.decompress(rc, ra, rs, block).astype(np.float32)
    R = -(-(-(-rows // world)) // stages) * stages
    Rs = R // stages
    chunk_bytes = stages * (-(-(Rs * d + 8 * (Rs * d // block)) // 256) * 256)
    for rank, out, r_chunk, sent in res:
        assert r_chunk == R
        assert out.shape == (rows, d)
        assert np.array_equal(out.view(np.uint32), ref.view(np.uint32)), f"rank {rank}"
        assert sent == {"all_to_all": (world - 1) * chunk_bytes, "all_gather": (world - 1) * chunk_bytes}


@pytest.mark.parametrize("world,rows,d,stages", [(2, 256, 256, 1), (3, 768, 128, 2)])
def test_two_shot_exchange_of_gemm_outputs_equals_the_reduce_of_all_ranks(world, rows, d, stages):
    """run_gemm: each rank's partial sum Y_r = A_r W_r^T is compressed by the
    GEMM step piece by piece; the result equals the oracle's reduce of every
    rank's fused GEMM + compress over the whole tensor (every block is
    independent)."""
    res = _run(world, ("gemm", rows, d, 128, stages))
    comp = [oracle.gemm_compress(*_gemm_operands(r, rows, d), 128) for r in range(world)]
    rc, ra, rs = oracle.reduce_shards(*zip(*comp), 128)
    ref = oracle.decompress(rc, ra, rs, 128).astype(np.float32)
    for rank, out, _, _ in res:
        assert out.shape == (rows, d)
        assert np.array_equal(out.view(np.uint32), ref.view(np.uint32)), f"rank {rank}"


def test_run_gemm_rejects_pieces_that_are_not_whole_tiles():
    """300 rows over 2 ranks are chunks of 150 rows: not whole 128-row tiles
    of the GEMM, so run_gemm refuses before it launches anything."""
    with pytest.raises(ValueError):
        _check_pieces(300, 256, 2, 1)


def _check_pieces(rows, d, world, stages):
    """run_gemm's piece check without a process group: a one-rank gloo group
    over a free port."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    dist.init_process_group("gloo", rank=0, world_size=1)
    try:
        ar = exchange.TwoShotAllReduce(rows, d, 128, device="cpu", ops=OracleOps, stages=stages)
        a = torch.zeros((rows, 64), dtype=torch.bfloat16)
        w = torch.zeros((d, 64), dtype=torch.bfloat16)
        ar.run_gemm(a, w)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,cb", [(2, 19), (3, 13)])
def test_agoq_exchange_equals_the_reduce_of_all_ranks(world, cb):
    """37 blocks: chunks of 19 (2 ranks) or 13 (3 ranks) blocks, the last one
    padded with zero codes and multipliers of 1."""
    n, block = 37 * 128, 128
    res = _run(world, ("agoq", n, None, block, 1))
    bufs = [_agoq_buffer(r, n, block) for r in range(world)]
    rc, rs = oracle.agoq_reduce([b[0] for b in bufs], [b[1] for b in bufs], block)
    for rank, (c, s), got_cb, _ in res:
        assert got_cb == cb
        assert np.array_equal(c, rc) and np.array_equal(s, rs), f"rank {rank}"


def test_chunking_covers_every_row_once():
    for rows in (1, 7, 64, 8192):
        for world in (1, 2, 3, 8):
            R = exchange.chunk_rows(rows, world)
            # W chunks of R rows hold every row, and no smaller chunk would
            assert R * world >= rows and (R - 1) * world < rows
    with pytest.raises(ValueError):
        exchange.chunk_rows(0, 2)
