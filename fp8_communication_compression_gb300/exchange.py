"""The two-shot AllReduce in compressed form across the ranks of a process
group: the exchange around the shard reduce.

TACO (gist.science summary of arXiv 2604.24088), 2.B.3: the tensor-parallel
AllReduce runs as a ReduceScatter followed by an AllGather, with the
intermediate tensor compressed before it travels and decompressed after.
AGoQ (gist.science summary of arXiv 2605.00539), 2.B: gradients travel as
FP8 shards through an All-to-All, each rank sums the shards it receives in
FP32 and requantises, and an All-Gather returns the reduced shards.

With W ranks, the rows (or, for a flat gradient buffer, the blocks) are cut
into W contiguous chunks of equal size; rank j owns chunk j.  One call:

  1. compress the whole local tensor (one launch);
  2. All-to-All of codes, alpha and s: chunk j of every rank lands on rank j,
     in the rank's own memory, in rank order;
  3. the shard reduce over the W received chunks (one launch);
  4. AllGather of the reduced chunk's codes and scalars;
  5. decompress the gathered tensor (one launch).

Rows that do not divide evenly are padded: the last chunk is filled up with
rows whose codes are 0 and whose scalars are 1, written once when the
buffers are allocated and never touched by the compressor, so they reduce
and decompress to exact zeros and are cut off the result.

The collectives are torch.distributed calls on buffers in the rank's own
memory (NCCL on GPUs); no kernel reads another GPU's memory.  ``ops`` selects
the implementation of the three local steps: by default the library's CUDA
kernels.  Tests of the exchange bookkeeping on CPU ranks (gloo) pass their
own.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import api


def chunk_rows(rows: int, world: int) -> int:
    """Rows of each rank's chunk: the rows split into ``world`` equal chunks,
    the last padded."""
    if rows < 1 or world < 1:
        raise ValueError("rows and world size must be positive")
    return -(-rows // world)


class CudaOps:
    """The three local steps on the library's CUDA kernels."""

    @staticmethod
    def compress(x, codes, alpha, scale, block, e_target, eps):
        api.taco_compress(x, block, e_target, eps, codes=codes, alpha=alpha, scale=scale)

    @staticmethod
    def reduce(codes, alpha, scale, block, e_target, eps, out_codes, out_alpha, out_scale):
        api.taco_reduce_shards(codes, alpha, scale, block, e_target, eps, out_codes, out_alpha, out_scale)

    @staticmethod
    def decompress(codes, alpha, scale, block, out):
        api.taco_decompress(codes, alpha, scale, block, out=out)

    @staticmethod
    def agoq_reduce(codes, scale, block, out_codes, out_scale):
        api.agoq_reduce_shards(codes, scale, block, out_codes, out_scale)


class TwoShotAllReduce:
    """Sum of a bf16 [rows, d] tensor over the ranks of ``group``, exchanged
    as ASH+DS FP8 codes (TACO 2.B.3).  Buffers are allocated once; ``run``
    only launches and communicates.  Every rank returns the same
    reconstruction [rows, d]."""

    def __init__(self, rows: int, d: int, block: int = 128, group=None, device="cuda",
                 e_target: float = api.E_TARGET, eps: float = api.EPS, out_dtype=torch.float32, ops=None):
        if d % block:
            raise ValueError("d must be a multiple of the block size")
        self.group = group
        self.W = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.rows, self.d, self.block = rows, d, block
        self.e_target, self.eps = e_target, eps
        self.ops = ops if ops is not None else CudaOps
        self.R = chunk_rows(rows, self.W)
        self.Rb = self.R * d // block  # blocks per chunk
        W, R, Rb = self.W, self.R, self.Rb
        u8, f32 = torch.uint8, torch.float32
        # send side: the local tensor's codes and scalars, chunk j at [j]
        self.codes = torch.zeros((W * R, d), dtype=u8, device=device)
        self.alpha = torch.ones(W * Rb, dtype=f32, device=device)
        self.scale = torch.ones(W * Rb, dtype=f32, device=device)
        # receive side: this rank's chunk of every rank, in rank order
        self.recv_codes = torch.empty((W, R, d), dtype=u8, device=device)
        self.recv_alpha = torch.empty((W, Rb), dtype=f32, device=device)
        self.recv_scale = torch.empty((W, Rb), dtype=f32, device=device)
        # the reduced chunk, then every rank's reduced chunk
        self.red_codes = torch.empty((R, d), dtype=u8, device=device)
        self.red_alpha = torch.empty(Rb, dtype=f32, device=device)
        self.red_scale = torch.empty(Rb, dtype=f32, device=device)
        self.gat_codes = torch.empty((W * R, d), dtype=u8, device=device)
        self.gat_alpha = torch.empty(W * Rb, dtype=f32, device=device)
        self.gat_scale = torch.empty(W * Rb, dtype=f32, device=device)
        self.out = torch.empty((W * R, d), dtype=out_dtype, device=device)
        nb = rows * d // block
        self._codes_live = self.codes[:rows]
        self._alpha_live = self.alpha[:nb]
        self._scale_live = self.scale[:nb]

    def bytes_exchanged(self) -> dict:
        """Bytes each rank sends per call in the two collectives (codes and
        both scalars of the W - 1 chunks that leave the rank)."""
        chunk = self.R * self.d + 8 * self.Rb
        return {"all_to_all": (self.W - 1) * chunk, "all_gather": (self.W - 1) * chunk}

    def compress(self, x: torch.Tensor):
        self.ops.compress(x, self._codes_live, self._alpha_live, self._scale_live, self.block, self.e_target,
                          self.eps)

    def exchange(self):
        """ReduceScatter in compressed form: chunk j of every rank to rank j."""
        g = self.group
        dist.all_to_all_single(self.recv_codes.view(-1), self.codes.view(-1), group=g)
        dist.all_to_all_single(self.recv_alpha.view(-1), self.alpha, group=g)
        dist.all_to_all_single(self.recv_scale.view(-1), self.scale, group=g)

    def reduce(self):
        self.ops.reduce(list(self.recv_codes), list(self.recv_alpha), list(self.recv_scale), self.block,
                        self.e_target, self.eps, self.red_codes, self.red_alpha, self.red_scale)

    def gather(self):
        g = self.group
        dist.all_gather_into_tensor(self.gat_codes.view(-1), self.red_codes.view(-1), group=g)
        dist.all_gather_into_tensor(self.gat_alpha, self.red_alpha, group=g)
        dist.all_gather_into_tensor(self.gat_scale, self.red_scale, group=g)

    def decompress(self) -> torch.Tensor:
        self.ops.decompress(self.gat_codes, self.gat_alpha, self.gat_scale, self.block, self.out)
        return self.out[:self.rows]

    def run(self, x: torch.Tensor) -> torch.Tensor:
        """x: this rank's bf16 [rows, d] -> the sum over ranks, reconstructed
        ([rows, d] view of the output buffer)."""
        if tuple(x.shape) != (self.rows, self.d):
            raise ValueError(f"x must be [{self.rows}, {self.d}]")
        self.compress(x)
        self.exchange()
        self.reduce()
        self.gather()
        return self.decompress()


class AgoqAllReduce:
    """Sum of FP8 gradient buffers (codes + one dequantisation multiplier per
    block) over the ranks of ``group`` (AGoQ 2.B): All-to-All of the FP8
    shards, the FP32 shard reduce on each rank's chunk, All-Gather of the
    reduced codes and multipliers.  The buffer's n elements are cut into W
    chunks of whole blocks; the last chunk is padded with zero codes and
    multipliers of 1.  Every rank ends with the same reduced buffer.

    The rank's gradient buffer is ``codes`` / ``scale`` (views of the
    All-to-All's send buffer, initialised to the zero gradient): accumulate
    the micro-batches into them with ``agoq_fp8_accumulate``, then ``run``."""

    def __init__(self, n: int, block: int = 128, group=None, device="cuda", ops=None):
        if n % block or n < block:
            raise ValueError("n must be a positive multiple of the block size")
        self.group = group
        self.W = dist.get_world_size(group)
        self.n, self.block = n, block
        self.ops = ops if ops is not None else CudaOps
        nb = n // block
        self.Cb = chunk_rows(nb, self.W)  # blocks per chunk
        W, Cb = self.W, self.Cb
        self.send_codes = torch.zeros(W * Cb * block, dtype=torch.uint8, device=device)
        self.send_scale = torch.ones(W * Cb, dtype=torch.float32, device=device)
        self.codes = self.send_codes[:n]
        self.scale = self.send_scale[:nb]
        self.recv_codes = torch.empty((W, Cb * block), dtype=torch.uint8, device=device)
        self.recv_scale = torch.empty((W, Cb), dtype=torch.float32, device=device)
        self.red_codes = torch.empty(Cb * block, dtype=torch.uint8, device=device)
        self.red_scale = torch.empty(Cb, dtype=torch.float32, device=device)
        self.gat_codes = torch.empty(W * Cb * block, dtype=torch.uint8, device=device)
        self.gat_scale = torch.empty(W * Cb, dtype=torch.float32, device=device)

    def run(self):
        """Reduce ``codes`` / ``scale`` over the ranks -> (codes [n], scale
        [n / block]) of the sum, views of the gathered buffers."""
        g = self.group
        dist.all_to_all_single(self.recv_codes.view(-1), self.send_codes, group=g)
        dist.all_to_all_single(self.recv_scale.view(-1), self.send_scale, group=g)
        self.ops.agoq_reduce(list(self.recv_codes), list(self.recv_scale), self.block, self.red_codes,
                             self.red_scale)
        dist.all_gather_into_tensor(self.gat_codes, self.red_codes, group=g)
        dist.all_gather_into_tensor(self.gat_scale, self.red_scale, group=g)
        return self.gat_codes[:self.n], self.gat_scale[:self.n // self.block]
