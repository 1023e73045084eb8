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

  1. compress the local tensor (one launch per chunk, into a packed send
     buffer: each chunk's codes, alphas and scales as one byte run), or, for
     a row-parallel layer, compute the local partial sum with the GEMM that
     compresses in its epilogue (``TwoShotAllReduce.run_gemm``);
  2. All-to-All of the packed chunks: chunk j of every rank lands on rank j,
     in the rank's own memory, in rank order;
  3. the shard reduce over the W received chunks (one launch);
  4. AllGather of the reduced chunk, packed the same way;
  5. decompress the gathered chunks (one launch per chunk).

With ``stages`` > 1 the chunks travel in pieces and the kernels of one
piece overlap the collectives of another (TwoShotAllReduce).

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
    def gemm_compress(a, w, codes, alpha, scale, block, e_target, eps):
        api.taco_gemm_compress(a, w, block, e_target, eps, codes=codes, alpha=alpha, scale=scale)

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
    reconstruction [rows, d].

    ``stages`` > 1 overlaps the kernels with the collectives (TACO 2.B.3:
    the compression and decompression kernels run while communication is in
    flight).  Each rank's chunk is cut into ``stages`` pieces of Rs rows;
    piece k of every chunk travels in stage k.  The compress of stage k + 1
    runs while stage k's All-to-All is in flight, the reduce of stage k + 1
    while stage k's AllGather is, and the decompress of stage k while later
    AllGathers are.  The collectives are issued asynchronously; on GPUs each
    one waits for the kernels queued before it on the current stream, and
    the kernels that read its result wait for it.  Stage k's pieces are not
    contiguous rows of the tensor, so its compress and decompress are one
    launch per chunk."""

    def __init__(self, rows: int, d: int, block: int = 128, group=None, device="cuda",
                 e_target: float = api.E_TARGET, eps: float = api.EPS, out_dtype=torch.float32, ops=None,
                 stages: int = 1):
        if d % block:
            raise ValueError("d must be a multiple of the block size")
        if stages < 1:
            raise ValueError("stages must be at least 1")
        self.group = group
        self.W = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.rows, self.d, self.block = rows, d, block
        self.e_target, self.eps = e_target, eps
        self.ops = ops if ops is not None else CudaOps
        self.S = stages
        self.R = -(-chunk_rows(rows, self.W) // stages) * stages  # rows per chunk, a multiple of S
        self.Rs = self.R // stages                                # rows per piece
        self.Rb = self.R * d // block                             # blocks per chunk
        W, S, Rs = self.W, self.S, self.Rs
        self.Rsb = Rs * d // block
        # One piece travels as one packed byte run: Rs * d codes, then Rsb
        # fp32 alphas, then Rsb fp32 scales, padded to a multiple of 256
        # bytes so that every piece's codes start 256-byte aligned (the
        # scalars follow at 4-byte aligned offsets: Rs * d is a multiple of
        # 128).  Each stage is then one All-to-All and one AllGather.
        self.piece_bytes = -(-(Rs * d + 8 * self.Rsb) // 256) * 256
        u8 = torch.uint8
        # per stage k: the send side holds piece k of every chunk of the
        # local tensor (chunk j at [j]; rows past the tensor stay code 0 and
        # scalars 1); the receive side this rank's piece k from every rank,
        # in rank order; then its reduced piece, and every rank's reduced piece
        self.send = torch.zeros((S, W, self.piece_bytes), dtype=u8, device=device)
        self._alpha_of(self.send).fill_(1.0)
        self._scale_of(self.send).fill_(1.0)
        self.recv = torch.empty((S, W, self.piece_bytes), dtype=u8, device=device)
        self.red = torch.empty((S, self.piece_bytes), dtype=u8, device=device)
        self.gat = torch.empty((S, W, self.piece_bytes), dtype=u8, device=device)
        self.out = torch.empty((W * self.R, d), dtype=out_dtype, device=device)

    # views of packed pieces (last dimension = one piece's bytes)
    def _codes_of(self, t):
        return t[..., :self.Rs * self.d].unflatten(-1, (self.Rs, self.d))

    def _alpha_of(self, t):
        o = self.Rs * self.d
        return t[..., o:o + 4 * self.Rsb].view(torch.float32)

    def _scale_of(self, t):
        o = self.Rs * self.d + 4 * self.Rsb
        return t[..., o:o + 4 * self.Rsb].view(torch.float32)

    def bytes_exchanged(self) -> dict:
        """Bytes each rank sends per call in the two collectives (codes and
        both scalars of the W - 1 chunks that leave the rank)."""
        chunk = self.S * self.piece_bytes
        return {"all_to_all": (self.W - 1) * chunk, "all_gather": (self.W - 1) * chunk}

    def _piece(self, j: int, k: int):
        """Rows of the tensor in piece k of chunk j (possibly fewer than Rs,
        or none, at the padded end)."""
        r0 = j * self.R + k * self.Rs
        return r0, max(r0, min(r0 + self.Rs, self.rows))

    def compress(self, x: torch.Tensor, k: int = 0):
        """Stage k's pieces of the local tensor into the send buffer."""
        nbr = self.d // self.block
        for j in range(self.W):
            r0, r1 = self._piece(j, k)
            if r1 > r0:
                n = r1 - r0
                piece = self.send[k, j]
                self.ops.compress(x[r0:r1], self._codes_of(piece)[:n], self._alpha_of(piece)[:n * nbr],
                                  self._scale_of(piece)[:n * nbr], self.block, self.e_target, self.eps)

    def compress_gemm(self, a: torch.Tensor, w: torch.Tensor, k: int = 0):
        """Stage k's pieces of this rank's partial sum Y = a w^T, computed
        and compressed by the GEMM with the compressor in its epilogue, one
        launch per piece, straight into the send buffer."""
        nbr = self.d // self.block
        for j in range(self.W):
            r0, r1 = self._piece(j, k)
            if r1 > r0:
                n = r1 - r0
                piece = self.send[k, j]
                self.ops.gemm_compress(a[r0:r1], w, self._codes_of(piece)[:n], self._alpha_of(piece)[:n * nbr],
                                       self._scale_of(piece)[:n * nbr], self.block, self.e_target, self.eps)

    def exchange(self, k: int = 0, async_op: bool = False):
        """ReduceScatter in compressed form: piece k of chunk j of every rank
        to rank j (codes and both scalars in one collective)."""
        return dist.all_to_all_single(self.recv[k].view(-1), self.send[k].view(-1), group=self.group,
                                      async_op=async_op)

    def reduce(self, k: int = 0):
        r, out = self.recv[k], self.red[k]
        self.ops.reduce(list(self._codes_of(r)), list(self._alpha_of(r)), list(self._scale_of(r)), self.block,
                        self.e_target, self.eps, self._codes_of(out), self._alpha_of(out), self._scale_of(out))

    def gather(self, k: int = 0, async_op: bool = False):
        return dist.all_gather_into_tensor(self.gat[k].view(-1), self.red[k], group=self.group, async_op=async_op)

    def decompress(self, k: int = 0) -> torch.Tensor:
        g = self.gat[k]
        for j in range(self.W):
            r0 = j * self.R + k * self.Rs
            self.ops.decompress(self._codes_of(g[j]), self._alpha_of(g[j]), self._scale_of(g[j]), self.block,
                                self.out[r0:r0 + self.Rs])
        return self.out[:self.rows]

    def run(self, x: torch.Tensor) -> torch.Tensor:
        """x: this rank's bf16 [rows, d] -> the sum over ranks, reconstructed
        ([rows, d] view of the output buffer)."""
        if tuple(x.shape) != (self.rows, self.d):
            raise ValueError(f"x must be [{self.rows}, {self.d}]")
        return self._run(lambda k: self.compress(x, k))

    def run_gemm(self, a: torch.Tensor, w: torch.Tensor) -> torch.Tensor:
        """The AllReduce of a row-parallel layer's output: this rank's partial
        sum is Y = a w^T (a bf16 [rows, K], w bf16 [d, K], its slice of the
        weight), produced already compressed by the GEMM's epilogue (AGoQ
        2.C's fusion applied to the TACO compressor), then exchanged as in
        ``run``.  Every piece must be a multiple of 128 rows (the GEMM's
        tile): rows a multiple of 128 and of 128 x world size x stages
        rows per chunk do it."""
        if a.dim() != 2 or w.dim() != 2 or a.shape[0] != self.rows or w.shape[0] != self.d or \
                a.shape[1] != w.shape[1]:
            raise ValueError(f"a must be [{self.rows}, K] and w [{self.d}, K]")
        for j in range(self.W):
            for k in range(self.S):
                r0, r1 = self._piece(j, k)
                if (r1 - r0) % 128:
                    raise ValueError(f"piece {k} of chunk {j} has {r1 - r0} rows, not a multiple of 128")
        return self._run(lambda k: self.compress_gemm(a, w, k))

    def _run(self, compress) -> torch.Tensor:
        if self.S == 1:
            compress(0)
            self.exchange()
            self.reduce()
            self.gather()
            return self.decompress()
        a2a = []
        for k in range(self.S):  # compress k + 1 is queued while exchange k is in flight
            compress(k)
            a2a.append(self.exchange(k, async_op=True))
        ag = []
        for k in range(self.S):
            a2a[k].wait()
            self.reduce(k)
            ag.append(self.gather(k, async_op=True))
        for k in range(self.S):
            ag[k].wait()
            self.decompress(k)
        return self.out[:self.rows]


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
