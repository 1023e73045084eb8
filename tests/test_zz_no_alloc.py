"""The no-allocation entry point, taco_two_shot_host_noalloc, called through
the C ABI.

It serves callers that cannot allocate device memory: code running inside an
allocator or memory-pool callback, sections where an allocation could block
or fail, programs whose device memory belongs to another component.  It
computes what the host pipeline (taco_host_pipeline_run) computes, with its
intermediate buffers in a fixed device array inside the library.  It is
checked against the pipeline on two calls in a row with different inputs,
at sizes that make each call go through the array in several chunks.

This file is collected last, so that a run stopping at its first failure
has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from fp8_communication_compression_gb300 import _lib
from fp8_communication_compression_gb300 import workloads as W

UNSUPPORTED = 2


def host_input(seed: int, P: int, rows: int, d: int, block: int) -> torch.Tensor:
    bits = np.stack([W.tp_activation(seed + p, rows, d, channel_scale=True, block=block) for p in range(P)])
    h = torch.empty((P, rows, d), dtype=torch.bfloat16, pin_memory=True)
    h.view(torch.int16).copy_(torch.from_numpy(bits.view(np.int16)))
    return h


def test_noalloc_rejects_a_row_that_does_not_fit_its_array():
    # 16 shards of 2^21-element rows need more than the array holds; the
    # call returns before any CUDA call
    lib = _lib.load()
    assert lib.taco_two_shot_host_noalloc(16, 1, 1 << 21, 128, 1 << 20, 1 << 21, 1.0, 1e-12, None) == UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("P,rows,d,block", [(4, 2100, 4096, 128), (3, 4000, 2560, 256)])
def test_noalloc_matches_the_host_pipeline_on_two_calls_in_a_row(P, rows, d, block):
    lib = _lib.load()
    ins = [host_input(700 + 10 * k, P, rows, d, block) for k in range(2)]

    # the existing entry point: the host pipeline with a caller-owned workspace
    h = ctypes.c_void_p()
    ws = ctypes.c_uint64()
    assert lib.taco_host_pipeline_create(P, rows, d, block, 4, 0, ctypes.byref(h), ctypes.byref(ws)) == 0
    workspace = torch.empty(ws.value, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    refs = []
    for x in ins:
        o = torch.empty((rows, d), dtype=torch.float32, pin_memory=True)
        assert lib.taco_host_pipeline_run(h, x.data_ptr(), o.data_ptr(), workspace.data_ptr(), 1.0, 1e-12,
                                          stream) == 0
        torch.cuda.synchronize()
        refs.append(o)
    assert lib.taco_host_pipeline_destroy(h) == 0

    # the no-allocation entry point, two calls in a row without synchronising
    outs = [torch.full((rows, d), float("nan"), dtype=torch.float32, pin_memory=True) for _ in range(2)]
    for x, o in zip(ins, outs):
        assert lib.taco_two_shot_host_noalloc(P, rows, d, block, x.data_ptr(), o.data_ptr(), 1.0, 1e-12,
                                              stream) == 0
    torch.cuda.synchronize()
    for o, r in zip(outs, refs):
        assert torch.equal(o.view(torch.int32), r.view(torch.int32))
