"""sda_decode_noalloc: the decode for callers that cannot allocate device
memory (hosts that give an operator only its input and output buffers, or C
callers without a device allocator).  Its scratch memory is a fixed device
array inside the library.

Checked through the C ABI (ctypes, no Python wrapper in between): two calls
in a row, on different workloads, each against the regular sda_decode entry
point on the same inputs and against the fp64 oracle, within the parity
tolerance of the other GPU tests.
This file is collected last on purpose; it passes alone in a fresh process
and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import parity
import sink_sda_decode_gb300 as sda
from sink_sda_decode_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20  # SDA_NOALLOC_SCRATCH_BYTES in include/sda.h


def _noalloc(lib, w, idx, ptr, out):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.sda_decode_noalloc(w.q.data_ptr(), w.unified_kv.data_ptr(), w.unified_kv.shape[0],
                                  idx.data_ptr(), idx.numel(), ptr.data_ptr(),
                                  w.attn_sink.data_ptr(), ctypes.c_float(w.softmax_scale), w.N,
                                  w.H, w.D, out.data_ptr(), stream)


def _check_against_decode(w, out, ref64=None):
    idx, ptr = parity.to_dev(w)
    ref = sda.decode(w.q, w.unified_kv, idx, ptr, w.attn_sink, w.softmax_scale)
    torch.cuda.synchronize()
    d = (out.double() - ref.double()).abs()
    assert d.max().item() <= parity.MAX_ABS and d.mean().item() <= parity.MEAN_ABS
    assert torch.all(out[torch.from_numpy(np.nonzero(w.lengths == 0)[0]).cuda()].view(torch.int16) == 0)
    # and against the fp64 oracle on the same inputs
    if ref64 is None:
        ref64 = parity.run_oracle(w)
    parity.assert_parity(parity.compare(out, ref64), "noalloc vs oracle")
    return ref64


def test_noalloc_two_calls_match_decode():
    lib = _lib.load()
    # call 1: the N=64, H=16, D=512, L=640 workload (lists split across CTAs)
    w1 = inputs.config(1, device="cuda")
    i1, p1 = parity.to_dev(w1)
    assert sda.workspace_size(w1.N, w1.H, w1.D, i1.numel()) <= SCRATCH_BYTES
    o1 = torch.full_like(w1.q, 9.0)
    assert _noalloc(lib, w1, i1, p1, o1) == 0
    torch.cuda.synchronize()
    ref1 = _check_against_decode(w1, o1)
    # call 2 right after, different shapes and lengths (empty, ragged, long)
    w2 = inputs.random_small(seed=77, N=6, H=32, D=512, P=40000,
                             lengths=[0, 1, 65, 640, 5000, 129], device="cuda")
    i2, p2 = parity.to_dev(w2)
    o2 = torch.full_like(w2.q, 9.0)
    assert _noalloc(lib, w2, i2, p2, o2) == 0
    torch.cuda.synchronize()
    _check_against_decode(w2, o2)
    # and call 1's output was not disturbed by call 2 sharing the scratch
    _check_against_decode(w1, o1, ref1)


def test_noalloc_rejects_sizes_beyond_the_array():
    lib = _lib.load()
    w = inputs.random_small(seed=78, N=300, H=128, D=512, P=4096, lengths=[64] * 300, device="cuda")
    idx, ptr = parity.to_dev(w)
    assert sda.workspace_size(w.N, w.H, w.D, idx.numel()) > SCRATCH_BYTES
    out = torch.full_like(w.q, 9.0)
    assert _noalloc(lib, w, idx, ptr, out) == 4  # SDA_ERR_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()
    assert torch.all(out == 9.0)
