"""The bounded-wait failure path of the tensor-core kernel, run on the GPU
without faulting anything: a test hook shortens every pipeline wait to 20 ms
and makes CTA 0's first loader warp withhold one mbarrier arrive, so that
the QK issuer's wait runs out.  The kernel must then raise the workspace
error word (1), drain its own copies and MMAs, and return; the next normal
call on the same workspace must be parity-green with the error word clear.
"""
import time

import pytest
import torch

import parity
import sink_sda_decode_gb300 as sda
from sink_sda_decode_gb300 import inputs

pytestmark = pytest.mark.gpu


def _call(w, idx, ptr, ws):
    return sda.decode(w.q, w.unified_kv, idx, ptr, w.attn_sink, w.softmax_scale, workspace=ws)


def test_withheld_arrive_times_out_reports_and_recovers():
    w = inputs.random_small(seed=21, N=4, H=64, D=512, P=20000, lengths=[700, 64, 0, 300],
                            device="cuda")
    assert sda.decode_kernel(w.H, w.D) == "one_cta"
    idx, ptr = parity.to_dev(w)
    ws = torch.empty(sda.workspace_size(w.N, w.H, w.D, idx.numel()), dtype=torch.uint8,
                     device="cuda")
    _call(w, idx, ptr, ws)  # normal call first: library and kernels loaded
    torch.cuda.synchronize()
    assert sda.decode_error_flag(ws) == 0
    sda.debug_wait_fault(True, 20_000_000)
    try:
        t0 = time.perf_counter()
        _call(w, idx, ptr, ws)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        flag = sda.decode_error_flag(ws)
    finally:
        sda.debug_wait_fault(False, 0)
    assert flag == 1
    # the 20 ms bound applied (the default bound is 2 s per wait)
    assert elapsed < 1.5, elapsed
    out = _call(w, idx, ptr, ws)
    torch.cuda.synchronize()
    assert sda.decode_error_flag(ws) == 0
    parity.assert_parity(parity.compare(out, parity.run_oracle(w)), "after a timed-out call")
