"""GPU parity of sda_decode against the fp64 oracle (through the C ABI).

Full sizes of the five workloads (and the sparse-prefill chunk) run in the
same launch configuration the benchmark times, and every token of every
workload is compared with the oracle, element by element.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import parity
import sink_sda_decode_gb300 as sda
from sink_sda_decode_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_forced_variant(monkeypatch):
    monkeypatch.delenv("SDA_FORCE_VARIANT", raising=False)


def _force(monkeypatch, variant):
    if variant != "default":
        monkeypatch.setenv("SDA_FORCE_VARIANT", variant)


@pytest.mark.parametrize("cfg", range(len(inputs.CONFIG_NAMES)), ids=inputs.CONFIG_NAMES)
def test_workload_parity(cfg):
    w = inputs.config(cfg, device="cuda")
    out = parity.run_gpu(w)
    torch.cuda.synchronize()
    ref = parity.run_oracle(w)
    st = parity.compare(out, ref)
    print(f"\n{inputs.CONFIG_NAMES[cfg]}: {st}")
    parity.assert_parity(st, inputs.CONFIG_NAMES[cfg])
    # padded tokens: exactly +0.0 (bf16 bit pattern 0)
    zero = np.nonzero(w.lengths == 0)[0]
    if zero.size:
        z = out[torch.from_numpy(zero).to(out.device)]
        assert torch.all(z.view(torch.int16) == 0)


def _ws_and_flag(w):
    idx, ptr = parity.to_dev(w)
    n = sda.workspace_size(w.N, w.H, w.D, idx.numel())
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = sda.decode(w.q, w.unified_kv, idx, ptr, w.attn_sink, w.softmax_scale, workspace=ws)
    return out, sda.decode_error_flag(ws)


def test_kernel_choice():
    """D = 512 with H in {16, 32, 64k} runs the one-CTA tensor-core kernel;
    other shapes the CUDA-core kernel."""
    for H in (16, 32, 64, 128):
        assert sda.decode_kernel(H, 512) == "one_cta"
    assert sda.decode_kernel(48, 512) == "simt"
    assert sda.decode_kernel(16, 128) == "simt"


def test_kernel_choice_forced(monkeypatch):
    """The environment switch reaches the CUDA-core kernel."""
    monkeypatch.setenv("SDA_FORCE_VARIANT", "simt")
    assert sda.decode_kernel(64, 512) == "simt"
    monkeypatch.setenv("SDA_FORCE_VARIANT", "umma")
    assert sda.decode_kernel(64, 512) == "one_cta"


def test_error_flag_clear_after_normal_call():
    w = inputs.config(1, device="cuda")
    _, flag = _ws_and_flag(w)
    assert flag == 0


# ----------------------------------------------------------------------------- shapes
SHAPES = [  # (H, D) -- tensor-core path for D=512 and H in {16,32,64k}; CUDA cores otherwise
    (16, 512), (32, 512), (64, 512), (128, 512), (192, 512), (256, 512),
    (8, 512), (48, 512), (1, 64), (3, 128), (8, 256), (24, 64),
]
LENGTHS = [0, 1, 2, 31, 63, 64, 65, 127, 128, 129, 300, 640, 1000, 2500]


@pytest.mark.parametrize("H,D", SHAPES, ids=[f"H{h}_D{d}" for h, d in SHAPES])
def test_shapes_and_ragged_lengths(H, D):
    _check_shape(H, D)


def _check_shape(H, D):
    w = inputs.random_small(seed=1000 + H + D, N=len(LENGTHS), H=H, D=D, P=20000, lengths=LENGTHS,
                            device="cuda")
    out = parity.run_gpu(w)
    ref = parity.run_oracle(w)
    st = parity.compare(out, ref)
    parity.assert_parity(st, f"H={H} D={D}")
    assert torch.all(out[0].view(torch.int16) == 0)


@pytest.mark.parametrize("variant", ["simt", "default"])
def test_split_long_lists(monkeypatch, variant):
    """Few tokens with long lists: the plan cuts every list into pieces and
    the combine kernel merges them (including the sink exactly once)."""
    _force(monkeypatch, variant)
    w = inputs.random_small(seed=7, N=3, H=64, D=512, P=1 << 17, lengths=[30000, 5, 12345],
                            sink_sigma=2.0, device="cuda")
    out = parity.run_gpu(w)
    ref = parity.run_oracle(w)
    parity.assert_parity(parity.compare(out, ref), f"split {variant}")


def test_split_merge_repeats_on_one_workspace(monkeypatch):
    """Split tokens over two head groups with +-inf and finite sinks, three
    calls on one workspace: identical outputs, each within the oracle bound."""
    w = inputs.random_small(seed=17, N=4, H=128, D=512, P=1 << 16, lengths=[9000, 3, 0, 4000],
                            sink_sigma=1.5, device="cuda")
    sink = w.attn_sink.clone()
    sink[0], sink[70], sink[127] = -math.inf, math.inf, 30.0
    idx, ptr = parity.to_dev(w)
    total = int(w.kv_indptr[-1])
    ws = torch.empty(sda.workspace_size(w.N, w.H, w.D, total), dtype=torch.uint8, device="cuda")
    ref = parity.run_oracle(w, sink=sink)
    outs = [sda.decode(w.q, w.unified_kv, idx, ptr, sink, w.softmax_scale, workspace=ws)
            for _ in range(3)]
    for k, out in enumerate(outs):
        parity.assert_parity(parity.compare(out, ref), f"split merge call {k}")
        assert torch.equal(out, outs[0])
    assert sda.decode_error_flag(ws) == 0


def test_variants_agree(monkeypatch):
    """CUDA-core and tensor-core kernels on the same input."""
    w = inputs.random_small(seed=8, N=5, H=64, D=512, P=50000, lengths=[1, 64, 700, 0, 129],
                            device="cuda")
    a = parity.run_gpu(w).float()
    monkeypatch.setenv("SDA_FORCE_VARIANT", "simt")
    b = parity.run_gpu(w).float()
    monkeypatch.delenv("SDA_FORCE_VARIANT")
    assert (a - b).abs().max().item() <= 2 * parity.MAX_ABS


# ----------------------------------------------------------------------------- edge cases
def test_sink_minus_inf_and_plus_inf():
    w = inputs.random_small(seed=9, N=4, H=16, D=512, P=4000, lengths=[0, 1, 50, 200], device="cuda")
    sink = torch.full((16,), -math.inf, device="cuda")
    out = parity.run_gpu(w, sink=sink)
    parity.assert_parity(parity.compare(out, parity.run_oracle(w, sink=sink)), "sink -inf")
    assert torch.all(out[0].view(torch.int16) == 0)  # empty list and no sink: 0 (reading)
    sink = torch.full((16,), math.inf, device="cuda")
    out = parity.run_gpu(w, sink=sink)
    assert torch.all(out.view(torch.int16) == 0)
    sink = torch.tensor([(-1) ** h * 30.0 for h in range(16)], device="cuda")  # huge sinks
    out = parity.run_gpu(w, sink=sink)
    parity.assert_parity(parity.compare(out, parity.run_oracle(w, sink=sink)), "sink +-30")


def test_single_slot_closed_form():
    w = inputs.random_small(seed=10, N=6, H=64, D=512, P=3000, lengths=[1] * 6, sink_sigma=2.0,
                            device="cuda")
    out = parity.run_gpu(w).double().cpu().numpy()
    q = w.q.double().cpu().numpy()
    kv = w.unified_kv.double().cpu().numpy()
    sink = w.attn_sink.double().cpu().numpy()
    for t in range(6):
        v = kv[w.kv_indices[t]]
        x = (q[t] @ v) * np.float32(w.softmax_scale)
        ref = (1.0 / (1.0 + np.exp(sink - x)))[:, None] * v[None, :]
        st = parity.compare(torch.from_numpy(out[t]), ref)
        parity.assert_parity(st, "single slot")


def test_duplicates_scale_zero_and_convexity():
    w = inputs.random_small(seed=11, N=4, H=32, D=512, P=100, lengths=[300, 64, 2, 1000],
                            duplicates=True, device="cuda")
    out = parity.run_gpu(w)
    parity.assert_parity(parity.compare(out, parity.run_oracle(w)), "duplicates")
    out0 = parity.run_gpu(w, scale=0.0)
    parity.assert_parity(parity.compare(out0, parity.run_oracle(w, scale=0.0)), "scale 0")
    kv = w.unified_kv.float()
    for t in range(4):
        rows = kv[torch.from_numpy(w.kv_indices[w.kv_indptr[t]:w.kv_indptr[t + 1]].astype(np.int64)).cuda()]
        bound = rows.abs().max(0).values
        assert torch.all(out[t].float().abs() <= bound[None, :] + 1e-6)


def test_permutation_invariance():
    w = inputs.random_small(seed=12, N=2, H=64, D=512, P=60000, lengths=[1500, 333], device="cuda")
    a = parity.run_gpu(w)
    idx = w.kv_indices.copy()
    rng = np.random.default_rng(0)
    for t in range(2):
        idx[w.kv_indptr[t]:w.kv_indptr[t + 1]] = rng.permutation(idx[w.kv_indptr[t]:w.kv_indptr[t + 1]])
    b = sda.decode(w.q, w.unified_kv, torch.from_numpy(idx).cuda(),
                   torch.from_numpy(w.kv_indptr).cuda(), w.attn_sink, w.softmax_scale)
    # the order changes which running max each p is rounded against (P is
    # bf16 for the tensor cores), so the two agree to the parity tolerance
    d = (a.double() - b.double()).abs()
    assert d.max().item() <= parity.MAX_ABS and d.mean().item() <= parity.MEAN_ABS
    parity.assert_parity(parity.compare(b, parity.run_oracle(w)), "permuted")


def test_growing_logits_rescale():
    """Lists sorted by increasing logit with a large score range, so the
    running max grows tile after tile and the O rescale path runs."""
    w = inputs.random_small(seed=13, N=3, H=64, D=512, P=40000, lengths=[2000, 700, 129],
                            device="cuda")
    # q[t, h] = 2 * (a pool row), lists sorted ascending by <q[t,0], k>
    kv = w.unified_kv
    for t in range(3):
        s = w.kv_indptr[t]
        e = w.kv_indptr[t + 1]
        rows = torch.from_numpy(w.kv_indices[s:e].astype(np.int64)).cuda()
        w.q[t] = (2.0 * kv[rows[-1]].float()).to(torch.bfloat16)[None, :].expand(w.H, -1)
        dots = (kv[rows].float() @ w.q[t, 0].float())
        w.kv_indices[s:e] = w.kv_indices[s:e][dots.argsort().cpu().numpy()]
    out = parity.run_gpu(w)
    parity.assert_parity(parity.compare(out, parity.run_oracle(w)), "growing logits")


def test_indptr_offset_and_subset_lists():
    """kv_indptr[0] != 0 and unused entries before/after the slices."""
    w = inputs.random_small(seed=14, N=4, H=16, D=512, P=5000, lengths=[10, 0, 100, 70], device="cuda")
    pad = np.full(37, 123456789, np.int32)  # never read: outside every slice
    idx = np.concatenate([pad, w.kv_indices, pad])
    ptr = w.kv_indptr + 37
    out = sda.decode(w.q, w.unified_kv, torch.from_numpy(idx).cuda(), torch.from_numpy(ptr).cuda(),
                     w.attn_sink, w.softmax_scale)
    parity.assert_parity(parity.compare(out, parity.run_oracle(w)), "offset indptr")


def test_bad_indptr_is_refused_on_device():
    """A decreasing kv_indptr: nothing is computed, the error word reads 2."""
    w = inputs.random_small(seed=15, N=3, H=16, D=512, P=5000, lengths=[10, 20, 30], device="cuda")
    idx, _ = parity.to_dev(w)
    bad = torch.tensor([0, 20, 10, 60], dtype=torch.int32, device="cuda")
    ws = torch.empty(sda.workspace_size(3, 16, 512, idx.numel()), dtype=torch.uint8, device="cuda")
    out = torch.full_like(w.q, 7.0)
    sda.decode(w.q, w.unified_kv, idx, bad, w.attn_sink, w.softmax_scale, out=out, workspace=ws)
    assert sda.decode_error_flag(ws) == 2
    assert torch.all(out == 7.0)


def test_guard_bytes_untouched():
    w = inputs.random_small(seed=16, N=5, H=128, D=512, P=9000, lengths=[0, 64, 65, 1, 900],
                            device="cuda")
    n = w.N * w.H * w.D
    buf = torch.full((n + 2 * 4096,), 3.0, dtype=torch.bfloat16, device="cuda")
    out = buf[4096:4096 + n].view(w.N, w.H, w.D)
    parity.run_gpu(w, out=out)
    assert torch.all(buf[:4096] == 3.0) and torch.all(buf[4096 + n:] == 3.0)
    parity.assert_parity(parity.compare(out, parity.run_oracle(w)), "guard")


def test_cuda_graph_capture_replay():
    w = inputs.random_small(seed=17, N=6, H=64, D=512, P=30000, lengths=[0, 5, 640, 3000, 64, 200],
                            device="cuda")
    idx, ptr = parity.to_dev(w)
    ws = torch.empty(sda.workspace_size(w.N, w.H, w.D, idx.numel()), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(w.q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sda.decode(w.q, w.unified_kv, idx, ptr, w.attn_sink, w.softmax_scale, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    ref = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sda.decode(w.q, w.unified_kv, idx, ptr, w.attn_sink, w.softmax_scale, out=out, workspace=ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # new lengths in the same buffers (the graph reads indptr on the device)
    new_ptr = torch.tensor([0, 3, 3, 600, 3600, 3664, 3864], dtype=torch.int32, device="cuda")
    ptr.copy_(new_ptr)
    g.replay()
    torch.cuda.synchronize()
    ref2 = oracle.sda_decode(w.q_bits(), oracle.bf16_bits(w.unified_kv), w.kv_indices,
                             new_ptr.cpu().numpy(), w.attn_sink.cpu().numpy(), w.softmax_scale)
    parity.assert_parity(parity.compare(out, ref2), "graph replay with new lengths")


def test_decode_host_e2e():
    w = inputs.random_small(seed=18, N=4, H=16, D=512, P=4000, lengths=[3, 0, 64, 100], device="cuda")
    q_h = w.q.cpu().pin_memory()
    idx_h = torch.from_numpy(w.kv_indices).pin_memory()
    ptr_h = torch.from_numpy(w.kv_indptr).pin_memory()
    out = sda.decode_host(q_h, w.unified_kv, idx_h, ptr_h, w.attn_sink, w.softmax_scale)
    assert not out.is_cuda
    parity.assert_parity(parity.compare(out, parity.run_oracle(w)), "host e2e")


def test_timing_hook_records_around_the_kernel():
    w = inputs.random_small(seed=19, N=8, H=64, D=512, P=30000, lengths=[640] * 8, device="cuda")
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    sda.set_timing_events(a, b)
    try:
        out = parity.run_gpu(w)
    finally:
        sda.set_timing_events(None, None)
    torch.cuda.synchronize()
    assert a.elapsed_time(b) > 0.0
    parity.assert_parity(parity.compare(out, parity.run_oracle(w)), "timing hook")


def test_negative_and_large_softmax_scale():
    """The kernels must not assume softmax_scale > 0 (the running max of the
    scaled logits comes from the smallest raw score when the scale is negative)."""
    w = inputs.random_small(seed=20, N=3, H=64, D=512, P=20000, lengths=[700, 64, 1], device="cuda")
    for scale in (-w.softmax_scale, 4.0 * w.softmax_scale):
        out = parity.run_gpu(w, scale=scale)
        parity.assert_parity(parity.compare(out, parity.run_oracle(w, scale=scale)), f"scale {scale}")


@pytest.mark.parametrize("variant", ["simt", "default"])
def test_plan_large_batch_with_tail_padding(monkeypatch, variant):
    """13 000 tokens (more than the work plan keeps in shared memory, so its
    token arrays live in the workspace), short ragged lists and a tail of
    3 000 padded tokens (zero-length slices, dealt round-robin over the CTAs):
    every token matches the oracle and every padded token is +0."""
    _force(monkeypatch, variant)
    rng = np.random.default_rng(31)
    N, pad = 13000, 3000
    lengths = list(rng.integers(0, 41, size=N - pad)) + [0] * pad
    w = inputs.random_small(seed=31, N=N, H=16, D=512, P=1 << 16, lengths=lengths, device="cuda")
    out = parity.run_gpu(w)
    parity.assert_parity(parity.compare(out, parity.run_oracle(w)), f"N={N} tail padding {variant}")
    assert not out[N - pad:].view(torch.int16).any()


@pytest.mark.parametrize("variant", ["simt", "default"])
def test_batch_without_slots(monkeypatch, variant):
    """Every slice empty: the plan has no ranges, every output is +0 and no
    error is raised."""
    _force(monkeypatch, variant)
    w = inputs.random_small(seed=32, N=300, H=64, D=512, P=4096, lengths=[0] * 300, device="cuda")
    idx, ptr = parity.to_dev(w)
    ws = torch.empty(sda.workspace_size(w.N, w.H, w.D, 0), dtype=torch.uint8, device="cuda")
    out = torch.full_like(w.q, 7.0)
    sda.decode(w.q, w.unified_kv, idx, ptr, w.attn_sink, w.softmax_scale, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert not out.view(torch.int16).any()
    assert sda.decode_error_flag(ws) == 0
