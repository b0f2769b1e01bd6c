"""sda_build_decode: the index build and the decode as one call (the builder's
scan and the decode's work plan share one CTA).  It must give exactly what
the two calls give back to back -- bit-identical lists, status and output --
and therefore match the oracle's build + decode."""
import numpy as np
import pytest
import torch

import oracle
import parity
import sink_sda_decode_gb300 as sda
from sink_sda_decode_gb300 import inputs

pytestmark = pytest.mark.gpu


def two_calls(w, bi, pool=None, capacity=None):
    idx, ptr, st = sda.build_indices(**bi, win=w.win, k_per_block=w.k_per_block,
                                     swa_pages=w.swa_pages, total_pages=w.total_pages,
                                     capacity=capacity)
    if pool is None:
        out = sda.decode(w.q, w.unified_kv, idx, ptr, w.attn_sink, w.softmax_scale)
    else:
        out = sda.decode_fp8(w.q, pool.codes, pool.scale, idx, ptr, w.attn_sink, w.softmax_scale)
    return out, idx, ptr, st


def fused(w, bi, pool=None, capacity=None):
    kv = w.unified_kv if pool is None else pool.codes
    return sda.build_decode(w.q, kv, w.attn_sink, w.softmax_scale, bi["state_slot"], bi["swa_len"],
                            bi["swa_head"], bi["comp_indptr"], bi["comp_block"], bi["comp_slot"],
                            win=w.win, k_per_block=w.k_per_block, swa_pages=w.swa_pages,
                            kv_scale=None if pool is None else pool.scale, capacity=capacity)


def assert_same(a, b):
    out_a, idx_a, ptr_a, st_a = a
    out_b, idx_b, ptr_b, st_b = b
    torch.cuda.synchronize()
    n = int(ptr_a[-1].item())
    assert int(st_a.item()) == int(st_b.item())
    assert torch.equal(ptr_a, ptr_b) and torch.equal(idx_a[:n], idx_b[:n])
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))


@pytest.mark.parametrize("cfg", [0, 1, 2, 4], ids=[inputs.CONFIG_NAMES[c] for c in (0, 1, 2, 4)])
def test_fused_equals_two_calls(cfg):
    w = inputs.config(cfg, device="cuda")
    bi = w.builder_inputs("cuda")
    assert_same(fused(w, bi), two_calls(w, bi))


def test_fused_fp8_equals_two_calls():
    w = inputs.config(2, device="cuda")
    bi = w.builder_inputs("cuda")
    pool = inputs.fp8_pool(w)
    assert_same(fused(w, bi, pool), two_calls(w, bi, pool))


def test_fused_matches_the_oracle_chain():
    w = inputs.config(1, device="cuda")
    bi = w.builder_inputs("cuda")
    out, idx, ptr, st = fused(w, bi)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_idx, o_ptr, o_st = oracle.build_indices(w.state_slot, w.swa_len, w.swa_head, w.comp_indptr,
                                              w.comp_block, w.comp_slot, w.win, w.k_per_block,
                                              w.swa_pages, w.total_pages)
    assert o_st == 0 and np.array_equal(ptr.cpu().numpy(), o_ptr)
    assert np.array_equal(idx.cpu().numpy()[: o_ptr[-1]], o_idx)
    parity.assert_parity(parity.compare(out, parity.run_oracle(w)), "fused build + decode")


def test_fused_bad_descriptors_and_capacity():
    """Bad tokens get empty slices (output +0) and their status bits; too
    small a capacity empties every list (bit 32) and every output is +0."""
    w = inputs.config(1, device="cuda")
    bi = {k: v.clone() for k, v in w.builder_inputs("cuda").items()}
    bi["swa_len"][3] = w.win + 1          # bit 1
    bi["comp_slot"][bi["comp_indptr"][5]] = w.k_per_block  # bit 8
    out, idx, ptr, st = fused(w, bi)
    ref = two_calls(w, bi)
    assert_same((out, idx, ptr, st), ref)
    assert int(st.item()) == 1 | 8
    assert not out[3].view(torch.int16).any() and not out[5].view(torch.int16).any()
    out, idx, ptr, st = fused(w, bi, capacity=100)
    torch.cuda.synchronize()
    assert int(st.item()) & 32 and not ptr.any() and not out.view(torch.int16).any()


def test_fused_graph_capture_and_empty_batch():
    w = inputs.config(1, device="cuda")
    bi = w.builder_inputs("cuda")
    cap = w.N * w.win + int(w.comp_block.size)
    idx = torch.empty(cap, dtype=torch.int32, device="cuda")
    ptr = torch.empty(w.N + 1, dtype=torch.int32, device="cuda")
    st = torch.empty(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(w.q)
    ws = torch.empty(sda.workspace_size(w.N, w.H, w.D, cap), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    kw = dict(win=w.win, k_per_block=w.k_per_block, swa_pages=w.swa_pages, capacity=cap, out=out,
              workspace=ws, kv_indices=idx, kv_indptr=ptr, status=st, stream=s)
    args = (w.q, w.unified_kv, w.attn_sink, w.softmax_scale, bi["state_slot"], bi["swa_len"],
            bi["swa_head"], bi["comp_indptr"], bi["comp_block"], bi["comp_slot"])
    with torch.cuda.stream(s):
        sda.build_decode(*args, **kw)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sda.build_decode(*args, **kw)
    out.zero_()
    ptr.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    assert_same((out, idx, ptr, st), two_calls(w, bi))
    # N = 0: the builder still writes kv_indptr[0] = 0 and a zero status
    e = torch.zeros(0, dtype=torch.int32, device="cuda")
    o, i, p, s0 = sda.build_decode(w.q[:0], w.unified_kv, w.attn_sink, w.softmax_scale, e, e, e,
                                   torch.zeros(1, dtype=torch.int32, device="cuda"), e, e,
                                   win=w.win, k_per_block=w.k_per_block, swa_pages=w.swa_pages)
    torch.cuda.synchronize()
    assert p.tolist() == [0] and int(s0.item()) == 0 and o.shape[0] == 0


def pinned(t):
    return t.cpu().pin_memory()


def host_call(w, bi, pool=None, out=None, status=None, workspace=None, stream=None):
    """One build_decode_host call on pinned copies of the inputs.  The copies
    are temporaries, so the call's stream is synchronised before they go out
    of scope (the kernels read them asynchronously)."""
    kv = w.unified_kv if pool is None else pool.codes
    h = {k: pinned(v) for k, v in bi.items()}
    hq = pinned(w.q)
    res = sda.build_decode_host(hq, kv, w.attn_sink, w.softmax_scale, h["state_slot"],
                                h["swa_len"], h["swa_head"], h["comp_indptr"], h["comp_block"],
                                h["comp_slot"], win=w.win, k_per_block=w.k_per_block,
                                swa_pages=w.swa_pages, kv_scale=None if pool is None else pool.scale,
                                out=out, status=status, workspace=workspace, stream=stream)
    (stream if stream is not None else torch.cuda.current_stream()).synchronize()
    return res


@pytest.mark.parametrize("cfg", [0, 1], ids=[inputs.CONFIG_NAMES[c] for c in (0, 1)])
def test_host_buffers_equal_the_device_call(cfg):
    """Inputs read by kernels straight from page-locked host memory and the
    result written back to it (batches below the pipelining size): bit-
    identical to the device-buffer call."""
    w = inputs.config(cfg, device="cuda")
    bi = w.builder_inputs("cuda")
    out_h, st_h = host_call(w, bi)
    out_d, _, _, st_d = fused(w, bi)
    torch.cuda.synchronize()
    assert int(st_h.item()) == int(st_d.item())
    assert torch.equal(out_h.view(torch.int16), out_d.cpu().view(torch.int16))


def test_host_buffers_fp8_and_bad_descriptors():
    w = inputs.config(1, device="cuda")
    bi = {k: v.clone() for k, v in w.builder_inputs("cuda").items()}
    bi["swa_len"][2] = -1  # bit 1: token 2 decodes to +0
    pool = inputs.fp8_pool(w)
    out_h, st_h = host_call(w, bi, pool)
    out_d, _, _, st_d = fused(w, bi, pool)
    torch.cuda.synchronize()
    assert int(st_h.item()) == int(st_d.item()) == 1
    assert torch.equal(out_h.view(torch.int16), out_d.cpu().view(torch.int16))
    assert not out_h[2].view(torch.int16).any()


def test_host_buffers_graph_replay_and_rejects_pageable():
    w = inputs.config(1, device="cuda")
    bi = w.builder_inputs("cuda")
    h = {k: pinned(v) for k, v in bi.items()}
    q_h = pinned(w.q)
    out_h = torch.empty(w.q.shape, dtype=torch.bfloat16, pin_memory=True)
    st_h = torch.empty(1, dtype=torch.int32, pin_memory=True)
    cap = w.N * w.win + int(w.comp_block.size)
    ws = torch.empty(sda.build_decode_host_workspace_size(w.N, w.H, w.D, int(w.comp_block.size), cap),
                     dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    args = (q_h, w.unified_kv, w.attn_sink, w.softmax_scale, h["state_slot"], h["swa_len"],
            h["swa_head"], h["comp_indptr"], h["comp_block"], h["comp_slot"])
    kw = dict(win=w.win, k_per_block=w.k_per_block, swa_pages=w.swa_pages, capacity=cap,
              out=out_h, status=st_h, workspace=ws, stream=s)
    with torch.cuda.stream(s):
        sda.build_decode_host(*args, **kw)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sda.build_decode_host(*args, **kw)
    out_h.zero_()
    st_h.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    out_d, _, _, st_d = fused(w, bi)
    torch.cuda.synchronize()
    assert int(st_h.item()) == int(st_d.item()) == 0
    assert torch.equal(out_h.view(torch.int16), out_d.cpu().view(torch.int16))
    with pytest.raises(ValueError):  # pageable host memory
        sda.build_decode_host(w.q.cpu(), *args[1:], **{**kw, "stream": None})


# Host batches whose q is at least 8 MB move through the host link in token
# chunks (copy-engine transfers on the library's two streams, the decode chunk
# by chunk on the caller's stream).  Each chunk gets its own work plan, so the
# output is not bit-identical to the one-call device path; it is checked
# against the oracle on every token, and the status word against the device
# call (the lists are built for the whole batch at once).
PIPELINE_BYTES = 8 << 20


@pytest.mark.parametrize("cfg", [2, 3], ids=[inputs.CONFIG_NAMES[c] for c in (2, 3)])
def test_host_buffers_large_batch_pipelined(cfg):
    w = inputs.config(cfg, device="cuda")
    assert w.N * w.H * w.D * 2 >= PIPELINE_BYTES
    bi = w.builder_inputs("cuda")
    out_h, st_h = host_call(w, bi)
    _, _, _, st_d = fused(w, bi)
    torch.cuda.synchronize()
    assert int(st_h.item()) == int(st_d.item()) == 0
    parity.assert_parity(parity.compare(out_h.cuda(), parity.run_oracle(w)),
                         f"{inputs.CONFIG_NAMES[cfg]} host batch in chunks")


def test_host_buffers_large_batch_bad_descriptors_and_graph_replay():
    """A bad token in a chunked host batch decodes to +0 with its status bit;
    the chunked call replays from a CUDA graph (the library's copy streams
    fork from and join the captured stream) and gives the same bits twice."""
    w = inputs.config(2, device="cuda")
    bi = {k: v.clone() for k, v in w.builder_inputs("cuda").items()}
    lens = np.asarray(w.lengths)
    bad = int(next(t for t in range(w.N // 2, w.N) if lens[t] > 0))  # a listed token of the second chunk
    bi["swa_len"][bad] = -1         # bit 1: empty slice, output +0
    h = {k: pinned(v) for k, v in bi.items()}
    q_h = pinned(w.q)
    out_h = torch.empty(w.q.shape, dtype=torch.bfloat16, pin_memory=True)
    st_h = torch.empty(1, dtype=torch.int32, pin_memory=True)
    cap = w.N * w.win + int(w.comp_block.size)
    ws = torch.empty(sda.build_decode_host_workspace_size(w.N, w.H, w.D, int(w.comp_block.size), cap),
                     dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    args = (q_h, w.unified_kv, w.attn_sink, w.softmax_scale, h["state_slot"], h["swa_len"],
            h["swa_head"], h["comp_indptr"], h["comp_block"], h["comp_slot"])
    kw = dict(win=w.win, k_per_block=w.k_per_block, swa_pages=w.swa_pages, capacity=cap,
              out=out_h, status=st_h, workspace=ws, stream=s)
    with torch.cuda.stream(s):
        sda.build_decode_host(*args, **kw)
    s.synchronize()
    first = out_h.clone()
    assert int(st_h.item()) == 1
    assert not out_h[bad].view(torch.int16).any()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sda.build_decode_host(*args, **kw)
    out_h.zero_()
    st_h.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    assert int(st_h.item()) == 1
    assert torch.equal(out_h.view(torch.int16), first.view(torch.int16))
    tokens = [t for t in range(w.N) if t != bad]
    ref = parity.run_oracle(w, tokens=tokens)
    parity.assert_parity(parity.compare(out_h[tokens].cuda(), ref), "chunked host batch, bad token")


def test_fused_large_batch_equals_two_calls():
    """9000 tokens: the plan beside the flat scatter, whose kv_indptr search
    runs in global memory (no shared-memory copy above 8191 tokens)."""
    rng = np.random.default_rng(9000)
    lens = rng.integers(0, 130, 9000)
    lens[::97] = 0
    w = inputs.random_small(9000, 9000, 16, 512, 1 << 16, lens, device="cuda")
    bi = w.builder_inputs("cuda")
    assert_same(fused(w, bi), two_calls(w, bi))


@pytest.mark.parametrize("offset", [0, 1])
def test_fused_bad_entries_unaligned(offset):
    """Bad compressed entries in several tokens, with the entry arrays passed
    as views that start `offset` entries into larger arrays (not 16-byte
    aligned for offset 1): the fused call's entry check and per-token
    re-check give exactly the two calls' lists, status and output."""
    w = inputs.config(2, device="cuda")
    bi = {k: v.clone() for k, v in w.builder_inputs("cuda").items()}
    cp = bi["comp_indptr"].cpu().numpy()
    for t in (3, 40, 41, 200):
        if cp[t + 1] > cp[t]:
            bi["comp_slot"][int(cp[t + 1]) - 1] = w.k_per_block      # bit 8
    bi["comp_block"][int(cp[100])] = (w.total_pages - w.swa_pages) // w.k_per_block + 7  # bit 16
    for k in ("comp_block", "comp_slot"):
        pad = torch.zeros(offset, dtype=torch.int32, device="cuda")
        bi[k] = torch.cat([pad, bi[k]])[offset:]
    a, b = fused(w, bi), two_calls(w, bi)
    assert_same(a, b)
    assert int(a[3].item()) & 8
