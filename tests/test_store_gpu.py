"""q/kv RMSNorm + GPT-J RoPE + SWA ring store (sda_qk_norm_rope_swa_store and
its FP8-pool form) on the GPU against the fp64 oracle.

The kernel computes in fp32 and rounds once; the oracle gives the exact
value v of every element.  An element passes if it is the correctly rounded
(nearest-even bf16, or nearest-even E4M3 of v / scale) form of some value
within tol of v, tol = 2^-18 * m, with m = |v| outside the rotated dims and
the length of v's RoPE pair inside them (the fp32 error of the norm is below
~25 units of 2^-24 relative, and a rotation's error scales with its pair).
Where tol is below half a rounding step -- every element but the few rotated
ones much smaller than their pair -- that is the exact rounding, or its
neighbour when v lies within tol of a midpoint.  Inputs built so that every
fp32 step is exact must match the oracle's rounding bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import parity
import sink_sda_decode_gb300 as sda
from sink_sda_decode_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL_REL = 2.0 ** -18


def element_mag(val: np.ndarray, R: int) -> np.ndarray:
    """|v| outside the last R dims; the length of the (2i, 2i+1) pair inside."""
    mag = np.abs(val).copy()
    if R:
        D = val.shape[-1]
        a, b = val[..., D - R::2], val[..., D - R + 1::2]
        pair = np.sqrt(a * a + b * b)
        mag[..., D - R::2] = pair
        mag[..., D - R + 1::2] = pair
    return mag


def _bf16_value(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_band_ok(got_bits: np.ndarray, val: np.ndarray, R: int) -> np.ndarray:
    """got is a nearest-even bf16 rounding of some value in [v - tol, v + tol]:
    rounding is monotone, so exactly the bf16 values between the roundings of
    the two ends."""
    tol = TOL_REL * element_mag(val, R)
    got = _bf16_value(got_bits.view(np.uint16))
    lo = _bf16_value(oracle.bf16_rne(val - tol))
    hi = _bf16_value(oracle.bf16_rne(val + tol))
    return (lo <= got) & (got <= hi)


_E4M3 = []


def e4m3_table() -> np.ndarray:
    if not _E4M3:
        _E4M3.append(oracle.e4m3_values())
    return _E4M3[0]


def fp8_rows_ok(codes: np.ndarray, scale: np.ndarray, val: np.ndarray, R: int):
    """(scale_ok [rows], code_ok [rows, D]) for quantised rows of exact values:
    the scale is the oracle's (or its neighbour where max |v| lies within tol
    of a power-of-two boundary); each code is a nearest-even E4M3 rounding of
    some value in [(v - tol) / scale, (v + tol) / scale]."""
    amax = np.abs(val).max(axis=1)
    e_alt = [{oracle.fp8_scale_exponent(a * (1 - TOL_REL)), oracle.fp8_scale_exponent(a),
              oracle.fp8_scale_exponent(a * (1 + TOL_REL))} for a in amax]
    scale_ok = np.array([float(s) in {math.ldexp(1.0, e) for e in es}
                         for s, es in zip(scale, e_alt)])
    sc = scale.astype(np.float64)[:, None]
    tol = TOL_REL * element_mag(val, R)
    table = e4m3_table()
    got = table[codes]
    lo = table[oracle.e4m3_rne_array((val - tol) / sc)]
    hi = table[oracle.e4m3_rne_array((val + tol) / sc)]
    return scale_ok, (lo <= got) & (got <= hi)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def run_oracle(w, si, tokens=None):
    """Oracle on the given tokens (the op is independent per token)."""
    tok = np.arange(w.N) if tokens is None else np.asarray(tokens)
    q = w.q_bits()[tok]
    kv = host_bits(si.kv_new)[tok]
    return oracle.qk_norm_rope_store(q, kv, host_bits(si.q_norm_w), host_bits(si.kv_norm_w),
                                     si.cos_cache.cpu().numpy(), si.sin_cache.cpu().numpy(),
                                     si.positions.cpu().numpy()[tok],
                                     si.state_slot.cpu().numpy()[tok], si.eps, w.win, w.swa_pages)


def call_store(w, si, pool=None, fp8=None, q_out=None, q=None):
    return sda.qk_norm_rope_swa_store(
        w.q if q is None else q, si.kv_new, si.q_norm_w, si.kv_norm_w, si.cos_cache, si.sin_cache,
        si.positions, si.state_slot, eps=si.eps, win=w.win, swa_pages=w.swa_pages,
        unified_kv=pool, kv_fp8=None if fp8 is None else fp8.codes,
        kv_scale=None if fp8 is None else fp8.scale, q_out=q_out)


def check_q(q_out, ref, tok, R, what):
    got = host_bits(q_out)[tok]
    ok = bf16_band_ok(got, ref["q_val"], R)
    assert ok.all(), (what, "q", int((~ok).sum()), np.argwhere(~ok)[:5])


def sample(w, k, seed):
    if k is None:
        return np.arange(w.N)
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(w.N, min(k, w.N), replace=False))


CFGS = [(1, None), (2, None), (3, 96)]


@pytest.mark.parametrize("cfg,k", CFGS, ids=[inputs.CONFIG_NAMES[c] for c, _ in CFGS])
def test_store_bf16_workload(cfg, k):
    w = inputs.config(cfg, device="cuda")
    si = inputs.store_inputs(w)
    R = si.cos_cache.shape[1] * 2
    before = w.unified_kv.clone()
    q_out, status = call_store(w, si, pool=w.unified_kv)
    torch.cuda.synchronize()
    tok = sample(w, k, 500 + cfg)
    ref = run_oracle(w, si, tok)
    assert int(status.item()) == ref["status"] == 0
    check_q(q_out, ref, tok, R, inputs.CONFIG_NAMES[cfg])
    live = ref["slot"] >= 0
    rows = w.unified_kv[torch.from_numpy(ref["slot"][live]).cuda()]
    ok = bf16_band_ok(host_bits(rows), ref["kv_val"][live], R)
    assert ok.all(), ("kv rows", int((~ok).sum()))
    # nothing but the tokens' own ring slots changed (all tokens, not only the sample)
    changed = torch.nonzero((w.unified_kv != before).any(dim=1)).flatten().cpu().numpy()
    st = si.state_slot.cpu().numpy().astype(np.int64)
    pos = si.positions.cpu().numpy().astype(np.int64)
    expect = np.unique((st * w.win + pos % w.win)[st >= 0])
    assert np.isin(changed, expect).all()
    # padded tokens: q_out = +0
    pad = np.nonzero(st < 0)[0]
    if pad.size:
        assert not host_bits(q_out)[pad].any()


@pytest.mark.parametrize("cfg,k", CFGS, ids=[inputs.CONFIG_NAMES[c] for c, _ in CFGS])
def test_store_fp8_workload(cfg, k):
    w = inputs.config(cfg, device="cuda")
    si = inputs.store_inputs(w)
    R = si.cos_cache.shape[1] * 2
    pool = inputs.fp8_pool(w)
    codes0, scale0 = pool.codes.clone(), pool.scale.clone()
    q_out, status = call_store(w, si, fp8=pool)
    torch.cuda.synchronize()
    tok = sample(w, k, 600 + cfg)
    ref = run_oracle(w, si, tok)
    assert int(status.item()) == ref["status"] == 0
    check_q(q_out, ref, tok, R, inputs.CONFIG_NAMES[cfg] + " fp8")
    live = ref["slot"] >= 0
    sl = torch.from_numpy(ref["slot"][live]).cuda()
    scale_ok, code_ok = fp8_rows_ok(pool.codes[sl].cpu().numpy(), pool.scale[sl].cpu().numpy(),
                                    ref["kv_val"][live], R)
    assert scale_ok.all() and code_ok.all(), (int((~scale_ok).sum()), int((~code_ok).sum()))
    changed = torch.nonzero((pool.codes != codes0).any(dim=1) | (pool.scale != scale0))
    st = si.state_slot.cpu().numpy().astype(np.int64)
    pos = si.positions.cpu().numpy().astype(np.int64)
    expect = np.unique((st * w.win + pos % w.win)[st >= 0])
    assert np.isin(changed.flatten().cpu().numpy(), expect).all()


def exact_case(N, H, D, R, seed, max_pos=40):
    """Rows of +-1 and +-3 (3D/8 threes) have mean square exactly 4, so with
    eps = 0 the norm factor is exactly 1/2; bf16 weights make y = x * w / 2
    exact in fp32; cos / sin in {0, +-1} make the rotation exact.  What is left
    is the final rounding, which both sides must then take identically."""
    rng = np.random.default_rng(seed)

    def rows(n):
        mag = np.ones((n, D))
        for r in range(n):
            mag[r, rng.choice(D, 3 * D // 8, replace=False)] = 3.0
        return mag * rng.choice([-1.0, 1.0], (n, D))

    q = rows(N * H).reshape(N, H, D)
    kv = rows(N)
    qw = rng.uniform(0.5, 2.0, D)
    kw = rng.uniform(0.5, 2.0, D)
    k = rng.integers(0, 4, (max_pos, R // 2))
    cos = np.choose(k, [1.0, 0.0, -1.0, 0.0]).astype(np.float32)
    sin = np.choose(k, [0.0, 1.0, 0.0, -1.0]).astype(np.float32)
    pos = rng.integers(0, max_pos, N).astype(np.int32)
    return q, kv, qw, kw, cos, sin, pos


@pytest.mark.parametrize("D,R,H", [(512, 64, 16), (64, 64, 3), (1024, 8, 2), (2048, 512, 1),
                                   (136, 0, 5)])
def test_store_exact_inputs_bit_identical(D, R, H):
    N, win = 7, 16
    q, kv, qw, kw, cos, sin, pos = exact_case(N, H, D, R, seed=D + R + H, max_pos=40)
    state = np.arange(N, dtype=np.int32)[::-1].copy()
    swa_pages, P = N * win, N * win + 8
    dev = "cuda"
    bf = lambda a: torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).to(dev)
    it = lambda a: torch.from_numpy(np.asarray(a, np.int32)).to(dev)
    qt, kvt, qwt, kwt = bf(q), bf(kv), bf(qw), bf(kw)
    cst = torch.from_numpy(cos).to(dev)
    snt = torch.from_numpy(sin).to(dev)
    ref = oracle.qk_norm_rope_store(host_bits(qt), host_bits(kvt), host_bits(qwt), host_bits(kwt),
                                    cos, sin, pos, state, 0.0, win, swa_pages)
    assert ref["status"] == 0
    # the construction is exact in fp32: the values are fp32 numbers
    assert np.array_equal(ref["q_val"].astype(np.float32).astype(np.float64), ref["q_val"])
    pool = torch.zeros((P, D), dtype=torch.bfloat16, device=dev)
    q_out, st = sda.qk_norm_rope_swa_store(qt, kvt, qwt, kwt, cst, snt, it(pos), it(state), eps=0.0,
                                           win=win, swa_pages=swa_pages, unified_kv=pool)
    codes = torch.zeros((P, D), dtype=torch.uint8, device=dev)
    scale = torch.zeros(P, dtype=torch.float32, device=dev)
    q_out8, st8 = sda.qk_norm_rope_swa_store(qt, kvt, qwt, kwt, cst, snt, it(pos), it(state),
                                             eps=0.0, win=win, swa_pages=swa_pages, kv_fp8=codes,
                                             kv_scale=scale)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st8.item()) == 0
    want_q = oracle.bf16_rne(ref["q_val"])
    assert np.array_equal(host_bits(q_out), want_q)
    assert np.array_equal(host_bits(q_out8), want_q)
    slots = torch.from_numpy(ref["slot"]).to(dev)
    assert np.array_equal(host_bits(pool[slots]), oracle.bf16_rne(ref["kv_val"]))
    want_codes, want_scale = oracle.fp8_quantise_rows(ref["kv_val"])
    assert np.array_equal(codes[slots].cpu().numpy(), want_codes)
    assert np.array_equal(scale[slots].cpu().numpy(), want_scale)


def small_case(N, H, D, R, seed, max_pos=50):
    rng = np.random.default_rng(seed)
    dev = "cuda"
    bf = lambda a: torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).to(dev)
    q = bf(rng.standard_normal((N, H, D)) * 3.0)
    kv = bf(rng.standard_normal((N, D)) * 0.01)
    qw = bf(rng.uniform(0.5, 1.5, D))
    kw = bf(rng.uniform(0.5, 1.5, D))
    cos, sin = inputs.rope_caches(max_pos, R, device=dev)
    return q, kv, qw, kw, cos, sin


def test_store_edge_cases_and_status_bits():
    """Padded tokens, positions outside the caches (bit 1), ring slots past the
    SWA region (bit 2), a large eps, and q updated in place."""
    N, H, D, R, win = 6, 4, 512, 64, 8
    q, kv, qw, kw, cos, sin = small_case(N, H, D, R, seed=91)
    pos = torch.tensor([3, -1, 50, 17, 9, 0], dtype=torch.int32, device="cuda")
    state = torch.tensor([0, 1, 2, -1, 4, 3], dtype=torch.int32, device="cuda")
    swa_pages = 4 * win  # token 4's slot 4*8+1 = 33 is past it
    pool = torch.full((40, D), 7.0, dtype=torch.bfloat16, device="cuda")
    before = pool.clone()
    q_in = q.clone()
    eps = 0.5
    q_out, st = sda.qk_norm_rope_swa_store(q, kv, qw, kw, cos, sin, pos, state, eps=eps, win=win,
                                           swa_pages=swa_pages, unified_kv=pool, q_out=q)  # in place
    torch.cuda.synchronize()
    ref = oracle.qk_norm_rope_store(host_bits(q_in), host_bits(kv), host_bits(qw), host_bits(kw),
                                    cos.cpu().numpy(), sin.cpu().numpy(), pos.cpu().numpy(),
                                    state.cpu().numpy(), eps, win, swa_pages)
    assert ref["slot"].tolist() == [3, -1, -1, -1, -1, 24]
    assert int(st.item()) == ref["status"] == 3
    assert q_out.data_ptr() == q.data_ptr()
    assert bf16_band_ok(host_bits(q), ref["q_val"], R).all()
    assert not host_bits(q)[[1, 2, 3]].any()
    rows = pool[torch.tensor([3, 24], device="cuda")]
    assert bf16_band_ok(host_bits(rows), ref["kv_val"][[0, 5]], R).all()
    keep = torch.ones(40, dtype=torch.bool, device="cuda")
    keep[[3, 24]] = False
    assert torch.equal(pool[keep], before[keep])


@pytest.mark.parametrize("D,R", [(64, 0), (128, 128), (200, 40), (1024, 64), (2048, 2048)])
def test_store_other_shapes(D, R):
    N, H, win = 5, 3, 4
    q, kv, qw, kw, cos, sin = small_case(N, H, D, R, seed=D + R)
    pos = torch.tensor([0, 5, 49, 12, 33], dtype=torch.int32, device="cuda")
    state = torch.arange(N, dtype=torch.int32, device="cuda")
    codes = torch.zeros((N * win, D), dtype=torch.uint8, device="cuda")
    scale = torch.zeros(N * win, dtype=torch.float32, device="cuda")
    q_out, st = sda.qk_norm_rope_swa_store(q, kv, qw, kw, cos, sin, pos, state, eps=1e-6, win=win,
                                           swa_pages=N * win, kv_fp8=codes, kv_scale=scale)
    torch.cuda.synchronize()
    ref = oracle.qk_norm_rope_store(host_bits(q), host_bits(kv), host_bits(qw), host_bits(kw),
                                    cos.cpu().numpy(), sin.cpu().numpy(), pos.cpu().numpy(),
                                    state.cpu().numpy(), 1e-6, win, N * win)
    assert int(st.item()) == 0
    assert bf16_band_ok(host_bits(q_out), ref["q_val"], R).all()
    sl = torch.from_numpy(ref["slot"]).cuda()
    scale_ok, code_ok = fp8_rows_ok(codes[sl].cpu().numpy(), scale[sl].cpu().numpy(),
                                    ref["kv_val"], R)
    assert scale_ok.all() and code_ok.all()


def test_store_empty_batch():
    q, kv, qw, kw, cos, sin = small_case(1, 2, 64, 8, seed=3)
    pool = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    e = torch.zeros(0, dtype=torch.int32, device="cuda")
    q_out, st = sda.qk_norm_rope_swa_store(q[:0], kv[:0], qw, kw, cos, sin, e, e, eps=1e-6, win=4,
                                           swa_pages=8, unified_kv=pool)
    torch.cuda.synchronize()
    assert q_out.shape == (0, 2, 64) and int(st.item()) == 0 and not pool.any()


def test_store_rejects_bad_arguments():
    N, H, D, R = 2, 2, 64, 8
    q, kv, qw, kw, cos, sin = small_case(N, H, D, R, seed=4)
    pos = torch.zeros(N, dtype=torch.int32, device="cuda")
    st = torch.arange(N, dtype=torch.int32, device="cuda")
    pool = torch.zeros((16, D), dtype=torch.bfloat16, device="cuda")
    kw_args = dict(eps=1e-6, win=4, swa_pages=8, unified_kv=pool)
    with pytest.raises(RuntimeError):  # rope_dim = 6 is not a multiple of 8
        sda.qk_norm_rope_swa_store(q, kv, qw, kw, cos[:, :3].contiguous(), sin[:, :3].contiguous(),
                                   pos, st, **kw_args)
    with pytest.raises(RuntimeError):  # negative eps
        sda.qk_norm_rope_swa_store(q, kv, qw, kw, cos, sin, pos, st, **{**kw_args, "eps": -1.0})
    with pytest.raises(RuntimeError):  # swa_pages > total_pages
        sda.qk_norm_rope_swa_store(q, kv, qw, kw, cos, sin, pos, st, **{**kw_args, "swa_pages": 17})
    big = torch.zeros(2 * N * H * D + 8, dtype=torch.bfloat16, device="cuda")
    q_a = big[: N * H * D].view(N, H, D)
    q_a.copy_(q)
    with pytest.raises(RuntimeError):  # q_out partly overlaps q
        sda.qk_norm_rope_swa_store(q_a, kv, qw, kw, cos, sin, pos, st, **kw_args,
                                   q_out=big[8: 8 + N * H * D].view(N, H, D))
    with pytest.raises(RuntimeError):  # misaligned kv (offset of one element)
        kv_m = torch.zeros(N * D + 1, dtype=torch.bfloat16, device="cuda")[1:].view(N, D)
        sda.qk_norm_rope_swa_store(q, kv_m, qw, kw, cos, sin, pos, st, **kw_args)
    with pytest.raises(ValueError):  # both pools
        sda.qk_norm_rope_swa_store(q, kv, qw, kw, cos, sin, pos, st, eps=1e-6, win=4, swa_pages=8,
                                   unified_kv=pool, kv_fp8=torch.zeros((16, D), dtype=torch.uint8,
                                                                       device="cuda"),
                                   kv_scale=torch.zeros(16, device="cuda"))
    with pytest.raises(TypeError):
        sda.qk_norm_rope_swa_store(q.float(), kv, qw, kw, cos, sin, pos, st, **kw_args)


def test_store_graph_capture_replay():
    w = inputs.config(1, device="cuda")
    si = inputs.store_inputs(w)
    R = si.cos_cache.shape[1] * 2
    q_out = torch.empty_like(w.q)
    status = torch.empty(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    args = (w.q, si.kv_new, si.q_norm_w, si.kv_norm_w, si.cos_cache, si.sin_cache, si.positions,
            si.state_slot)
    kw = dict(eps=si.eps, win=w.win, swa_pages=w.swa_pages, unified_kv=w.unified_kv, q_out=q_out,
              status=status, stream=s)
    with torch.cuda.stream(s):
        sda.qk_norm_rope_swa_store(*args, **kw)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sda.qk_norm_rope_swa_store(*args, **kw)
    q_out.zero_()
    status.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    ref = run_oracle(w, si)
    assert int(status.item()) == 0
    check_q(q_out, ref, np.arange(w.N), R, "graph")


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
def test_store_build_decode_pipeline(fp8):
    """One decode step as the three calls run it: store the new rows, build
    the lists, attend.  The oracle runs the same chain on its own results:
    its stored rows (rounded as the pool stores them) replace the seeded
    pool's rows at the ring slots."""
    w = inputs.config(1, device="cuda")
    si = inputs.store_inputs(w)
    tok = sample(w, 24, 77)
    # the oracle's pool rows, taken before the GPU store touches the pool
    lists = [w.kv_indices[w.kv_indptr[t]:w.kv_indptr[t + 1]] for t in range(w.N)]
    need = np.unique(np.concatenate([lists[t] for t in tok]))
    pool = inputs.fp8_pool(w) if fp8 else None
    if fp8:
        codes_h = pool.codes[torch.from_numpy(need).cuda()].cpu().numpy()
        scale_h = pool.scale[torch.from_numpy(need).cuda()].cpu().numpy()
    else:
        rows_h = host_bits(w.unified_kv[torch.from_numpy(need).cuda()])
    # GPU: store -> build -> decode
    q_out, st = call_store(w, si, pool=None if fp8 else w.unified_kv, fp8=pool)
    b = w.builder_inputs("cuda")
    idx, ptr, bst = sda.build_indices(**b, win=w.win, k_per_block=w.k_per_block,
                                      swa_pages=w.swa_pages, total_pages=w.total_pages)
    if fp8:
        out = sda.decode_fp8(q_out, pool.codes, pool.scale, idx, ptr, w.attn_sink, w.softmax_scale)
    else:
        out = sda.decode(q_out, w.unified_kv, idx, ptr, w.attn_sink, w.softmax_scale)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(bst.item()) == 0
    # oracle: store -> build -> decode on the sampled tokens
    ref = run_oracle(w, si)
    o_idx, o_ptr, o_st = oracle.build_indices(w.state_slot, w.swa_len, w.swa_head, w.comp_indptr,
                                              w.comp_block, w.comp_slot, w.win, w.k_per_block,
                                              w.swa_pages, w.total_pages)
    assert o_st == 0
    live = ref["slot"] >= 0
    hit = np.isin(ref["slot"], need) & live
    where = np.searchsorted(need, ref["slot"][hit])
    if fp8:
        c, s = oracle.fp8_quantise_rows(ref["kv_val"][hit])
        codes_h[where], scale_h[where] = c, s
    else:
        rows_h[where] = oracle.bf16_rne(ref["kv_val"][hit])
    q_bits = oracle.bf16_rne(ref["q_val"])[tok]
    sub = [o_idx[o_ptr[t]:o_ptr[t + 1]] for t in tok]
    sub_ptr = np.zeros(len(tok) + 1, np.int32)
    sub_ptr[1:] = np.cumsum([len(x) for x in sub])
    sub_idx = np.searchsorted(need, np.concatenate(sub)).astype(np.int32)
    sink = w.attn_sink.cpu().numpy()
    if fp8:
        want = oracle.sda_decode_fp8(q_bits, codes_h, scale_h, sub_idx, sub_ptr, sink, w.softmax_scale)
    else:
        want = oracle.sda_decode(q_bits, rows_h, sub_idx, sub_ptr, sink, w.softmax_scale)
    got = out[torch.from_numpy(tok).cuda()]
    parity.assert_parity(parity.compare(got, want), "store+build+decode" + (" fp8" if fp8 else ""))
