"""Pins that tie the fp64 oracle to the pages and to mathematics (CPU only).

Each pin checks the oracle against something other than itself: a library
routine (torch's scaled-dot-product attention and softmax in float64), a
closed form, an invariant, or a hand-worked example of the slot formulas.
The functions take an oracle library handle so that the mutation tests can
run the same pins against deliberately broken builds of the oracle.

Source of the definitions: the docstring of paged_decode.py quoted on the
sglang PR 28392 summary page ("为 AMD V4 内核添加 ATOM 来源注释", section
"关键源码片段"): caller convention (unified_kv, kv_indices, kv_indptr,
attn_sink, softmax_scale), returns, numerics.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def random_case(rng, N, H, D, P, lens, dup=False, sink_sigma=1.0):
    q = bf16_bits(rng.standard_normal((N, H, D)))
    kv = bf16_bits(rng.standard_normal((P, D)))
    lists = [rng.integers(0, P, L) if dup else rng.choice(P, L, replace=False) for L in lens]
    ptr = np.zeros(N + 1, np.int32)
    ptr[1:] = np.cumsum([len(x) for x in lists])
    idx = np.concatenate(lists).astype(np.int32) if ptr[-1] else np.zeros(0, np.int32)
    sink = (rng.standard_normal(H) * sink_sigma).astype(np.float32)
    return q, kv, idx, ptr, sink


def sdpa_reference(q, kv, idx, ptr, sink, scale):
    """Attention with a sink written as ordinary softmax attention (torch SDPA,
    float64) over the listed keys plus one extra all-zero key/value row whose
    logit is biased by attn_sink[h] through an additive mask."""
    N, H, D = q.shape
    qf = torch.from_numpy(bits_to_f64(q))
    kvf = torch.from_numpy(bits_to_f64(kv))
    sink_t = torch.from_numpy(np.asarray(sink, np.float64))
    out = torch.zeros((N, H, D), dtype=torch.float64)
    for t in range(N):
        rows = kvf[torch.from_numpy(idx[ptr[t]:ptr[t + 1]].astype(np.int64))]
        L = rows.shape[0]
        keys = torch.cat([rows, torch.zeros(1, D, dtype=torch.float64)], 0)
        keys = keys.unsqueeze(0).expand(H, L + 1, D)
        mask = torch.zeros(H, 1, L + 1, dtype=torch.float64)
        mask[:, 0, L] = sink_t
        out[t] = F.scaled_dot_product_attention(qf[t].unsqueeze(1), keys, keys, attn_mask=mask,
                                                scale=float(np.float32(scale)))[:, 0, :]
    return out.numpy()


def logits(q, kv, idx, ptr, t, h, scale):
    rows = bits_to_f64(kv[idx[ptr[t]:ptr[t + 1]]])
    return float(np.float32(scale)) * rows @ bits_to_f64(q[t, h])


# ----------------------------------------------------------------------------- pins
def pin_sdpa(lib):
    """Random small cases (empty, short and full-tile lists) vs torch SDPA fp64."""
    rng = np.random.default_rng(11)
    for N, H, D, P in [(1, 1, 8, 50), (4, 3, 16, 300), (6, 8, 64, 4096), (3, 2, 128, 900)]:
        lens = rng.integers(0, 70, N)
        lens[0] = 0
        q, kv, idx, ptr, sink = random_case(rng, N, H, D, P, lens)
        scale = rng.uniform(0.05, 0.5)
        got = oracle.sda_decode(q, kv, idx, ptr, sink, scale, lib=lib)
        ref = sdpa_reference(q, kv, idx, ptr, sink, scale)
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def pin_sink_minus_inf_is_softmax(lib):
    """attn_sink -> -inf reduces to ordinary softmax attention (torch.softmax)."""
    rng = np.random.default_rng(12)
    N, H, D, P = 3, 4, 32, 500
    q, kv, idx, ptr, _ = random_case(rng, N, H, D, P, [5, 40, 1])
    sink = np.full(H, -np.inf, np.float32)
    scale = 0.2
    got = oracle.sda_decode(q, kv, idx, ptr, sink, scale, lib=lib)
    for t in range(N):
        v = torch.from_numpy(bits_to_f64(kv[idx[ptr[t]:ptr[t + 1]]]))
        for h in range(H):
            x = torch.from_numpy(logits(q, kv, idx, ptr, t, h, scale))
            ref = torch.softmax(x, 0) @ v
            np.testing.assert_allclose(got[t, h], ref.numpy(), rtol=0, atol=1e-12)


def pin_single_slot(lib):
    """One slot: out = v * e^x / (e^x + e^sink) = v * logistic(x - sink)."""
    rng = np.random.default_rng(13)
    N, H, D, P = 5, 6, 64, 256
    q, kv, idx, ptr, sink = random_case(rng, N, H, D, P, [1] * N, sink_sigma=2.0)
    scale = 0.125
    got = oracle.sda_decode(q, kv, idx, ptr, sink, scale, lib=lib)
    for t in range(N):
        v = bits_to_f64(kv[idx[ptr[t]]])
        for h in range(H):
            x = logits(q, kv, idx, ptr, t, h, scale)[0]
            w = 1.0 / (1.0 + math.exp(float(sink[h]) - x))
            np.testing.assert_allclose(got[t, h], w * v, rtol=1e-13, atol=1e-14)


def pin_duplicate_adds_ln2(lib):
    """A slot listed twice weighs like one occurrence with its logit + ln 2."""
    rng = np.random.default_rng(14)
    D, P, H = 32, 100, 3
    q = bf16_bits(rng.standard_normal((1, H, D)))
    kv = bf16_bits(rng.standard_normal((P, D)))
    sink = rng.standard_normal(H).astype(np.float32)
    s = 17
    idx = np.array([s, s], np.int32)
    ptr = np.array([0, 2], np.int32)
    scale = 0.3
    got = oracle.sda_decode(q, kv, idx, ptr, sink, scale, lib=lib)
    v = bits_to_f64(kv[s])
    for h in range(H):
        x = logits(q, kv, idx[:1], np.array([0, 1], np.int32), 0, h, scale)[0]
        w = 1.0 / (1.0 + math.exp(float(sink[h]) - (x + math.log(2.0))))
        np.testing.assert_allclose(got[0, h], w * v, rtol=1e-13, atol=1e-14)


def pin_zero_length(lib):
    """Empty slice -> exactly +0.0, with a finite sink and with sink = -inf."""
    rng = np.random.default_rng(15)
    q, kv, idx, ptr, sink = random_case(rng, 3, 4, 16, 64, [0, 3, 0])
    sink[1] = -np.inf
    out = oracle.sda_decode(q, kv, idx, ptr, sink, 0.25, lib=lib)
    assert np.all(out[0] == 0.0) and np.all(out[2] == 0.0)
    assert not np.signbit(out[0]).any()


def pin_permutation(lib):
    """Order within a token's list does not change the result."""
    rng = np.random.default_rng(16)
    q, kv, idx, ptr, sink = random_case(rng, 2, 4, 64, 2000, [200, 37])
    a = oracle.sda_decode(q, kv, idx, ptr, sink, 0.125, lib=lib)
    idx2 = idx.copy()
    for t in range(2):
        idx2[ptr[t]:ptr[t + 1]] = rng.permutation(idx[ptr[t]:ptr[t + 1]])
    b = oracle.sda_decode(q, kv, idx2, ptr, sink, 0.125, lib=lib)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def pin_sink_factor(lib):
    """out(sink) = out(-inf) * Zk / (Zk + e^sink), Zk = sum_j e^{x_j}."""
    rng = np.random.default_rng(17)
    q, kv, idx, ptr, sink = random_case(rng, 2, 3, 32, 400, [9, 50])
    scale = 0.2
    with_sink = oracle.sda_decode(q, kv, idx, ptr, sink, scale, lib=lib)
    no_sink = oracle.sda_decode(q, kv, idx, ptr, np.full(3, -np.inf, np.float32), scale, lib=lib)
    for t in range(2):
        for h in range(3):
            x = logits(q, kv, idx, ptr, t, h, scale)
            zk = np.exp(x).sum()
            f = zk / (zk + math.exp(float(sink[h])))
            np.testing.assert_allclose(with_sink[t, h], no_sink[t, h] * f, rtol=1e-12, atol=1e-14)


def pin_scale_zero(lib):
    """softmax_scale = 0: every logit is 0, out = sum_j v_j / (L + e^sink)."""
    rng = np.random.default_rng(18)
    q, kv, idx, ptr, sink = random_case(rng, 2, 2, 16, 300, [4, 33])
    got = oracle.sda_decode(q, kv, idx, ptr, sink, 0.0, lib=lib)
    for t in range(2):
        v = bits_to_f64(kv[idx[ptr[t]:ptr[t + 1]]])
        L = v.shape[0]
        for h in range(2):
            ref = v.sum(0) / (L + math.exp(float(sink[h])))
            np.testing.assert_allclose(got[t, h], ref, rtol=1e-13, atol=1e-14)


def pin_convexity(lib):
    """Weights are non-negative and sum to < 1: |out| <= max_j |kv[S_j, d]|."""
    rng = np.random.default_rng(19)
    q, kv, idx, ptr, sink = random_case(rng, 4, 4, 64, 3000, [1, 10, 100, 640])
    got = oracle.sda_decode(q, kv, idx, ptr, sink, 1 / 8, lib=lib)
    for t in range(4):
        bound = np.abs(bits_to_f64(kv[idx[ptr[t]:ptr[t + 1]]])).max(0)
        assert np.all(np.abs(got[t]) <= bound[None, :] + 1e-12)


def pin_hard_attention_limit(lib):
    """Huge scale: the softmax becomes an argmax; with sink -inf out -> v_argmax."""
    rng = np.random.default_rng(20)
    q, kv, idx, ptr, _ = random_case(rng, 1, 2, 16, 200, [12])
    sink = np.full(2, -np.inf, np.float32)
    got = oracle.sda_decode(q, kv, idx, ptr, sink, 1e4, lib=lib)
    for h in range(2):
        x = logits(q, kv, idx, ptr, 0, h, 1e4)
        j = int(np.argmax(x))
        np.testing.assert_allclose(got[0, h], bits_to_f64(kv[idx[j]]), rtol=0, atol=1e-12)


def pin_sink_plus_inf(lib):
    """sink = +inf absorbs all the mass (reading): out = 0."""
    rng = np.random.default_rng(21)
    q, kv, idx, ptr, sink = random_case(rng, 2, 2, 16, 100, [3, 0])
    sink[:] = np.inf
    assert np.all(oracle.sda_decode(q, kv, idx, ptr, sink, 0.5, lib=lib) == 0.0)


def pin_token_subset(lib):
    """Evaluating a subset of tokens gives exactly the same rows."""
    rng = np.random.default_rng(22)
    q, kv, idx, ptr, sink = random_case(rng, 5, 2, 16, 100, [3, 0, 7, 1, 9])
    full = oracle.sda_decode(q, kv, idx, ptr, sink, 0.5, lib=lib)
    sub = oracle.sda_decode(q, kv, idx, ptr, sink, 0.5, tokens=[4, 0, 2], lib=lib)
    assert np.array_equal(sub, full[[4, 0, 2]])


def read_golden_builder():
    vals = {}
    with open(os.path.join(GOLDEN, "build_indices_example.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = line.split(":", 1)
            vals[k.strip()] = [int(x) for x in v.split()]
    return vals


def pin_builder_golden(lib):
    """Hand-worked example of the two slot formulas (golden fixture)."""
    g = read_golden_builder()
    idx, ptr, st = oracle.build_indices(
        g["state_slot"], g["swa_len"], g["swa_head"], g["comp_indptr"], g["comp_block"],
        g["comp_slot"], g["win"][0], g["k_per_block"][0], g["swa_pages"][0], g["total_pages"][0],
        lib=lib)
    assert idx.tolist() == g["kv_indices"], (idx.tolist(), g["kv_indices"])
    assert ptr.tolist() == g["kv_indptr"]
    assert st == g["status"][0]


def pin_builder_ring_closed_form(lib):
    """A full ring with newest entry at `head` lists the state's win slots, oldest
    first: state*win + (head+1), ..., state*win + head (mod win)."""
    win, N = 8, 5
    heads = np.array([0, 3, 7, 5, 1], np.int32)
    idx, ptr, st = oracle.build_indices(np.arange(N), np.full(N, win), heads, np.zeros(N + 1),
                                        [], [], win, 4, N * win, N * win, lib=lib)
    assert st == 0 and ptr.tolist() == [0, 8, 16, 24, 32, 40]
    for t in range(N):
        expect = [t * win + (heads[t] + 1 + j) % win for j in range(win)]
        assert idx[ptr[t]:ptr[t + 1]].tolist() == expect


def pin_builder_capacity(lib):
    """Over-capacity output: status bit 32 and every slice empty."""
    idx, ptr, st = oracle.build_indices([0, 1], [2, 2], [1, 1], [0, 0, 0], [], [], 4, 4, 8, 8,
                                        capacity=3, lib=lib)
    assert st == 32 and ptr.tolist() == [0, 0, 0] and idx.size == 0


def pin_builder_comp_range(lib):
    """A compressed range that ends past the last entry: that token is empty
    with status bit 4, the token before it is unaffected (worked by hand:
    t0 = ring slot 0*4 + 0 and compressed 8 + 0*4 + 2)."""
    idx, ptr, st = oracle.build_indices([0, 1], [1, 1], [0, 0], [0, 1, 3], [0], [2], 4, 4, 8, 16,
                                        lib=lib)
    assert st == 4 and ptr.tolist() == [0, 2, 2] and idx.tolist() == [0, 10]


def pin_validate(lib):
    """Validation flags: decreasing indptr, indptr out of range, bad slots (counted)."""
    assert oracle.validate_indices([0, 1, 2], [0, 1, 3], 3, lib=lib) == (0, 0)
    assert oracle.validate_indices([0, 5, 2, -1], [0, 2, 4], 3, lib=lib) == (4, 2)
    assert oracle.validate_indices([0, 1], [0, 2, 1], 3, lib=lib) == (1, 0)
    assert oracle.validate_indices([0, 1], [0, 3], 3, lib=lib) == (2, 0)
    assert oracle.validate_indices([2, 3], [0, 2], 3, lib=lib) == (4, 1)  # slot == total_pages


# ----------------------------------------------------------------------------- FP8 pool
def pin_e4m3_table(lib):
    """All 256 E4M3 codes decode as torch's float8_e4m3fn conversion does (a
    library routine of the same format): the finite values exactly, NaN at
    S.1111.111."""
    got = oracle.e4m3_values(lib)
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def fp8_case(rng, N, H, D, P, lens):
    """Random finite E4M3 codes, power-of-two row scales, and the bf16 bits of
    the exactly dequantised pool (computed with torch, not with the oracle)."""
    codes = rng.integers(0, 256, (P, D)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    scale = np.ldexp(1.0, rng.integers(-6, 4, P)).astype(np.float32)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32) * torch.from_numpy(scale)[:, None]
    kv_bits = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert torch.equal(vals.to(torch.bfloat16).to(torch.float32), vals)  # exact in bf16
    q, _, idx, ptr, sink = random_case(rng, N, H, D, P, lens)
    return q, codes, scale, kv_bits, idx, ptr, sink


def pin_fp8_equals_bf16_pool(lib):
    """On a pool whose dequantised values are exact in bf16, the FP8 entry
    point equals the bf16 one (whose own pins tie it to the definition)."""
    rng = np.random.default_rng(41)
    q, codes, scale, kv_bits, idx, ptr, sink = fp8_case(rng, 4, 3, 16, 40, [0, 1, 7, 20])
    a = oracle.sda_decode_fp8(q, codes, scale, idx, ptr, sink, 0.25, lib=lib)
    b = oracle.sda_decode(q, kv_bits, idx, ptr, sink, 0.25, lib=lib)
    assert np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(b)))


def pin_fp8_zero_scale_row(lib):
    """A row with scale 0 is an all-zero key and value: its logit is 0, it
    adds e^0 to the denominator and nothing to the output (closed form with
    one ordinary slot beside it)."""
    D = 8
    codes = np.full((2, D), 0x38, np.uint8)  # e4m3 1.0 everywhere
    scale = np.array([0.5, 0.0], np.float32)
    q = bf16_bits(np.full((1, 1, D), 0.25))
    out = oracle.sda_decode_fp8(q, codes, scale, [0, 1], [0, 2], [0.375], 1.0, lib=lib)
    x = 0.25 * 0.5 * D
    want = math.exp(x) * 0.5 / (math.exp(0.375) + math.exp(x) + 1.0)
    assert np.allclose(out[0, 0], want, rtol=0, atol=1e-14)


FP8_PINS = [pin_e4m3_table, pin_fp8_equals_bf16_pool, pin_fp8_zero_scale_row]


# ----------------------------------------------------------------------------- q/kv norm + RoPE + store
# Source: the sglang PR 25898 summary page ("修复 DSV4 在 AMD GPU 上的运行时崩溃与
# JIT 不兼容"), sections "关键文件" / "关键符号" (fused_qk_norm_rope_store.py:
# Q per-head RMSNorm, KV RMSNorm, GPT-J RoPE, FP8 quantisation, paged SWA store;
# cos_cache / sin_cache in "实现拆解" item 2) and the SWA slot formula
# state_slot * win + ring of the paged_decode.py docstring (PR 28392 page).
def store_case(rng, N, H, D, R, max_pos=64, sigma=1.0):
    q = bf16_bits(rng.standard_normal((N, H, D)) * sigma)
    kv = bf16_bits(rng.standard_normal((N, D)) * sigma)
    qw = bf16_bits(rng.uniform(0.5, 1.5, D))
    kw = bf16_bits(rng.uniform(0.5, 1.5, D))
    ang = rng.uniform(-math.pi, math.pi, (max_pos, R // 2))
    cos = np.cos(ang).astype(np.float32)
    sin = np.sin(ang).astype(np.float32)
    pos = rng.integers(0, max_pos, N).astype(np.int32)
    return q, kv, qw, kw, cos, sin, pos


def pin_store_matches_torch(lib):
    """torch's RMSNorm (F.rms_norm, float64) followed by RoPE written as the
    complex product (y_d + i y_{d+1}) * (cos + i sin) of each adjacent pair of
    the last R dims: a library routine and a different formulation of the
    same rotation."""
    rng = np.random.default_rng(81)
    N, H, D, R = 5, 3, 32, 8
    q, kv, qw, kw, cos, sin, pos = store_case(rng, N, H, D, R)
    eps = 0.75  # large, so that a dropped eps shows
    ss = np.arange(N, dtype=np.int32)
    res = oracle.qk_norm_rope_store(q, kv, qw, kw, cos, sin, pos, ss, eps, 16, 1 << 20, lib=lib)
    assert res["status"] == 0

    def torch_ref(x_bits, w_bits):
        x = torch.from_numpy(bits_to_f64(x_bits))
        w = torch.from_numpy(bits_to_f64(w_bits))
        y = F.rms_norm(x, (D,), w, eps)
        rot = torch.view_as_complex(y[..., D - R:].reshape(*y.shape[:-1], R // 2, 2).contiguous())
        p = torch.from_numpy(pos.astype(np.int64))
        c = torch.from_numpy(cos.astype(np.float64))[p]
        s = torch.from_numpy(sin.astype(np.float64))[p]
        if y.dim() == 3:
            c, s = c[:, None, :], s[:, None, :]
        rot = torch.view_as_real(rot * torch.complex(c, s)).reshape(*y.shape[:-1], R)
        return torch.cat([y[..., :D - R], rot], -1).numpy()

    assert np.allclose(res["q_val"], torch_ref(q, qw), rtol=0, atol=1e-13)
    assert np.allclose(res["kv_val"], torch_ref(kv, kw), rtol=0, atol=1e-13)


def pin_store_closed_forms(lib):
    """eps = 0: a constant row c normalises to sign(c) * w; a row with one
    non-zero element x_0 to sqrt(D) * sign(x_0) * w_0 there; a quarter turn
    (cos 0, sin 1) maps the pair (a, b) to (-b, a); R = 0 leaves the norm."""
    D, R = 16, 4
    w = bf16_bits(np.linspace(0.5, 2.0, D))
    wf = bits_to_f64(w)
    q = bf16_bits(np.stack([np.full(D, -3.0), np.eye(D)[0] * 5.0])[None])      # N=1, H=2
    kv = bf16_bits(np.full((1, D), 0.125))
    cos = np.zeros((1, R // 2), np.float32)
    sin = np.ones((1, R // 2), np.float32)
    res = oracle.qk_norm_rope_store(q, kv, w, w, cos, sin, [0], [0], 0.0, 4, 4, lib=lib)
    quarter = lambda y: np.concatenate([y[:D - R], np.stack([-y[D - R + 1::2], y[D - R::2]], 1).ravel()])
    assert np.array_equal(res["q_val"][0, 0], quarter(-wf))
    one_hot = np.zeros(D)
    one_hot[0] = math.sqrt(D) * wf[0]
    assert np.allclose(res["q_val"][0, 1], quarter(one_hot), rtol=1e-15, atol=0)
    assert np.array_equal(res["kv_val"][0], quarter(wf))
    res0 = oracle.qk_norm_rope_store(q, kv, w, w, np.zeros((1, 0), np.float32),
                                     np.zeros((1, 0), np.float32), [0], [0], 0.0, 4, 4, lib=lib)
    assert np.array_equal(res0["kv_val"][0], wf)


def pin_store_rotation_invariants(lib):
    """Rotating by an angle and then by its negative restores the row; each
    pair's length is kept; rotation at position p uses row p of the caches."""
    rng = np.random.default_rng(82)
    N, H, D, R = 4, 2, 16, 8
    q, kv, qw, kw, cos, sin, pos = store_case(rng, N, H, D, R, max_pos=8)
    plain = oracle.qk_norm_rope_store(q, kv, qw, kw, np.ones_like(cos), np.zeros_like(sin),
                                      pos, np.arange(N), 1e-6, 8, 64, lib=lib)
    rot = oracle.qk_norm_rope_store(q, kv, qw, kw, cos, sin, pos, np.arange(N), 1e-6, 8, 64, lib=lib)
    y0, y1 = plain["q_val"][..., D - R:], rot["q_val"][..., D - R:]
    n0 = y0[..., 0::2] ** 2 + y0[..., 1::2] ** 2
    n1 = y1[..., 0::2] ** 2 + y1[..., 1::2] ** 2
    c = cos[pos].astype(np.float64)[:, None, :]
    s = sin[pos].astype(np.float64)[:, None, :]
    assert np.allclose(n1, n0 * (c * c + s * s), rtol=1e-12, atol=0)  # fp32 caches: c^2+s^2 ~ 1
    assert np.array_equal(plain["q_val"][..., :D - R], rot["q_val"][..., :D - R])
    back_a = y1[..., 0::2] * c + y1[..., 1::2] * s
    back_b = y1[..., 1::2] * c - y1[..., 0::2] * s
    assert np.allclose(back_a, y0[..., 0::2] * (c * c + s * s), rtol=1e-12, atol=1e-12)
    assert np.allclose(back_b, y0[..., 1::2] * (c * c + s * s), rtol=1e-12, atol=1e-12)


def pin_store_slots(lib):
    """Ring slot = state_slot * win + pos mod win (worked by hand); padded
    tokens store nothing and give q = 0; a position outside the caches or a
    slot outside the SWA region raises its status bit."""
    D, R = 8, 2
    rng = np.random.default_rng(83)
    q, kv, qw, kw, cos, sin, _ = store_case(rng, 6, 1, D, R, max_pos=300)
    pos = [0, 129, 255, 7, 300, 1]
    ss = [0, 2, 1, -1, 0, 5]
    res = oracle.qk_norm_rope_store(q, kv, qw, kw, cos, sin, pos, ss, 1e-6, 128, 5 * 128, lib=lib)
    # token 0: 0*128 + 0; token 1: 2*128 + 1; token 2: 128 + 127; 3 padded; 4 pos out of range;
    # token 5: 5*128 + 1 = 641 >= 640 -> not stored
    assert res["slot"].tolist() == [0, 257, 255, -1, -1, -1]
    assert res["status"] == 3
    assert not res["q_val"][3].any() and not res["q_val"][4].any() and not res["kv_val"][4].any()
    assert res["q_val"][5].any() and res["kv_val"][5].any()


def pin_bf16_rne(lib):
    """Round to nearest even bf16: equal to torch's float32 -> bfloat16
    conversion on values exact in fp32 (no double rounding possible there),
    and correct on hand cases where rounding through fp32 would not be."""
    rng = np.random.default_rng(84)
    v = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-40, 38, 4000),
                        np.float32(1.0) + np.arange(-64, 64) * np.float32(2.0 ** -9)]).astype(np.float32)
    v = v[np.isfinite(v)]
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_rne(v.astype(np.float64), lib=lib), want)
    hand = [(1.0 + 2.0 ** -8, 0x3F80), (1.0 + 3 * 2.0 ** -8, 0x3F82),
            (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81), (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
            (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000), (3.0 * 2.0 ** -134, 0x0002),
            (0.0, 0x0000), (-0.0, 0x8000), (1e39, 0x7F80), (-3.0, 0xC040)]
    got = oracle.bf16_rne([v for v, _ in hand], lib=lib)
    assert got.tolist() == [b for _, b in hand]


def pin_e4m3_rne(lib):
    """E4M3 rounding: every code's value maps back to that code, and a dense
    sweep of fp32 values (midpoints included) equals torch's float8_e4m3fn
    conversion after clamping to +-448; hand cases for ties and saturation."""
    vals = oracle.e4m3_values(lib)
    for c in range(256):
        if not np.isnan(vals[c]) and c != 0x80:
            assert oracle.e4m3_rne(vals[c], lib=lib) == c
    fin = np.sort(np.unique(vals[~np.isnan(vals)]))
    mids = (fin[1:] + fin[:-1]) / 2
    rng = np.random.default_rng(85)
    sweep = np.concatenate([fin, mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf),
                            rng.uniform(-500, 500, 3000), rng.standard_normal(3000) * 1e-2]).astype(np.float32)
    want = torch.from_numpy(sweep).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_rne(float(x), lib=lib) for x in sweep], np.uint8)
    assert np.array_equal(oracle.e4m3_rne_array(sweep.astype(np.float64), lib=lib), got)
    zero = sweep == 0  # the sign of a zero is kept by both; compare magnitudes there
    assert np.array_equal(got[~zero], want[~zero]) and np.all((got[zero] & 0x7F) == 0)
    # 17 = 1.0625 * 2^4: exponent field 11, mantissa tie 0.5 -> even 0: 0x58
    hand = [(2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (470.0, 0x7E), (-1e9, 0xFE), (1.0, 0x38),
            (1.0625, 0x38), (1.1875, 0x3A), (17.0, 0x58), (2.0 ** -9, 0x01), (-0.0, 0x80)]
    assert [oracle.e4m3_rne(v, lib=lib) for v, _ in hand] == [c for _, c in hand]


def pin_fp8_scale(lib):
    """Row scale 2^e, e the least integer with 448 * 2^e >= amax (hand cases at
    and around the powers of two), and quantised rows that dequantise to
    within half a code step of every value, with the largest at |code| > 224."""
    hand = {0.0: 0, 448.0: 0, 448.0 * (1 + 2.0 ** -40): 1, 1.0: -8, 1.75: -8, 1.7500001: -7,
            224.0: -1, 3.5: -7, 448.0 * 2.0 ** -130: -126}
    assert [oracle.fp8_scale_exponent(a, lib=lib) for a in hand] == list(hand.values())
    rng = np.random.default_rng(86)
    y = rng.standard_normal((64, 32)) * 10.0 ** rng.integers(-3, 4, (64, 1))
    y[3] = 0.0
    codes, scale = oracle.fp8_quantise_rows(y, lib=lib)
    assert scale[3] == 1.0 and not (codes[3] & 0x7F).any()
    table = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    deq = table[codes] * scale[:, None]
    for r in range(64):
        if r == 3:
            continue
        amax = np.abs(y[r]).max()
        assert 448.0 * scale[r] >= amax > 224.0 * scale[r]
        x = y[r] / scale[r]
        step = np.where(np.abs(x) < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(x), 1e-300))) - 3))
        assert np.all(np.abs(deq[r] - y[r]) <= 0.5 * step * scale[r] * (1 + 1e-12))


# ----------------------------------------------------------------------------- top-k -> slot lists
# Source: the sglang attention tag page, entry "DSV4.1 新增索引器内核，重做 Top-K v2
# 分派" (NaN padding below a legitimate -inf; a separate page-table transform),
# and the compressed-slot formula block_id * K_PER_BLOCK + slot_in_block of the
# paged_decode.py docstring (PR 28392 page).
def topk_numpy(scores, lengths, block_table, k, kpb):
    """The same selection with numpy's lexsort: non-NaN before NaN, then
    larger score (so -0 == +0), then smaller position; kept positions in
    increasing order, mapped through the block table."""
    ptr, blks, slots = [0], [], []
    S = scores.shape[1]
    for t in range(scores.shape[0]):
        n = int(lengths[t]) if 0 <= lengths[t] <= S else 0
        s = scores[t, :n].astype(np.float64)
        nan = np.isnan(s)
        order = np.lexsort((np.arange(n), -np.where(nan, 0.0, s), nan))
        keep = np.sort(order[:min(k, n)])
        blks += [int(block_table[t, p // kpb]) for p in keep]
        slots += [int(p % kpb) for p in keep]
        ptr.append(ptr[-1] + len(keep))
    return np.array(ptr), np.array(blks, np.int64), np.array(slots, np.int64)


def topk_case(rng, N, S, lens, kpb, tie_values=None):
    if tie_values is None:
        scores = rng.standard_normal((N, S)).astype(np.float32)
    else:
        scores = rng.choice(np.asarray(tie_values, np.float32), (N, S))
    B = -(-S // kpb)
    bt = rng.integers(0, 1000, (N, B)).astype(np.int32)
    return scores, np.asarray(lens, np.int32), bt


def pin_topk_matches_lexsort(lib):
    """Random scores, heavy ties (+-0, -inf, NaN among few values), ragged
    lengths around k: equal to numpy's lexsort formulation."""
    rng = np.random.default_rng(87)
    for ties in (None, [1.0, 0.0, -0.0, -np.inf, np.nan, 2.5, -1.0]):
        for k in (1, 5, 16):
            scores, lens, bt = topk_case(rng, 7, 40, [0, 1, 5, 16, 17, 40, 33], 8, ties)
            ptr, blk, slot, st = oracle.topk_slots(scores, lens, bt, k, 8, lib=lib)
            want = topk_numpy(scores, lens, bt, k, 8)
            assert np.array_equal(ptr, want[0]) and np.array_equal(blk, want[1])
            assert np.array_equal(slot, want[2])
            assert st == (8 if ties is not None and np.isnan(scores).any() and
                          any(np.isnan(scores[t, :lens[t]]).any() for t in range(7)) else 0)


def pin_topk_closed_forms(lib):
    """k >= n keeps every position; constant scores keep the first k; rising
    scores keep the last k; a worked example with ties, -0, -inf and NaN; bad
    lengths and negative block ids raise their status bits."""
    bt = np.array([[7, 9, 11]], np.int32)
    s = np.arange(12, dtype=np.float32)[None]
    assert oracle.topk_slots(s, [12], bt, 20, 4, lib=lib)[2].tolist() == [0, 1, 2, 3] * 3
    const = np.full((1, 12), 0.5, np.float32)
    ptr, blk, slot, _ = oracle.topk_slots(const, [12], bt, 5, 4, lib=lib)
    assert ptr.tolist() == [0, 5] and blk.tolist() == [7, 7, 7, 7, 9] and slot.tolist() == [0, 1, 2, 3, 0]
    ptr, blk, slot, _ = oracle.topk_slots(s, [12], bt, 3, 4, lib=lib)
    assert blk.tolist() == [11, 11, 11] and slot.tolist() == [1, 2, 3]
    # scores 0.5, 2, -inf, 2, NaN, 1, 0, -0 (block size 4, blocks 7 and 9): the
    # best five are p1, p3 (2.0), p5 (1.0), p0 (0.5) and p6 (0 ties -0, p6 first)
    ex = np.array([[0.5, 2.0, -np.inf, 2.0, np.nan, 1.0, 0.0, -0.0]], np.float32)
    bt2 = np.array([[7, 9]], np.int32)
    ptr, blk, slot, st = oracle.topk_slots(ex, [8], bt2, 5, 4, lib=lib)
    assert blk.tolist() == [7, 7, 7, 9, 9] and slot.tolist() == [0, 1, 3, 1, 2] and st == 8
    # seven: -0 (p7) and then -inf (p2) join; the NaN (p4) is last
    ptr, blk, slot, _ = oracle.topk_slots(ex, [8], bt2, 7, 4, lib=lib)
    assert slot.tolist() == [0, 1, 2, 3, 1, 2, 3]
    # length 0 and a length past the row (bit 1) keep nothing; a negative block id (bit 4)
    two = np.zeros((3, 8), np.float32)
    btn = np.array([[1, 2], [3, 4], [-5, 6]], np.int32)
    ptr, blk, slot, st = oracle.topk_slots(two, [0, 9, 2], btn, 4, 4, lib=lib)
    assert ptr.tolist() == [0, 0, 0, 2] and blk.tolist() == [-5, -5] and st == 1 | 4


TOPK_PINS = [pin_topk_matches_lexsort, pin_topk_closed_forms]
STORE_PINS = [pin_store_matches_torch, pin_store_closed_forms, pin_store_rotation_invariants,
              pin_store_slots]
ROUNDING_PINS = [pin_bf16_rne, pin_e4m3_rne, pin_fp8_scale]

DECODE_PINS = [pin_sdpa, pin_sink_minus_inf_is_softmax, pin_single_slot, pin_duplicate_adds_ln2,
               pin_zero_length, pin_permutation, pin_sink_factor, pin_scale_zero, pin_convexity,
               pin_hard_attention_limit, pin_sink_plus_inf, pin_token_subset]
BUILDER_PINS = [pin_builder_golden, pin_builder_ring_closed_form, pin_builder_capacity,
                pin_builder_comp_range]
VALIDATE_PINS = [pin_validate]
ALL_PINS = (DECODE_PINS + BUILDER_PINS + VALIDATE_PINS + FP8_PINS + STORE_PINS + ROUNDING_PINS
            + TOPK_PINS)


def failing_pins(lib, pins=ALL_PINS):
    """Names of the pins that fail (any exception counts) for this oracle build."""
    bad = []
    for p in pins:
        try:
            p(lib)
        except Exception:  # noqa: BLE001 - a failing pin is the signal
            bad.append(p.__name__)
    return bad
