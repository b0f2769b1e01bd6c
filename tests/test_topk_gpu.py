"""Top-k selection into the compressed slot lists (sda_topk_slots) on the GPU
against the oracle.  Integer output: comp_indptr, comp_block, comp_slot and
the status word must be bit-identical (the order -- larger score first, -0
equal to +0, NaN below -inf, ties by position, output in position order --
makes the kept set and its order unique)."""
import numpy as np
import pytest
import torch

import oracle
import parity
import sink_sda_decode_gb300 as sda
from sink_sda_decode_gb300 import inputs

pytestmark = pytest.mark.gpu


def run_both(scores, lengths, bt, k, kpb, capacity=None):
    ptr, blk, slot, st = sda.topk_slots(scores, lengths, bt, k=k, k_per_block=kpb, capacity=capacity)
    torch.cuda.synchronize()
    ref = oracle.topk_slots(scores.cpu().numpy(), lengths.cpu().numpy(), bt.cpu().numpy(), k, kpb)
    return (ptr.cpu().numpy(), blk.cpu().numpy(), slot.cpu().numpy(), int(st.item())), ref


def assert_equal(got, ref, what=""):
    ptr, blk, slot, st = got
    rptr, rblk, rslot, rst = ref
    assert np.array_equal(ptr, rptr), (what, "indptr")
    n = int(rptr[-1])
    assert np.array_equal(blk[:n], rblk), (what, "block", np.nonzero(blk[:n] != rblk)[0][:5])
    assert np.array_equal(slot[:n], rslot), (what, "slot", np.nonzero(slot[:n] != rslot)[0][:5])
    assert st == rst, (what, "status", st, rst)


@pytest.mark.parametrize("cfg", [1, 2, 3], ids=[inputs.CONFIG_NAMES[c] for c in (1, 2, 3)])
def test_topk_workloads(cfg):
    w = inputs.config(cfg, device="cuda")
    ti = inputs.topk_inputs(w)
    got, ref = run_both(ti.scores, ti.lengths, ti.block_table, ti.k, w.k_per_block)
    assert_equal(got, ref, inputs.CONFIG_NAMES[cfg])


def special_scores(rng, N, S):
    vals = np.array([1.0, 0.0, -0.0, -np.inf, np.inf, np.nan, 2.5, -1.0, 1e-30], np.float32)
    s = rng.standard_normal((N, S)).astype(np.float32)
    mask = rng.random((N, S)) < 0.5
    s[mask] = rng.choice(vals, int(mask.sum()))
    return s


@pytest.mark.parametrize("S,kpb", [(64, 8), (3000, 64), (9216, 64), (9217, 7), (40000, 64)])
def test_topk_ties_specials_and_lengths(S, kpb):
    """Half of the scores from a few values (ties, +-0, +-inf, NaN); lengths
    around k and at the row's end; rows staged in shared memory and rows too
    long for it (read from L2 by each pass)."""
    rng = np.random.default_rng(S + kpb)
    k = 33
    lens = np.array([0, 1, k - 1, k, k + 1, S, S - 1, S // 2], np.int32)
    N = len(lens)
    scores = torch.from_numpy(special_scores(rng, N, S)).cuda()
    B = -(-S // kpb)
    bt = torch.from_numpy(rng.integers(0, 10**6, (N, B)).astype(np.int32)).cuda()
    got, ref = run_both(scores, torch.from_numpy(lens).cuda(), bt, k, kpb)
    assert_equal(got, ref, f"S={S}")
    assert ref[3] == 8  # NaN candidates were present


@pytest.mark.parametrize("k", [1, 2, 100, 4096])
def test_topk_k_sweep_with_all_ties(k):
    """All-equal rows keep the first k positions; rows of distinct values keep
    the largest; k past every length keeps everything."""
    N, S, kpb = 4, 5000, 64
    rng = np.random.default_rng(k)
    s = np.zeros((N, S), np.float32)
    s[1] = -np.inf
    s[2] = rng.permutation(S).astype(np.float32)
    s[3] = rng.standard_normal(S).astype(np.float32)
    lens = np.array([S, S, S, 1234], np.int32)
    bt = torch.from_numpy(rng.integers(0, 1000, (N, -(-S // kpb))).astype(np.int32)).cuda()
    got, ref = run_both(torch.from_numpy(s).cuda(), torch.from_numpy(lens).cuda(), bt, k, kpb)
    assert_equal(got, ref, f"k={k}")


def test_topk_status_bits_and_capacity():
    rng = np.random.default_rng(5)
    N, S, kpb, k = 5, 100, 10, 7
    scores = torch.from_numpy(rng.standard_normal((N, S)).astype(np.float32)).cuda()
    lens = torch.tensor([5, -1, 101, 100, 30], dtype=torch.int32, device="cuda")
    bt_h = rng.integers(0, 50, (N, 10)).astype(np.int32)
    bt_h[4, :] = -3  # every block of token 4 is negative
    bt = torch.from_numpy(bt_h).cuda()
    got, ref = run_both(scores, lens, bt, k, kpb)
    assert_equal(got, ref, "status")
    assert ref[3] == 1 | 4
    # capacity below the total: every list empty, bit 32
    got, ref_ = run_both(scores, lens, bt, k, kpb, capacity=10)
    assert got[0].tolist() == [0] * (N + 1) and got[3] & 32
    # k = 0 and an empty batch
    got, ref = run_both(scores, lens, bt, 0, kpb)
    assert_equal(got, ref, "k=0")
    e = torch.zeros((0, S), dtype=torch.float32, device="cuda")
    ptr, _, _, st = sda.topk_slots(e, torch.zeros(0, dtype=torch.int32, device="cuda"),
                                   torch.zeros((0, 10), dtype=torch.int32, device="cuda"), k=k,
                                   k_per_block=kpb)
    torch.cuda.synchronize()
    assert ptr.tolist() == [0] and int(st.item()) == 0


def test_topk_rejects_bad_arguments():
    s = torch.zeros((2, 100), dtype=torch.float32, device="cuda")
    ln = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(RuntimeError):  # block table too short for the row
        sda.topk_slots(s, ln, torch.zeros((2, 9), dtype=torch.int32, device="cuda"), k=4,
                       k_per_block=10)
    with pytest.raises(RuntimeError):  # k_per_block <= 0
        sda.topk_slots(s, ln, torch.zeros((2, 10), dtype=torch.int32, device="cuda"), k=4,
                       k_per_block=0)
    with pytest.raises(TypeError):
        sda.topk_slots(s.double(), ln, torch.zeros((2, 10), dtype=torch.int32, device="cuda"),
                       k=4, k_per_block=10)


def test_topk_graph_capture_replay():
    w = inputs.config(1, device="cuda")
    ti = inputs.topk_inputs(w)
    N = w.N
    ptr = torch.empty(N + 1, dtype=torch.int32, device="cuda")
    blk = torch.empty(N * ti.k, dtype=torch.int32, device="cuda")
    slot = torch.empty(N * ti.k, dtype=torch.int32, device="cuda")
    st = torch.empty(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    kw = dict(k=ti.k, k_per_block=w.k_per_block, comp_indptr=ptr, comp_block=blk, comp_slot=slot,
              status=st, stream=s)
    with torch.cuda.stream(s):
        sda.topk_slots(ti.scores, ti.lengths, ti.block_table, **kw)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sda.topk_slots(ti.scores, ti.lengths, ti.block_table, **kw)
    blk.fill_(-7)
    ptr.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.topk_slots(ti.scores.cpu().numpy(), ti.lengths.cpu().numpy(),
                            ti.block_table.cpu().numpy(), ti.k, w.k_per_block)
    assert_equal((ptr.cpu().numpy(), blk.cpu().numpy(), slot.cpu().numpy(), int(st.item())), ref)


def test_topk_build_decode_pipeline():
    """Select -> build -> decode on the GPU against the oracle's own chain
    (its selection, its index build, its decode) on sampled tokens."""
    w = inputs.config(2, device="cuda")
    ti = inputs.topk_inputs(w)
    ptr, blk, slot, st = sda.topk_slots(ti.scores, ti.lengths, ti.block_table, k=ti.k,
                                        k_per_block=w.k_per_block)
    b = w.builder_inputs("cuda")
    idx, iptr, bst = sda.build_indices(b["state_slot"], b["swa_len"], b["swa_head"], ptr, blk,
                                       slot, win=w.win, k_per_block=w.k_per_block,
                                       swa_pages=w.swa_pages, total_pages=w.total_pages)
    out = sda.decode(w.q, w.unified_kv, idx, iptr, w.attn_sink, w.softmax_scale)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(bst.item()) == 0
    rptr, rblk, rslot, rst = oracle.topk_slots(ti.scores.cpu().numpy(), ti.lengths.cpu().numpy(),
                                               ti.block_table.cpu().numpy(), ti.k, w.k_per_block)
    o_idx, o_ptr, o_st = oracle.build_indices(w.state_slot, w.swa_len, w.swa_head, rptr, rblk,
                                              rslot, w.win, w.k_per_block, w.swa_pages,
                                              w.total_pages)
    assert o_st == 0 and rst == 0
    rng = np.random.default_rng(11)
    tok = np.sort(rng.choice(w.N, 24, replace=False))
    lists = [o_idx[o_ptr[t]:o_ptr[t + 1]] for t in tok]
    need = np.unique(np.concatenate(lists)) if sum(len(x) for x in lists) else np.zeros(0, np.int64)
    rows = inputs.bf16_to_bits(w.unified_kv[torch.from_numpy(need.astype(np.int64)).cuda()])
    sub_ptr = np.zeros(len(tok) + 1, np.int32)
    sub_ptr[1:] = np.cumsum([len(x) for x in lists])
    sub_idx = (np.searchsorted(need, np.concatenate(lists)) if len(need)
               else np.zeros(0, np.int64)).astype(np.int32)
    want = oracle.sda_decode(w.q_bits()[tok], rows, sub_idx, sub_ptr, w.attn_sink.cpu().numpy(),
                             w.softmax_scale)
    parity.assert_parity(parity.compare(out[torch.from_numpy(tok).cuda()], want), "topk+build+decode")


@pytest.mark.parametrize("N,S", [(4200, 200), (4097, 11268)])
def test_topk_large_batches(N, S):
    """More than 4096 tokens: comp_indptr comes from the separate scan kernel
    (smaller batches compute it inside the selection kernel); rows staged in
    shared memory and rows read from L2."""
    rng = np.random.default_rng(N + S)
    scores = special_scores(rng, N, S)
    lens = rng.integers(0, S + 1, N).astype(np.int32)
    lens[::7] = S
    kpb = 32
    bt = rng.integers(0, 10**5, (N, -(-S // kpb))).astype(np.int32)
    got, ref = run_both(torch.from_numpy(scores).cuda(), torch.from_numpy(lens).cuda(),
                        torch.from_numpy(bt).cuda(), 9, kpb)
    assert_equal(got, ref, f"N={N} S={S}")


@pytest.mark.parametrize("N,S", [(100, 3000), (150, 12000), (76, 700)])
def test_topk_mid_size_batches(N, S):
    """Mid-size batches with special values and ties, rows staged in shared
    memory and rows read from L2, lengths from 0 to the whole row, k from 1
    to past most lengths."""
    rng = np.random.default_rng(N * 7 + S)
    scores = special_scores(rng, N, S)
    lens = rng.integers(0, S + 1, N).astype(np.int32)
    lens[:4] = [0, 1, 40, S]
    kpb = 16
    bt = rng.integers(0, 10**5, (N, -(-S // kpb))).astype(np.int32)
    for k in (1, 40, 1000):
        got, ref = run_both(torch.from_numpy(scores).cuda(), torch.from_numpy(lens).cuda(),
                            torch.from_numpy(bt).cuda(), k, kpb)
        assert_equal(got, ref, f"N={N} S={S} k={k}")
