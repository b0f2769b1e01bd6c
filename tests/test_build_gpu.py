"""GPU index builder and validator: bit-exact against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins
import sink_sda_decode_gb300 as sda
from sink_sda_decode_gb300 import inputs

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def gpu_build(ss, sl, sh, cp, cb, cs, win, kpb, swa_pages, total_pages, capacity=None):
    idx, ptr, st = sda.build_indices(dev(ss), dev(sl), dev(sh), dev(cp), dev(cb), dev(cs), win=win,
                                     k_per_block=kpb, swa_pages=swa_pages, total_pages=total_pages,
                                     capacity=capacity)
    ptr_h = ptr.cpu().numpy()
    return idx.cpu().numpy()[:ptr_h[-1]], ptr_h, int(st.item())


def test_golden_example():
    g = oracle_pins.read_golden_builder()
    idx, ptr, st = gpu_build(g["state_slot"], g["swa_len"], g["swa_head"], g["comp_indptr"],
                             g["comp_block"], g["comp_slot"], g["win"][0], g["k_per_block"][0],
                             g["swa_pages"][0], g["total_pages"][0])
    assert idx.tolist() == g["kv_indices"]
    assert ptr.tolist() == g["kv_indptr"]
    assert st == g["status"][0]


@pytest.mark.parametrize("cfg", range(len(inputs.CONFIG_NAMES)), ids=inputs.CONFIG_NAMES)
def test_workload_lists_bit_exact(cfg):
    w = inputs.config(cfg, device="cuda")
    args = (w.state_slot, w.swa_len, w.swa_head, w.comp_indptr, w.comp_block, w.comp_slot, w.win,
            w.k_per_block, w.swa_pages, w.total_pages)
    idx, ptr, st = gpu_build(*args)
    assert st == 0
    assert np.array_equal(ptr, w.kv_indptr)
    assert np.array_equal(idx, w.kv_indices)
    o_idx, o_ptr, o_st = oracle.build_indices(*args)
    assert np.array_equal(idx, o_idx) and np.array_equal(ptr, o_ptr) and st == o_st


def random_descriptors(rng, N, win, kpb, n_states, n_blocks, bad=True, max_comp=40):
    swa_pages = n_states * win
    total_pages = swa_pages + n_blocks * kpb
    ss = rng.integers(-1, n_states, N)
    sl = rng.integers(0, win + 1, N)
    sh = rng.integers(0, win, N)
    cl = rng.integers(0, max_comp, N)
    cp = np.zeros(N + 1, np.int64)
    cp[1:] = np.cumsum(cl)
    cb = rng.integers(0, n_blocks, cp[-1])
    cs = rng.integers(0, kpb, cp[-1])
    if bad:
        k = rng.integers(0, N, 6)
        sl[k[0]] = win + 1                      # bit 1
        sh[k[1]] = win; sl[k[1]] = 3            # bit 2
        ss[k[2]] = n_states + 2; sl[k[2]] = 1   # bit 16 (SWA slot outside its region)
        if cp[-1] > 2:
            cs[0] = kpb                         # bit 8
            cb[1] = n_blocks                    # bit 16 (compressed slot >= total_pages)
            cb[2] = -5                          # bit 8
    return ss, sl, sh, cp.astype(np.int32), cb, cs, win, kpb, swa_pages, total_pages


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("N", [1, 7, 1000, 5000])
def test_random_descriptors_bit_exact(seed, N):
    rng = np.random.default_rng(seed * 7919 + N)
    args = random_descriptors(rng, N, win=16, kpb=8, n_states=max(N // 2, 1), n_blocks=300)
    idx, ptr, st = gpu_build(*args)
    o_idx, o_ptr, o_st = oracle.build_indices(*args)
    assert st == o_st
    assert np.array_equal(ptr, o_ptr)
    assert np.array_equal(idx, o_idx)


@pytest.mark.parametrize("seed", [1, 2])
@pytest.mark.parametrize("N", [1, 9, 300])
def test_long_lists_bit_exact(seed, N):
    """Thousands of compressed entries per token (each token's entries take
    several passes of its CTA's threads); bad entries sit at the ends of long
    lists."""
    rng = np.random.default_rng(seed * 104729 + N)
    ss, sl, sh, cp, cb, cs, win, kpb, swa_pages, total_pages = random_descriptors(
        rng, N, win=16, kpb=8, n_states=max(N // 2, 1), n_blocks=5000, max_comp=6000)
    for t in rng.integers(0, N, 3):
        if cp[t + 1] - cp[t] > 10:
            cs[cp[t + 1] - 1] = kpb if rng.random() < 0.5 else cs[cp[t + 1] - 1]
            cb[cp[t + 1] - 2] = 5000 if rng.random() < 0.5 else cb[cp[t + 1] - 2]
    args = (ss, sl, sh, cp, cb, cs, win, kpb, swa_pages, total_pages)
    idx, ptr, st = gpu_build(*args)
    o_idx, o_ptr, o_st = oracle.build_indices(*args)
    assert st == o_st
    assert np.array_equal(ptr, o_ptr)
    assert np.array_equal(idx, o_idx)


def test_capacity_overflow_and_empty_batch():
    args = random_descriptors(np.random.default_rng(5), 50, 8, 4, 50, 10, bad=False)
    total = oracle.build_indices(*args)[1][-1]
    idx, ptr, st = gpu_build(*args, capacity=int(total) - 1)
    assert st & 32 and np.all(ptr == 0)
    e = np.zeros(0, np.int32)
    idx, ptr, st = gpu_build(e, e, e, np.zeros(1, np.int32), e, e, 4, 4, 0, 10)
    assert ptr.tolist() == [0] and st == 0


def test_validate_matches_oracle():
    rng = np.random.default_rng(3)
    for _ in range(5):
        n = int(rng.integers(1, 3000))
        idx = rng.integers(-3, 1000, n).astype(np.int32)
        ptr = np.sort(rng.integers(0, n + 1, 41)).astype(np.int32)
        if rng.random() < 0.5:
            ptr[5], ptr[6] = ptr[6] + 1, ptr[5]
        if rng.random() < 0.3:
            ptr[-1] = n + 4
        st = sda.validate_indices(dev(idx), dev(ptr), 997).cpu().numpy()
        assert tuple(int(x) for x in st) == oracle.validate_indices(idx, ptr, 997)


def check_against_oracle(args, capacity=None, offset=0):
    """GPU build of `args` (capacity as given) against the oracle.  offset > 0
    passes comp_block / comp_slot as views that start `offset` entries into
    larger arrays, so that their addresses are not 16-byte aligned."""
    ss, sl, sh, cp, cb, cs, win, kpb, swa_pages, total_pages = args
    cbd, csd = dev(np.concatenate([np.zeros(offset, np.int32), cb])), \
        dev(np.concatenate([np.zeros(offset, np.int32), cs]))
    idx, ptr, st = sda.build_indices(dev(ss), dev(sl), dev(sh), dev(cp), cbd[offset:], csd[offset:],
                                     win=win, k_per_block=kpb, swa_pages=swa_pages,
                                     total_pages=total_pages, capacity=capacity)
    ptr_h = ptr.cpu().numpy()
    o_idx, o_ptr, o_st = oracle.build_indices(*args, capacity=capacity)
    assert int(st.item()) == o_st
    assert np.array_equal(ptr_h, o_ptr)
    assert np.array_equal(idx.cpu().numpy()[:ptr_h[-1]], o_idx)
    return o_st


def test_entry_check_overlapping_and_stray_entries():
    """The length pass checks the entry array in slices without knowing the
    tokens, and the scan re-checks the tokens that overlap a flagged slice.
    With a non-monotone comp_indptr, token ranges overlap: an entry listed
    by two tokens marks both, an entry listed only by a token whose range is
    bad (bit 4) or by a padded token marks none, nor does one that no token
    lists."""
    win, kpb, n_blocks = 8, 4, 50
    swa_pages = 4 * win
    total_pages = swa_pages + n_blocks * kpb
    n_entries = 20003  # not a multiple of 4: the last chunk runs past the arrays' end
    rng = np.random.default_rng(11)
    cb = rng.integers(0, n_blocks, n_entries).astype(np.int32)
    cs = rng.integers(0, kpb, n_entries).astype(np.int32)
    # token 0 [0, 9000); token 1 [9000, 3000): bit 4; token 2 [3000, 5000)
    # and token 3 [5000, 15000), both inside token 0's range in part;
    # token 4 padded over [15000, 20000); token 5 [20000, 15000): bit 4;
    # entries [20000, 20003) belong to no token
    ss = np.array([0, 1, 2, 3, -1, 0], np.int32)
    sl = np.array([2, 0, 3, 1, 0, 0], np.int32)
    sh = np.array([1, 0, 5, 7, 0, 0], np.int32)
    cp = np.array([0, 9000, 3000, 5000, 15000, 20000, 15000], np.int32)
    cap = 40000  # overlapping ranges list some entries twice
    assert check_against_oracle((ss, sl, sh, cp, cb, cs, win, kpb, swa_pages, total_pages), cap) == 4
    cases = {  # entry -> the bit it raises
        "listed by tokens 0 and 3": (6000, 8),
        "listed by tokens 0 and 2": (4000, 16),
        "listed by token 0 (and the bad-range token 1)": (8999, 8),
        "listed only by the padded token 4": (17000, 8),
        "listed by no token": (20001, 16),
    }
    for what, (e, bit) in cases.items():
        cb2, cs2 = cb.copy(), cs.copy()
        if bit == 16:
            cb2[e] = n_blocks + 3
        else:
            cs2[e] = kpb
        st = check_against_oracle((ss, sl, sh, cp, cb2, cs2, win, kpb, swa_pages, total_pages), cap)
        assert st & 4 and not st & 32, what
    # every entry bad: every token with a good range and a real slot is marked
    check_against_oracle((ss, sl, sh, cp, np.full_like(cb, -1), cs, win, kpb, swa_pages, total_pages),
                         cap)


@pytest.mark.parametrize("offset", [0, 1, 3])
@pytest.mark.parametrize("capacity", ["auto", 0, 5, 2000])
def test_entry_check_alignment_and_capacity(offset, capacity):
    """Entry arrays that are not 16-byte aligned (checked one entry per
    load), and capacities that leave the flags little room or none (0: the
    single flag goes through the status word)."""
    rng = np.random.default_rng(offset * 31 + (7 if capacity == "auto" else capacity))
    args = random_descriptors(rng, 400, win=16, kpb=8, n_states=200, n_blocks=3000, max_comp=900)
    cap = None if capacity == "auto" else capacity
    check_against_oracle(args, capacity=cap, offset=offset)


@pytest.mark.parametrize("N", [305, 2000])
def test_long_lists_flat_scatter(N):
    """Batches above one wave of one-token CTAs take the scatter that is flat
    over the packed output: a 65 536-entry list among short ones, lists that
    end inside a thread's four outputs, empty and padded tokens between."""
    rng = np.random.default_rng(N)
    ss, sl, sh, cp, cb, cs, win, kpb, swa_pages, total_pages = random_descriptors(
        rng, N, win=16, kpb=8, n_states=N, n_blocks=20000, bad=False, max_comp=7)
    lens = np.diff(cp.astype(np.int64))
    lens[N // 3] = 65536
    lens[N // 2] = 0
    ss[N // 2 + 1] = -1
    cp = np.zeros(N + 1, np.int64)
    cp[1:] = np.cumsum(lens)
    cb = rng.integers(0, 20000, cp[-1]).astype(np.int32)
    cs = rng.integers(0, kpb, cp[-1]).astype(np.int32)
    st = check_against_oracle((ss, sl, sh, cp.astype(np.int32), cb, cs, win, kpb, swa_pages,
                               total_pages))
    assert st == 0


@pytest.mark.parametrize("N", [9000, 13000])
def test_large_batches_unstaged_scatter(N):
    """Batches above 8191 tokens: the flat scatter searches kv_indptr in
    global memory instead of a shared-memory copy."""
    rng = np.random.default_rng(N + 17)
    args = random_descriptors(rng, N, win=16, kpb=8, n_states=N, n_blocks=5000, max_comp=30)
    check_against_oracle(args)
