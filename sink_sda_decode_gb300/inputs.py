"""Seeded synthetic workloads for sparse sink decode attention.

This module only draws random inputs; it holds none of the attention or
index-building arithmetic, so that both the CUDA path and the CPU oracle can
be fed the very same inputs without sharing any of the method's code.

Shapes, sizes and value distributions follow the five benchmark workloads
of the project (tiny, H=16, ragged H=64, H=128, long-tail H=64); the
per-workload recipe is written next to each generator.  Everything is seeded:
index lists, q and attn_sink come from NumPy's PCG64 on the host (so they are
identical on every machine); the big unified KV pool is drawn with torch's
seeded generator directly on the target device (it is gigabytes) and copied
back only where a CPU consumer needs rows of it.

Per-token slot lists are drawn first; the index-builder descriptors
(state_slot / swa_len / swa_head + compressed (block, slot) pairs) are then
the plain inverse of how the slot ids are laid out in the pool:
SWA slot = state_slot * win + ring, compressed slot = swa_pages +
block * k_per_block + slot_in_block.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

SEED_BASE = 20261202
K_PER_BLOCK = 64
WIN = 128


@dataclasses.dataclass
class Workload:
    name: str
    N: int
    H: int
    D: int
    total_pages: int
    softmax_scale: float
    q: torch.Tensor              # [N, H, D] bf16 (device)
    unified_kv: torch.Tensor     # [total_pages, D] bf16 (device)
    attn_sink: torch.Tensor      # [H] fp32 (device)
    kv_indices: np.ndarray       # [sum L] int32, the intended packed lists
    kv_indptr: np.ndarray        # [N + 1] int32
    # index-builder descriptors (host, int32)
    state_slot: np.ndarray
    swa_len: np.ndarray
    swa_head: np.ndarray
    comp_indptr: np.ndarray
    comp_block: np.ndarray
    comp_slot: np.ndarray
    win: int
    k_per_block: int
    swa_pages: int
    recipe: str = ""
    seed: int = 0                # the generator seed (distinct per shard)

    @property
    def lengths(self) -> np.ndarray:
        return np.diff(self.kv_indptr)

    @property
    def total_len(self) -> int:
        return int(self.kv_indptr[-1] - self.kv_indptr[0])

    def q_bits(self) -> np.ndarray:
        return bf16_to_bits(self.q)

    def kv_rows_for(self, tokens=None):
        """Host copy of the pool restricted to the rows the given tokens read.

        Returns (kv_bits [R, D] uint16, kv_indices remapped into [0, R),
        kv_indptr rebased for the selected tokens, token order).  Pools of at
        most 256 MiB are copied whole (indices unchanged).
        """
        ptr = self.kv_indptr.astype(np.int64)
        if tokens is None:
            tokens = np.arange(self.N)
        tokens = np.asarray(tokens, dtype=np.int64)
        pieces = [self.kv_indices[ptr[t]:ptr[t + 1]] for t in tokens]
        lens = np.array([len(p) for p in pieces], dtype=np.int64)
        sub_idx = np.concatenate(pieces) if len(pieces) else np.zeros(0, np.int32)
        sub_ptr = np.zeros(len(tokens) + 1, dtype=np.int32)
        sub_ptr[1:] = np.cumsum(lens)
        if self.unified_kv.numel() * 2 <= (256 << 20):
            return bf16_to_bits(self.unified_kv), sub_idx.astype(np.int32), sub_ptr
        uniq, inv = np.unique(sub_idx, return_inverse=True)
        rows = self.unified_kv.index_select(
            0, torch.from_numpy(uniq.astype(np.int64)).to(self.unified_kv.device))
        return bf16_to_bits(rows), inv.astype(np.int32), sub_ptr

    def builder_inputs(self, device):
        def t(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
        return dict(state_slot=t(self.state_slot), swa_len=t(self.swa_len),
                    swa_head=t(self.swa_head), comp_indptr=t(self.comp_indptr),
                    comp_block=t(self.comp_block), comp_slot=t(self.comp_slot))


def bf16_to_bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _to_bf16(a: np.ndarray, device) -> torch.Tensor:
    # fp32 -> bf16 with round-to-nearest-even (torch's conversion)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).to(device)


def random_pool(total_pages: int, D: int, seed: int, device, chunk_rows: int = 1 << 20):
    """[total_pages, D] bf16 ~ N(0,1) drawn with torch's seeded generator on `device`."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    out = torch.empty((total_pages, D), dtype=torch.bfloat16, device=dev)
    for r0 in range(0, total_pages, chunk_rows):
        r1 = min(total_pages, r0 + chunk_rows)
        out[r0:r1] = torch.randn((r1 - r0, D), generator=g, device=dev, dtype=torch.float32)
    return out


E4M3_MAX = 448.0  # largest finite FP8 E4M3 magnitude


@dataclasses.dataclass
class Fp8Pool:
    """A pool stored as FP8: row s is e4m3(codes[s]) * scale[s]."""
    codes: torch.Tensor  # [P, D] uint8 E4M3 codes (device of the workload)
    scale: torch.Tensor  # [P] fp32


def fp8_pool(w: "Workload", pow2: bool = True, chunk_rows: int = 1 << 19) -> Fp8Pool:
    """The workload's bf16 pool quantised row by row the way an FP8 cache store
    fills one: code = E4M3 of row / scale rounded to nearest even (torch's
    float8_e4m3fn conversion, clamped to the finite range first) with
    scale = max|row| / 448 (1 for an all-zero row), or with `pow2` that value
    rounded up to a power of two (as block-scaled FP8 formats with 8-bit
    exponent scales store it), which makes code * scale exact in bf16."""
    P, D = w.unified_kv.shape
    dev = w.unified_kv.device
    codes = torch.empty((P, D), dtype=torch.uint8, device=dev)
    scale = torch.empty(P, dtype=torch.float32, device=dev)
    for r0 in range(0, P, chunk_rows):
        r1 = min(P, r0 + chunk_rows)
        rows = w.unified_kv[r0:r1].float()
        amax = rows.abs().amax(dim=1)
        sc = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
        if pow2:
            sc = torch.exp2(torch.ceil(torch.log2(sc)))
        x = (rows / sc[:, None]).clamp_(-E4M3_MAX, E4M3_MAX)
        codes[r0:r1] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        scale[r0:r1] = sc
    return Fp8Pool(codes=codes, scale=scale)


ROPE_DIM = 64        # rotated trailing dims of each 512-wide row
ROPE_BASE = 10000.0
MAX_POS = 1 << 16


@dataclasses.dataclass
class StoreInputs:
    """Inputs of the q/kv norm + RoPE + SWA store step of one decode step."""
    kv_new: torch.Tensor      # [N, D] bf16, the step's new latent row per token
    q_norm_w: torch.Tensor    # [D] bf16
    kv_norm_w: torch.Tensor   # [D] bf16
    cos_cache: torch.Tensor   # [max_pos, R/2] fp32
    sin_cache: torch.Tensor   # [max_pos, R/2] fp32
    positions: torch.Tensor   # [N] int32
    state_slot: torch.Tensor  # [N] int32 (< 0: padded)
    eps: float
    recipe: str = ""


def rope_caches(max_pos: int, rope_dim: int, base: float = ROPE_BASE, device="cpu"):
    """cos / sin tables [max_pos, rope_dim/2] of the angles pos * base^(-2i/R),
    evaluated in float64 and stored as fp32 (the usual RoPE frequency ladder)."""
    inv = base ** (-np.arange(0, rope_dim, 2, dtype=np.float64) / max(rope_dim, 1))
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    cos = torch.from_numpy(np.cos(ang).astype(np.float32)).to(device)
    sin = torch.from_numpy(np.sin(ang).astype(np.float32)).to(device)
    return cos, sin


def store_inputs(w: "Workload", rope_dim: int = ROPE_DIM, max_pos: int = MAX_POS,
                 seed: int | None = None, eps: float = 1e-6) -> StoreInputs:
    """Store-step inputs matching a decode workload: each live token's position
    is congruent to its ring head modulo win (so its new row lands on the
    newest SWA entry of its own list) and at least win; new KV rows ~ N(0,1)
    bf16; norm weights ~ U[0.5, 1.5) bf16; RoPE tables of base 10000 on the
    last `rope_dim` dims.  Padded tokens keep state_slot < 0."""
    rng = np.random.default_rng(w.seed + 700 if seed is None else seed)
    dev = w.q.device
    N, D, win = w.N, w.D, w.win
    kv_new = _to_bf16(rng.standard_normal((N, D)), dev)
    qw = _to_bf16(rng.uniform(0.5, 1.5, D), dev)
    kw = _to_bf16(rng.uniform(0.5, 1.5, D), dev)
    laps = rng.integers(1, max(2, max_pos // win), N)
    pos = (w.swa_head.astype(np.int64) + laps * win).astype(np.int64)
    pos = np.minimum(pos, max_pos - win + w.swa_head.astype(np.int64)).astype(np.int32)
    cos, sin = rope_caches(max_pos, rope_dim, device=dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    return StoreInputs(kv_new=kv_new, q_norm_w=qw, kv_norm_w=kw, cos_cache=cos, sin_cache=sin,
                       positions=t(pos), state_slot=t(w.state_slot), eps=eps,
                       recipe=f"new KV N(0,1) bf16, weights U[0.5,1.5), RoPE base 1e4 on the last "
                              f"{rope_dim} dims, positions = ring head + win * U{{1..{max_pos // win - 1}}}")


TOPK_K = 512          # compressed entries kept per token (the workloads' compressed lists)
TOPK_CANDIDATES = 8192


@dataclasses.dataclass
class TopkInputs:
    """Inputs of the top-k -> slot-list step: per-token indexer scores over
    the token's compressed-cache positions and its block table."""
    scores: torch.Tensor       # [N, S] fp32
    lengths: torch.Tensor      # [N] int32 (0 for padded tokens)
    block_table: torch.Tensor  # [N, S / k_per_block] int32, distinct blocks per token
    k: int
    recipe: str = ""


def topk_inputs(w: "Workload", candidates: int = TOPK_CANDIDATES, k: int = TOPK_K,
                seed: int | None = None, ragged: bool | None = None) -> TopkInputs:
    """Top-k inputs matching a decode workload: scores ~ N(0,1) fp32 over
    `candidates` positions per token (uniform U{0..candidates} lengths when
    `ragged`, by default for workloads that pad tokens), length 0 for padded
    tokens, and a block table of distinct random blocks of the workload's
    compressed region."""
    rng = np.random.default_rng(w.seed + 900 if seed is None else seed)
    dev = w.q.device
    N, kpb = w.N, w.k_per_block
    B = -(-candidates // kpb)
    n_blocks = (w.total_pages - w.swa_pages) // kpb
    scores = rng.standard_normal((N, candidates), dtype=np.float32)
    if ragged is None:
        ragged = bool((w.state_slot < 0).any())
    lens = rng.integers(0, candidates + 1, N) if ragged else np.full(N, candidates)
    lens[w.state_slot < 0] = 0
    bt = np.stack([rng.choice(n_blocks, B, replace=False) for _ in range(N)]).astype(np.int32)
    return TopkInputs(scores=torch.from_numpy(scores).to(dev),
                      lengths=torch.from_numpy(lens.astype(np.int32)).to(dev),
                      block_table=torch.from_numpy(bt).to(dev), k=k,
                      recipe=f"scores N(0,1) fp32 over {candidates} positions"
                             f"{' (lengths U{0..%d})' % candidates if ragged else ''}, k={k}, "
                             f"{B} distinct random blocks per token")


def fp8_rows_for(w: "Workload", pool: Fp8Pool, tokens=None):
    """Host copy of an FP8 pool restricted to the rows the given tokens read:
    (codes [R, D] uint8, scale [R] fp32, kv_indices remapped into [0, R),
    kv_indptr rebased), as Workload.kv_rows_for."""
    ptr = w.kv_indptr.astype(np.int64)
    if tokens is None:
        tokens = np.arange(w.N)
    tokens = np.asarray(tokens, dtype=np.int64)
    pieces = [w.kv_indices[ptr[t]:ptr[t + 1]] for t in tokens]
    lens = np.array([len(p) for p in pieces], dtype=np.int64)
    sub_idx = np.concatenate(pieces) if len(pieces) else np.zeros(0, np.int32)
    sub_ptr = np.zeros(len(tokens) + 1, dtype=np.int32)
    sub_ptr[1:] = np.cumsum(lens)
    uniq, inv = np.unique(sub_idx, return_inverse=True)
    sel = torch.from_numpy(uniq.astype(np.int64)).to(pool.codes.device)
    codes = pool.codes.index_select(0, sel).cpu().numpy() if uniq.size else np.zeros((0, w.D), np.uint8)
    scale = pool.scale.index_select(0, sel).cpu().numpy() if uniq.size else np.zeros(0, np.float32)
    return codes, scale, inv.astype(np.int32), sub_ptr


def _descriptors(lists, swa_parts, swa_pages, win, kpb):
    """Builder descriptors that reproduce `lists` (SWA part first, then compressed)."""
    N = len(lists)
    state_slot = np.full(N, -1, np.int32)
    swa_len = np.zeros(N, np.int32)
    swa_head = np.zeros(N, np.int32)
    comp_ptr = np.zeros(N + 1, np.int64)
    blocks, slots = [], []
    for t, (lst, sp) in enumerate(zip(lists, swa_parts)):
        if sp is None:                      # padded token
            comp_ptr[t + 1] = comp_ptr[t]
            continue
        state, n_swa, head = sp
        state_slot[t] = state
        swa_len[t] = n_swa
        swa_head[t] = head
        comp = np.asarray(lst[n_swa:], dtype=np.int64) - swa_pages
        b, s = np.divmod(comp, kpb)
        blocks.append(b)
        slots.append(s)
        comp_ptr[t + 1] = comp_ptr[t] + len(comp)
    cb = np.concatenate(blocks).astype(np.int32) if blocks else np.zeros(0, np.int32)
    cs = np.concatenate(slots).astype(np.int32) if slots else np.zeros(0, np.int32)
    return state_slot, swa_len, swa_head, comp_ptr.astype(np.int32), cb, cs


def _ring(state, n_swa, head, win):
    """SWA slots of one state, oldest -> newest (head = newest ring position)."""
    pos = (head - n_swa + 1 + np.arange(n_swa)) % win
    return state * win + pos


def _assemble(name, N, H, D, P, lists, swa_parts, swa_pages, sink_sigma, seed, device, recipe,
              win=WIN, kpb=K_PER_BLOCK, q_rng=None):
    rng = q_rng
    q = _to_bf16(rng.standard_normal((N, H, D), dtype=np.float32), device)
    sink = torch.from_numpy((rng.standard_normal(H) * sink_sigma).astype(np.float32)).to(device)
    lens = np.array([len(x) for x in lists], dtype=np.int64)
    ptr = np.zeros(N + 1, np.int64)
    ptr[1:] = np.cumsum(lens)
    idx = (np.concatenate([np.asarray(x, np.int64) for x in lists]) if lens.sum()
           else np.zeros(0, np.int64)).astype(np.int32)
    desc = _descriptors(lists, swa_parts, swa_pages, win, kpb)
    kv = random_pool(P, D, seed + 7919, device)
    return Workload(name=name, N=N, H=H, D=D, total_pages=P, softmax_scale=1.0 / math.sqrt(D),
                    q=q, unified_kv=kv, attn_sink=sink, kv_indices=idx,
                    kv_indptr=ptr.astype(np.int32), state_slot=desc[0], swa_len=desc[1],
                    swa_head=desc[2], comp_indptr=desc[3], comp_block=desc[4], comp_slot=desc[5],
                    win=win, k_per_block=kpb, swa_pages=swa_pages, recipe=recipe, seed=seed)


def tiny(device="cpu", seed=SEED_BASE + 0):
    """N=4, H=8, D=64, pool 4096; lengths {0,1,17,64} in random order, slots
    uniform without replacement; sink ~ N(0,1); scale 1/sqrt(D)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    N, H, D, P = 4, 8, 64, 4096
    lens = rng.permutation(np.array([0, 1, 17, 64]))
    lists, swa = [], []
    for L in lens:
        lists.append(rng.choice(P, int(L), replace=False))
        swa.append(None if L == 0 else (0, 0, 0))
    return _assemble("tiny N=4 H=8 D=64", N, H, D, P, lists, swa, 0, 1.0, seed, device,
                     tiny.__doc__, q_rng=rng)


def _swa_plus_random(rng, N, P, comp_lens, zero_tokens=()):
    swa_pages = N * WIN
    lists, swa = [], []
    zero = set(int(z) for z in zero_tokens)
    for t in range(N):
        if t in zero:
            lists.append(np.zeros(0, np.int64))
            swa.append(None)
            continue
        head = int(rng.integers(0, WIN))
        ring = _ring(t, WIN, head, WIN)
        comp = swa_pages + rng.choice(P - swa_pages, int(comp_lens[t]), replace=False)
        lists.append(np.concatenate([ring, comp]))
        swa.append((t, WIN, head))
    return lists, swa, swa_pages


def h16(device="cpu", seed=SEED_BASE + 1):
    """N=64, H=16, D=512, pool 2^20 (first 8192 slots = SWA region, 64 states x
    win 128); each token: its 128 ring slots + 512 compressed slots uniform
    without replacement from the rest (L=640); sink ~ N(0,1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    N, H, D, P = 64, 16, 512, 1 << 20
    lists, swa, swa_pages = _swa_plus_random(rng, N, P, np.full(N, 512))
    return _assemble("N=64 H=16 D=512 L=640", N, H, D, P, lists, swa, swa_pages, 1.0, seed, device,
                     h16.__doc__, q_rng=rng)


def ragged_h64(device="cpu", seed=SEED_BASE + 2):
    """N=256, H=64, D=512, pool 2^21 (SWA region 256 x 128); 26 tokens (10%,
    seeded choice) zero-length padding; the others 128 ring slots + U{0..2048}
    compressed slots; sink ~ N(0,1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    N, H, D, P = 256, 64, 512, 1 << 21
    zero = rng.choice(N, int(round(0.1 * N)), replace=False)
    comp_lens = rng.integers(0, 2049, size=N)
    lists, swa, swa_pages = _swa_plus_random(rng, N, P, comp_lens, zero)
    return _assemble("N=256 H=64 D=512 ragged", N, H, D, P, lists, swa, swa_pages, 1.0, seed, device,
                     ragged_h64.__doc__, q_rng=rng)


def h128(device="cpu", seed=SEED_BASE + 3):
    """N=1024, H=128, D=512, pool 2^21 (SWA region 1024 x 128); each token 128
    ring slots + 512 random compressed slots (L=640); sink ~ N(0,1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    N, H, D, P = 1024, 128, 512, 1 << 21
    lists, swa, swa_pages = _swa_plus_random(rng, N, P, np.full(N, 512))
    return _assemble("N=1024 H=128 D=512 L=640", N, H, D, P, lists, swa, swa_pages, 1.0, seed,
                     device, h128.__doc__, q_rng=rng)


def longtail_h64(device="cpu", seed=SEED_BASE + 4):
    """N=512, H=64, D=512, pool 2^22 slots (4 GiB), no SWA region; L_t =
    round(2^u), u ~ U[0,13] (log-uniform in [1, 8192]), except token 1 with
    L=65536; even tokens read contiguous runs of 64 slots (whole compressed
    blocks at distinct random block ids, last run truncated), odd tokens read
    uniform random slots without replacement; sink ~ N(0, 2^2)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    N, H, D, P = 512, 64, 512, 1 << 22
    lens = np.rint(2.0 ** rng.uniform(0.0, 13.0, size=N)).astype(np.int64)
    lens[1] = 65536
    lists, swa = [], []
    n_blocks = P // K_PER_BLOCK
    for t in range(N):
        L = int(lens[t])
        if t % 2 == 0:
            nb = -(-L // K_PER_BLOCK)
            blocks = rng.choice(n_blocks, nb, replace=False)
            lst = (blocks[:, None] * K_PER_BLOCK + np.arange(K_PER_BLOCK)[None, :]).reshape(-1)[:L]
        else:
            lst = rng.choice(P, L, replace=False)
        lists.append(lst)
        swa.append((0, 0, 0))
    return _assemble("N=512 H=64 D=512 long-tail", N, H, D, P, lists, swa, 0, 2.0, seed, device,
                     longtail_h64.__doc__, q_rng=rng)


def prefill_h64(device="cpu", seed=SEED_BASE + 5):
    """Sparse prefill: one chunk of N=2048 consecutive tokens of a sequence,
    H=64, D=512, pool 2^21 slots, no SWA region.  Token i attends over its
    causal window of the chunk's own rows (slots max(0, i-127) .. i of a
    staging region at the start of the pool, where the chunk's new K/V rows
    sit: 1..128 entries) and over 512 compressed entries drawn for it from a
    2048-entry candidate set the whole chunk shares (neighbouring tokens'
    selections over the same context overlap heavily); sink ~ N(0,1).  The
    lists go through the index builder as compressed (block, slot) pairs."""
    rng = np.random.Generator(np.random.PCG64(seed))
    N, H, D, P = 2048, 64, 512, 1 << 21
    cand = N + rng.choice(P - N, 2048, replace=False)
    lists, swa = [], []
    for i in range(N):
        window = np.arange(max(0, i - WIN + 1), i + 1)
        lists.append(np.concatenate([window, rng.choice(cand, 512, replace=False)]))
        swa.append((0, 0, 0))
    return _assemble("N=2048 H=64 D=512 prefill chunk", N, H, D, P, lists, swa, 0, 1.0, seed,
                     device, prefill_h64.__doc__, q_rng=rng)


GENERATORS = [tiny, h16, ragged_h64, h128, longtail_h64, prefill_h64]
CONFIG_NAMES = ["tiny", "h16", "ragged_h64", "h128", "longtail_h64", "prefill_h64"]


SHARD_SEED_STRIDE = 1000


def config(i: int, device="cpu", shard: int = 0) -> Workload:
    """Workload i (0..5) with its fixed seed SEED_BASE + i.

    `shard` > 0 draws another batch of the same recipe (seed offset by
    SHARD_SEED_STRIDE per shard): under data parallelism each process decodes
    its own independent token batch; shard 0 is the workload itself."""
    if shard < 0:
        raise ValueError("shard must be >= 0")
    return GENERATORS[i](device=device, seed=SEED_BASE + i + SHARD_SEED_STRIDE * shard)


def random_small(seed: int, N: int, H: int, D: int, P: int, lengths, sink_sigma=1.0,
                 device="cpu", duplicates=False) -> Workload:
    """Small random case for parity sweeps: given per-token lengths, slots drawn
    uniformly (with replacement if `duplicates`), q/kv/sink normal."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lists, swa = [], []
    for L in lengths:
        L = int(L)
        if duplicates:
            lists.append(rng.integers(0, P, size=L))
        else:
            lists.append(rng.choice(P, L, replace=False))
        swa.append((0, 0, 0))
    return _assemble(f"random N={N} H={H} D={D}", N, H, D, P, lists, swa, 0, sink_sigma,
                     seed, device, "random_small", q_rng=rng)
