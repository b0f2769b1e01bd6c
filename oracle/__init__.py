"""fp64 CPU oracle for sparse sink decode attention and its index builder.

TEST INFRASTRUCTURE ONLY.  The only code that may import this package is the
test suite (``tests/``), the smoke check in ``__graft_entry__.py`` and the
CPU-baseline / reference leg of ``bench.py``.  The product library never
imports, links or calls it, and it imports nothing from the product package.

The arithmetic lives in ``sda_oracle.c`` (plain C, double precision, one
OpenMP loop over (token, head)); this module only compiles it with gcc on
first use and marshals NumPy arrays through ctypes.

``sda_decode_fp8`` is the same attention over a pool stored as FP8 E4M3
codes with one fp32 scale per row (a format the pages do not fix; it serves
the FP8-pool variant of the path).

``qk_norm_rope_store`` is the step that fills the pool before decode: the
per-head RMSNorm of q, the RMSNorm of the step's new KV row, GPT-J RoPE on
the last R dims and the store of the KV row into its SWA ring slot (sglang PR
25898 summary page, sections "关键文件" and "关键符号"); ``bf16_rne`` and
``fp8_quantise_rows`` give the rounded forms it stores.

``topk_slots`` is the step before the index builder: per token, the k
best-scored compressed-cache positions (NaN padding ranks below -inf, ties in
position order), emitted in position order and mapped through the token's
block table to (block, slot in block) pairs (sglang attention tag page,
entry "DSV4.1 新增索引器内核，重做 Top-K v2 分派").

What it computes follows the docstring of ``paged_decode.py`` quoted on the
sglang PR 28392 summary page ("为 AMD V4 内核添加 ATOM 来源注释", section
"关键源码片段": caller convention, returns, numerics):

    x_j = softmax_scale * <q[t,h,:], kv[S_j,:]>
    out[t,h,:] = sum_j e^{x_j} kv[S_j,:] / (e^{sink_h} + sum_j e^{x_j})

with S = kv_indices[kv_indptr[t]:kv_indptr[t+1]].  The pins that tie this to
the pages and to mathematics, not to itself, are in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sda_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_ERRORS = {1: "bad shape", 2: "bad kv_indptr", 3: "slot out of range", 4: "out of memory"}

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False, src: str = _SRC, dst: str = _LIB) -> str:
    """Compile the C oracle into a shared library (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(dst) and os.path.getmtime(dst) >= os.path.getmtime(src):
        return dst
    tmp = dst + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, dst)
    return dst


def _bind(lib):
    lib.oracle_sda_decode.restype = ctypes.c_int
    lib.oracle_sda_decode.argtypes = [
        _u16p, _u16p, ctypes.c_int64, _i32p, ctypes.c_int64, _i32p, _f32p, ctypes.c_float,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int, _f64p]
    lib.oracle_sda_decode_fp8.restype = ctypes.c_int
    lib.oracle_sda_decode_fp8.argtypes = [
        _u16p, _u8p, _f32p, ctypes.c_int64, _i32p, ctypes.c_int64, _i32p, _f32p, ctypes.c_float,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int, _f64p]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_build_indices.restype = ctypes.c_int
    lib.oracle_build_indices.argtypes = [
        _i32p, _i32p, _i32p, _i32p, _i32p, _i32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _i32p, ctypes.c_int64, _i32p, _i32p]
    lib.oracle_validate_indices.restype = ctypes.c_int
    lib.oracle_validate_indices.argtypes = [
        _i32p, ctypes.c_int64, _i32p, ctypes.c_int, ctypes.c_int64, _i32p]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_qk_norm_rope_store.restype = ctypes.c_int
    lib.oracle_qk_norm_rope_store.argtypes = [
        _u16p, _u16p, _u16p, _u16p, _f32p, _f32p, ctypes.c_int, _i32p, _i32p, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int64,
        _f64p, _f64p, _i64p, _i32p]
    lib.oracle_bf16_rne_array.restype = None
    lib.oracle_bf16_rne_array.argtypes = [_f64p, ctypes.c_int64, _u16p]
    lib.oracle_fp8_quantise_rows.restype = None
    lib.oracle_fp8_quantise_rows.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int, _u8p, _f32p]
    lib.oracle_topk_slots.restype = ctypes.c_int
    lib.oracle_topk_slots.argtypes = [
        _f32p, ctypes.c_int64, _i32p, _i32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, _i32p, _i32p, _i32p, _i32p]
    lib.oracle_e4m3_rne_array.restype = None
    lib.oracle_e4m3_rne_array.argtypes = [_f64p, ctypes.c_int64, _u8p]
    lib.oracle_e4m3_rne.restype = ctypes.c_uint8
    lib.oracle_e4m3_rne.argtypes = [ctypes.c_double]
    lib.oracle_fp8_scale_exponent.restype = ctypes.c_int
    lib.oracle_fp8_scale_exponent.argtypes = [ctypes.c_double]
    return lib


def load(path: str | None = None):
    """Return the ctypes handle of the oracle library, compiling it if needed."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def num_threads(lib=None) -> int:
    """Threads the oracle's OpenMP loop uses (OMP_NUM_THREADS or all cores)."""
    return int((lib or load()).oracle_num_threads())


def bf16_bits(x) -> np.ndarray:
    """View a bf16 array (uint16 bit patterns or a torch bf16 tensor) as uint16."""
    if hasattr(x, "detach"):  # torch tensor
        import torch

        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    return _as(np.asarray(x).view(np.uint16), np.uint16)


def sda_decode(q_bits, kv_bits, kv_indices, kv_indptr, attn_sink, softmax_scale,
               tokens=None, lib=None) -> np.ndarray:
    """fp64 sparse sink decode attention.

    q_bits [N,H,D] and kv_bits [P,D] are bf16 bit patterns (uint16).  Returns
    float64 [len(tokens) or N, H, D].  ``softmax_scale`` is rounded to fp32,
    as the CUDA entry point receives it.
    """
    lib = lib or load()
    q = _as(q_bits, np.uint16)
    kv = _as(kv_bits, np.uint16)
    N, H, D = q.shape
    assert kv.ndim == 2 and kv.shape[1] == D
    idx = _as(kv_indices, np.int32)
    ptr = _as(kv_indptr, np.int32)
    sink = _as(attn_sink, np.float32)
    assert ptr.shape == (N + 1,) and sink.shape == (H,)
    if tokens is None:
        tok = None
        n_tok = N
    else:
        tok = _as(tokens, np.int32)
        n_tok = int(tok.size)
    out = np.zeros((n_tok, H, D), dtype=np.float64)
    idx_arg = idx if idx.size else np.zeros(1, np.int32)
    rc = lib.oracle_sda_decode(_ptr(q, ctypes.c_uint16), _ptr(kv, ctypes.c_uint16), kv.shape[0],
                               _ptr(idx_arg, ctypes.c_int32), idx.size, _ptr(ptr, ctypes.c_int32),
                               _ptr(sink, ctypes.c_float), float(np.float32(softmax_scale)),
                               N, H, D, None if tok is None else _ptr(tok, ctypes.c_int32), n_tok,
                               _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle_sda_decode: {_ERRORS.get(rc, rc)}")
    return out


def e4m3_values(lib=None) -> np.ndarray:
    """The 256 FP8 E4M3 codes decoded to float64 by the oracle (index = code)."""
    lib = lib or load()
    return np.array([lib.oracle_e4m3_to_double(c) for c in range(256)], dtype=np.float64)


def fp8_codes(x) -> np.ndarray:
    """View an FP8 array (uint8 codes or a torch float8_e4m3fn / uint8 tensor) as uint8."""
    if hasattr(x, "detach"):  # torch tensor
        import torch

        x = x.detach().cpu().contiguous().view(torch.uint8).numpy()
    return _as(np.asarray(x).view(np.uint8), np.uint8)


def sda_decode_fp8(q_bits, kv_codes, kv_scale, kv_indices, kv_indptr, attn_sink, softmax_scale,
                   tokens=None, lib=None) -> np.ndarray:
    """fp64 sparse sink decode attention over an FP8 pool.

    Row s, element d of the pool is e4m3(kv_codes[s, d]) * kv_scale[s];
    otherwise as sda_decode.  q_bits [N,H,D] bf16 bits, kv_codes [P,D] uint8
    E4M3 codes, kv_scale [P] fp32.
    """
    lib = lib or load()
    q = _as(q_bits, np.uint16)
    kv = _as(kv_codes, np.uint8)
    sc = _as(kv_scale, np.float32)
    N, H, D = q.shape
    assert kv.ndim == 2 and kv.shape[1] == D and sc.shape == (kv.shape[0],)
    idx = _as(kv_indices, np.int32)
    ptr = _as(kv_indptr, np.int32)
    sink = _as(attn_sink, np.float32)
    assert ptr.shape == (N + 1,) and sink.shape == (H,)
    if tokens is None:
        tok = None
        n_tok = N
    else:
        tok = _as(tokens, np.int32)
        n_tok = int(tok.size)
    out = np.zeros((n_tok, H, D), dtype=np.float64)
    idx_arg = idx if idx.size else np.zeros(1, np.int32)
    rc = lib.oracle_sda_decode_fp8(_ptr(q, ctypes.c_uint16), _ptr(kv, ctypes.c_uint8),
                                   _ptr(sc, ctypes.c_float), kv.shape[0],
                                   _ptr(idx_arg, ctypes.c_int32), idx.size,
                                   _ptr(ptr, ctypes.c_int32), _ptr(sink, ctypes.c_float),
                                   float(np.float32(softmax_scale)), N, H, D,
                                   None if tok is None else _ptr(tok, ctypes.c_int32), n_tok,
                                   _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle_sda_decode_fp8: {_ERRORS.get(rc, rc)}")
    return out


def build_indices(state_slot, swa_len, swa_head, comp_indptr, comp_block, comp_slot, win,
                  k_per_block, swa_pages, total_pages, capacity=None, lib=None):
    """Reference index builder.  Returns (kv_indices[:indptr[N]], kv_indptr, status)."""
    lib = lib or load()
    ss = _as(state_slot, np.int32)
    N = int(ss.size)
    sl = _as(swa_len, np.int32)
    sh = _as(swa_head, np.int32)
    cp = _as(comp_indptr, np.int32)
    cb = _as(comp_block, np.int32)
    cs = _as(comp_slot, np.int32)
    assert cb.size == cs.size and cp.size == N + 1
    if capacity is None:
        capacity = N * int(win) + int(cb.size)
    out = np.full(max(int(capacity), 1), -1, dtype=np.int32)
    ptr = np.zeros(N + 1, dtype=np.int32)
    st = np.zeros(1, dtype=np.int32)
    one = np.zeros(1, np.int32)
    rc = lib.oracle_build_indices(
        _ptr(ss if N else one, ctypes.c_int32), _ptr(sl if N else one, ctypes.c_int32),
        _ptr(sh if N else one, ctypes.c_int32), _ptr(cp, ctypes.c_int32),
        _ptr(cb if cb.size else one, ctypes.c_int32), _ptr(cs if cs.size else one, ctypes.c_int32),
        cb.size, N, int(win), int(k_per_block), int(swa_pages), int(total_pages),
        _ptr(out, ctypes.c_int32), int(capacity), _ptr(ptr, ctypes.c_int32),
        _ptr(st, ctypes.c_int32))
    if rc != 0:
        raise ValueError(f"oracle_build_indices: {_ERRORS.get(rc, rc)}")
    return out[: ptr[N]].copy(), ptr, int(st[0])


def validate_indices(kv_indices, kv_indptr, total_pages, lib=None):
    """Reference index validation.  Returns (flags, n_bad_slots)."""
    lib = lib or load()
    idx = _as(kv_indices, np.int32)
    ptr = _as(kv_indptr, np.int32)
    st = np.zeros(2, dtype=np.int32)
    one = np.zeros(1, np.int32)
    rc = lib.oracle_validate_indices(_ptr(idx if idx.size else one, ctypes.c_int32), idx.size,
                                     _ptr(ptr, ctypes.c_int32), ptr.size - 1, int(total_pages),
                                     _ptr(st, ctypes.c_int32))
    if rc != 0:
        raise ValueError(f"oracle_validate_indices: {_ERRORS.get(rc, rc)}")
    return int(st[0]), int(st[1])


def qk_norm_rope_store(q_bits, kv_bits, q_norm_w_bits, kv_norm_w_bits, cos_cache, sin_cache,
                       positions, state_slot, eps, win, swa_pages, lib=None) -> dict:
    """fp64 fused q/kv RMSNorm + GPT-J RoPE (last R dims) + SWA ring slot.

    q_bits [N,H,D], kv_bits [N,D], weights [D]: bf16 bits; cos_cache and
    sin_cache [max_pos, R/2] fp32; positions, state_slot [N] int32.  Returns
    ``q_val`` [N,H,D] and ``kv_val`` [N,D] (exact results, float64), ``slot``
    [N] int64 (pool row of the KV store, -1 if none) and ``status``.
    """
    lib = lib or load()
    q = _as(q_bits, np.uint16)
    kv = _as(kv_bits, np.uint16)
    N, H, D = q.shape
    assert kv.shape == (N, D)
    qw = _as(q_norm_w_bits, np.uint16)
    kw = _as(kv_norm_w_bits, np.uint16)
    assert qw.shape == (D,) and kw.shape == (D,)
    cs = _as(cos_cache, np.float32)
    sn = _as(sin_cache, np.float32)
    assert cs.ndim == 2 and cs.shape == sn.shape
    max_pos, half = cs.shape
    pos = _as(positions, np.int32)
    ss = _as(state_slot, np.int32)
    assert pos.shape == (N,) and ss.shape == (N,)
    q_val = np.zeros((N, H, D), np.float64)
    kv_val = np.zeros((N, D), np.float64)
    slot = np.full(max(N, 1), -1, np.int64)
    st = np.zeros(1, np.int32)
    one16 = np.zeros(1, np.uint16)
    one32 = np.zeros(1, np.int32)
    onef = np.zeros(1, np.float32)
    rc = lib.oracle_qk_norm_rope_store(
        _ptr(q if N else one16, ctypes.c_uint16), _ptr(kv if N else one16, ctypes.c_uint16),
        _ptr(qw, ctypes.c_uint16), _ptr(kw, ctypes.c_uint16),
        _ptr(cs if cs.size else onef, ctypes.c_float), _ptr(sn if sn.size else onef, ctypes.c_float),
        max_pos, _ptr(pos if N else one32, ctypes.c_int32), _ptr(ss if N else one32, ctypes.c_int32),
        N, H, D, 2 * half, float(np.float32(eps)), int(win), int(swa_pages),
        _ptr(q_val if N else np.zeros(1), ctypes.c_double),
        _ptr(kv_val if N else np.zeros(1), ctypes.c_double), _ptr(slot, ctypes.c_int64),
        _ptr(st, ctypes.c_int32))
    if rc != 0:
        raise ValueError(f"oracle_qk_norm_rope_store: {_ERRORS.get(rc, rc)}")
    return {"q_val": q_val, "kv_val": kv_val, "slot": slot[:N].copy(), "status": int(st[0])}


def bf16_rne(values, lib=None) -> np.ndarray:
    """bf16 bit patterns of float64 values rounded to nearest even."""
    lib = lib or load()
    v = _as(values, np.float64)
    out = np.zeros(v.shape, np.uint16)
    if v.size:
        lib.oracle_bf16_rne_array(_ptr(v, ctypes.c_double), v.size, _ptr(out, ctypes.c_uint16))
    return out


def e4m3_rne(value, lib=None) -> int:
    """E4M3 code of one float64 value rounded to nearest even (saturating)."""
    return int((lib or load()).oracle_e4m3_rne(float(value)))


def e4m3_rne_array(values, lib=None) -> np.ndarray:
    """E4M3 codes of float64 values rounded to nearest even (saturating)."""
    lib = lib or load()
    v = _as(values, np.float64)
    out = np.zeros(v.shape, np.uint8)
    if v.size:
        lib.oracle_e4m3_rne_array(_ptr(v, ctypes.c_double), v.size, _ptr(out, ctypes.c_uint8))
    return out


def fp8_scale_exponent(amax, lib=None) -> int:
    """e of the power-of-two row scale 2^e: the smallest e with 448 * 2^e >= amax."""
    return int((lib or load()).oracle_fp8_scale_exponent(float(amax)))


def fp8_quantise_rows(values, lib=None):
    """(codes [rows, D] uint8, scale [rows] fp32) of float64 rows [rows, D]."""
    lib = lib or load()
    v = _as(values, np.float64)
    rows, D = v.shape
    codes = np.zeros((rows, D), np.uint8)
    scale = np.zeros(rows, np.float32)
    if rows:
        lib.oracle_fp8_quantise_rows(_ptr(v, ctypes.c_double), rows, D,
                                     _ptr(codes, ctypes.c_uint8), _ptr(scale, ctypes.c_float))
    return codes, scale


def topk_slots(scores, lengths, block_table, k, k_per_block, lib=None):
    """Reference top-k -> (comp_indptr [N+1], comp_block, comp_slot, status).

    scores [N, S] fp32 (token t's candidates are scores[t, :lengths[t]]),
    lengths [N] int32, block_table [N, B] int32 with B * k_per_block >= S."""
    lib = lib or load()
    sc = _as(scores, np.float32)
    N, S = sc.shape
    ln = _as(lengths, np.int32)
    bt = _as(block_table, np.int32)
    assert ln.shape == (N,) and bt.ndim == 2 and bt.shape[0] == N
    cap = max(1, N * int(k))  # room for k per token whatever the lengths say
    ptr = np.zeros(N + 1, np.int32)
    blk = np.zeros(cap, np.int32)
    slot = np.zeros(cap, np.int32)
    st = np.zeros(1, np.int32)
    one_f = np.zeros(1, np.float32)
    one_i = np.zeros(1, np.int32)
    rc = lib.oracle_topk_slots(_ptr(sc if sc.size else one_f, ctypes.c_float), S,
                               _ptr(ln if N else one_i, ctypes.c_int32),
                               _ptr(bt if bt.size else one_i, ctypes.c_int32), bt.shape[1], N,
                               int(k), int(k_per_block), _ptr(ptr, ctypes.c_int32),
                               _ptr(blk, ctypes.c_int32), _ptr(slot, ctypes.c_int32),
                               _ptr(st, ctypes.c_int32))
    if rc != 0:
        raise ValueError(f"oracle_topk_slots: {_ERRORS.get(rc, rc)}")
    return ptr, blk[: ptr[N]].copy(), slot[: ptr[N]].copy(), int(st[0])
