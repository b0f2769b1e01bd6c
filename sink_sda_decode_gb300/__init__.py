"""Sparse decode attention with an attention sink over a unified KV pool (GB300).

Thin Python binding of the C ABI in include/sda.h (libsda.so, built in this
package directory).  The functions only check and marshal arguments: torch is
used for device memory and streams, and every step of the computation runs in
the library's CUDA kernels.  There is no CPU or PyTorch fallback; calling
without the built library raises.

    out = decode(q, unified_kv, kv_indices, kv_indptr, attn_sink, softmax_scale)

computes, for every token t and head h, attention of q[t, h] over the rows
unified_kv[kv_indices[kv_indptr[t]:kv_indptr[t+1]]] (each row is key and
value), with attn_sink[h] as a key of value zero; see decode() for details.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

__all__ = ["decode", "workspace_size", "build_indices", "validate_indices", "decode_error_flag",
           "decode_kernel", "decode_fp8", "workspace_size_fp8", "qk_norm_rope_swa_store", "topk_slots", "build_decode",
           "build_decode_host", "build_decode_host_workspace_size",
           "decode_host", "set_timing_events", "decode_noalloc", "library_path"]

library_path = _lib.LIB_PATH


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _workspace_for(nbytes: int, dev, stream) -> torch.Tensor:
    """A workspace from torch's caching allocator that the allocator knows is
    in use on `stream` (the stream the kernels run on), so that the block is
    not handed out again while those kernels may still touch it."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=dev)
    if isinstance(stream, torch.cuda.Stream):
        ws.record_stream(stream)
    return ws


def _req(t: torch.Tensor, name: str, dtype, ndim=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_size(N: int, H: int, D: int, total_indices: int) -> int:
    """Bytes of workspace decode() needs on the current CUDA device."""
    lib = _lib.load()
    n = ctypes.c_size_t(0)
    _lib.check(lib.sda_decode_workspace_size(int(N), int(H), int(D), int(total_indices),
                                             ctypes.byref(n)), "sda_decode_workspace_size")
    return int(n.value)


def decode(q: torch.Tensor, unified_kv: torch.Tensor, kv_indices: torch.Tensor,
           kv_indptr: torch.Tensor, attn_sink: torch.Tensor, softmax_scale: float,
           out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
           stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Sparse sink decode attention (paged_decode.py docstring semantics).

    q [N, H, D] bf16; unified_kv [P, D] bf16 (one row = key and value of a
    slot); kv_indices int32 (every listed entry must be a valid slot);
    kv_indptr [N + 1] int32 (empty slice = padded token -> out 0); attn_sink
    [H] fp32 sink logits; returns out [N, H, D] bf16.  `workspace` (uint8,
    >= workspace_size(...) bytes) may be passed to keep the call free of
    allocations, e.g. for CUDA-graph capture.  Asynchronous on `stream`.
    """
    lib = _lib.load()
    _req(q, "q", torch.bfloat16, 3)
    dev = q.device
    _req(unified_kv, "unified_kv", torch.bfloat16, 2, dev)
    _req(kv_indices, "kv_indices", torch.int32, 1, dev)
    _req(kv_indptr, "kv_indptr", torch.int32, 1, dev)
    _req(attn_sink, "attn_sink", torch.float32, 1, dev)
    N, H, D = q.shape
    if unified_kv.shape[1] != D:
        raise ValueError("unified_kv row length must equal q's head dim")
    if kv_indptr.numel() != N + 1 or attn_sink.numel() != H:
        raise ValueError("kv_indptr must have N+1 entries and attn_sink H entries")
    if out is None:
        out = torch.empty_like(q)
    else:
        _req(out, "out", torch.bfloat16, 3, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    with torch.cuda.device(dev):
        need = workspace_size(N, H, D, kv_indices.numel())
        if workspace is None:
            workspace = _workspace_for(need, dev, stream)
        else:
            _req(workspace, "workspace", torch.uint8, 1, dev)
        rc = lib.sda_decode(q.data_ptr(), unified_kv.data_ptr(), unified_kv.shape[0],
                            kv_indices.data_ptr() if kv_indices.numel() else None,
                            kv_indices.numel(), kv_indptr.data_ptr(), attn_sink.data_ptr(),
                            float(softmax_scale), N, H, D, out.data_ptr(), workspace.data_ptr(),
                            workspace.numel(), _stream_ptr(stream))
    _lib.check(rc, "sda_decode")
    return out


def workspace_size_fp8(N: int, H: int, D: int, total_indices: int) -> int:
    """Bytes of workspace decode_fp8() needs on the current CUDA device."""
    lib = _lib.load()
    n = ctypes.c_size_t(0)
    _lib.check(lib.sda_decode_fp8_workspace_size(int(N), int(H), int(D), int(total_indices),
                                                 ctypes.byref(n)), "sda_decode_fp8_workspace_size")
    return int(n.value)


def decode_fp8(q: torch.Tensor, kv_fp8: torch.Tensor, kv_scale: torch.Tensor,
               kv_indices: torch.Tensor, kv_indptr: torch.Tensor, attn_sink: torch.Tensor,
               softmax_scale: float, out: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None,
               stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """decode() over a pool stored in FP8: row s of the pool is
    e4m3(kv_fp8[s]) * kv_scale[s].

    kv_fp8 [P, D] float8_e4m3fn (or uint8 holding E4M3 codes); kv_scale [P]
    fp32; the other arguments and the result as decode().  D = 512 with
    H in {16, 32} or a multiple of 64 up to 256.
    """
    lib = _lib.load()
    _req(q, "q", torch.bfloat16, 3)
    dev = q.device
    if kv_fp8.dtype == torch.float8_e4m3fn:
        kv_fp8 = kv_fp8.view(torch.uint8)
    _req(kv_fp8, "kv_fp8", torch.uint8, 2, dev)
    _req(kv_scale, "kv_scale", torch.float32, 1, dev)
    _req(kv_indices, "kv_indices", torch.int32, 1, dev)
    _req(kv_indptr, "kv_indptr", torch.int32, 1, dev)
    _req(attn_sink, "attn_sink", torch.float32, 1, dev)
    N, H, D = q.shape
    if kv_fp8.shape[1] != D or kv_scale.numel() != kv_fp8.shape[0]:
        raise ValueError("kv_fp8 rows must have q's head dim and kv_scale one entry per row")
    if kv_indptr.numel() != N + 1 or attn_sink.numel() != H:
        raise ValueError("kv_indptr must have N+1 entries and attn_sink H entries")
    if out is None:
        out = torch.empty_like(q)
    else:
        _req(out, "out", torch.bfloat16, 3, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    with torch.cuda.device(dev):
        need = workspace_size_fp8(N, H, D, kv_indices.numel())
        if workspace is None:
            workspace = _workspace_for(need, dev, stream)
        else:
            _req(workspace, "workspace", torch.uint8, 1, dev)
        rc = lib.sda_decode_fp8(q.data_ptr(), kv_fp8.data_ptr(), kv_scale.data_ptr(),
                                kv_fp8.shape[0],
                                kv_indices.data_ptr() if kv_indices.numel() else None,
                                kv_indices.numel(), kv_indptr.data_ptr(), attn_sink.data_ptr(),
                                float(softmax_scale), N, H, D, out.data_ptr(), workspace.data_ptr(),
                                workspace.numel(), _stream_ptr(stream))
    _lib.check(rc, "sda_decode_fp8")
    return out


def decode_noalloc(q: torch.Tensor, unified_kv: torch.Tensor, kv_indices: torch.Tensor,
                   kv_indptr: torch.Tensor, attn_sink: torch.Tensor, softmax_scale: float,
                   out: torch.Tensor, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """decode() for callers that may not allocate device memory: `out` must be
    given, and the scratch memory is the library's fixed 16 MiB device array
    (calls that would need more raise; overlapping calls on the GPU race on
    the shared array).  Asynchronous on `stream`."""
    lib = _lib.load()
    _req(q, "q", torch.bfloat16, 3)
    dev = q.device
    _req(unified_kv, "unified_kv", torch.bfloat16, 2, dev)
    _req(kv_indices, "kv_indices", torch.int32, 1, dev)
    _req(kv_indptr, "kv_indptr", torch.int32, 1, dev)
    _req(attn_sink, "attn_sink", torch.float32, 1, dev)
    _req(out, "out", torch.bfloat16, 3, dev)
    N, H, D = q.shape
    if out.shape != q.shape or kv_indptr.numel() != N + 1 or attn_sink.numel() != H:
        raise ValueError("shape mismatch")
    with torch.cuda.device(dev):
        rc = lib.sda_decode_noalloc(q.data_ptr(), unified_kv.data_ptr(), unified_kv.shape[0],
                                    kv_indices.data_ptr() if kv_indices.numel() else None,
                                    kv_indices.numel(), kv_indptr.data_ptr(), attn_sink.data_ptr(),
                                    float(softmax_scale), N, H, D, out.data_ptr(),
                                    _stream_ptr(stream))
    _lib.check(rc, "sda_decode_noalloc")
    return out


KERNEL_NAMES = {0: "simt", 1: "one_cta"}


def decode_kernel(H: int, D: int, device=None) -> str:
    """Name of the attention kernel decode() launches for (H, D) on `device`
    ("simt" or "one_cta")."""
    lib = _lib.load()
    k = ctypes.c_int(-1)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _lib.check(lib.sda_decode_kernel(H, D, ctypes.byref(k)), "sda_decode_kernel")
    return KERNEL_NAMES[k.value]


def decode_error_flag(workspace: torch.Tensor, stream=None) -> int:
    """Device error word of the last decode() on `workspace` (synchronises).

    0 = fine; 1 = a pipeline wait timed out; 2 = kv_indptr was not a prefix
    sum inside [0, len(kv_indices)] (nothing was computed)."""
    lib = _lib.load()
    flag = torch.zeros(1, dtype=torch.int32, device=workspace.device)
    with torch.cuda.device(workspace.device):
        _lib.check(lib.sda_decode_error_flag(workspace.data_ptr(), flag.data_ptr(),
                                             _stream_ptr(stream)), "sda_decode_error_flag")
    return int(flag.item())


def debug_wait_fault(withhold_arrive: bool, timeout_ns: int = 0) -> None:
    """Test hook of the tensor-core kernels' bounded waits: every later launch
    bounds each pipeline wait by `timeout_ns` (0 = the default 2 s) and, with
    withhold_arrive, CTA 0's first loader warp skips one arrive so that a wait
    runs out (the error word then reads 1).  Reset with (False, 0)."""
    lib = _lib.load()
    _lib.check(lib.sda_debug_wait_fault(1 if withhold_arrive else 0, int(timeout_ns)),
               "sda_debug_wait_fault")


def set_timing_events(before: torch.cuda.Event | None, after: torch.cuda.Event | None) -> None:
    """Record `before` / `after` around the attention kernel of every later
    decode() / decode_fp8() and around the kernel of every later
    qk_norm_rope_swa_store() / topk_slots() on this thread (None, None turns
    it off).
    Events must be created with enable_timing=True."""
    lib = _lib.load()
    handles = []
    for ev in (before, after):
        if ev is None:
            handles.append(None)
            continue
        if not ev.cuda_event:  # torch creates the CUDA event on its first record()
            ev.record()
        if not ev.cuda_event:
            raise ValueError("could not create the CUDA event")
        handles.append(ev.cuda_event)
    _lib.check(lib.sda_set_timing_events(handles[0], handles[1]), "sda_set_timing_events")


def build_indices(state_slot, swa_len, swa_head, comp_indptr, comp_block, comp_slot, *, win,
                  k_per_block, swa_pages, total_pages, capacity=None, kv_indices=None,
                  kv_indptr=None, status=None, stream=None):
    """Pack SWA ring slots and compressed slots into ragged kv_indices.

    Returns (kv_indices [capacity], kv_indptr [N+1], status [1]) int32 device
    tensors; status bits are documented in include/sda.h (0 = all fine)."""
    lib = _lib.load()
    _req(state_slot, "state_slot", torch.int32, 1)
    dev = state_slot.device
    for name, t in (("swa_len", swa_len), ("swa_head", swa_head), ("comp_indptr", comp_indptr),
                    ("comp_block", comp_block), ("comp_slot", comp_slot)):
        _req(t, name, torch.int32, 1, dev)
    N = state_slot.numel()
    if capacity is None:
        capacity = N * int(win) + comp_block.numel()
    if kv_indices is None:
        kv_indices = torch.empty(max(int(capacity), 1), dtype=torch.int32, device=dev)
    if kv_indptr is None:
        kv_indptr = torch.empty(N + 1, dtype=torch.int32, device=dev)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        rc = lib.sda_build_indices(
            state_slot.data_ptr(), swa_len.data_ptr(), swa_head.data_ptr(), comp_indptr.data_ptr(),
            comp_block.data_ptr() if comp_block.numel() else None,
            comp_slot.data_ptr() if comp_slot.numel() else None, comp_block.numel(), N, int(win),
            int(k_per_block), int(swa_pages), int(total_pages), kv_indices.data_ptr(),
            int(capacity), kv_indptr.data_ptr(), status.data_ptr(), _stream_ptr(stream))
    _lib.check(rc, "sda_build_indices")
    return kv_indices, kv_indptr, status


def build_decode(q, unified_kv, attn_sink, softmax_scale, state_slot, swa_len, swa_head,
                 comp_indptr, comp_block, comp_slot, *, win, k_per_block, swa_pages,
                 kv_scale=None, capacity=None, out=None, workspace=None, kv_indices=None,
                 kv_indptr=None, status=None, stream=None):
    """build_indices followed by decode (decode_fp8 when `kv_scale` is given;
    `unified_kv` then holds the E4M3 codes) in one call with one launch fewer.
    Returns (out, kv_indices, kv_indptr, status)."""
    lib = _lib.load()
    _req(q, "q", torch.bfloat16, 3)
    dev = q.device
    N, H, D = q.shape
    if kv_scale is None:
        _req(unified_kv, "unified_kv", torch.bfloat16, 2, dev)
    else:
        if unified_kv.dtype == torch.float8_e4m3fn:
            unified_kv = unified_kv.view(torch.uint8)
        _req(unified_kv, "kv_fp8", torch.uint8, 2, dev)
        _req(kv_scale, "kv_scale", torch.float32, 1, dev)
        if kv_scale.numel() != unified_kv.shape[0]:
            raise ValueError("kv_scale must have one entry per pool row")
    if unified_kv.shape[1] != D:
        raise ValueError("pool rows must have D elements")
    _req(attn_sink, "attn_sink", torch.float32, 1, dev)
    _req(state_slot, "state_slot", torch.int32, 1, dev)
    for name, t in (("swa_len", swa_len), ("swa_head", swa_head), ("comp_indptr", comp_indptr),
                    ("comp_block", comp_block), ("comp_slot", comp_slot)):
        _req(t, name, torch.int32, 1, dev)
    if state_slot.numel() != N or attn_sink.numel() != H:
        raise ValueError("state_slot must be [N] and attn_sink [H]")
    if capacity is None:
        capacity = N * int(win) + comp_block.numel()
    if kv_indices is None:
        kv_indices = torch.empty(max(int(capacity), 1), dtype=torch.int32, device=dev)
    if kv_indptr is None:
        kv_indptr = torch.empty(N + 1, dtype=torch.int32, device=dev)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        size = (workspace_size if kv_scale is None else workspace_size_fp8)(N, H, D, int(capacity))
        workspace = _workspace_for(size, dev, stream)
    with torch.cuda.device(dev):
        rc = lib.sda_build_decode(
            state_slot.data_ptr(), swa_len.data_ptr(), swa_head.data_ptr(), comp_indptr.data_ptr(),
            comp_block.data_ptr() if comp_block.numel() else None,
            comp_slot.data_ptr() if comp_slot.numel() else None, comp_block.numel(), int(win),
            int(k_per_block), int(swa_pages), kv_indices.data_ptr(), int(capacity),
            kv_indptr.data_ptr(), status.data_ptr(), q.data_ptr(), unified_kv.data_ptr(),
            None if kv_scale is None else kv_scale.data_ptr(), unified_kv.shape[0],
            attn_sink.data_ptr(), float(softmax_scale), N, H, D, out.data_ptr(),
            workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    _lib.check(rc, "sda_build_decode")
    return out, kv_indices, kv_indptr, status


def build_decode_host_workspace_size(N, H, D, comp_total, capacity, fp8=False) -> int:
    """Device workspace bytes build_decode_host needs."""
    lib = _lib.load()
    n = ctypes.c_size_t(0)
    _lib.check(lib.sda_build_decode_host_workspace_size(int(N), int(H), int(D), int(comp_total),
                                                        int(capacity), int(bool(fp8)),
                                                        ctypes.byref(n)),
               "sda_build_decode_host_workspace_size")
    return int(n.value)


def build_decode_host(q, unified_kv, attn_sink, softmax_scale, state_slot, swa_len, swa_head,
                      comp_indptr, comp_block, comp_slot, *, win, k_per_block, swa_pages,
                      kv_scale=None, capacity=None, out=None, status=None, workspace=None,
                      stream=None):
    """build_decode from page-locked HOST tensors (q, the descriptors, and the
    outputs out / status): kernels read the inputs from host memory and write
    the result back, with no copy-engine transfer.  The pool and attn_sink stay
    on the device.  Asynchronous on `stream`; returns (out, status) host
    tensors, valid once the stream has reached this call.  The caller must
    keep every host tensor passed in alive (and pinned) until then: the
    kernels read and write them after this function returns."""
    lib = _lib.load()

    def kind(t, name, dtype, ndim):
        if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.dim() != ndim:
            raise TypeError(f"{name} must be a {ndim}-d {dtype} tensor")

    def host(t, name, dtype, ndim):
        kind(t, name, dtype, ndim)
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous page-locked (pinned) host tensor")
    descriptors = (("state_slot", state_slot), ("swa_len", swa_len), ("swa_head", swa_head),
                   ("comp_indptr", comp_indptr), ("comp_block", comp_block),
                   ("comp_slot", comp_slot))
    kind(q, "q", torch.bfloat16, 3)
    N, H, D = q.shape
    for name, t in descriptors:
        kind(t, name, torch.int32, 1)
    # the kernels trust these extents: check every one (host memory is reached
    # over the chip-to-chip link, and an undersized buffer would be read past)
    if state_slot.numel() != N or swa_len.numel() != N or swa_head.numel() != N:
        raise ValueError("state_slot, swa_len and swa_head must have N entries")
    if comp_indptr.numel() != N + 1:
        raise ValueError("comp_indptr must have N + 1 entries")
    if comp_block.numel() != comp_slot.numel():
        raise ValueError("comp_block and comp_slot must have the same length")
    if out is not None:
        kind(out, "out", torch.bfloat16, 3)
        if tuple(out.shape) != (N, H, D):
            raise ValueError("out must have q's shape")
    if status is not None:
        kind(status, "status", torch.int32, 1)
        if status.numel() < 1:
            raise ValueError("status must hold one int32")
    host(q, "q", torch.bfloat16, 3)
    for name, t in descriptors:
        host(t, name, torch.int32, 1)
    if not isinstance(unified_kv, torch.Tensor):
        raise TypeError("unified_kv must be a torch.Tensor")
    dev = unified_kv.device
    if kv_scale is None:
        _req(unified_kv, "unified_kv", torch.bfloat16, 2, dev)
    else:
        if unified_kv.dtype == torch.float8_e4m3fn:
            unified_kv = unified_kv.view(torch.uint8)
        _req(unified_kv, "kv_fp8", torch.uint8, 2, dev)
        _req(kv_scale, "kv_scale", torch.float32, 1, dev)
        if kv_scale.numel() != unified_kv.shape[0]:
            raise ValueError("kv_scale must have one entry per pool row")
    if unified_kv.shape[1] != D:
        raise ValueError("pool rows must have D elements")
    _req(attn_sink, "attn_sink", torch.float32, 1, dev)
    if attn_sink.numel() != H:
        raise ValueError("attn_sink must have H entries")
    if capacity is None:
        capacity = N * int(win) + comp_block.numel()
    if out is None:
        out = torch.empty((N, H, D), dtype=torch.bfloat16, pin_memory=True)
    else:
        host(out, "out", torch.bfloat16, 3)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, pin_memory=True)
    else:
        host(status, "status", torch.int32, 1)
    if workspace is None:
        with torch.cuda.device(dev):
            size = build_decode_host_workspace_size(N, H, D, comp_block.numel(), capacity,
                                                    kv_scale is not None)
        workspace = _workspace_for(size, dev, stream)
    with torch.cuda.device(dev):
        rc = lib.sda_build_decode_host(
            state_slot.data_ptr() if N else None, swa_len.data_ptr() if N else None,
            swa_head.data_ptr() if N else None, comp_indptr.data_ptr(),
            comp_block.data_ptr() if comp_block.numel() else None,
            comp_slot.data_ptr() if comp_slot.numel() else None, comp_block.numel(), int(win),
            int(k_per_block), int(swa_pages), int(capacity), q.data_ptr() if N else None,
            unified_kv.data_ptr(), None if kv_scale is None else kv_scale.data_ptr(),
            unified_kv.shape[0], attn_sink.data_ptr(), float(softmax_scale), N, H, D,
            out.data_ptr() if N else None, status.data_ptr(), workspace.data_ptr(),
            workspace.numel(), _stream_ptr(stream))
    _lib.check(rc, "sda_build_decode_host")
    return out, status


def validate_indices(kv_indices, kv_indptr, total_pages, status=None, stream=None):
    """Device check of the index contract; returns status [2] int32 (flags, n_bad)."""
    lib = _lib.load()
    _req(kv_indptr, "kv_indptr", torch.int32, 1)
    dev = kv_indptr.device
    _req(kv_indices, "kv_indices", torch.int32, 1, dev)
    if status is None:
        status = torch.empty(2, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        rc = lib.sda_validate_indices(kv_indices.data_ptr() if kv_indices.numel() else None,
                                      kv_indices.numel(), kv_indptr.data_ptr(),
                                      kv_indptr.numel() - 1, int(total_pages), status.data_ptr(),
                                      _stream_ptr(stream))
    _lib.check(rc, "sda_validate_indices")
    return status


def topk_slots(scores, lengths, block_table, *, k, k_per_block, capacity=None, comp_indptr=None,
               comp_block=None, comp_slot=None, status=None, stream=None):
    """Per token, the k best of scores[t, :lengths[t]] (NaN below -inf, ties by
    position), in increasing position, as (block, slot in block) pairs through
    block_table [N, B]: the comp_indptr / comp_block / comp_slot inputs of
    build_indices.  Returns (comp_indptr [N+1], comp_block [capacity],
    comp_slot [capacity], status [1]) int32 device tensors."""
    lib = _lib.load()
    _req(scores, "scores", torch.float32, 2)
    dev = scores.device
    _req(lengths, "lengths", torch.int32, 1, dev)
    _req(block_table, "block_table", torch.int32, 2, dev)
    N, S = scores.shape
    if lengths.numel() != N or block_table.shape[0] != N:
        raise ValueError("lengths must be [N] and block_table [N, B]")
    if capacity is None:
        capacity = N * int(k)
    if comp_indptr is None:
        comp_indptr = torch.empty(N + 1, dtype=torch.int32, device=dev)
    if comp_block is None:
        comp_block = torch.empty(max(int(capacity), 1), dtype=torch.int32, device=dev)
    if comp_slot is None:
        comp_slot = torch.empty(max(int(capacity), 1), dtype=torch.int32, device=dev)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        rc = lib.sda_topk_slots(scores.data_ptr() if scores.numel() else None, S,
                                lengths.data_ptr() if N else None,
                                block_table.data_ptr() if block_table.numel() else None,
                                block_table.shape[1], N, int(k), int(k_per_block),
                                comp_indptr.data_ptr(), comp_block.data_ptr(),
                                comp_slot.data_ptr(), int(capacity), status.data_ptr(),
                                _stream_ptr(stream))
    _lib.check(rc, "sda_topk_slots")
    return comp_indptr, comp_block, comp_slot, status


def qk_norm_rope_swa_store(q, kv, q_norm_w, kv_norm_w, cos_cache, sin_cache, positions,
                           state_slot, *, eps, win, swa_pages, unified_kv=None, kv_fp8=None,
                           kv_scale=None, q_out=None, status=None, stream=None):
    """Per-head RMSNorm of q and RMSNorm of the new KV rows, GPT-J RoPE on the
    last cos_cache.shape[1] * 2 dims, and the store of each token's KV row into
    its ring slot state_slot * win + position mod win of the pool: bf16
    (`unified_kv`) or E4M3 codes + power-of-two row scales (`kv_fp8`,
    `kv_scale`).  Returns (q_out [N, H, D] bf16, status [1] int32); the status
    bits are documented in include/sda.h.  `q_out` may be `q` (in place)."""
    lib = _lib.load()
    _req(q, "q", torch.bfloat16, 3)
    dev = q.device
    N, H, D = q.shape
    _req(kv, "kv", torch.bfloat16, 2, dev)
    _req(q_norm_w, "q_norm_w", torch.bfloat16, 1, dev)
    _req(kv_norm_w, "kv_norm_w", torch.bfloat16, 1, dev)
    _req(cos_cache, "cos_cache", torch.float32, 2, dev)
    _req(sin_cache, "sin_cache", torch.float32, 2, dev)
    _req(positions, "positions", torch.int32, 1, dev)
    _req(state_slot, "state_slot", torch.int32, 1, dev)
    if kv.shape != (N, D) or q_norm_w.numel() != D or kv_norm_w.numel() != D:
        raise ValueError("kv must be [N, D] and the norm weights [D]")
    if cos_cache.shape != sin_cache.shape or positions.numel() != N or state_slot.numel() != N:
        raise ValueError("cos_cache / sin_cache must match; positions, state_slot must be [N]")
    max_pos, half = cos_cache.shape
    if (unified_kv is None) == (kv_fp8 is None):
        raise ValueError("pass exactly one of unified_kv (bf16 pool) or kv_fp8 + kv_scale")
    if unified_kv is not None:
        _req(unified_kv, "unified_kv", torch.bfloat16, 2, dev)
        total_pages = unified_kv.shape[0]
        if unified_kv.shape[1] != D:
            raise ValueError("unified_kv must be [total_pages, D]")
    else:
        if kv_fp8.dtype == torch.float8_e4m3fn:
            kv_fp8 = kv_fp8.view(torch.uint8)
        _req(kv_fp8, "kv_fp8", torch.uint8, 2, dev)
        _req(kv_scale, "kv_scale", torch.float32, 1, dev)
        total_pages = kv_fp8.shape[0]
        if kv_fp8.shape[1] != D or kv_scale.numel() != total_pages:
            raise ValueError("kv_fp8 must be [total_pages, D] and kv_scale [total_pages]")
    if q_out is None:
        q_out = torch.empty_like(q)
    else:
        _req(q_out, "q_out", torch.bfloat16, 3, dev)
        if q_out.shape != q.shape:
            raise ValueError("q_out must have q's shape")
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    common = (q.data_ptr(), kv.data_ptr(), q_norm_w.data_ptr(), kv_norm_w.data_ptr(),
              cos_cache.data_ptr() if cos_cache.numel() else None,
              sin_cache.data_ptr() if sin_cache.numel() else None, int(max_pos),
              positions.data_ptr(), state_slot.data_ptr(), N, H, D, 2 * int(half),
              float(eps), int(win), int(swa_pages), int(total_pages), q_out.data_ptr())
    with torch.cuda.device(dev):
        if unified_kv is not None:
            rc = lib.sda_qk_norm_rope_swa_store(*common, unified_kv.data_ptr(), status.data_ptr(),
                                                _stream_ptr(stream))
        else:
            rc = lib.sda_qk_norm_rope_swa_store_fp8(*common, kv_fp8.data_ptr(),
                                                    kv_scale.data_ptr(), status.data_ptr(),
                                                    _stream_ptr(stream))
    _lib.check(rc, "sda_qk_norm_rope_swa_store")
    return q_out, status


def decode_host(q_host: torch.Tensor, unified_kv: torch.Tensor, kv_indices_host: torch.Tensor,
                kv_indptr_host: torch.Tensor, attn_sink: torch.Tensor, softmax_scale: float,
                out_host: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """End-to-end call from host buffers: copies q and the index lists to the
    device (pinned host memory -> async copies), runs decode on the resident
    pool and copies out back to the host.  Synchronises the stream."""
    dev = unified_kv.device
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.stream(s):
        q = q_host.to(dev, non_blocking=True)
        idx = kv_indices_host.to(dev, non_blocking=True)
        ptr = kv_indptr_host.to(dev, non_blocking=True)
        out = decode(q, unified_kv, idx, ptr, attn_sink, softmax_scale, stream=s)
        if out_host is None:
            out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        out_host.copy_(out, non_blocking=True)
    s.synchronize()
    return out_host
