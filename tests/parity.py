"""Parity helpers shared by the GPU tests: run the CUDA path, run the oracle
on the same inputs, compare element by element.

Tolerance (stated for unit-normal q and kv, the workloads' distribution):
max |gpu - ref| <= 8e-3 and mean |gpu - ref| <= 1e-3 against the fp64
oracle.  The output is bf16, whose half-ULP is 2^-8 * 2^e: for |ref| >= 4
correct round-to-nearest-even alone can exceed 8e-3, so an element also
passes if it is within one bf16 ULP of ref (the rounding-aware bound); the
raw violations are counted and reported separately.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import sink_sda_decode_gb300 as sda

MAX_ABS = 8e-3
MEAN_ABS = 1e-3


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def compare(gpu: torch.Tensor, ref: np.ndarray) -> dict:
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    allowed = np.maximum(MAX_ABS, bf16_ulp(ref))
    raw = err > MAX_ABS
    return {
        "max_abs": float(err.max()) if err.size else 0.0,
        "mean_abs": float(err.mean()) if err.size else 0.0,
        "n": int(err.size),
        "raw_violations": int(raw.sum()),
        "raw_violation_max_ref": float(np.abs(ref[raw]).min()) if raw.any() else 0.0,
        "rounding_aware_violations": int((err > allowed).sum()),
        "nonfinite": int((~np.isfinite(g)).sum()),
    }


def assert_parity(stats: dict, what: str = ""):
    assert stats["nonfinite"] == 0, (what, stats)
    assert stats["mean_abs"] <= MEAN_ABS, (what, stats)
    assert stats["rounding_aware_violations"] == 0, (what, stats)
    # every raw violation must be an output-rounding case (|ref| >= 2)
    if stats["raw_violations"]:
        assert stats["raw_violation_max_ref"] >= 2.0, (what, stats)


def to_dev(w, device="cuda"):
    idx = torch.from_numpy(np.ascontiguousarray(w.kv_indices, np.int32)).to(device)
    ptr = torch.from_numpy(np.ascontiguousarray(w.kv_indptr, np.int32)).to(device)
    return idx, ptr


def run_gpu(w, idx=None, ptr=None, sink=None, scale=None, out=None):
    if idx is None:
        idx, ptr = to_dev(w)
    return sda.decode(w.q, w.unified_kv, idx, ptr, w.attn_sink if sink is None else sink,
                      w.softmax_scale if scale is None else scale, out=out)


def run_oracle(w, tokens=None, sink=None, scale=None, kv_indices=None, kv_indptr=None):
    """fp64 oracle on the workload's inputs for `tokens` (None = all)."""
    if kv_indices is not None:
        kv_bits = oracle.bf16_bits(w.unified_kv)
        q_bits = w.q_bits()
        return oracle.sda_decode(q_bits, kv_bits, kv_indices, kv_indptr,
                                 (w.attn_sink if sink is None else sink).cpu().numpy(),
                                 w.softmax_scale if scale is None else scale, tokens=tokens)
    kv_bits, sub_idx, sub_ptr = w.kv_rows_for(tokens)
    q_bits = w.q_bits()
    if tokens is not None:
        q_bits = q_bits[np.asarray(tokens)]
    return oracle.sda_decode(q_bits, kv_bits, sub_idx, sub_ptr,
                             (w.attn_sink if sink is None else sink).cpu().numpy(),
                             w.softmax_scale if scale is None else scale)
