"""Benchmark of the sparse sink decode attention hot path on one GB300.

One step = the whole hot path over one batch: the index build (SWA ring
slots + compressed slots -> ragged kv_indices) followed by the decode
(device-side split plan, tensor-core attention kernel, log-sum-exp combine),
made by one sda_build_decode call and replayed as one CUDA graph.

Prints ONE JSON line.  Default workload: N=1024 tokens, H=128, D=512, 640
slots per token (128 SWA ring slots + 512 random compressed slots) over a
2^21-slot pool, the largest of the five decode workloads that fits one GPU.
`--config` picks another workload (the five decode workloads, or a
2048-token sparse-prefill chunk, prefill_h64, through the same path).  The
default decode run also times the five decode workloads one after another
in the same way (`per_config`: tokens/s, attention-kernel time, roofline
fraction) and, in its CPU-baseline leg, compares a bounded token sample of
each with the fp64 oracle (`parity_sample`).

  value     decode tokens/s with inputs resident in HBM (graph replays,
            CUDA events, L2 flushed between steps: a 256 MiB write, then a
            256 MiB read so that the written lines are back in HBM and the
            step pays for none of the flush's write-backs)
  e2e       the same metric through the public API from pinned host
            memory: sda_build_decode_host, replayed as one CUDA graph (small
            batches: kernels read q and the index descriptors from page-
            locked host memory and write out back; batches with >= 8 MB of
            q: token chunks over copy-engine streams, overlapped with the
            decode); other paths: one packed H2D copy in, D2H copies out
  roofline  the attention kernel alone (events recorded around it by the
            library's timing hook): algorithmic bytes / time vs measured HBM;
            also distinct_row_bytes / frac_distinct_rows, each distinct pool
            row counted once (the HBM figure of a prefill chunk, whose tokens
            share most rows)
  cpu_baseline  the fp64 CPU oracle on the host cores (bounded sample)

--path topk times the step in front of the index build: per token, the k
best-scored of its compressed-cache positions, as (block, slot) lists.
--path store times the step that fills the pool instead (per-head RMSNorm of
q, RMSNorm of the new KV row, GPT-J RoPE, store into the SWA ring slot: one
kernel); --path layer times the three calls of a decode layer's attention
together (store, index build, decode) as one CUDA graph.

--impl reference times the fp64 CPU oracle instead (same config and metric).
Under torchrun (N>1 GPUs) every rank decodes its own batch of the same
recipe (seeded per rank; tokens are independent: weak scaling, no collective
on the data path); rank 0 prints all ranks' tokens over the slowest rank's
time.  The reference arm runs on rank 0 alone.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sink_sda_decode_gb300 import inputs  # noqa: E402

METRIC = "decode tokens/s and gathered-KV GB/s; % of binding roofline (HBM vs bf16)"
STORE_METRIC = "q/kv RMSNorm + RoPE + SWA store tokens/s; % of HBM roofline"
TOPK_METRIC = "top-k -> slot list tokens/s; % of HBM roofline"
BUILDER_KEYS = ("state_slot", "swa_len", "swa_head", "comp_indptr", "comp_block", "comp_slot")
DEFAULT_CONFIG = 3  # h128: N=1024 H=128 D=512 L=640, the largest single-GPU workload
L2_FLUSH_BYTES = 256 << 20
HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0


# ----------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS, "fallback"


# The source files that define each measured kernel (its own file, the
# headers it includes): a committed ncu figure is used only while these are
# unchanged.
KERNEL_SOURCES = {
    "decode": ("sda_decode_umma.cu", "umma_ptx.cuh", "sda_internal.cuh"),
    "store": ("sda_store.cu", "sda_internal.cuh"),
    "topk": ("sda_topk.cu", "sda_internal.cuh"),
}


def _code_only(src):
    """The source without comments and blank lines: a comment edit leaves the
    compiled kernel, and so its measured figures, unchanged."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_source_hash(kernel="decode"):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sink_sda_decode_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(config_name, kernel="decode"):
    """DRAM bytes per launch of the measured kernel from the committed ncu
    summary, only if it was taken on the current sources of that kernel."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(config_name)
        if e and e.get("kernel_sources") == kernel_source_hash(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class _Nvml:
    """Read-only NVML through ctypes (libnvidia-ml ships with the driver):
    current / maximum SM clock and the active clock-event reasons."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index):
        import ctypes
        self.c = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        bus = None
        try:
            p = torch.cuda.get_device_properties(cuda_index)
            bus = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:
            pass
        ok = bus is not None and lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle")
        get = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.get_reasons = get or lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
        self.max_mhz = float(mx.value)

    def sample(self):
        mhz = self.c.c_uint(0)
        r = self.c.c_ulonglong(0)
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.c.byref(mhz))
        self.get_reasons(self.h, self.c.byref(r))
        return float(mhz.value), int(r.value)


class ClockSampler:
    """SM clock and clock-event reasons sampled during the timed region:
    NVML polled about every millisecond in a thread (nvidia-smi at 10 ms
    intervals where NVML cannot be loaded)."""

    def __init__(self, index):
        self.index = index
        self.samples = []  # (host time, mhz, set of reason names)
        self.window = None
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None

    def __enter__(self):
        try:
            nv = _Nvml(self.index)
            self.max_mhz, self.source = nv.max_mhz, "nvml"

            def poll():
                while not self._stop.is_set():
                    mhz, bits = nv.sample()
                    self.samples.append((time.perf_counter(), mhz,
                                         {n for b, n in _Nvml.REASONS.items() if bits & b}))
                    time.sleep(0.001)
                nv.lib.nvmlShutdown()
            self._thread = threading.Thread(target=poll, daemon=True)
            self._thread.start()
        except Exception:
            self._start_smi()
        return self

    def _start_smi(self):
        fields = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={fields}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"

            def read():
                for ln in self._proc.stdout:
                    parts = [x.strip() for x in ln.split(",")]
                    if len(parts) != 6:
                        continue
                    try:
                        mhz, self.max_mhz = float(parts[0]), float(parts[1])
                    except ValueError:
                        continue
                    self.samples.append((time.perf_counter(), mhz,
                                         {n for n, v in zip(names, parts[2:]) if v.lower() == "active"}))
            self._thread = threading.Thread(target=read, daemon=True)
            self._thread.start()
        except Exception:
            self._proc = None

    def __exit__(self, *a):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def wait_first(self, timeout=5.0):
        t0 = time.perf_counter()
        while not self.samples and time.perf_counter() - t0 < timeout:
            time.sleep(0.001)

    def mark(self, t_start, t_end):
        """Host-time window of the timed region (first launch .. final sync)."""
        self.window = (t_start, t_end)

    def summary(self):
        sel = [x for x in self.samples
               if self.window is None or self.window[0] <= x[0] <= self.window[1]]
        sm = [m for _, m, _ in sel]
        reasons = set()
        for _, _, r in sel:
            reasons |= r
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(sm), "source": self.source}


def algorithmic_bytes(w, kv="bf16"):
    """Bytes the method must move per decode: gathered KV rows + q + out +
    kv_indices + kv_indptr.  An FP8 pool row is D one-byte codes plus its
    4-byte scale."""
    L = int(w.total_len)
    row = w.D * 2 if kv == "bf16" else w.D + 4
    return L * row + 2 * w.N * w.H * w.D * 2 + L * 4 + (w.N + 1) * 4


def distinct_row_bytes(w, kv="bf16"):
    """algorithmic_bytes with each distinct pool row counted once, however
    many tokens' lists hold it: the least the step could read from HBM.  The
    decode workloads' lists barely overlap, so it is close to
    algorithmic_bytes; a prefill chunk's neighbouring tokens share most of
    their rows, and the fraction against these bytes is its HBM figure."""
    n = int(np.unique(np.asarray(w.kv_indices)).size)
    L = int(w.total_len)
    row = w.D * 2 if kv == "bf16" else w.D + 4
    return n * row + 2 * w.N * w.H * w.D * 2 + L * 4 + (w.N + 1) * 4


def store_algorithmic_bytes(w, rope_dim, kv="bf16"):
    """Bytes the store step must move: q read and written (bf16), the new KV
    row read (bf16) and written to the pool (bf16, or D codes + a 4-byte
    scale), each token's position and state slot, its RoPE cache rows (R/2
    cos + R/2 sin, fp32) and the two norm weights once."""
    row_out = w.D * 2 if kv == "bf16" else w.D + 4
    per_token = 2 * w.H * w.D * 2 + w.D * 2 + row_out + 4 + 4 + rope_dim * 4
    return w.N * per_token + 2 * w.D * 2


def topk_algorithmic_bytes(lengths, k, kpb):
    """Bytes the top-k step must move: every candidate score (fp32) once, the
    lengths, the block-table rows of the candidates, and the output lists
    (indptr + a block id and a slot per kept position)."""
    n = np.asarray(lengths, np.int64)
    kept = np.minimum(n, k)
    return int((n * 4).sum() + n.size * 4 + (-(-n // kpb) * 4).sum() + (n.size + 1) * 4
               + (kept * 8).sum())


def algorithmic_flops(w):
    return 4 * w.H * w.D * int(w.total_len)


# ----------------------------------------------------------------------------- GPU arm
class L2Flush:
    """Run before each timed step (outside its events): write 256 MiB, which
    evicts everything the previous step left in the 126 MiB L2, then read
    another 256 MiB, which writes those dirty lines back to HBM and leaves L2
    holding clean lines of an unrelated buffer.  The step starts cold and
    pays for none of the flush's write-backs."""

    def __init__(self, device):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.amax()



class Step:
    """Device-resident inputs and buffers of one step of the chosen path:
    "decode" (index build + decode), "store" (q/kv norm + RoPE + SWA store)
    or "layer" (store, then build + decode on the stored pool and the rotated
    q).  `ins` holds the per-step inputs, the tensors the end-to-end run
    copies from the host."""

    def __init__(self, w, device, pool=None, path="decode"):
        import sink_sda_decode_gb300 as sda
        self.sda = sda
        self.w = w
        self.path = path
        self.pool = pool  # an FP8 pool (inputs.Fp8Pool) replaces the bf16 one
        self.dev = device
        if path == "topk":
            self.ti = inputs.topk_inputs(w)
            self.ins = {"scores": self.ti.scores, "lengths": self.ti.lengths,
                        "block_table": self.ti.block_table}
            cap = w.N * self.ti.k
            self.comp = [torch.empty(w.N + 1, dtype=torch.int32, device=device),
                         torch.empty(cap, dtype=torch.int32, device=device),
                         torch.empty(cap, dtype=torch.int32, device=device)]
            self.topk_status = torch.empty(1, dtype=torch.int32, device=device)
            self.results = list(self.comp)
            self.launches_per_step = 2
            return
        self.ins = {"q": w.q}
        if path != "store":
            self.ins.update(w.builder_inputs(device))
            self.capacity = w.N * w.win + int(w.comp_block.size)
            self.kv_indices = torch.empty(max(self.capacity, 1), dtype=torch.int32, device=device)
            self.kv_indptr = torch.empty(w.N + 1, dtype=torch.int32, device=device)
            self.status = torch.empty(1, dtype=torch.int32, device=device)
            self.out = torch.empty_like(w.q)
            size = (sda.workspace_size if pool is None else sda.workspace_size_fp8)(
                w.N, w.H, w.D, self.capacity)
            self.ws = torch.empty(size, dtype=torch.uint8, device=device)
        if path != "decode":
            self.si = inputs.store_inputs(w)
            self.ins["kv_new"] = self.si.kv_new
            self.ins["positions"] = self.si.positions
            self.ins.setdefault("state_slot", self.si.state_slot)
            self.q_rot = torch.empty_like(w.q)
            self.store_status = torch.empty(1, dtype=torch.int32, device=device)
        self.results = [self.q_rot if path == "store" else self.out]
        # decode: builder lengths, scan, plan + scatter, attention, combine
        self.launches_per_step = {"decode": 5, "store": 1, "layer": 6}[path]

    @property
    def rope_dim(self):
        return self.si.cos_cache.shape[1] * 2

    def run(self, ins=None, stream=None, timing=None):
        """One step.  `timing` = (before, after) events: recorded around the
        store kernel on the store path, around the attention kernel otherwise."""
        w = self.w
        ins = ins or self.ins
        if self.path == "topk":
            if timing:
                self.sda.set_timing_events(*timing)
            self.sda.topk_slots(ins["scores"], ins["lengths"], ins["block_table"], k=self.ti.k,
                                k_per_block=w.k_per_block, comp_indptr=self.comp[0],
                                comp_block=self.comp[1], comp_slot=self.comp[2],
                                status=self.topk_status, stream=stream)
            self.sda.set_timing_events(None, None)
            return
        q = ins["q"]
        if self.path != "decode":
            si = self.si
            if timing and self.path == "store":
                self.sda.set_timing_events(*timing)
            self.sda.qk_norm_rope_swa_store(
                q, ins["kv_new"], si.q_norm_w, si.kv_norm_w, si.cos_cache, si.sin_cache,
                ins["positions"], ins["state_slot"], eps=si.eps, win=w.win,
                swa_pages=w.swa_pages, unified_kv=w.unified_kv if self.pool is None else None,
                kv_fp8=None if self.pool is None else self.pool.codes,
                kv_scale=None if self.pool is None else self.pool.scale, q_out=self.q_rot,
                status=self.store_status, stream=stream)
            self.sda.set_timing_events(None, None)
            q = self.q_rot
        if self.path == "store":
            return
        # index build + decode in one call (the builder's scan and the decode's
        # work plan share a CTA)
        if timing:
            self.sda.set_timing_events(*timing)
        self.sda.build_decode(q, w.unified_kv if self.pool is None else self.pool.codes,
                              w.attn_sink, w.softmax_scale,
                              *(ins[k] for k in BUILDER_KEYS), win=w.win,
                              k_per_block=w.k_per_block, swa_pages=w.swa_pages,
                              kv_scale=None if self.pool is None else self.pool.scale,
                              capacity=self.capacity, out=self.out, workspace=self.ws,
                              kv_indices=self.kv_indices, kv_indptr=self.kv_indptr,
                              status=self.status, stream=stream)
        self.sda.set_timing_events(None, None)

    def check_status(self):
        if self.path == "topk":
            if int(self.topk_status.item()) != 0:
                raise RuntimeError(f"top-k status {int(self.topk_status.item())}")
            return
        if self.path != "store" and int(self.status.item()) != 0:
            raise RuntimeError(f"index builder status {int(self.status.item())}")
        if self.path != "decode" and int(self.store_status.item()) != 0:
            raise RuntimeError(f"store status {int(self.store_status.item())}")


def gpu_arm(args, w, device, ws, rank, pool=None):
    step = Step(w, device, pool, getattr(args, "path", "decode"))
    flush = L2Flush(device)
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        for _ in range(max(args.warmup, 3)):
            step.run(stream=s)
    torch.cuda.current_stream(device).wait_stream(s)
    torch.cuda.synchronize(device)
    step.check_status()
    # whole step as one CUDA graph
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step.run(stream=s)
    torch.cuda.synchronize(device)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)

    # ---- timed region 1: K graph replays, L2 flushed before each step
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with ClockSampler(torch.cuda.current_device() if device.index is None else device.index) as cs:
        cs.wait_first()
        barrier()
        t_start = time.perf_counter()
        with torch.cuda.stream(s):
            for a, b in evs:
                flush()
                a.record(s)
                g.replay()
                b.record(s)
        barrier()
        cs.mark(t_start, time.perf_counter())
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms_per_step = sum(step_ms) / len(step_ms)

    # ---- timed region 2: the dominant kernel alone (library timing hook)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier()
    with torch.cuda.stream(s):
        for a, b in kev:
            flush()
            step.run(stream=s, timing=(a, b))
    barrier()
    kernel_ms = sum(a.elapsed_time(b) for a, b in kev) / len(kev)

    # ---- timed region 3: end to end from pinned host memory.  The step's
    # inputs (q, the builder's descriptors, the new KV rows and positions)
    # sit packed in one pinned host buffer: one H2D copy, the public calls on
    # views of the device copy, one D2H copy of the result (out, or the
    # rotated q of the store path) -- replayed as one CUDA graph, as a
    # serving loop replays its decode step.
    names = list(step.ins)
    parts = [step.ins[k].reshape(-1).view(torch.uint8) for k in names]
    offs, total = [], 0
    for t_ in parts:
        offs.append(total)
        total += (t_.numel() + 255) // 256 * 256
    h_in = torch.zeros(max(total, 256), dtype=torch.uint8, pin_memory=True)
    for o, t_ in zip(offs, parts):
        h_in[o:o + t_.numel()].copy_(t_.cpu())
    d_in = torch.empty_like(h_in, device=device)
    views = {k: d_in[o:o + p.numel()].view(step.ins[k].dtype).view(step.ins[k].shape)
             for k, o, p in zip(names, offs, parts)}
    outs_h = [torch.empty(t_.shape, dtype=t_.dtype, pin_memory=True) for t_ in step.results]
    h2d = sum(t_.numel() for t_ in parts)
    d2h = sum(o.numel() * o.element_size() for o in outs_h)

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        step.run(ins=views, stream=s)
        for o, t_ in zip(outs_h, step.results):
            o.copy_(t_, non_blocking=True)

    if step.path == "decode":
        # The decode step's own host-buffer call: kernels read q and the
        # builder's descriptors from page-locked host memory and write out and
        # the status word back (sda_build_decode_host; large batches go through
        # its chunked copy-engine pipeline).
        hq = w.q.cpu().pin_memory()
        hd = {k: step.ins[k].cpu().pin_memory() for k in BUILDER_KEYS}
        h_out = torch.empty(w.q.shape, dtype=w.q.dtype, pin_memory=True)
        h_st = torch.empty(1, dtype=torch.int32, pin_memory=True)
        pool = step.pool
        ws_host = torch.empty(step.sda.build_decode_host_workspace_size(
            w.N, w.H, w.D, int(w.comp_block.size), step.capacity, pool is not None),
            dtype=torch.uint8, device=device)
        h2d = hq.numel() * hq.element_size() + sum(t_.numel() * 4 for t_ in hd.values())
        d2h = h_out.numel() * h_out.element_size() + 4

        def e2e_step():
            step.sda.build_decode_host(
                hq, w.unified_kv if pool is None else pool.codes, w.attn_sink, w.softmax_scale,
                *(hd[k] for k in BUILDER_KEYS), win=w.win, k_per_block=w.k_per_block,
                swa_pages=w.swa_pages, kv_scale=None if pool is None else pool.scale,
                capacity=step.capacity, out=h_out, status=h_st, workspace=ws_host, stream=s)

    with torch.cuda.stream(s):
        for _ in range(max(args.warmup, 3)):
            e2e_step()
    torch.cuda.synchronize(device)
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge, stream=s):
        e2e_step()
    torch.cuda.synchronize(device)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    barrier()
    with torch.cuda.stream(s):
        for a, b in e2e_ev:
            flush()
            a.record(s)
            ge.replay()
            b.record(s)
    barrier()
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_ev) / len(e2e_ev)
    return dict(ms_per_step=ms_per_step, kernel_ms=kernel_ms, e2e_ms=e2e_ms, clocks=cs.summary(),
                h2d=h2d, d2h=d2h, launches_per_step=step.launches_per_step,
                rope_dim=step.rope_dim if step.path in ("store", "layer") else None,
                topk_bytes=(topk_algorithmic_bytes(step.ti.lengths.cpu().numpy(), step.ti.k,
                                                   w.k_per_block) if step.path == "topk" else None))


def measure_decode(w, device, steps, warmup):
    """Step and attention-kernel time (ms) of the decode step on workload w,
    timed as in gpu_arm (graph replays after an L2 flush; the kernel alone
    through the library's timing hook).  Returns the output of the last step
    too, for the sampled oracle comparison."""
    step = Step(w, device, None, "decode")
    flush = L2Flush(device)
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        for _ in range(max(warmup, 3)):
            step.run(stream=s)
    torch.cuda.synchronize(device)
    step.check_status()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step.run(stream=s)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize(device)
    with torch.cuda.stream(s):
        for a, b in evs:
            flush()
            a.record(s)
            g.replay()
            b.record(s)
        for a, b in kev:
            flush()
            step.run(stream=s, timing=(a, b))
    torch.cuda.synchronize(device)
    ms_step = sum(a.elapsed_time(b) for a, b in evs) / steps
    ms_kernel = sum(a.elapsed_time(b) for a, b in kev) / steps
    return ms_step, ms_kernel, step.out.clone()


def per_config_entry(w, ms_step, ms_kernel):
    hbm, bf16, _ = peaks()
    nbytes, flops = algorithmic_bytes(w), algorithmic_flops(w)
    bound = "hbm" if nbytes / (hbm * 1e9) >= flops / (bf16 * 1e12) else "tensor"
    achieved = (nbytes / 1e9 if bound == "hbm" else flops / 1e12) / (ms_kernel * 1e-3)
    return {"workload": w.name, "N": w.N, "H": w.H, "total_slots": int(w.total_len),
            "value": w.N / (ms_step * 1e-3), "unit": "tokens/s", "ms_per_step": ms_step,
            "kernel_ms": ms_kernel, "bound": bound,
            "frac": achieved / (hbm if bound == "hbm" else bf16),
            "gathered_kv_gbs": int(w.total_len) * w.D * 2 / (ms_kernel * 1e-3) / 1e9}


PER_CONFIGS = ("tiny", "h16", "ragged_h64", "h128", "longtail_h64")


# ----------------------------------------------------------------------------- job-wide report
def reduce_over_ranks(times_ms, units, ws, device):
    """Job-wide timings and units of a data-parallel run.

    Each per-rank time becomes its MAX over ranks (the slowest rank bounds
    the job); the units (decoded tokens) are SUMMED, since every rank decodes
    its own batch.  Two all_reduce calls on the default process group, on
    tensors placed on `device` (the GPU for NCCL, the CPU for gloo); a single
    process returns its own numbers."""
    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=device)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    if ws > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    return [float(x) for x in t.cpu()], float(u.cpu().item())


STEP_TEXT = {
    "topk": "top-k of each token's scores -> compressed (block, slot) lists (2 kernels) as one "
            "CUDA graph",
    "decode": "index build + decode (plan, attention, combine), one sda_build_decode call, as "
              "one CUDA graph",
    "store": "q/kv RMSNorm + GPT-J RoPE + SWA ring store (one kernel) as one CUDA graph",
    "layer": "q/kv norm + RoPE + SWA store, index build, decode as one CUDA graph",
}


def report_line(args, w, ws, ms_step, ms_kernel, ms_e2e, tokens_total, r):
    """The JSON line of the GPU arm from job-wide numbers (rank 0 prints it).

    `value` and `e2e.value` are all ranks' tokens over the slowest rank's step
    time; the roofline is the dominant kernel of this rank's workload (the
    attention kernel, or the store kernel on the store path), whose shape
    every rank shares."""
    hbm, bf16, peak_src = peaks()
    kv = getattr(args, "kv", "bf16")
    path = getattr(args, "path", "decode")
    value = tokens_total / (ms_step * 1e-3)
    if path == "store":
        nbytes = store_algorithmic_bytes(w, r["rope_dim"], kv)
        flops = 0
        bound = "hbm"
        kernel = "q/kv norm + RoPE + SWA store kernel"
        traffic_key = "store_" + args.config
    elif path == "topk":
        nbytes = r["topk_bytes"]
        flops = 0
        bound = "hbm"
        kernel = "top-k slot-list kernels (indptr scan + per-token radix select)"
        traffic_key = "topk_" + args.config
    else:
        nbytes = algorithmic_bytes(w, kv)
        flops = algorithmic_flops(w)
        bound = "hbm" if nbytes / (hbm * 1e9) >= flops / (bf16 * 1e12) else "tensor"
        kernel = "sda decode attention kernel"
        traffic_key = args.config
    if kv != "bf16":
        traffic_key += "_fp8"
    t_bound = nbytes / (hbm * 1e9) if bound == "hbm" else flops / (bf16 * 1e12)
    # achieved rate of the binding resource: GB/s of algorithmic bytes, or
    # TFLOP/s of algorithmic FLOPs
    achieved = (nbytes / 1e9 if bound == "hbm" else flops / 1e12) / (ms_kernel * 1e-3)
    line = {
        "metric": {"store": STORE_METRIC, "topk": TOPK_METRIC}.get(path, METRIC), "value": value,
        "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if path == "topk" else "bf16", "data": "synthetic",
        "config": {"workload": w.name, "N": w.N, "H": w.H, "D": w.D,
                   "total_slots": int(w.total_len), "pool_slots": w.total_pages,
                   "kv": "bf16" if kv == "bf16" else "fp8 e4m3, fp32 scale per row",
                   "path": path, "step": STEP_TEXT[path],
                   "l2": "flushed before every timed step (256 MiB write, then 256 MiB read)",
                   "parallelism": f"dp{ws} (independent token batches)"},
        "roofline": {"bound": bound, "achieved": achieved,
                     "peak": hbm if bound == "hbm" else bf16,
                     "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                     "frac": achieved / (hbm if bound == "hbm" else bf16),
                     "traffic": ncu_traffic(traffic_key, path if path in ("store", "topk")
                                            else "decode"),
                     "peak_source": peak_src,
                     "kernel": kernel, "kernel_ms": ms_kernel,
                     "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                     "step_frac_of_roofline": t_bound / (ms_step * 1e-3)},
        "e2e": {"value": tokens_total / (ms_e2e * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": r["launches_per_step"] * args.steps,
        "clocks": r["clocks"],
    }
    if path == "store":
        line["config"]["rope_dim"] = r["rope_dim"]
    elif path == "topk":
        line["config"]["topk"] = {"k": inputs.TOPK_K, "candidates": inputs.TOPK_CANDIDATES}
    else:
        line["gathered_kv_gbs"] = (int(w.total_len) * (w.D * 2 if kv == "bf16" else w.D + 4)
                                   / (ms_step * 1e-3) / 1e9)
        if bound == "hbm":
            db = distinct_row_bytes(w, kv)
            line["roofline"]["distinct_row_bytes"] = db
            line["roofline"]["frac_distinct_rows"] = db / 1e9 / (ms_kernel * 1e-3) / hbm
    return line


# ----------------------------------------------------------------------------- CPU oracle
def oracle_inputs(w, tokens, pool=None):
    """Arguments of the oracle call for `tokens` (bf16 pool, or an FP8 pool)."""
    q_bits = w.q_bits()[np.asarray(tokens)]
    if pool is None:
        kv_bits, sub_idx, sub_ptr = w.kv_rows_for(tokens)
        return q_bits, kv_bits, sub_idx, sub_ptr, w.attn_sink.cpu().numpy()
    codes, scale, sub_idx, sub_ptr = inputs.fp8_rows_for(w, pool, tokens)
    return q_bits, codes, scale, sub_idx, sub_ptr, w.attn_sink.cpu().numpy()


def oracle_decode(oargs, w):
    import oracle
    fn = oracle.sda_decode if len(oargs) == 5 else oracle.sda_decode_fp8
    return fn(*oargs, w.softmax_scale)


def oracle_sample(w, budget_tokens):
    """Deterministic token sample whose slot count is about budget_tokens x mean L."""
    rng = np.random.default_rng(0)
    k = max(1, min(w.N, budget_tokens))
    return np.sort(rng.choice(w.N, k, replace=False))


def oracle_job(w, toks, pool=None, path="decode"):
    """The oracle's share of one step on the token sample `toks`, as a
    callable: the store (exact values, then the rounding the pool stores)
    and / or the decode."""
    import oracle
    calls = []
    if path == "topk":
        ti = inputs.topk_inputs(w)
        targs = (ti.scores.cpu().numpy()[toks], ti.lengths.cpu().numpy()[toks],
                 ti.block_table.cpu().numpy()[toks], ti.k, w.k_per_block)
        return lambda: oracle.topk_slots(*targs)
    if path != "decode":
        si = inputs.store_inputs(w)
        bits = inputs.bf16_to_bits
        sargs = (w.q_bits()[toks], bits(si.kv_new)[toks], bits(si.q_norm_w), bits(si.kv_norm_w),
                 si.cos_cache.cpu().numpy(), si.sin_cache.cpu().numpy(),
                 si.positions.cpu().numpy()[toks], si.state_slot.cpu().numpy()[toks], si.eps,
                 w.win, w.swa_pages)

        def store():
            res = oracle.qk_norm_rope_store(*sargs)
            oracle.bf16_rne(res["q_val"])
            if pool is None:
                oracle.bf16_rne(res["kv_val"])
            else:
                oracle.fp8_quantise_rows(res["kv_val"])
        calls.append(store)
    if path != "store":
        oargs = oracle_inputs(w, toks, pool)
        calls.append(lambda: oracle_decode(oargs, w))
    return lambda: [c() for c in calls]


def oracle_budget(w, path):
    """Tokens per oracle pass: all of them where a pass is cheap."""
    return w.N if path in ("store", "topk") or w.total_len <= 200000 else 16


def sampled_parity(w, out, max_tokens=48):
    """The CPU-baseline leg's check of the GPU output: a deterministic sample
    of tokens (always the longest and the shortest list) against the fp64
    oracle, with the tolerance of the parity tests (max |err| <= 8e-3 or one
    bf16 ULP of the reference where that is larger, mean |err| <= 1e-3)."""
    lens = w.lengths
    rng = np.random.default_rng(1)
    toks = set(rng.choice(w.N, min(w.N, max_tokens), replace=False).tolist())
    toks |= {int(np.argmax(lens)), int(np.argmin(lens))}
    toks = np.array(sorted(toks))
    ref = oracle_decode(oracle_inputs(w, toks), w)
    got = out[torch.from_numpy(toks).to(out.device)].float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    ax = np.abs(ref)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(ax, 2.0 ** -126))) - 7)
    return {"tokens": int(toks.size), "elements": int(err.size),
            "max_abs": float(err.max()) if err.size else 0.0,
            "mean_abs": float(err.mean()) if err.size else 0.0,
            "raw_violations": int((err > 8e-3).sum()),
            "rounding_aware_violations": int((err > np.maximum(8e-3, ulp)).sum())}


def time_oracle(w, seconds, max_tokens, pool=None, path="decode"):
    import oracle
    toks = oracle_sample(w, max_tokens)
    job = oracle_job(w, toks, pool, path)
    done_tokens, t0 = 0, time.perf_counter()
    passes = 0
    while True:
        job()
        done_tokens += len(toks)
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return done_tokens / el, oracle.num_threads(), toks, passes, el


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", default=inputs.CONFIG_NAMES[DEFAULT_CONFIG],
                    choices=inputs.CONFIG_NAMES)
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="pool format: bf16 rows, or FP8 E4M3 codes with one fp32 scale per row "
                         "(the workload's pool quantised row by row)")
    ap.add_argument("--path", choices=["decode", "store", "layer", "topk"], default="decode",
                    help="decode: index build + decode; store: q/kv norm + RoPE + SWA store; "
                         "layer: store + build + decode; topk: top-k -> slot lists")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip timing the five decode workloads after the main one")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    ws, rank, local = dist_env()
    cfg_idx = inputs.CONFIG_NAMES.index(args.config)

    if args.impl == "reference":
        if rank != 0:
            return
        w = inputs.config(cfg_idx, device="cuda" if torch.cuda.is_available() else "cpu")
        import oracle
        pool = inputs.fp8_pool(w) if args.kv == "fp8" else None
        toks = oracle_sample(w, oracle_budget(w, args.path))
        job = oracle_job(w, toks, pool, args.path)
        for _ in range(args.warmup):
            job()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            job()
        el = time.perf_counter() - t0
        tps = len(toks) * args.steps / el
        sample = f"{len(toks)} of {w.N} tokens per step"
        line = {"metric": {"store": STORE_METRIC, "topk": TOPK_METRIC}.get(args.path, METRIC),
                "value": tps,
                "unit": "tokens/s", "impl": "reference",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32" if args.path == "topk" else "f64",
                "data": "synthetic",
                "config": {"workload": w.name, "N": w.N, "H": w.H, "D": w.D,
                           "total_slots": w.total_len, "kv": args.kv, "path": args.path},
                "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": oracle.num_threads(),
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if ws > 1:
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w = inputs.config(cfg_idx, device=device, shard=rank)
    pool = inputs.fp8_pool(w) if args.kv == "fp8" else None
    r = gpu_arm(args, w, device, ws, rank, pool)

    (ms_step, ms_kernel, ms_e2e), tokens_total = reduce_over_ranks(
        [r["ms_per_step"], r["kernel_ms"], r["e2e_ms"]], w.N, ws, device)
    if rank != 0:
        torch.distributed.destroy_process_group()
        return

    line = report_line(args, w, ws, ms_step, ms_kernel, ms_e2e, tokens_total, r)
    outs = {}
    if args.per_config and ws == 1 and args.path == "decode" and args.kv == "bf16":
        # the five decode workloads, one after another, timed the same way
        per = []
        for name in PER_CONFIGS:
            wc = w if name == args.config else inputs.config(inputs.CONFIG_NAMES.index(name),
                                                             device=device)
            ms_s, ms_k, outs[name] = measure_decode(wc, device, args.steps, args.warmup)
            per.append(dict(config=name, **per_config_entry(wc, ms_s, ms_k)))
            if wc is not w:
                del wc
                torch.cuda.empty_cache()
        line["per_config"] = per
    if not args.no_cpu_baseline and ws == 1:
        tps, cores, toks, passes, el = time_oracle(w, args.cpu_seconds,
                                                   oracle_budget(w, args.path), pool, args.path)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"{len(toks)} of {w.N} tokens x {passes} passes, "
                                          f"{el:.1f} s"}
        if outs:
            # the same leg checks each workload's GPU output on a token sample
            for entry in line["per_config"]:
                name = entry["config"]
                wc = w if name == args.config else inputs.config(inputs.CONFIG_NAMES.index(name),
                                                                 device=device)
                entry["parity_sample"] = sampled_parity(wc, outs[name])
                if wc is not w:
                    del wc
                    torch.cuda.empty_cache()
    print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
