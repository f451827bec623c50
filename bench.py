#!/usr/bin/env python3
"""Benchmark of the MTP draft block + verify-accept hot path.

One step of a draft workload = one mtp_draft_block call (N chained draft
steps, one persistent launch) + one mtp_verify_greedy call on the target's
(1+N) x V verify logits.  Metric: drafted tokens per second = B * N / (draft
+ verify time).  The headline is the Gemma-assistant-shaped workload (bf16,
d_t 5120, d_a 1024, 4 blocks, 16 x 256 query heads over 4 KV heads, GeGLU
4096, vocab 262144, B = 1, N = 3, 8192 cached positions; 3 blocks attend a
1024-window sliding layer, 1 a full layer).  The default run also times the
same model at B = 16 (N = 4, ragged 2k-32k contexts) and B = 64 (N = 2,
context 4096), exact temp > 0 verification alone (mtp_verify_sample,
B = 32, N = 3, V = 248320; that configuration has no draft block), and an
Edge-shaped drafter with the centroid-routed LM head (B = 1, N = 3), the
headline workload with Q8_0 and with Q4_0 projections, and the dense NextN drafter
(Qwen-shaped, B = 1: two catch-up rows then N = 3 drafts from its own KV of
4096 rows, one mtp_nextn_draft call + greedy verify), each
reported under per_workload with its own roofline fraction, end-to-end
number and CPU baseline.  `--workload K` times one of them alone.

Prints ONE JSON line.  `--impl reference` times the CPU oracle instead (a
bounded sample per step), with the same config.  Multi-GPU (torchrun): every
rank runs an independent replica (the path has no cross-sequence exchange);
the value is the sum of drafted tokens over the max time across ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "drafted tok/s (MTP draft block + verify) at B=1..64; % of HBM/tensor roofline"
UNIT = "tok/s"
HEADLINE = 1
OTHERS = (2, 3, 4, 5, 6, 8, 7)
NEXTN = 7


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=None, choices=[0, 1, 2, 3, 4, 5, 6, 7, 8],
                    help="time this workload alone (default: the headline plus workloads 2-8)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The largest x over all ranks of the initialised process group (x itself
    for one rank): the whole-job time of independent replicas."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# workloads and their configs (one description for both arms)
# ----------------------------------------------------------------------------

L2_FLUSH_BYTES = 256 << 20   # written between timed verify-sample launches (its 111 MB of logits fit in L2)


def _common(world: int, flushed: bool) -> dict:
    return {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": (f"flushed before every timed launch ({L2_FLUSH_BYTES >> 20} MB written)" if flushed
                   else "inputs larger than L2 (weights streamed every step), no flush")}


def draft_config(w, world: int = 1) -> dict:
    m = w.model
    head = (f"centroid-routed: {m.n_centroids} lists of {m.vocab // m.n_centroids}, top {m.centroid_top_k}"
            if m.n_centroids else "dense tied")
    return dict({"workload": w.name, "B": w.B, "N": w.N, "vocab": m.vocab, "d_t": m.d_t, "d_a": m.d_a,
                 "n_blocks": m.n_blocks, "kv_len_max": int(w.kv_len.max()), "kv_len_min": int(w.kv_len.min()),
                 "lm_head": head,
                 "projections": {"q8_0": "Q8_0 (bf16 table and KV)", "q4_0": "Q4_0 (bf16 table and KV)"}.get(m.wquant,
                                                                                                       m.dtype)},
                **_common(world, False))


def nextn_config(w, world: int = 1) -> dict:
    m = w.model
    return dict({"workload": w.name, "B": w.B, "N": w.N, "vocab": m.vocab, "d": m.d, "heads": m.n_q_heads,
                 "kv_heads": m.n_kv_heads, "head_dim": m.head_dim, "d_ff": m.d_ff,
                 "drafter_kv_rows": int(w.kv_len.max()), "catch_up_rows": int(w.n_cu.max()),
                 "lm_head": "dense tied (shared head)", "projections": m.dtype,
                 "path": "mtp_nextn_draft (catch-up + drafts, one launch) + mtp_verify_greedy"},
                **_common(world, False))


def sample_config(inp, world: int = 1) -> dict:
    B, R, V = inp.target.shape
    return dict({"workload": synth.WORKLOADS[4], "B": B, "N": R - 1, "vocab": V, "history": int(inp.hist.shape[1]),
                 "path": "mtp_verify_sample alone (this configuration has no draft block)"}, **_common(world, True))


# ----------------------------------------------------------------------------
# algorithmic bytes (the byte floor: every tensor the step must read, once)
# ----------------------------------------------------------------------------

def kv_bytes_per_step(w) -> int:
    """Distinct KV bytes one draft step reads: each view's readable positions,
    K and V, every KV head; a view read by several blocks counts once."""
    m = w.model
    esz = 2 if m.dtype == "bf16" else 4
    used = sorted(set(m.block_view))
    tot = 0
    for vi in used:
        vd = w.views[vi]
        for b in range(w.B):
            n = len(synth.view_positions(vd["window"], int(w.kv_len[b]), vd.get("sink", 0)))
            tot += 2 * n * m.n_kv_heads * m.head_dim * esz
    return tot


def head_bytes_per_step(w) -> int:
    """The LM head's bytes: the dense head reads the whole table; the
    centroid-routed head the centroids, and per sequence the top_k lists'
    ids and their table rows."""
    m = w.model
    esz = 2 if m.dtype == "bf16" else 4
    if not m.n_centroids:
        return m.vocab * m.d_t * esz
    cand = m.centroid_top_k * (m.vocab // m.n_centroids)
    return m.n_centroids * m.d_t * esz + w.B * cand * (m.d_t * esz + 4)


def draft_bytes_per_launch(w) -> int:
    """Weights (the head's share per head_bytes_per_step), each view's KV
    once, and the consumed tokens' embedding rows, per step."""
    m = w.model
    esz = 2 if m.dtype == "bf16" else 4
    head_w = m.vocab * m.d_t * esz + sum(int(w.weights[n].nbytes) for n in ("centroids", "token_ordering")
                                         if n in w.weights)
    wb = w.weight_bytes()
    if m.wquant in ("q8_0", "q4_0"):   # quantised projections: a byte (Q4_0: half) per weight, 2 bytes per 32
        per = 1 if m.wquant == "q8_0" else 0.5
        for n in synth.projection_names(m):
            a = w.weights[n]
            wb += a.size * (per + 2 / 32) - a.nbytes
    per_step = (wb - head_w + head_bytes_per_step(w) + kv_bytes_per_step(w) + w.B * m.d_t * esz)
    return int(w.N * per_step)


def draft_flops_per_launch(w) -> float:
    m = w.model
    attn = 0
    for l in range(m.n_blocks):
        vd = w.views[m.block_view[l]]
        for b in range(w.B):
            n = len(synth.view_positions(vd["window"], int(w.kv_len[b]), vd.get("sink", 0)))
            attn += 4 * m.n_q_heads * m.head_dim * n
    return float(w.N * (2 * m.params() * w.B + attn))


def nextn_bytes_per_launch(w) -> int:
    """The NextN drafter's byte floor for one call.  Weights: every catch-up
    iteration (as many as the largest catch-up count) reads eh_proj and the
    key and value rows of w_qkv; every draft step all weights (the table once:
    it is also the head).  Per sequence: each catch-up row's embedding row and
    hidden state, each step's embedding row and the drafter KV's rows
    [0, pos], and the key and value rows the call writes."""
    m = w.model
    esz = 2 if m.dtype == "bf16" else 4
    d, hd, Hkv = m.d, m.head_dim, m.n_kv_heads
    W = w.weights
    kv_row = 2 * Hkv * hd * esz
    tot = int(w.n_cu.max()) * (int(W["eh_proj"].nbytes) + 2 * Hkv * hd * d * esz)
    tot += w.N * sum(int(a.nbytes) for a in W.values())
    for b in range(w.B):
        nc = int(w.n_cu[b])
        tot += nc * (d * esz + 4 * d)
        for k in range(w.N):
            tot += (int(w.kv_len[b]) + nc + k + 1) * kv_row + d * esz
        tot += (nc + w.N) * kv_row
    return int(tot)


def verify_sample_bytes(inp) -> int:
    """Algorithmic bytes of one mtp_verify_sample call: one read of the target
    and draft logits (the history and drafts are a few KB)."""
    return int(inp.target.nbytes + inp.draft.nbytes)


# ----------------------------------------------------------------------------
# clocks during the timed regions
# ----------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples (200 ms) taken only while a timed region runs:
    start()/pause() bracket each region, summary() covers them all."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.th = None
        self.failed = False

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            self.failed = True
            return
        self.th = threading.Thread(target=self._read, args=(self.proc,), daemon=True)
        self.th.start()
        time.sleep(0.3)

    def _read(self, proc):
        for line in proc.stdout:
            self.lines.append(line.strip())

    def pause(self):
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.th:
            self.th.join(timeout=2)
        self.proc = None

    def summary(self) -> dict:
        self.pause()
        if self.failed and not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_hash() -> str:
    """sha256 prefix over the library's CUDA sources and its public header:
    ties a recorded ncu traffic figure to the kernel it was taken on."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mtp_speculative_decoding_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.endswith((".cu", ".cuh", ".h")):
            h.update(fn.encode())
            with open(os.path.join(csrc, fn), "rb") as f:
                h.update(f.read())
    with open(os.path.join(ROOT, "include", "mtp.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the workload's dominant kernel
    from the committed ncu record (one line per workload), or None when that
    capture was taken on other kernel sources."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    src = kernel_source_hash()
    with open(p) as f:
        for line in f:
            kv = dict(t.split("=", 1) for t in line.split() if "=" in t)
            if kv.get("workload") == workload and kv.get("source_hash") == src:
                return int(kv["dram_bytes_per_launch"])
    return None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


# ----------------------------------------------------------------------------
# our implementation
# ----------------------------------------------------------------------------

def bench_draft(wid, args, world, clocks, reuse=None):
    """Draft block + greedy verify of workload wid.  Returns (fields, device
    draft object for reuse, workload)."""
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import to_device, upload_draft

    w = synth.make_draft_inputs(wid)
    m = w.model
    B, N, V = w.B, w.N, m.vocab
    dev = upload_draft(w, extra_ws_for=(B, N, V), reuse=reuse)
    ws = dev.ws
    drafts = torch.empty((B, N), dtype=torch.int32, device="cuda")
    h_last = torch.empty((B, m.d_t), dtype=torch.float32, device="cuda")
    # one untimed draft to plant the verify logits' accept lengths against the real drafts
    dev.run(drafts, h_last)
    torch.cuda.synchronize()
    if mtp.last_error(ws) != 0:
        raise RuntimeError(f"draft block status {mtp.last_error(ws)}")
    d_host = drafts.cpu().numpy()
    vin = synth.make_verify_greedy_inputs(wid, B=B, N=N, V=V)
    logits_np = synth.plant_greedy_logits(
        synth.bf16_bits_to_f32(vin.logits) if vin.dtype == "bf16" else vin.logits, d_host, vin.planted, vin.dtype)
    logits = to_device(logits_np, vin.dtype)
    out_tok = torch.empty((B, N + 1), dtype=torch.int32, device="cuda")
    n_acc = torch.empty((B,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        dev.run(drafts, h_last)
        mtp.verify_greedy(logits, drafts, out_tok, n_acc, ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert mtp.last_error(ws) == 0
    got_n = n_acc.cpu().numpy()
    if not np.array_equal(got_n, vin.planted):
        raise RuntimeError(f"verify accepted {got_n}, planted {vin.planted}")

    # per-kernel events on the launch stream: draft launch and verify launch separately
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        a, b_, c = ev[i]
        a.record(stream)
        dev.run(drafts, h_last)
        b_.record(stream)
        mtp.verify_greedy(logits, drafts, out_tok, n_acc, ws)
        c.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.pause()
    total_ms = t_start.elapsed_time(t_end)
    draft_ms = [e[0].elapsed_time(e[1]) for e in ev]
    verify_ms = [e[1].elapsed_time(e[2]) for e in ev]
    total_ms = max_over_ranks(total_ms, world)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ms_per_step = total_ms / args.steps
    value = world * B * N * args.steps / (total_ms / 1e3)

    # end-to-end through the public API with host buffers (pinned), copies inside the timed region
    h_tok = torch.from_numpy(w.last_tok.copy()).pin_memory()
    h_h = torch.from_numpy(w.h_prev.copy()).pin_memory()
    h_kv = torch.from_numpy(w.kv_len.copy()).pin_memory()
    h_logits = torch.empty(logits.shape, dtype=logits.dtype).pin_memory()
    h_logits.copy_(logits.cpu())
    h_out = torch.empty((B, N + 1), dtype=torch.int32).pin_memory()
    h_n = torch.empty((B,), dtype=torch.int32).pin_memory()
    h_dr = torch.empty((B, N), dtype=torch.int32).pin_memory()
    bi = h_tok.numel() * 4 + h_h.numel() * 4 + h_kv.numel() * 4 + h_logits.numel() * h_logits.element_size()
    bo = h_out.numel() * 4 + h_n.numel() * 4 + h_dr.numel() * 4

    def e2e_step():
        dev.last_tok.copy_(h_tok, non_blocking=True)
        dev.h_prev.copy_(h_h, non_blocking=True)
        dev.kv_len.copy_(h_kv, non_blocking=True)
        logits.copy_(h_logits, non_blocking=True)
        dev.run(drafts, h_last)
        mtp.verify_greedy(logits, drafts, out_tok, n_acc, ws)
        h_dr.copy_(drafts, non_blocking=True)
        h_out.copy_(out_tok, non_blocking=True)
        h_n.copy_(n_acc, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks.start()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.pause()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = world * B * N * args.steps / (e2e_ms / 1e3)
    if not np.array_equal(h_n.numpy(), vin.planted):
        raise RuntimeError("end-to-end verify disagrees with the planted accept lengths")

    peak, peak_kind = measured_peaks()
    alg = draft_bytes_per_launch(w)
    achieved = alg / (statistics.mean(draft_ms) / 1e3) / 1e9
    fields = {
        "value": round(value, 2), "ms_per_step": round(ms_per_step, 4),
        "config": draft_config(w, world),
        "breakdown": {"draft_ms_mean": round(statistics.mean(draft_ms), 4),
                      "verify_ms_mean": round(statistics.mean(verify_ms), 4)},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": int(bi),
                "d2h_bytes_per_step": int(bo)},
        "roofline": {"bound": "hbm", "kernel": "draft_kernel", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": alg, "traffic": recorded_traffic(w.name)},
        "gpu_launches": 2 * args.steps,
        "dtype": "bf16" if m.dtype == "bf16" else "f32",
    }
    return fields, dev, w


def bench_nextn(args, world, clocks):
    """The NextN drafter (workload 7): one mtp_nextn_draft call (catch-up rows,
    then N drafts from its own KV) + greedy verify.  Returns (fields, workload)."""
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import to_device, upload_nextn

    w = synth.make_nextn_inputs(NEXTN)
    m = w.model
    B, N, V = w.B, w.N, m.vocab
    dev = upload_nextn(w)
    ws = mtp.alloc_workspace(max(int(dev.ws.numel()), mtp.workspace_size(None, B, N, V)))
    dev.ws = ws
    drafts = torch.empty((B, N), dtype=torch.int32, device="cuda")
    h_last = torch.empty((B, m.d), dtype=torch.float32, device="cuda")
    # every call writes the same drafter-KV rows (kv_len is not advanced): the timed calls repeat one call
    dev.run(drafts, h_last)
    torch.cuda.synchronize()
    if mtp.last_error(ws) != 0:
        raise RuntimeError(f"NextN drafter status {mtp.last_error(ws)}")
    d_host = drafts.cpu().numpy()
    vin = synth.make_verify_greedy_inputs(NEXTN, B=B, N=N, V=V)
    logits_np = synth.plant_greedy_logits(synth.bf16_bits_to_f32(vin.logits), d_host, vin.planted, vin.dtype)
    logits = to_device(logits_np, vin.dtype)
    out_tok = torch.empty((B, N + 1), dtype=torch.int32, device="cuda")
    n_acc = torch.empty((B,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        dev.run(drafts, h_last)
        mtp.verify_greedy(logits, drafts, out_tok, n_acc, ws)
    torch.cuda.synchronize()
    assert mtp.last_error(ws) == 0
    if not np.array_equal(n_acc.cpu().numpy(), vin.planted):
        raise RuntimeError("NextN verify disagrees with the planted accept lengths")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        a, b_, c = ev[i]
        a.record(stream)
        dev.run(drafts, h_last)
        b_.record(stream)
        mtp.verify_greedy(logits, drafts, out_tok, n_acc, ws)
        c.record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clocks.pause()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    draft_ms = [e[0].elapsed_time(e[1]) for e in ev]
    verify_ms = [e[1].elapsed_time(e[2]) for e in ev]
    value = world * B * N * args.steps / (total_ms / 1e3)

    # end to end: the call's inputs up from pinned host memory, the tokens back
    host = {n: getattr(dev, n).cpu().pin_memory() for n in ("last_tok", "h_prev", "kv_len", "n_cu", "cu_tok", "cu_h")}
    h_logits = torch.empty(logits.shape, dtype=logits.dtype).pin_memory()
    h_logits.copy_(logits.cpu())
    h_out = torch.empty((B, N + 1), dtype=torch.int32).pin_memory()
    h_n = torch.empty((B,), dtype=torch.int32).pin_memory()
    h_dr = torch.empty((B, N), dtype=torch.int32).pin_memory()
    bi = sum(t.numel() * t.element_size() for t in host.values()) + h_logits.numel() * h_logits.element_size()
    bo = (h_out.numel() + h_n.numel() + h_dr.numel()) * 4

    def e2e_step():
        for n, t in host.items():
            getattr(dev, n).copy_(t, non_blocking=True)
        logits.copy_(h_logits, non_blocking=True)
        dev.run(drafts, h_last)
        mtp.verify_greedy(logits, drafts, out_tok, n_acc, ws)
        h_dr.copy_(drafts, non_blocking=True)
        h_out.copy_(out_tok, non_blocking=True)
        h_n.copy_(n_acc, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.start()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.pause()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    if not np.array_equal(h_n.numpy(), vin.planted):
        raise RuntimeError("end-to-end NextN verify disagrees with the planted accept lengths")

    peak, peak_kind = measured_peaks()
    alg = nextn_bytes_per_launch(w)
    achieved = alg / (statistics.mean(draft_ms) / 1e3) / 1e9
    fields = {
        "value": round(value, 2), "ms_per_step": round(total_ms / args.steps, 4),
        "config": nextn_config(w, world),
        "breakdown": {"draft_ms_mean": round(statistics.mean(draft_ms), 4),
                      "verify_ms_mean": round(statistics.mean(verify_ms), 4)},
        "e2e": {"value": round(world * B * N * args.steps / (e2e_ms / 1e3), 2), "unit": UNIT,
                "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo)},
        "roofline": {"bound": "hbm", "kernel": "draft_kernel (NextN)", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": alg, "traffic": recorded_traffic(w.name)},
        "gpu_launches": 2 * args.steps,
        "dtype": m.dtype,
    }
    return fields, w


def bench_verify_sample(args, world, clocks):
    """Exact temp > 0 verification alone (workload 4).  Returns (fields, inputs)."""
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import to_device

    inp = synth.make_verify_sample_inputs()
    B, R, V = inp.target.shape
    N = R - 1
    tg, df = to_device(inp.target, inp.dtype), to_device(inp.draft, inp.dtype)
    hi = torch.from_numpy(np.ascontiguousarray(inp.hist, dtype=np.int32)).cuda()
    out = torch.empty((B, R), dtype=torch.int32, device="cuda")
    n_acc = torch.empty((B,), dtype=torch.int32, device="cuda")
    ws = mtp.alloc_workspace(mtp.workspace_size(None, B, N, V))
    # the drafter's tokens: draws from q_i = sample_dist(draft row i), untimed
    dr = torch.empty((B, N), dtype=torch.int32, device="cuda")
    mtp.sample_drafts(df, hi, inp.params, inp.seed, inp.offset, dr, ws)
    torch.cuda.synchronize()
    if mtp.last_error(ws) != 0:
        raise RuntimeError(f"sample_drafts status {mtp.last_error(ws)}")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i):
        mtp.verify_sample(tg, df, dr, hi, inp.params, inp.seed, i, out, n_acc, ws)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    if mtp.last_error(ws) != 0:
        raise RuntimeError(f"verify_sample status {mtp.last_error(ws)}")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for i in range(args.steps):
        flush.fill_(float(i))   # evict the logits from L2
        ev[i][0].record(stream)
        step(1000 + i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks.pause()
    if mtp.last_error(ws) != 0:
        raise RuntimeError(f"verify_sample status {mtp.last_error(ws)}")
    ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(ms), world)
    value = world * B * N * args.steps / (total_ms / 1e3)

    # end-to-end through the public API with pinned host buffers: the logits,
    # drafts and history go up, the emitted tokens and accept counts come back
    h_tg = torch.empty(tg.shape, dtype=tg.dtype).pin_memory()
    h_tg.copy_(tg.cpu())
    h_df = torch.empty(df.shape, dtype=df.dtype).pin_memory()
    h_df.copy_(df.cpu())
    h_dr = dr.cpu().pin_memory()
    h_hi = hi.cpu().pin_memory()
    h_out = torch.empty((B, R), dtype=torch.int32).pin_memory()
    h_n = torch.empty((B,), dtype=torch.int32).pin_memory()
    bi = sum(t.numel() * t.element_size() for t in (h_tg, h_df, h_dr, h_hi))
    bo = h_out.numel() * 4 + h_n.numel() * 4

    def e2e_step(i):
        tg.copy_(h_tg, non_blocking=True)
        df.copy_(h_df, non_blocking=True)
        dr.copy_(h_dr, non_blocking=True)
        hi.copy_(h_hi, non_blocking=True)
        step(i)
        h_out.copy_(out, non_blocking=True)
        h_n.copy_(n_acc, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.start()
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(2000 + i)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.pause()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = world * B * N * args.steps / (e2e_ms / 1e3)

    peak, peak_kind = measured_peaks()
    alg = verify_sample_bytes(inp)
    achieved = alg / (statistics.mean(ms) / 1e3) / 1e9
    fields = {
        "value": round(value, 2), "ms_per_step": round(total_ms / args.steps, 4),
        "config": sample_config(inp, world),
        "breakdown": {"verify_ms_mean": round(statistics.mean(ms), 4),
                      "n_accept_mean": round(float(n_acc.float().mean().item()), 4)},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": int(bi),
                "d2h_bytes_per_step": int(bo)},
        "roofline": {"bound": "hbm", "kernel": "sample_kernel", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": alg, "traffic": recorded_traffic(synth.WORKLOADS[4])},
        "gpu_launches": args.steps,
        "dtype": inp.dtype,
    }
    return fields, inp


# ----------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample of the workload
# ----------------------------------------------------------------------------

def _timed_units(run_unit, min_seconds):
    reps, t0 = 0, time.perf_counter()
    while True:
        run_unit(reps)
        reps += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    return reps, time.perf_counter() - t0


def cpu_baseline_draft(w, min_seconds: float = 8.0) -> dict:
    """Whole draft blocks of single sequences (cycling through the batch, N
    steps each) + their greedy verify rows, on all host cores until
    min_seconds of work, then one sequence on one core."""
    import oracle
    vin = synth.make_verify_greedy_inputs(0 if w.model.dtype == "f32" else 1, B=1, N=w.N, V=w.model.vocab)

    def unit(r):
        oracle.draft_block(w, seqs=[r % w.B], want_logits=False)
        oracle.verify_greedy(vin.logits, vin.dtype, vin.drafts)

    cores = oracle.num_threads()
    reps, dt = _timed_units(unit, min_seconds)
    oracle.set_threads(1)
    try:
        t0 = time.perf_counter()
        unit(0)
        dt1 = time.perf_counter() - t0
    finally:
        oracle.set_threads(cores)
    return {"value": round(reps * w.N / dt, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} single-sequence draft blocks (N={w.N}) + greedy verify, cycling over the "
                      f"batch's sequences, {dt:.1f} s",
            "single_thread": {"value": round(w.N / dt1, 4), "cores": 1, "sample": "one sequence's draft block"},
            "cpu_model": cpu_model()}


def cpu_baseline_nextn(w, min_seconds: float = 8.0) -> dict:
    """Whole NextN drafting calls of single sequences (catch-up rows + N
    steps) + their greedy verify rows, on all host cores until min_seconds of
    work, then one call on one core."""
    import oracle
    vin = synth.make_verify_greedy_inputs(NEXTN, B=1, N=w.N, V=w.model.vocab)

    def unit(r):
        oracle.nextn_draft(w, seqs=[r % w.B], want_logits=False)
        oracle.verify_greedy(vin.logits, vin.dtype, vin.drafts)

    cores = oracle.num_threads()
    reps, dt = _timed_units(unit, min_seconds)
    oracle.set_threads(1)
    try:
        t0 = time.perf_counter()
        unit(0)
        dt1 = time.perf_counter() - t0
    finally:
        oracle.set_threads(cores)
    return {"value": round(reps * w.N / dt, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} single-sequence NextN calls (catch-up + N={w.N}) + greedy verify, {dt:.1f} s",
            "single_thread": {"value": round(w.N / dt1, 4), "cores": 1, "sample": "one sequence's call"},
            "cpu_model": cpu_model()}


def cpu_baseline_verify_sample(inp, min_seconds: float = 8.0) -> dict:
    """The oracle's exact sampling verify, whole calls until min_seconds (the
    drafter's draws, by the oracle, untimed), then one call on one core."""
    import oracle
    inp.drafts, _ = oracle.sample_drafts(inp.draft, inp.dtype, inp.hist, inp.params, inp.seed, inp.offset)
    B, R, _ = inp.target.shape

    def unit(r):
        oracle.verify_sample(inp.target, inp.draft, inp.dtype, inp.drafts, inp.hist, inp.params, inp.seed, r)

    cores = oracle.num_threads()
    reps, dt = _timed_units(unit, min_seconds)
    oracle.set_threads(1)
    try:
        t0 = time.perf_counter()
        unit(0)
        dt1 = time.perf_counter() - t0
    finally:
        oracle.set_threads(cores)
    return {"value": round(reps * B * (R - 1) / dt, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} full verify_sample calls (B={B}, N={R - 1}), {dt:.1f} s",
            "single_thread": {"value": round(B * (R - 1) / dt1, 4), "cores": 1, "sample": "one full call"},
            "cpu_model": cpu_model()}


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from mtp_speculative_decoding_gb300 import build as mtp_build
    mtp_build.build()
    clocks = ClockSampler(local)
    want_cpu = rank == 0 and not args.no_cpu_baseline

    order = [args.workload] if args.workload is not None else [HEADLINE] + list(OTHERS)
    results = {}
    reuse = None
    for wid in order:
        if wid == 4:
            fields, inp = bench_verify_sample(args, world, clocks)
            if want_cpu:
                fields["cpu_baseline"] = cpu_baseline_verify_sample(inp)
            del inp
        elif wid == NEXTN:
            reuse = None   # a different model: the assistant's weights go
            torch.cuda.empty_cache()
            fields, w = bench_nextn(args, world, clocks)
            if want_cpu:
                fields["cpu_baseline"] = cpu_baseline_nextn(w)
            del w
        else:
            fields, dev, w = bench_draft(wid, args, world, clocks, reuse=reuse)
            if want_cpu:
                fields["cpu_baseline"] = cpu_baseline_draft(w)
            reuse = dev if w.model.dtype == "bf16" else None
            del w
        results[wid] = fields
        torch.cuda.synchronize()
    del reuse
    torch.cuda.empty_cache()

    head = results[order[0]]
    result = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
        "data": "synthetic (seeded; random-init weights of the workloads' shapes)",
        "config": head["config"], "e2e": head["e2e"], "roofline": head["roofline"],
        "breakdown": head["breakdown"],
        "gpu_launches": sum(r["gpu_launches"] for r in results.values()),
        "clocks": clocks.summary(),
    }
    if len(order) > 1:   # the other workloads, each with the same fields as the headline
        result["per_workload"] = {results[wid]["config"]["workload"]: {
            k: results[wid][k] for k in ("value", "ms_per_step", "config", "breakdown", "e2e", "roofline",
                                         "cpu_baseline", "gpu_launches") if k in results[wid]}
            for wid in order[1:]}
    if "cpu_baseline" in head:
        result["cpu_baseline"] = head["cpu_baseline"]
    if rank == 0:
        print(json.dumps(result))


# ----------------------------------------------------------------------------
# reference arm: the oracle on the host cores, same config as ours
# ----------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    wid = HEADLINE if args.workload is None else args.workload
    if wid == 4:
        inp = synth.make_verify_sample_inputs()
        inp.drafts, _ = oracle.sample_drafts(inp.draft, inp.dtype, inp.hist, inp.params, inp.seed, inp.offset)
        B, R, _ = inp.target.shape
        for i in range(args.warmup):
            oracle.verify_sample(inp.target, inp.draft, inp.dtype, inp.drafts, inp.hist, inp.params, inp.seed, i)
        times = []
        for i in range(args.steps):
            t0 = time.perf_counter()
            oracle.verify_sample(inp.target, inp.draft, inp.dtype, inp.drafts, inp.hist, inp.params, inp.seed, 1000 + i)
            times.append(time.perf_counter() - t0)
        units = B * (R - 1) * args.steps
        config = sample_config(inp, world)
        sample = f"{args.steps} full verify_sample calls"
        dtype = "f32"
    elif wid == NEXTN:
        w = synth.make_nextn_inputs(NEXTN)
        vin = synth.make_verify_greedy_inputs(NEXTN, B=1, N=w.N, V=w.model.vocab)
        for r in range(args.warmup):
            oracle.nextn_draft(w, seqs=[r % w.B], want_logits=False)
        times = []
        for r in range(args.steps):
            t0 = time.perf_counter()
            oracle.nextn_draft(w, seqs=[r % w.B], want_logits=False)
            oracle.verify_greedy(vin.logits, vin.dtype, vin.drafts)
            times.append(time.perf_counter() - t0)
        units = w.N * args.steps
        config = nextn_config(w, world)
        sample = f"{args.steps} single-sequence NextN calls + greedy verify"
        dtype = "f64"
    else:
        w = synth.make_draft_inputs(wid)
        vin = synth.make_verify_greedy_inputs(0 if w.model.dtype == "f32" else 1, B=1, N=w.N, V=w.model.vocab)
        # each step: one sequence's draft block (cycling over the batch) + its verify rows
        for r in range(args.warmup):
            oracle.draft_block(w, seqs=[r % w.B], want_logits=False)
        times = []
        for r in range(args.steps):
            t0 = time.perf_counter()
            oracle.draft_block(w, seqs=[r % w.B], want_logits=False)
            oracle.verify_greedy(vin.logits, vin.dtype, vin.drafts)
            times.append(time.perf_counter() - t0)
        units = w.N * args.steps
        config = draft_config(w, world)
        sample = f"{args.steps} single-sequence draft blocks + greedy verify, cycling over the batch"
        dtype = "f64"
    tot = sum(times)
    value = units / tot
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
            "data": "synthetic (seeded; random-init weights of the workloads' shapes)", "config": config,
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
