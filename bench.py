#!/usr/bin/env python
"""Decode-step benchmark of the paged sparse/sliding-window MQA decode path.

A step is one full decode call over a batch: dsa_decode_run (gather +
dequant + attention, one fused kernel) then dsa_decode_combine (split-KV
merge). Default workload: 1024 decode tokens, 64 query heads, fp8 sliding
window list of 128 over a 2^16-slot cache plus a 4096-wide NVFP4 list over a
4M-slot (1.2 GB) cache, sink and RoPE on -- the bandwidth-stress
configuration at its largest batch. All inputs are seeded synthetic data.

Prints ONE JSON line (rank 0). ``--impl reference`` times the fp64 CPU oracle
instead (the reference arm); ``--gpus N`` under torchrun runs N replicas.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from swa_paged_decode_gb300 import workloads as W  # noqa: E402

METRIC = "decode tokens/s; gathered-KV HBM GB/s as % of GB300 peak (1 GPU)"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20        # > 2x the 126 MB L2
MX_GROUP = 8   # heads per o-fused output group of the V4.1 variant (open on the pages)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic of tc_decode_kernel<64> from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum, one launch of the
# bandwidth-stress workload at 256 tokens), per gathered KV row; valid only
# while the kernel sources hash to `sources`. The capture is summarised under
# profiles/ with the command that made it.
NCU_TRAFFIC = {
    "sources": "0024d884f97371c5",
    "workload": "config5_T256_H64",
    "bytes_per_launch": 444022784 + 26824192,
    "rows_per_launch": 256 * (128 + 4096),
}
KERNEL_SOURCES = ("swa_paged_decode_gb300/csrc/dsa_tc.cu", "swa_paged_decode_gb300/csrc/tc_ptx.cuh",
                  "swa_paged_decode_gb300/csrc/dsa_internal.cuh")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=5, help="workload 1..5")
    ap.add_argument("--variant", choices=["base", "v41", "model1", "v32"], default="base",
                    help="v41: ue8m0 fp8 records, GPT-J RoPE, MXFP8 o-fused output "
                         f"({MX_GROUP} heads per group); model1: MODEL1 (584 B) records "
                         "in place of the fp8-528 lists; v32: V3.2 (656 B, 576-dim keys) "
                         "records in every list, no RoPE")
    ap.add_argument("--tokens", type=int, default=None, help="batch size (default: config's)")
    ap.add_argument("--per-config", dest="per_config", action="store_true", default=True)
    ap.add_argument("--quick", dest="per_config", action="store_false",
                    help="skip the per-configuration table")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false", default=True)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU work for the oracle baseline sample")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------ accounting

def kept_rows(w: W.Workload) -> torch.Tensor:
    """Per-token kept rows per list (bench-side accounting of the algorithmic
    work: positions below clamp(len, 0, width) whose id is a cache slot)."""
    cnt = []
    for c, l in ((w.swa_cache, w.swa), (w.extra_cache, w.extra)):
        if l is None:
            continue
        r = torch.arange(l.width, device=l.ids.device)[None, :]
        lim = l.lens.clamp(0, l.width).to(torch.int64)[:, None]
        ok = (r < lim) & (l.ids >= 0) & (l.ids.to(torch.int64) < c.num_slots)
        cnt.append((ok.sum(1), c.record_bytes))
    return cnt


def algorithmic(w: W.Workload, mx: bool = False):
    cnt = kept_rows(w)
    rows = sum(int(k.sum()) for k, _ in cnt)
    gathered = sum(int(k.sum()) * rb for k, rb in cnt)
    dqk = int(w.q.shape[-1])                     # 512, or 576 with V3.2 records
    flops = 2 * (dqk + W.HEAD_DIM) * w.H * rows  # QK^T (dqk) and PV (512), 2 flops per MAC
    ids_bytes = 4 * (w.swa.width + (0 if w.extra is None else w.extra.width)) * w.T
    out_bytes = w.T * w.H * (W.HEAD_DIM + W.HEAD_DIM // 32) if mx else w.T * w.H * W.HEAD_DIM * 2
    io_bytes = w.T * w.H * dqk * 2 + out_bytes + w.T * w.H * 4   # q in, out, lse
    return dict(rows=rows, gathered_bytes=gathered, flops=flops,
                total_bytes=gathered + ids_bytes + io_bytes)


# ------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock / throttle reasons while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return self
        # start timing only once the sampler is producing lines
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            self.file.flush()
            if os.path.getsize(f"/proc/self/fd/{self.file.fileno()}") > 0:
                break
            time.sleep(0.02)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.file is None or self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ GPU arm

class Step:
    def __init__(self, w: W.Workload, B, mx: bool = False):
        self.w = w
        self.B = B
        self.mx = mx
        self.dec = B.Decoder(w, mx_group=MX_GROUP if mx else None)
        self.has_combine = self.dec.plan.split_tokens > 0 and not self.dec.plan.merge_in_run

    def __call__(self, ev_k0=None, ev_k1=None):
        w, B, d = self.w, self.B, self.dec
        ei = None if w.extra is None else w.extra.ids
        el = None if w.extra is None else w.extra.lens
        if ev_k0 is not None:
            ev_k0.record()
        if self.mx:
            B.dsa_decode_run_v41(d.plan, d.workspace, w.q, w.swa_cache, w.swa.ids, w.swa.lens,
                                 w.extra_cache, ei, el, w.sink, w.positions, w.cos_sin,
                                 w.rope_style, w.scale, None, d.mx, d.lse)
        else:
            B.dsa_decode_run(d.plan, d.workspace, w.q, w.swa_cache, w.swa.ids, w.swa.lens,
                             w.extra_cache, ei, el, w.sink, w.positions, w.cos_sin, w.scale,
                             d.out, d.lse)
        if ev_k1 is not None:
            ev_k1.record()
        if self.mx:
            B.dsa_decode_combine_v41(d.plan, d.workspace, w.sink, w.positions, w.cos_sin,
                                     w.rope_style, None, d.mx, d.lse)
        else:
            B.dsa_decode_combine(d.plan, d.workspace, w.sink, d.out, d.lse)


def rank_barrier(world: int):
    """Barrier across the replicas (one process per GPU); no-op alone."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest replica's figure (every rank gets it)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_steps(step: Step, steps: int, warmup: int, flush: torch.Tensor, clocks=None,
               world: int = 1):
    """Timed region: `steps` whole steps (run then combine issued back to
    back, as a caller issues them; L2 flushed before each), events only
    around each step. Then, outside it, a second pass with events around
    the decode kernel alone (an event between run and combine would hold
    back the combine's programmatic early launch, so it is not in the timed
    steps)."""
    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    rank_barrier(world)            # all replicas start the timed region together
    torch.cuda.synchronize()
    E = lambda: torch.cuda.Event(enable_timing=True)
    evs = [(E(), E()) for _ in range(steps)]
    ctx = clocks if clocks is not None else _Null()
    with ctx:
        for s0, s1 in evs:
            flush.zero_()
            s0.record()
            step()
            s1.record()
        torch.cuda.synchronize()
    rank_barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    kev = [(E(), E()) for _ in range(steps)]
    for k0, k1 in kev:
        flush.zero_()
        step(k0, k1)
    torch.cuda.synchronize()
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    return sum(step_ms), step_ms, kern_ms


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def e2e_steps(w: W.Workload, B, steps: int, warmup: int, mx: bool = False):
    """Same step through the public API from pinned HOST buffers: per step the
    per-token inputs (Q, slot lists, lengths, positions) go host->device and
    out + lse come back device->host inside the timed region. The caches and
    the sink (model state) stay resident.

    Steps are double-buffered as a serving loop runs them: step k's inputs
    are copied on one copy stream while step k-1 computes, and step k-1's
    result is copied back on another; two sets of device buffers alternate.
    The timed region spans all `steps` steps, from the first copy in to the
    last copy out.

    No L2 flush here: the cache (1.2 GB at the headline workload) is larger
    than L2, and consecutive steps gather different records -- odd steps
    use the slot ids shifted by half the cache (mod its slot count; -1
    stays -1), the same lengths and the same amount of work -- so no step
    finds the previous step's records in L2."""
    names = ["q", "swa_ids", "swa_lens"] + (["extra_ids", "extra_lens"] if w.extra is not None else []) \
        + (["positions"] if w.positions is not None else [])
    src = {"q": w.q, "swa_ids": w.swa.ids, "swa_lens": w.swa.lens,
           "extra_ids": None if w.extra is None else w.extra.ids,
           "extra_lens": None if w.extra is None else w.extra.lens, "positions": w.positions}
    host = {n: src[n].cpu().pin_memory() for n in names}

    def shifted(ids, slots):
        v = ids.cpu()
        return torch.where(v >= 0, (v.to(torch.int64) + slots // 2) % slots, v).to(ids.dtype).pin_memory()

    host_odd = dict(host)
    host_odd["swa_ids"] = shifted(w.swa.ids, w.swa_cache.num_slots)
    if w.extra is not None:
        host_odd["extra_ids"] = shifted(w.extra.ids, w.extra_cache.num_slots)
    hosts = [host, host_odd]
    dec = B.Decoder(w, mx_group=MX_GROUP if mx else None)
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    E = lambda: torch.cuda.Event()
    pinned = lambda t: torch.empty(t.shape, dtype=t.dtype).pin_memory()
    sets = []
    for _ in range(2):
        if mx:
            m = B.MxOut(w.T, w.H, MX_GROUP, w.q.device)
            outs = {"mx": m, "res": [m.data, m.scale]}
        else:
            o = torch.empty_like(dec.out)
            outs = {"out": o, "res": [o]}
        lse = torch.empty_like(dec.lse)
        outs["res"].append(lse)
        sets.append(dict(outs, dev={n: torch.empty_like(src[n]) for n in names}, lse=lse,
                         res_h=[pinned(t) for t in outs["res"]],
                         in_ready=E(), comp_done=E(), out_done=E(), used=False))
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = sum(t.numel() * t.element_size() for t in sets[0]["res"])

    def step(k):
        b = sets[k % 2]
        if b["used"]:                       # its previous result has been read back
            s_in.wait_event(b["out_done"])
        b["used"] = True
        with torch.cuda.stream(s_in):
            for n in names:
                b["dev"][n].copy_(hosts[k % 2][n], non_blocking=True)
            b["in_ready"].record(s_in)
        comp.wait_event(b["in_ready"])
        d = b["dev"]
        if mx:
            B.dsa_decode_run_v41(dec.plan, dec.workspace, d["q"], w.swa_cache, d["swa_ids"],
                                 d["swa_lens"], w.extra_cache, d.get("extra_ids"),
                                 d.get("extra_lens"), w.sink, d.get("positions"), w.cos_sin,
                                 w.rope_style, w.scale, None, b["mx"], b["lse"], comp)
            B.dsa_decode_combine_v41(dec.plan, dec.workspace, w.sink, d.get("positions"),
                                     w.cos_sin, w.rope_style, None, b["mx"], b["lse"], comp)
        else:
            B.dsa_decode_run(dec.plan, dec.workspace, d["q"], w.swa_cache, d["swa_ids"],
                             d["swa_lens"], w.extra_cache, d.get("extra_ids"),
                             d.get("extra_lens"), w.sink, d.get("positions"), w.cos_sin, w.scale,
                             b["out"], b["lse"], comp)
            B.dsa_decode_combine(dec.plan, dec.workspace, w.sink, b["out"], b["lse"], comp)
        b["comp_done"].record(comp)
        s_out.wait_event(b["comp_done"])
        with torch.cuda.stream(s_out):
            for hst, dv in zip(b["res_h"], b["res"]):
                hst.copy_(dv, non_blocking=True)
            b["out_done"].record(s_out)

    for k in range(warmup):
        step(k)
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    s_in.wait_stream(comp)
    for k in range(steps):
        step(k)
    comp.wait_stream(s_out)
    e.record(comp)
    e.synchronize()
    return a.elapsed_time(e), h2d, d2h


def roofline(w: W.Workload, alg, kern_ms_avg: float, peaks, peak_kind, captured: bool = True):
    hbm = peaks["hbm_gbs"]
    tf = peaks["bf16_tflops"]
    intensity = alg["flops"] / max(alg["gathered_bytes"], 1)
    ridge = tf * 1e12 / (hbm * 1e9)
    s = kern_ms_avg * 1e-3
    if intensity > ridge:
        ach = alg["flops"] / s / 1e12
        r = {"bound": "tensor", "achieved": ach, "peak": tf, "unit": "TFLOP/s",
             "frac": ach / tf}
    else:
        ach = alg["gathered_bytes"] / s / 1e9
        r = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm}
    r["traffic"] = ncu_traffic(alg["rows"]) if captured else None
    r["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback"
    r["intensity_flop_per_byte"] = intensity
    r["kernel_ms"] = kern_ms_avg
    return r


def sources_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(rows: int):
    """Captured DRAM bytes per launch scaled to `rows` gathered rows (the
    traffic grows with the rows: same per-token lists, more tokens); None
    once the kernel sources differ from the captured ones."""
    if sources_hash() != NCU_TRAFFIC["sources"]:
        return None
    return int(NCU_TRAFFIC["bytes_per_launch"] * rows / NCU_TRAFFIC["rows_per_launch"])


def gpu_arm(args, rank, world, B, peaks, peak_kind):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    mx = args.variant == "v41"
    w = W.make_config(args.config, T=args.tokens, device=dev, v41=mx,
                      model1=args.variant == "model1", v32=args.variant == "v32")
    alg = algorithmic(w, mx)
    step = Step(w, B, mx)
    clocks = ClockSampler(dev.index)
    total_ms, step_ms, kern_ms = time_steps(step, args.steps, args.warmup, flush, clocks, world)
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = w.T * world / (ms_per_step * 1e-3)
    kern_avg = sum(kern_ms) / len(kern_ms)
    e2e_ms, h2d, d2h = e2e_steps(w, B, max(3, args.steps // 2), args.warmup, mx)
    e2e_value = w.T * world / (e2e_ms / max(3, args.steps // 2) * 1e-3)
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if step.dec.plan.kernel == 1 else "fp32",
        "dtype_detail": ("tcgen05 kind::f16 MMAs on f16 tiles (fp8 rows normalized per row "
                         "by a power of two), fp32 accumulate and softmax, bf16 out"
                         if step.dec.plan.kernel == 1 else "CUDA-core fp32, bf16 out"),
        "data": "synthetic (seeded N(0,1) rows quantized to fp8/NVFP4 records, random slot lists)",
        "config": {"workload": w.name, "T": w.T, "H": w.H,
                   "swa": f"{W.FMT_NAMES[w.swa_cache.fmt]} w{w.swa.width} page "
                          f"{w.swa_cache.page_size} {w.swa_cache.num_slots} slots",
                   "extra": None if w.extra is None else
                   f"{W.FMT_NAMES[w.extra_cache.fmt]} w{w.extra.width} page "
                   f"{w.extra_cache.page_size} {w.extra_cache.num_slots} slots",
                   "sink": w.sink is not None, "rope": w.cos_sin is not None,
                   "rope_style": ["neox", "gptj"][w.rope_style],
                   "out": f"mxfp8 o-fused, {MX_GROUP} heads per group" if mx else "bf16",
                   "global_batch": w.T * world,
                   "l2": ("value: flushed (256 MiB write before every step); e2e: not flushed, "
                          "the cache is larger than L2 and odd steps gather other records "
                          "(slot ids shifted by half the cache)"),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "kernel": ["simt", "tcgen05"][step.dec.plan.kernel]},
        "gathered_hbm": {"bytes_per_step": alg["gathered_bytes"],
                         "gbs": alg["gathered_bytes"] / (kern_avg * 1e-3) / 1e9,
                         "frac_of_peak": alg["gathered_bytes"] / (kern_avg * 1e-3) / 1e9 / peaks["hbm_gbs"],
                         "gbs_step": alg["gathered_bytes"] / (ms_per_step * 1e-3) / 1e9},
        "roofline": roofline(w, alg, kern_avg, peaks, peak_kind, captured=args.variant == "base"),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        # decode, combine (when a token is split), MXFP8 cast (V4.1 output)
        "gpu_launches": args.steps * (1 + (1 if step.has_combine else 0) + (1 if mx else 0)),
        "clocks": clocks.summary(),
    }
    return res, w, step


def per_config_table(B, peaks, peak_kind, steps=20, warmup=3):
    dev = torch.device("cuda", torch.cuda.current_device())
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    rows = []
    for k, T in [(1, None), (2, None), (3, None), (4, None)] + [(5, t) for t in W.CONFIG5_BATCHES]:
        w = W.make_config(k, T=T, device=dev)
        alg = algorithmic(w)
        step = Step(w, B)
        total, step_ms, kern_ms = time_steps(step, steps, warmup, flush)
        med = statistics.median(step_ms)
        kmed = statistics.median(kern_ms)
        rows.append({"workload": w.name, "tokens_per_s": w.T / (med * 1e-3),
                     "ms_step_median": med, "ms_kernel_median": kmed,
                     "gathered_gbs": alg["gathered_bytes"] / (kmed * 1e-3) / 1e9,
                     "gathered_frac_hbm": alg["gathered_bytes"] / (kmed * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "tflops": alg["flops"] / (kmed * 1e-3) / 1e12,
                     "tensor_frac": alg["flops"] / (kmed * 1e-3) / 1e12 / peaks["bf16_tflops"],
                     "splits": step.dec.plan.ctas_per_group})
        del step, w
        torch.cuda.empty_cache()
    return rows


# ------------------------------------------------------------ CPU (oracle) arm

def oracle_run(a, tok, cores: int, mx: bool):
    """The oracle on tokens `tok` (and, for the V4.1 variant, its MXFP8
    output epilogue on the result); returns (out, lse, kept, checksum)."""
    import oracle
    res = oracle.decode(a["q"], a["caches"], a["lists"], scale=a["scale"], sink=a["sink"],
                        positions=a["positions"], cos_sin=a["cos_sin"],
                        rope_style=a["rope_style"], tokens=tok, nthreads=cores)
    if mx:
        pos = None if a["positions"] is None else a["positions"].cpu().numpy()[tok]
        oracle.mxfp8_epilogue(res[0], group_size=MX_GROUP, positions=pos, cos_sin=a["cos_sin"],
                              rope_style=a["rope_style"])
    return res


def oracle_timing(w: W.Workload, target_s: float, seed: int = 0, mx: bool = False,
                  max_s: float = 90.0):
    """Time the fp64 oracle on workload w, on every host core and on one.

    All cores: every token of the workload when that fits in ``max_s``
    seconds (estimated from a first sample of one token per core), else a
    seeded sample of about ``target_s`` seconds. The oracle's results on
    these tokens are returned for the parity record. One core: a seeded
    sample of about target_s / 3 seconds.
    Returns (cpu_baseline dict, (tokens, oracle out, lse, kept, checksum))."""
    import numpy as np

    a = W.oracle_args(w)
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(seed)
    n = min(w.T, cores)
    tok = np.sort(rng.choice(w.T, size=n, replace=False))
    t0 = time.perf_counter()
    oracle_run(a, tok, cores, mx)
    per_tok = (time.perf_counter() - t0) / n
    n2 = w.T if w.T * per_tok <= max_s else int(max(1, min(w.T, target_s / max(per_tok, 1e-9))))
    tok = np.arange(w.T) if n2 == w.T else np.sort(rng.choice(w.T, size=n2, replace=False))
    t0 = time.perf_counter()
    res = oracle_run(a, tok, cores, mx)
    dt = time.perf_counter() - t0
    n1 = int(max(1, min(w.T, target_s / 3 / max(per_tok * cores, 1e-9))))
    tok1 = np.sort(rng.choice(w.T, size=n1, replace=False))
    t0 = time.perf_counter()
    oracle_run(a, tok1, 1, mx)
    dt1 = time.perf_counter() - t0
    base = {"value": n2 / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n2} of {w.T} tokens of {w.name} (fp64 C oracle, {cores} threads), {dt:.1f} s",
            "one_core": {"value": n1 / dt1, "unit": UNIT, "cores": 1,
                         "sample": f"{n1} of {w.T} tokens, 1 thread, {dt1:.1f} s"}}
    return base, (tok, *res)


def parity_record(step: "Step", ref, mx: bool):
    """GPU output of the timed workload (the buffers of the last timed step;
    every step decodes the same inputs) against the oracle on the tokens it
    evaluated, with the decode tolerances: out max |err| <= 2e-2 and
    per-(token, head) cosine >= 0.9999 against the fp64 oracle, |dlse| <=
    1e-3, row selection (kept count, checksum) bit-exact. For MXFP8 output
    each dequantized value must lie within 2e-2 plus half an e4m3 step of
    the oracle epilogue's input (and its scale byte within 1)."""
    import numpy as np

    tok, r_out, r_lse, r_kept, r_chk = ref
    d = step.dec
    kept, chk = d.selection()
    if d.lse.is_cuda:
        torch.cuda.synchronize()
    ti = torch.as_tensor(tok, device=d.lse.device, dtype=torch.long)
    lse = d.lse.index_select(0, ti).double().cpu().numpy()
    k = kept.index_select(0, ti).cpu().numpy()
    c = chk.index_select(0, ti).cpu().numpy().view(np.uint32)
    fin = np.isfinite(r_lse)
    rec = {"tokens_checked": int(len(tok)), "of_tokens": int(step.w.T),
           "selection_exact": bool(np.array_equal(k, r_kept) and np.array_equal(c, r_chk)),
           "lse_inf_pattern_exact": bool(np.array_equal(np.isfinite(lse), fin)),
           "max_abs_dlse": float(np.abs(lse[fin] - r_lse[fin]).max()) if fin.any() else 0.0}
    if not mx:
        o = d.out.index_select(0, ti).double().cpu().numpy()
        rec["max_abs_err"] = float(np.abs(o - r_out).max())
        rn, on = np.linalg.norm(r_out, axis=-1), np.linalg.norm(o, axis=-1)
        nz = rn > 0
        cos = (o * r_out).sum(-1)[nz] / np.maximum(on[nz] * rn[nz], 1e-300)
        rec["min_cosine"] = float(cos.min()) if cos.size else 1.0
        rec["zero_rows_exact"] = bool(np.all(o[~nz] == 0))
        ok_out = rec["max_abs_err"] <= 2e-2 and rec["min_cosine"] >= 0.9999 and rec["zero_rows_exact"]
    else:
        import oracle
        w = step.w
        G = d.mx.group_size
        pos = None if w.positions is None else w.positions.cpu().numpy()[tok]
        _, r_sc, x = oracle.mxfp8_epilogue(r_out, group_size=G, positions=pos,
                                           cos_sin=None if w.cos_sin is None else w.cos_sin.cpu(),
                                           rope_style=w.rope_style)
        table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
        sc = d.mx.scale_bytes().index_select(0, ti).cpu().numpy().astype(np.int64)
        got = table[d.mx.data.index_select(0, ti).cpu().numpy()] * \
            np.repeat(np.ldexp(1.0, sc - 127), 32, axis=-1)
        n, H = x.shape[:2]
        want = x.astype(np.float64).reshape(n, H // G, G, 16, 32).transpose(0, 1, 3, 2, 4)
        want = want.reshape(n, H // G, G * 512)
        err = np.abs(got - want)
        rec["max_abs_err"] = float(err.max())
        rec["mx_values_within_bound"] = bool(np.all(err <= 2e-2 + np.abs(want) * 2.0 ** -4 * 1.001))
        rec["mx_scale_bytes_within_1"] = bool(np.all(np.abs(sc - r_sc) <= 1))
        ok_out = rec["mx_values_within_bound"] and rec["mx_scale_bytes_within_1"]
    rec["pass"] = bool(ok_out and rec["selection_exact"] and rec["lse_inf_pattern_exact"]
                       and rec["max_abs_dlse"] <= 1e-3)
    rec["tolerance"] = ("out max|err| <= 2e-2, cosine >= 0.9999, |dlse| <= 1e-3, selection exact"
                        if not mx else "MXFP8 values within 2e-2 + half an e4m3 step, scale bytes "
                        "within 1, |dlse| <= 1e-3, selection exact")
    return rec


def reference_arm(args):
    """The fp64 oracle as the reference arm: K steps, each a bounded token
    sample of the same workload, on this host's cores."""
    import numpy as np

    mx = args.variant == "v41"
    w = W.make_config(args.config, T=args.tokens, device="cpu", v41=mx,
                      model1=args.variant == "model1", v32=args.variant == "v32")
    a = W.oracle_args(w)
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(0)
    n = min(w.T, max(1, cores))
    def one():
        tok = np.sort(rng.choice(w.T, size=n, replace=False))
        t0 = time.perf_counter()
        oracle_run(a, tok, cores, mx)
        return time.perf_counter() - t0
    for _ in range(args.warmup):
        one()
    tot = sum(one() for _ in range(args.steps))
    value = n * args.steps / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "T": w.T, "H": w.H,
                                            "step": f"{n} sampled tokens"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{n} tokens per step of {w.name}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return line


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            # oracle runs on host cores only; the rendezvous is not needed
            print(json.dumps(reference_arm(args)), flush=True)
        return
    from swa_paged_decode_gb300 import binding as B
    from swa_paged_decode_gb300 import build as BLD
    if rank == 0:
        BLD.build()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        dist.barrier()
    B.load()
    peaks, peak_kind = load_peaks()
    res, w, step = gpu_arm(args, rank, world, B, peaks, peak_kind)
    if rank == 0 and world == 1:
        if args.per_config and args.variant == "base":
            res["per_config"] = per_config_table(B, peaks, peak_kind)
        if args.cpu_baseline:
            mx = args.variant == "v41"
            res["cpu_baseline"], ref = oracle_timing(w, args.cpu_seconds, mx=mx)
            res["parity"] = parity_record(step, ref, mx)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
