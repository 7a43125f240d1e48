#!/usr/bin/env python3
"""Benchmark: differentiated KV-cache compaction throughput on GB300.

One step = reset the page pool (dkv_init_pool) + one dkv_compact over the
whole batch (significance reduce, classification, page scan, quantise +
pack + scatter, table commit).  Default workload: Llama-3-8B-shaped prefill
compaction (32 layers, 16 x 4096 tokens, 32 query / 8 KV heads, page 16).

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on
the host cores instead (a bounded sample of the same workload per step).
Multi-GPU (torchrun): every rank compacts its own batch on its own GPU (the
units are independent: replicas, weak scaling); only the timing is reduced.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV tokens compacted/sec (token-rows: one token x one (layer, KV head))"
UNIT = "token-rows/s"


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="llama")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="keep only this many layers (a reduced case for profiler captures; named in config)")
    ap.add_argument("--requests", type=int, default=0,
                    help="keep only the first this-many requests (a reduced case; named in config)")
    ap.add_argument("--window", type=int, default=0,
                    help="decode: recent window W (tokens kept at K8V4; 0 = none)")
    ap.add_argument("--decode-mode", type=int, default=0, choices=[0, 1],
                    help="decode: 0 re-scores every older token, 1 only the one leaving the window")
    ap.add_argument("--scheme", type=int, default=0, choices=[0, 1, 2],
                    help="precision scheme of the pool: 0 K8V4/K4V2, 1 K8V2/K4V1, 2 K4V8/K2V4 (prefill workloads)")
    ap.add_argument("--op", default="step", choices=["step", "attention", "prefill-attention"],
                    help="decode: the generation step or the attention over the pages; prefill workloads: "
                         "the compaction step or the prefill attention that produces its significance inputs")
    return ap.parse_args()


def workload(a):
    """The named workload, cut to --layers / --requests when given."""
    import dataclasses

    from differentiated_kv_cache_dkv_gb300 import workloads as W

    w = W.get(a.workload)
    if getattr(a, "scheme", 0):
        w = dataclasses.replace(w, scheme=a.scheme)
    if a.layers:
        w = dataclasses.replace(w, L=min(a.layers, w.L))
    if a.requests:
        w = dataclasses.replace(w, lens=list(w.lens[:a.requests]))
    return w


def workload_name(a) -> str:
    name = a.workload
    if getattr(a, "op", "step") == "attention":
        name += " attention"
    if getattr(a, "op", "step") == "prefill-attention":
        name += " prefill attention"
    if getattr(a, "window", 0) or getattr(a, "decode_mode", 0):
        name += f" (window {a.window}, {'single candidate' if a.decode_mode else 'every token re-scored'})"
    if getattr(a, "scheme", 0):
        name += " " + SCHEME_NAMES[a.scheme]
    if a.layers or a.requests:
        name += f" (reduced: {a.layers or 'all'} layers, {a.requests or 'all'} requests)"
    return name


SCHEME_NAMES = {0: "K8V4/K4V2", 1: "K8V2/K4V1", 2: "K4V8/K2V4"}


# DRAM traffic of one full k_pack launch on the Llama-shaped workload, from one
# ncu capture of the same kernel on 2 of its 32 layers scaled by the units
# processed (profiles/k_pack_llama_prefill.md); valid only for the kernel
# source it was measured on.
PACK_TRAFFIC = {"workload": "llama", "source_sha1": "99bd3387b01d", "bytes": 16 * (537.732608 + 130.183424) * 1e6}

# DRAM traffic of k_reclass per algorithmic byte, from one ncu capture on 4
# layers x 64 requests of the decode workload (180.6 MB for 176.2 MB; traffic
# grows with the live rows) (profiles/decode_step.md); valid only for the
# kernel source it was measured on.  That source is decode.cu up to the next
# kernel's definition (k_candidate): k_reclass and every device helper it
# calls precede it, so later edits to the apply kernels keep the figure.
RECLASS_TRAFFIC = {"workload": "decode", "source_sha1": "a334c0a2478c", "upto": b"k_candidate(DecodeArgs a)",
                   "per_byte": (177.17376 + 3.397632) / 176.177616}


def _source_sha(name: str, upto: bytes = None):
    """First 12 hex digits of the SHA-1 of a csrc file, or of its lines before
    the first line holding `upto` (None if the file or the marker is missing)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "differentiated_kv_cache_dkv_gb300", "csrc", name), "rb") as f:
            data = f.read()
    except OSError:
        return None
    if upto is not None:
        lines = data.split(b"\n")
        cut = next((i for i, line in enumerate(lines) if upto in line), None)
        if cut is None:
            return None
        data = b"\n".join(lines[:cut])
    return hashlib.sha1(data).hexdigest()[:12]


def _pack_traffic(workload: str):
    if workload != PACK_TRAFFIC["workload"] or _source_sha("pack.cu") != PACK_TRAFFIC["source_sha1"]:
        return None
    return PACK_TRAFFIC["bytes"]


def _reclass_traffic(workload: str, alg_bytes: float):
    if workload != RECLASS_TRAFFIC["workload"] or _source_sha("decode.cu", RECLASS_TRAFFIC["upto"]) != RECLASS_TRAFFIC["source_sha1"]:
        return None
    return RECLASS_TRAFFIC["per_byte"] * alg_bytes


def scheme_bits(scheme: int) -> int:
    """K + V bits of the high class of a scheme (the low class has half)."""
    return {0: 12, 1: 10, 2: 12}[scheme]


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------- ranks -----

def max_over_ranks(ms: float, device, world: int) -> float:
    """The slowest rank's time: every rank times its own replica between two
    barriers; the whole job took as long as its slowest rank."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Units all ranks processed per second (replicas: every rank processes
    the same number of units)."""
    return world * units_per_rank / (ms_max / 1000.0)


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- oracle ----

def oracle_sample(w, seconds: float):
    """Time the CPU oracle, as it stands, on layer 0 of the workload (repeated
    until `seconds` of CPU work).  Returns (rows/s, reps, rows per rep)."""
    import oracle
    from differentiated_kv_cache_dkv_gb300 import workloads as W

    inp = W.to_numpy(W.make_inputs(w, layers=[0]))
    rows = w.T * w.Hkv
    reps, t_total = 0, 0.0
    while t_total < seconds or reps == 0:
        pool = oracle.Pool(w.Hkv * sum(-(-n // w.P) + 1 for n in w.lens), w.P)
        tab = oracle.Tables(w.R * w.Hkv, w.pmax, rows)
        t = time.perf_counter()
        st = oracle.compact(inp, w.alpha_h, w.alpha_l, pool, tab)
        t_total += time.perf_counter() - t
        assert st == oracle.OK, st
        reps += 1
    return rows * reps / t_total, reps, rows, t_total


def run_reference(a):
    """CPU oracle arm: each step compacts layer 0 of the workload on one host core."""
    from differentiated_kv_cache_dkv_gb300 import workloads as W

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload(a)
    for _ in range(a.warmup):
        oracle_sample(w, 0.0)
    times = []
    rows = w.T * w.Hkv
    for _ in range(a.steps):
        r = oracle_sample(w, 0.0)
        times.append(r[3])
    total = sum(times)
    value = rows * a.steps / total
    sample = f"layer 0 of {a.workload} ({rows} token-rows) per step, single-threaded oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": a.gpus, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": 1000.0 * total / a.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_name(a), "layers": w.L, "requests": w.R, "tokens": w.T, "Hq": w.Hq,
                   "Hkv": w.Hkv, "page_tokens": w.P},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- native ----

def run_native(a):
    import torch
    import torch.distributed as dist

    from differentiated_kv_cache_dkv_gb300 import libdkv
    from differentiated_kv_cache_dkv_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    libdkv.load()
    w = workload(a)
    dev = torch.device("cuda", local)
    inp = W.make_inputs(w, seed=W.SEED_BASE + 1000 * rank, device=dev)
    comp = libdkv.Compactor(w.L, w.R, w.Hq, w.Hkv, w.T, max(w.lens), w.P, w.pool_pages, device=dev,
                            scheme=w.scheme)
    stream = torch.cuda.current_stream()

    def step(profiler=None):
        libdkv.dkv_init_pool(comp.pool)
        comp.compact(inp, w.alpha_h, w.alpha_l, profiler=profiler)

    for _ in range(a.warmup):
        step()
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_OK
    torch.cuda.synchronize()

    # per-step workload facts (identical every step)
    rows = w.rows
    classes = comp.classes[:rows]
    n_pruned = int((classes == 0).sum())
    n_surv = rows - n_pruned
    pages = int(comp.pool.cursors[0])
    hdr = comp.tables.unit_hdr
    n_hi, n_lo = int(hdr[:, 0].sum()), int(hdr[:, 1].sum())

    prof = libdkv.Profiler(a.steps)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(a.steps):
        step(prof)
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_OK
    kt = prof.read()
    prof.close()
    kernel_ms = {n: statistics.mean(c[i] for c in kt) for i, n in enumerate(libdkv.KERNEL_NAMES)}

    ms_max = max_over_ranks(ms, dev, world)
    value = whole_job_rate(rows * a.steps, world, ms_max)

    # roofline of the dominant kernel (k_pack): algorithmic bytes per launch,
    # the per-row figure of the measurement spec (every K / V row of the batch
    # read, as the kernel's tiles do) plus the pages it writes, the free-list
    # ids, tile descriptors and unit headers it reads
    peak, peak_kind = _peaks()
    U = w.U
    pb = libdkv.dkv_page_bytes(w.scheme, w.P)
    ntiles = w.L * w.Hkv * sum(-(-n // 128) for n in w.lens)
    pack_bytes = rows * 512 + pages * (pb + 4) + ntiles * 40 + U * 16
    pack_ms = kernel_ms["k_pack"]
    pack_gbs = pack_bytes / (pack_ms / 1000.0) / 1e9
    # the whole step by the spec's count: read every K / V row, the sums and
    # counts; write the pages, class bytes, unit headers and the fwd + rev
    # entries of the allocated pages
    spec_read = rows * 512 + w.L * w.T * w.Hq * 4 + w.T * 4
    spec_write = pages * pb + rows + U * 16 + pages * (4 + 8)
    spec_gbs = (spec_read + spec_write) / (ms_max / a.steps / 1000.0) / 1e9
    # and with what the step touches besides: only surviving rows' K / V
    # count as read, but the pool reset and the full forward rows do count
    step_read = n_surv * 512 + w.L * w.T * w.Hq * 4 + w.T * 4
    step_write = rows + pages * (pb + 13) + U * (w.pmax * 4 + 16) + w.pool_pages * 13
    step_gbs = (step_read + step_write) / (ms_max / a.steps / 1000.0) / 1e9

    # end to end through the public API with host buffers
    e2e = None
    if a.e2e_steps > 0:
        host = {k: inp[k].to("cpu").pin_memory() for k in ("k", "v", "sig_sum", "sig_cnt", "lens")}
        out_hdr = torch.empty_like(hdr, device="cpu").pin_memory()
        out_cur = torch.empty(2, dtype=torch.int64).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_hdr.numel() * 4 + 16

        def e2e_step():
            for k_, t_ in host.items():
                inp[k_].copy_(t_, non_blocking=True)
            step()
            out_hdr.copy_(hdr, non_blocking=True)
            out_cur.copy_(comp.pool.cursors, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(a.e2e_steps):
            e2e_step()
        s1.record(stream)
        torch.cuda.synchronize()
        te = max_over_ranks(s0.elapsed_time(s1), dev, world)
        e2e = {"value": whole_job_rate(rows * a.e2e_steps, world, te), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": a.e2e_steps}
        del host

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        v, reps, rrows, tt = oracle_sample(w, a.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"layer 0 of {a.workload} ({rrows} token-rows) x {reps}, single-threaded, {tt:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms_max / a.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_name(a), "layers": w.L, "requests": w.R, "tokens_per_request": w.lens[0]
                       if len(set(w.lens)) == 1 else "ragged", "Hq": w.Hq, "Hkv": w.Hkv, "page_tokens": w.P,
                       "alpha_h": w.alpha_h, "alpha_l": w.alpha_l, "scheme": SCHEME_NAMES[w.scheme],
                       "rows_per_step": rows,
                       "l2": "inputs (%.1f GB) larger than L2" % ((rows * 512 + w.L * w.T * w.Hq * 4) / 1e9),
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": "k_pack", "achieved": pack_gbs, "peak": peak, "unit": "GB/s",
                         "frac": pack_gbs / peak, "peak_kind": peak_kind, "traffic": _pack_traffic(workload_name(a)),
                         "algorithmic_bytes": pack_bytes, "ms": pack_ms},
            "step_hbm_spec": {"achieved": spec_gbs, "frac": spec_gbs / peak, "bytes": spec_read + spec_write,
                              "counted": "all K/V rows, sums, counts read; pages, classes, headers, fwd+rev written"},
            "step_hbm": {"achieved": step_gbs, "frac": step_gbs / peak, "bytes": step_read + step_write,
                         "counted": "surviving K/V rows, sums, counts read; pool reset, pages, classes, full "
                                    "forward rows written"},
            "kernels_ms": kernel_ms,
            "request_tokens_per_s": value / (w.L * w.Hkv),
            "classes": {"k8v4": n_hi / rows, "k4v2": n_lo / rows, "pruned": n_pruned / rows},
            "pages_per_step": pages,
            "payload_fraction": ((scheme_bits(w.scheme)) * (n_hi + 0.5 * n_lo)) / (32 * rows),
            "gpu_launches": a.steps * (2 + libdkv.DKV_PROFILE_KERNELS),  # pool reset, 5 kernels, k_clear_hi
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------- decode ----

from differentiated_kv_cache_dkv_gb300.decode_setup import DECODE_SLACK, decode_cap, decode_prefill, decode_setup  # noqa: E402,F401


class DecodeOracleSample:
    """The oracle's generation step on a bounded sample of the decode
    workload: layer 0 of its first n_req requests, prefilled by the oracle
    (untimed) and then stepped with the same seeded updates."""

    def __init__(self, w, n_req: int = 16, window: int = 0, mode: int = 0):
        import dataclasses

        self.w = dataclasses.replace(w, L=1, lens=list(w.lens[:n_req]))
        self.window, self.mode = window, mode
        self.max_steps = int(w.extra.get("steps", 100))  # the workload's own run length
        self.steps = 0
        self._fresh()

    def _fresh(self):
        from oracle.host_decode import HostDecode

        self.hd = HostDecode(self.w, decode_cap(self.w, self.max_steps), window=self.window, mode=self.mode)
        self.local = 0

    def step(self):
        """One timed oracle step: (seconds, live token-rows).  Every
        max_steps steps the sample starts again from its prefill (untimed)."""
        from differentiated_kv_cache_dkv_gb300 import workloads as W

        if self.local == self.max_steps:
            self._fresh()
        upd = W.decode_update_inputs(self.w, self.hd.ctx, self.local)
        live = int((self.hd.ctx["ctx_lens"] + upd["new_lens"]).sum()) * self.w.Hkv
        t = time.perf_counter()
        st = self.hd.step(upd)
        dt = time.perf_counter() - t
        assert st == 0, st
        self.steps += 1
        self.local += 1
        return dt, live


def decode_oracle_sample(w, seconds: float, window: int = 0, mode: int = 0):
    """(live token-rows/s, steps, rows per step, seconds) of the oracle stepped
    until `seconds` of step time."""
    smp = DecodeOracleSample(w, window=window, mode=mode)
    t_total, rows = 0.0, 0
    while t_total < seconds or smp.steps == 0:
        dt, live = smp.step()
        t_total += dt
        rows += live
    return rows / t_total, smp.steps, rows / smp.steps, t_total


def run_native_decode(a):
    import torch

    from differentiated_kv_cache_dkv_gb300 import libdkv
    from differentiated_kv_cache_dkv_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    libdkv.load()
    w = workload(a)
    dev = torch.device("cuda", local)
    total = a.warmup + a.steps + a.e2e_steps + 1
    dec, ctx, cap, used = decode_setup(w, dev, W.SEED_BASE + 1000 * rank, total, window=a.window,
                                       mode=a.decode_mode)
    F = dec.pool.F
    stream = torch.cuda.current_stream()
    head0 = int(dec.pool.cursors[0])

    def inputs(step):
        upd = W.decode_update_inputs(w, ctx, step, device=dev)
        return upd, {"k_new": upd["k_new"], "v_new": upd["v_new"], "sig_sum": ctx["sig_sum"],
                     "sig_cnt": ctx["sig_cnt"], "ctx_lens": ctx["ctx_lens"], "new_lens": upd["new_lens"]}

    step_no = 0
    for _ in range(a.warmup):
        upd, d = inputs(step_no)
        dec.step(d, w.alpha_h, w.alpha_l)
        ctx["ctx_lens"] += upd["new_lens"]
        step_no += 1
    assert libdkv.dkv_get_status(dec.pool) == libdkv.DKV_OK

    prof = libdkv.Profiler(a.steps)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    # the step's row counts, summed on the device so that the timed loop never
    # waits on the host (a read-back here would leave the GPU idle before
    # every step's first launch)
    cnt_t = torch.zeros(3, dtype=torch.int64, device=dev)  # live rows, new rows, scored tokens
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(a.steps):
        upd, d = inputs(step_no)
        cnt_t[0] += (ctx["ctx_lens"] + upd["new_lens"]).sum()
        cnt_t[1] += upd["new_lens"].sum()
        # tokens whose significance the step reads: outside the window (mode
        # 0), or the one leaving it (mode 1), plus a classified new token
        nl = ctx["ctx_lens"] + upd["new_lens"]
        if a.decode_mode == 0:
            cnt_t[2] += (nl - a.window).clamp(min=0).sum()
        else:
            cnt_t[2] += ((ctx["ctx_lens"] - a.window >= 0) & (upd["new_lens"] > 0)).sum()
        evs[i][0].record(stream)
        dec.step(d, w.alpha_h, w.alpha_l, profiler=prof)
        evs[i][1].record(stream)
        ctx["ctx_lens"] += upd["new_lens"]
        step_no += 1
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    st = libdkv.dkv_get_status(dec.pool)
    assert st == libdkv.DKV_OK, libdkv.status_string(st)
    live_rows = int(cnt_t[0]) * w.L * w.Hkv
    new_rows = int(cnt_t[1]) * w.L * w.Hkv
    scored = int(cnt_t[2])
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs)
    kt = prof.read()
    prof.close()
    names = ("reset", "k_candidate" if a.decode_mode else "k_reclass", "k_dscan", "k_apply", "k_demote")
    kernel_ms = {n: statistics.mean(c[i] for c in kt) for i, n in enumerate(names)}
    ms_max = max_over_ranks(ms, dev, world)
    value = whole_job_rate(live_rows, world, ms_max)

    peak, peak_kind = _peaks()
    tok_per_step = live_rows / a.steps / (w.L * w.Hkv)
    sc_per_step = scored / a.steps
    rc_bytes = w.L * sc_per_step * (w.Hq * 4 + w.Hkv) + sc_per_step * 4
    rc_name = names[1]
    rc_ms = kernel_ms[rc_name]
    rc_gbs = rc_bytes / (rc_ms / 1000.0) / 1e9
    step_gbs = rc_bytes / (ms_max / a.steps / 1000.0) / 1e9

    e2e = None
    if a.e2e_steps > 0:
        # end to end: this step's inputs (new K / V, significance sums and
        # counts, lengths) copied from pinned host buffers, then the step, then
        # the unit headers and cursors read back
        upd, d = inputs(step_no)
        host = {"k_new": upd["k_new"].cpu().pin_memory(), "v_new": upd["v_new"].cpu().pin_memory(),
                "sig_sum": ctx["sig_sum"].cpu().pin_memory(), "sig_cnt": ctx["sig_cnt"].cpu().pin_memory(),
                "ctx_lens": ctx["ctx_lens"].cpu().pin_memory(), "new_lens": upd["new_lens"].cpu().pin_memory()}
        out_hdr = torch.empty(dec.tables.unit_hdr.shape, dtype=torch.int32).pin_memory()
        out_cur = torch.empty(2, dtype=torch.int64).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in host.values())
        d2h = out_hdr.numel() * 4 + 16
        te = 0.0
        e_rows = 0
        for i in range(a.e2e_steps):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            s0.record(stream)
            for k_, x in host.items():
                d[k_].copy_(x, non_blocking=True)
            dec.step(d, w.alpha_h, w.alpha_l)
            out_hdr.copy_(dec.tables.unit_hdr, non_blocking=True)
            out_cur.copy_(dec.pool.cursors, non_blocking=True)
            s1.record(stream)
            torch.cuda.synchronize()
            te += s0.elapsed_time(s1)
            e_rows += int((ctx["ctx_lens"] + upd["new_lens"]).sum()) * w.L * w.Hkv
            ctx["ctx_lens"] += upd["new_lens"]
            step_no += 1
            if i + 1 < a.e2e_steps:
                upd, d = inputs(step_no)
                for k_ in host:
                    host[k_].copy_(d[k_])
        assert libdkv.dkv_get_status(dec.pool) == libdkv.DKV_OK
        te = max_over_ranks(te, dev, world)
        e2e = {"value": whole_job_rate(e_rows, world, te), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": a.e2e_steps}
        del host
    head1 = int(dec.pool.cursors[0])

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        v, nsteps, rrows, tt = decode_oracle_sample(w, a.cpu_seconds, a.window, a.decode_mode)
        cpu = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"layer 0 of the first 16 requests of {a.workload} ({rrows:.0f} live token-rows per "
                         f"step) x {nsteps} steps, single-threaded, {tt:.1f} s"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms_max / a.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_name(a), "layers": w.L, "requests": w.R, "context": "uniform 2048..8192",
                       "Hq": w.Hq, "Hkv": w.Hkv, "page_tokens": w.P, "alpha_h": w.alpha_h, "alpha_l": w.alpha_l,
                       "cap": cap, "updates": "0.5% pruned + 0.5% demoted per (layer, request, KV head, token)",
                       "timed": "dkv_decode_step only (significance updates between steps untimed)",
                       "l2": "significance sums (%.1f GB) larger than L2" % (w.L * w.R * cap * w.Hq * 4 / 1e9),
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": rc_name, "achieved": rc_gbs, "peak": peak, "unit": "GB/s",
                         "frac": rc_gbs / peak, "peak_kind": peak_kind,
                         "traffic": _reclass_traffic(workload_name(a), rc_bytes) if rc_name == "k_reclass" else None,
                         "algorithmic_bytes": rc_bytes, "ms": rc_ms},
            "step_hbm": {"achieved": step_gbs, "frac": step_gbs / peak, "bytes": rc_bytes},
            "kernels_ms": kernel_ms,
            "new_token_rows_per_s": whole_job_rate(new_rows, world, ms_max),
            "pool": {"F": F, "prefill_pages": used, "head_start": head0, "head_end": head1,
                     "wraps": head1 // F - head0 // F},
            "gpu_launches": a.steps * 4,  # counter reset is a memset: k_reclass, k_dscan, k_apply, k_demote
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference_decode(a):
    """CPU oracle arm of the decode workload: each step is one oracle
    generation step on layer 0 of the first 16 requests."""
    from differentiated_kv_cache_dkv_gb300 import workloads as W

    if int(os.environ.get("RANK", "0")) != 0:
        return
    w = workload(a)
    smp = DecodeOracleSample(w, window=a.window, mode=a.decode_mode)
    for _ in range(a.warmup):
        smp.step()
    total, rows = 0.0, 0
    for _ in range(a.steps):
        dt, live = smp.step()
        total += dt
        rows += live
    value = rows / total
    sample = "one generation step on layer 0 of the first 16 requests per step, single-threaded oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": a.gpus, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": 1000.0 * total / a.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_name(a), "layers": w.L, "requests": w.R, "Hq": w.Hq, "Hkv": w.Hkv,
                   "page_tokens": w.P},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)


# ------------------------------------------------------------- attention ---

ATTN_METRIC = "KV tokens attended/sec (token-rows: one held token x one (layer, KV head), its G query heads)"
ATTN_SCALE = 0.08838834764831845  # 1 / sqrt(128)


class AttentionOracleSample:
    """The oracle's decode attention on a bounded sample of the decode
    workload: layer 0 of its first n_req requests, prefilled by the oracle
    (untimed)."""

    def __init__(self, w, n_req: int = 4):
        import dataclasses

        import torch

        from differentiated_kv_cache_dkv_gb300 import workloads as W
        from oracle.host_decode import HostDecode

        self.w = dataclasses.replace(w, L=1, lens=list(w.lens[:n_req]))
        self.cap = decode_cap(self.w, 1)
        self.hd = HostDecode(self.w, self.cap)
        q = W.decode_queries(self.w, 1, W.SEED_BASE)
        upd = W.decode_update_inputs(self.w, {k: (v.clone() if torch.is_tensor(v) else v)
                                              for k, v in self.hd.ctx.items()}, 0)
        b16 = lambda t: t.contiguous().view(torch.int16).numpy().view("uint16")  # noqa: E731
        self.a = {"L": 1, "R": self.w.R, "Hq": self.w.Hq, "Hkv": self.w.Hkv, "cap": self.cap, "layer0": 0,
                  "n_layers": 1, "q": b16(q), "k_new": b16(upd["k_new"]), "v_new": b16(upd["v_new"]),
                  "new_lens": upd["new_lens"].numpy().astype("int32"),
                  "ctx_lens": self.hd.ctx["ctx_lens"].numpy(), "scale": ATTN_SCALE}
        self.rows = (int(self.hd.tab.unit_hdr[:, :2].sum()) + int(upd["new_lens"].sum()) * self.w.Hkv)

    def step(self):
        import oracle

        t = time.perf_counter()
        st, _, _ = oracle.decode_attention(self.a, self.hd.pool, self.hd.tab)
        dt = time.perf_counter() - t
        assert st == 0, st
        return dt, self.rows


def run_native_attention(a):
    import torch

    from differentiated_kv_cache_dkv_gb300 import libdkv
    from differentiated_kv_cache_dkv_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    libdkv.load()
    w = workload(a)
    dev = torch.device("cuda", local)
    dec, ctx, cap, used = decode_setup(w, dev, W.SEED_BASE + 1000 * rank, 2)
    stream = torch.cuda.current_stream()
    q = W.decode_queries(w, w.L, W.SEED_BASE + rank, device=dev)
    upd = W.decode_update_inputs(w, {k: (v.clone() if torch.is_tensor(v) else v) for k, v in ctx.items()}, 0,
                                 device=dev)
    k_new, v_new, new_lens = upd["k_new"], upd["v_new"], upd["new_lens"]
    out = torch.empty((w.L, w.R, w.Hq, 128), dtype=torch.float32, device=dev)
    sig = ctx["sig_sum"]
    hdr = dec.tables.unit_hdr.long()
    n_hi, n_lo = int(hdr[:, 0].sum()), int(hdr[:, 1].sum())
    n_new = int(new_lens.sum()) * w.L * w.Hkv
    rows = n_hi + n_lo + n_new
    G = w.Hq // w.Hkv
    # algorithmic bytes: every held slot's codes, metadata and position; the
    # new tokens' K and V; queries and outputs; the forward rows and headers
    # read; each attended position's G significance sums read and written
    pages_used = int(hdr[:, 2].sum() + hdr[:, 3].sum())
    kv = scheme_bits(w.scheme)  # K + V bits of the high class; the low class has half
    alg = (n_hi * (16 * kv + 12) + n_lo * (8 * kv + 12) + n_new * 512
           + w.L * w.R * w.Hq * (256 + 512) + pages_used * 4 + w.U * 16 + rows * G * 8)

    def call():
        dec.attend(q, ctx["ctx_lens"], out, ATTN_SCALE, k_new=k_new, v_new=v_new, new_lens=new_lens, sig_sum=sig)

    for _ in range(a.warmup):
        call()
    torch.cuda.synchronize()
    assert libdkv.dkv_get_status(dec.pool) == libdkv.DKV_OK
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(a.steps):
        evs[i][0].record(stream)
        call()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    st = libdkv.dkv_get_status(dec.pool)
    assert st == libdkv.DKV_OK, libdkv.status_string(st)
    per = [e0.elapsed_time(e1) for e0, e1 in evs]
    ms = sum(per)
    ms_max = max_over_ranks(ms, dev, world)
    value = whole_job_rate(rows * a.steps, world, ms_max)
    peak, peak_kind = _peaks()
    att_ms = statistics.mean(per)
    gbs = alg / (att_ms / 1000.0) / 1e9

    e2e = None
    if a.e2e_steps > 0:
        # end to end: queries, new K / V and lengths from pinned host memory,
        # the call, the outputs read back (significance stays on the device)
        host = {"q": q.cpu().pin_memory(), "k_new": k_new.cpu().pin_memory(), "v_new": v_new.cpu().pin_memory(),
                "ctx": ctx["ctx_lens"].cpu().pin_memory(), "new": new_lens.cpu().pin_memory()}
        dst = {"q": q, "k_new": k_new, "v_new": v_new, "ctx": ctx["ctx_lens"], "new": new_lens}
        out_h = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in host.values())
        d2h = out_h.numel() * 4
        te = 0.0
        for _ in range(a.e2e_steps):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            s0.record(stream)
            for k_, x in host.items():
                dst[k_].copy_(x, non_blocking=True)
            call()
            out_h.copy_(out, non_blocking=True)
            s1.record(stream)
            torch.cuda.synchronize()
            te += s0.elapsed_time(s1)
        te = max_over_ranks(te, dev, world)
        e2e = {"value": whole_job_rate(rows * a.e2e_steps, world, te), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": a.e2e_steps}

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        smp = AttentionOracleSample(w)
        tt, rr, n = 0.0, 0, 0
        while tt < a.cpu_seconds or n == 0:
            dt, r_ = smp.step()
            tt += dt
            rr += r_
            n += 1
        cpu = {"value": rr / tt, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"layer 0 of the first 4 requests of {a.workload} ({smp.rows} token-rows per call) x {n} "
                         f"calls, single-threaded, {tt:.1f} s"}
    if rank == 0:
        line = {
            "metric": ATTN_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms_max / a.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_name(a), "layers": w.L, "requests": w.R, "context": "uniform 2048..8192",
                       "Hq": w.Hq, "Hkv": w.Hkv, "page_tokens": w.P, "cap": cap,
                       "held": {"k8v4": n_hi, "k4v2": n_lo, "new": n_new},
                       "timed": "one dkv_decode_attention over every layer (significance update included)",
                       "l2": "pages (%.1f GB) larger than L2" % (pages_used * 216 * w.P / 1e9),
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": "k_attend", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "peak_kind": peak_kind, "traffic": None, "algorithmic_bytes": alg,
                         "ms": att_ms},
            "gpu_launches": a.steps,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference_attention(a):
    """CPU oracle arm of decode attention: each step is one oracle attention
    call on layer 0 of the first 4 requests."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    w = workload(a)
    smp = AttentionOracleSample(w)
    for _ in range(a.warmup):
        smp.step()
    total, rows = 0.0, 0
    for _ in range(a.steps):
        dt, r_ = smp.step()
        total += dt
        rows += r_
    value = rows / total
    sample = "one oracle attention call on layer 0 of the first 4 requests per step, single-threaded"
    print(json.dumps({
        "impl": "reference", "metric": ATTN_METRIC, "value": value, "unit": UNIT, "n_gpus": a.gpus,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1000.0 * total / a.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(a), "layers": w.L, "requests": w.R, "Hq": w.Hq, "Hkv": w.Hkv,
                   "page_tokens": w.P},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)


# ----------------------------------------------------- prefill attention ---

PREFILL_METRIC = "KV tokens attended in prefill/sec (token-rows: one token x one (layer, KV head)), significance produced"


def _prefill_pairs(lens) -> int:
    return sum(n * (n + 1) // 2 for n in lens)


class PrefillOracleSample:
    """The oracle's prefill attention on a bounded sample: layer 0 of the first
    request, its first two query heads (one KV head)."""

    def __init__(self, w):
        import dataclasses

        import torch

        from differentiated_kv_cache_dkv_gb300 import workloads as W

        G = w.Hq // w.Hkv
        nq = min(2, G)
        self.w = dataclasses.replace(w, L=1, lens=[w.lens[0]], Hq=nq, Hkv=1)
        b16 = lambda t: t.contiguous().view(torch.int16).numpy().view("uint16")  # noqa: E731
        kv = dataclasses.replace(w, L=1, lens=[w.lens[0]])
        self.k = b16(W.make_kv_layer(kv, W.SEED_BASE, 0, 0)[:, :1][None])
        self.v = b16(W.make_kv_layer(kv, W.SEED_BASE, 0, 1)[:, :1][None])
        self.q = b16(W.prefill_queries(self.w, W.SEED_BASE, 0)[None])
        self.rows = w.lens[0]  # token-rows of one (layer, KV head), attended by nq of its G heads

    def step(self):
        import oracle

        t = time.perf_counter()
        st, _, _, _ = oracle.prefill_attention(self.q, self.k, self.v, self.w.lens, ATTN_SCALE)
        dt = time.perf_counter() - t
        assert st == 0, st
        return dt, self.rows


def run_native_prefill_attention(a):
    import torch

    from differentiated_kv_cache_dkv_gb300 import libdkv
    from differentiated_kv_cache_dkv_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    libdkv.load()
    w = workload(a)
    dev = torch.device("cuda", local)
    seed = W.SEED_BASE + 1000 * rank
    k = torch.empty((w.L, w.T, w.Hkv, 128), dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    q = torch.empty((w.L, w.T, w.Hq, 128), dtype=torch.bfloat16, device=dev)
    for l in range(w.L):
        k[l] = W.make_kv_layer(w, seed, l, 0, dev)
        v[l] = W.make_kv_layer(w, seed, l, 1, dev)
        q[l] = W.prefill_queries(w, seed, l, dev)
    lens = torch.tensor(w.lens, dtype=torch.int32, device=dev)
    out = torch.empty((w.L, w.T, w.Hq, 128), dtype=torch.float32, device=dev)
    sig = torch.empty((w.L, w.T, w.Hq), dtype=torch.float32, device=dev)
    cnt = torch.empty((w.T,), dtype=torch.int32, device=dev)
    pool = libdkv.DevicePool(1, 16, dev)
    libdkv.dkv_init_pool(pool)
    stream = torch.cuda.current_stream()

    def call():
        libdkv.dkv_prefill_attention(q, k, v, lens, max(w.lens), ATTN_SCALE, out, sig, cnt, pool)

    for _ in range(a.warmup):
        call()
    torch.cuda.synchronize()
    assert libdkv.dkv_get_status(pool) == libdkv.DKV_OK
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(a.steps):
        evs[i][0].record(stream)
        call()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    assert libdkv.dkv_get_status(pool) == libdkv.DKV_OK
    per = [e0.elapsed_time(e1) for e0, e1 in evs]
    ms_max = max_over_ranks(sum(per), dev, world)
    rows = w.T * w.L * w.Hkv
    value = whole_job_rate(rows * a.steps, world, ms_max)
    # algorithmic flops: q . k and p v over the causal pairs, every query head
    flops = 4.0 * 128 * _prefill_pairs(w.lens) * w.Hq * w.L
    tf = flops / (statistics.mean(per) / 1000.0) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        peak, peak_kind = float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), "measured (sustained bf16)"
    except Exception:
        peak, peak_kind = 1700.0, "fallback (sustained bf16)"

    e2e = None
    if a.e2e_steps > 0:
        host = {"q": q.cpu().pin_memory(), "k": k.cpu().pin_memory(), "v": v.cpu().pin_memory()}
        dst = {"q": q, "k": k, "v": v}
        sig_h = torch.empty(sig.shape, dtype=torch.float32).pin_memory()
        cnt_h = torch.empty(cnt.shape, dtype=torch.int32).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in host.values())
        d2h = sig_h.numel() * 4 + cnt_h.numel() * 4
        te = 0.0
        for _ in range(a.e2e_steps):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            s0.record(stream)
            for k_, x in host.items():
                dst[k_].copy_(x, non_blocking=True)
            call()
            sig_h.copy_(sig, non_blocking=True)
            cnt_h.copy_(cnt, non_blocking=True)
            s1.record(stream)
            torch.cuda.synchronize()
            te += s0.elapsed_time(s1)
        te = max_over_ranks(te, dev, world)
        e2e = {"value": whole_job_rate(rows * a.e2e_steps, world, te), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": a.e2e_steps,
               "note": "outputs stay on the device; the significance sums and counts are read back"}
        del host

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        smp = PrefillOracleSample(w)
        tt, rr, nn = 0.0, 0, 0
        while tt < a.cpu_seconds or nn == 0:
            dt, r_ = smp.step()
            tt += dt
            rr += r_
            nn += 1
        G = w.Hq // w.Hkv
        # the sample attends nq of a KV head's G query heads: scale its time to all G
        cpu = {"value": rr / (tt * G / smp.w.Hq), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"layer 0, request 0 ({smp.rows} tokens), {smp.w.Hq} of the {G} query heads of KV "
                         f"head 0, x {nn} calls, {tt:.1f} s single-threaded; time scaled to all {G} heads"}
    if rank == 0:
        print(json.dumps({
            "metric": PREFILL_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms_max / a.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_name(a), "layers": w.L, "requests": w.R, "tokens": w.T, "Hq": w.Hq,
                       "Hkv": w.Hkv, "timed": "one dkv_prefill_attention over every layer (outputs, significance "
                                              "sums and counts)",
                       "l2": "inputs (%.1f GB) larger than L2" % ((q.numel() + 2 * k.numel()) * 2 / 1e9),
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "kernel": "k_prefill", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": tf / peak, "peak_kind": peak_kind, "traffic": None, "algorithmic_flops": flops,
                         "ms": statistics.mean(per)},
            "gpu_launches": a.steps * 2,  # k_sigcnt, k_prefill (the zeroing is a memset)
            "clocks": clk, "e2e": e2e, "cpu_baseline": cpu}), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference_prefill_attention(a):
    """CPU oracle arm of prefill attention: each step is one oracle call on the
    bounded sample (layer 0, request 0, two query heads)."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    w = workload(a)
    smp = PrefillOracleSample(w)
    for _ in range(a.warmup):
        smp.step()
    total, rows = 0.0, 0
    for _ in range(a.steps):
        dt, r_ = smp.step()
        total += dt
        rows += r_
    G = w.Hq // w.Hkv
    value = rows / (total * G / smp.w.Hq)
    sample = "oracle prefill attention of layer 0, request 0, two query heads per step; time scaled to all G heads"
    print(json.dumps({
        "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": UNIT, "n_gpus": a.gpus,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1000.0 * total / a.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(a), "layers": w.L, "requests": w.R, "Hq": w.Hq, "Hkv": w.Hkv},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)


def main():
    a = _args()
    decode = a.workload == "decode"
    if a.op == "prefill-attention" and not decode:
        run_reference_prefill_attention(a) if a.impl == "reference" else run_native_prefill_attention(a)
    elif decode and a.op == "attention":
        run_reference_attention(a) if a.impl == "reference" else run_native_attention(a)
    elif a.impl == "reference":
        run_reference_decode(a) if decode else run_reference(a)
    else:
        run_native_decode(a) if decode else run_native(a)


if __name__ == "__main__":
    main()
