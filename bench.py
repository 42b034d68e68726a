#!/usr/bin/env python3
"""Ring attention fwd+bwd throughput on GB300 (one JSON line on rank 0).

A step is one pass of the whole hot path over one batch of synthetic input: the fused ring
forward (all D steps, online-softmax merge, finalise) and the ring backward (preprocess,
K/V-tile kernel, postprocess), on shard-major inputs resident in HBM. ``value`` is
algorithmic fwd+bwd TFLOP/s (causal pairs only, backward = 2.5x forward) on the
long-context workload: 131072 tokens, 32 query / 8 K/V heads, head_dim 128, D = 16,
zigzag, causal, bf16.

``--impl reference`` times the float64 CPU oracle on the host cores instead (a bounded
sample of query rows per step). With ``--gpus N`` under torchrun each rank runs its own
replica of the workload (the path has no cross-GPU exchange); rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "ring-attn fwd+bwd TFLOP/s (causal bf16, 1×GB300) and % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch from an ncu capture, with the hash of the kernel source (with the
# shared headers and the plan construction) they were taken on: a changed kernel reports
# null until re-measured.
TRAFFIC = {
    ("ring_bwd_tc (K/V-tile pass)", "long_s131072_gqa32x8_dh128_D16_zigzag"):
        {"bytes": 55050429696 + 541969408, "source_sha": "f32b290a402a8697"},
    ("ring_fwd_tc", "long_s131072_gqa32x8_dh128_D16_zigzag"):
        {"bytes": 118658146816 + 1258202880, "source_sha": "2b895ee9cb12a15d"},
    ("ring_bwd_dq_tc (dq pass)", "long_s131072_gqa32x8_dh128_D16_zigzag"):
        {"bytes": 16206185984 + 1060122624, "source_sha": "8733957a884564f0"},
    ("merge_kernel", "long_s131072_gqa32x8_dh128_D16_zigzag"):
        {"bytes": 3255621888 + 2109105664, "source_sha": "59a72745c75670f4"},
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=W.LONG128K.name, choices=sorted(W.NAMED))
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of one oracle sample")
    ap.add_argument("--secondary", type=int, default=1,
                    help="also time the unfused per-step path and the deterministic backward")
    ap.add_argument("--once", action="store_true",
                    help="run the forward, the backward and the merge once each on the "
                         "workload and exit (a short command to put under a profiler)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def fwd_bwd_flops(w: W.Workload) -> tuple[float, float]:
    f = w.fwd_flops()
    return f, 2.5 * f


# ------------------------------------------------------------------------ CPU oracle sample

def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return os.uname().machine


def oracle_sample(w: W.Workload, target_s: float, inputs=None):
    """Time the float64 oracle (forward + backward) on a stratified sample of query rows of
    the longest sequence: R strata of equal length, one seeded random row in each, every
    query head, each row against its whole causal key range. R doubles until one sample
    takes about ``target_s`` / 4 or more.

    Returns (TFLOP/s, seconds, description, extrapolated seconds of the full workload)."""
    from oracle import attention as A

    if inputs is None:
        q, k, v = W.make_qkv(w)
        do = W.make_dout(w)
    else:
        q, k, v, do = inputs
    pk = lambda x: x.reshape(-1, x.shape[-2], x.shape[-1])
    q, k, v, do = pk(q), pk(k), pk(v), pk(do)
    i = int(np.argmax(w.lengths))
    cu = w.cu_seqlens
    s0, s1 = int(cu[i]), int(cu[i + 1])
    n_tok = s1 - s0
    qs, ks, vs, dos = q[s0:s1], k[s0:s1], v[s0:s1], do[s0:s1]
    cu1 = np.array([0, n_tok])
    rng = np.random.default_rng(2024)

    def run(nrows):
        edges = np.linspace(0, n_tok, nrows + 1).astype(np.int64)
        rows = np.unique(np.array([rng.integers(a, max(a + 1, b)) for a, b in zip(edges[:-1], edges[1:])]))
        t0 = time.perf_counter()
        A.attention_fwd(qs, ks, vs, cu1, w.causal, rows=rows)
        A.attention_bwd(qs, ks, vs, dos, cu1, w.causal, rows=rows)
        dt = time.perf_counter() - t0
        pairs = float(sum((r + 1) if w.causal else n_tok for r in rows)) * w.hq
        return dt, 3.5 * 4.0 * w.head_dim * pairs, rows.size

    n = 8
    dt, fl, got = run(n)
    while dt < target_s / 4 and n < n_tok:
        n = min(n_tok, max(n * 2, int(n * target_s / max(dt, 1e-3) * 0.8)))
        dt, fl, got = run(n)
    rate = fl / dt
    full_s = sum(fwd_bwd_flops(w)) / rate
    desc = (f"oracle fwd+bwd (float64 NumPy) on {got} query rows of the longest sequence "
            f"({n_tok} tokens), one seeded row per equal stratum, all {w.hq} query heads, "
            f"each row against its whole causal key range; CPU {cpu_model()}")
    return rate / 1e12, dt, desc, full_s


def cores_used() -> int:
    return os.cpu_count() or 1


# ------------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------ our arm

def kernel_source_hash(name: str) -> str:
    """sha256 prefix of a kernel's source file together with the headers every kernel
    shares (launch plan, layouts, PTX wrappers) and the plan construction (item order)."""
    csrc = os.path.join(ROOT, "context_blockwise_attention_step_gb300", "csrc")
    h = hashlib.sha256()
    for part in (name, "ra_plan.h", "ra_layout.h", "ra_ptx.cuh", "ra_api.cu"):
        with open(os.path.join(csrc, part), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def run_ours(args, rank, world, local_rank):
    import torch

    import context_blockwise_attention_step_gb300 as ra

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    ra.build()
    w = W.NAMED[args.workload]
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    q, k, v = W.make_qkv(w)
    do = W.make_dout(w)
    np_inputs = (q, k, v, do)
    host = [torch.from_numpy(x).to(tdt).pin_memory() for x in np_inputs]
    nat = [h.to(dev, non_blocking=True) for h in host]
    prob = ra.problem_for(nat[0], nat[1], D=w.D, layout=w.layout, causal=w.causal,
                          cu_seqlens=w.cu_seqlens if w.varlen else None)
    qs, ks, vs, dos = (ra.shard_tokens(x, prob) for x in nat)
    out = torch.empty_like(qs)
    lse = torch.empty(ra.ops._lse_shape(prob), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(qs), torch.empty_like(ks), torch.empty_like(vs)
    ws = torch.empty(max(ra.workspace_bytes(prob), 1), device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)
    if args.once:
        ra.ring_attn_fwd(qs, ks, vs, prob, out=out, lse=lse)
        ra.ring_attn_bwd(dos, qs, ks, vs, out, lse, prob, dq=dq, dk=dk, dv=dv, workspace=ws)
        mo = torch.zeros(qs.shape, device=dev, dtype=torch.float32)
        ml = torch.full(lse.shape, float("-inf"), device=dev, dtype=torch.float32)
        ra.update_out_and_lse(mo, ml, out, lse, prob)
        torch.cuda.synchronize(dev)
        status = ra.check_device_status()
        if status != 0:
            raise RuntimeError(f"device status: {ra.last_error()}")
        print(json.dumps({"once": w.name, "status": status}), flush=True)
        return None
    in_bytes = sum(x.numel() * x.element_size() for x in (qs, ks, vs, dos))
    flush = None if in_bytes > 2 * L2_BYTES else torch.empty(2 * L2_BYTES // 4, device=dev)

    for _ in range(args.warmup):
        ra.ring_attn_fwd(qs, ks, vs, prob, out=out, lse=lse)
        ra.ring_attn_bwd(dos, qs, ks, vs, out, lse, prob, dq=dq, dk=dk, dv=dv, workspace=ws)
    torch.cuda.synchronize(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    st = [ev() for _ in range(args.steps)]
    sp = [ev() for _ in range(args.steps)]
    kf = [(ev(), ev()) for _ in range(args.steps)]
    kb = [(ev(), ev()) for _ in range(args.steps)]
    km = [ev() for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            st[i].record(stream)
            ra.profile_events(*kf[i])
            ra.ring_attn_fwd(qs, ks, vs, prob, out=out, lse=lse)
            ra.profile_events(*kb[i])
            ra.profile_split_event(km[i])
            ra.ring_attn_bwd(dos, qs, ks, vs, out, lse, prob, dq=dq, dk=dk, dv=dv, workspace=ws)
            ra.profile_events(None, None)
            ra.profile_split_event(None)
            sp[i].record(stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(st, sp)]
    fwd_ms = [a.elapsed_time(b) for a, b in kf]
    bwd_ms = [a.elapsed_time(b) for a, b in kb]
    kv_ms = [a.elapsed_time(m) for (a, _), m in zip(kb, km)]
    if ra.check_device_status() != 0:
        raise RuntimeError(f"device status after the timed region: {ra.last_error()}")

    # ---- end to end: host buffers in, host buffers out, through the public API
    outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (out, lse, dq, dk, dv)]
    dev_nat = [torch.empty_like(x) for x in nat]
    dev_out_nat = [torch.empty_like(t) for t in (out, lse, dq, dk, dv)]

    copy_stream = torch.cuda.Stream(dev)

    def e2e_step():
        # Copies run on their own stream, overlapped with the kernels: q, k, v first (the
        # forward needs them), dO during the forward, out and lse back during the backward,
        # dq, dk, dv back at the end. The step ends when the last copy has landed.
        copy_stream.wait_stream(stream)
        with torch.cuda.stream(copy_stream):
            for h, d in zip(host[:3], dev_nat[:3]):
                d.copy_(h, non_blocking=True)
            qkv_in = torch.cuda.Event()
            qkv_in.record(copy_stream)
            dev_nat[3].copy_(host[3], non_blocking=True)
            do_in = torch.cuda.Event()
            do_in.record(copy_stream)
        stream.wait_event(qkv_in)
        sm = [ra.shard_tokens(x, prob) for x in dev_nat[:3]]
        o, l = ra.ring_attn_fwd(sm[0], sm[1], sm[2], prob)
        ra.unshard_tokens(o, prob, out=dev_out_nat[0])
        ra.unshard_lse(l, prob, out=dev_out_nat[1])
        fwd_done = torch.cuda.Event()
        fwd_done.record(stream)
        stream.wait_event(do_in)
        sdo = ra.shard_tokens(dev_nat[3], prob)
        g = ra.ring_attn_bwd(sdo, sm[0], sm[1], sm[2], o, l, prob, workspace=ws)
        copy_stream.wait_event(fwd_done)
        with torch.cuda.stream(copy_stream):
            for d, h in zip(dev_out_nat[:2], outs_h[:2]):
                h.copy_(d, non_blocking=True)
        for t, d in zip(g, dev_out_nat[2:]):
            ra.unshard_tokens(t, prob, out=d)
        copy_stream.wait_stream(stream)
        with torch.cuda.stream(copy_stream):
            for d, h in zip(dev_out_nat[2:], outs_h[2:]):
                h.copy_(d, non_blocking=True)
        stream.wait_stream(copy_stream)

    e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = ev(), ev()
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    h2d = sum(h.numel() * h.element_size() for h in host)
    d2h = sum(h.numel() * h.element_size() for h in outs_h)

    merge = measure_merge(ra, prob, qs, lse, w, stream)
    secondary = measure_secondary(ra, w, nat, prob, (qs, ks, vs, dos), ev, stream) if args.secondary else None

    per = torch.tensor([sum(step_ms) / args.steps, e2e_ms, statistics.mean(fwd_ms),
                        statistics.mean(bwd_ms), statistics.mean(kv_ms)], device=dev,
                       dtype=torch.float64)
    if dist is not None:
        dist.all_reduce(per, op=dist.ReduceOp.MAX)
    ms_step, e2e_ms, fwd_mean, bwd_mean, kv_mean = per.tolist()
    dq_mean = bwd_mean - kv_mean

    ff, fb = fwd_bwd_flops(w)
    value = world * (ff + fb) / (ms_step * 1e-3) / 1e12
    e2e_value = world * (ff + fb) / (e2e_ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak_sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    peak_burst = peaks["bf16_tflops"]
    merge["frac_of_hbm"] = merge["gbs"] / peaks["hbm_gbs"]
    merge["hbm_peak_gbs"] = peaks["hbm_gbs"]
    mtr = TRAFFIC.get(("merge_kernel", w.name))
    merge["traffic"] = (mtr["bytes"] if mtr and mtr["source_sha"] == kernel_source_hash("ra_misc.cu")
                        else None)
    # Algorithmic FLOP per kernel: the forward's 2 GEMMs; of the backward's 5 (S recompute,
    # dP, dV, dK, dQ) the K/V-tile pass does 4 and the dq pass adds dQ (its S and dP
    # recomputation is executed work the method does not count).
    kern = {
        "ring_fwd_tc": {"ms": fwd_mean, "algorithmic_tflop_per_launch": ff / 1e12,
                        "executed_tflop_per_launch": ff / 1e12},
        "ring_bwd_tc (K/V-tile pass)": {"ms": kv_mean, "algorithmic_tflop_per_launch": 2.0 * ff / 1e12,
                                        "executed_tflop_per_launch": 2.0 * ff / 1e12},
        "ring_bwd_dq_tc (dq pass)": {"ms": dq_mean, "algorithmic_tflop_per_launch": 0.5 * ff / 1e12,
                                     "executed_tflop_per_launch": 1.5 * ff / 1e12},
    }
    for kv in kern.values():
        kv["tflops"] = kv["algorithmic_tflop_per_launch"] / (kv["ms"] * 1e-3)
        kv["executed_tflops"] = kv["executed_tflop_per_launch"] / (kv["ms"] * 1e-3)
        kv["frac_of_sustained_peak"] = kv["tflops"] / peak_sus
        kv["frac_of_burst_peak"] = kv["tflops"] / peak_burst
        kv["executed_frac_of_sustained_peak"] = kv["executed_tflops"] / peak_sus
        kv["share_of_step"] = kv["ms"] / ms_step
    backward = {"ms": bwd_mean, "tflops": fb / (bwd_mean * 1e-3) / 1e12,
                "algorithmic_tflop": fb / 1e12}
    backward["frac_of_sustained_peak"] = backward["tflops"] / peak_sus
    dom = max(kern, key=lambda n: kern[n]["ms"])
    src = {"ring_fwd_tc": "ra_fwd_tc.cu", "ring_bwd_tc (K/V-tile pass)": "ra_bwd_tc.cu",
           "ring_bwd_dq_tc (dq pass)": "ra_bwd_dq_tc.cu"}[dom]
    tr = TRAFFIC.get((dom, w.name))
    traffic = tr["bytes"] if tr and tr["source_sha"] == kernel_source_hash(src) else None
    result = None
    if rank == 0:
        cpu = None
        if world == 1:
            v_cpu, t_cpu, desc, full_s = oracle_sample(w, args.cpu_seconds, np_inputs)
            cpu = {"value": v_cpu, "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                   "sample": desc, "seconds": t_cpu,
                   "extrapolated_full_workload_s": full_s}
        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded N(0,1), rounded to bf16)",
            "config": {"workload": w.name, "batch": w.batch or None, "seq_len": w.seqlen or None,
                       "total_tokens": w.total_tokens, "hq": w.hq, "hkv": w.hkv,
                       "head_dim": w.head_dim, "D": w.D, "layout": w.layout, "causal": w.causal,
                       "varlen": w.varlen, "parallelism": f"replicas{world}",
                       "l2": ("inputs larger than L2" if flush is None
                              else "L2 flushed between steps (outside the timed windows)"),
                       "fwd_tflop": ff / 1e12, "bwd_tflop": fb / 1e12},
            "pct_of_peak": 100.0 * value / world / peak_sus,
            "pct_of_peak_burst": 100.0 * value / world / peak_burst,
            "peak_tflops": {"sustained": peak_sus, "burst": peak_burst, "source": peak_src},
            "tokens_per_s": world * w.total_tokens / (ms_step * 1e-3),
            "roofline": {"bound": "tensor", "kernel": dom, "achieved": kern[dom]["tflops"],
                         "peak": peak_sus, "peak_source": f"{peak_src} bf16_tflops_sustained",
                         "unit": "TFLOP/s", "frac": kern[dom]["tflops"] / peak_sus,
                         "frac_burst": kern[dom]["tflops"] / peak_burst,
                         "traffic": traffic,
                         "algorithmic_unit": "2 x head_dim FLOP per causal (query, key) pair for "
                                             "each of the path's seven GEMMs (fwd QK^T, PV; bwd S, "
                                             "dP, dV, dK, dQ) the kernel performs, over S^2/2 pairs "
                                             "per sequence and query head"},
            "kernels": kern,
            "backward_both_passes": backward,
            "merge_kernel": merge,
            "secondary": secondary,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": 4 * args.steps,  # forward; backward preprocess, K/V pass, dq pass
            "clocks": clocks.summary(),
            "step_ms": step_ms,
        }
    if dist is not None:
        dist.destroy_process_group()
    return result


def measure_merge(ra, prob, qs, lse, w, stream, reps=5):
    """HBM GB/s of the standalone update_out_and_lse kernel on the workload's rows: float32
    out / lse updated in place with a bf16 block. Algorithmic bytes per (token, head) row:
    read + write out (2 x 4 x Dh), read the bf16 block (2 x Dh), read + write lse and read
    the block lse (12): 1292 B at Dh = 128."""
    import torch

    out = torch.zeros(qs.shape, device=qs.device, dtype=torch.float32)
    mlse = torch.full(lse.shape, float("-inf"), device=qs.device, dtype=torch.float32)
    block = torch.randn(qs.shape, device=qs.device, dtype=torch.float32).to(torch.bfloat16)
    blse = torch.randn(lse.shape, device=qs.device, dtype=torch.float32)
    for _ in range(2):
        ra.update_out_and_lse(out, mlse, block, blse, prob)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
    for i in range(reps):
        ev[2 * i].record(stream)
        ra.update_out_and_lse(out, mlse, block, blse, prob)
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(reps))
    rows = w.total_tokens * w.hq
    per_row = 2 * 4 * w.head_dim + 2 * w.head_dim + 12
    del out, mlse, block, blse
    return {"ms": ms, "bytes_per_launch": rows * per_row, "bytes_per_row": per_row,
            "gbs": rows * per_row / (ms * 1e-3) / 1e9, "launches_timed": reps}


def measure_secondary(ra, w, nat, prob, sm, ev, stream, reps=2):
    """TFLOP/s of (a) the unfused path: D block forwards merged one step at a time, then D
    per-step block backwards added into float32 accumulators; (b) the deterministic
    backward (K/V-tile pass without dq + query-tile dq pass). Same algorithmic FLOP as the
    fused step."""
    import torch

    qs, ks, vs, dos = sm
    ff, fb = fwd_bwd_flops(w)
    out, lse = ra.ring_attn_fwd(qs, ks, vs, prob)
    lse_shape = lse.shape
    res = {}

    def unfused():
        o = torch.zeros(qs.shape, device=qs.device, dtype=torch.float32)
        l = torch.full(lse_shape, float("-inf"), device=qs.device, dtype=torch.float32)
        bo = torch.empty(qs.shape, device=qs.device, dtype=torch.bfloat16)
        bl = torch.empty(lse_shape, device=qs.device, dtype=torch.float32)
        for s in range(w.D):
            ra.block_attn_fwd(qs, ks, vs, prob, rank=-1, step=s, out_dtype=torch.bfloat16,
                              block_out=bo, block_lse=bl)
            ra.update_out_and_lse(o, l, bo, bl, prob)
        acc = [torch.zeros(t.shape, device=qs.device, dtype=torch.float32) for t in (qs, ks, vs)]
        for s in range(w.D):
            ra.block_attn_bwd(dos, qs, ks, vs, out, lse, prob, -1, s, *acc)

    det = ra.problem_for(nat[0], nat[1], D=w.D, layout=w.layout, causal=w.causal,
                         cu_seqlens=w.cu_seqlens if w.varlen else None, deterministic=True)
    ws = torch.empty(max(ra.workspace_bytes(det), 1), device=qs.device, dtype=torch.uint8)

    def deterministic():
        ra.ring_attn_bwd(dos, qs, ks, vs, out, lse, det, workspace=ws)

    for name, fn, flop in (("unfused_fwd_bwd", unfused, ff + fb), ("deterministic_bwd", deterministic, fb)):
        fn()
        torch.cuda.synchronize()
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        res[name] = {"ms": ms, "tflops": flop / (ms * 1e-3) / 1e12}
    if ra.check_device_status() != 0:
        raise RuntimeError(f"device status after the secondary measurements: {ra.last_error()}")
    return res


# ------------------------------------------------------------------------ reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = W.NAMED[args.workload]
    q, k, v = W.make_qkv(w)
    do = W.make_dout(w)
    inputs = (q, k, v, do)
    per_step = max(5.0, min(args.cpu_seconds, 180.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, per_step, inputs)
    vals, secs, desc = [], [], ""
    for _ in range(args.steps):
        v_, t_, desc, _ = oracle_sample(w, per_step, inputs)
        vals.append(v_)
        secs.append(t_)
    value = statistics.mean(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), rounded to bf16)",
        "config": {"workload": w.name, "seq_len": w.seqlen or None, "total_tokens": w.total_tokens,
                   "hq": w.hq, "hkv": w.hkv, "head_dim": w.head_dim, "D": w.D,
                   "layout": w.layout, "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
