"""Benchmark: full-vocabulary Jacobi refinement on the batched-decode workload.

One step = one ``xp_jacobi_refine`` call over a batch of N=32 draft blocks of
B=16 slots, V=151936, bf16: the hidden cache, the init argmax and K=15 passes
of latent + tensor-core readout/argmax.  ``value`` = Jacobi passes per second
over the whole job (all ranks), inputs resident in HBM.  ``e2e`` = the same
metric through the same C-ABI call with the step's inputs copied in from
pinned host memory and blk copied back, every step.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Multi-GPU (torchrun, one rank per GPU): every rank refines its own batch
(weak scaling, no collective on the data path); timing is the max over ranks.
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

WORKLOAD = "batched-decode"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "refine_persist_batched_decode.json")
PERSIST_SRC = os.path.join(ROOT, "jacobi_speculative_decode_gb300", "csrc", "k_persist.cu")
READOUT_TRAFFIC = os.path.join(ROOT, "profiles", "readout_tc_batched_decode.json")
PASS_MODES = {"auto": 0, "persistent": 1, "per-stage": 2}   # XP_PASSES_* of include/xp.h
READOUT_SRC = os.path.join(ROOT, "jacobi_speculative_decode_gb300", "csrc", "k_readout_tc.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--K", type=int, default=None,
                    help="passes per step (default: the workload's); for short profiler captures")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-breakdown", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the single-request, top-C and max-batch side measurements")
    ap.add_argument("--pass-mode", default="auto", choices=["auto", "persistent", "per-stage"],
                    help="how the step runs its passes (xp_set_pass_mode); default: the library's "
                         "automatic choice")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def workload_config(wl):
    """The workload's identity; the same dict in both arms."""
    return {"workload": wl.name, "N": wl.N, "B": wl.B, "V": wl.V, "r": wl.r,
            "hidden": wl.hidden, "H": wl.H, "K": wl.K, "topc": wl.topc}


def pass_bytes(wl):
    """Algorithmic HBM bytes of one full-vocabulary pass: w2 and the draft rows' base
    streamed once, plus the latent side (projected-embedding rows gathered per slot
    (fp32), xh, the latent written and read back, the SwiGLU and mixer weights, blk)."""
    es = 2 if wl.dtype == "bf16" else 4
    readout = wl.V * wl.r * es + wl.rows * wl.V * es
    latent = (wl.N * wl.B * wl.r * 4            # E[prev] rows
              + wl.N * wl.B * wl.r * 4          # xh
              + 2 * wl.rows * wl.r * es         # lat out and back in
              + 3 * wl.H * wl.r * es            # w_gate, w_up, w_down
              + wl.B * wl.B * wl.r * es         # folded mixer
              + 2 * wl.N * wl.B * 8)            # blk read and written
    return readout + latent


def roofline_step(wl, passes_per_s):
    """The headline rate against the HBM roofline: per-pass algorithmic bytes x passes/s.
    The once-per-step hidden cache and init are inside the measured rate but not counted
    in the bytes, so the fraction is a lower bound."""
    hbm, kind = peaks()
    b = pass_bytes(wl)
    achieved = b * passes_per_s / 1e9
    return {"bound": "hbm", "bytes_per_pass": b, "achieved": round(achieved, 1), "peak": hbm,
            "unit": "GB/s", "frac": round(achieved / hbm, 4),
            "peak_kind": f"{kind} (copy bandwidth)"}


def l2_note(wl):
    es = 2 if wl.dtype == "bf16" else 4
    base_mb, w2_mb = wl.rows * wl.V * es / 1e6, wl.V * wl.r * es / 1e6
    return (f"no flush between steps: every pass streams base {base_mb:.0f} MB + w2 {w2_mb:.0f} MB, "
            f"{base_mb + w2_mb:.0f} MB against a 129 MB L2")


def src_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def committed_traffic(profile, src, rows, key, times=1):
    """DRAM bytes (read + write) from a committed ncu summary: its per-unit figure `key` x
    times, if the kernel source is unchanged since the capture and the rows match."""
    try:
        with open(profile) as f:
            p = json.load(f)
        if p.get("source_sha256_16") != src_hash(src) or p.get("rows") != rows:
            return None
        return float(p[key]) * times
    except Exception:
        return None


class Clocks:
    """nvidia-smi sampled every 200 ms during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        out_dir = os.environ.get("XP_BENCH_OUT", os.path.join(ROOT, "bench_out"))
        self.path = os.path.join(out_dir, f"clocks_rank{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        try:
            rows = [ln.split(",") for ln in open(self.path).read().strip().splitlines() if ln.strip()]
        except Exception:
            return None
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() in ("active", "1"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------

def run_native(args, rank, world, local):
    import torch
    from jacobi_speculative_decode_gb300 import inputs as I
    from jacobi_speculative_decode_gb300 import xp

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from jacobi_speculative_decode_gb300 import shard
    wl = I.workload(args.workload)
    wl = I.workload(args.workload, seed=shard.rank_seed(wl.seed, rank))   # this rank's own batch
    if args.K is not None:
        wl = I.workload(args.workload, seed=wl.seed, K=args.K)
    d = I.make_inputs(wl)
    head, _ = xp.head_from_inputs(d, wl)
    xp.xp_set_pass_mode(head.handle, PASS_MODES[args.pass_mode])
    base = xp.to_device(d["base"], wl.dtype)
    h = xp.to_device(d["h_full"], wl.dtype)
    anchor = torch.from_numpy(d["anchor"]).cuda()
    am1 = torch.from_numpy(d["am1"]).cuda()
    blk = torch.empty(wl.N, wl.B, dtype=torch.int64, device=dev)
    ws = head.workspace(wl.N, wl.topc)
    sn, sb = (wl.B - 1) * wl.V, wl.V
    stream = torch.cuda.current_stream()

    def step():
        xp.xp_jacobi_refine(head.handle, base, sn, sb, h, anchor, am1, wl.N, wl.K, wl.topc, blk, ws)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    status = xp.xp_get_error(head.handle)
    if status != xp.XP_OK:
        raise RuntimeError(f"device error after warm-up: {xp.status_str(status)}")

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        barrier()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        barrier()
    ms = shard.max_over_ranks(e0.elapsed_time(e1), device=dev)
    status = xp.xp_get_error(head.handle)
    if status != xp.XP_OK:
        raise RuntimeError(f"device error in the timed region: {xp.status_str(status)}")

    passes = wl.K * args.steps * world
    value = passes / (ms / 1e3)
    # tensor-core hidden cache (GEMM + reduce) and the init beside it (3), or the hidden
    # cache and the top-C select (+ the w2 row copy when it is no larger than w2); then
    # 2 per pass (latent, readout)
    persistent = persistent_path(xp, head, wl, base, sn, sb)
    if wl.topc == 0:
        # hidden-cache GEMM, init argmax, reduce; then one persistent launch for all passes,
        # or 2 launches per pass (latent, readout)
        launches_per_step = 3 + (1 if persistent else 2 * wl.K)
    else:
        copies = 1 if wl.N * (wl.B - 1) * min(wl.topc, wl.V) <= wl.V else 0
        launches_per_step = 2 + 1 + copies + 2 * wl.K
    out = {
        "metric": "Jacobi passes/s at N=32,B=16,V=151936 bf16; % of HBM roofline",
        "value": round(value, 2), "unit": "passes/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generator; random-init head weights)",
        "config": workload_config(wl),
        "parallelism": f"blocks sharded, {world} independent replica(s)",
        "passes": "persistent launch" if persistent else "per stage (latent, readout)",
        "l2": l2_note(wl),
        "rows_per_s": round(value * wl.rows, 1),
        "roofline_step": roofline_step(wl, value),
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }

    # --- per-kernel breakdown: the same pass issued stage by stage, events per kernel
    if not args.no_breakdown:
        out.update(breakdown(wl, head, base, sn, sb, h, anchor, am1, ws, stream, rank,
                             PASS_MODES[args.pass_mode]))

    # --- end to end through the C ABI with host buffers
    if not args.no_e2e:
        out["e2e"] = e2e(wl, head, d, ws, args, stream, world)

    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl, d, budget_s=12.0)
    head.close()
    del d, base, h, ws
    if rank == 0 and world == 1 and not args.no_extras:
        out["other_workloads"] = other_workloads(args)
    return out


def other_workloads(args):
    """Side measurements on the other workloads (not the headline): passes/s of a full
    step, and for top-C the per-pass candidate readout against the HBM roofline."""
    import torch
    from jacobi_speculative_decode_gb300 import inputs as I
    from jacobi_speculative_decode_gb300 import xp
    res = {}
    hbm, kind = peaks()
    for name in ("single-request", "topc", "max-batch"):
        wl = I.workload(name)
        d = I.make_inputs(wl)
        head, _ = xp.head_from_inputs(d, wl)
        base = xp.to_device(d["base"], wl.dtype)
        h = xp.to_device(d["h_full"], wl.dtype)
        anchor = torch.from_numpy(d["anchor"]).cuda()
        am1 = torch.from_numpy(d["am1"]).cuda()
        blk = torch.empty(wl.N, wl.B, dtype=torch.int64, device="cuda")
        ws = head.workspace(wl.N, wl.topc)
        sn, sb = (wl.B - 1) * wl.V, wl.V
        stream = torch.cuda.current_stream()

        def step():
            xp.xp_jacobi_refine(head.handle, base, sn, sb, h, anchor, am1, wl.N, wl.K, wl.topc,
                                blk, ws)

        for _ in range(2):
            step()
        steps = 5
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        r = {"passes_per_s": round(wl.K / (ms / 1e3), 1), "ms_per_step": round(ms, 4),
             "rows_per_s": round(wl.K * wl.rows / (ms / 1e3), 1),
             "config": {"N": wl.N, "B": wl.B, "V": wl.V, "hidden": wl.hidden, "K": wl.K,
                        "topc": wl.topc}}
        if not wl.topc:
            r["roofline_step_frac"] = round(pass_bytes(wl) * wl.K / (ms / 1e3) / 1e9 / hbm, 4)
            # the latent's share of a pass, from the single-pass entry points chained as in a step
            xh = torch.empty(wl.N, wl.B, wl.r, dtype=torch.float32, device="cuda")
            lat = torch.empty(wl.N, wl.B - 1, wl.r, dtype=xp.torch_dtype(wl.dtype), device="cuda")
            xp.xp_hidden_cache(head.handle, h, wl.N, xh, ws)
            xp.xp_init_argmax(head.handle, base, sn, sb, anchor, wl.N, blk, None, ws)

            def chained_us(fn, n=30):
                for _ in range(3):
                    fn()
                c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c0.record(stream)
                for _ in range(n):
                    fn()
                c1.record(stream)
                torch.cuda.synchronize()
                return c0.elapsed_time(c1) / n * 1e3

            def readout():
                xp.xp_readout_argmax(head.handle, lat, base, sn, sb, wl.N, blk, None, ws)

            def one_pass():
                xp.xp_latent_pass(head.handle, blk, am1, xh, wl.N, lat)
                readout()

            ro_us, pass_us = chained_us(readout), chained_us(one_pass)
            r["readout_us"] = round(ro_us, 2)
            r["pass_us"] = round(pass_us, 2)
            r["latent_share_of_pass"] = round(max(pass_us - ro_us, 0.0) / pass_us, 4)
            del xh, lat
        if xp.xp_get_error(head.handle) != xp.XP_OK:
            r["device_error"] = True
        if wl.topc:
            C = wl.topc
            cand = torch.empty(wl.N, wl.B - 1, C, dtype=torch.int64, device="cuda")
            base_c = torch.empty(wl.N, wl.B - 1, C, dtype=torch.bfloat16, device="cuda")
            w2c = torch.empty(wl.N, wl.B - 1, C, wl.r, dtype=torch.bfloat16, device="cuda")
            lat = torch.empty(wl.N, wl.B - 1, wl.r, dtype=torch.bfloat16, device="cuda")
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            xp.xp_topc_gather(head.handle, base, sn, sb, wl.N, C, cand, base_c, w2c, blk)
            g1.record(stream)
            lat.copy_(torch.randn_like(lat, dtype=torch.float32).to(torch.bfloat16))
            for _ in range(3):
                xp.xp_topc_readout_argmax(head.handle, lat, base_c, cand, w2c, wl.N, C, blk, None)
            n = 20
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(n):
                xp.xp_topc_readout_argmax(head.handle, lat, base_c, cand, w2c, wl.N, C, blk, None)
            t1.record(stream)
            torch.cuda.synchronize()
            us = t0.elapsed_time(t1) / n * 1e3
            rows = wl.rows
            nbytes = rows * C * wl.r * 2 + rows * C * 2 + rows * C * 8 + rows * wl.r * 2 + rows * 8
            r["topc_readout"] = {"us": round(us, 2), "algorithmic_bytes": nbytes,
                                 "achieved_gbs": round(nbytes / us / 1e3, 1),
                                 "frac_of_hbm": round(nbytes / us / 1e3 / hbm, 4),
                                 "w2_rows": "copied once per step (w2c)"}
            # the same pass reading the candidates' rows by id from w2 (L2-resident)
            t0.record(stream)
            for _ in range(n):
                xp.xp_topc_readout_argmax(head.handle, lat, base_c, cand, None, wl.N, C, blk, None)
            t1.record(stream)
            torch.cuda.synchronize()
            r["topc_readout_by_id_us"] = round(t0.elapsed_time(t1) / n * 1e3, 2)
            r["topc_gather_us"] = round(g0.elapsed_time(g1) * 1e3, 1)
            del cand, base_c, w2c, lat
        res[name] = r
        head.close()
        del d, base, h, ws, blk
        torch.cuda.empty_cache()
    return res


def persistent_path(xp, head, wl, base, sn, sb):
    """Whether xp_jacobi_refine runs this workload's passes in the persistent kernel."""
    return wl.topc == 0 and xp.xp_passes_persistent(head.handle, base, sn, sb, wl.N)


def timeline_summary(xp, head, wl, step):
    """Phase structure of the persistent kernel from one step with per-CTA stamps: the pass
    period, each CTA's readout phase, and the part of a pass in which no CTA is in its
    readout (the latent stage and its hand-offs, exposed)."""
    import torch
    need = xp.xp_profile_timeline(head.handle, None, wl.K)
    buf = torch.zeros(need // 8, dtype=torch.int64, device="cuda")
    xp.xp_profile_timeline(head.handle, buf, wl.K)
    step()
    torch.cuda.synchronize()
    xp.xp_profile_timeline(head.handle, None, wl.K)
    a = buf.cpu().numpy().reshape(-1, wl.K, 12).astype(np.float64) / 1e3   # us
    rs, re = a[:, :, 2], a[:, :, 3]
    used = rs[:, 0] > 0
    rs, re = rs[used], re[used]
    first = rs.min(axis=0)
    period = np.diff(first)
    gap = first[1:] - re[:, :-1].max(axis=0)
    dur = (re - rs)[:, 1:]
    return {"us_per_pass": round(float(np.median(period)), 2),
            "readout_phase_us_median_cta": round(float(np.median(dur)), 2),
            "readout_phase_us_slowest_cta": round(float(np.median(dur.max(axis=0))), 2),
            "latent_gap_us": round(float(np.median(gap)), 2),
            "latent_share_of_pass": round(float(np.median(gap / period)), 4),
            "definition": "gap = first readout start of pass k+1 - last readout end of pass k "
                          "(no CTA streams then: latent stage and its hand-offs); share = gap / "
                          "pass period; medians over passes 1..K-1 of one step"}


def breakdown(wl, head, base, sn, sb, h, anchor, am1, ws, stream, rank, mode):
    import torch
    from jacobi_speculative_decode_gb300 import xp
    rows = wl.rows
    xh = torch.empty(wl.N, wl.B, wl.r, dtype=torch.float32, device="cuda")
    lat = torch.empty(wl.N, wl.B - 1, wl.r, dtype=xp.torch_dtype(wl.dtype), device="cuda")
    blk = torch.empty(wl.N, wl.B, dtype=torch.int64, device="cuda")
    xp.xp_hidden_cache(head.handle, h, wl.N, xh, ws)
    xp.xp_init_argmax(head.handle, base, sn, sb, anchor, wl.N, blk, None, ws)
    n = max(3 * wl.K, 30)

    def loop_us(fn, reps=5):
        # average launch duration over n back-to-back launches (the kernels chain through
        # programmatic dependent launch as inside a step); best of a few repeats
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / n)
        return best

    def latent():
        xp.xp_latent_pass(head.handle, blk, am1, xh, wl.N, lat)

    def readout():
        xp.xp_readout_argmax(head.handle, lat, base, sn, sb, wl.N, blk, None, ws)

    def one_pass():
        latent()
        readout()

    ro_ms = loop_us(readout)
    lat_ms = loop_us(latent)
    pass_ms = loop_us(one_pass)
    persistent = persistent_path(xp, head, wl, base, sn, sb)
    # the K passes alone as the step runs them, timed back to back
    blk2 = blk.clone()
    n_saved = n
    n = 10
    passes_K = lambda: xp.xp_jacobi_passes(head.handle, base, sn, sb, xh, am1, wl.N, wl.K, blk2,
                                           ws)
    passes_ms = loop_us(passes_K)
    n = n_saved
    # the unfused readout: the same rows' fp32 logits written out instead of their argmax
    out = torch.empty(rows, wl.V, dtype=torch.float32, device="cuda")
    lg_ms = loop_us(lambda: xp.xp_refine_logits(head.handle, lat, base, sn, sb, wl.N, out, wl.V))
    del out
    # algorithmic bytes of one readout launch: w2 + base rows + latents in + blk out
    es = 2 if wl.dtype == "bf16" else 4
    ro_bytes = wl.V * wl.r * es + rows * wl.V * es + rows * wl.r * es + rows * 8
    lg_bytes = wl.V * wl.r * es + rows * wl.V * es + rows * wl.r * es + rows * wl.V * 4
    hbm, kind = peaks()

    def persist_roofline(launch_ms):
        # one launch = K passes, each pass_bytes of algorithmic traffic
        k_bytes = wl.K * pass_bytes(wl)
        achieved = k_bytes / (launch_ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4),
                "traffic": committed_traffic(PROFILE_TRAFFIC, PERSIST_SRC, rows,
                                             "dram_bytes_per_pass", wl.K),
                "kernel": "refine_persist_kernel (all K passes)",
                "algorithmic_bytes_per_launch": k_bytes, "launch_us": round(launch_ms * 1e3, 2),
                "peak_kind": f"{kind} (copy bandwidth, sustained loop of one launch per call)"}

    if persistent:
        roof = persist_roofline(passes_ms)
    else:
        achieved = ro_bytes / (ro_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4),
                "traffic": committed_traffic(READOUT_TRAFFIC, READOUT_SRC, rows,
                                             "dram_bytes_per_launch"),
                "kernel": xp.xp_readout_kernel_name(head.handle),
                "algorithmic_bytes_per_launch": ro_bytes, "launch_us": round(ro_ms * 1e3, 2),
                "peak_kind": f"{kind} (copy bandwidth, burst)"}
    out = {
        "roofline": roof,
        "kernel_us": {"readout_argmax": round(ro_ms * 1e3, 2), "latent": round(lat_ms * 1e3, 2),
                      "pass": round(pass_ms * 1e3, 2),
                      "passes_K": round(passes_ms * 1e3, 2),
                      "pass_in_passes_K": round(passes_ms * 1e3 / wl.K, 2),
                      "note": "readout_argmax, latent and pass: the single-pass entry points "
                              "chained back to back; passes_K: xp_jacobi_passes (K passes)"},
        # w2 + base rows + latents in, rows x V fp32 logits out
        "refine_logits": {"us": round(lg_ms * 1e3, 2), "bytes": lg_bytes,
                          "achieved_gbs": round(lg_bytes / (lg_ms / 1e3) / 1e9, 1),
                          "frac": round(lg_bytes / (lg_ms / 1e3) / 1e9 / hbm, 4)},
        # single-pass kernels: what the latent launch adds to a pass
        "latent_share_of_pass_single_pass_kernels": round(max(pass_ms - ro_ms, 0.0) / pass_ms, 4),
    }
    step = lambda: xp.xp_jacobi_refine(head.handle, base, sn, sb, h, anchor, am1, wl.N, wl.K, 0,
                                       blk2, ws)
    if not persistent and wl.topc == 0:
        # the persistent kernel (all K passes in one launch) measured beside the automatic
        # choice, with its phase structure
        xp.xp_set_pass_mode(head.handle, xp.XP_PASSES_PERSISTENT)
        if persistent_path(xp, head, wl, base, sn, sb):
            n_saved = n
            n = 10
            p_launch_ms = loop_us(passes_K)
            p_step_ms = loop_us(step)
            n = n_saved
            out["persistent_kernel"] = {
                "passes_per_s_step": round(wl.K / (p_step_ms / 1e3), 1),
                "roofline": persist_roofline(p_launch_ms),
                **timeline_summary(xp, head, wl, step)}
        xp.xp_set_pass_mode(head.handle, mode)
    if persistent:
        out["persistent"] = timeline_summary(xp, head, wl, step)
        out["latent_share_of_pass"] = out["persistent"]["latent_share_of_pass"]
    else:
        out["latent_share_of_pass"] = out["latent_share_of_pass_single_pass_kernels"]
    return out


def e2e(wl, head, d, ws, args, stream, world):
    """The step through the public call with host buffers: every step copies its inputs
    from pinned host memory and reads blk back, inside the timed region.  Two device
    buffer sets alternate: step i+1's inputs are copied on a second stream while step i
    computes (a step's refine waits for its own copy; a copy waits until the refine
    that last read its buffer set is done)."""
    import torch
    from jacobi_speculative_decode_gb300 import xp
    pin = lambda a: xp.to_device(a, wl.dtype, device="cpu").pin_memory()
    base_h = pin(d["base"])
    h_h = pin(d["h_full"])
    anc_h = torch.from_numpy(d["anchor"]).pin_memory()
    am1_h = torch.from_numpy(d["am1"]).pin_memory()
    blk_h = torch.empty(wl.N, wl.B, dtype=torch.int64).pin_memory()
    sets = []
    for _ in range(2):
        sets.append({"base": torch.empty_like(base_h, device="cuda"),
                     "h": torch.empty_like(h_h, device="cuda"),
                     "anchor": torch.empty_like(anc_h, device="cuda"),
                     "am1": torch.empty_like(am1_h, device="cuda"),
                     "blk": torch.empty(wl.N, wl.B, dtype=torch.int64, device="cuda"),
                     "copied": torch.cuda.Event(), "consumed": torch.cuda.Event()})
    copy_stream = torch.cuda.Stream()
    sn, sb = (wl.B - 1) * wl.V, wl.V

    def copy_in(b):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(b["consumed"])
            b["base"].copy_(base_h, non_blocking=True)
            b["h"].copy_(h_h, non_blocking=True)
            b["anchor"].copy_(anc_h, non_blocking=True)
            b["am1"].copy_(am1_h, non_blocking=True)
            b["copied"].record(copy_stream)

    def compute(b):
        stream.wait_event(b["copied"])
        xp.xp_jacobi_refine(head.handle, b["base"], sn, sb, b["h"], b["anchor"], b["am1"], wl.N,
                            wl.K, wl.topc, b["blk"], ws)
        blk_h.copy_(b["blk"], non_blocking=True)
        b["consumed"].record(stream)

    def run(n):
        copy_in(sets[0])
        for i in range(n):
            if i + 1 < n:
                copy_in(sets[(i + 1) % 2])
            compute(sets[i % 2])

    for b in sets:
        b["consumed"].record(stream)
    run(args.warmup)
    torch.cuda.synchronize()
    # the first step's copy cannot overlap anything: enough steps that the measured rate
    # is the pipeline's steady state (the fill stays inside the timed region)
    steps = max(20, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    h2d = sum(t.numel() * t.element_size() for t in (base_h, h_h, anc_h, am1_h))
    d2h = blk_h.numel() * blk_h.element_size()
    return {"value": round(wl.K * steps * world / (ms / 1e3), 2), "unit": "passes/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / steps, 4), "steps": steps,
            "overlap": "step i+1's host copies run on a second stream during step i"}


# ---------------------------------------------------------------------------
# the fp64 CPU oracle as the baseline / reference arm
# ---------------------------------------------------------------------------

def cpu_baseline(wl, d, budget_s=12.0):
    """Time the oracle as it stands on this host: hidden cache + init once, then full
    passes over the whole batch until the budget is used; scaled to one step of K passes."""
    from oracle import xp_oracle as O
    p = O.params_from_inputs(d, wl.dtype)
    base = O.decode(d["base"], wl.dtype)
    hf = O.decode(d["h_full"], wl.dtype)
    t0 = time.perf_counter()
    xh = O.xh_from_cache(O.hidden_cache(hf, p.down_h, p.down_g), p.in_proj)
    blk = O.init_blk(base, d["anchor"])
    t_fixed = time.perf_counter() - t0
    n = 0
    t1 = time.perf_counter()
    while True:
        blk = O.full_pass(blk, d["am1"], xh, base, p)[0]
        n += 1
        if time.perf_counter() - t1 > budget_s or n >= wl.K:
            break
    t_pass = (time.perf_counter() - t1) / n
    step_s = t_fixed + wl.K * t_pass
    return {"value": round(wl.K / step_s, 4), "unit": "passes/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"hidden cache + init + {n} of {wl.K} full-vocabulary fp64 passes on the "
                      f"whole {wl.N}-block batch, scaled to one {wl.K}-pass step"}


def run_reference(args, rank, world):
    """The fp64 oracle as the reference arm.  One step = one measured sample: the hidden
    cache, the init and ONE full-vocabulary pass over the whole batch.  ms_per_step is
    that sample's measured wall time; value is the rate one K-pass step would have at
    the measured times (hidden cache and init once, then K passes), and the line says so
    under "extrapolated"."""
    if rank != 0:
        return None
    from jacobi_speculative_decode_gb300 import inputs as I
    wl = I.workload(args.workload)
    d = I.make_inputs(wl)
    from oracle import xp_oracle as O
    p = O.params_from_inputs(d, wl.dtype)
    base = O.decode(d["base"], wl.dtype)
    hf = O.decode(d["h_full"], wl.dtype)

    def one_step():
        t0 = time.perf_counter()
        xh = O.xh_from_cache(O.hidden_cache(hf, p.down_h, p.down_g), p.in_proj)
        blk = O.init_blk(base, d["anchor"])
        t1 = time.perf_counter()
        O.full_pass(blk, d["am1"], xh, base, p)
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1

    for _ in range(args.warmup):
        one_step()
    t_start = time.perf_counter()
    samples = [one_step() for _ in range(args.steps)]
    wall = time.perf_counter() - t_start
    t_fixed = sum(a for a, _ in samples) / len(samples)
    t_pass = sum(b for _, b in samples) / len(samples)
    value = wl.K / (t_fixed + wl.K * t_pass)
    return {"impl": "reference",
            "metric": "Jacobi passes/s at N=32,B=16,V=151936 bf16; % of HBM roofline",
            "value": round(value, 4), "unit": "passes/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator; random-init head weights)",
            "config": workload_config(wl),
            "extrapolated": {"passes_timed_per_step": 1, "passes_per_step_in_value": wl.K,
                             "timed_s": round(wall, 3), "fixed_s_per_step": round(t_fixed, 4),
                             "pass_s": round(t_pass, 4)},
            "cpu_baseline": {"value": round(value, 4), "unit": "passes/s",
                             "cores": os.cpu_count(), "kind": "oracle",
                             "sample": "per step: hidden cache + init + one fp64 full-vocabulary "
                                       f"pass over the whole batch (measured); value scales the "
                                       f"measured times to one {wl.K}-pass step"},
            "e2e": {"value": round(value, 4), "unit": "passes/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_native(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1 and args.impl == "native":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
