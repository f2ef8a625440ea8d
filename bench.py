"""Benchmark of the packed verify + OPD-loss pass on GB300.

One step = the whole path over one batch through the C ABI: verification, the
clipped reverse-KL + CE loss and its gradient, in one adaflash_opd_loss_fwd_bwd call
(on this workload: the row pass with the gradient, which reads every logit byte from
HBM once, then the acceptance scan / loss kernel K2).  The same batch is also timed
as separate forward (K1 + K2) and backward (K3) calls.
Default workload: concurrency 128 (V = 151936, bf16 logits, 128 requests with
k_i from a truncated geometric on 1..16, clip c = 0.5).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.  Multi-GPU (torchrun): every rank processes its
own batch (weak scaling, no data-path collective); time is the max over ranks.
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "logit rows/s for fused verify + clipped reverse-KL fwd/bwd; % of HBM peak"
FALLBACK_HBM_GBS = 6800.0


SAMPLED_T = 0.8  # temperature of the sampled-verification measurement
LMHEAD_HIDDEN = 4096  # Qwen3-8B hidden size for the logit-free measurement
LMHEAD_CALLS = 10


# Sources that decide each kernel's code; a recorded ncu figure is used only while they are unchanged.
KERNEL_SOURCES = {
    "rowpass_kernel": ("rowpass.cu", "rowstats.cuh", "common.cuh", "kernels.h"),
    "rowpass_kernel_grad": ("rowpass.cu", "rowstats.cuh", "common.cuh", "kernels.h"),
    "fused_kernel": ("fused.cu", "rowstats.cuh", "common.cuh", "kernels.h"),
    "bwd_kernel": ("backward.cu", "common.cuh", "kernels.h"),
    "lse_rows_kernel": ("sampled.cu", "common.cuh", "kernels.h"),
    "sampled_draw_kernel": ("sampled.cu", "common.cuh", "kernels.h"),
    "lmhead_gemm_kernel": ("lmhead.cu", "tc.cuh", "common.cuh", "kernels.h"),
}


def source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "serving_packed_var_gb300", "csrc", name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _sum_traffic(traffic, names):
    if not all(n in traffic for n in names):
        return None
    return sum(traffic[n]["dram_bytes_per_launch"] for n in names)


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, for the kernels unchanged since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return {}
    return {k: v for k, v in rec.get("kernels", {}).items()
            if k in KERNEL_SOURCES and v.get("source_sha") == source_hash(k)}


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]), hw=f[5], hwt=f[6],
                                 swt=f[7], pcap=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in busy:
            if r["hw"].lower() == "active":
                reasons.add("hw_slowdown")
            if r["hwt"].lower() == "active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"].lower() == "active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"].lower() == "active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in busy), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(busy),
                "power_w_median": statistics.median(r["power"] for r in busy)}


# ---------------------------------------------------------------------------
# distributed helpers (torchrun, one GPU per rank)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rows_per_s(rows_per_rank: int, world: int, ms_max: float, steps: int) -> float:
    """Weak scaling: every rank processes rows_per_rank rows per step; time is the slowest rank's."""
    return world * rows_per_rank / (ms_max * 1e-3 / steps)


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

K_MIX = {
    "tiny": "k_i = {16, 9, 3, 1}, L_i ~ U{0..k_i}",
    "single": "k = 16, L ~ U{0..16}",
    "c32": "k_i ~ U{1..16}, L_i ~ Bin(k_i, 0.6)",
    "c128": "k_i truncated-geometric (p = 0.07) on 1..16, L_i ~ Bin(k_i, 0.6), 5% of rows with 64 entries at "
            "target -30 / draft +6",
    "c128_clip": "as c128 with draft +16 on the planted entries",
    "stress": "k_i = 16, L_i ~ U{0..16}, 1% exact-tie target rows, 1% draft == target rows, rows off the "
              "16-byte grid (ld = V)",
}


def workload_text(w):
    return (f"{w.name}: concurrency {w.num_requests}, V={w.vocab}, {w.d_dtype} draft / {w.t_dtype} target, "
            f"{K_MIX.get(w.name.split('[')[0], 'k_i as generated')}, clip c={w.clip_c}")


def workload_from_args(args, make_workload, seed=0):
    """The named workload, or its first --requests requests (same rows, same planted structure)."""
    import numpy as np
    w = make_workload(args.workload, seed=seed)
    n = getattr(args, "requests", 0)
    if n and n < w.num_requests:
        nd = int(np.sum(w.k[:n]))
        nt = nd + n
        over = dict(k=w.k[:n], planted_accept=w.planted_accept[:n])
        for key, lim in (("clip_rows", nd), ("equal_rows", nd), ("tie_rows", nt), ("constant_target_rows", nt)):
            rows = getattr(w, key)
            over[key] = rows[rows < lim]
        w = make_workload(args.workload, seed=seed, **over)
        w.name = f"{args.workload}[:{n}]"
    return w


def workload_config(w):
    return {
        "workload": workload_text(w) + ", fwd+bwd",
        "num_requests": w.num_requests, "draft_rows": w.num_draft_rows, "target_rows": w.num_target_rows,
        "vocab": w.vocab, "input_dtype": w.d_dtype, "clip_c": w.clip_c, "ce_weight": w.ce_weight,
        "l2": "inputs larger than L2 (no flush): forward reads and backward traffic exceed 129 MB",
        "parallelism": "replica per GPU (weak scaling)",
    }


def single_pass_bytes(w):
    """adaflash_opd_loss_fwd_bwd on a batch of many rows: every logit byte read once, dz written once."""
    V = w.vocab
    bz, bt = w.bytes_per_draft_elem, w.bytes_per_target_elem
    return (w.num_draft_rows * (bz + bt + 4) + w.num_requests * bt) * V


def algorithmic_bytes(w):
    V = w.vocab
    bz, bt = w.bytes_per_draft_elem, w.bytes_per_target_elem
    fwd = (w.num_draft_rows * (bz + bt) + w.num_requests * bt) * V
    bwd = w.num_draft_rows * (bz + bt + 4) * V
    return fwd, bwd


def cpu_baseline(b, budget_s=10.0):
    """The plain C++ float64 oracle as it stands (forward + gradient per draft row) on a bounded
    sample of this workload's draft rows: one thread, then every host core (std::thread over rows)."""
    import numpy as np

    from oracle import cpp
    w = b.w
    cores = os.cpu_count() or 1
    cpp.build()

    def run(threads, budget):
        rows, t0 = 0, time.perf_counter()
        while rows < w.num_draft_rows and time.perf_counter() - t0 < budget:
            sel = np.arange(rows, min(w.num_draft_rows, rows + 2 * threads), dtype=np.int32)
            cpp.opd_rows(b.draft, w.d_dtype, b.target, w.t_dtype, b.doff, w.vocab, w.clip_c, w.ce_weight,
                         rows=sel, grad=True, threads=threads)
            rows += len(sel)
        return rows, time.perf_counter() - t0

    r1, e1 = run(1, budget_s / 4)
    rn, en = run(cores, budget_s * 3 / 4)
    return {"value": rn / en, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "value_1core": r1 / e1,
            "sample": f"plain C++ float64 oracle (oracle/opd_ref.cpp), forward + gradient per draft row of the "
                      f"same workload: {r1} rows on 1 thread in {e1:.1f} s, then {rn} rows on {cores} threads "
                      f"(std::thread over rows) in {en:.1f} s"}


def run_ours(args):
    import numpy as np
    import torch

    import serving_packed_var_gb300 as af
    from synth import make_workload, materialize

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from serving_packed_var_gb300.build import build
    if rank == 0 or world == 1:
        build()
    barrier()

    w = workload_from_args(args, make_workload, seed=rank)
    b = materialize(w)
    Nd, R = w.num_draft_rows, w.num_requests

    def dev_from(arr, dtype):
        if dtype == "bf16":
            return torch.from_numpy(arr.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(arr).to(dev)

    z = dev_from(b.draft, w.d_dtype)
    t = dev_from(b.target, w.t_dtype)
    tok = torch.from_numpy(b.tokens).to(dev)
    doff = torch.from_numpy(b.doff).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = None
    grad = torch.empty((Nd, w.vocab), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    fbo = {"grad": grad}

    def step():
        nonlocal fbo
        fbo = af.adaflash_opd_loss_fwd_bwd(z, t, tok, doff, w.clip_c, w.ce_weight, grad_scale=1.0 / Nd, out=fbo,
                                           status=status)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    # ---- the timed region: K steps, one adaflash_opd_loss_fwd_bwd call each ----
    K = args.steps
    launches0 = af.adaflash_kernel_launches()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(K):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
    barrier()
    launches = af.adaflash_kernel_launches() - launches0
    ms_local = start.elapsed_time(stop)
    ms = max_over_ranks(ms_local, dev if world > 1 else None)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    # the same step as separate forward and backward calls (per-call events)
    Ks = max(20, K // 2)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(Ks)]
    for i in range(Ks + 3):
        if i >= 3:
            ev[i - 3][0].record(stream)
        out = af.adaflash_opd_loss_fwd(z, t, tok, doff, w.clip_c, w.ce_weight, out=out, status=status)
        if i >= 3:
            ev[i - 3][1].record(stream)
        af.adaflash_opd_loss_bwd(z, t, doff, out["target_argmax"], out["row_stats"], w.clip_c, w.ce_weight,
                                 grad_scale=1.0 / Nd, out=grad, status=status)
        if i >= 3:
            ev[i - 3][2].record(stream)
    torch.cuda.synchronize()
    fwd_ms = sum(e0.elapsed_time(e1) for e0, e1, _ in ev) / Ks
    bwd_ms = sum(e1.elapsed_time(e2) for _, e1, e2 in ev) / Ks
    sep_ms = sum(e0.elapsed_time(e2) for e0, _, e2 in ev) / Ks
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    # the forward pass alone (back to back, no backward in between)
    fa, fb_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    Kf = max(20, K // 2)
    torch.cuda.synchronize()
    fa.record(stream)
    for _ in range(Kf):
        out = af.adaflash_opd_loss_fwd(z, t, tok, doff, w.clip_c, w.ce_weight, out=out, status=status)
    fb_.record(stream)
    torch.cuda.synchronize()
    fwd_alone_ms = fa.elapsed_time(fb_) / Kf

    fwd_bwd_ms = ms_local / K

    # greedy verification alone (adaflash_verify_packed: target rows only), calls back to back
    vout = af.adaflash_verify_packed(t, tok, doff, status=status)
    torch.cuda.synchronize()
    va, vb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    va.record(stream)
    for _ in range(Kf):
        vout = af.adaflash_verify_packed(t, tok, doff, out=vout, status=status)
    vb.record(stream)
    torch.cuda.synchronize()
    verify_ms = va.elapsed_time(vb) / Kf

    # temperature-sampled verification of the same batch (seeded uniforms, T = 0.8), calls back to back
    urng = np.random.default_rng(1000 + rank)
    u_acc = torch.from_numpy(urng.random(Nd, dtype=np.float32)).to(dev)
    u_smp = torch.from_numpy(urng.random(R, dtype=np.float32)).to(dev)
    sout = af.adaflash_verify_sampled(z, t, tok, doff, SAMPLED_T, u_acc, u_smp, status=status)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sa.record(stream)
    for _ in range(Kf):
        sout = af.adaflash_verify_sampled(z, t, tok, doff, SAMPLED_T, u_acc, u_smp, out=sout, status=status)
    sb.record(stream)
    torch.cuda.synchronize()
    sampled_ms = sa.elapsed_time(sb) / Kf
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    # cold-HBM per-call times: an L2-sized flush (twice the L2) before every call
    if args.profile_only:
        # a profiling run: the warm-up, the timed steps, the separate calls, verification
        # and sampled verification only
        print(json.dumps({"profile_only": True, "workload": workload_text(w), "ms_per_step": ms_local / K,
                          "launches": launches}), flush=True)
        return
    cold = run_cold(w, dev, af, torch, np, z, t, tok, doff, status, out, grad, stream, fbo)
    cold_clean = run_cold(w, dev, af, torch, np, z, t, tok, doff, status, out, grad, stream, fbo, by_read=True)

    # concurrency 1 (one request of 16 draft rows): the step eager and replayed from a CUDA graph
    small = run_small_batch_graph(dev, af, torch, np, make_workload, materialize)

    # the other benchmark configurations (concurrency 1 and 32, the stress batch)
    configs = run_configs(dev, af, torch, np, stream, hbm_peak()[0], make_workload, materialize)

    # the logit-free forward from hidden states at Qwen3-8B shapes (H = 4096, shared head),
    # the same packed layout as this workload
    lm = run_lmhead(args, w, dev, af, torch, np, stream)

    # end to end: pinned host inputs -> device, step, verify outputs + loss back to host
    e2e = run_e2e(args, b, w, dev, af, torch, np)
    e2e_grad = run_e2e(args, b, w, dev, af, torch, np, grad_to_host=True)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    peak, peak_kind = hbm_peak()
    fb, bb = algorithmic_bytes(w)
    spb = single_pass_bytes(w)
    vb_bytes = w.num_target_rows * w.bytes_per_target_elem * w.vocab  # every target logit once
    traffic = ncu_traffic()
    fwd_gbs = fb / (fwd_ms * 1e-3) / 1e9
    bwd_gbs = bb / (bwd_ms * 1e-3) / 1e9
    fwd_alone_gbs = fb / (fwd_alone_ms * 1e-3) / 1e9
    kernels = {
        "fwd_pass": {"kernels": "rowpass (K1) + finalize (K2), in the separate-call step (after the previous "
                                "backward)",
                     "ms": fwd_ms, "bytes": fb, "achieved_gbs": fwd_gbs,
                     "frac": fwd_gbs / peak, "rows_per_s": Nd / (fwd_ms * 1e-3)},
        "fwd_alone": {"kernels": "rowpass (K1) + finalize (K2), forward calls back to back", "ms": fwd_alone_ms,
                      "bytes": fb, "achieved_gbs": fwd_alone_gbs, "frac": fwd_alone_gbs / peak,
                      "rows_per_s": Nd / (fwd_alone_ms * 1e-3)},
        "bwd": {"kernels": "bwd (K3)", "ms": bwd_ms, "bytes": bb, "achieved_gbs": bwd_gbs, "frac": bwd_gbs / peak,
                "rows_per_s": Nd / (bwd_ms * 1e-3)},
        "fwd_bwd_call": {"kernels": "adaflash_opd_loss_fwd_bwd (the step): the row pass with the gradient (one "
                                    "launch on this batch; each slice read from HBM once, re-read from L2 for dz) "
                                    "+ K2; calls back to back",
                         "ms": fwd_bwd_ms, "bytes": spb, "achieved_gbs": spb / (fwd_bwd_ms * 1e-3) / 1e9,
                         "frac": spb / (fwd_bwd_ms * 1e-3) / 1e9 / peak, "rows_per_s": Nd / (fwd_bwd_ms * 1e-3),
                         "traffic": traffic.get("rowpass_kernel_grad", {}).get("dram_bytes_per_launch")},
        "step_separate": {"kernels": "adaflash_opd_loss_fwd (K1 + K2) then adaflash_opd_loss_bwd (K3), per-call "
                                     "events", "ms": sep_ms, "bytes": fb + bb,
                          "achieved_gbs": (fb + bb) / (sep_ms * 1e-3) / 1e9,
                          "frac": (fb + bb) / (sep_ms * 1e-3) / 1e9 / peak, "rows_per_s": Nd / (sep_ms * 1e-3)},
        "verify_packed": {"kernels": "rowpass (K1, target rows only) + finalize (K2): adaflash_verify_packed, calls back "
                                     "to back", "ms": verify_ms, "bytes": vb_bytes,
                          "achieved_gbs": vb_bytes / (verify_ms * 1e-3) / 1e9,
                          "frac": vb_bytes / (verify_ms * 1e-3) / 1e9 / peak, "rows_per_s": Nd / (verify_ms * 1e-3)},
        "sampled_verify": {"kernels": f"lse_rows (S1) + accept/draw (S2), T = {SAMPLED_T}, calls back to back",
                           "ms": sampled_ms, "bytes": fb, "achieved_gbs": fb / (sampled_ms * 1e-3) / 1e9,
                           "frac": fb / (sampled_ms * 1e-3) / 1e9 / peak, "rows_per_s": Nd / (sampled_ms * 1e-3),
                           "traffic": _sum_traffic(traffic, ("lse_rows_kernel", "sampled_draw_kernel"))},
    }
    # The step's dominant kernel is the row pass with the gradient; its time is taken as
    # the whole call's (the acceptance scan / loss kernel adds a few microseconds).
    roofline = {"bound": "hbm", "achieved": kernels["fwd_bwd_call"]["achieved_gbs"], "peak": peak, "unit": "GB/s",
                "frac": kernels["fwd_bwd_call"]["frac"],
                "traffic": traffic.get("rowpass_kernel_grad", {}).get("dram_bytes_per_launch"),
                "kernel": "row pass with the gradient (one launch on this batch) + K2, per adaflash_opd_loss_fwd_bwd call",
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s", "algorithmic_bytes_per_launch": spb}
    roofline_bwd = {"bound": "hbm", "achieved": bwd_gbs, "peak": peak, "unit": "GB/s", "frac": bwd_gbs / peak,
                    "traffic": traffic.get("bwd_kernel", {}).get("dram_bytes_per_launch"),
                    "kernel": "bwd (K3) in the separate-call step", "algorithmic_bytes_per_launch": bb}
    roofline_lmhead = None
    if lm is not None:
        tpeak, tkind = tensor_peak()
        kernels["lmhead_fwd"] = {"kernels": "L0 gather + L1 tcgen05 head GEMM with per-tile row reduction + "
                                            "L2 combine + K2 (adaflash_lmhead_opd_fwd), calls back to back",
                                 "ms": lm["ms"], "flops": lm["flops"], "achieved_tflops": lm["tflops"],
                                 "frac": lm["tflops"] / tpeak, "rows_per_s": Nd / (lm["ms"] * 1e-3),
                                 "hidden": lm["hidden"], "vocab": lm["vocab"], "e2e": lm["e2e"]}
        roofline_lmhead = {"bound": "tensor", "achieved": lm["tflops"], "peak": tpeak, "unit": "TFLOP/s",
                           "frac": lm["tflops"] / tpeak,
                           "traffic": traffic.get("lmhead_gemm_kernel", {}).get("dram_bytes_per_launch"),
                           "kernel": "logit-free verify + loss forward (head GEMM dominant)",
                           "algorithmic_flops_per_launch": lm["flops"],
                           "peak_source": f"{tkind} (MEASURED_PEAKS.json bf16_tflops, burst)"}
    roofline_fwd = {"bound": "hbm", "achieved": fwd_alone_gbs, "peak": peak, "unit": "GB/s",
                    "frac": fwd_alone_gbs / peak,
                    "traffic": traffic.get("rowpass_kernel", {}).get("dram_bytes_per_launch"),
                    "kernel": "fused verify + loss forward (K1 + K2), calls back to back",
                    "algorithmic_bytes_per_launch": fb, "in_step_frac": fwd_gbs / peak}
    value = whole_job_rows_per_s(Nd, world, ms, K)
    head_cfg = {"workload": workload_text(w), "draft_rows": Nd, "target_rows": w.num_target_rows,
                "fwd": _entry(fwd_alone_ms, fb, Nd, peak), "step": _entry(fwd_bwd_ms, spb, Nd, peak),
                "note": "the headline configuration: the step is the timed region above"}
    order = ["single", "c32", w.name, "stress"]
    all_configs = {k: (head_cfg if k == w.name else configs[k]) for k in dict.fromkeys(order) if
                   k == w.name or k in configs}
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded; no datasets or weights)",
        "config": workload_config(w), "roofline": roofline, "roofline_fwd": roofline_fwd, "roofline_bwd": roofline_bwd,
        "roofline_lmhead": roofline_lmhead, "kernels": kernels, "configs": all_configs, "small_batch": small, "cold": cold, "cold_clean": cold_clean,
        "e2e": e2e, "e2e_grad_to_host": e2e_grad, "gpu_launches": launches, "clocks": clk.summary(),
        "cpu_baseline": cpu_baseline(b) if world == 1 or rank == 0 else None,
        "impl": "ours",
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def run_cold(w, dev, af, torch, np, z, t, tok, doff, status, out, grad, stream, fbo, reps=21, by_read=False):
    """The step call, the forward call and the backward call, each timed after evicting the L2
    with a pass over twice its size (cold HBM); median and 10th / 90th percentiles over the reps.

    by_read=False writes the buffer, which leaves about an L2 of dirty lines that the timed call
    then writes back; by_read=True reads it (a reduction), which leaves clean lines, so the timed
    call pays for its own traffic only."""
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (129 << 20)
    flush = torch.zeros(2 * l2 // 4, dtype=torch.int32, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)

    def evict(r):
        if by_read:
            torch.sum(flush, dim=0, dtype=torch.int32, out=sink[0])
        else:
            flush.fill_(r & 0xff)

    Nd = w.num_draft_rows
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for r in range(reps):
        evict(r + 7)
        a, b = evs[r]
        a.record(stream)
        af.adaflash_opd_loss_fwd_bwd(z, t, tok, doff, w.clip_c, w.ce_weight, grad_scale=1.0 / Nd, out=fbo,
                                     status=status)
        b.record(stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2 * reps)]
    for r in range(reps):
        evict(r)
        a, b = ev[2 * r]
        a.record(stream)
        af.adaflash_opd_loss_fwd(z, t, tok, doff, w.clip_c, w.ce_weight, out=out, status=status)
        b.record(stream)
        evict(r + 1)
        a, b = ev[2 * r + 1]
        a.record(stream)
        af.adaflash_opd_loss_bwd(z, t, doff, out["target_argmax"], out["row_stats"], w.clip_c, w.ce_weight,
                                 grad_scale=1.0 / Nd, out=grad, status=status)
        b.record(stream)
    torch.cuda.synchronize()
    stp = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    fwd = sorted(ev[2 * r][0].elapsed_time(ev[2 * r][1]) * 1e3 for r in range(reps))
    bwd = sorted(ev[2 * r + 1][0].elapsed_time(ev[2 * r + 1][1]) * 1e3 for r in range(reps))
    del flush

    def q(xs, f):
        return xs[min(len(xs) - 1, int(round(f * (len(xs) - 1))))]

    return {"flush_bytes": 2 * l2, "reps": reps, "flush": "read (clean lines)" if by_read else "write (dirty lines)",
            "step_us": {"median": q(stp, 0.5), "p10": q(stp, 0.1), "p90": q(stp, 0.9)},
            "fwd_us": {"median": q(fwd, 0.5), "p10": q(fwd, 0.1), "p90": q(fwd, 0.9)},
            "bwd_us": {"median": q(bwd, 0.5), "p10": q(bwd, 0.1), "p90": q(bwd, 0.9)}}


def _entry(ms, nbytes, rows, peak):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": ms, "bytes": nbytes, "achieved_gbs": gbs, "frac": gbs / peak, "rows_per_s": rows / (ms * 1e-3)}


def _back_to_back(torch, stream, fn, n, warm_s=0.3):
    """Mean time per call (ms) of n calls back to back on `stream`, after about warm_s of warm-up calls."""
    t0, k = time.perf_counter(), 0
    while k < 3 or (time.perf_counter() - t0 < warm_s and k < 5000):
        fn()
        k += 1
        if k % 8 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def _graph_replay(torch, fn, n):
    """Mean time per replay (ms) of fn captured once in a CUDA graph."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    for _ in range(20):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(n):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def run_configs(dev, af, torch, np, stream, peak, make_workload, materialize):
    """Every benchmark configuration besides the headline one, each on its own batch:
    concurrency 1 (the forward alone, as the configuration states, eager and replayed from
    a CUDA graph; and the single-call step), concurrency 32 (the step and the forward) and
    the stress batch (the step, the forward, the separate calls and greedy verification).
    Times are means over calls back to back (the forward and the step as calls marshalled
    once with prepare()); bytes are algorithmic (every logit byte read once, dz written once)."""
    res = {}
    for name in ("single", "c32", "stress"):
        b = materialize(make_workload(name))
        w = b.w
        Nd, R, V = w.num_draft_rows, w.num_requests, w.vocab

        def dev_from(arr, dtype):
            if dtype == "bf16":
                return torch.from_numpy(arr.view(np.int16)).to(dev).view(torch.bfloat16)
            return torch.from_numpy(arr).to(dev)

        z, t = dev_from(b.draft, w.d_dtype), dev_from(b.target, w.t_dtype)
        tok, doff = torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.doff).to(dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        grad = torch.empty((Nd, V), dtype=torch.float32, device=dev)
        fb, bb = algorithmic_bytes(w)
        spb = single_pass_bytes(w)
        o = {"out": af.adaflash_opd_loss_fwd(z, t, tok, doff, w.clip_c, w.ce_weight, status=st)}
        fbo = af.adaflash_opd_loss_fwd_bwd(z, t, tok, doff, w.clip_c, w.ce_weight, grad_scale=1.0 / Nd,
                                           out={"grad": grad}, status=st)

        def fwd():
            af.adaflash_opd_loss_fwd(z, t, tok, doff, w.clip_c, w.ce_weight, out=o["out"], status=st)

        def step():
            af.adaflash_opd_loss_fwd_bwd(z, t, tok, doff, w.clip_c, w.ce_weight, grad_scale=1.0 / Nd, out=fbo,
                                         status=st)

        # eager calls marshalled once (prepare): at concurrency 1 the host's time per call
        # through the Python binding would otherwise be the floor
        fwd_prep, _ = af.prepare(af.adaflash_opd_loss_fwd, z, t, tok, doff, w.clip_c, w.ce_weight, out=o["out"],
                                 status=st)
        step_prep, _ = af.prepare(af.adaflash_opd_loss_fwd_bwd, z, t, tok, doff, w.clip_c, w.ce_weight,
                                  grad_scale=1.0 / Nd, out=fbo, status=st)

        n = {"single": 400, "c32": 200, "stress": 40}[name]
        e = {"workload": workload_text(w), "draft_rows": Nd, "target_rows": w.num_target_rows}
        e["fwd"] = _entry(_back_to_back(torch, stream, fwd_prep, n), fb, Nd, peak)
        e["step"] = _entry(_back_to_back(torch, stream, step_prep, n), spb, Nd, peak)
        if name == "single":
            e["fwd_graph"] = _entry(_graph_replay(torch, fwd, n), fb, Nd, peak)
            e["step_graph"] = _entry(_graph_replay(torch, step, n), spb, Nd, peak)
        if name == "stress":
            def separate():
                fwd()
                af.adaflash_opd_loss_bwd(z, t, doff, o["out"]["target_argmax"], o["out"]["row_stats"], w.clip_c,
                                         w.ce_weight, grad_scale=1.0 / Nd, out=grad, status=st)
            e["step_separate"] = _entry(_back_to_back(torch, stream, separate, n), fb + bb, Nd, peak)
            vo = {"v": af.adaflash_verify_packed(t, tok, doff, status=st)}

            def verify():
                af.adaflash_verify_packed(t, tok, doff, out=vo["v"], status=st)
            e["verify_packed"] = _entry(_back_to_back(torch, stream, verify, n),
                                        w.num_target_rows * w.bytes_per_target_elem * V, Nd, peak)
            urng = np.random.default_rng(2000)
            u_acc = torch.from_numpy(urng.random(Nd, dtype=np.float32)).to(dev)
            u_smp = torch.from_numpy(urng.random(R, dtype=np.float32)).to(dev)
            so = {"s": af.adaflash_verify_sampled(z, t, tok, doff, SAMPLED_T, u_acc, u_smp, status=st)}

            def sampled():
                af.adaflash_verify_sampled(z, t, tok, doff, SAMPLED_T, u_acc, u_smp, out=so["s"], status=st)
            e["sampled_verify"] = _entry(_back_to_back(torch, stream, sampled, n), fb, Nd, peak)
        torch.cuda.synchronize()
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())} ({name})")
        res[name] = e
        del z, t, grad, o, fbo
        torch.cuda.empty_cache()
    return res


def run_small_batch_graph(dev, af, torch, np, make_workload, materialize):
    """Concurrency 1 (`single`: 16 draft rows, 17 target rows): the single-call step eager,
    and the same call captured once in a CUDA graph and replayed (launch-bound at this size)."""
    b = materialize(make_workload("single"))
    w = b.w
    z = torch.from_numpy(b.draft.view(np.int16)).to(dev).view(torch.bfloat16)
    t = torch.from_numpy(b.target.view(np.int16)).to(dev).view(torch.bfloat16)
    tok, doff = torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.doff).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream()
    n = 200
    with torch.cuda.stream(s):
        out = af.adaflash_opd_loss_fwd_bwd(z, t, tok, doff, w.clip_c, w.ce_weight, grad_scale=1.0 / w.num_draft_rows,
                                           status=st)
        for _ in range(10):
            af.adaflash_opd_loss_fwd_bwd(z, t, tok, doff, w.clip_c, w.ce_weight, grad_scale=1.0 / w.num_draft_rows,
                                         out=out, status=st)
        a, bb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(n):
            af.adaflash_opd_loss_fwd_bwd(z, t, tok, doff, w.clip_c, w.ce_weight, grad_scale=1.0 / w.num_draft_rows,
                                         out=out, status=st)
        bb.record(s)
    s.synchronize()
    eager_us = a.elapsed_time(bb) / n * 1e3
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        af.adaflash_opd_loss_fwd_bwd(z, t, tok, doff, w.clip_c, w.ce_weight, grad_scale=1.0 / w.num_draft_rows,
                                     out=out, status=st)
    for _ in range(10):
        graph.replay()
    torch.cuda.synchronize()
    a.record()
    for _ in range(n):
        graph.replay()
    bb.record()
    torch.cuda.synchronize()
    graph_us = a.elapsed_time(bb) / n * 1e3
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())} (small batch)")
    return {"workload": "single: 1 request, k = 16, V = 151936, bf16, fwd + bwd in one call (the on-chip fused kernel)",
            "eager_us_per_step": eager_us, "graph_us_per_step": graph_us,
            "rows_per_s_graph": w.num_draft_rows / (graph_us * 1e-6)}


def run_lmhead(args, w, dev, af, torch, np, stream):
    """Time adaflash_lmhead_opd_fwd on hidden states of this workload's packed layout."""
    if args.no_lmhead:
        return None
    from synth.lmhead import LMHeadWorkload, materialize_lmhead
    lw = LMHeadWorkload(name="lm_" + w.name, vocab=w.vocab, hidden=LMHEAD_HIDDEN, k=w.k,
                        planted_accept=w.planted_accept, clip_c=w.clip_c, ce_weight=w.ce_weight, seed=w.seed)
    lb = materialize_lmhead(lw)

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    hd, ht, wh = dev_bf16(lb.hd), dev_bf16(lb.ht), dev_bf16(lb.wt)
    tok = torch.from_numpy(lb.tokens).to(dev)
    doff = torch.from_numpy(lb.doff).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    R, Nd = lw.num_requests, lw.num_draft_rows
    ws = torch.empty(af.adaflash_lmhead_workspace_bytes(R, Nd, lw.vocab, lw.hidden), dtype=torch.uint8, device=dev)
    out = af.adaflash_lmhead_opd_fwd(hd, ht, wh, wh, tok, doff, lw.clip_c, lw.ce_weight, workspace=ws, status=st)
    for _ in range(2):
        af.adaflash_lmhead_opd_fwd(hd, ht, wh, wh, tok, doff, lw.clip_c, lw.ce_weight, workspace=ws, out=out,
                                   status=st)
    torch.cuda.synchronize()
    n = LMHEAD_CALLS
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        af.adaflash_lmhead_opd_fwd(hd, ht, wh, wh, tok, doff, lw.clip_c, lw.ce_weight, workspace=ws, out=out,
                                   status=st)
    b.record(stream)
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())} (lmhead)")
    ms = a.elapsed_time(b) / n
    flops = 2.0 * (2 * Nd + R) * lw.hidden * lw.vocab

    # End to end: every step copies the draft and target hidden states (and the tokens and
    # offsets) from pinned host memory, runs the call with the head resident on the device,
    # and reads the verification outputs and the loss back.
    hdh = torch.from_numpy(np.ascontiguousarray(lb.hd).view(np.int16)).pin_memory()
    hth = torch.from_numpy(np.ascontiguousarray(lb.ht).view(np.int16)).pin_memory()
    tokh, doffh = torch.from_numpy(lb.tokens).pin_memory(), torch.from_numpy(lb.doff).pin_memory()
    hdd, htd = torch.empty_like(hdh, device=dev), torch.empty_like(hth, device=dev)
    tokd, doffd = torch.empty_like(tokh, device=dev), torch.empty_like(doffh, device=dev)
    res_h = {k: torch.empty(R, dtype=dt).pin_memory() for k, dt in
             (("accept_len", torch.int32), ("bonus_token", torch.int32), ("accept_rate", torch.float32))}
    res_h["loss"] = torch.empty(1, dtype=torch.float32).pin_memory()

    def e2e_step():
        hdd.copy_(hdh, non_blocking=True)
        htd.copy_(hth, non_blocking=True)
        tokd.copy_(tokh, non_blocking=True)
        doffd.copy_(doffh, non_blocking=True)
        af.adaflash_lmhead_opd_fwd(hdd.view(torch.bfloat16), htd.view(torch.bfloat16), wh, wh, tokd, doffd,
                                   lw.clip_c, lw.ce_weight, workspace=ws, out=out, status=st)
        for k2, v in res_h.items():
            v.copy_(out[k2], non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    blocks = []
    for _ in range(3):  # the median of three timed blocks, as for the step's end-to-end figure
        t0 = time.perf_counter()
        for _ in range(n):
            e2e_step()
        torch.cuda.synchronize()
        blocks.append(time.perf_counter() - t0)
    el = statistics.median(blocks)
    bi = sum(x.numel() * x.element_size() for x in (hdh, hth, tokh, doffh))
    bo = sum(x.numel() * x.element_size() for x in res_h.values())
    e2e = {"value": Nd * n / el, "unit": "rows/s", "ms_per_step": el / n * 1e3, "h2d_bytes_per_step": bi,
           "d2h_bytes_per_step": bo, "steps": n, "blocks_ms_per_step": [round(b / n * 1e3, 4) for b in blocks],
           "returns": "verification outputs and loss to host memory (the heads stay resident on the device)"}
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())} (lmhead e2e)")
    del hd, ht, wh, ws, hdd, htd
    return {"ms": ms, "flops": flops, "tflops": flops / (ms * 1e-3) / 1e12, "hidden": lw.hidden, "vocab": lw.vocab,
            "e2e": e2e}


def run_e2e(args, b, w, dev, af, torch, np, grad_to_host=False):
    """Same step through the public API from pinned host buffers, copies inside the timed region.

    Every step copies its inputs from pinned host memory and reads its results back:
    the verification outputs and the loss, and with grad_to_host the float32 gradient
    too (otherwise dz stays on the device, where an optimiser step would consume it).
    The copy of step i + 1 (on a copy stream, into the other of two device input
    buffers) overlaps the kernels of step i, as a serving loop would pipeline them.
    """
    Nd = w.num_draft_rows
    zh = torch.from_numpy(b.draft.view(np.int16) if w.d_dtype == "bf16" else b.draft).pin_memory()
    th = torch.from_numpy(b.target.view(np.int16) if w.t_dtype == "bf16" else b.target).pin_memory()
    tokh = torch.from_numpy(b.tokens).pin_memory()
    doffh = torch.from_numpy(b.doff).pin_memory()
    bufs = []
    for _ in range(2):
        zd, td = torch.empty_like(zh, device=dev), torch.empty_like(th, device=dev)
        bufs.append(dict(z=zd, t=td, tok=torch.empty_like(tokh, device=dev), doff=torch.empty_like(doffh, device=dev),
                         zv=zd.view(torch.bfloat16) if w.d_dtype == "bf16" else zd,
                         tv=td.view(torch.bfloat16) if w.t_dtype == "bf16" else td))
    R = w.num_requests
    res_h = {"accept_len": torch.empty(R, dtype=torch.int32).pin_memory(),
             "bonus_token": torch.empty(R, dtype=torch.int32).pin_memory(),
             "accept_rate": torch.empty(R, dtype=torch.float32).pin_memory(),
             "loss": torch.empty(1, dtype=torch.float32).pin_memory()}
    grad = torch.empty((Nd, w.vocab), dtype=torch.float32, device=dev)
    if grad_to_host:
        res_h["grad"] = torch.empty((Nd, w.vocab), dtype=torch.float32).pin_memory()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    comp = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]
    for e in consumed:
        e.record(comp)
    out = None
    bi = sum(x.numel() * x.element_size() for x in (zh, th, tokh, doffh))
    bo = sum(x.numel() * x.element_size() for x in res_h.values())
    steps = max(3, min(args.steps, 50))
    it = [0]

    def step():
        nonlocal out
        k = it[0] % 2
        it[0] += 1
        bf = bufs[k]
        copy_stream.wait_event(consumed[k])  # the kernels that last read this buffer are done
        with torch.cuda.stream(copy_stream):
            bf["z"].copy_(zh, non_blocking=True)
            bf["t"].copy_(th, non_blocking=True)
            bf["tok"].copy_(tokh, non_blocking=True)
            bf["doff"].copy_(doffh, non_blocking=True)
            copied[k].record(copy_stream)
        comp.wait_event(copied[k])
        out = af.adaflash_opd_loss_fwd_bwd(bf["zv"], bf["tv"], bf["tok"], bf["doff"], w.clip_c, w.ce_weight,
                                           grad_scale=1.0 / Nd, out=out if out is not None else {"grad": grad},
                                           status=status)
        consumed[k].record(comp)
        for key, v in res_h.items():
            v.copy_(out[key], non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    # three timed blocks, the median reported: a host-side stall in one block (the copies
    # go through host memory) does not decide the figure
    world = int(os.environ.get("WORLD_SIZE", "1"))
    blocks = []
    for _ in range(3):
        barrier()
        t0 = time.perf_counter()
        for _ in range(steps):
            step()
        torch.cuda.synchronize()
        blocks.append(max_over_ranks(time.perf_counter() - t0, dev if world > 1 else None))
    el = statistics.median(blocks)
    return {"value": world * Nd * steps / el, "unit": "rows/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "steps": steps, "ms_per_step": el / steps * 1e3,
            "blocks_ms_per_step": [round(b / steps * 1e3, 4) for b in blocks],
            "returns": ("verification outputs, loss and the float32 gradient to host memory" if grad_to_host else
                        "verification outputs and loss to host memory; the float32 gradient stays on the device "
                        "for an on-device optimiser step"),
            "pipelined": "the copy of step i + 1 overlaps the kernels of step i (two device input buffers)"}


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from synth import make_workload, materialize
    w = workload_from_args(args, make_workload, seed=0)
    b = materialize(w)
    base = None
    # the whole run (warm-up and timed steps) is bounded to about two minutes of host time
    # whatever K and W are: each step is a sample of at least one block of rows per thread
    # count, with a time budget of 120 s / (K + W), at most 20 s
    budget = max(0.02, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(b, budget_s=budget)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        base = cpu_baseline(b, budget_s=budget)
        vals.append(base["value"])
    el = time.perf_counter() - t0
    value = statistics.mean(vals)
    line = {"metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el / max(1, args.steps) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": workload_config(w), "impl": "reference",
            "cpu_baseline": dict(base, value=value),
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c128")
    ap.add_argument("--no-lmhead", action="store_true", help="skip the logit-free (hidden-state) measurement")
    ap.add_argument("--requests", type=int, default=0,
                    help="take only the first N requests of the workload (a smaller case of the same shape)")
    ap.add_argument("--profile-only", action="store_true",
                    help="warm-up, timed steps and the separate calls only; prints a short JSON line (for ncu)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
