"""Benchmark of the vocabulary-sharded embedding + globally normalised
cross-entropy step on one GB300 (or N independent replicas under torchrun).

One step = embedding lookup of the step's token ids, loss forward, loss
backward (dH and the tied dW), embedding backward into the same dW, on the
Qwen3-like tied workload (T=8192, H=2048, V=151936, S=8, bf16). Inputs are
seeded and synthetic and already resident in HBM when the timed region starts;
W (622 MB) and the per-pass G chunks (256 MB) are larger than L2, so no extra
flush is done between steps.

Prints ONE JSON line (rank 0). `--impl reference` times the CPU oracle instead
(the slow fp64 definition, on the host cores, on a bounded token sample).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused vocab-CE fwd+bwd tokens/s & % BF16 TC peak; embed gather/bwd GB/s vs HBM"
WORKLOAD = "qwen3_tied"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of the loss path's
# tensor-core launches in one step of a workload, from one ncu capture whose
# summary is kept under profiles/. `source` is the sha256 prefix of the
# tensor-core kernel's source file that the capture ran: once that file has
# changed the figure is stale, and the line reports null until it is retaken.
MEASURED_TRAFFIC = {
    "qwen3_tied": {"bytes_per_step": 18608047360,
                   "per_kernel": {"tc_fwd": 942013952, "tc_grad": 3408379136, "tc_dh": 7139366400,
                                  "tc_dw": 7118287872},
                   "source": "b9152a7d87535d8d",
                   "profile": "profiles/tc_loss_kernel_qwen3_T8192.md"},
}
TC_SOURCE = os.path.join(ROOT, "vocab_embedding_cross_gb300", "csrc", "loss_tc.cu")


def measured_traffic(workload: str):
    """The captured loss-path traffic of `workload` if it belongs to the
    tensor-core kernel as it is now, else None."""
    import hashlib
    rec = MEASURED_TRAFFIC.get(workload)
    if rec is None:
        return None
    with open(TC_SOURCE, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    return rec if sha == rec["source"] else None


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return pk, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def arm_config(workload: str, world: int) -> dict:
    """The `config` object of the JSON line; both arms print the same one."""
    from vocab_embedding_cross_gb300 import inputs as I
    wl = I.WORKLOADS[workload]
    return {"workload": f"{workload}: T={wl.T} H={wl.H} V_real={wl.V_real} Vp={wl.Vp} S={wl.S} tied={wl.tied}",
            "step": "embed_fwd_plan (the lookup, beside the sort of the ids for the backward) + loss_fwd + "
                    "loss_bwd (writes the tied dW) + embed_bwd_apply (adds into it)",
            "l2": "inputs larger than L2 (W 622 MB, G chunks of 1.25 GB); no extra flush",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def max_over_ranks(ms: float, world: int, device="cuda") -> float:
    """The slowest replica's time per step: every rank gets the maximum over
    ranks (all-reduce MAX, then a barrier). One rank returns its own time."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_rank: int, world: int, ms: float) -> float:
    """Replicas: every rank processes its own batch, so the job's throughput is
    all ranks' tokens over the slowest rank's step time (weak scaling)."""
    return world * tokens_per_rank / (ms / 1e3)


class Clocks:
    """Samples nvidia-smi during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        import tempfile
        self.gpu = gpu_index
        self.proc = None
        # the raw samples are kept for inspection: VCE_CLOCK_LOG_DIR, else the temp dir
        log_dir = os.environ.get("VCE_CLOCK_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from vocab_embedding_cross_gb300 import _lib as vce
    if not os.path.exists(vce.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    from vocab_embedding_cross_gb300 import device as D
    from vocab_embedding_cross_gb300 import inputs as I

    wl = I.WORKLOADS[args.workload]
    # each replica draws its own batch (weak scaling); W is shared by seed
    t_gen = time.time()
    d = I.make_all(wl, ("W", "h", "targets", "ids", "dE"))
    gen_s = time.time() - t_gen
    T, H, Vp, V = wl.T, wl.H, wl.Vp, wl.V_real
    p = vce.problem(T, H, Vp, V, wl.S, vce.VCE_BF16, tied=wl.tied)
    # The tied gradient dW = dW_head + dW_embed is built in two calls: the
    # head's backward writes dW (the overwrite form of vce_loss_bwd, which
    # also zeroes the padded rows), and the embedding backward adds its rows.
    # No separate zeroing of the 1.24 GB buffer is needed.
    p_head = vce.problem(T, H, Vp, V, wl.S, vce.VCE_BF16, tied=False)
    W = D.to_device(d["W"])
    h = D.to_device(d["h"])
    ids = torch.from_numpy(d["ids"]).cuda()
    y = torch.from_numpy(d["targets"]).cuda()
    dE = D.to_device(d["dE"])
    E = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    loss = torch.empty(1, device="cuda")
    lse = torch.empty(T, device="cuda")
    dH = torch.empty((T, H), device="cuda")
    dW = torch.empty((Vp, H), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_f = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_LOSS_FWD))
    ws_b_bytes = vce.vce_workspace_size(p, vce.VCE_OP_LOSS_BWD)
    if args.bwd_cols:   # G chunk of that many columns plus the dH K-part partials
        ws_b_bytes = 256 + T * 2 * args.bwd_cols + (0 if args.no_dh_split else 8 * (-(-T // 256) * 256) * H * 4)
    ws_b = D.workspace(ws_b_bytes)
    ws_e = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_EMBED_BWD))
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    # The embedding backward's plan (the sort of the ids) is made at the lookup,
    # where the ids are known, beside the lookup's row copies; the backward
    # then only applies it to dE.
    def step_ops():
        vce.vce_embed_fwd_plan(p, ids, W, E, ws_e, dev_status=st, stream=sp)
        vce.vce_loss_fwd(p, h, W, y, loss, lse, ws=ws_f, dev_status=st, stream=sp)
        vce.vce_loss_bwd(p_head, h, W, y, lse, 1.0, dH, dW, ws_b, dev_status=st, stream=sp)
        vce.vce_embed_bwd_apply(p, dE, dW, ws_e, dev_status=st, stream=sp)

    def step():
        step_ops()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert int(st.item()) == 0, vce.status_str(int(st.item()))

    # ---- timed region: K steps, device resident ----
    clocks = Clocks(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    n0 = vce.vce_launch_count()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    launches = vce.vce_launch_count() - n0
    clk = clocks.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)
    value = whole_job_tokens_per_s(T, world, ms)

    # ---- per-launch timing: K more steps, right after the timed ones ----
    # Events after every launch. The pass follows the timed steps with no
    # pause, so that the kernels run in the same power-capped state (a cooled
    # GPU runs the first steps at a higher clock). A short spin kernel first
    # holds the stream so that the first launches are queued before the GPU
    # reaches them; later launches are queued far ahead of the GPU anyway.
    cap = 8192
    per_kind = {}
    reps = args.steps
    torch.cuda._sleep(2_000_000)
    vce.vce_profile_begin(cap, stream=sp)
    for _ in range(reps):
        step_ops()
    prof = vce.vce_profile_end(cap)
    for k, dt in prof:
        tot, n = per_kind.get(k, (0.0, 0))
        per_kind[k] = (tot + dt, n + 1)
    per_kind = {k: (tot / reps, n // reps) for k, (tot, n) in per_kind.items()}

    # ---- roofline: the loss path, credited 6*T*H*V_real FLOP ----
    # The headline fraction is the credited work of the loss forward and
    # backward (2*T*H*V_real each for the logits, dH and dW; the backward's
    # recompute of the logits is not credited) over the summed per-launch
    # times of the loss path's kernels, against the measured burst bf16 rate.
    # Each tensor-core mode's executed rate (2*T*H*V_real per step) is kept
    # beside it.
    peaks, peak_src = load_peaks()
    dh_part = 0 if args.no_dh_split else 8 * (-(-T // 256) * 256) * H * 4
    vc = min((ws_b_bytes - 256 - dh_part) // (T * 2), -(-V // 256) * 256)
    tc_kinds = ["tc_fwd", "tc_grad", "tc_dh", "tc_dw"]
    loss_kinds = tc_kinds + ["dh_reduce", "merge", "loss_mean", "count_valid"]
    loss_ms = sum(per_kind.get(k, (0.0, 0))[0] for k in loss_kinds)
    credited_flops = 6.0 * T * H * V
    roofline = None
    if loss_ms > 0:
        achieved = credited_flops / (loss_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        tr = measured_traffic(args.workload) if not (args.bwd_cols or args.no_dh_split) else None
        per_tc = {}
        for k in tc_kinds:
            if k in per_kind:
                tf = 2.0 * T * H * V / (per_kind[k][0] / 1e3) / 1e12
                per_tc[k] = {"ms_per_step": round(per_kind[k][0], 4), "launches_per_step": per_kind[k][1],
                             "executed_TFLOPs": round(tf, 1), "frac_of_burst": round(tf / peak, 4),
                             "frac_of_sustained": round(tf / peaks["bf16_tflops_sustained"], 4)}
        roofline = {"bound": "tensor", "kernel": "loss path: tc_loss_kernel FWD, GRAD, DH, DW and the merge, "
                                                "mean, valid-count and dH-part kernels",
                    "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                    "frac": round(achieved / peak, 4),
                    "traffic": tr["bytes_per_step"] if tr else None,
                    "traffic_unit": "bytes per step of the loss path's tensor-core launches "
                                    "(ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                    "traffic_source": (f"{tr['profile']} (tensor-core source sha256 {tr['source']})" if tr
                                       else "stale or not captured for this configuration"),
                    "credited_flops_per_step": credited_flops, "ms_per_step": round(loss_ms, 4),
                    "peak_kind": f"bf16_tflops burst ({peak_src})",
                    "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                    "per_kernel_executed": per_tc}
    credited = credited_flops
    loss_tflops = credited / (loss_ms / 1e3) / 1e12 if loss_ms else None
    valid = (d["ids"] >= 0) & (d["ids"] < V)
    U = int(np.unique(d["ids"][valid]).size)
    gather_bytes = 8 * T + U * H * 2 + T * H * 2
    bwd_bytes = 8 * T + T * H * 2 + U * H * 8
    emb = {}
    if "embed_gather" in per_kind:
        g_ms = per_kind["embed_gather"][0]
        emb["gather_GBps"] = round(gather_bytes / (g_ms / 1e3) / 1e9, 1)
        emb["gather_us"] = round(g_ms * 1e3, 2)
    if "embed_reduce" in per_kind:
        sorts = ("embed_sort", "embed_sort_cluster")
        b_ms = sum(per_kind.get(k, (0.0, 0))[0] for k in ("embed_hdr", "embed_reduce") + sorts)
        emb["bwd_GBps"] = round(bwd_bytes / (b_ms / 1e3) / 1e9, 1)
        emb["bwd_us"] = round(b_ms * 1e3, 2)
        emb["bwd_sort_us"] = round(sum(per_kind.get(k, (0.0, 0))[0] for k in sorts) * 1e3, 2)
        # the backward's own launch in the step: the plan's application (the plan
        # is made after the lookup)
        a_ms = per_kind["embed_reduce"][0]
        emb["bwd_apply_GBps"] = round(bwd_bytes / (a_ms / 1e3) / 1e9, 1)
        emb["bwd_apply_us"] = round(a_ms * 1e3, 2)
    emb["hbm_peak_GBps"] = peaks["hbm_gbs"]
    for k in ("gather", "bwd", "bwd_apply"):
        if f"{k}_GBps" in emb:
            emb[f"{k}_frac"] = round(emb[f"{k}_GBps"] / peaks["hbm_gbs"], 4)

    # ---- the head backward in its tied (+=) form at this size ----
    tied_flag = run_tied_flag(args, vce, p, p_head, h, W, y, lse, dH, dW, ws_b, stream)

    # ---- end to end through the C ABI with host buffers ----
    e2e = run_e2e(args, vce, D, d, p, p_head, W, E, loss, lse, dH, dW, st, ws_f, ws_b, ws_e, stream, wl)
    # the library's launches made by each leg, in order (they split a profiler's launch list)
    leg_marks = [("step", vce.vce_launch_count())]

    # ---- the embedding on the GPT-OSS-shaped table ----
    emb_gptoss = run_embedding(args, vce, D, I, stream, peaks, "gptoss_embed")
    leg_marks.append(("embedding_gptoss", vce.vce_launch_count()))
    # the main workload's lookup and backward, each call timed alone the same way
    # (the figures above come from the step's per-launch events)
    emb["isolated"] = {k: v for k, v in run_embedding(args, vce, D, I, stream, peaks, args.workload).items()
                       if k != "workload"}
    leg_marks.append(("embedding_isolated", vce.vce_launch_count()))

    # ---- greedy argmax over the same head (decoding), device resident ----
    greedy = run_greedy(args, vce, D, p, h, W, stream, T, H, V, peaks)
    leg_marks.append(("greedy_argmax", vce.vce_launch_count()))

    # ---- the OT-H auxiliary head on the same workload ----
    oth = run_oth(args, vce, D, p, h, W, y, stream, T, H, Vp, V, wl.S, peaks)
    leg_marks.append(("oth_head", vce.vce_launch_count()))

    # ---- the loss alone on the GPT-2-like head and on the GPT-OSS shapes ----
    loss_configs = {name: run_loss_config(args, vce, D, I, stream, peaks, name)
                    for name in ("gpt2_head", "gptoss_embed")}
    leg_marks.append(("loss_configs", vce.vce_launch_count()))

    # ---- hashed n-gram input embeddings on the same ids ----
    ngram = run_ngram(args, vce, D, I, wl, d, p, W, dE, stream, peaks)
    leg_marks.append(("ngram_embedding", vce.vce_launch_count()))

    # ---- sampled-softmax variant, against the full-vocabulary loss ----
    sampled = run_sampled(args, vce, D, I, stream, peaks, full_loss_tok_s=T / (loss_ms / 1e3) if loss_ms else None)
    leg_marks.append(("sampled_softmax", vce.vce_launch_count()))
    leg_launches = {name: n - (leg_marks[i - 1][1] if i else 0) for i, (name, n) in enumerate(leg_marks)}

    # ---- CPU baseline (rank 0, N = 1 only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args, sample_tokens=args.cpu_sample)
        # one-thread figures on the small configurations: the whole fp32 case, and
        # a 64-token sample of the GPT-2-like head
        cpu["one_thread"] = {w: cpu_baseline(args, sample_tokens=n, threads=1, workload=w)
                             for w, n in (("tiny_f32", 64), ("gpt2_head", 64))}
        # every core, per operation, on the other loss configurations
        cpu["configs"] = {w: cpu_baseline(args, sample_tokens=n, workload=w)
                          for w, n in (("tiny_f32", 64), ("gpt2_head", 128), ("gptoss_embed", 128))}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; Zipf(1.1) token ids, RMS-normalised h, W ~ N(0, 0.02^2))",
            "config": arm_config(args.workload, world),
            "roofline": roofline,
            "per_launch_sum_ms": round(sum(v[0] for v in per_kind.values()), 4),
            "step_credited_frac_of_burst": round(credited / (ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
            "loss_fwd_bwd": {"ms": round(loss_ms, 4), "credited_flops": credited,
                             "credited_TFLOPs": round(loss_tflops, 1) if loss_tflops else None,
                             "frac_of_burst": round(loss_tflops / peaks["bf16_tflops"], 4) if loss_tflops else None,
                             "frac_of_sustained": round(loss_tflops / peaks["bf16_tflops_sustained"], 4)
                             if loss_tflops else None,
                             "executed_flops": 8.0 * T * H * V, "vc": int(vc)},
            "head_bwd_tied_flag": tied_flag,
            "embedding": emb,
            "sampled_softmax": sampled,
            "embedding_gptoss": emb_gptoss,
            "greedy_argmax": greedy,
            "loss_configs": loss_configs,
            "oth_head": oth,
            "ngram_embedding": ngram,
            "per_kernel_ms": {k: round(v[0], 4) for k, v in sorted(per_kind.items())},
            "per_kernel_launches": {k: v[1] for k, v in sorted(per_kind.items())},
            "gpu_launches": int(launches),
            "leg_launches": leg_launches,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "input_gen_s": round(gen_s, 1),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_tied_flag(args, vce, p, p_head, h, W, y, lse, dH, dW, ws_b, stream):
    """vce_loss_bwd with tied_weights = 1 (dW += G^T h, a TMA reduce-add into
    the fp32 gradient) against the overwrite form the step uses (the head's
    dW written, then the embedding's rows added), on the main workload. A
    caller of the tied form zeroes dW once per step; that fill is timed too."""
    import torch
    sp = stream.cuda_stream
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def timed(fn, n):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    n = max(3, args.steps // 4)
    ow = timed(lambda: vce.vce_loss_bwd(p_head, h, W, y, lse, 1.0, dH, dW, ws_b, dev_status=st, stream=sp), n)
    acc = timed(lambda: vce.vce_loss_bwd(p, h, W, y, lse, 1.0, dH, dW, ws_b, dev_status=st, stream=sp), n)
    zero = timed(lambda: dW.zero_(), n)
    assert int(st.item()) == 0, vce.status_str(int(st.item()))
    return {"overwrite_ms": round(ow, 4), "accumulate_ms": round(acc, 4), "dW_zero_ms": round(zero, 4),
            "calls": n}


def run_greedy(args, vce, D, p, h, W, stream, T, H, V, peaks):
    """vce_greedy_argmax on the main workload's h and W (T tokens, all V
    classes, S shards): tokens/s and the logit GEMM's TFLOP/s (2*T*H*V)."""
    import torch
    arg = torch.empty(T, dtype=torch.int64, device="cuda")
    ws = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_GREEDY_ARGMAX))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sp = stream.cuda_stream
    for _ in range(3):
        vce.vce_greedy_argmax(p, h, W, arg, ws=ws, dev_status=st, stream=sp)
    torch.cuda.synchronize()
    n = max(5, args.steps // 4)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        vce.vce_greedy_argmax(p, h, W, arg, ws=ws, dev_status=st, stream=sp)
    e1.record(stream)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, vce.status_str(int(st.item()))
    ms = e0.elapsed_time(e1) / n
    tf = 2.0 * T * H * V / (ms / 1e3) / 1e12
    return {"tokens_per_s": round(T / (ms / 1e3), 1), "ms_per_call": round(ms, 4), "calls": n,
            "TFLOPs": round(tf, 1), "frac_of_burst": round(tf / peaks["bf16_tflops"], 4)}


def run_oth(args, vce, D, p, h, W, y, stream, T, H, Vp, V, S, peaks):
    """The OT-H auxiliary head on the main workload: head one scores h on the
    next tokens, head two (its own weights W2, here a copy of W) scores h[:-1]
    on the tokens two ahead at weight 0.1 and adds its dH into head one's
    (VCE_FLAG_ACCUMULATE_DH). One step is both heads' forward and backward;
    the plain head's forward and backward is timed beside it."""
    import torch
    W2 = W.clone()
    y2 = y[1:]
    p1 = vce.problem(T, H, Vp, V, S, vce.VCE_BF16)
    p2 = vce.problem(T - 1, H, Vp, V, S, vce.VCE_BF16)
    p2_acc = vce.problem(T - 1, H, Vp, V, S, vce.VCE_BF16, flags=vce.VCE_FLAG_ACCUMULATE_DH)
    loss1 = torch.empty(1, device="cuda")
    loss2 = torch.empty(1, device="cuda")
    lse1 = torch.empty(T, device="cuda")
    lse2 = torch.empty(T - 1, device="cuda")
    dH = torch.empty((T, H), device="cuda")
    dW1 = torch.empty((Vp, H), device="cuda")
    dW2 = torch.empty((Vp, H), device="cuda")
    ws_f = D.workspace(vce.vce_workspace_size(p1, vce.VCE_OP_LOSS_FWD))
    ws_b = D.workspace(vce.vce_workspace_size(p1, vce.VCE_OP_LOSS_BWD))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sp = stream.cuda_stream

    def one_head():
        vce.vce_loss_fwd(p1, h, W, y, loss1, lse1, ws=ws_f, dev_status=st, stream=sp)
        vce.vce_loss_bwd(p1, h, W, y, lse1, 1.0, dH, dW1, ws_b, dev_status=st, stream=sp)

    def two_heads():
        one_head()
        vce.vce_loss_fwd(p2, h, W2, y2, loss2, lse2, ws=ws_f, dev_status=st, stream=sp)
        vce.vce_loss_bwd(p2_acc, h, W2, y2, lse2, 0.1, dH, dW2, ws_b, dev_status=st, stream=sp)

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    n = max(3, args.steps // 4)
    ms1 = timed(one_head, n)
    ms2 = timed(two_heads, n)
    assert int(st.item()) == 0, vce.status_str(int(st.item()))
    del W2, dW1, dW2, ws_f, ws_b
    torch.cuda.empty_cache()
    return {"step": "head one fwd+bwd, head two (T-1 rows, weight 0.1) fwd+bwd adding into dH",
            "ms_per_step": round(ms2, 4), "tokens_per_s": round(T / (ms2 / 1e3), 1),
            "one_head_ms": round(ms1, 4), "ratio_to_one_head": round(ms2 / ms1, 4), "steps": n}


def run_loss_config(args, vce, D, I, stream, peaks, name):
    """Loss forward + backward alone on another configuration's shapes (inputs
    resident in HBM, larger than L2): tokens/s and 6*T*H*V_real credited FLOP
    over the measured time, against the bf16 peaks."""
    import torch
    wl = I.WORKLOADS[name]
    d = I.make_all(wl, ("W", "h", "targets"))
    T, H, V = wl.T, wl.H, wl.V_real
    p = vce.problem(T, H, wl.Vp, V, wl.S, vce.VCE_BF16)
    W, h = D.to_device(d["W"]), D.to_device(d["h"])
    y = torch.from_numpy(d["targets"]).cuda()
    loss = torch.empty(1, device="cuda")
    lse = torch.empty(T, device="cuda")
    dH = torch.empty((T, H), device="cuda")
    dW = torch.empty((wl.Vp, H), device="cuda")
    ws_f = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_LOSS_FWD))
    ws_b = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_LOSS_BWD))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sp = stream.cuda_stream

    def step():
        vce.vce_loss_fwd(p, h, W, y, loss, lse, ws=ws_f, dev_status=st, stream=sp)
        vce.vce_loss_bwd(p, h, W, y, lse, 1.0, dH, dW, ws_b, dev_status=st, stream=sp)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    n = max(5, args.steps // 4)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, vce.status_str(int(st.item()))
    ms = e0.elapsed_time(e1) / n
    tf = 6.0 * T * H * V / (ms / 1e3) / 1e12
    del W, h, dH, dW, ws_f, ws_b
    torch.cuda.empty_cache()
    return {"workload": f"{name}: T={T} H={H} V_real={V} Vp={wl.Vp} S={wl.S} bf16 untied",
            "tokens_per_s": round(T / (ms / 1e3), 1), "ms_per_step": round(ms, 4), "steps": n,
            "credited_TFLOPs": round(tf, 1), "frac_of_burst": round(tf / peaks["bf16_tflops"], 4),
            "frac_of_sustained": round(tf / peaks["bf16_tflops_sustained"], 4)}


def run_embedding(args, vce, D, I, stream, peaks, name):
    """Masked lookup and deterministic backward on a named workload (the
    GPT-OSS-shaped table [201088, 3072] with T=16384 Zipf ids, 2% padding and
    1% out-of-range ids; or the main workload's): microseconds per call and
    GB/s of the algorithmic bytes (ids, the distinct valid rows read, E
    written; dE read, touched dW rows read-modify-written in fp32).

    L2 is flushed before every call by writing a 256 MB buffer. The headline
    figures then read another 256 MB buffer, so that the L2 holds clean lines
    and the timed call is not charged for writing back the flush buffer's dirty
    lines; the `*_dirty_l2` figures skip that read.

    `bwd_*` is the one-call backward (vce_embed_bwd: the sort of the ids, then
    the addition of dE into dW); `bwd_plan_us` the sort alone
    (vce_embed_bwd_plan); `gather_with_plan_*` the lookup with the plan made
    beside it (vce_embed_fwd_plan), credited with the lookup's bytes;
    `bwd_apply_*` the addition by a plan made earlier (vce_embed_bwd_apply),
    which is all the backward runs once the plan is made at the lookup, and
    which moves all of the backward's bytes."""
    import torch
    wl = I.WORKLOADS[name]
    d = I.make_all(wl, ("W", "ids", "dE"))
    T, H = wl.T, wl.H
    p = vce.problem(T, H, wl.Vp, wl.V_real, wl.S, vce.VCE_BF16)
    W, dE = D.to_device(d["W"]), D.to_device(d["dE"])
    ids = torch.from_numpy(d["ids"]).cuda()
    E = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    dW = torch.zeros((wl.Vp, H), device="cuda")
    ws = D.workspace(vce.vce_workspace_size(p, vce.VCE_OP_EMBED_BWD))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sp = stream.cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    clean = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")
    valid = (d["ids"] >= 0) & (d["ids"] < wl.V_real)
    import numpy as np
    U = int(np.unique(d["ids"][valid]).size)
    gather_bytes = 8 * T + U * H * 2 + T * H * 2
    bwd_bytes = 8 * T + T * H * 2 + U * H * 8
    logical_bytes = 8 * T + int(valid.sum()) * H * 2 + T * H * 2

    def timed(fn, n, clean_l2=True):
        tot = 0.0
        for i in range(n + 3):
            flush.zero_()
            if clean_l2:
                torch.sum(clean.view(torch.int32), dtype=torch.int64)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                tot += e0.elapsed_time(e1)
        return tot / n

    n = max(10, args.steps // 2)
    fwd = lambda: vce.vce_embed_fwd(p, ids, W, E, dev_status=st, stream=sp)
    bwd = lambda: vce.vce_embed_bwd(p, ids, dE, dW, ws, dev_status=st, stream=sp)
    plan = lambda: vce.vce_embed_bwd_plan(p, ids, ws, dev_status=st, stream=sp)
    apply = lambda: vce.vce_embed_bwd_apply(p, dE, dW, ws, dev_status=st, stream=sp)
    fwd_plan = lambda: vce.vce_embed_fwd_plan(p, ids, W, E, ws, dev_status=st, stream=sp)
    g_ms, b_ms = timed(fwd, n), timed(bwd, n)
    g_dirty, b_dirty = timed(fwd, n, clean_l2=False), timed(bwd, n, clean_l2=False)
    # The backward split at its plan: the sort of the ids alone, the lookup
    # with the plan made beside it, then the application of the plan to dE (the
    # workspace holds the plan of these ids, and every application leaves it in
    # place).
    plan_ms = timed(plan, n)
    gp_ms = timed(fwd_plan, n)
    a_ms, a_dirty = timed(apply, n), timed(apply, n, clean_l2=False)
    assert int(st.item()) == 0, vce.status_str(int(st.item()))
    del W, dE, E, dW, ws, flush, clean
    torch.cuda.empty_cache()
    frac = lambda b, ms: round(b / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)
    return {"workload": f"{name}: W[{wl.Vp},{H}] bf16, T={T} Zipf(1.1) ids, {100 * wl.pad_id_frac:g}% padding id, "
                        f"{100 * wl.oor_id_frac:g}% out of range, {U} distinct valid rows",
            "l2": "flushed before every call: a 256 MB write, then a 256 MB read of another buffer (clean lines); "
                  "*_dirty_l2: the write alone",
            "gather_us": round(g_ms * 1e3, 2), "gather_GBps": round(gather_bytes / (g_ms / 1e3) / 1e9, 1),
            "gather_frac": frac(gather_bytes, g_ms),
            "bwd_us": round(b_ms * 1e3, 2), "bwd_GBps": round(bwd_bytes / (b_ms / 1e3) / 1e9, 1),
            "bwd_frac": frac(bwd_bytes, b_ms),
            "gather_us_dirty_l2": round(g_dirty * 1e3, 2), "gather_frac_dirty_l2": frac(gather_bytes, g_dirty),
            "bwd_us_dirty_l2": round(b_dirty * 1e3, 2), "bwd_frac_dirty_l2": frac(bwd_bytes, b_dirty),
            "bwd_plan_us": round(plan_ms * 1e3, 2),
            "gather_with_plan_us": round(gp_ms * 1e3, 2), "gather_with_plan_frac": frac(gather_bytes, gp_ms),
            "bwd_apply_us": round(a_ms * 1e3, 2), "bwd_apply_GBps": round(bwd_bytes / (a_ms / 1e3) / 1e9, 1),
            "bwd_apply_frac": frac(bwd_bytes, a_ms),
            "bwd_apply_us_dirty_l2": round(a_dirty * 1e3, 2), "bwd_apply_frac_dirty_l2": frac(bwd_bytes, a_dirty),
            "gather_bytes": gather_bytes, "bwd_bytes": bwd_bytes,
            # every valid row counted as read (repeats hit L2), and the nominal 8 TB/s HBM3e
            "gather_logical_bytes": logical_bytes,
            "gather_frac_of_8TBps": round(gather_bytes / (g_ms / 1e3) / 8e12, 4),
            "bwd_frac_of_8TBps": round(bwd_bytes / (b_ms / 1e3) / 8e12, 4)}


def run_ngram(args, vce, D, I, wl, d, p, W, dE, stream, peaks):
    """vce_ngram_embed_fwd / _bwd on the main workload's ids (4 sequences of
    2048) with two hashed tables of 2^18 rows: time per call and GB/s of the
    algorithmic bytes (ids, distinct rows read, E written; dE read once per
    table, touched rows read-modify-written in fp32). The backward is also
    timed in its two parts: the plan (vce_ngram_embed_bwd_plan) and its
    application (vce_ngram_embed_bwd_apply), which moves all of its bytes."""
    import torch
    M, L = I.NGRAM_ROWS, I.NGRAM_SEQ_LEN
    T, H = wl.T, wl.H
    T2 = D.to_device(I.make_ngram_table(wl, 2, M))
    T3 = D.to_device(I.make_ngram_table(wl, 3, M))
    ids = torch.from_numpy(d["ids"]).cuda()
    E = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    dW = torch.zeros((wl.Vp, H), device="cuda")
    dT2 = torch.zeros((M, H), device="cuda")
    dT3 = torch.zeros((M, H), device="cuda")
    ws = D.workspace(vce.vce_ngram_workspace_size(p))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sp = stream.cuda_stream
    idx = torch.empty(T, dtype=torch.int64, device="cuda")
    uniq = []
    for n, Mn in ((1, wl.V_real), (2, M), (3, M)):
        vce.vce_ngram_hash(ids, n, wl.V_real, Mn, idx, seq_len=L, stream=sp)
        uniq.append(int(torch.unique(idx[idx >= 0]).numel()))
    fwd_bytes = 8 * T + sum(uniq) * H * 2 + T * H * 2
    bwd_bytes = 8 * T + 3 * T * H * 2 + sum(uniq) * H * 8

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    n = max(10, args.steps)
    f_ms = timed(lambda: vce.vce_ngram_embed_fwd(p, ids, W, T2, M, T3, M, E, seq_len=L, dev_status=st, stream=sp), n)
    b_ms = timed(lambda: vce.vce_ngram_embed_bwd(p, ids, dE, dW, dT2, M, dT3, M, ws, seq_len=L, dev_status=st,
                                                 stream=sp), n)
    # the backward split at its plan (row indices and the three sorts), then
    # the application alone (the workspace keeps the plan of these ids)
    pl_ms = timed(lambda: vce.vce_ngram_embed_bwd_plan(p, ids, M, M, ws, seq_len=L, dev_status=st, stream=sp), n)
    a_ms = timed(lambda: vce.vce_ngram_embed_bwd_apply(p, dE, dW, dT2, M, dT3, M, ws, dev_status=st, stream=sp), n)
    assert int(st.item()) == 0, vce.status_str(int(st.item()))
    del T2, T3, dT2, dT3, dW, ws
    torch.cuda.empty_cache()
    return {"workload": f"ids of {wl.name} (T={T}, sequences of {L}), H={H}, tables V={wl.V_real}, 2^18, 2^18",
            "distinct_rows": uniq, "fwd_us": round(f_ms * 1e3, 2),
            "fwd_GBps": round(fwd_bytes / (f_ms / 1e3) / 1e9, 1),
            "fwd_frac": round(fwd_bytes / (f_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
            "bwd_us": round(b_ms * 1e3, 2), "bwd_GBps": round(bwd_bytes / (b_ms / 1e3) / 1e9, 1),
            "bwd_frac": round(bwd_bytes / (b_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
            "bwd_plan_us": round(pl_ms * 1e3, 2),
            "bwd_apply_us": round(a_ms * 1e3, 2), "bwd_apply_GBps": round(bwd_bytes / (a_ms / 1e3) / 1e9, 1),
            "bwd_apply_frac": round(bwd_bytes / (a_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)}


def run_sampled(args, vce, D, I, stream, peaks, full_loss_tok_s):
    """The sampled-softmax loss step (T=16384, H=2048, V=151936, P=8192
    candidates: candidate list, gather of W[cand], cross-entropy over the
    candidates forward and backward, scatter of dW into the candidate rows),
    one vce_sampled_loss call per step, device resident, timed like the main
    step; compared with the full-vocabulary loss fwd+bwd of the main workload."""
    import torch
    wl = I.WORKLOADS["sampled"]
    P = I.SAMPLED_P
    d = I.make_all(wl, ("W", "h", "targets"))
    T, H = wl.T, wl.H
    p = vce.problem(T, H, wl.Vp, wl.V_real, wl.S, vce.VCE_BF16)
    W, h = D.to_device(d["W"]), D.to_device(d["h"])
    y = torch.from_numpy(d["targets"]).cuda()
    draws = torch.from_numpy(I.make_negative_draws(wl, P)).cuda()
    loss = torch.empty(1, device="cuda")
    dH = torch.empty((T, H), device="cuda")
    dW = torch.zeros((wl.Vp, H), device="cuda")
    cand = torch.empty(P, dtype=torch.int64, device="cuda")
    pos = torch.empty(T, dtype=torch.int64, device="cuda")
    nu = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = D.workspace(vce.vce_sampled_workspace_size(p, P))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sp = stream.cuda_stream

    def step():
        vce.vce_sampled_loss(p, h, W, y, draws, P, 1.0, loss, None, dH, dW, cand, pos, nu, ws, dev_status=st,
                             stream=sp)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert int(st.item()) == 0, vce.status_str(int(st.item()))
    n = max(5, args.steps // 2)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    torch.cuda._sleep(100_000_000)
    vce.vce_profile_begin(1024, stream=sp)
    for _ in range(3):
        step()
    per = {}
    for k, dt in vce.vce_profile_end(1024):
        per[k] = per.get(k, 0.0) + dt / 3
    tok_s = T / (ms / 1e3)
    credited = 6.0 * T * H * P
    out = {"workload": f"sampled: T={T} H={H} V={wl.V_real} P={P} S={wl.S} untied, Zipf(1.1) targets",
           "step": "vce_sampled_loss (candidates + gather + CE fwd/bwd over P + dW scatter)",
           "tokens_per_s": round(tok_s, 1), "ms_per_step": round(ms, 4), "steps": n,
           "n_unique_targets": int(nu.item()),
           "credited_TFLOPs": round(credited / (ms / 1e3) / 1e12, 1),
           "frac_of_burst": round(credited / (ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
           "per_kernel_ms": {k: round(v, 4) for k, v in sorted(per.items())},
           "full_vocab_loss_tokens_per_s": round(full_loss_tok_s, 1) if full_loss_tok_s else None,
           "speedup_vs_full_vocab_loss": round(tok_s / full_loss_tok_s, 3) if full_loss_tok_s else None}
    del W, h, dW, dH, ws
    torch.cuda.empty_cache()
    return out


def run_e2e(args, vce, D, d, p, p_head, W, E, loss, lse, dH, dW, st, ws_f, ws_b, ws_e, stream, wl):
    """The same step through the C ABI with every step's inputs (ids, targets,
    h, dE) copied from pinned host memory and its loss read back. The copies
    run on a second stream into two alternating sets of device buffers, so the
    copy of step i+1's inputs overlaps step i's kernels; every copy and every
    read-back lies inside the timed region."""
    import torch
    sp = stream.cuda_stream
    host = {k: D.to_device(d[k], device="cpu") if k in ("h", "dE") else torch.from_numpy(d[k])
            for k in ("ids", "targets", "h", "dE")}
    host = {k: v.pin_memory() for k, v in host.items()}
    dev = [{k: torch.empty_like(v, device="cuda") for k, v in host.items()} for _ in range(2)]
    loss_h = torch.empty(1, dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    cs = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        b = i % 2
        cs.wait_event(used[b])          # the step that last read these buffers is done
        with torch.cuda.stream(cs):
            for k in host:
                dev[b][k].copy_(host[k], non_blocking=True)
            ready[b].record(cs)

    def compute(i):
        b = i % 2
        stream.wait_event(ready[b])
        x = dev[b]
        vce.vce_embed_fwd_plan(p, x["ids"], W, E, ws_e, dev_status=st, stream=sp)
        vce.vce_loss_fwd(p, x["h"], W, x["targets"], loss, lse, ws=ws_f, dev_status=st, stream=sp)
        vce.vce_loss_bwd(p_head, x["h"], W, x["targets"], lse, 1.0, dH, dW, ws_b, dev_status=st, stream=sp)
        vce.vce_embed_bwd_apply(p, x["dE"], dW, ws_e, dev_status=st, stream=sp)
        used[b].record(stream)
        loss_h.copy_(loss, non_blocking=True)

    def run(n):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            compute(i)

    for e in used:
        e.record(stream)
    run(max(1, args.warmup))
    torch.cuda.synchronize()
    n = max(3, args.steps // 2)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    cs.wait_event(e0)
    for e in used:
        e.record(stream)
    run(n)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t0) / n
    ms = e0.elapsed_time(e1) / n
    return {"value": round(wl.T / (max(ms, wall * 1e3) / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 4, "ms_per_step": round(max(ms, wall * 1e3), 4),
            "copies": "pinned host -> device on a second stream, double-buffered, overlapping the previous step"}


# ---------------------------------------------------------------------------
# CPU oracle (bench's cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def cpu_baseline(args, sample_tokens, steps=1, warmup=0, threads=None, workload=None):
    """Runs the oracle in a child process with an explicit BLAS thread count
    (every core the process may use, unless `threads` is given): `warmup`
    untimed steps, then `steps` timed ones, each on the same sample."""
    cores = threads or len(os.sched_getaffinity(0))
    env = dict(os.environ, OMP_NUM_THREADS=str(cores), OPENBLAS_NUM_THREADS=str(cores),
               MKL_NUM_THREADS=str(cores))
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-child", "--workload", workload or args.workload,
           "--cpu-sample", str(sample_tokens), "--steps", str(steps), "--warmup", str(warmup)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=1800)
    try:
        out = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception:
        return {"value": None, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                "sample": f"failed: {r.stderr[-300:]}"}
    out["cores"] = cores
    return out


def oracle_child(args):
    import numpy as np
    from oracle import vce_oracle as O
    from vocab_embedding_cross_gb300 import inputs as I

    wl = I.WORKLOADS[args.workload]
    d = I.make_all(wl, ("W", "h", "targets", "ids", "dE"))
    n = min(args.cpu_sample, wl.T)
    # a bounded sample of the workload: the first n tokens, full vocabulary and hidden size
    h, y, ids, dE = d["h"][:n], d["targets"][:n], d["ids"][:n], d["dE"][:n]
    ops = {
        "embed_fwd": lambda: O.embed_forward(ids, d["W"], wl.V_real),
        "loss_fwd": lambda: O.cross_entropy_forward(h, d["W"], y, wl.V_real),
        "loss_bwd": lambda: O.cross_entropy_backward(h, d["W"], y, wl.V_real, wl.Vp),
        "embed_bwd": lambda: O.embed_backward(ids, dE, wl.V_real, wl.Vp),
    }

    for _ in range(max(0, args.warmup)):
        for fn in ops.values():
            fn()
    steps = max(1, args.steps)
    per_op = {k: 0.0 for k in ops}
    for _ in range(steps):
        for k, fn in ops.items():   # one step: the four calls in the path's order, each timed
            t0 = time.perf_counter()
            fn()
            per_op[k] += time.perf_counter() - t0
    per_op = {k: v / steps for k, v in per_op.items()}
    t = sum(per_op.values())
    print(json.dumps({"value": round(n / t, 3), "unit": "tokens/s", "kind": "oracle",
                      "sample": f"first {n} of {wl.T} tokens of {args.workload}, full V={wl.V_real} and "
                                f"H={wl.H}; embed fwd + loss fwd + loss bwd + embed bwd in fp64 numpy",
                      "seconds": round(t, 3), "steps": steps,
                      "per_op": {k: {"seconds": round(v, 4), "tokens_per_s": round(n / v, 3) if v > 0 else None}
                                 for k, v in per_op.items()}}))


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    cores = len(os.sched_getaffinity(0))
    res = cpu_baseline(argparse.Namespace(workload=args.workload), sample_tokens=args.cpu_sample,
                       steps=args.steps, warmup=args.warmup)
    secs = res.get("seconds")
    line = {"impl": "reference", "metric": METRIC, "value": res.get("value"), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs * 1e3, 1) if secs else None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": arm_config(args.workload, world),
            "cpu_baseline": {"value": res.get("value"), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": res.get("sample")},
            "e2e": {"value": res.get("value"), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--cpu-sample", type=int, default=128)
    ap.add_argument("--no-dh-split", action="store_true", help="with --bwd-cols: no room for dH K parts")
    ap.add_argument("--bwd-cols", type=int, default=0,
                    help="vocabulary columns per backward pass (sizes the workspace); 0 = library default")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-child", action="store_true")
    args = ap.parse_args()
    if args.oracle_child:
        oracle_child(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
