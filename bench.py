"""Benchmark: causal attention forward + backward TFLOP/s on one GB300.

One step = dfa_attn_fwd followed by dfa_attn_bwd (from the saved O and lse)
over one batch of seeded synthetic inputs of the chosen workload (default:
the Llama-7B attention shape at 128K tokens, bf16).  FLOPs are algorithmic
causal FLOPs: pairs = B*H*S(S+1)/2, 4D per pair forward and 10D per pair
backward (P is recomputed from the saved lse), 14D per pair in total.

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on a bounded sample of the same workload instead.

Multi-GPU (torchrun): the path does not exchange data between GPUs; each rank
runs its own batch of the workload (weak scaling) and the slowest rank's time
is reported.
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

NOMINAL_BF16_TFLOPS = 2250.0
DEFAULT_WORKLOAD = "llama7b_s128k"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["dfa", "reference"], default="dfa")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--shape", default=None,
                    help="B,H,H_kv,S,D: a custom bf16 shape instead of a named workload (profiling cases)")
    ap.add_argument("--sched", choices=["balanced", "unbalanced", "split_kv"], default="balanced")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-chunk-step", action="store_true", help="skip the per-worker chunk-step timing")
    ap.add_argument("--window", type=int, default=2, help="chunks per local window for the extra local-window timing (0: skip)")
    ap.add_argument("--no-varlen", action="store_true", help="skip the packed-batch timing")
    ap.add_argument("--no-split-kv", action="store_true", help="skip the small-problem split-kv forward timing")
    ap.add_argument("--cpu-seconds", type=float, default=8.0, help="target oracle sample time")
    ap.add_argument("--no-unbalanced", action="store_true", help="skip the unbalanced work-list timing")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the timing of the other Llama-7B workloads (32K, GQA 64K, 512K)")
    return ap.parse_args()


# DRAM bytes (read + write) of one launch of the backward kernel, measured by
# ncu on one launch of the 32K Llama-7B workload (one kernel, one launch, a few
# GB on the device), and the forward kernel's the same way.  A larger workload
# of the same head shape is scaled by its ratio of causal (query, key) pairs:
# an estimate, because how much of the fp32 dQ accumulator stays in L2 changes
# with the size.  Valid only for the kernel builds they were taken on.
NCU_TRAFFIC_REF = {"workload": "llama7b_s32k", "bwd": 1.6716e9 + 1.0668e9, "fwd": 0.8989e9 + 0.2509e9}


def config_of(w, sched):
    """The `config` object of both arms' JSON lines (the same for the same workload)."""
    return {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.H_kv, "S": w.S, "D": w.D,
            "n_chunks": w.n_chunks, "sched": sched, "causal": True,
            "l2": "inputs larger than L2 (each tensor exceeds 129 MB)"}


def scaled_traffic(w, kernel):
    """DRAM bytes per launch of `kernel` ("bwd" or "fwd") for workload w, scaled
    from the single-launch capture of NCU_TRAFFIC_REF, or None."""
    from long_context_causal_gb300.inputs import WORKLOADS
    measured = NCU_TRAFFIC_REF[kernel]
    ref = WORKLOADS[NCU_TRAFFIC_REF["workload"]]
    if measured is None or w.D != ref.D or w.H // w.H_kv != ref.H // ref.H_kv:
        return None
    return measured * w.causal_flops() / ref.causal_flops()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower().startswith("active")})
        pw = []
        for r in self.rows:
            try:
                pw.append(float(r[3]))
            except ValueError:
                pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows),
                "power_w": statistics.median(pw) if pw else None}


def dist_setup(n_gpus, backend="nccl"):
    """One process per GPU (torchrun sets RANK/LOCAL_RANK/WORLD_SIZE/MASTER_*).
    backend "gloo" runs the same rank logic on CPU (tests)."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    elif backend == "nccl":
        torch.cuda.set_device(0)
    return rank, world, local


def rank_seed(base_seed, rank):
    """Weak scaling: every rank draws its own independent copy of the workload."""
    return base_seed + rank


def job_value(flops_per_rank, ms_per_step, world):
    """Whole-job throughput (TFLOP/s): all ranks' work over the slowest rank's time."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- CPU oracle sample
def oracle_sample(w, seconds, seed=0):
    """Times the fp64 oracle on sampled query rows of workload `w`.

    Returns (flops, elapsed_s, cores, description).  Each sampled row gets its
    forward (O, lse: 4D FLOPs per visible key) and its dQ (recomputed scores,
    dP and dQ: 6D per visible key)."""
    import numpy as np
    import torch

    import oracle
    from long_context_causal_gb300.inputs import make

    # Inputs of one (batch, head) pair drawn with the workload's recipe; the
    # oracle needs keys up to the sampled row only.
    rng = np.random.default_rng(seed)
    Hs = 1
    Skv = w.S
    q, k, v, do = make(1, Hs, 1, Skv, w.D, w.dtype, seed=w.seed, device="cpu", k_scale=w.k_scale)
    f = lambda t: t.float().numpy().astype(np.float64)
    q, k, v, do = f(q), f(k), f(v), f(do)
    cores = oracle.num_threads()
    # Calibrate: rows of average length S/2 cost ~10*D*S/2 FLOPs; aim for `seconds`.
    rows_done, flops, elapsed = 0, 0.0, 0.0
    batch = max(cores, 8)
    while elapsed < seconds:
        rows = np.sort(rng.integers(0, w.S, size=batch))
        idx = np.stack([np.zeros_like(rows), np.zeros_like(rows), rows], axis=1)
        t0 = time.perf_counter()
        oracle.attn_fwd_rows(q, k, v, idx, scale=w.scale)
        oracle.attn_dq_rows(q, k, v, do, idx, scale=w.scale)
        elapsed += time.perf_counter() - t0
        flops += float(np.sum(rows + 1)) * w.D * 10
        rows_done += batch
    desc = (f"{rows_done} random query rows of one head of {w.name} (S={w.S}, D={w.D}); "
            f"forward O/lse and dQ per row in fp64")
    return flops, elapsed, cores, desc


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per_step = max(1.0, min(args.cpu_seconds, 180.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, per_step / 4, seed=1)
    tot_f, tot_t, cores, desc = 0.0, 0.0, 1, ""
    for s in range(args.steps):
        fl, el, cores, desc = oracle_sample(w, per_step, seed=100 + s)
        tot_f += fl
        tot_t += el
    val = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": "causal attn fwd+bwd TFLOP/s (bf16, Llama-7B head shape)",
        "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args.sched),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def chunk_step_timing(w, q, k, v, O, lse, do, stream, dfa, reps=5):
    """One worker's calls of the distributed method on this workload's chunks
    (C = S / n_chunks): the chunk step (partial O + lse) and its backward step
    (partial dQ/dK/dV from the saved O/lse), on the last query chunk against
    the first key chunk (no mask) and on the diagonal pair.  Reported beside
    the headline, not part of it."""
    import torch
    if w.n_chunks < 2:
        return None
    C = -(-w.S // w.n_chunks)     # the library's chunk length: ceil(S / n_chunks), the last chunk shorter
    last = (w.n_chunks - 1) * C   # first token of the last chunk
    Cq = w.S - last
    out = {"C": C}
    f32 = dict(dtype=torch.float32, device=q.device)
    ws = torch.empty(max(dfa.dfa_chunk_bwd_workspace_size(w.B, w.H, w.H_kv, Cq, C, w.D), 16),
                     dtype=torch.uint8, device=q.device)
    Op = torch.empty((w.B, Cq, w.H, w.D), **f32)
    lp = torch.empty((w.B, w.H, Cq), **f32)
    acc = (torch.zeros((w.B, Cq, w.H, w.D), **f32), torch.zeros((w.B, C, w.H_kv, w.D), **f32),
           torch.zeros((w.B, C, w.H_kv, w.D), **f32))
    for name, (qa, ka, Lk) in (("off_diagonal", (last, 0, C)), ("diagonal", (last, last, Cq))):
        qs, ks = slice(qa, qa + Cq), slice(ka, ka + Lk)
        qc, kc, vc, dc = (t.contiguous() for t in (q[:, qs], k[:, ks], v[:, ks], do[:, qs]))
        Oc, lc = O[:, qs].contiguous(), lse[:, :, qs].contiguous()

        def fwd():
            dfa.dfa_chunk_attn_fwd(qc, kc, vc, q_offset=qa, kv_offset=ka, scale=w.scale, O_partial=Op,
                                   lse=lp, stream=stream)

        def bwd():
            dfa.dfa_chunk_attn_bwd(qc, kc, vc, Oc, lc, dc, q_offset=qa, kv_offset=ka, scale=w.scale,
                                   dQ_acc=acc[0], dK_acc=acc[1][:, :Lk], dV_acc=acc[2][:, :Lk], workspace_buf=ws,
                                   stream=stream)

        res = {}
        for tag, fn, per_pair in (("fwd", fwd, 4), ("bwd", bwd, 10)):
            for _ in range(2):
                fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(q.device)
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
            torch.cuda.synchronize(q.device)
            ms = a.elapsed_time(b) / reps
            pairs = w.B * w.H * (Cq * Lk if qa != ka else Cq * (Cq + 1) // 2)
            res[f"{tag}_ms"] = ms
            res[f"{tag}_tflops"] = pairs * w.D * per_pair / (ms * 1e-3) / 1e12
        out[name] = res
        if name == "off_diagonal":   # keep this step's partial for the merge below
            Op_first, lp_first = Op.clone(), lp.clone()
    # The owner's merge of two chunk partials (rescale-and-merge): HBM-bound,
    # three [B, C, H, D] fp32 tensors and three [B, H, C] lse per call.
    Om, lm = torch.empty_like(Op), torch.empty_like(lp)

    def merge():
        dfa.dfa_merge_partials(Op_first, lp_first, Op, lp, O_out=Om, lse_out=lm, stream=stream)
    for _ in range(2):
        merge()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(q.device)
    a.record(stream)
    for _ in range(reps):
        merge()
    b.record(stream)
    torch.cuda.synchronize(q.device)
    ms = a.elapsed_time(b) / reps
    nbytes = 3 * (Op.numel() + lp.numel()) * 4
    peaks, kind = measured_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["merge"] = {"ms": ms, "bytes": nbytes, "gbs": gbs, "frac_of_hbm_peak": gbs / float(peaks["hbm_gbs"]),
                    "peak_kind": kind}
    dfa.dfa_check_errors(stream)
    return out


def local_window_pairs(S, C, window):
    """Visible (query, key) pairs per head of causal attention restricted to a
    local window of `window` chunks of C tokens."""
    import numpy as np
    qp = np.arange(S, dtype=np.int64)
    lo = np.maximum(0, (qp // C - (window - 1)) * C)
    return int(np.sum(qp - lo + 1))


def local_window_timing(w, window, q, k, v, do, stream, dfa, reps=3):
    """Forward + backward with the pages' local sliding window (App. F) on the
    same workload; FLOPs counted on the visible pairs only.  Reported beside
    the headline, not part of it."""
    import torch
    if w.n_chunks < 2 or window >= w.n_chunks:
        return None
    C = -(-w.S // w.n_chunks)     # the library's chunk length: ceil(S / n_chunks)
    O = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=q.device)
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsf = dfa.workspace(w.B, w.H, w.H_kv, w.S, w.D, w.n_chunks, False, q.device)
    wsb = dfa.workspace(w.B, w.H, w.H_kv, w.S, w.D, w.n_chunks, True, q.device)

    def fwd():
        dfa.dfa_attn_fwd_local(q, k, v, n_chunks=w.n_chunks, window=window, scale=w.scale, O=O, lse=lse,
                               workspace_buf=wsf, stream=stream)

    def bwd():
        dfa.dfa_attn_bwd_local(q, k, v, O, lse, do, n_chunks=w.n_chunks, window=window, scale=w.scale,
                               dQ=dQ, dK=dK, dV=dV, workspace_buf=wsb, stream=stream)

    pairs = w.B * w.H * local_window_pairs(w.S, C, window)
    out = {"window": window, "chunk": C}
    for tag, fn, per_pair in (("fwd", fwd, 4), ("bwd", bwd, 10)):
        fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(q.device)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(q.device)
        ms = a.elapsed_time(b) / reps
        out[f"{tag}_ms"] = ms
        out[f"{tag}_tflops"] = pairs * w.D * per_pair / (ms * 1e-3) / 1e12
    dfa.dfa_check_errors(stream)
    return out


SPLIT_KV_SHAPES = [(1, 1, 1, 32768, 128), (1, 1, 1, 16384, 128)]


def split_kv_timing(device, stream, dfa, reps=10):
    """Causal forward and backward of problems with fewer 256-row query blocks
    (forward) or key-tile pairs (backward) than SMs, with the plain balanced
    list and with split-kv helper items (pieces of each block's key range, or
    of each key tile's query range, computed by other CTAs, then merged or
    added).  Inputs of these sizes stay in L2; both passes are compute-bound
    either way.  Reported beside the headline."""
    import torch
    from long_context_causal_gb300.inputs import make
    out = []
    for B, H, Hkv, S, D in SPLIT_KV_SHAPES:
        q, k, v, do = make(B, H, Hkv, S, D, torch.bfloat16, seed=3, device=device)
        O = torch.empty_like(q)
        lse = torch.empty((B, H, S), dtype=torch.float32, device=device)
        dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        wsf = dfa.workspace(B, H, Hkv, S, D, 1, False, device)
        wsb = dfa.workspace(B, H, Hkv, S, D, 1, True, device)
        pairs = B * H * S * (S + 1) // 2 * D
        row = {"B": B, "H": H, "H_kv": Hkv, "S": S, "D": D}
        for sched in ("balanced", "split_kv"):
            def fwd():
                dfa.dfa_attn_fwd(q, k, v, sched=sched, O=O, lse=lse, workspace_buf=wsf, stream=stream)

            def bwd():
                dfa.dfa_attn_bwd(q, k, v, O, lse, do, sched=sched, dQ=dQ, dK=dK, dV=dV, workspace_buf=wsb,
                                 stream=stream)
            for tag, fn, per_pair in (("fwd", fwd, 4), ("bwd", bwd, 10)):
                for _ in range(3):
                    fn()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize(device)
                e0.record(stream)
                for _ in range(reps):
                    fn()
                e1.record(stream)
                torch.cuda.synchronize(device)
                ms = e0.elapsed_time(e1) / reps
                row[f"{sched}_{tag}_ms"] = ms
                row[f"{sched}_{tag}_tflops"] = pairs * per_pair / (ms * 1e-3) / 1e12
        row["fwd_speedup"] = row["balanced_fwd_ms"] / row["split_kv_fwd_ms"]
        row["bwd_speedup"] = row["balanced_bwd_ms"] / row["split_kv_bwd_ms"]
        out.append(row)
    dfa.dfa_check_errors(stream)
    return out


VARLEN_LENS = [57344, 28672, 16384, 12288, 8192, 4096, 2048, 1024, 512, 512]   # 131072 tokens


def varlen_timing(device, stream, dfa, H=32, Hkv=32, D=128, reps=3):
    """A packed batch of sequences of very different lengths (a long-tail mix of
    128K tokens at the Llama-7B head shape): causal forward + backward as one
    launch each through the packed entry points, against one dense call per
    sequence.  FLOPs on each sequence's own causal triangle.  Each packed
    tensor (1 GB) exceeds L2.  Reported beside the headline."""
    import numpy as np
    import torch
    from long_context_causal_gb300.inputs import make
    lens = VARLEN_LENS
    T = sum(lens)
    q, k, v, do = (x[0] for x in make(1, H, Hkv, T, D, torch.bfloat16, seed=5, device=device))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    O = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=device)
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsf = dfa.varlen_workspace(cu, H, Hkv, D, False, device)
    wsb = dfa.varlen_workspace(cu, H, Hkv, D, True, device)
    pairs = sum(L * (L + 1) // 2 for L in lens) * H
    segs = [(int(a), int(b)) for a, b in zip(cu[:-1], cu[1:])]
    seg_lse = [torch.empty((1, H, b - a), dtype=torch.float32, device=device) for a, b in segs]
    wsd = {b - a: (dfa.workspace(1, H, Hkv, b - a, D, 1, False, device),
                   dfa.workspace(1, H, Hkv, b - a, D, 1, True, device)) for a, b in segs}

    def packed_fwd():
        dfa.dfa_attn_fwd_varlen(q, k, v, cu, O=O, lse=lse, workspace_buf=wsf, stream=stream)

    def packed_bwd():
        dfa.dfa_attn_bwd_varlen(q, k, v, O, lse, do, cu, dQ=dQ, dK=dK, dV=dV, workspace_buf=wsb, stream=stream)

    def loop_fwd():
        for (a, b), l in zip(segs, seg_lse):
            dfa.dfa_attn_fwd(q[None, a:b], k[None, a:b], v[None, a:b], O=O[None, a:b], lse=l,
                             workspace_buf=wsd[b - a][0], stream=stream)

    def loop_bwd():
        for (a, b), l in zip(segs, seg_lse):
            dfa.dfa_attn_bwd(q[None, a:b], k[None, a:b], v[None, a:b], O[None, a:b], l, do[None, a:b],
                             dQ=dQ[None, a:b], dK=dK[None, a:b], dV=dV[None, a:b], workspace_buf=wsd[b - a][1],
                             stream=stream)

    out = {"lens": lens, "H": H, "H_kv": Hkv, "D": D}
    for tag, fn, per_pair in (("packed_fwd", packed_fwd, 4), ("packed_bwd", packed_bwd, 10),
                              ("per_sequence_fwd", loop_fwd, 4), ("per_sequence_bwd", loop_bwd, 10)):
        fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(device)
        ms = a.elapsed_time(b) / reps
        out[f"{tag}_ms"] = ms
        out[f"{tag}_tflops"] = pairs * D * per_pair / (ms * 1e-3) / 1e12
    dfa.dfa_check_errors(stream)
    return out


def timed_ms(fn, device, stream, reps, warm=1):
    """Mean device time of fn() over reps calls (CUDA events on `stream`)."""
    import torch
    for _ in range(warm):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    torch.cuda.synchronize(device)
    return a.elapsed_time(b) / reps


def fwd_bwd_legs(w, q, k, v, do, O, lse, dQ, dK, dV, wsf, wsb, sched, stream, dfa, reps, warm):
    """fwd, bwd and fwd + bwd ms and TFLOP/s of one workload under one schedule."""
    def fwd():
        dfa.dfa_attn_fwd(q, k, v, n_chunks=w.n_chunks, scale=w.scale, sched=sched, O=O, lse=lse,
                         workspace_buf=wsf, stream=stream)

    def bwd():
        dfa.dfa_attn_bwd(q, k, v, O, lse, do, n_chunks=w.n_chunks, scale=w.scale, sched=sched,
                         dQ=dQ, dK=dK, dV=dV, workspace_buf=wsb, stream=stream)
    f_ms = timed_ms(fwd, q.device, stream, reps, warm)
    b_ms = timed_ms(bwd, q.device, stream, reps, warm)
    dfa.dfa_check_errors(stream)
    ff, bf = w.causal_flops(True, False), w.causal_flops(False, True)
    return {"fwd_ms": f_ms, "bwd_ms": b_ms, "total_ms": f_ms + b_ms,
            "fwd_tflops": ff / (f_ms * 1e-3) / 1e12, "bwd_tflops": bf / (b_ms * 1e-3) / 1e12,
            "tflops": (ff + bf) / ((f_ms + b_ms) * 1e-3) / 1e12,
            "pct_of_nominal_bf16_peak": 100.0 * (ff + bf) / ((f_ms + b_ms) * 1e-3) / 1e12 / NOMINAL_BF16_TFLOPS}


def unbalanced_timing(w, tensors, stream, dfa, balanced, reps=3):
    """The same workload with the unbalanced work list (each persistent CTA
    takes one contiguous token range per head, the pages' baseline
    distribution of the causal triangle, DISTFLASHATTN §4.5 / Fig. 4) against
    the balanced list of the headline."""
    out = fwd_bwd_legs(w, *tensors, "unbalanced", stream, dfa, reps, 1)
    out["balanced_over_unbalanced"] = out["total_ms"] / balanced["total_ms"]
    out["balanced"] = balanced
    return out


OTHER_WORKLOADS = ("llama7b_s32k", "llama7b_gqa8_s64k", "llama7b_s512k")


def workloads_timing(device, stream, dfa, names=OTHER_WORKLOADS):
    """fwd / bwd / fwd + bwd of the other Llama-7B workloads (32K, GQA 32/8
    heads at 64K with K x 2, 512K), balanced list, each on its own inputs
    (freed before the next).  The 512K step takes about 8 s: one warm-up step
    and one timed step there, three elsewhere."""
    import torch
    from long_context_causal_gb300.inputs import WORKLOADS, make_workload
    out = {}
    for name in names:
        w = WORKLOADS[name]
        q, k, v, do = make_workload(w, device)
        O, lse = torch.empty_like(q), torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=device)
        dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        wsf = dfa.workspace(w.B, w.H, w.H_kv, w.S, w.D, w.n_chunks, False, device)
        wsb = dfa.workspace(w.B, w.H, w.H_kv, w.S, w.D, w.n_chunks, True, device)
        reps = 1 if w.S >= 262144 else 3
        r = fwd_bwd_legs(w, q, k, v, do, O, lse, dQ, dK, dV, wsf, wsb, "balanced", stream, dfa, reps, 1)
        r.update({"B": w.B, "H": w.H, "H_kv": w.H_kv, "S": w.S, "D": w.D, "n_chunks": w.n_chunks, "reps": reps})
        out[name] = r
        del q, k, v, do, O, lse, dQ, dK, dV, wsf, wsb
        torch.cuda.empty_cache()
    return out


def gpu_numa_cpus(index):
    """(NUMA node, its CPU list) of GPU `index` from sysfs, or (None, None)."""
    try:
        bus = subprocess.run(["nvidia-smi", f"--id={index}", "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip().lower()
        # nvidia-smi prints an 8-digit PCI domain; sysfs uses 4 digits
        dom, rest = bus.split(":", 1)
        path = f"/sys/bus/pci/devices/{dom[-4:]}:{rest}/numa_node"
        node = int(open(path).read().strip())
        if node < 0:
            return None, None
        cpus = set()
        for part in open(f"/sys/devices/system/node/node{node}/cpulist").read().strip().split(","):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        return node, sorted(cpus)
    except Exception:
        return None, None


def copy_bandwidth(hin, xin, hout, yout, s_in, s_out, device, dfa, reps=3):
    """GB/s of the step's host-to-device copies alone, of its device-to-host
    copies alone, and of both at once, on the same pinned buffers and streams
    as the end-to-end leg (copy engines); and of each direction through the SMs
    (dfa_copy)."""
    import torch

    def run_sm(h2d):
        cur = torch.cuda.current_stream(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        a.record(cur)
        for _ in range(reps):
            for h_, d_ in (zip(hin, xin) if h2d else zip(hout, yout)):
                if h2d:
                    dfa.dfa_copy(d_, h_, stream=cur)
                else:
                    dfa.dfa_copy(h_, d_, stream=cur)
        b.record(cur)
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) / reps

    def run(h2d, d2h):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream(device)
        torch.cuda.synchronize(device)
        a.record(cur)
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        for _ in range(reps):
            if h2d:
                with torch.cuda.stream(s_in):
                    for d_, h_ in zip(xin, hin):
                        d_.copy_(h_, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s_out):
                    for h_, d_ in zip(hout, yout):
                        h_.copy_(d_, non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)
        b.record(cur)
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) / reps
    bi = sum(t.numel() * t.element_size() for t in hin)
    bo = sum(t.numel() * t.element_size() for t in hout)
    run(True, True)
    t_in, t_out, t_both = run(True, False), run(False, True), run(True, True)
    run_sm(True)
    s_in_ms, s_out_ms = run_sm(True), run_sm(False)
    return {"h2d_gbs": bi / (t_in * 1e-3) / 1e9, "d2h_gbs": bo / (t_out * 1e-3) / 1e9,
            "h2d_ms": t_in, "d2h_ms": t_out, "both_ms": t_both,
            "both_gbs": (bi + bo) / (t_both * 1e-3) / 1e9,
            "sm_h2d_gbs": bi / (s_in_ms * 1e-3) / 1e9, "sm_d2h_gbs": bo / (s_out_ms * 1e-3) / 1e9}


# ---------------------------------------------------------------- GPU arm
def main():
    args = parse()
    from long_context_causal_gb300.inputs import WORKLOADS, Workload
    if args.shape:
        import torch
        B, H, Hkv, S, D = (int(x) for x in args.shape.split(","))
        w = Workload(f"custom_B{B}_H{H}_Hkv{Hkv}_S{S}_D{D}", B, H, Hkv, S, D, 1, torch.bfloat16)
    else:
        w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch

    from long_context_causal_gb300 import dfa
    from long_context_causal_gb300.inputs import make

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local if world > 1 else 0)
    seed = rank_seed(w.seed, rank)
    q, k, v, do = make(w.B, w.H, w.H_kv, w.S, w.D, w.dtype, seed=seed, device=dev, k_scale=w.k_scale)
    O = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsf = dfa.workspace(w.B, w.H, w.H_kv, w.S, w.D, w.n_chunks, False, dev)
    wsb = dfa.workspace(w.B, w.H, w.H_kv, w.S, w.D, w.n_chunks, True, dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        dfa.dfa_attn_fwd(q, k, v, n_chunks=w.n_chunks, scale=w.scale, sched=args.sched, O=O, lse=lse,
                         workspace_buf=wsf, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        dfa.dfa_attn_bwd(q, k, v, O, lse, do, n_chunks=w.n_chunks, scale=w.scale, sched=args.sched,
                         dQ=dQ, dK=dK, dV=dV, workspace_buf=wsb, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    dfa.dfa_check_errors(stream)

    launches0 = sum(dfa.dfa_launch_count(kd) for kd in dfa.KERNEL_KINDS)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local if world > 1 else 0) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.5)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        step(evs[s])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop() if clocks else None
    dfa.dfa_check_errors(stream)
    launches = sum(dfa.dfa_launch_count(kd) for kd in dfa.KERNEL_KINDS) - launches0

    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    flops = w.causal_flops()
    ms_step = total_ms / args.steps
    value = job_value(flops, ms_step, world)

    peaks, peak_kind = measured_peaks()
    peak_tc = float(peaks["bf16_tflops"])
    bwd_flops = w.causal_flops(fwd=False, bwd=True)
    fwd_flops = w.causal_flops(fwd=True, bwd=False)
    bwd_tflops = bwd_flops / (bwd_ms * 1e-3) / 1e12
    fwd_tflops = fwd_flops / (fwd_ms * 1e-3) / 1e12

    # End to end through the public API with host buffers: every step copies its
    # inputs in from pinned host memory and reads every result back, inside the
    # timing.  Three schedules: the copies on their own streams (DMA copy
    # engines), overlapping the neighbouring steps' compute (device inputs and
    # outputs double-buffered, events order the reuse of each buffer), as a
    # training loop streaming its batches would run; in, compute, out one after
    # another on one stream with the copy engines; or the same with the copies
    # through the SMs (dfa_copy).  Which is fastest depends on the host link:
    # where concurrent copies slow the kernels down more than they save, a
    # serial one wins, and after heavy CPU work on the host the copy engines can
    # run at a fraction of the link's rate while SM copies keep it.  Each is
    # tried for two steps and the fastest is timed.
    e2e = None
    if not args.no_e2e:
        # Pinned host buffers on the GPU's own NUMA node: pages are placed when
        # they are pinned, on the node of the CPU that pins them, so the
        # allocating thread runs on that node's CPUs meanwhile (no GPU setting
        # is touched; the previous CPU affinity is restored).
        node, cpus = gpu_numa_cpus(local if world > 1 else 0)
        old_aff = os.sched_getaffinity(0)
        if cpus:
            try:
                os.sched_setaffinity(0, cpus)
            except OSError:
                node = None
        try:
            hin = [t.cpu().pin_memory() for t in (q, k, v, do)]
            hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (O, lse, dQ, dK, dV)]
        finally:
            os.sched_setaffinity(0, old_aff)
        h2d = sum(t.numel() * t.element_size() for t in hin)
        d2h = sum(t.numel() * t.element_size() for t in hout)
        xin = [(q, k, v, do), tuple(torch.empty_like(t) for t in (q, k, v, do))]
        yout = [(O, lse, dQ, dK, dV), tuple(torch.empty_like(t) for t in (O, lse, dQ, dK, dV))]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_ready, comp_done, out_done = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

        def issue_in(n):     # H2D of step n's inputs, once step n-2 has finished reading that slot
            b = n % 2
            if n >= 2:
                s_in.wait_event(comp_done[b])
            with torch.cuda.stream(s_in):
                for d_, h_ in zip(xin[b], hin):
                    d_.copy_(h_, non_blocking=True)
            in_ready[b].record(s_in)

        comp_ev = []

        def issue_comp(n):   # fwd + bwd of step n, once its inputs are in and step n-2's results are out
            b = n % 2
            stream.wait_event(in_ready[b])
            if n >= 2:
                stream.wait_event(out_done[b])
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            comp_ev.append(ev)
            ev[0].record(stream)
            qq, kk, vv, dd = xin[b]
            OO, ll, gq, gk, gv = yout[b]
            dfa.dfa_attn_fwd(qq, kk, vv, n_chunks=w.n_chunks, scale=w.scale, sched=args.sched, O=OO, lse=ll,
                             workspace_buf=wsf, stream=stream)
            dfa.dfa_attn_bwd(qq, kk, vv, OO, ll, dd, n_chunks=w.n_chunks, scale=w.scale, sched=args.sched,
                             dQ=gq, dK=gk, dV=gv, workspace_buf=wsb, stream=stream)
            comp_done[b].record(stream)
            ev[1].record(stream)

        def issue_out(n):    # D2H of step n's results
            b = n % 2
            s_out.wait_event(comp_done[b])
            with torch.cuda.stream(s_out):
                for h_, d_ in zip(hout, yout[b]):
                    h_.copy_(d_, non_blocking=True)
            out_done[b].record(s_out)

        def e2e_run(n_steps, mode, t0=None, t1=None):
            if t0 is not None:
                t0.record(stream)
            if mode == "overlapped":
                s_in.wait_stream(stream)
                s_out.wait_stream(stream)
                issue_in(0)
                for n in range(n_steps):
                    if n + 1 < n_steps:
                        issue_in(n + 1)
                    issue_comp(n)
                    issue_out(n)
                stream.wait_stream(s_in)
                stream.wait_stream(s_out)
            else:
                sm = mode == "serial_sm"
                for n in range(n_steps):
                    with torch.cuda.stream(stream):
                        for d_, h_ in zip(xin[0], hin):
                            if sm:
                                dfa.dfa_copy(d_, h_, stream=stream)
                            else:
                                d_.copy_(h_, non_blocking=True)
                    in_ready[0].record(stream)
                    issue_comp(0)
                    with torch.cuda.stream(stream):
                        for h_, d_ in zip(hout, yout[0]):
                            if sm:
                                dfa.dfa_copy(h_, d_, stream=stream)
                            else:
                                h_.copy_(d_, non_blocking=True)
                    out_done[0].record(stream)
            if t1 is not None:
                t1.record(stream)

        trial = {}
        for mode in ("overlapped", "serial", "serial_sm"):
            e2e_run(1, mode)
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e2e_run(2, mode, a, b)
            torch.cuda.synchronize(dev)
            trial[mode] = max_over_ranks(a.elapsed_time(b), world) / 2
        mode = min(trial, key=trial.get)
        n_e2e = max(1, min(args.steps, 10))
        barrier(world)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        comp_ev.clear()
        e2e_clocks = ClockSampler(local if world > 1 else 0)
        e2e_clocks.start()
        e2e_run(n_e2e, mode, a, b)
        torch.cuda.synchronize(dev)
        e2e_clk = e2e_clocks.stop()
        barrier(world)
        dfa.dfa_check_errors(stream)
        e2e_ms = max_over_ranks(a.elapsed_time(b), world) / n_e2e
        # the forward + backward kernels' own time inside the end-to-end run: near
        # the device-timed step, the copies are hidden; well above it, concurrent
        # copies slow the kernels down
        comp_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in comp_ev)
        bw = copy_bandwidth(hin, xin[1], hout, yout[1], s_in, s_out, dev, dfa)
        e2e = {"value": job_value(flops, e2e_ms, world), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": n_e2e,
               "copies": {"overlapped": "overlapped with the neighbouring steps' compute on two copy streams",
                          "serial": "in, compute, out one after another on the compute stream (copy engines)",
                          "serial_sm": "in, compute, out one after another on the compute stream, copies through "
                                       "the SMs (dfa_copy)"}[mode],
               "schedule_trial_ms": trial,
               "pinned_numa_node": node, **bw, "compute_ms_in_e2e": comp_ms,
               # SM clock and board power while the end-to-end steps ran: host copies
               # add power on a capped part, and the clock gives way
               "clocks": e2e_clk,
               # a step costs at least max(compute, copies); the copies bound it when they take longer
               "link_bound": bw["both_ms"] > ms_step}
        del xin, yout

    balanced = {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "total_ms": fwd_ms + bwd_ms, "tflops": flops / ((fwd_ms + bwd_ms) * 1e-3) / 1e12}
    unbal = None
    if not args.no_unbalanced and args.sched == "balanced":
        unbal = unbalanced_timing(w, (q, k, v, do, O, lse, dQ, dK, dV, wsf, wsb), stream, dfa, balanced)
    chunk = None if args.no_chunk_step else chunk_step_timing(w, q, k, v, O, lse, do, stream, dfa)
    local_win = None if args.window <= 0 else local_window_timing(w, args.window, q, k, v, do, stream, dfa)
    split = None if args.no_split_kv else split_kv_timing(q.device, stream, dfa)
    varlen = None if args.no_varlen else varlen_timing(q.device, stream, dfa)
    others = None
    if not args.no_workloads and args.shape is None and w.name == "llama7b_s128k":
        del wsf, wsb
        torch.cuda.empty_cache()
        others = workloads_timing(q.device, stream, dfa)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fl, el, cores, desc = oracle_sample(w, args.cpu_seconds)
        rate = fl / el
        cpu = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
               # extrapolation, not a measurement: the whole workload's forward + backward
               # FLOPs at the sampled rate (a row's cost grows with its visible keys)
               "extrapolated_full_s": flops / rate,
               "extrapolated_full_note": "extrapolated: full fwd+bwd FLOPs divided by the sampled rate"}

    if rank != 0:
        return
    line = {
        "metric": "causal attn fwd+bwd TFLOP/s (bf16, Llama-7B head shape)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype.is_floating_point and w.dtype.itemsize == 2 else "f32",
        "data": "synthetic",
        "config": config_of(w, args.sched),
        "pct_of_nominal_bf16_peak": 100.0 * value / world / NOMINAL_BF16_TFLOPS,
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops,
        # the backward counted at 8D per pair (without recomputing S = QK^T), for other conventions
        "bwd_tflops_8d": bwd_tflops * 0.8,
        "roofline": {"bound": "tensor", "kernel": "dfa_attn_bwd (delta + bwd + dQ convert)",
                     "achieved": bwd_tflops, "peak": peak_tc, "unit": "TFLOP/s",
                     "frac": bwd_tflops / peak_tc,
                     "traffic": scaled_traffic(w, "bwd"),
                     "traffic_note": f"DRAM bytes of one launch captured on {NCU_TRAFFIC_REF['workload']}, "
                                     "scaled by the ratio of causal pairs (estimate)",
                     "peak_kind": f"{peak_kind} bf16 burst"},
        "roofline_fwd": {"bound": "tensor", "achieved": fwd_tflops, "peak": peak_tc, "unit": "TFLOP/s",
                         "frac": fwd_tflops / peak_tc, "traffic": scaled_traffic(w, "fwd")},
        "cpu_baseline": cpu,
        "chunk_step": chunk,
        "local_window": local_win,
        "split_kv": split,
        "varlen": varlen,
        "unbalanced": unbal,
        "workloads": others,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
