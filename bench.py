"""Benchmark: attention fwd+bwd per 16,384-token packed microbatch on GB300.

One step = the whole hot path over one synthetic microbatch: the forward
kernel, then the backward (rowsum preprocess, dK/dV pass, dQ pass), all
through the library's C ABI.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

The headline workload is the context-4,096 global-causal microbatch; the
window-512 and context-512 microbatches, the context sweep (512 ... 4,096,
global and window 512) and the 65,536-token 16/4-head long-context case are
measured in the same run under "also"; the Gated DeltaNet local layer
(include/gdn_varlen.h) on the context-4,096 and context-512 microbatches under
"also.gdn".

Timing: CUDA events on the launching stream around every kernel of every
step; the L2 (129 MB) is flushed by writing a 512 MiB buffer between steps,
outside the events.  SM clocks are sampled with nvidia-smi during the timed
steps.  Multi-GPU: replicas only (every rank runs its own microbatch; there
is no data-path collective), weak scaling.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from varlen_sliding_window_gb300 import synth  # noqa: E402

METRIC = "attn fwd+bwd ms per 16K-token microbatch; unmasked TFLOPS & % of bf16 peak"
# The page's FlashAttention-2 fwd+bwd per layer on its own (unnamed, clock-capped)
# GPU, for the same workloads: reported as context ("page_context"), not as a
# baseline and not as a target.
PAGE_FA2_MS = {"ctx512_global": 0.68, "ctx4096_global": 1.43, "ctx4096_w512": 0.95,
               "sweep_ctx512_global": 0.68, "sweep_ctx1024_global": 0.94, "sweep_ctx2048_global": 1.26,
               "sweep_ctx4096_global": 1.43, "sweep_ctx512_w512": 0.69, "sweep_ctx1024_w512": 0.85,
               "sweep_ctx2048_w512": 0.91, "sweep_ctx4096_w512": 0.95}
# The page's Gated DeltaNet layer (flash-linear-attention kernels), fwd+bwd per
# step at context 4,096 on the same unnamed GPU (research.dws.rip/llm/kernels,
# section 03, Fig. 5): context for the Gated DeltaNet leg.
PAGE_GDN_MS = 1.73
PAGE_KDA_MS = 3.32  # the same for the Kimi Delta layer
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GEMM units (2*d*Hq*pairs flops each) each kernel does that the counting rule
# credits: forward QK^T + PV; dK/dV pass S, dP, dV, dK; dQ pass dQ only (its
# recomputed S and dP are not counted).
KERNEL_UNITS = {"fwd": 2.0, "bwd_preprocess": 0.0, "bwd_dkdv": 4.0, "bwd_dq": 1.0}
# Kernels of this library per step: forward, preprocess, planner, dK/dV, dQ.
KERNELS_PER_STEP = 5


def gdn_flops(cu: np.ndarray, nh: int, d: int, per_channel: bool = False) -> tuple[float, float]:
    """Matrix-product FLOPs the Gated DeltaNet (or, per_channel, Kimi Delta)
    kernels perform, per call (forward, backward), summed over chunks of
    n <= 64 tokens and heads.  Gated DeltaNet: forward 2d(5n^2 + 3nd) (K K^T,
    Q K^T, the two WY factors, W H, Q H, the masked Q K^T block times E,
    K^T E); backward, which recomputes the forward without O,
    2d(4n^2 + 2nd) + 2d(n^2 + 3nd) + 2d(4n^2 + 5nd) + 14dn^2 + 4n^3
    (recomputation, state-gradient pass, the two local passes).  Kimi Delta:
    K K^T and Q K^T only in the 10 of 16 blocks of 16 rows on or below the
    diagonal; its local passes take 2d(n^2 + 3nd) and 8dn^2 + 4n^3, and the
    four decay-weighted sums of its last pass 4 d n^2."""
    fwd = bwd = 0.0
    for L in np.diff(cu.astype(np.int64)):
        for c0 in range(0, int(L), 64):
            n = float(min(64, int(L) - c0))
            qk = 2 * 2 * d * n * n * (10.0 / 16.0 if per_channel else 1.0)  # K K^T and Q K^T
            wu = 2 * 2 * d * n * n                                           # W, U
            fwd += qk + wu + 2 * d * (n * n + 3 * n * d)
            rec = qk + wu + 2 * 2 * n * d * d
            state = 2 * d * (n * n + 3 * n * d)
            if per_channel:
                bwd += rec + state + 2 * d * (n * n + 3 * n * d) + 8 * d * n * n + 4 * n ** 3 + 4 * d * n * n
            else:
                bwd += rec + state + 2 * d * (4 * n * n + 5 * n * d) + 14 * d * n * n + 4 * n ** 3
    return fwd * nh, bwd * nh


def unmasked_pairs(cu: np.ndarray, window: int) -> int:
    """Closed form of sum_i |V(i)| per segment (global: L(L+1)/2; window w:
    (w+1)(w+2)/2 + (L-w-1)(w+1) when L > w+1)."""
    n = 0
    for L in np.diff(cu.astype(np.int64)):
        L = int(L)
        if window < 0 or L <= window + 1:
            n += L * (L + 1) // 2
        else:
            n += (window + 1) * (window + 2) // 2 + (L - window - 1) * (window + 1)
    return n


def algorithmic_bytes(w) -> int:
    """HBM bytes one step must move at least: the forward reads q, k, v and
    writes out, lse; the backward reads q, k, v, out, dout, lse, writes dq, dk,
    dv, and writes then reads D (fp32 [Hq, T])."""
    T, row_q, row_kv = w.total, w.hq * w.d * 2, w.hkv * w.d * 2
    stat = 4 * w.hq * T
    fwd = T * (row_q + 2 * row_kv + row_q) + stat
    bwd = T * (row_q + 2 * row_kv + 2 * row_q) + stat + T * (row_q + 2 * row_kv) + 2 * stat
    return fwd + bwd


# ex2 results per clock per SM, measured on a GB300 with a microbenchmark of
# back-to-back independent ex2.approx.f32 instructions.
MUFU_EX2_PER_CLK_SM = 31.0
# bf16 mma.sync m16n8k16 (the warp-level instruction the linear-attention
# kernels use): one per 2 cycles per SM, 1,024 FMA per clock per SM, measured
# on a GB300 with a microbenchmark (20 cycles latency; 4 warps with 4
# independent accumulators reach it).
MMA_SYNC_FMA_PER_CLK_SM = 1024.0
NUM_SMS = 152


def roofs(w, pairs: int, ms: float, peak_t: float, peak_hbm: float, sm_mhz) -> dict:
    """Both roofs for one step: counted tensor FLOPs against the bf16 peak,
    algorithmic bytes against the HBM copy peak, and the exp count (pairs * Hq
    in the forward, twice that in the backward) against the ex2 rate."""
    sec = ms * 1e-3
    flops = 4.0 * w.d * w.hq * pairs * 3.5
    nbytes = algorithmic_bytes(w)
    nexp = 3 * pairs * w.hq
    mhz = sm_mhz or 2032.0
    exp_peak = MUFU_EX2_PER_CLK_SM * NUM_SMS * mhz * 1e6
    return {"tensor": {"achieved_tflops": flops / sec / 1e12, "frac": flops / sec / 1e12 / peak_t},
            "hbm": {"bytes": nbytes, "achieved_gbs": nbytes / sec / 1e9, "frac": nbytes / sec / 1e9 / peak_hbm},
            "exp": {"count": nexp, "per_s": nexp / sec, "frac": nexp / sec / exp_peak,
                    "peak_per_s": exp_peak, "peak_basis": f"{MUFU_EX2_PER_CLK_SM:g} ex2/clk/SM x {NUM_SMS} SMs x {mhz:g} MHz"},
            "intensity_flop_per_byte": flops / nbytes}


def csrc_hash() -> str:
    """sha1 (12 hex digits) of the attention kernels' sources: attn_*.cu, then
    *.cuh, then *.h, each sorted (the Gated DeltaNet file does not change them)."""
    import glob
    import hashlib
    d = os.path.join(ROOT, "varlen_sliding_window_gb300", "csrc")
    h = hashlib.sha1()
    for pat in ("attn_*.cu", "*.cuh", "*.h"):
        for f in sorted(glob.glob(os.path.join(d, pat))):
            h.update(open(f, "rb").read())
    return h.hexdigest()[:12]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"vsw_bench_clocks_{os.getpid()}_gpu{gpu_index}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_time(inp, window: int, scale: float, budget_s: float):
    """Times the float64 oracle (fwd + bwd) on whole segments, longest first,
    until `budget_s` seconds have passed; returns (ms per full microbatch,
    sample description, cores).  The oracle's work per segment and head is
    proportional to the segment's unmasked (query, key) pairs (L(L+1)/2 for
    global causal, about L (w+1) for a window w), so the sample is scaled to
    the microbatch by the pair count."""
    import oracle
    cu = inp.cu_seqlens
    segs = [(int(a), int(b)) for a, b in zip(cu[:-1], cu[1:]) if b > a]
    # Longest first so that the sample includes the dominant segments.
    segs.sort(key=lambda s: -(s[1] - s[0]))
    seg_pairs = {s: unmasked_pairs(np.array([0, s[1] - s[0]]), window) for s in segs}
    total_w = sum(seg_pairs.values())
    done_w, elapsed, n = 0, 0.0, 0
    for a, b in segs:
        sl = slice(a, b)
        c = np.array([0, b - a])
        t0 = time.perf_counter()
        oracle.forward(inp.q[sl], inp.k[sl], inp.v[sl], c, window, scale)
        oracle.backward(inp.dout[sl], inp.q[sl], inp.k[sl], inp.v[sl], c, window, scale)
        elapsed += time.perf_counter() - t0
        done_w += seg_pairs[(a, b)]
        n += 1
        if elapsed >= budget_s:
            break
    ms = 1e3 * elapsed * total_w / done_w
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = (f"{n} of {len(segs)} segments (longest first, {done_w / total_w:.1%} of the unmasked pairs), all heads, "
              f"oracle fwd+bwd in numpy float64; scaled to the microbatch by the unmasked pair count")
    return ms, sample, cores


def workload_config(wl, cu, pairs: int, world: int) -> dict:
    """The "config" object of a bench line, the same for both arms."""
    return {"workload": wl.name, "tokens": wl.total, "context": wl.context, "window_left": wl.window_left,
            "hq": wl.hq, "hkv": wl.hkv, "head_dim": wl.d, "segments": int(len(cu) - 1),
            "doc_seed": wl.doc_seed, "tensor_seed": wl.tensor_seed, "unmasked_pairs": int(pairs),
            "l2": "flushed between steps (512 MiB write)", "parallelism": f"replicas x{world}"}


def job_ms_per_microbatch(timed_ms: float, steps: int, world: int, device) -> float:
    """Whole-job value: every rank times `steps` steps of its own microbatch
    (replicas, weak scaling); the job takes as long as its slowest rank, and
    it processed steps * world microbatches.  With world > 1 the caller's
    process group does the MAX (NCCL on GPUs; gloo works the same on CPU)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([timed_ms], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item() / (steps * world)


def run_reference(args, wl):
    """The reference arm: the CPU oracle as it stands, timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = wl.inputs()
    budget = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_time(inp, wl.window_left, wl.softmax_scale, budget)
    vals = []
    sample = cores = None
    for _ in range(args.steps):
        ms, sample, cores = oracle_time(inp, wl.window_left, wl.softmax_scale, budget)
        vals.append(ms)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "ms", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": value, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, inp.cu_seqlens, unmasked_pairs(inp.cu_seqlens, wl.window_left),
                                      int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": value, "unit": "ms", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="ctx4096_global")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--also", default="ctx4096_w512,ctx512_global",
                    help="extra workloads measured in full in the same run (comma list, '' for none)")
    ap.add_argument("--sweep", default=",".join(f"sweep_ctx{c}_{t}" for t in ("global", "w512")
                                                for c in (512, 1024, 2048, 4096)) + ",long65536_global,long65536_w4096",
                    help="workloads whose step and kernel times are reported under also.sweep ('' for none)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--gdn", default="gdn_ctx4096,gdn_ctx512,kda_ctx4096,kda_ctx512",
                    help="Gated DeltaNet / Kimi Delta workloads measured under also.gdn ('' for none)")
    args = ap.parse_args()
    wls = synth.workloads()
    wl = wls[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)

    import torch
    import torch.distributed as dist

    from varlen_sliding_window_gb300 import binding

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load_library()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()

    def prepare(w):
        inp = w.inputs()
        cu = inp.cu_seqlens
        to = lambda bits: torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(dev)  # noqa: E731
        t = {"q": to(inp.q_bits), "k": to(inp.k_bits), "v": to(inp.v_bits), "dout": to(inp.dout_bits),
             "cu": torch.from_numpy(cu).to(dev)}
        t["out"] = torch.empty_like(t["q"])
        t["lse"] = torch.empty(w.hq, w.total, dtype=torch.float32, device=dev)
        t["ws"] = torch.empty(binding.attn_varlen_bwd_workspace_bytes(w.total, w.hq), dtype=torch.uint8, device=dev)
        t["dq"], t["dk"], t["dv"] = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
        return inp, t

    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def step(w, t, evs=None):
        """One step through the C ABI, kernel by kernel; evs = 5 events recorded
        between the forward, the preprocess (with the one-CTA planner beside
        it), the dK/dV pass and the dQ pass."""
        ms, win, sc = w.context, w.window_left, w.softmax_scale
        if evs:
            evs[0].record(stream)
        binding.attn_varlen_fwd(t["q"], t["k"], t["v"], t["cu"], ms, win, sc, t["out"], t["lse"])
        if evs:
            evs[1].record(stream)
        binding.attn_varlen_bwd_preprocess(t["dout"], t["out"], t["ws"])
        binding.attn_varlen_bwd_plan(t["cu"], ms, win, t["ws"], w.total, w.hq, w.hkv)
        if evs:
            evs[2].record(stream)
        binding.attn_varlen_bwd_dkdv(t["dout"], t["q"], t["k"], t["v"], t["lse"], t["ws"], t["cu"], ms, win, sc,
                                     t["dk"], t["dv"])
        if evs:
            evs[3].record(stream)
        binding.attn_varlen_bwd_dq(t["dout"], t["q"], t["k"], t["v"], t["lse"], t["ws"], t["cu"], ms, win, sc,
                                   t["dq"])
        if evs:
            evs[4].record(stream)

    def step_api(w, t, mid_ev=None):
        """One step as a user makes it: the forward call, then the backward call
        (mid_ev, if given, is recorded between the two)."""
        ms, win, sc = w.context, w.window_left, w.softmax_scale
        binding.attn_varlen_fwd(t["q"], t["k"], t["v"], t["cu"], ms, win, sc, t["out"], t["lse"])
        if mid_ev is not None:
            mid_ev.record(stream)
        binding.attn_varlen_bwd(t["dout"], t["q"], t["k"], t["v"], t["out"], t["lse"], t["cu"], ms, win, sc,
                                t["dq"], t["dk"], t["dv"])

    def measure(w, steps, warmup, sample_clocks=False):
        """Times whole steps (fwd + bwd calls, events around the step only: the
        dQ kernel may overlap the dK/dV kernel's tail), then the four kernels
        one by one (events between them, which also stops that overlap)."""
        inp, t = prepare(w)
        for _ in range(warmup):
            step_api(w, t)
            flush.fill_(1.0)
        torch.cuda.synchronize()
        step_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        sampler = ClockSampler(local) if sample_clocks else None
        if sampler:
            sampler.__enter__()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for s in range(steps):
            flush.fill_(float(s))  # L2 flush between steps, outside the events
            step_evs[s][0].record(stream)
            step_api(w, t, step_evs[s][1])
            step_evs[s][2].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        if sampler:
            sampler.__exit__(None, None, None)
        for _ in range(warmup):
            step(w, t)
            flush.fill_(1.0)
        torch.cuda.synchronize()
        evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
        for s in range(steps):
            flush.fill_(float(s))
            step(w, t, evsets[s])
        torch.cuda.synchronize()
        status = binding.attn_varlen_get_status()
        if status:
            raise RuntimeError(f"device status word {status}")
        names = ["fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq"]
        per = {n: [] for n in names}
        tot = [ev[0].elapsed_time(ev[2]) for ev in step_evs]
        fwd = [ev[0].elapsed_time(ev[1]) for ev in step_evs]
        bwd = [ev[1].elapsed_time(ev[2]) for ev in step_evs]
        for ev in evsets:
            for i, n in enumerate(names):
                per[n].append(ev[i].elapsed_time(ev[i + 1]))
        pairs = unmasked_pairs(inp.cu_seqlens, w.window_left)
        return {"inp": inp, "t": t, "total_ms": tot, "fwd_ms": fwd, "bwd_ms": bwd, "per_ms": per, "pairs": pairs,
                "wall_s": wall,
                "clocks": sampler.summary() if sampler else None}

    def graph_replay(w, steps, warmup):
        """The step as a training loop records it (research.dws.rip/llm/kernels,
        section 06 and Fig. 8): forward + backward captured once in a CUDA graph
        over a boundary list padded with empty segments to a fixed count (42,
        or the next multiple of 8 when a batch has more segments), then replayed
        on three microbatches with different boundaries.  Every batch's replay
        is compared bit for bit with eager calls on its unpadded boundaries."""
        seeds = [w.doc_seed + i for i in range(3)]
        cus = [synth.pack_microbatch(w.total, w.context, sd, w.cap) for sd in seeds]
        most = max(len(c) - 1 for c in cus)
        nseg = 42 if most <= 42 else -(-most // 8) * 8
        batches = []
        for i, cu in enumerate(cus):
            inp = synth.make_inputs(cu, w.hq, w.hkv, w.d, tensor_seed=w.tensor_seed + 100 + i)
            to = lambda bits: torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(dev)  # noqa: E731
            batches.append({"q": to(inp.q_bits), "k": to(inp.k_bits), "v": to(inp.v_bits), "dout": to(inp.dout_bits),
                            "cu": torch.from_numpy(cu).to(dev),
                            "cu_pad": torch.from_numpy(synth.pad_cu_seqlens(cu, nseg)).to(dev),
                            "pairs": unmasked_pairs(cu, w.window_left)})
        st = {n: torch.empty_like(batches[0][n]) for n in ("q", "k", "v", "dout", "cu_pad")}
        st["out"], st["dq"] = torch.empty_like(st["q"]), torch.empty_like(st["q"])
        st["dk"], st["dv"] = torch.empty_like(st["k"]), torch.empty_like(st["k"])
        st["lse"] = torch.empty(w.hq, w.total, dtype=torch.float32, device=dev)
        ms_, win, sc = w.context, w.window_left, w.softmax_scale

        def load(b):
            for n in ("q", "k", "v", "dout", "cu_pad"):
                st[n].copy_(b[n])

        def rec():
            binding.attn_varlen_fwd(st["q"], st["k"], st["v"], st["cu_pad"], ms_, win, sc, st["out"], st["lse"])
            binding.attn_varlen_bwd(st["dout"], st["q"], st["k"], st["v"], st["out"], st["lse"], st["cu_pad"], ms_,
                                    win, sc, st["dq"], st["dk"], st["dv"])

        side = torch.cuda.Stream()
        side.wait_stream(stream)
        load(batches[0])
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            rec()  # outside capture: the library's per-device set-up happens here
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            rec()
        bit_exact = True
        for b in batches:
            load(b)
            g.replay()
            torch.cuda.synchronize()
            got = [st[n].clone() for n in ("out", "lse", "dq", "dk", "dv")]
            ref = {"out": torch.empty_like(b["q"]), "dq": torch.empty_like(b["q"]), "dk": torch.empty_like(b["k"]),
                   "dv": torch.empty_like(b["k"]), "lse": torch.empty_like(st["lse"])}
            binding.attn_varlen_fwd(b["q"], b["k"], b["v"], b["cu"], ms_, win, sc, ref["out"], ref["lse"])
            binding.attn_varlen_bwd(b["dout"], b["q"], b["k"], b["v"], ref["out"], ref["lse"], b["cu"], ms_, win, sc,
                                    ref["dq"], ref["dk"], ref["dv"])
            torch.cuda.synchronize()
            for x, n in zip(got, ("out", "lse", "dq", "dk", "dv")):
                bit_exact = bit_exact and bool(torch.equal(x, ref[n]))
            del got, ref

        def timed(fn):
            for i in range(warmup):
                load(batches[i % 3])
                fn()
            torch.cuda.synchronize()
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
            for i in range(steps):
                load(batches[i % 3])
                flush.fill_(float(i))
                evs[i][0].record(stream)
                fn()
                evs[i][1].record(stream)
            torch.cuda.synchronize()
            return [e[0].elapsed_time(e[1]) for e in evs]

        replay_ms = timed(g.replay)
        eager_ms = timed(rec)
        status = binding.attn_varlen_get_status()
        del g
        pairs = [b["pairs"] for b in batches]
        mean_pairs = sum(pairs[i % 3] for i in range(steps)) / steps
        res = {"ms": statistics.mean(replay_ms), "eager_ms": statistics.mean(eager_ms),
               "tflops": tflops(w, mean_pairs, statistics.mean(replay_ms)), "pad_segments": nseg,
               "segments": [len(c) - 1 for c in cus], "doc_seeds": seeds, "bit_exact_vs_eager_unpadded": bit_exact,
               "status": status}
        return res

    def layer_leg(w, steps, warmup):
        """One attention layer around the kernels (QKV projection, attention on
        strided views of the fused projection output, output projection,
        loss = sum(y * g), and the whole backward), as the page's Fig. 8 times
        it: eager steps against one CUDA graph replayed, on three microbatches
        with boundaries padded to a fixed count.  The replay is checked bit
        for bit against an eager step on the last batch."""
        from varlen_sliding_window_gb300.layer import AttentionLayer
        cus = [synth.pack_microbatch(w.total, w.context, w.doc_seed + i, w.cap) for i in range(3)]
        most = max(len(c) - 1 for c in cus)
        nseg = 42 if most <= 42 else -(-most // 8) * 8
        d_model = w.hq * w.d
        lay = AttentionLayer(w.total, d_model, w.hq, w.hkv, w.context, w.window_left, nseg, seed=w.tensor_seed)
        gen = torch.Generator(device="cpu").manual_seed(w.tensor_seed + 7)
        lay.x.copy_(torch.randn(w.total, d_model, generator=gen).to(torch.bfloat16))
        lay.g.copy_(torch.randn(w.total, d_model, generator=gen).to(torch.bfloat16))
        pads = [torch.from_numpy(synth.pad_cu_seqlens(c, nseg)).to(dev) for c in cus]
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        lay.cu.copy_(pads[0])
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            lay.step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            lay.step()

        def timed(fn):
            for i in range(warmup):
                lay.cu.copy_(pads[i % 3])
                fn()
            torch.cuda.synchronize()
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
            for i in range(steps):
                lay.cu.copy_(pads[i % 3])
                flush.fill_(float(i))
                evs[i][0].record(stream)
                fn()
                evs[i][1].record(stream)
            torch.cuda.synchronize()
            return statistics.mean(e[0].elapsed_time(e[1]) for e in evs)

        eager_ms = timed(lay.step)
        graph_ms = timed(graph.replay)
        lay.cu.copy_(pads[2])
        graph.replay()
        torch.cuda.synchronize()
        names = ("qkv", "out", "lse", "y", "loss", "d_out", "d_qkv", "dw_qkv", "dw_o", "dx")
        got = {n: getattr(lay, n).clone() for n in names}
        lay.step()
        torch.cuda.synchronize()
        exact = all(torch.equal(got[n], getattr(lay, n)) for n in names)
        gemm_flops = 2.0 * w.total * d_model * ((w.hq + 2 * w.hkv) * w.d) * 3 + 2.0 * w.total * w.hq * w.d * d_model * 3
        del graph, lay
        return {"eager_ms": eager_ms, "graph_ms": graph_ms, "d_model": d_model, "pad_segments": nseg,
                "projection_gflop": gemm_flops / 1e9, "bit_exact_replay_vs_eager": exact,
                "what": "x@W_qkv, attention on strided views of qkv, @W_o, loss=sum(y*g), full backward "
                        "(dW_qkv, dW_o, dx); projections via torch.matmul (cuBLAS)"}

    def tflops(w, pairs, ms):
        return 4.0 * w.d * w.hq * pairs * 3.5 / (ms * 1e-3) / 1e12

    main_res = measure(wl, args.steps, args.warmup, sample_clocks=True)
    step_ms = statistics.mean(main_res["total_ms"])
    value = job_ms_per_microbatch(sum(main_res["total_ms"]), args.steps, world, dev)
    peak_t = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tf = tflops(wl, main_res["pairs"], step_ms)

    def dominant_roofline(w, res):
        """Roofline of the kernel with the largest CUDA-event time in the
        per-kernel run: its credited GEMM units x 2 d Hq pairs, over its mean
        launch time, against the bf16 peak."""
        kern = {n: statistics.mean(v) for n, v in res["per_ms"].items()}
        dom = max(kern, key=kern.get)
        gemm_unit = 2.0 * w.d * w.hq * res["pairs"]
        achieved = KERNEL_UNITS[dom] * gemm_unit / (kern[dom] * 1e-3) / 1e12
        traffic = None
        tpath = os.path.join(ROOT, "profiles", "dram_traffic.json")
        if os.path.exists(tpath):
            try:
                rec = json.load(open(tpath))
                # Counters only count while the kernels are the ones they were taken on.
                if rec.get("csrc_hash") == csrc_hash():
                    traffic = rec.get(w.name, {}).get(dom)
            except Exception:
                traffic = None
        return kern, {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
                      "frac": achieved / peak_t, "traffic": traffic,
                      "peak_source": f"bf16 dense burst, {'of measured' if peak_src == 'measured' else 'of fallback'}"}

    kern_ms, roofline = dominant_roofline(wl, main_res)

    # e2e through the public calls with host buffers and copies in the timed region.
    inp, t = main_res["inp"], main_res["t"]
    pin = {n: t[n].cpu().pin_memory() for n in ("q", "k", "v", "dout", "cu")}
    host_out = {n: torch.empty(t[n].shape, dtype=t[n].dtype).pin_memory() for n in ("out", "lse", "dq", "dk", "dv")}
    h2d = sum(pin[n].numel() * pin[n].element_size() for n in pin)
    d2h = sum(host_out[n].numel() * host_out[n].element_size() for n in host_out)

    def e2e_step():
        for n in pin:
            t[n].copy_(pin[n], non_blocking=True)
        binding.attn_varlen_fwd(t["q"], t["k"], t["v"], t["cu"], wl.context, wl.window_left, wl.softmax_scale,
                                t["out"], t["lse"])
        binding.attn_varlen_bwd(t["dout"], t["q"], t["k"], t["v"], t["out"], t["lse"], t["cu"], wl.context,
                                wl.window_left, wl.softmax_scale, t["dq"], t["dk"], t["dv"])
        for n in host_out:
            host_out[n].copy_(t[n], non_blocking=True)

    for _ in range(max(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_times = []
    for _ in range(args.steps):
        flush.fill_(0.5)
        e_s.record(stream)
        e2e_step()
        e_e.record(stream)
        e_e.synchronize()
        e2e_times.append(e_s.elapsed_time(e_e))
    e2e_serial_ms = statistics.mean(e2e_times)

    # The same steps overlapped the way a training loop overlaps them: while
    # step s computes, step s+1's inputs go up on one copy stream and step
    # s-1's results come down on another.  Every step still copies its own
    # inputs from pinned host memory and reads all of its results back; two
    # device slots of inputs and outputs, events order their reuse.
    ins, outs = ("q", "k", "v", "dout", "cu"), ("out", "lse", "dq", "dk", "dv")
    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
    slots = [{n: torch.empty_like(t[n]) for n in ins + outs} for _ in range(2)]
    host_res = [{n: torch.empty(t[n].shape, dtype=t[n].dtype).pin_memory() for n in outs} for _ in range(2)]
    up_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    down_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_pipelined(nsteps):
        for s in range(nsteps):
            k = s % 2
            d = slots[k]
            with torch.cuda.stream(s_up):
                if s >= 2:
                    s_up.wait_event(comp_done[k])  # step s-2 has read this input slot
                for n in ins:
                    d[n].copy_(pin[n], non_blocking=True)
                up_done[k].record(s_up)
            stream.wait_event(up_done[k])
            if s >= 2:
                stream.wait_event(down_done[k])  # step s-2's results have left this output slot
            binding.attn_varlen_fwd(d["q"], d["k"], d["v"], d["cu"], wl.context, wl.window_left, wl.softmax_scale,
                                    d["out"], d["lse"])
            binding.attn_varlen_bwd(d["dout"], d["q"], d["k"], d["v"], d["out"], d["lse"], d["cu"], wl.context,
                                    wl.window_left, wl.softmax_scale, d["dq"], d["dk"], d["dv"])
            comp_done[k].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(comp_done[k])
                for n in outs:
                    host_res[k][n].copy_(d[n], non_blocking=True)
                down_done[k].record(s_down)
        for k in range(min(2, nsteps)):
            stream.wait_event(down_done[k])

    e2e_pipelined(max(3, args.warmup))
    torch.cuda.synchronize()
    flush.fill_(0.25)
    e_s.record(stream)
    e2e_pipelined(args.steps)
    e_e.record(stream)
    e_e.synchronize()
    e2e_ms = e_s.elapsed_time(e_e) / args.steps
    for k in range(2):  # the results that came back are the device's
        for n in outs:
            assert torch.equal(host_res[k][n], slots[k][n].cpu()), n

    # Spread over document seeds 0-4 of the same workload recipe (the
    # headline is seed 0): step ms and counted TFLOP/s per seed.
    import dataclasses
    spread = []
    for sd in range(5):
        w_s = dataclasses.replace(wl, doc_seed=sd)
        r = measure(w_s, max(5, args.steps // 2), 3)
        ms_s = statistics.mean(r["total_ms"])
        spread.append({"doc_seed": sd, "segments": int(len(r["inp"].cu_seqlens) - 1), "pairs": r["pairs"],
                       "ms": ms_s, "tflops": tflops(w_s, r["pairs"], ms_s)})
        del r
    sm_mhz = (main_res["clocks"] or {}).get("sm_mhz")
    peak_hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    graph_main = graph_replay(wl, args.steps, args.warmup)
    layer_main = layer_leg(wl, args.steps, args.warmup)
    also = {}
    for name in [x for x in args.also.split(",") if x]:
        w2 = wls[name]
        r = measure(w2, max(5, args.steps // 2), 3)
        ms2 = statistics.mean(r["total_ms"])
        k2, rl2 = dominant_roofline(w2, r)
        also[name] = {"ms": ms2, "tflops": tflops(w2, r["pairs"], ms2), "frac": tflops(w2, r["pairs"], ms2) / peak_t,
                      "fwd_ms": statistics.mean(r["fwd_ms"]), "bwd_ms": statistics.mean(r["bwd_ms"]),
                      "pairs": r["pairs"], "segments": int(len(r["inp"].cu_seqlens) - 1),
                      "kernel_ms": k2, "roofline": rl2,
                      "roofs": roofs(w2, r["pairs"], ms2, peak_t, peak_hbm, sm_mhz)}
        if w2.name in PAGE_FA2_MS:
            also[name]["page_context"] = {"fa2_ms": PAGE_FA2_MS[w2.name], "ratio": ms2 / PAGE_FA2_MS[w2.name]}
        del r
        also[name]["graph"] = graph_replay(w2, max(6, args.steps // 2), 3)
    # The context sweep (research.dws.rip/llm/kernels, section 02, Figs. 3
    # and 4) and the long-context case: step and per-kernel times.
    sweep = {}
    for name in [x for x in args.sweep.split(",") if x]:
        w2 = wls[name]
        r = measure(w2, max(5, args.steps // 2), 3)
        ms2 = statistics.mean(r["total_ms"])
        k2, rl2 = dominant_roofline(w2, r)
        sweep[name] = {"ms": ms2, "tflops": tflops(w2, r["pairs"], ms2), "frac": tflops(w2, r["pairs"], ms2) / peak_t,
                       "fwd_ms": statistics.mean(r["fwd_ms"]), "bwd_ms": statistics.mean(r["bwd_ms"]),
                       "pairs": r["pairs"], "segments": int(len(r["inp"].cu_seqlens) - 1), "tokens": w2.total,
                       "context": w2.context, "window_left": w2.window_left, "hq": w2.hq, "hkv": w2.hkv,
                       "kernel_ms": k2, "dominant": {"kernel": rl2["kernel"], "frac": rl2["frac"]}}
        if w2.name in PAGE_FA2_MS:
            sweep[name]["page_context"] = {"fa2_ms": PAGE_FA2_MS[w2.name], "ratio": ms2 / PAGE_FA2_MS[w2.name]}
        del r
    if sweep:
        also["sweep"] = sweep

    def gdn_leg(gw, steps, warmup):
        """The Gated DeltaNet local layer (include/gdn_varlen.h) on one packed
        microbatch: the forward and the backward call each timed with CUDA
        events on the stream, L2 flushed between steps; FLOPs as the kernels
        perform them (gdn_flops), HBM bytes as the inputs and outputs of each
        call."""
        gi = gw.inputs()
        to = lambda bits: torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(dev)  # noqa: E731
        q, k, v, do = (to(b) for b in (gi.q_bits, gi.k_bits, gi.v_bits, gi.do_bits))
        g_ = torch.from_numpy(gi.g).to(dev)
        be = torch.from_numpy(gi.beta).to(dev)
        cu = torch.from_numpy(gi.cu_seqlens).to(dev)
        nseg = len(gi.cu_seqlens) - 1
        o = torch.empty_like(q)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dg, db = torch.empty_like(g_), torch.empty_like(be)
        # Kimi Delta (a decay per key channel) or Gated DeltaNet: the same calls' shapes
        f_fwd, f_bwd, f_ws = ((binding.kda_varlen_fwd, binding.kda_varlen_bwd, binding.kda_varlen_bwd_workspace_bytes)
                              if gw.per_channel else
                              (binding.gdn_varlen_fwd, binding.gdn_varlen_bwd, binding.gdn_varlen_bwd_workspace_bytes))
        ws = torch.empty(f_ws(gw.total, gw.nh, nseg), dtype=torch.uint8, device=dev)
        fwd = lambda: f_fwd(q, k, v, g_, be, cu, gw.scale, o, ws)  # noqa: E731
        bwd = lambda: f_bwd(q, k, v, g_, be, do, cu, gw.scale, dq, dk, dv, dg, db, ws)  # noqa: E731

        def timed(fwd, bwd):
            for _ in range(warmup):
                fwd()
                bwd()
                flush.fill_(1.0)
            torch.cuda.synchronize()
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
            for i in range(steps):
                flush.fill_(float(i))
                evs[i][0].record(stream)
                fwd()
                evs[i][1].record(stream)
                flush.fill_(float(i) + 0.5)
                evs[i][2].record(stream)
                bwd()
                evs[i][3].record(stream)
            torch.cuda.synchronize()
            return (statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
                    statistics.mean(e[2].elapsed_time(e[3]) for e in evs))

        f_ms, b_ms = timed(fwd, bwd)
        # The training pair that keeps the forward's factors, states and E for
        # the backward (the *_fwd_save / *_bwd_saved calls), on the same
        # workspace: its times, and its outputs against the pair above, bit for bit.
        ref_plain = [x.clone() for x in (o, dq, dk, dv, dg, db)]
        f_save, f_saved = ((binding.kda_varlen_fwd_save, binding.kda_varlen_bwd_saved) if gw.per_channel else
                           (binding.gdn_varlen_fwd_save, binding.gdn_varlen_bwd_saved))
        fs_ms, bs_ms = timed(lambda: f_save(q, k, v, g_, be, cu, gw.scale, o, ws),
                             lambda: f_saved(q, k, v, g_, be, do, cu, gw.scale, dq, dk, dv, dg, db, ws))
        saved_res = {"fwd_ms": fs_ms, "bwd_ms": bs_ms, "step_ms": fs_ms + bs_ms,
                     "page_ratio": ((fs_ms + bs_ms) / (PAGE_KDA_MS if gw.per_channel else PAGE_GDN_MS)
                                    if gw.context == 4096 else None),
                     "bit_exact_vs_recomputing": all(torch.equal(a, b)
                                                     for a, b in zip(ref_plain, (o, dq, dk, dv, dg, db)))}
        # The same step captured in a CUDA graph over the boundary list padded
        # with empty segments to 42 (the page replays these layers too, section
        # 06): replay time, and its outputs against the eager step's bits.
        graph_res = None
        if nseg <= 42:
            ref = [x.clone() for x in (o, dq, dk, dv, dg, db)]
            cu_pad = torch.from_numpy(synth.pad_cu_seqlens(gi.cu_seqlens, 42)).to(dev)
            ws_pad = torch.empty(f_ws(gw.total, gw.nh, 42), dtype=torch.uint8, device=dev)

            def padded():
                f_fwd(q, k, v, g_, be, cu_pad, gw.scale, o, ws_pad)
                f_bwd(q, k, v, g_, be, do, cu_pad, gw.scale, dq, dk, dv, dg, db, ws_pad)

            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                padded()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                padded()
            graph.replay()
            torch.cuda.synchronize()
            exact = all(torch.equal(a, b) for a, b in zip(ref, (o, dq, dk, dv, dg, db)))
            gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
            for i in range(steps):
                flush.fill_(float(i))
                gev[i][0].record(stream)
                graph.replay()
                gev[i][1].record(stream)
            torch.cuda.synchronize()
            graph_res = {"ms": statistics.mean(e[0].elapsed_time(e[1]) for e in gev), "eager_ms": f_ms + b_ms,
                         "pad_segments": 42, "bit_exact_vs_eager_unpadded": exact}
            del graph, ws_pad
        status = binding.attn_varlen_get_status()
        ff, fb = gdn_flops(gi.cu_seqlens, gw.nh, gw.d, gw.per_channel)
        tok = gw.total * gw.nh * gw.d * 2
        gates = gw.total * gw.nh * 4 * (gw.d if gw.per_channel else 1)
        bytes_f = 4 * tok + 2 * gates            # q, k, v in, o out; g, beta
        bytes_b = 7 * tok + 4 * gates            # q, k, v, d_o in; dq, dk, dv out; g, beta in; dg, dbeta out
        tf_f, tf_b = ff / (f_ms * 1e-3) / 1e12, fb / (b_ms * 1e-3) / 1e12
        dom = "bwd" if b_ms >= f_ms else "fwd"
        layer, page_ms = ("Kimi Delta", PAGE_KDA_MS) if gw.per_channel else ("Gated DeltaNet", PAGE_GDN_MS)
        ach = tf_b if dom == "bwd" else tf_f
        mhz_g = sm_mhz or 2032.0
        mma_sync_peak = 2 * MMA_SYNC_FMA_PER_CLK_SM * NUM_SMS * mhz_g * 1e6 / 1e12
        del ws
        return {"fwd_ms": f_ms, "bwd_ms": b_ms, "step_ms": f_ms + b_ms, "segments": nseg, "tokens": gw.total,
                "heads": gw.nh, "gflop_fwd": ff / 1e9, "gflop_bwd": fb / 1e9, "tflops_fwd": tf_f, "tflops_bwd": tf_b,
                "hbm_gbs_fwd": bytes_f / (f_ms * 1e-3) / 1e9, "hbm_gbs_bwd": bytes_b / (b_ms * 1e-3) / 1e9,
                "roofline": {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak_t, "unit": "TFLOP/s",
                             "frac": ach / peak_t, "traffic": None,
                             "peak_source": f"bf16 dense burst, {'of measured' if peak_src == 'measured' else 'of fallback'}",
                             "note": "warp-level mma.sync bf16 products; the peak is the tcgen05/cuBLAS one",
                             "mma_sync": {"peak": mma_sync_peak, "frac": ach / mma_sync_peak,
                                          "peak_basis": f"{MMA_SYNC_FMA_PER_CLK_SM:g} FMA/clk/SM x 2 x {NUM_SMS} "
                                                        f"SMs x {mhz_g:g} MHz (measured instruction rate)"}},
                "page_context": ({"page_ms": page_ms, "ratio": (f_ms + b_ms) / page_ms,
                                  "what": f"the page's {layer} layer fwd+bwd per step at context 4,096 on its "
                                          "own unnamed GPU (research.dws.rip/llm/kernels, Fig. 5)"}
                                 if gw.context == 4096 else None),
                "graph": graph_res,
                "saved": saved_res,
                "status": status}

    gdn = {}
    gwls = {**synth.gdn_workloads(), **synth.kda_workloads()}
    for name in [x for x in args.gdn.split(",") if x]:
        gdn[name] = gdn_leg(gwls[name], max(5, args.steps // 2), 3)
    if gdn:
        also["gdn"] = gdn

    line = None
    if rank == 0:
        cpu_ms, sample, cores = oracle_time(inp, wl.window_left, wl.softmax_scale, args.cpu_budget)
        line = {
            "metric": METRIC, "value": value, "unit": "ms", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None,
            "page_context": ({"fa2_ms": PAGE_FA2_MS[wl.name], "ratio": value / PAGE_FA2_MS[wl.name],
                              "what": "the page's FlashAttention-2 fwd+bwd per layer on its own unnamed, "
                                      "clock-capped GPU (research.dws.rip/llm/kernels, Figs. 3 and 4)"}
                             if wl.name in PAGE_FA2_MS else None),
            "dtype": "bf16", "data": "synthetic",
            "config": workload_config(wl, inp.cu_seqlens, main_res["pairs"], world),
            "tflops": tf, "pct_of_bf16_peak": 100.0 * tf / peak_t,
            "fwd_ms": statistics.mean(main_res["fwd_ms"]), "bwd_ms": statistics.mean(main_res["bwd_ms"]),
            "kernel_ms": kern_ms,
            "roofs": roofs(wl, main_res["pairs"], step_ms, peak_t, peak_hbm, sm_mhz),
            "seed_spread": spread,
            "graph": graph_main,
            "layer": layer_main,
            "roofline": roofline,
            "cpu_baseline": {"value": cpu_ms, "unit": "ms", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps_overlapped": True, "serial_ms": e2e_serial_ms,
                    "how": "attn_varlen_fwd + attn_varlen_bwd per step, inputs copied up from pinned host memory "
                           "and all five results copied back every step; copies of neighbouring steps overlap "
                           "the compute on two copy streams (serial_ms: one step at a time)"},
            "gpu_launches": KERNELS_PER_STEP * args.steps,
            "clocks": main_res["clocks"],
            "also": also,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
