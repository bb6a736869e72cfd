"""Benchmark of the channelwise gated delta rule hot path on one GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * one decode step at B=64, H=32, dk=dv=128 (bf16 q/k/v, fp32 per-channel
    log-decay, fp32 state of 134 MB carried from step to step), and
  * one chunked prefill at B=1, H=32, dk=dv=128, T=4000, chunk 64 (zero
    initial state).
The L2 cache (129 MB) is flushed before every kernel, outside the timed
brackets: a 256 MiB buffer is written and then read back, so the kernel starts
with no data of its own in L2 and no dirty lines of the flush left to write
back during its run; kernels are timed with CUDA events on the stream they
run on.

Headline value: decode state GB/s = 2*B*H*dk*dv*4 bytes per step / decode
time, sustained: back-to-back decode steps rotating over three distinct
134 MB states (402 MB, larger than L2), so that no step finds its state in L2
and the write-back of one step's dirty lines is paid inside the next step.
The per-launch time after an L2 flush (median) is reported beside it.  The
prefill rate (tokens/s, o in bf16 as a bf16 model runs it) is reported beside
it too.  `roofline` is for the kernel with the larger share of the step (the
prefill kernel); the decode kernel's roofline is under `decode_roofline`.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas, weak scaling, no collective on the data path); the step time is
the max over ranks.  `--impl reference` times the fp64 CPU oracle instead,
on rank 0 only.
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

METRIC = "decode state GB/s (% HBM peak) at B=64; prefill tokens/s at T=4000, 32 heads"
DEC = dict(B=64, H=32, dk=128, dv=128)
PRE = dict(B=1, H=32, T=4000, dk=128, dv=128, chunk=64)
DEC_STATE_BYTES = 2 * DEC["B"] * DEC["H"] * DEC["dk"] * DEC["dv"] * 4           # 268,435,456
# prefill algorithmic bytes: q,k,v bf16 + g fp32 + beta fp32 + o + state in and out fp32;
# o in bf16 (the timed configuration) or fp32 (reported beside it)
def prefill_bytes(B, T, H, o_bytes):
    return B * T * H * (3 * 128 * 2 + 128 * 4 + 4 + 128 * o_bytes) + 2 * B * H * 128 * 128 * 4


PRE_BYTES = prefill_bytes(PRE["B"], PRE["T"], PRE["H"], 2)                        # 201,314,304
PRE_BYTES_F32O = prefill_bytes(PRE["B"], PRE["T"], PRE["H"], 4)                   # 234,082,304
# prefill tensor flops per token-head: 10*C*d (intra-chunk) + 6*dk*dv (carry)
PRE_FLOPS = PRE["B"] * PRE["T"] * PRE["H"] * (10 * PRE["chunk"] * 128 + 6 * 128 * 128)
L2_FLUSH_BYTES = 256 << 20
# kernel name and the sources that define it, per prefill path (1 = per head, 2 = cluster, 5 = cooperative)
PREFILL_KERNELS = {1: ("prefill_tc05_kernel", ["prefill_tc05.cu", "prefill_tc05_chunk.cuh", "tc05.cuh"]),
                   2: ("prefill_cluster_kernel", ["prefill_cluster.cu", "prefill_tc05_chunk.cuh", "tc05.cuh"]),
                   5: ("prefill_coop_kernel", ["prefill_cluster.cu", "prefill_tc05_chunk.cuh", "tc05.cuh"])}
DECODE_KERNEL = ("decode_kernel", ["decode.cu", "cgdr_internal.cuh"])


def bench_config(world):
    """The workload both arms report (the reference arm times bounded samples of it)."""
    return {"workload": "decode_b64 + prefill_t4000",
            "decode": {"B": 64, "H": 32, "dk": 128, "dv": 128, "state": "fp32", "inputs": "bf16",
                       "gate": "per-channel fp32"},
            "prefill": {"B": 1, "H": 32, "T": 4000, "dk": 128, "dv": 128, "chunk": 64, "inputs": "bf16",
                        "o": "bf16"},
            "l2": "decode (headline): inputs larger than L2 (three 134 MB states in rotation, back to back); "
                  "per-launch decode and prefill: L2 flushed before every kernel (256 MiB written, then read "
                  "back), outside the timed brackets",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def max_over_ranks(values, world, device):
    """The element-wise max over ranks of this rank's timing totals (one all_reduce)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_rates(dec_total_ms, pre_total_ms, world, steps):
    """Whole-job rates from the slowest rank's totals: every rank runs the same
    workload on its own GPU (replicas, weak scaling), so the job moves `world`
    times one rank's state bytes and tokens in the slowest rank's time."""
    dec_gbs = world * steps * DEC_STATE_BYTES / (dec_total_ms / 1e3) / 1e9
    pre_tps = world * steps * PRE["B"] * PRE["T"] / (pre_total_ms / 1e3)
    return dec_gbs, pre_tps


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def sources_sha256(sources) -> str:
    """sha256 of the concatenated kernel sources (csrc/), in the order listed."""
    h = hashlib.sha256()
    for src in sources:
        with open(os.path.join(ROOT, "gated_delta_rule_channelwise_gb300", "csrc", src), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _traffic(kernel: str, sources):
    """DRAM bytes per launch from the committed ncu summary, if it is for these sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        sha = sources_sha256(sources)
        for line in open(path):
            kv = dict(x.split("=", 1) for x in line.split() if "=" in x)
            if kv.get("kernel") == kernel and kv.get("source_sha256") == sha:
                return int(kv["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = os.path.join("/tmp", "cgdr_clocks_%d.csv" % os.getpid())
        try:
            import torch
            bus = torch.cuda.get_device_properties(device_index).pci_bus_id
            sel = ["-i", "%04x:%02x:%02x.0" % (torch.cuda.get_device_properties(device_index).pci_domain_id, bus,
                                                torch.cuda.get_device_properties(device_index).pci_device_id)]
        except Exception:
            sel = ["-i", str(device_index)]
        self.cmd = ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits", "-lms", "100", *sel]

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(self.cmd, stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, x in enumerate(r) if x.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import gated_delta_rule_channelwise_gb300 as cg
    from gated_delta_rule_channelwise_gb300 import build as cbuild
    from gated_delta_rule_channelwise_gb300.synth import WORKLOADS, make_inputs

    if rank == 0 or world == 1:
        cbuild.build()
    if world > 1:
        dist.barrier()
    cbuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()

    # ---- resident inputs
    wd, wp = WORKLOADS["decode_b64"], WORKLOADS["prefill_t4000"]
    dsteps = 16                                   # distinct decode inputs, cycled
    dinp = make_inputs(wd, T=dsteps, device=dev, seed=wd.seed + 97 * rank)
    dstate = dinp["S0"].clone()
    dstates = [dstate, dinp["S0"].clone(), dinp["S0"].clone()]    # 3 x 134 MB, rotated back to back
    dout = torch.empty(DEC["B"], DEC["H"], DEC["dv"], dtype=torch.float32, device=dev)
    pinp = make_inputs(wp, device=dev, seed=wp.seed + 97 * rank)
    pstate = torch.zeros_like(pinp["S0"])
    pout = torch.empty(pinp["v"].shape, dtype=torch.bfloat16, device=dev)
    pkw = dict(g=pinp["g"], beta=pinp["beta"], chunk=64)
    pws = torch.empty(max(1, cg.prefill_workspace_size(pinp["q"], pinp["k"], pinp["v"], pstate, pout, **pkw)),
                      dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()                         # write > L2 ...
        torch.sum(flush, dim=0, out=sink)     # ... then read it back: L2 holds clean flush lines only
        # ~100 us of GPU-side spin after the flush: the next launch is queued behind it before the
        # GPU reaches the start event, so host-side marshalling never falls inside a timed interval
        torch.cuda._sleep(200000)

    def decode(i, state=dstate):
        t = i % dsteps
        cg.decode(dinp["q"][:, t], dinp["k"][:, t], dinp["v"][:, t], state, dout,
                  g=dinp["g"][:, t], beta=dinp["beta"][:, t])

    def prefill():
        cg.prefill(pinp["q"], pinp["k"], pinp["v"], pstate, pout, workspace=pws, **pkw)

    pre_path = cg.prefill_path_for(pinp["q"], pinp["k"], pinp["v"], pstate, pout, **pkw)
    pre_kernel = PREFILL_KERNELS[pre_path]
    K = args.steps
    NS = max(64, K)                               # sustained back-to-back decode steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    es0, es1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the clock sampler runs from before the warm-up, so that its start-up pause is not an idle gap
    # between the warm-up and the timed launches
    with ClockSampler(local_rank) as clk:
        for i in range(args.warmup):
            flush_l2(); decode(i); flush_l2(); pstate.zero_(); prefill()
        for i in range(3):
            decode(i, dstates[i % 3])
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for i in range(K):
            flush_l2()
            ev[i][0].record(stream); decode(i); ev[i][1].record(stream)
            flush_l2()
            pstate.zero_()
            ev[i][2].record(stream)
            prefill()
            ev[i][3].record(stream)
        es0.record(stream)
        for i in range(NS):
            decode(i, dstates[i % 3])
        es1.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    dec_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    pre_ms = [ev[i][2].elapsed_time(ev[i][3]) for i in range(K)]
    sus_ms = es0.elapsed_time(es1)
    dec_total, pre_total, sus_total = max_over_ranks([sum(dec_ms), sum(pre_ms), sus_ms], world, dev)

    # ---- end to end: host (pinned) buffers, copies inside the timed region
    e2e = run_e2e(args, cg, dinp, dstate, pinp, dev, stream, world)
    secondary = run_secondary(cg, dev, stream, flush_l2) if (rank == 0 and not args.no_secondary) else None

    if rank != 0:
        return None
    hbm, tflops, peak_kind = _peaks()
    sus_step_s = sus_total / NS / 1e3
    dec_gbs = world * DEC_STATE_BYTES / sus_step_s / 1e9              # whole job, sustained
    _, pre_tps = job_rates(dec_total, pre_total, world, K)
    dec_launch_s = statistics.median(dec_ms) / 1e3
    pre_launch_s = statistics.median(pre_ms) / 1e3
    pre_ach = PRE_BYTES / pre_launch_s / 1e9
    dec_ach_flushed = DEC_STATE_BYTES / dec_launch_s / 1e9
    dec_ach_sus = DEC_STATE_BYTES / sus_step_s / 1e9
    tr_pre = _traffic(*pre_kernel)
    tr_dec = _traffic(*DECODE_KERNEL)
    out = {
        "metric": METRIC, "value": round(dec_gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(sus_step_s * 1e3 + pre_total / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "dtype_note": "bf16 q/k/v inputs; fp32 state, gates and accumulation; the prefill's tensor-core "
                      "operands are TF32 (anchored causal terms) and fp16 (the other products, range-checked)",
        "config": bench_config(world),
        "pct_hbm_peak": round(100.0 * dec_gbs / world / hbm, 2),
        "prefill": {"metric": "prefill tokens/s at T=4000, 32 heads", "value": round(pre_tps, 1),
                    "unit": "tokens/s", "ms_per_launch_median": round(pre_launch_s * 1e3, 5),
                    "ms_per_launch_mean": round(statistics.mean(pre_ms), 5), "o_dtype": "bf16",
                    "kernel": pre_kernel[0]},
        "decode": {"ms_per_step_sustained": round(sus_step_s * 1e3, 5), "sustained_steps": NS,
                   "ms_per_launch_flushed_median": round(dec_launch_s * 1e3, 5),
                   "ms_per_launch_flushed_mean": round(statistics.mean(dec_ms), 5)},
        "roofline": {"kernel": pre_kernel[0], "bound": "hbm", "achieved": round(pre_ach, 2), "peak": hbm,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(pre_ach / hbm, 4),
                     "traffic": tr_pre, "algorithmic_bytes": PRE_BYTES, "o_dtype": "bf16",
                     "time": "median per-launch CUDA-event time after an L2 flush",
                     "tensor_flops": PRE_FLOPS, "tensor_frac": round(PRE_FLOPS / pre_launch_s / 1e12 / tflops, 4)},
        "decode_roofline": {"kernel": "decode_kernel", "bound": "hbm", "achieved": round(dec_ach_sus, 2),
                            "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(dec_ach_sus / hbm, 4),
                            "time": "sustained: %d back-to-back steps over three rotating states" % NS,
                            "achieved_flushed": round(dec_ach_flushed, 2),
                            "frac_flushed": round(dec_ach_flushed / hbm, 4),
                            "traffic": tr_dec, "algorithmic_bytes": DEC_STATE_BYTES},
        "e2e": e2e,
        "secondary": secondary,
        "gpu_launches": 2 * K + NS,
        "wall_s_timed_region": round(t_wall, 3),
    }
    out["clocks"] = clk.summary()
    return out


def run_secondary(cg, dev, stream, flush_l2):
    """The other workloads, timed once each: the fused GatedDeltaNet decode at B=1
    (256 steps, eager and as one CUDA graph) and the long prefill (B=4, T=16411)."""
    import torch
    from gated_delta_rule_channelwise_gb300.synth import WORKLOADS, Workload, gate_kwargs, make_inputs
    out = {}
    w = WORKLOADS["gdn_decode_b1"]
    inp = make_inputs(w, device=dev)
    st = inp["S0"].clone()
    o = torch.empty(w.T, 1, w.Hv, w.dv, dtype=torch.float32, device=dev)

    def steps():
        for t in range(w.T):
            cg.decode(inp["q"][:, t], inp["k"][:, t], inp["v"][:, t], st, o[t], a=inp["a"][:, t], b=inp["b"][:, t],
                      A_log=inp["A_log"], dt_bias=inp["dt_bias"])

    steps()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream); steps(); e1.record(stream); torch.cuda.synchronize()
    eager_us = e0.elapsed_time(e1) * 1e3 / w.T
    graph_us = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            steps()
        g.replay(); torch.cuda.synchronize()
        e0.record(stream); g.replay(); e1.record(stream); torch.cuda.synchronize()
        graph_us = e0.elapsed_time(e1) * 1e3 / w.T
    except Exception as exc:  # pragma: no cover - reported, not hidden
        graph_us = "capture failed: %s" % exc
    state_bytes = 2 * w.B * w.Hv * w.dk * w.dv * 4
    out["gdn_decode_b1"] = {"workload": "fused GatedDeltaNet decode B=1, 16 k-heads -> 32 v-heads, packed bf16 qkv",
                            "us_per_step_eager": round(eager_us, 3),
                            "us_per_step_cuda_graph": round(graph_us, 3) if isinstance(graph_us, float) else graph_us,
                            "state_bytes_per_step": state_bytes, "steps": w.T,
                            "note": "the 4.2 MB state stays resident in the 129 MB L2 from step to step: "
                                    "these are L2 rates, not HBM rates"}
    del inp, st, o
    hbm, _, _ = _peaks()

    def time_prefill(inp, st, o, path):
        ws = torch.empty(max(1, cg.prefill_workspace_size(inp["q"], inp["k"], inp["v"], st, o, chunk=64, path=path,
                                                          **gate_kwargs(inp))), dtype=torch.uint8, device=dev)
        ms = []
        for _ in range(3):
            st.copy_(inp["S0"])
            flush_l2()
            e0.record(stream)
            cg.prefill(inp["q"], inp["k"], inp["v"], st, o, chunk=64, path=path, workspace=ws, **gate_kwargs(inp))
            e1.record(stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        return round(min(ms[1:]), 4)

    w = WORKLOADS["prefill_long"]
    inp = make_inputs(w, device=dev)
    st = torch.empty_like(inp["S0"])
    o = torch.empty(inp["v"].shape, dtype=torch.bfloat16, device=dev)
    o32 = torch.empty(inp["v"].shape, dtype=torch.float32, device=dev)
    t = time_prefill(inp, st, o, cg.PREFILL_AUTO)
    nbytes = prefill_bytes(w.B, w.T, w.Hv, 2)
    out["prefill_long"] = {"workload": "prefill B=4 H=32 T=16411 chunk 64, g = -softplus(N(1,1)), o bf16",
                           "ms_per_launch": t, "tokens_per_s": round(w.B * w.T / (t / 1e3), 1),
                           "algorithmic_bytes": nbytes, "roofline_frac": round(nbytes / (t / 1e3) / 1e9 / hbm, 4),
                           "ms_per_launch_cluster_kernel": time_prefill(inp, st, o, cg.PREFILL_CLUSTER),
                           "ms_per_launch_per_head_kernel": time_prefill(inp, st, o, cg.PREFILL_PER_HEAD),
                           "ms_per_launch_o_fp32": time_prefill(inp, st, o32, cg.PREFILL_AUTO),
                           "algorithmic_bytes_o_fp32": prefill_bytes(w.B, w.T, w.Hv, 4)}
    del inp, st, o, o32
    w = WORKLOADS["prefill_t4000"]
    inp = make_inputs(w, device=dev)
    st = torch.empty_like(inp["S0"])
    o = torch.empty(inp["v"].shape, dtype=torch.bfloat16, device=dev)
    o32 = torch.empty(inp["v"].shape, dtype=torch.float32, device=dev)
    out["prefill_t4000_by_kernel"] = {"o": "bf16",
                                      "ms_per_launch_coop_kernel": time_prefill(inp, st, o, cg.PREFILL_COOP),
                                      "ms_per_launch_cluster_kernel": time_prefill(inp, st, o, cg.PREFILL_CLUSTER),
                                      "ms_per_launch_per_head_kernel": time_prefill(inp, st, o, cg.PREFILL_PER_HEAD),
                                      "ms_per_launch_o_fp32": time_prefill(inp, st, o32, cg.PREFILL_AUTO),
                                      "algorithmic_bytes_o_fp32": PRE_BYTES_F32O}
    del o32
    del inp, st, o
    # prefill over a range of lengths and batches (same shapes and distributions as the T = 4000
    # workload), by the kernel the library picks; small T at B = 64 also by the chunked kernel, and
    # B = 2, 3 (64 and 96 heads: two and three waves of clusters) by both tensor-core kernels
    sweep = {}
    for B, T in ((1, 8), (1, 16), (1, 128), (1, 512), (1, 4000), (2, 4000), (3, 4000), (64, 2), (64, 4), (64, 8)):
        wl = Workload("sweep", B=B, Hk=32, Hv=32, dk=128, dv=128, T=T, dtype="bf16", gate="channel",
                      s0_std=0.0, seed=5000 + T)
        inp = make_inputs(wl, device=dev)
        st = torch.empty_like(inp["S0"])
        o = torch.empty(inp["v"].shape, dtype=torch.bfloat16, device=dev)
        key = "B%d_T%d" % (B, T)
        pth = cg.prefill_path_for(inp["q"], inp["k"], inp["v"], st, o, chunk=64, **gate_kwargs(inp))
        t_auto = time_prefill(inp, st, o, cg.PREFILL_AUTO)
        sweep[key] = {"kernel": {cg.PREFILL_PER_HEAD: "per_head", cg.PREFILL_CLUSTER: "cluster",
                                 cg.PREFILL_SIMT: "simt", cg.PREFILL_RECURRENT: "recurrent",
                                 cg.PREFILL_COOP: "coop"}.get(pth, str(pth)),
                      "ms": t_auto, "tokens_per_s": round(B * T / (t_auto / 1e3), 1)}
        if pth == cg.PREFILL_RECURRENT:
            sweep[key]["ms_chunked_per_head"] = time_prefill(inp, st, o, cg.PREFILL_PER_HEAD)
        elif B > 1:
            sweep[key]["ms_per_head"] = time_prefill(inp, st, o, cg.PREFILL_PER_HEAD)
            sweep[key]["ms_cluster"] = time_prefill(inp, st, o, cg.PREFILL_CLUSTER)
            sweep[key]["ms_coop"] = time_prefill(inp, st, o, cg.PREFILL_COOP)
        del inp, st, o
    out["prefill_sweep"] = sweep
    torch.cuda.empty_cache()
    return out


def run_e2e(args, cg, dinp, dstate, pinp, dev, stream, world):
    """Decode and prefill through the public API with pinned host inputs and outputs.

    Every step copies its inputs host -> device and its output device -> host
    inside the timed region.  The copies run on two streams of their own, double
    buffered, so that step i+1's inputs go in and step i's output comes back while
    the GPU computes (the state is carried on the device from step to step).  The
    headline replays a run of such steps from one CUDA graph (the host issues one
    launch for many steps); the same steps issued call by call from Python are
    reported beside it."""
    import torch
    K = max(3, min(args.steps, 200))

    def packed(tensors, device):
        """One buffer (pinned on the host) holding all the tensors, and views of it in their shapes."""
        offs, n = [], 0
        for x in tensors.values():
            offs.append(n)
            n += (x.numel() * x.element_size() + 255) // 256 * 256
        buf = torch.empty(n, dtype=torch.uint8, device=device)
        if device == "cpu":
            buf = buf.pin_memory()
        views = {k: buf[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
                 for (k, x), o in zip(tensors.items(), offs)}
        return buf, views

    def pipeline(host_in, out_like, compute, cs):
        """A runner of n steps: copy in (s_in) -> compute (cs) -> copy out (s_out), two slots.
        The inputs travel as one packed copy.  Every event a run waits on is recorded inside the
        run, so the same runner can be captured into a CUDA graph on cs."""
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        hbuf, hviews = packed(host_in, "cpu")
        for k, x in host_in.items():
            hviews[k].copy_(x)
        dev_in = [packed(host_in, dev) for _ in range(2)]
        dev_out = [torch.empty_like(out_like, device=dev) for _ in range(2)]
        host_out = [torch.empty_like(out_like).pin_memory() for _ in range(2)]
        in_ready, in_free, out_ready, out_free = ([torch.cuda.Event() for _ in range(2)] for _ in range(4))

        def run(n):
            for e in in_free + out_free:                       # everything before the run is done with both slots
                e.record(cs)
            for i in range(n):
                j = i & 1
                s_in.wait_event(in_free[j])                    # step i-2 has finished reading slot j
                with torch.cuda.stream(s_in):
                    dev_in[j][0].copy_(hbuf, non_blocking=True)
                in_ready[j].record(s_in)
                cs.wait_event(in_ready[j])
                cs.wait_event(out_free[j])                     # step i-2's output has left slot j
                with torch.cuda.stream(cs):
                    compute(dev_in[j][1], dev_out[j])
                in_free[j].record(cs)
                out_ready[j].record(cs)
                s_out.wait_event(out_ready[j])
                with torch.cuda.stream(s_out):
                    host_out[j].copy_(dev_out[j], non_blocking=True)
                out_free[j].record(s_out)
            cs.wait_event(out_free[(n - 1) & 1])               # the last output is on the host
        return run

    def graphed(host_in, out_like, compute, n_steps):
        """The same pipeline captured as one CUDA graph of n_steps steps; returns a replay function."""
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        run = pipeline(host_in, out_like, compute, cap)
        run(2)                                                 # eager once: per-device set-up outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            run(n_steps)
        graph.replay()
        torch.cuda.synchronize()
        return graph.replay

    def timed(fn, n_calls, steps_per_call):
        fn()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(n_calls):
            fn()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / (n_calls * steps_per_call)

    # decode: q, k, v, g, beta in, o out
    h = {k: dinp[k][:, 0].contiguous().cpu().pin_memory() for k in ("q", "k", "v", "g", "beta")}
    o_like = torch.empty(DEC["B"], DEC["H"], DEC["dv"], dtype=torch.float32)
    h2d_dec = sum(x.numel() * x.element_size() for x in h.values())
    d2h_dec = o_like.numel() * o_like.element_size()

    def dcompute(d, o):
        cg.decode(d["q"], d["k"], d["v"], dstate, o, g=d["g"], beta=d["beta"])

    # prefill: q, k, v, g, beta in, o out (zero initial state each step, as in the timed kernel)
    hp = {k: pinp[k].contiguous().cpu().pin_memory() for k in ("q", "k", "v", "g", "beta")}
    po_like = torch.empty(pinp["v"].shape, dtype=torch.bfloat16)
    ps = torch.zeros_like(pinp["S0"])
    h2d_pre = sum(x.numel() * x.element_size() for x in hp.values())
    d2h_pre = po_like.numel() * po_like.element_size()
    ws = torch.empty(max(1, cg.prefill_workspace_size(pinp["q"], pinp["k"], pinp["v"], ps,
                                                      torch.empty(pinp["v"].shape, dtype=torch.bfloat16, device=dev),
                                                      g=pinp["g"], beta=pinp["beta"], chunk=64)),
                     dtype=torch.uint8, device=dev)

    def pcompute(d, o):
        ps.zero_()
        cg.prefill(d["q"], d["k"], d["v"], ps, o, g=d["g"], beta=d["beta"], chunk=64, workspace=ws)

    drun, prun = pipeline(h, o_like, dcompute, stream), pipeline(hp, po_like, pcompute, stream)
    drun(3)
    prun(3)
    dms, pms = timed(lambda: drun(K), 1, K), timed(lambda: prun(K), 1, K)
    D_STEPS, P_STEPS = 64, 8
    graph_dms = timed(graphed(h, o_like, dcompute, D_STEPS), 4, D_STEPS)
    graph_pms = timed(graphed(hp, po_like, pcompute, P_STEPS), 3, P_STEPS)
    return {"value": round(world * DEC_STATE_BYTES / (graph_dms / 1e3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d_dec + h2d_pre, "d2h_bytes_per_step": d2h_dec + d2h_pre,
            "decode_ms": round(graph_dms, 5), "prefill_ms": round(graph_pms, 5),
            "prefill_tokens_per_s": round(world * PRE["T"] / (graph_pms / 1e3), 1),
            "eager_pipelined": {"decode_ms": round(dms, 5), "prefill_ms": round(pms, 5),
                                "value": round(world * DEC_STATE_BYTES / (dms / 1e3) / 1e9, 2)},
            "note": f"every step copies its inputs in (one packed copy from pinned host memory) and its o out "
                    f"inside the timed region, on two copy streams double-buffered against the compute; value: "
                    f"{D_STEPS} decode / {P_STEPS} prefill steps replayed from one CUDA graph; eager_pipelined: "
                    f"the same steps issued call by call from Python; the decode state stays resident on the device"}


# ------------------------------------------------------------------ oracle timing
def oracle_sample(seconds_budget: float):
    """Time the fp64 CPU oracle, as it stands, on bounded samples of both workloads.

    Decode: every (b, h) unit of a B=64, H=32 batch for one token, on all host cores and on
    one; prefill: all 32 heads for the first `n_tok` tokens of the T=4000 sequence.  Returns
    (decode GB/s of fp32-state traffic, prefill tokens/s, threads, description, single-thread
    decode GB/s).
    """
    import oracle
    from gated_delta_rule_channelwise_gb300.synth import WORKLOADS, make_inputs
    threads = oracle.default_threads()
    wd, wp = WORKLOADS["decode_b64"], WORKLOADS["prefill_t4000"]
    di = make_inputs(wd, T=1, device="cpu")
    t = time.perf_counter()
    oracle.recurrence(di["q"], di["k"], di["v"], g=di["g"], beta=di["beta"], S0=di["S0"], threads=threads)
    dsec = time.perf_counter() - t
    # one thread, on an eighth of the units (scaled to the full batch)
    d1 = make_inputs(wd, T=1, B=8, device="cpu")
    t = time.perf_counter()
    oracle.recurrence(d1["q"], d1["k"], d1["v"], g=d1["g"], beta=d1["beta"], S0=d1["S0"], threads=1)
    dsec1 = (time.perf_counter() - t) * 8
    n_tok = 64
    pi = make_inputs(wp, T=n_tok, device="cpu")
    t = time.perf_counter()
    reps = 0
    while True:
        oracle.recurrence(pi["q"], pi["k"], pi["v"], g=pi["g"], beta=pi["beta"], S0=pi["S0"], threads=threads)
        reps += 1
        if time.perf_counter() - t > seconds_budget / 2 or reps >= 50:
            break
    psec = (time.perf_counter() - t) / reps
    desc = ("decode: all 2048 (b,h) units of B=64,H=32 for 1 token (single-thread figure: 256 units, "
            "scaled); prefill: 32 heads x %d tokens of the T=4000 sequence, %d repeats" % (n_tok, reps))
    return DEC_STATE_BYTES / dsec / 1e9, n_tok / psec, threads, desc, DEC_STATE_BYTES / dsec1 / 1e9


def run_reference(args):
    """Reference arm: the fp64 CPU oracle on the host cores, K steps of a bounded sample."""
    import numpy as np
    import oracle
    from gated_delta_rule_channelwise_gb300.synth import WORKLOADS, make_inputs
    oracle.build()
    threads = oracle.default_threads()
    wd, wp = WORKLOADS["decode_b64"], WORKLOADS["prefill_t4000"]
    units = 2 * threads                          # decode units per step (a sample of the 2048)
    di = make_inputs(wd, T=1, B=max(1, units // 32), device="cpu")
    pi = make_inputs(wp, T=8, device="cpu")
    pi = {k: (v[:, :, :1] if k in ("q", "k", "v", "g", "beta") else (v[:, :1] if k == "S0" else v))
          for k, v in pi.items()}
    bytes_per_unit = 2 * 128 * 128 * 4

    def step():
        t0 = time.perf_counter()
        oracle.recurrence(di["q"], di["k"], di["v"], g=di["g"], beta=di["beta"], S0=di["S0"], threads=threads)
        t1 = time.perf_counter()
        oracle.recurrence(pi["q"], pi["k"], pi["v"], g=pi["g"], beta=pi["beta"], S0=pi["S0"], threads=1)
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1

    for _ in range(args.warmup):
        step()
    dsum = psum = 0.0
    for _ in range(args.steps):
        a, b = step()
        dsum += a
        psum += b
    n_units = di["v"].shape[0] * di["v"].shape[2]
    gbs = args.steps * n_units * bytes_per_unit / dsum / 1e9
    tps = args.steps * 8 * 32 / (psum * 32)      # one head timed; 32 heads per token at this rate
    sample = ("per step: one decode token for %d of the 2048 (b,h) units of B=64,H=32; prefill: 8 tokens of one "
              "head of the T=4000 sequence (scaled to 32 heads)" % n_units)
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round((dsum + psum) / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(1),
            "prefill": {"value": round(tps, 2), "unit": "tokens/s"},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_case(name):
    """One small case of a kernel, run twice, for a profiler to capture (prints 'ok')."""
    import torch
    import gated_delta_rule_channelwise_gb300 as cg
    from gated_delta_rule_channelwise_gb300 import build as cbuild
    from gated_delta_rule_channelwise_gb300.synth import Workload, gate_kwargs, make_inputs
    cbuild.build()
    if name.startswith("prefill_t1024"):
        path = {"prefill_t1024_per_head": cg.PREFILL_PER_HEAD,
                "prefill_t1024_cluster": cg.PREFILL_CLUSTER}.get(name, cg.PREFILL_AUTO)
        w = Workload("p", B=1, Hk=32, Hv=32, dk=128, dv=128, T=1024, dtype="bf16", gate="channel", seed=1)
        inp = make_inputs(w, device="cuda")
        o = torch.empty(inp["v"].shape, dtype=torch.bfloat16, device="cuda")
        for _ in range(2):
            st = torch.zeros_like(inp["S0"])
            cg.prefill(inp["q"], inp["k"], inp["v"], st, o, chunk=64, path=path, **gate_kwargs(inp))
    elif name == "decode_b16":
        w = Workload("d", B=16, Hk=32, Hv=32, dk=128, dv=128, T=2, dtype="bf16", gate="channel", seed=1)
        inp = make_inputs(w, device="cuda")
        st = inp["S0"].clone()
        for t in range(2):
            cg.decode(inp["q"][:, t], inp["k"][:, t], inp["v"][:, t], st, g=inp["g"][:, t], beta=inp["beta"][:, t])
    torch.cuda.synchronize()
    print("ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-baseline-seconds", type=float, default=20.0)
    ap.add_argument("--no-secondary", action="store_true", help="skip the B=1 decode and T=16411 prefill timings")
    ap.add_argument("--case", choices=["prefill_t1024", "prefill_t1024_per_head", "prefill_t1024_cluster", "decode_b16"],
                    help="run one small case twice (for a profiler) and exit")
    args = ap.parse_args()
    if args.case:
        run_case(args.case)
        return
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if world == 1:
            dgbs, ptps, cores, desc, dgbs1 = oracle_sample(args.cpu_baseline_seconds)
            out["cpu_baseline"] = {"value": round(dgbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                   "sample": desc, "prefill_tokens_per_s": round(ptps, 2),
                                   "value_one_thread": round(dgbs1, 4)}
        else:
            out["cpu_baseline"] = None
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
