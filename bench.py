"""Benchmark of the LAGA MLA attention block, forward + backward, on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Workload (default): the DeepSeek-V3-dimension MLA layer (n_h=128, d_c=512,
d_nope=128, d_rope=64, d_v=128), sequence 16384 split over SP=8 ranks, the
last rank's shard (2048 queries at q_offset=14336 against the full latent),
causal, batch 1, bf16 storage with fp32 accumulation. One step = one forward
and one backward of that shard (reconstruction, attention, attention
backward, reconstruction backward). Inputs are seeded synthetic N(0,1) data
(weights N(0, 1/d_c)), generated on the host.

Printed: one JSON line. `value` is algorithmic TFLOP/s (fwd flops
2*P*n_h*(d_qk+d_v) + 2*B*Skv_eff*d_c*n_h*(d_nope+d_v), bwd = 2 x fwd) summed
over ranks; ranks run independent replicas of the shard (no collective).
L2 is flushed (a 512 MB buffer is written) before every timed step, outside
the step's own CUDA events.

--impl reference times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload (a subset of heads per step).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from mla_attention_sequence_gb300.configs import GROUPS, NAMED, DSV3_LAST_RANK, Problem  # noqa: E402
from mla_attention_sequence_gb300.synth import make_inputs  # noqa: E402

METRIC = "MLA attn-block fwd+bwd TFLOP/s & tokens/s, % of GB300 bf16 peak"
UNIT = "TFLOP/s"
SEED = 2007


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                "bf16_tflops_sustained": pk.get("bf16_tflops_sustained", pk["bf16_tflops"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# DRAM traffic per launch of a kernel, from one ncu capture of the kernel source
# identified by `src_sha` (sha256 of the kernel file followed by csrc/ptx.cuh,
# first 16 hex digits). It is reported only while the source is unchanged.
# attn_bwd_dkdv: dram__bytes_read.sum + dram__bytes_write.sum = 741.1 + 563.5 MB
# on the n_h = 64 last-rank shard (the full n_h = 128 shard exceeds the size rule
# for a multi-pass capture); the kernel's work and both byte streams (K/V and
# Q/dO tiles in, dK/dV and the head-group RoPE-key partials out) scale with the
# head count, so x2.
MEASURED_TRAFFIC = {
    "attn_bwd_dkdv": {"src": "attn_bwd_dkdv_tc.cu", "src_sha": "bfc25970d5f2b0f6",
                      "bytes_per_launch": {"dsv3_sp8_rank7_S16384_h128": 2 * (741.058304e6 + 563.450880e6)}},
}


def kernel_traffic(kernel: str, workload: str):
    import hashlib
    m = MEASURED_TRAFFIC.get(kernel)
    if not m or workload not in m["bytes_per_launch"]:
        return None
    csrc = os.path.join(ROOT, "mla_attention_sequence_gb300", "csrc")
    try:
        h = hashlib.sha256()
        for name in (m["src"], "ptx.cuh"):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    return m["bytes_per_launch"][workload] if h.hexdigest()[:16] == m["src_sha"] else None


def workload_config(p: Problem, extra=None):
    c = {"workload": p.name, "B": p.B, "Sq": p.Sq, "S": p.S, "n_h": p.n_h, "d_c": p.d_c, "d_nope": p.d_nope,
         "d_rope": p.d_rope, "d_v": p.d_v, "q_offset": p.q_offset, "causal": p.causal, "sp": 8,
         "flops_per_step": p.flops_step(), "tokens_per_step": p.B * p.Sq,
         "l2": "flushed before each timed step (512 MB write)", "parallelism": "replicas"}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over ranks (identity for one process)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------- CPU oracle timing
def oracle_sample(p: Problem, x: dict, heads: list[int], keep: dict | None = None):
    """Run the fp64 oracle's forward+backward for the given heads, over every
    batch element. Returns the algorithmic flops of that sample; `keep` (if
    given) collects each head's results by head index: batch 0's per-row outputs
    (out, lse, dq) and the head's weight gradients summed over the batch, as the
    library's dW_UK / dW_UV are."""
    import oracle
    x64 = x if all(v.dtype == np.float64 for v in x.values()) else {k: v.astype(np.float64) for k, v in x.items()}
    pos = oracle.query_positions(p.Sq, p.q_offset, p.q_split, p.q_offset2) if p.q_split > 0 else p.q_offset
    for h in heads:
        g = None
        for bi in range(p.B):
            gb = oracle.mla_backward_head(x64["q"], x64["c_kv"], x64["k_rope"], x64["W_UK"], x64["W_UV"],
                                          x64["dout"], bi, h, pos, p.causal)
            if g is None:
                g = gb
            else:
                g["dW_UK_h"] = g["dW_UK_h"] + gb["dW_UK_h"]
                g["dW_UV_h"] = g["dW_UV_h"] + gb["dW_UV_h"]
        if keep is not None:
            keep[h] = g
    return p.with_(n_h=len(heads)).flops_step()


def time_oracle(p: Problem, x: dict, budget_s: float = 15.0, max_heads: int = 64, keep: dict | None = None):
    """Time the oracle over as many heads as fit the time budget (at least one)."""
    x = {k: v.astype(np.float64) for k, v in x.items()}
    t0 = time.perf_counter()
    flops = 0
    heads = 0
    while heads < min(max_heads, p.n_h) and (time.perf_counter() - t0) < budget_s:
        flops += oracle_sample(p, x, [heads], keep)
        heads += 1
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, heads, dt


def sampled_errors(p: Problem, buf, ref_heads: dict) -> dict:
    """max|gpu - oracle| / max|oracle| per output tensor over the oracle's sampled
    heads (out, lse, dq of batch 0; dW_UK, dW_UV summed over the batch)."""
    acc = {}
    for h, g in ref_heads.items():
        pairs = {"out": (buf.out[0, :, h], g["out_h"]), "lse": (buf.lse[0, h], g["lse_h"]),
                 "dq": (buf.grads["dq"][0, :, h], g["dq_h"]),
                 "dW_UK": (buf.grads["dW_UK"][:, h * p.d_nope:(h + 1) * p.d_nope], g["dW_UK_h"]),
                 "dW_UV": (buf.grads["dW_UV"][:, h * p.d_v:(h + 1) * p.d_v], g["dW_UV_h"])}
        for k, (a, r) in pairs.items():
            a = a.float().cpu().numpy().astype(np.float64)
            e, m = float(np.abs(a - r).max()), float(np.abs(r).max())
            pe, pm = acc.get(k, (0.0, 0.0))
            acc[k] = (max(pe, e), max(pm, m))
    return {k: e / m if m > 0 else e for k, (e, m) in acc.items()}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- reference arm
def run_reference(args, p: Problem):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    x = make_inputs(p, SEED)
    x64 = {k: v.astype(np.float64) for k, v in x.items()}
    heads_per_step = 1
    for i in range(args.warmup):
        oracle_sample(p, x64, [i % p.n_h])
    times = []
    flops = 0
    for i in range(args.steps):
        t0 = time.perf_counter()
        flops += oracle_sample(p, x64, [(args.warmup + i) % p.n_h])
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = flops / total / 1e12
    cores = host_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(p, {"sample": f"{heads_per_step} head(s) of {p.n_h} per step"}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"fp64 oracle fwd+bwd of {heads_per_step} head per step (of {p.n_h}), "
                                   f"every batch element of the shard; TFLOP/s of that sample's algorithmic flops"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def shard_inputs(name: str, seed: int):
    """Problems of one step and their host inputs. A single shard draws its own
    inputs; the all-ranks group draws the full sequence once and gives each rank
    its query / dout rows with the shared latent, RoPE key and weights."""
    if name not in GROUPS:
        p = NAMED[name]
        return [p], [make_inputs(p, seed)]
    shards = GROUPS[name]
    p0 = shards[0]
    full = p0.with_(Sq=p0.S, q_offset=0)
    x = make_inputs(full, seed)
    xs = []
    for p in shards:
        rows = np.concatenate([np.arange(off, off + n) for _, n, off in p.segments()])
        xs.append({k: (np.ascontiguousarray(v[:, rows]) if k in ("q", "dout") else v) for k, v in x.items()})
    return shards, xs


def kernel_flops(p: Problem) -> dict:
    """Algorithmic flops each timed step of one shard's forward+backward owns."""
    attn_fwd = 2 * p.pairs * p.n_h * (p.d_qk + p.d_v)
    recon = 2 * p.B * p.skv_eff * p.d_c * p.n_h * (p.d_nope + p.d_v)
    # backward attention = 2 x forward, split by the products each kernel owns:
    # dK/dV kernel dV + dP + dK (128 + 128 + 192 per pair and head), dq kernel dQ (192)
    unit = 2 * p.pairs * p.n_h
    return {"attn_fwd": attn_fwd, "attn_bwd_dkdv": unit * (p.d_v + p.d_v + p.d_qk), "attn_bwd_dq": unit * p.d_qk,
            "recon_fwd_gemm": recon, "recon_bwd_dc_gemm": recon, "recon_bwd_dw_gemm": recon}


def run_ours(args, name: str):
    import ctypes

    import torch

    from mla_attention_sequence_gb300 import build as build_mod
    from mla_attention_sequence_gb300 import laga

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    build_mod.build()
    L = laga.lib()

    problems, xs = shard_inputs(name, SEED + rank)
    dt = torch.bfloat16 if problems[0].dtype == "bf16" else torch.float32
    shared = {}
    dinps = []
    for x in xs:
        d = {}
        for k, v in x.items():
            key = (k, id(v))
            if key not in shared:  # inputs shared by shards are staged once
                hv = torch.from_numpy(v).to(dt).pin_memory()
                shared[key] = (hv, hv.to(dev, non_blocking=True))
            d[k] = shared[key][1]
        dinps.append(d)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    bufs = [laga.alloc_step(p, d, args.variant) for p, d in zip(problems, dinps)]
    stream = torch.cuda.current_stream(dev)

    def step():
        for buf in bufs:
            laga.step(buf, args.variant)

    step()
    torch.cuda.synchronize()
    # device memory of one step: inputs, outputs, gradients and the one workspace
    # the forward and backward share (the library allocates nothing itself)
    mem = {"peak_mem_bytes": int(torch.cuda.max_memory_allocated(dev)),
           "workspace_bytes": int(sum(b.ws.numel() if b.ws is not None else 0 for b in bufs)),
           "inputs_bytes": int(sum(t.numel() * t.element_size() for t in {id(v): v for d in dinps
                                                                             for v in d.values()}.values())),
           "what": "torch.cuda.max_memory_allocated over staging the inputs, allocating outputs, gradients "
                   "and workspace, and one forward+backward (the L2 flush buffer is allocated afterwards)"}
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    for _ in range(args.warmup):
        step()
    laga.check(dev)
    torch.cuda.synchronize()

    # ---- device-resident timed region
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    L.laga_mla_profile_enable(1)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    nmax = 64 * args.steps * len(bufs)
    names = (ctypes.c_char_p * nmax)()
    ms = (ctypes.c_float * nmax)()
    nrec = L.laga_mla_profile_read(ctypes.cast(names, ctypes.POINTER(ctypes.c_char_p)), ms, nmax)
    L.laga_mla_profile_enable(0)
    laga.check(dev)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = reduce_max(sum(step_ms), world, dev)
    per_kernel = {}
    for i in range(min(nrec, nmax)):
        per_kernel.setdefault(names[i].decode(), []).append(ms[i])

    # ---- end-to-end through the public API with host buffers. Every step copies its
    # inputs pinned host -> device and all its results device -> host inside the timed
    # region. The copies run on their own streams over two buffer sets, so step i+1's
    # inputs land and step i-1's results leave while step i computes (the input
    # prefetch of a training loop); a set is refilled only after the step that used it
    # has finished, and overwritten only after its results have left.
    sets = []
    for rep in range(2):
        if rep == 0:
            dev_in = {key: dv for key, (hv, dv) in shared.items()}
            sbufs = bufs
        else:
            dev_in = {key: torch.empty_like(dv) for key, (hv, dv) in shared.items()}
            dins = [{k: dev_in[(k, id(v))] for k, v in x.items()} for x in xs]
            sbufs = [laga.alloc_step(p, d, args.variant) for p, d in zip(problems, dins)]
        outs_host = []
        for buf in sbufs:
            oh = {"out": torch.empty(buf.out.shape, dtype=dt).pin_memory(),
                  "lse": torch.empty(buf.lse.shape, dtype=torch.float32).pin_memory()}
            for k, v in buf.grads.items():
                oh[k] = torch.empty(v.shape, dtype=dt).pin_memory()
            outs_host.append(oh)
        sets.append((dev_in, sbufs, outs_host))
    h2d = sum(hv.numel() * hv.element_size() for hv, _ in shared.values())
    d2h = sum(v.numel() * v.element_size() for oh in sets[0][2] for v in oh.values())
    copy_in = torch.cuda.Stream(dev)
    copy_out = torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    # the compute of each step inside the end-to-end loop, to tell copy/compute
    # interference (compute slower) from dependency stalls (gaps between steps)
    c_start = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    c_end = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    # and each step's copies on their streams, to tell slow host copies (a step
    # waiting for its inputs) from a host thread that enqueues too late
    cp_ev = {k: [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] for k in ("h0", "h1", "o0", "o1")}
    barrier(world)
    torch.cuda.synchronize()
    e_start.record(stream)
    copy_in.wait_stream(stream)
    copy_out.wait_stream(stream)
    host_t0 = time.perf_counter()
    for i in range(args.steps):
        b = i % 2
        dev_in, sbufs, outs_host = sets[b]
        if i >= 2:
            copy_in.wait_event(done[b])  # step i-2 has finished reading this set's inputs
        with torch.cuda.stream(copy_in):
            cp_ev["h0"][i].record(copy_in)
            for key, (hv, _) in shared.items():
                dev_in[key].copy_(hv, non_blocking=True)
            cp_ev["h1"][i].record(copy_in)
            in_ready[b].record(copy_in)
        stream.wait_event(in_ready[b])
        if i >= 2:
            stream.wait_event(out_done[b])  # step i-2's results have left this set
        c_start[i].record(stream)
        for buf in sbufs:
            laga.step(buf, args.variant)
        c_end[i].record(stream)
        done[b].record(stream)
        copy_out.wait_event(done[b])
        with torch.cuda.stream(copy_out):
            cp_ev["o0"][i].record(copy_out)
            for buf, oh in zip(sbufs, outs_host):
                oh["out"].copy_(buf.out, non_blocking=True)
                oh["lse"].copy_(buf.lse, non_blocking=True)
                for k, v in buf.grads.items():
                    oh[k].copy_(v, non_blocking=True)
            cp_ev["o1"][i].record(copy_out)
            out_done[b].record(copy_out)
    stream.wait_stream(copy_out)
    e_end.record(stream)
    host_enqueue_ms = (time.perf_counter() - host_t0) * 1e3  # the host thread's time to enqueue every step
    torch.cuda.synchronize()
    barrier(world)
    laga.check(dev)
    e2e_ms = reduce_max(e_start.elapsed_time(e_end), world, dev)
    e2e_compute_ms = float(np.mean([a.elapsed_time(z) for a, z in zip(c_start, c_end)]))
    e2e_gap_ms = float(np.mean([c_end[i].elapsed_time(c_start[i + 1]) for i in range(args.steps - 1)])) \
        if args.steps > 1 else 0.0
    e2e_h2d_ms = float(np.mean([a.elapsed_time(z) for a, z in zip(cp_ev["h0"], cp_ev["h1"])]))
    e2e_d2h_ms = float(np.mean([a.elapsed_time(z) for a, z in zip(cp_ev["o0"], cp_ev["o1"])]))

    flops = sum(p.flops_step() for p in problems)
    tokens = sum(p.B * p.Sq for p in problems)
    value = world * flops * args.steps / (total_ms * 1e-3) / 1e12
    e2e_value = world * flops * args.steps / (e2e_ms * 1e-3) / 1e12
    tokens_s = world * tokens * args.steps / (total_ms * 1e-3)
    peaks = load_peaks()

    # roofline of the dominant kernel (largest total time): algorithmic flops of
    # all its launches in a step over their measured time in that step
    kflops = {}
    for p in problems:
        for k, v in kernel_flops(p).items():
            kflops[k] = kflops.get(k, 0) + v
    kernel_ms = {k: float(np.mean(v)) for k, v in per_kernel.items()}
    dom = max(per_kernel, key=lambda k: sum(per_kernel[k])) if per_kernel else None
    roof = None
    if dom in kflops:
        t_step = sum(per_kernel[dom]) / args.steps
        achieved = kflops[dom] / (t_step * 1e-3) / 1e12
        # The kernel runs a few ms inside a ~9 ms step, in a timed region well under a
        # second at the maximum SM clock: burst conditions, so the burst peak applies.
        peak = peaks["bf16_tflops"]
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "traffic": kernel_traffic(dom, problems[0].name) if len(problems) == 1 else None,
                "peak_kind": f"bf16 dense, burst, {peaks['source']}",
                "flops_per_launch": kflops[dom] / len(problems), "ms_per_launch": t_step / len(problems),
                "launches_per_step": len(problems)}
    launches_per_step = {"simt_fwd": 3, "simt_bwd": 10}  # every other timed step is one kernel
    gpu_launches = sum(launches_per_step.get(k, 1) * len(v) for k, v in per_kernel.items())

    cpu = None
    errors = None
    oracle_s = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ref_heads = {}
        tf, heads, secs = time_oracle(problems[-1], xs[-1], budget_s=args.cpu_budget, keep=ref_heads)
        oracle_s = secs
        cpu = {"value": tf, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": f"fp64 oracle fwd+bwd of {heads} head(s) (of {problems[-1].n_h}) of shard "
                         f"{problems[-1].name}, {secs:.1f} s; TFLOP/s of the sample's algorithmic flops"}
        # the same heads of the GPU's last step (same inputs) against the oracle
        errors = sampled_errors(problems[-1], bufs[-1], ref_heads)
        errors["heads"] = sorted(ref_heads)

    if rank == 0:
        cfg = workload_config(problems[-1], {"variant": args.variant})
        if len(problems) > 1:
            cfg.update({"workload": name, "Sq": tokens, "q_offset": [p.q_offset for p in problems],
                        "shards_per_step": len(problems), "flops_per_step": flops, "tokens_per_step": tokens})
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": cfg,
            "tokens_per_s": tokens_s,
            # secondary: FlashAttention convention (adds the backward's score recompute)
            "tflops_fa_convention": world * sum(p.flops_step_fa() for p in problems) * args.steps
            / (total_ms * 1e-3) / 1e12,
            "pct_of_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
            "peak_source": peaks["source"],
            "roofline": roof,
            "kernels_ms_per_launch": kernel_ms,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "compute_ms_per_step": e2e_compute_ms,
                    "gap_ms_between_steps": e2e_gap_ms, "h2d_ms_per_step": e2e_h2d_ms,
                    "d2h_ms_per_step": e2e_d2h_ms, "host_enqueue_ms_per_step": host_enqueue_ms / args.steps,
                    "ms_per_step": e2e_ms / args.steps},
            "gpu_launches": gpu_launches,
            "clocks": clk,
            "cpu_baseline": cpu,
            "max_err_over_max_ref": errors,
            "oracle_s": oracle_s,
            "memory": mem,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------- forward variants
def _time_events(fn, steps, flush, stream):
    """Median CUDA-event time (ms) of fn over `steps` runs, L2 flushed before each."""
    import torch
    times = []
    for _ in range(steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e))
    return float(np.median(times))


def run_variant_sweep(args):
    """The sweep over the last-rank SP=8 shards (sequence length x heads): per shape,
    forward + backward of the materialised-K/V variant (the path AUTO takes; the
    backward reuses the forward's K/V), and the forward of both K/V variants:
    'materialize' (reconstruction GEMM to HBM + attention) against 'fused_recon'
    (K/V tiles rebuilt inside the attention kernel; forward only, no backward is
    built for it). Algorithmic flops as in the main line; one JSON line per shape."""
    import ctypes

    import torch

    from mla_attention_sequence_gb300 import build as build_mod
    from mla_attention_sequence_gb300 import laga
    from mla_attention_sequence_gb300.configs import sweep_points

    build_mod.build()
    L = laga.lib()
    dev = torch.device("cuda", 0)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for p in sweep_points():
        if args.sweep_filter and args.sweep_filter not in p.name:
            continue
        x = make_inputs(p, SEED)
        t = {k: torch.from_numpy(v).to(dev).to(torch.bfloat16) for k, v in x.items()}
        line = {"mode": "sweep", "workload": p.name, "S": p.S, "n_h": p.n_h, "Sq": p.Sq, "q_offset": p.q_offset,
                "flops_step": p.flops_step(), "flops_fwd": p.flops_fwd()}
        # forward + backward, materialised K/V (one workspace shared by both calls)
        buf = laga.alloc_step(p, t, "materialize")

        def step():
            laga.step(buf, "materialize")
        for _ in range(args.warmup):
            step()
        laga.check(dev)
        L.laga_mla_profile_enable(1)
        ms_step = _time_events(step, args.steps, flush, stream)
        nmax = 16 * args.steps
        names = (ctypes.c_char_p * nmax)()
        ms = (ctypes.c_float * nmax)()
        n = L.laga_mla_profile_read(ctypes.cast(names, ctypes.POINTER(ctypes.c_char_p)), ms, nmax)
        L.laga_mla_profile_enable(0)
        per = {}
        for i in range(min(n, nmax)):
            per.setdefault(names[i].decode(), []).append(ms[i])
        line["materialize"] = {"ms_step": ms_step, "tflops_step": p.flops_step() / (ms_step * 1e-3) / 1e12,
                               "pct_of_bf16_peak": 100.0 * p.flops_step() / (ms_step * 1e-3) / 1e12
                               / load_peaks()["bf16_tflops"],
                               "kernels_ms": {k: float(np.median(v)) for k, v in per.items()},
                               "workspace_bytes": int(buf.ws.numel()) if buf.ws is not None else 0}
        del buf
        out = torch.empty((p.B, p.Sq, p.n_h, p.d_v), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((p.B, p.n_h, p.Sq), dtype=torch.float32, device=dev)
        for variant in ("materialize", "fused_recon"):
            nbytes = laga.fwd_workspace_bytes(p, variant)
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None

            def run():
                laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, p.causal, None, variant,
                         ws, out, lse)
            for _ in range(args.warmup):
                run()
            laga.check(dev)
            t_ms = _time_events(run, args.steps, flush, stream)
            key = "materialize" if variant == "materialize" else "fused_recon"
            line.setdefault(key, {}).update({"ms_fwd": t_ms, "tflops_fwd": p.flops_fwd() / (t_ms * 1e-3) / 1e12,
                                             "fwd_workspace_bytes": nbytes})
            del ws
        line["fused_recon"]["bwd"] = "not built (forward-only variant)"
        print(json.dumps(line), flush=True)
        del t, out, lse
        torch.cuda.empty_cache()
    return 0


# ---------------------------------------------------------------- eager (unfused) baseline
def eager_forward_backward(t: dict, p: Problem, scale: float, saved: dict | None = None):
    """The attention block written as separate library operations, the 'eager'
    setting: reconstruction matmuls, the RoPE-key concat, QK^T, mask, softmax in
    fp32, PV, each a separate cuBLAS / PyTorch kernel with its intermediates in
    HBM, and torch autograd for the backward. bf16 matmuls with fp32 softmax.
    `saved` (if given) receives the memory autograd holds after the forward."""
    import torch
    B, Sq, n_h, S = p.B, p.Sq, p.n_h, p.skv_eff
    q = t["q"].detach().requires_grad_()
    c = t["c_kv"].detach().requires_grad_()
    kr = t["k_rope"].detach().requires_grad_()
    wk = t["W_UK"].detach().requires_grad_()
    wv = t["W_UV"].detach().requires_grad_()
    base = torch.cuda.memory_allocated(q.device)
    k_nope = (c[:, :S] @ wk).view(B, S, n_h, p.d_nope)
    v = (c[:, :S] @ wv).view(B, S, n_h, p.d_v)
    k = torch.cat([k_nope, kr[:, :S, None, :].expand(B, S, n_h, p.d_rope)], dim=-1)
    sc = torch.matmul(q.permute(0, 2, 1, 3), k.permute(0, 2, 3, 1)).float() * scale  # [B, n_h, Sq, S]
    if p.causal:
        pos = torch.arange(Sq, device=q.device) + p.q_offset
        mask = torch.arange(S, device=q.device)[None, :] > pos[:, None]
        sc = sc.masked_fill(mask, float("-inf"))
    with torch.no_grad():
        lse = torch.logsumexp(sc, dim=-1)
    prob = torch.softmax(sc, dim=-1).to(torch.bfloat16)
    out = torch.matmul(prob, v.permute(0, 2, 1, 3)).permute(0, 2, 1, 3)
    if saved is not None:
        torch.cuda.synchronize()
        saved["bytes"] = torch.cuda.memory_allocated(q.device) - base
    out.backward(t["dout"])
    return out.detach(), lse.detach(), {"dq": q.grad, "dc_kv": c.grad, "dk_rope": kr.grad, "dW_UK": wk.grad,
                                        "dW_UV": wv.grad}


def eager_absorbed_forward_backward(t: dict, p: Problem, scale: float, saved: dict | None = None):
    """The absorbed MLA form as separate library operations (the eager setting):
    q_lat = q_nope W_UK^T per head, scores against [c_kv | k_rope], softmax in fp32,
    attention over the latent, output through W_UV, torch autograd backward.
    `saved` (if given) receives the memory autograd holds after the forward."""
    import torch
    B, Sq, n_h, S = p.B, p.Sq, p.n_h, p.skv_eff
    q = t["q"].detach().requires_grad_()
    c = t["c_kv"].detach().requires_grad_()
    kr = t["k_rope"].detach().requires_grad_()
    wk = t["W_UK"].detach().requires_grad_()
    wv = t["W_UV"].detach().requires_grad_()
    base = torch.cuda.memory_allocated(q.device)
    q_lat = torch.einsum("bihd,chd->bihc", q[..., :p.d_nope], wk.view(p.d_c, n_h, p.d_nope))
    q_abs = torch.cat([q_lat, q[..., p.d_nope:]], dim=-1)  # [B, Sq, n_h, d_c + d_rope]
    key = torch.cat([c[:, :S], kr[:, :S]], dim=-1)  # one key for every head
    sc = torch.einsum("bihc,bjc->bhij", q_abs, key).float() * scale
    if p.causal:
        pos = torch.arange(Sq, device=q.device) + p.q_offset
        sc = sc.masked_fill(torch.arange(S, device=q.device)[None, :] > pos[:, None], float("-inf"))
    prob = torch.softmax(sc, dim=-1).to(torch.bfloat16)
    ctx = torch.einsum("bhij,bjc->bihc", prob, c[:, :S])
    out = torch.einsum("bihc,chd->bihd", ctx, wv.view(p.d_c, n_h, p.d_v))
    if saved is not None:
        torch.cuda.synchronize()
        saved["bytes"] = torch.cuda.memory_allocated(q.device) - base
    out.backward(t["dout"])
    return out.detach(), {"dq": q.grad, "dc_kv": c.grad, "dk_rope": kr.grad, "dW_UK": wk.grad, "dW_UV": wv.grad}


def run_memory_sweep(args):
    """Device memory of one training step (forward + backward) of the attention
    block, per implementation, over the last-rank SP=8 shards of seq in
    {4096, 8192, 16384} x n_h in {32, 64, 128}: the bytes kept from the forward for
    the backward ('saved': autograd's holdings for the eager forms; the outputs
    and the kept workspace for the library's) and the step's peak above the
    inputs ('peak'). One JSON line per shape, then a fit of the absorbed-minus-LAGA
    gap against seq x n_h."""
    import torch

    from mla_attention_sequence_gb300 import build as build_mod
    from mla_attention_sequence_gb300 import laga
    from mla_attention_sequence_gb300.configs import dsv3_rank

    build_mod.build()
    dev = torch.device("cuda", 0)
    rows = []
    for seq in (4096, 8192, 16384):
        for n_h in (32, 64, 128):
            p = dsv3_rank(7, seq=seq, n_h=n_h)
            x = make_inputs(p, SEED)
            t = {k: torch.from_numpy(v).to(dev).to(torch.bfloat16) for k, v in x.items()}
            scale = 1.0 / float(np.sqrt(p.d_qk))
            line = {"mode": "memory", "workload": p.name, "S": seq, "n_h": n_h, "Sq": p.Sq}
            outs_bytes = (p.B * p.Sq * p.n_h * p.d_v * 2 + p.B * p.n_h * p.Sq * 4)

            def measure(fn):
                torch.cuda.synchronize()
                torch.cuda.empty_cache()
                base = torch.cuda.memory_allocated(dev)
                torch.cuda.reset_peak_memory_stats(dev)
                info = fn() or {}
                torch.cuda.synchronize()
                info["peak"] = int(torch.cuda.max_memory_allocated(dev) - base)
                return info

            def laga_reuse():
                buf = laga.alloc_step(p, t)
                laga.step(buf)
                # kept from the forward for the backward: the rebuilt K_nope / V (the
                # forward's part of the shared workspace) and out, lse
                return {"saved": int(laga.fwd_workspace_bytes(p)) + outs_bytes, "workspace": int(buf.ws.numel())}

            def laga_rebuild():
                ws_f = laga.fwd_workspace_bytes(p)
                out, lse = laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True)
                torch.cuda.synchronize()
                torch.cuda.empty_cache()  # the forward's workspace is gone; K/V are rebuilt in the backward
                laga.bwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], out, lse, t["dout"], p.q_offset, True)
                return {"saved": outs_bytes, "fwd_workspace": int(ws_f), "bwd_workspace": int(laga.bwd_workspace_bytes(p))}

            def absorbed():
                nb = laga.absorbed_workspace_bytes(p)
                ws = torch.empty(nb, dtype=torch.uint8, device=dev)
                laga.absorbed_fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True,
                                  workspace=ws)
                # the absorbed form's backward needs q_lat and ctx (the workspace) kept
                return {"saved": int(nb) + outs_bytes, "workspace": int(nb), "note": "forward only on the GPU"}

            def eager_expl():
                saved = {}
                r = eager_forward_backward(t, p, scale, saved)
                del r
                return {"saved": int(saved["bytes"])}

            def eager_abs():
                saved = {}
                r = eager_absorbed_forward_backward(t, p, scale, saved)
                del r
                return {"saved": int(saved["bytes"])}

            # forward times (median of 5, L2 flushed): the library's forward and the absorbed form's
            flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
            stream = torch.cuda.current_stream(dev)
            ws_l = torch.empty(laga.fwd_workspace_bytes(p), dtype=torch.uint8, device=dev)
            ws_a = torch.empty(laga.absorbed_workspace_bytes(p), dtype=torch.uint8, device=dev)
            f_l = lambda: laga.fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True,
                                   workspace=ws_l)
            f_a = lambda: laga.absorbed_fwd(t["q"], t["c_kv"], t["k_rope"], t["W_UK"], t["W_UV"], p.q_offset, True,
                                            workspace=ws_a)
            f_l(), f_a()
            line["ms_fwd"] = {"laga": _time_events(f_l, 5, flush, stream), "absorbed": _time_events(f_a, 5, flush, stream)}
            del flush, ws_l, ws_a
            line["laga_reuse_kv"] = measure(laga_reuse)
            line["laga_rebuild_kv"] = measure(laga_rebuild)
            line["absorbed"] = measure(absorbed)
            if not args.no_eager:
                line["eager_explicit"] = measure(eager_expl)
                line["eager_absorbed"] = measure(eager_abs)
            print(json.dumps(line), flush=True)
            rows.append(line)
            del t
            torch.cuda.empty_cache()
    # the absorbed form's extra saved bytes against LAGA's (rebuild): linear in Sq x n_h?
    xs = np.array([r["Sq"] * r["n_h"] for r in rows], dtype=float)
    gap = np.array([r["absorbed"]["saved"] - r["laga_rebuild_kv"]["saved"] for r in rows], dtype=float)
    A = np.vstack([xs, np.ones_like(xs)]).T
    coef, res, _, _ = np.linalg.lstsq(A, gap, rcond=None)
    pred = A @ coef
    print(json.dumps({"mode": "memory_fit", "quantity": "absorbed saved - laga (rebuild) saved, bytes",
                      "bytes_per_query_row_and_head": coef[0], "intercept": coef[1],
                      "max_rel_residual": float(np.max(np.abs(pred - gap) / np.maximum(np.abs(gap), 1.0)))}),
          flush=True)
    if not args.no_eager:
        # eager forms: the absorbed-minus-explicit gap per score element (query x key x head)
        els = np.array([r["Sq"] * r["S"] * r["n_h"] for r in rows], dtype=float)
        eg = np.array([r["eager_absorbed"]["saved"] - r["eager_explicit"]["saved"] for r in rows], dtype=float)
        ratio = eg / els
        print(json.dumps({"mode": "memory_fit", "quantity": "eager absorbed saved - eager explicit saved, bytes",
                          "bytes_per_score_element": {"min": float(ratio.min()), "max": float(ratio.max())},
                          "relative_gap_pct": [round(100 * (r["eager_absorbed"]["saved"] /
                                                            r["eager_explicit"]["saved"] - 1), 2) for r in rows]}),
              flush=True)
    return 0


def run_eager(args, name: str):
    """Times the eager baseline beside the fused path on the same shard and inputs,
    checks one head of each against the fp64 oracle, and prints one JSON line."""
    import torch

    from mla_attention_sequence_gb300 import build as build_mod
    from mla_attention_sequence_gb300 import laga

    build_mod.build()
    p = NAMED[name]
    dev = torch.device("cuda", 0)
    x = make_inputs(p, SEED)
    t = {k: torch.from_numpy(v).to(dev).to(torch.bfloat16) for k, v in x.items()}
    scale = 1.0 / float(np.sqrt(p.d_qk))
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    buf = laga.alloc_step(p, t)
    for _ in range(args.warmup):
        laga.step(buf)
    laga.check(dev)
    ms_fused = _time_events(lambda: laga.step(buf), args.steps, flush, stream)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    res = {}

    def eager():
        res["r"] = eager_forward_backward(t, p, scale)
    for _ in range(max(1, args.warmup // 3)):
        eager()
    torch.cuda.synchronize()
    peak_eager = torch.cuda.max_memory_allocated(dev) - base
    ms_eager = _time_events(eager, max(2, args.steps // 4), flush, stream)
    # one head of each against the oracle
    import oracle
    x64 = {k: v.astype(np.float64) for k, v in x.items()}
    h = p.n_h - 1
    g = oracle.mla_backward_head(x64["q"], x64["c_kv"], x64["k_rope"], x64["W_UK"], x64["W_UV"], x64["dout"], 0, h,
                                 p.q_offset, p.causal)
    eo, el, eg = res["r"]

    def err(a, r):
        a = a.float().cpu().numpy().astype(np.float64)
        return float(np.abs(a - r).max() / np.abs(r).max())
    errs = {}
    for tag, (o, l, gr) in {"eager": (eo, el, eg), "fused": (buf.out, buf.lse, buf.grads)}.items():
        errs[tag] = {"out": err(o[0, :, h], g["out_h"]), "lse": err(l[0, h], g["lse_h"]),
                     "dq": err(gr["dq"][0, :, h], g["dq_h"]),
                     "dW_UK": err(gr["dW_UK"][:, h * p.d_nope:(h + 1) * p.d_nope], g["dW_UK_h"]),
                     "dW_UV": err(gr["dW_UV"][:, h * p.d_v:(h + 1) * p.d_v], g["dW_UV_h"])}
    flops = p.flops_step()
    print(json.dumps({"mode": "eager_vs_fused", "workload": p.name, "flops_per_step": flops,
                      "fused": {"ms_step": ms_fused, "tflops": flops / (ms_fused * 1e-3) / 1e12,
                                "workspace_bytes": int(buf.ws.numel()) if buf.ws is not None else 0},
                      "eager": {"ms_step": ms_eager, "tflops": flops / (ms_eager * 1e-3) / 1e12,
                                "peak_extra_bytes": int(peak_eager),
                                "what": "cuBLAS bf16 matmuls (reconstruction, QK^T, PV), fp32 mask/softmax, "
                                        "torch autograd backward; intermediates in HBM"},
                      "speedup_fused_over_eager": ms_eager / ms_fused,
                      "max_err_over_max_ref_head": {"head": h, **errs}}), flush=True)
    return 0


def free_port() -> int:
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def relaunch(n: int, argv: list) -> int:
    """Run this script under torch.distributed.run with n local ranks (rendezvous on
    127.0.0.1); returns its exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DSV3_LAST_RANK.name, choices=sorted(NAMED) + sorted(GROUPS))
    ap.add_argument("--variant", default="auto", choices=["auto", "materialize", "simt"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle timing for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--variant-sweep", action="store_true",
                    help="time fwd+bwd (materialised K/V) and the forward of both K/V variants over the sweep "
                         "shapes instead")
    ap.add_argument("--sweep-filter", default="", help="only sweep shapes whose name contains this string")
    ap.add_argument("--memory-sweep", action="store_true",
                    help="device memory of one training step per implementation over the sweep shapes instead")
    ap.add_argument("--no-eager", action="store_true", help="memory sweep without the eager (torch) forms")
    ap.add_argument("--eager", action="store_true",
                    help="time the unfused (eager) baseline beside the fused path on --workload instead")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least three untimed steps
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # --gpus N outside a launcher: start the N ranks (one process per GPU) here
        return relaunch(args.gpus, sys.argv[1:] if argv is None else list(argv))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; reporting n_gpus={world}", file=sys.stderr)
    if args.variant_sweep:
        return run_variant_sweep(args)
    if args.eager:
        return run_eager(args, args.workload)
    if args.memory_sweep:
        return run_memory_sweep(args)
    if args.impl == "reference":
        p = GROUPS[args.workload][-1] if args.workload in GROUPS else NAMED[args.workload]
        return run_reference(args, p)
    return run_ours(args, args.workload)


if __name__ == "__main__":
    sys.exit(main())
