#!/usr/bin/env python3
"""Benchmark of the ModernBERT-base attention block on GB300.

One step = the whole hot path over one batch: a global layer and a local
layer of the attention block over one packed batch (default: one sequence of
8192 tokens, qkv [8192, 2304] bf16 ~ N(0, 1), seed 3).  `value` is tokens/s
through that layer pair, all ranks together; the per-layer figures, the
TFLOP/s and the roofline fractions are reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun, one process per GPU, each rank on its own copy of
the batch (weak scaling, no collective on the data path; a barrier and a max
over ranks of the timed region only).  `--impl reference` times the fp64 CPU
oracle on a bounded sample of the same workload (rank 0 only).

Inputs stay resident in HBM during the timed region; 6 rotating sets of
input/output buffers (377 MB, about 3x the 129 MB L2) keep each step's reads
out of L2.  The `e2e` figure goes through the public API with pinned host
buffers and counts the host<->device copies.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from encoder_only_transformer_gb300 import workloads as W  # noqa: E402

METRIC = "attention tokens/s and TFLOP/s (local & global layer) at 8192 tok, % of roofline"
UNIT = "tokens/s"
HEADS, HEAD_DIM = 12, 64
FLOP_PER_PAIR = 4 * HEAD_DIM * HEADS           # QK^T + PV, all heads: 3072
BYTES_PER_TOKEN = (2304 + 768) * 2             # read qkv once, write out once
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
N_SETS = 6

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) on the
# one-sequence 8192-token workload: the median over the kernel's launches in
# one ncu capture of this bench command.  Reported only while the kernel
# sources still hash to what was captured.
NCU_TRAFFIC = {
    "global": {"bytes": 38.63e6, "kernel": "attn_global_kernel",
               "sources": {"attn_global.cu": "87cc8c905c71723d", "common.cuh": "c9dc0987f95761ca"}},
    "local": {"bytes": 37.83e6, "kernel": "attn_local_kernel",
              "sources": {"attn_local.cu": "061aa162a27f1530", "common.cuh": "c9dc0987f95761ca"}},
    "out_proj": {"bytes": 26.38e6, "kernel": "out_proj_kernel",
                 "sources": {"projections.cu": "0c50f79aa2716b43", "common.cuh": "c9dc0987f95761ca"}},
    "qkv_proj": {"bytes": 16.15e6, "kernel": "qkv_proj_kernel",
                 "sources": {"projections.cu": "0c50f79aa2716b43", "common.cuh": "c9dc0987f95761ca"}},
    "layernorm": {"bytes": 12.59e6, "kernel": "layernorm_kernel",
                  "sources": {"layernorm.cu": "e66f36105992687b", "common.cuh": "c9dc0987f95761ca"}},
    "mlp_up": {"bytes": 16.17e6, "kernel": "mlp_up_kernel",
               "sources": {"projections.cu": "0c50f79aa2716b43", "common.cuh": "c9dc0987f95761ca"}},
    "mlp_down": {"bytes": 33.26e6, "kernel": "mlp_down_kernel",
                 "sources": {"projections.cu": "0c50f79aa2716b43", "common.cuh": "c9dc0987f95761ca"}},
}

WORKLOADS = {
    "config3": (3, "1 sequence x 8192 tokens, qkv [8192,2304] bf16 ~ N(0,1), seed 3"),
    "config4": (4, "65536 tokens, L ~ U{128..8192} packed, qkv bf16 ~ N(0,0.5), seed 4"),
}


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------

def admitted_pairs(lengths, kind, half_window=64):
    """Sum over rows of the admitted-set size per head: L^2 on a global
    layer; on a local layer 129 L - 4160 for L >= 65 (L^2 below)."""
    tot = 0
    for L in lengths:
        if kind == "global" or L <= half_window + 1:
            tot += L * L
        else:
            # 2hw+1 keys per row, minus hw - i missing keys for row i < hw at
            # each end of the sequence
            tot += (2 * half_window + 1) * L - half_window * (half_window + 1)
    return tot


def work(lengths, kind):
    T = sum(lengths)
    return {"flops": FLOP_PER_PAIR * admitted_pairs(lengths, kind),
            "bytes": BYTES_PER_TOKEN * T}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def captured_traffic(kind, workload):
    """DRAM bytes per launch of a kernel ("global" / "local": the layer's
    attention kernel; "out_proj", "qkv_proj", "layernorm": the projections
    and the norm), or None if no capture applies (none taken, another
    workload, or the kernel source changed since)."""
    import hashlib
    rec = NCU_TRAFFIC.get(kind)
    if rec is None or workload != "config3":
        return None
    csrc = os.path.join(ROOT, "encoder_only_transformer_gb300", "csrc")
    for name, digest in rec["sources"].items():
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest()[:16] != digest:
                    return None
        except OSError:
            return None
    return rec["bytes"]


def bench_config(workload, desc, wl, world):
    """The `config` object of both arms' JSON lines (the same workload)."""
    return {"workload": f"{workload}: {desc}; step = 1 global + 1 local layer",
            "tokens_per_step_per_gpu": wl.T, "n_seqs": wl.n_seqs,
            "l2": f"inputs larger than L2 across steps: {N_SETS} rotating qkv/out buffer sets "
                  "on the GPU (the oracle arm reads host memory)",
            "parallelism": f"{world} independent replica(s), no collective"}


def max_over_ranks(x: float, world: int, device) -> float:
    """Max of a per-rank float over all ranks (the slowest rank's time)."""
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return x


def whole_job_tokens_per_s(tokens_per_rank: int, world: int, max_ms: float) -> float:
    """Weak scaling: every rank processes its own batch; the job's rate is
    the tokens of all ranks over the slowest rank's time."""
    return world * tokens_per_rank / (max_ms / 1e3)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class Clocks:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device):
        self.proc = None
        self.ident = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.ident = str(device.index)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100", "-i", self.ident],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"error": "nvidia-smi unavailable"}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out = self.proc.communicate(timeout=10)[0]
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out = self.proc.communicate()[0]
        sm, mx, reasons = [], [], set()
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[3:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"error": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample
# ---------------------------------------------------------------------------

def time_oracle(wl, rows_global, rows_local, seed=0, threads=0):
    """Seconds per query row (all 12 heads) of the fp64 oracle, per kind, on
    `threads` host threads (0: all)."""
    import oracle
    bits = W.bf16_bits(wl.qkv)
    cu = wl.cu_seqlens.numpy()
    out = {}
    for kind, n in (("global", rows_global), ("local", rows_local)):
        per_seq = max(2, n // max(1, wl.n_seqs))
        rows = W.sample_rows(wl.cu_seqlens, per_seq, seed + (kind == "local"))
        t0 = time.perf_counter()
        oracle.attention_kind(bits, cu, kind, rows=rows, threads=threads)
        out[kind] = ((time.perf_counter() - t0) / len(rows), len(rows))
    return out, (threads if threads > 0 else oracle.max_threads())


def cpu_baseline(wl, budget_s=15.0):
    """The oracle as it stands, on a sample sized to ~budget_s of CPU work,
    extrapolated to tokens/s through one global + one local layer."""
    probe, cores = time_oracle(wl, 16, 128)
    share = budget_s / 2
    ng = int(min(wl.T, max(16, share / max(probe["global"][0], 1e-9))))
    nl = int(min(wl.T, max(128, share / max(probe["local"][0], 1e-9))))
    per_row, cores = time_oracle(wl, ng, nl, seed=1)
    sec_per_token = per_row["global"][0] + per_row["local"][0]
    # the same oracle on one host thread, on a sample of about budget_s / 4
    # seconds (a row on one thread costs about `cores` times its share above)
    ng1 = int(min(wl.T, max(8, share / 4 / max(per_row["global"][0] * cores, 1e-9))))
    nl1 = int(min(wl.T, max(64, share / 4 / max(per_row["local"][0] * cores, 1e-9))))
    one, _ = time_oracle(wl, ng1, nl1, seed=2, threads=1)
    sec_one = one["global"][0] + one["local"][0]
    return {"value": 1.0 / sec_per_token, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"fp64 oracle, {per_row['global'][1]} sampled query rows of the global "
                       f"layer and {per_row['local'][1]} of the local layer (all 12 heads), "
                       f"time per row extrapolated to {wl.T} tokens"),
            "one_thread": {"value": 1.0 / sec_one, "unit": UNIT, "cores": 1,
                           "sample": (f"{one['global'][1]} global and {one['local'][1]} local "
                                      "sampled query rows on one host thread")}}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch.distributed as dist
    from encoder_only_transformer_gb300 import binding

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg_id, desc = WORKLOADS[args.workload]
    wl = W.config(cfg_id)
    T, L = wl.T, wl.max_seqlen
    attn = binding.Attention(dev.index)
    attn.reserve(T, wl.n_seqs)
    cu = wl.cu_seqlens.to(dev)
    qkv_sets = [wl.qkv.to(dev) for _ in range(N_SETS)]
    out_sets = [(torch.empty(T, 768, dtype=torch.bfloat16, device=dev),
                 torch.empty(T, 768, dtype=torch.bfloat16, device=dev)) for _ in range(N_SETS)]

    def step(i, kinds=("global", "local")):
        q = qkv_sets[i % N_SETS]
        og, ol = out_sets[i % N_SETS]
        for kind in kinds:
            attn.forward(q, cu, kind, max_seqlen=L, out=og if kind == "global" else ol)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if attn.get_error() != 0:
        raise RuntimeError("device error during warm-up")

    # --- the timed region: K steps as the library runs them (each kernel's
    # launch may overlap the end of the one before it), one event pair
    # around all of them
    clocks = Clocks(dev)
    attn.profile_read()
    barrier()
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        step(i)
    e1.record()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    _, _, launches = attn.profile_read()
    if attn.get_error() != 0:
        raise RuntimeError("device error in the timed region")

    # --- the same K steps again with a CUDA event pair around every
    # attention kernel (the events keep each kernel apart from its
    # neighbours): the kernel durations behind the roofline figures
    attn.profile(True)
    barrier()
    for i in range(args.steps):
        step(i)
    barrier()
    clock_rec = clocks.stop()
    kern_ms, kern_n, _ = attn.profile_read()
    attn.profile(False)
    if attn.get_error() != 0:
        raise RuntimeError("device error in the profiled steps")

    # A call's host side (argument checks, launch) can take longer than a
    # short kernel, and then an event pair around the call also times the
    # idle GPU waiting for the launch.  The loops below that time one kind of
    # call alone first queue a spin kernel, so that the host enqueues the
    # calls ahead of the GPU and the events see only device work.
    def queue_ahead(calls):
        torch.cuda._sleep(int(calls * 60e-6 * 2.0e9))    # ~60 us of host time per call

    # --- per layer kind: the whole call (all its kernels), timed alone
    per_kind = {}
    kk = max(3, args.steps // 2)
    for kind in ("global", "local"):
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        queue_ahead(kk)
        a.record()
        for i in range(kk):
            step(i, (kind,))
        b.record()
        barrier()
        per_kind[kind] = max_over_ranks(a.elapsed_time(b), world, dev) / kk

    # --- the step after the block: y = x + out Wo^T on the global layer's
    # output (synthetic Wo ~ N(0, 1/768), x ~ N(0, 1)), timed alone
    gw = torch.Generator().manual_seed(4242)
    wo = (torch.randn(768, 768, generator=gw) / 768 ** 0.5).to(torch.bfloat16).to(dev)
    x_sets = [torch.randn(T, 768, generator=gw).to(torch.bfloat16).to(dev) for _ in range(N_SETS)]
    y_sets = [torch.empty(T, 768, dtype=torch.bfloat16, device=dev) for _ in range(N_SETS)]
    for i in range(3):
        attn.out_proj(out_sets[i % N_SETS][0], wo, x_sets[i % N_SETS], out=y_sets[i % N_SETS])
    kp = max(20, args.steps)
    attn.profile_read()
    attn.profile(True)
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    queue_ahead(kp)
    a.record()
    for i in range(kp):
        attn.out_proj(out_sets[i % N_SETS][0], wo, x_sets[i % N_SETS], out=y_sets[i % N_SETS])
    b.record()
    barrier()
    attn.profile(False)
    proj_call_ms = max_over_ranks(a.elapsed_time(b), world, dev) / kp
    p_ms, p_n, _ = attn.profile_read()
    proj_ms = max_over_ranks(p_ms["out_proj"], world, dev) / max(1, p_n["out_proj"])

    # --- the step before the block: qkv = LayerNorm(x) Wqkv^T on the same
    # residual rows x (synthetic norm weight 1 + 0.1 N(0, 1), Wqkv ~
    # N(0, 1/768)), timed alone: the norm kernel and the GEMM separately
    gq = torch.Generator().manual_seed(4243)
    norm_w = (1.0 + 0.1 * torch.randn(768, generator=gq)).to(torch.bfloat16).to(dev)
    wqkv = (torch.randn(2304, 768, generator=gq) / 768 ** 0.5).to(torch.bfloat16).to(dev)
    lnq_out = [torch.empty(T, 2304, dtype=torch.bfloat16, device=dev) for _ in range(N_SETS)]
    for i in range(3):
        attn.ln_qkv(x_sets[i % N_SETS], norm_w, wqkv, out=lnq_out[i % N_SETS])
    attn.profile_read()
    attn.profile(True)
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    queue_ahead(kp)
    a.record()
    for i in range(kp):
        attn.ln_qkv(x_sets[i % N_SETS], norm_w, wqkv, out=lnq_out[i % N_SETS])
    b.record()
    barrier()
    attn.profile(False)
    lnq_call_ms = max_over_ranks(a.elapsed_time(b), world, dev) / kp
    p_ms, p_n, _ = attn.profile_read()
    qkvp_ms = max_over_ranks(p_ms["qkv_proj"], world, dev) / max(1, p_n["qkv_proj"])
    ln_ms = max_over_ranks(p_ms["layernorm"], world, dev) / max(1, p_n["layernorm"])
    del lnq_out

    # --- the layer's second block: y = x + MLP(LayerNorm(x)) on the residual
    # rows (synthetic norm weight 1 + 0.1 N(0, 1), Wi ~ N(0, 1/768), Wo ~
    # N(0, 1/1152)), timed alone: its three kernels separately
    gm = torch.Generator().manual_seed(4244)
    mlp_w = (1.0 + 0.1 * torch.randn(768, generator=gm)).to(torch.bfloat16).to(dev)
    mlp_wi = (torch.randn(2304, 768, generator=gm) / 768 ** 0.5).to(torch.bfloat16).to(dev)
    mlp_wo = (torch.randn(768, 1152, generator=gm) / 1152 ** 0.5).to(torch.bfloat16).to(dev)
    for i in range(3):
        attn.mlp(x_sets[i % N_SETS], mlp_w, mlp_wi, mlp_wo, out=y_sets[i % N_SETS])
    attn.profile_read()
    attn.profile(True)
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    queue_ahead(kp)
    a.record()
    for i in range(kp):
        attn.mlp(x_sets[i % N_SETS], mlp_w, mlp_wi, mlp_wo, out=y_sets[i % N_SETS])
    b.record()
    barrier()
    attn.profile(False)
    mlp_call_ms = max_over_ranks(a.elapsed_time(b), world, dev) / kp
    p_ms, p_n, _ = attn.profile_read()
    mlp_ms = {k: max_over_ranks(p_ms[k], world, dev) / max(1, p_n[k])
              for k in ("layernorm", "mlp_up", "mlp_down")}

    # --- a whole encoder layer of each kind from the library's calls:
    # qkv = LN(x) Wqkv^T, attention, x1 = x + a Wo^T, y = x1 + MLP(x1), on
    # the step's packing; one event pair around each run of layers
    lay_qkv = torch.empty(T, 2304, dtype=torch.bfloat16, device=dev)
    lay_a = torch.empty(T, 768, dtype=torch.bfloat16, device=dev)
    lay_x1 = torch.empty(T, 768, dtype=torch.bfloat16, device=dev)

    def layer(i, kind):
        x_in = x_sets[i % N_SETS]
        attn.ln_qkv(x_in, norm_w, wqkv, out=lay_qkv)
        attn.forward(lay_qkv, cu, kind, max_seqlen=L, out=lay_a)
        attn.out_proj(lay_a, wo, x_in, out=lay_x1)
        attn.mlp(lay_x1, mlp_w, mlp_wi, mlp_wo, out=y_sets[i % N_SETS])

    layer_ms = {}
    for kind in ("global", "local"):
        for i in range(3):
            layer(i, kind)
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        queue_ahead(4 * kk)
        a.record()
        for i in range(kk):
            layer(i, kind)
        b.record()
        barrier()
        layer_ms[kind] = max_over_ranks(a.elapsed_time(b), world, dev) / kk
    del lay_qkv, lay_a, lay_x1

    # --- the padded-batch call: 8 rows of 2048 positions holding sequences
    # of U{128..2048} real tokens (seeded), each layer kind, against the
    # packed call on the same tokens
    rng = np.random.default_rng(4245)
    pad_B, pad_S = 8, 2048
    pad_len = rng.integers(128, pad_S + 1, pad_B)
    pad_mask = torch.zeros(pad_B, pad_S, dtype=torch.int32)
    for bb, Lb in enumerate(pad_len):
        pad_mask[bb, :Lb] = 1
    gp = torch.Generator().manual_seed(4245)
    pad_qkv = torch.randn(pad_B, pad_S, 2304, generator=gp).to(torch.bfloat16).to(dev)
    pad_mask = pad_mask.to(dev)
    pad_out = torch.empty(pad_B, pad_S, 768, dtype=torch.bfloat16, device=dev)
    pk_qkv = torch.cat([pad_qkv[bb, :Lb] for bb, Lb in enumerate(pad_len)])
    pk_cu = torch.tensor(np.concatenate([[0], np.cumsum(pad_len)]), dtype=torch.int32, device=dev)
    pk_out = torch.empty(pk_qkv.shape[0], 768, dtype=torch.bfloat16, device=dev)
    padded = {"batch": pad_B, "seq_len": pad_S, "real_tokens": int(pad_len.sum())}
    for kind in ("global", "local"):
        res = {}
        for name, call in (("padded", lambda: attn.forward_padded(pad_qkv, pad_mask, kind, out=pad_out)),
                           ("packed", lambda: attn.forward(pk_qkv, pk_cu, kind, max_seqlen=pad_S, out=pk_out))):
            for _ in range(3):
                call()
            barrier()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            queue_ahead(kk)
            a.record()
            for _ in range(kk):
                call()
            b.record()
            barrier()
            res[name] = max_over_ranks(a.elapsed_time(b), world, dev) / kk
        padded[kind] = {"ms_padded": res["padded"], "ms_packed": res["packed"],
                        "real_tokens_per_s": int(pad_len.sum()) / (res["padded"] / 1e3)}
    padded["note"] = ("forward_padded (pack, attention kernels, unpack) against forward on the "
                      "same tokens packed; not part of the step")
    del pad_qkv, pad_out, pk_qkv, pk_out

    # --- the 22-layer schedule: 32 packed sequences of 8192 tokens (262144
    # tokens), layer i global iff i % 3 == 0, each layer's qkv ~ N(0, 1)
    # drawn from seed 1000 + i by the device's generator (drawing 22 x 604 M
    # values on the host would take minutes).  One event pair around each
    # pass of all 22 layers; the attention kernels' own durations from one
    # more pass with an event pair around each kernel.
    sched_raw = None
    if not args.no_schedule:
        s_len = [8192] * 32
        s_T = sum(s_len)
        s_cu = W.cu_from_lengths(s_len).to(dev)
        s_kinds = [W.layer_kind(i) for i in range(22)]
        s_qkv = []
        for i in range(22):
            gd = torch.Generator(device=dev)
            gd.manual_seed(1000 + i)
            s_qkv.append(torch.randn(s_T, 2304, generator=gd, device=dev).to(torch.bfloat16))
        s_out = torch.empty(s_T, 768, dtype=torch.bfloat16, device=dev)
        attn.reserve(s_T, len(s_len))

        def sched_pass():
            for i in range(22):
                attn.forward(s_qkv[i], s_cu, s_kinds[i], max_seqlen=8192, out=s_out)

        sched_pass()
        barrier()
        reps = 3
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            sched_pass()
        b.record()
        barrier()
        s_ms = max_over_ranks(a.elapsed_time(b), world, dev) / reps
        attn.profile_read()
        attn.profile(True)
        sched_pass()
        barrier()
        sk_ms, sk_n, _ = attn.profile_read()
        attn.profile(False)
        if attn.get_error() != 0:
            raise RuntimeError("device error in the 22-layer schedule")
        sched_raw = (s_len, s_kinds, reps, s_ms,
                     {k: max_over_ranks(sk_ms[k], world, dev) / max(1, sk_n[k]) for k in ("global", "local")})
        del s_qkv, s_out

    # --- end to end through the public API, pinned host buffers.  Every step
    # uploads both layers' qkv and reads both outputs back.  Copies and
    # compute are pipelined the way a serving loop would run them: uploads
    # on one stream, the two attention calls on another, downloads on a
    # third, device buffers double-buffered across steps.
    host_in = [wl.qkv.pin_memory(), wl.qkv.clone().pin_memory()]
    host_out = [[torch.empty(T, 768, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
                for _ in range(2)]
    dev_in = [[torch.empty_like(qkv_sets[0]) for _ in range(2)] for _ in range(2)]
    dev_out = [[torch.empty(T, 768, dtype=torch.bfloat16, device=dev) for _ in range(2)]
               for _ in range(2)]
    s_up, s_comp, s_down = (torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev))
    ev = lambda: torch.cuda.Event()
    in_free = [[None, None], [None, None]]      # compute done reading dev_in[b][j]
    out_free = [[None, None], [None, None]]     # download done with dev_out[b][j]

    def e2e_step(i):
        b = i & 1
        for j, kind in enumerate(("global", "local")):
            up = ev()
            with torch.cuda.stream(s_up):
                if in_free[b][j] is not None:
                    s_up.wait_event(in_free[b][j])
                dev_in[b][j].copy_(host_in[j], non_blocking=True)
                up.record(s_up)
            done = ev()
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(up)
                if out_free[b][j] is not None:
                    s_comp.wait_event(out_free[b][j])
                binding.attention(dev_in[b][j], cu, kind, max_seqlen=L, out=dev_out[b][j])
                done.record(s_comp)
            in_free[b][j] = done
            down = ev()
            with torch.cuda.stream(s_down):
                s_down.wait_event(done)
                host_out[b][j].copy_(dev_out[b][j], non_blocking=True)
                down.record(s_down)
            out_free[b][j] = down

    def all_sync():
        for st in (s_up, s_comp, s_down):
            st.synchronize()

    for i in range(3):
        e2e_step(i)
    all_sync()
    ke = max(3, args.steps // 4)
    barrier()
    t0 = time.perf_counter()
    for i in range(ke):
        e2e_step(i)
    all_sync()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world, dev) / ke
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    peaks, src = load_peaks()
    ms_step = ms / args.steps
    layers = {}
    for kind in ("global", "local"):
        wk = work(wl.lengths, kind)
        t_kernel = kern_ms[kind] / max(1, kern_n[kind]) / 1e3
        t_call = per_kind[kind] / 1e3
        roof_t = max(wk["flops"] / (peaks["bf16_tflops"] * 1e12), wk["bytes"] / (peaks["hbm_gbs"] * 1e9))
        layers[kind] = {
            "tokens_per_s": T / t_call,
            "ms_per_call": per_kind[kind],
            "attn_kernel_ms": t_kernel * 1e3,
            "tflops": wk["flops"] / t_kernel / 1e12,
            "hbm_gbs": wk["bytes"] / t_kernel / 1e9,
            "bound": "tensor" if wk["flops"] / (peaks["bf16_tflops"] * 1e12) >= wk["bytes"] / (peaks["hbm_gbs"] * 1e9) else "hbm",
            "roofline_frac_kernel": roof_t / t_kernel,
            "roofline_frac_call": roof_t / t_call,
            "gflop": wk["flops"] / 1e9,
            "mbytes": wk["bytes"] / 1e6,
        }
    pf = 2.0 * T * 768 * 768
    pb = 2.0 * (3 * T * 768 + 768 * 768)       # read out and x, write y, read Wo once
    p_roof = max(pf / (peaks["bf16_tflops"] * 1e12), pb / (peaks["hbm_gbs"] * 1e9))
    out_proj = {"kernel": "out_proj_kernel", "kernel_ms": proj_ms, "ms_per_call": proj_call_ms,
                "tflops": pf / (proj_ms / 1e3) / 1e12, "hbm_gbs": pb / (proj_ms / 1e3) / 1e9,
                "bound": "hbm" if pb / (peaks["hbm_gbs"] * 1e9) >= pf / (peaks["bf16_tflops"] * 1e12) else "tensor",
                "roofline_frac": p_roof / (proj_ms / 1e3), "gflop": pf / 1e9, "mbytes": pb / 1e6,
                "traffic": captured_traffic("out_proj", args.workload),
                "note": "y = x + out Wo^T after the global layer, timed alone over "
                        f"{kp} calls enqueued ahead of the GPU: kernel_ms from a CUDA event "
                        "pair around each launch, ms_per_call from one pair around all "
                        "calls; not part of the step"}
    qf = 2.0 * T * 768 * 2304
    qb = 2.0 * (T * 768 + T * 2304 + 2304 * 768)   # read h, write qkv, read Wqkv once
    q_roof = max(qf / (peaks["bf16_tflops"] * 1e12), qb / (peaks["hbm_gbs"] * 1e9))
    lb = 2.0 * (2 * T * 768 + 768)                 # read x, write h, read the weight
    l_roof = lb / (peaks["hbm_gbs"] * 1e9)
    ln_qkv = {
        "ms_per_call": lnq_call_ms,
        "qkv_proj": {"kernel": "qkv_proj_kernel", "kernel_ms": qkvp_ms,
                     "tflops": qf / (qkvp_ms / 1e3) / 1e12, "hbm_gbs": qb / (qkvp_ms / 1e3) / 1e9,
                     "bound": "tensor" if qf / (peaks["bf16_tflops"] * 1e12) >= qb / (peaks["hbm_gbs"] * 1e9) else "hbm",
                     "roofline_frac": q_roof / (qkvp_ms / 1e3), "gflop": qf / 1e9, "mbytes": qb / 1e6,
                     "traffic": captured_traffic("qkv_proj", args.workload)},
        "layernorm": {"kernel": "layernorm_kernel", "kernel_ms": ln_ms,
                      "hbm_gbs": lb / (ln_ms / 1e3) / 1e9, "bound": "hbm",
                      "roofline_frac": l_roof / (ln_ms / 1e3), "mbytes": lb / 1e6,
                      "traffic": captured_traffic("layernorm", args.workload)},
        "note": "qkv = LayerNorm(x) Wqkv^T from the residual rows x (the step before the "
                f"block), timed alone over {kp} calls enqueued ahead of the GPU; kernel_ms "
                "from a CUDA event pair around each launch; not part of the step"}
    uf, df = 2.0 * T * 768 * 2304, 2.0 * T * 1152 * 768
    ub = 2.0 * (T * 768 + T * 1152 + 2304 * 768)          # read h, write GELU(g) * u, read Wi
    db = 2.0 * (T * 1152 + 2 * T * 768 + 768 * 1152)      # read it and x, write y, read Wo

    def gemm_rec(kernel, flops, nbytes, ms):
        t = ms / 1e3
        roof = max(flops / (peaks["bf16_tflops"] * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9))
        return {"kernel": kernel, "kernel_ms": ms, "tflops": flops / t / 1e12,
                "hbm_gbs": nbytes / t / 1e9,
                "bound": "tensor" if flops / (peaks["bf16_tflops"] * 1e12) >= nbytes / (peaks["hbm_gbs"] * 1e9) else "hbm",
                "roofline_frac": roof / t, "gflop": flops / 1e9, "mbytes": nbytes / 1e6}
    mlp = {"ms_per_call": mlp_call_ms,
           "layernorm": {"kernel": "layernorm_kernel", "kernel_ms": mlp_ms["layernorm"],
                         "hbm_gbs": lb / (mlp_ms["layernorm"] / 1e3) / 1e9,
                         "roofline_frac": l_roof / (mlp_ms["layernorm"] / 1e3)},
           "mlp_up": dict(gemm_rec("mlp_up_kernel", uf, ub, mlp_ms["mlp_up"]),
                          traffic=captured_traffic("mlp_up", args.workload)),
           "mlp_down": dict(gemm_rec("mlp_down_kernel", df, db, mlp_ms["mlp_down"]),
                            traffic=captured_traffic("mlp_down", args.workload)),
           "note": "y = x + (GELU(g) * u) Wo^T after the MLP's LayerNorm, timed alone over "
                   f"{kp} calls enqueued ahead of the GPU; not part of the step"}
    layer_flops = {k: qf + pf + uf + df + layers[k]["gflop"] * 1e9 for k in ("global", "local")}
    encoder_layer = {
        k: {"ms_per_layer": layer_ms[k], "tokens_per_s": whole_job_tokens_per_s(T, world, layer_ms[k]),
            "tflops": layer_flops[k] / (layer_ms[k] / 1e3) / 1e12,
            "calls": "ln_qkv, attention, out_proj, mlp (8 or 9 kernels)"}
        for k in ("global", "local")}
    encoder_layer["note"] = ("one whole encoder layer from the library's calls on the step's "
                             f"packing, {kk} layers per event pair, enqueued ahead of the GPU; "
                             "synthetic weights; not part of the step")
    schedule = None
    if sched_raw is not None:
        s_len, s_kinds, reps, s_ms, sk = sched_raw
        s_T = sum(s_len)
        sw = {k: work(s_len, k) for k in ("global", "local")}
        s_roof = {k: max(sw[k]["flops"] / (peaks["bf16_tflops"] * 1e12), sw[k]["bytes"] / (peaks["hbm_gbs"] * 1e9))
                  for k in sw}
        s_flops = sum(sw[k]["flops"] for k in s_kinds)
        s_bytes = sum(sw[k]["bytes"] for k in s_kinds)
        s_t = s_ms / 1e3
        schedule = {
            "workload": f"config5: {len(s_len)} sequences x 8192 tokens = {s_T} tokens, 22 layers "
                        f"({s_kinds.count('global')} global, {s_kinds.count('local')} local; layer i "
                        "global iff i % 3 == 0), qkv per layer ~ N(0, 1) bf16 from seed 1000 + i "
                        "on the device's generator",
            "ms_per_schedule": s_ms,
            "layer_tokens_per_s": 22 * s_T / s_t,
            "tflops": s_flops / s_t / 1e12,
            "tflop": s_flops / 1e12,
            "gbytes": s_bytes / 1e9,
            "roofline_frac": sum(s_roof[k] for k in s_kinds) / s_t,
            "global": {"attn_kernel_ms": sk["global"], "tflops": sw["global"]["flops"] / (sk["global"] / 1e3) / 1e12,
                       "bound": "tensor", "roofline_frac": s_roof["global"] / (sk["global"] / 1e3)},
            "local": {"attn_kernel_ms": sk["local"], "hbm_gbs": sw["local"]["bytes"] / (sk["local"] / 1e3) / 1e9,
                      "bound": "hbm", "roofline_frac": s_roof["local"] / (sk["local"] / 1e3)},
            "note": f"not part of the step; one CUDA event pair around each of {reps} passes of "
                    "the 22 layers' attention calls; kernel durations from one more pass with an "
                    "event pair around each attention kernel; roofline_frac of the schedule = the "
                    "sum of the layers' roofline times over the measured time"}
    g, lo = layers["global"], layers["local"]
    calls = {"global": "plan_rope_kernel, attn_global_kernel",
             "local": "attn_local_kernel" if wl.n_seqs <= 256 else "plan_kernel, attn_local_kernel"}
    # The dominant kernel (the global layer's) against the tensor peak; the
    # local layer's kernel, HBM bound, against the copy bandwidth.  Kernel
    # times are CUDA-event pairs around each launch over a second pass of
    # the same K steps (the timed region itself carries no per-kernel
    # events), with the SM clock at its maximum (see "clocks"), so the burst
    # peaks.
    roofline = {"bound": "tensor", "achieved": g["tflops"], "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": g["tflops"] / peaks["bf16_tflops"],
                "frac_call": g["roofline_frac_call"],
                "traffic": captured_traffic("global", args.workload),
                "kernel": "attn_global_kernel (global layer)",
                "call": f"frac_call: the whole global call ({calls['global']}), from one event "
                        f"pair around {kk} back-to-back calls enqueued ahead of the GPU",
                "peak_source": f"{src} bf16_tflops (burst)"}
    roofline_local = {"bound": "hbm", "achieved": lo["hbm_gbs"], "peak": peaks["hbm_gbs"],
                      "unit": "GB/s", "frac": lo["hbm_gbs"] / peaks["hbm_gbs"],
                      "frac_call": lo["roofline_frac_call"],
                      "traffic": captured_traffic("local", args.workload),
                      "kernel": "attn_local_kernel (local layer)",
                      "call": f"frac_call: the whole local call ({calls['local']}), from one event "
                              f"pair around {kk} back-to-back calls enqueued ahead of the GPU",
                      "peak_source": f"{src} hbm_gbs"}
    rec = {
        "metric": METRIC,
        "value": whole_job_tokens_per_s(T, world, ms_step),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": bench_config(args.workload, desc, wl, world),
        "timing": "value: one CUDA event pair around K steps; kernel durations: an event "
                  "pair around each attention kernel over a second pass of the K steps",
        "layers": layers,
        "out_proj": out_proj,
        "ln_qkv": ln_qkv,
        "mlp": mlp,
        "encoder_layer": encoder_layer,
        "padded": padded,
        "schedule": schedule,
        "roofline": roofline,
        "roofline_local": roofline_local,
        "gpu_launches": launches,
        "clocks": clock_rec,
        "e2e": {"value": whole_job_tokens_per_s(T, world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": 2 * T * 2304 * 2, "d2h_bytes_per_step": 2 * T * 768 * 2},
    }
    if not args.no_cpu_baseline:
        rec["cpu_baseline"] = cpu_baseline(wl, args.cpu_budget)
    if world > 1:
        dist.destroy_process_group()
    return rec


# ---------------------------------------------------------------------------
# reference arm: the oracle, as it stands, on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    cfg_id, desc = WORKLOADS[args.workload]
    wl = W.config(cfg_id)
    probe, cores = time_oracle(wl, 16, 128)
    # each step: a sample sized so that warm-up + steps take ~args.cpu_budget * 8 s in all
    per_step = max(0.05, args.cpu_budget * 8 / max(1, args.steps + args.warmup))
    ng = int(min(wl.T, max(2, per_step / 2 / max(probe["global"][0], 1e-9))))
    nl = int(min(wl.T, max(2, per_step / 2 / max(probe["local"][0], 1e-9))))
    for i in range(args.warmup):
        time_oracle(wl, ng, nl, seed=100 + i)
    per_token = 0.0
    rows = None
    t0 = time.perf_counter()
    for i in range(args.steps):
        r, cores = time_oracle(wl, ng, nl, seed=1000 + i)
        per_token += r["global"][0] + r["local"][0]
        rows = (r["global"][1], r["local"][1])
    wall_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    sec_per_token = per_token / args.steps
    value = 1.0 / sec_per_token
    sample = (f"fp64 oracle, per step {rows[0]} sampled query rows of the global layer and "
              f"{rows[1]} of the local layer (all 12 heads); tokens/s = 1 / (seconds per "
              "row of the global layer + seconds per row of the local layer)")
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": wall_ms,
        "ms_per_step_extrapolated": 1e3 * sec_per_token * wl.T,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": bench_config(args.workload, desc, wl, world),
        "timing": "ms_per_step: wall time of each timed step, a bounded sample of the "
                  "workload's query rows; ms_per_step_extrapolated: the same rate over every "
                  f"row of the {wl.T}-token step",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="config3")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-schedule", action="store_true",
                    help="skip the 22-layer schedule over 262144 tokens")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rec = run_reference(args) if args.impl == "reference" else run_ours(args)
    if rec is not None:
        print(json.dumps(rec), flush=True)


if __name__ == "__main__":
    main()
