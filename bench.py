#!/usr/bin/env python3
"""Throughput of the pre-LN ViT encoder block forward on GB300.

One step = one vit_block call over one batch: every stage of the block (LN1, QKV
GEMM, attention, Wo GEMM + residual, LN2, W1 GEMM + GELU, W2 GEMM + residual) on
N sequences of the chosen block shape. Default workload: the ViT-B/16-shaped block
(N 256, T 197, D 768, H 12, F 3072) in bf16 with fp32 accumulation.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config vit_b16]
  python bench.py --impl reference ...   # the float64 CPU oracle, as the reference arm

Prints one JSON line (rank 0). For N > 1 (torchrun, one process per GPU) each rank
runs the whole workload on its own GPU with its own seed (independent sequences, no
collective on the data path); value = all ranks' tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from vision_transformer_encoder_gb300 import api  # noqa: E402
from vision_transformer_encoder_gb300.inputs import CONFIGS, make_config_inputs, make_encoder_inputs  # noqa: E402

METRIC = "ViT block tokens/s and TFLOP/s (% of GB300 dense peak) at ViT-B/16 bf16, 1 GPU"
METRIC_F32 = "ViT block tokens/s and TFLOP/s at ViT-B/16 fp32 (3xTF32 tensor-core products), 1 GPU"
# fp32 path: its products are three TF32 tensor-core products each, so its contraction peak
# is the measured bf16 peak x the nominal TF32 / BF16 dense ratio (1.1 / 2.25) / 3; an
# attention the tensor-core kernel does not take (head width other than 64, or T > 224)
# runs on the CUDA cores: 152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz.
TF32X3_OF_BF16 = (1.1 / 2.25) / 3.0
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
UNIT = "tokens/s"
PATCH_METRIC = "ViT patch-embedding front end tokens/s at ViT-B/16 width bf16, 1 GPU"
ENCODER_METRIC = "ViT encoder (%d blocks + final LN) tokens/s at ViT-B/16 width bf16, 1 GPU"
CLS_METRIC = "ViT CLS-only last block tokens/s at ViT-B/16 bf16, 1 GPU"
ENCODER_CLS_METRIC = ("ViT encoder (%d blocks, the last CLS-only, + final LN of the CLS rows) tokens/s at "
                      "ViT-B/16 width bf16, 1 GPU")
L2_FLUSH_BYTES = 512 << 20  # > 126 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def workload_name(name, c):
    label = {"vit_b16": "ViT-B/16", "vit_ti16": "ViT-Ti/16", "vit_l16_384": "ViT-L/16@384",
             "vit_h14_448": "ViT-H/14@448", "tiny": "tiny"}[name]
    return ("%s-shaped pre-LN encoder block forward: N=%d sequences x T=%d tokens, D=%d, H=%d "
            "(d_h=%d), F=%d, eps=%g" % (label, c["N"], c["T"], c["D"], c["H"], c["D"] // c["H"],
                                        c["F"], c["eps"]))


def flops_per_step(c):
    N, T, D, F = c["N"], c["T"], c["D"], c["F"]
    return 2 * N * T * (4 * D * D + 2 * D * F) + 4 * N * T * T * D


def cls_flops_per_step(c):
    """The CLS-only block: K/V projections of every row; query, attention, output
    projection and MLP of the N CLS rows."""
    N, T, D, F = c["N"], c["T"], c["D"], c["F"]
    return 2 * N * T * D * 2 * D + 2 * N * (2 * D * D + 2 * D * F) + 4 * N * T * D


def kernel_work(c, f32=False):
    """Algorithmic work per launch of each kernel: (bound, amount, unit). f32: the fp32
    path (fp32 activations, 3xTF32 tensor-core products in the GEMMs and, at head width 64
    and T <= 224, in the attention; CUDA-core attention otherwise)."""
    N, T, D, F = c["N"], c["T"], c["D"], c["F"]
    M = N * T
    if f32:
        return {
            # LayerNorms read fp32 rows and write xn and its low part (the next product's A_lo)
            "ln1": ("hbm", M * D * (4 + 4 + 4), "bytes"),
            "qkv_gemm": ("tensor", 2 * M * D * 3 * D, "flops"),
            "attention": ("tensor" if D // c["H"] == 64 and T <= 224 else "alu", 4 * N * T * T * D, "flops"),
            "wo_gemm_residual": ("tensor", 2 * M * D * D, "flops"),
            "ln2": ("hbm", M * D * (4 + 4 + 4), "bytes"),
            "w1_gemm_gelu": ("tensor", 2 * M * D * F, "flops"),
            "w2_gemm_residual": ("tensor", 2 * M * F * D, "flops"),
            # weights read once, written twice (transposed high and low parts)
            "tf32_weight_split": ("hbm", (4 * D * D + 2 * D * F) * 4 * 3, "bytes"),
        }
    return {
        "ln1": ("hbm", M * D * (2 + 2), "bytes"),          # read x bf16, write xn bf16
        "qkv_gemm": ("tensor", 2 * M * D * 3 * D, "flops"),
        "attention": ("tensor", 4 * N * T * T * D, "flops"),
        "wo_gemm_residual": ("tensor", 2 * M * D * D, "flops"),
        "ln2": ("hbm", M * D * (4 + 2), "bytes"),          # read y fp32, write yn bf16
        "w1_gemm_gelu": ("tensor", 2 * M * D * F, "flops"),
        "w2_gemm_residual": ("tensor", 2 * M * F * D, "flops"),
        # LayerNorm folded into the GEMMs (opt-in, VIT_LN_FOLD=1): LN1 reduces to row
        # statistics of x; the fold's column terms are computed once per call
        "ln1_row_stats": ("hbm", M * D * 2 + M * 8, "bytes"),
        "ln_fold_prep": ("hbm", (3 * D * D + D * F) * 2 + (3 * D + F) * 8, "bytes"),
        # stacks: the final LayerNorm reads the fp32 stream and writes bf16
        "final_ln": ("hbm", M * D * (4 + 2), "bytes"),
        # patch-embedding front end (images 3 x 224 x 224, P 16: T - 1 patches of 768)
        "patchify": ("hbm", N * (T - 1) * 768 * 2 * 2, "bytes"),
        "patch_gemm": ("tensor", 2 * N * (T - 1) * 768 * D, "flops"),
        "patch_assemble": ("hbm", N * (T - 1) * D * 4 + M * D * 2, "bytes"),
        # CLS-only last block: K/V of all rows; one query row per sequence
        "kv_gemm": ("tensor", 2 * M * D * 2 * D, "flops"),
        "cls_q_gemm": ("tensor", 2 * N * D * D, "flops"),
        "cls_attention": ("hbm", M * 2 * D * 2 + N * D * 2 * 2, "bytes"),   # K, V read; q read, o written
        "cls_wo_gemm_residual": ("tensor", 2 * N * D * D, "flops"),
        "cls_ln2": ("hbm", N * D * (4 + 2), "bytes"),
        "cls_w1_gemm_gelu": ("tensor", 2 * N * D * F, "flops"),
        "cls_w2_gemm_residual": ("tensor", 2 * N * F * D, "flops"),
    }


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic():
    """DRAM bytes per launch from a committed ncu summary, keyed by kernel; an entry is
    used only while the source file it was measured on is unchanged (same sha256)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic_vit_b16.txt")
    out = {}
    if not os.path.exists(p):
        return out
    for line in open(p):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if len(parts) != 4:
            continue
        kern, nbytes, src, sha = parts
        path = os.path.join(ROOT, src)
        if os.path.exists(path) and hashlib.sha256(open(path, "rb").read()).hexdigest()[:16] == sha:
            out[kern] = int(float(nbytes))
    return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms in the background."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "20"]
        if self.gpu_id is not None:
            cmd += ["-i", str(self.gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        window = [r for r in rows if t0 <= r[0] <= t1]
        note = "sampled every 20 ms during the timed region"
        if len(window) < 3:
            window = rows
            note = "timed region shorter than 3 samples: warm-up and timed region together"
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in window for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in window),
                "sm_max_mhz": max(r[2] for r in window), "reasons": reasons,
                "samples": len(window), "note": note}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def reduce_max(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_baseline(name, c):
    """The float64 oracle on the host cores, on a bounded sample of the workload."""
    import oracle
    cores = oracle.max_threads()
    # sixteen sequences per host core (the whole ViT-B/16 batch on a 16-core host): about
    # ten seconds of oracle time
    n = max(1, min(16 * cores, c["N"]))
    inp = make_config_inputs(name, dtype=torch.bfloat16, N=n)
    t = time.perf_counter()
    oracle.vit_block(inp.x, *inp.weights(), c["H"], c["eps"], nthreads=cores)
    dt = time.perf_counter() - t
    return {"value": n * c["T"] / dt, "unit": UNIT, "cores": min(cores, n), "kind": "oracle",
            "sample": "%d of the %d sequences (%d tokens each), float64 straight loops, OpenMP "
                      "over sequences, %.1f s wall" % (n, c["N"], c["T"], dt)}


def run_reference(args):
    """Reference arm: the float64 CPU oracle as it stands, on the host cores."""
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import oracle
    name = args.config
    c = CONFIGS[name]
    cores = oracle.max_threads()
    K, W = args.steps, args.warmup
    # one sequence per host core: a step costs about one sequence's time on one core
    n = max(1, min(cores, c["N"]))
    inp = make_config_inputs(name, dtype=torch.bfloat16, N=n)
    x = inp.x[:n]
    ws = inp.weights()
    for _ in range(W):
        oracle.vit_block(x, *ws, c["H"], c["eps"], nthreads=cores)
    times = []
    for _ in range(K):
        t = time.perf_counter()
        oracle.vit_block(x, *ws, c["H"], c["eps"], nthreads=cores)
        times.append(time.perf_counter() - t)
    total = sum(times)
    value = K * n * c["T"] / total
    sample = ("each step: %d of the %d sequences (%d tokens each) of the workload, float64 "
              "straight loops, OpenMP over sequences" % (n, c["N"], c["T"]))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": K, "warmup": W, "ms_per_step": 1e3 * total / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(name, c), "tokens_per_step": n * c["T"]},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(cores, n), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# the other block shapes of the workload list in bf16, and the fp32 path (3xTF32 tensor
# cores) at the ViT-Ti/16 shape, which the list gives in fp32 too, and at ViT-B/16
OTHER_CONFIGS = (("vit_ti16", False), ("vit_l16_384", False), ("vit_h14_448", False),
                 ("vit_ti16", True), ("vit_b16", True))


def time_other_configs(K, W, flush, stream, sampler):
    """The other workloads, after the headline: per workload W warm-up steps, K steps
    timed with events on the launching stream (L2 flushed between steps, outside the
    events), then K steps with per-kernel events for the slowest kernel. Returns
    {name: figures}; fp32 entries are named "<shape>_f32" and their fractions are of the
    3xTF32 contraction peak."""
    peaks, _ = load_peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    res = {}
    for name, f32 in OTHER_CONFIGS:
        c = CONFIGS[name]
        dt = torch.float32 if f32 else torch.bfloat16
        tc_peak = peaks["bf16_tflops"] * (TF32X3_OF_BF16 if f32 else 1.0)
        d = make_config_inputs(name, seed=0, dtype=dt).to(device=dev)
        out = torch.empty_like(d.x)

        def step():
            api.vit_block(d.x, *d.weights(), c["H"], c["eps"], out=out, stream=stream)

        for _ in range(W):
            step()
        torch.cuda.synchronize()
        t0 = time.time()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        ms = sum(a.elapsed_time(b) for a, b in ev) / K
        api.timing_reset()
        api.timing_enable(True)
        for _ in range(K):
            flush.zero_()
            step()
        torch.cuda.synchronize()
        api.timing_enable(False)
        pk = {k: v for k, v in api.timing_collect().items() if v[1] > 0}
        dom = max(pk, key=lambda k: pk[k][0])
        bound, amount, _u = kernel_work(c, f32)[dom]
        dom_s = pk[dom][0] / pk[dom][1] / 1e3
        tfl = flops_per_step(c) / (ms / 1e3) / 1e12
        dom_fig = amount / dom_s / (1e9 if bound == "hbm" else 1e12)
        dom_peak = {"tensor": tc_peak, "alu": FP32_ALU_TFLOPS, "hbm": peaks["hbm_gbs"]}[bound]
        res[name + ("_f32" if f32 else "")] = {
                     "workload": workload_name(name, c), "dtype": "f32" if f32 else "bf16", "ms_per_step": ms,
                     "tokens_per_s": c["N"] * c["T"] / (ms / 1e3), "tflops": tfl,
                     "frac_of_peak": tfl / tc_peak, "steps": K, "warmup": W,
                     "dominant_kernel": {"kernel": dom, "avg_us": dom_s * 1e6, "bound": bound,
                                         "achieved": dom_fig, "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                                         "frac": dom_fig / dom_peak},
                     "kernels_us": {k: 1e3 * v[0] / v[1] for k, v in pk.items()},
                     "clocks": sampler.summary(t0, t1)}
        del d, out
    return res


def time_prepared(inp, c, K, W, flush, stream):
    """The headline block on prepared weights (vit_weights_create / vit_block_w), plain
    and with both LayerNorms folded into the products that follow them; K steps each,
    timed as the headline. Returns {"plain_ms", "fold_ms", "fold_speedup"}."""
    dev = torch.device("cuda", torch.cuda.current_device())
    d = inp.to(device=dev)
    layer = dict(zip(("w_q", "w_k", "w_v", "w_o", "w_mlp1", "w_mlp2"), d.weights()))
    out = torch.empty_like(d.x)
    res = {}
    for key, fold in (("plain_ms", 0), ("fold_ms", 1)):
        w = api.VitWeights(layer, c["H"], fold=fold)
        for _ in range(W):
            api.vit_block_w(d.x, w, c["eps"], out=out, stream=stream)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            api.vit_block_w(d.x, w, c["eps"], out=out, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
        res[key] = sum(a.elapsed_time(b) for a, b in ev) / K
        w.close()
    res["fold_speedup"] = res["plain_ms"] / res["fold_ms"]
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="vit_b16", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=30,
                    help="steps of the host-buffer end-to-end measurement (0: skip it)")
    ap.add_argument("--n-seq", type=int, default=None,
                    help="override the number of sequences N (profiling of a smaller case)")
    ap.add_argument("--patch-embed", action="store_true",
                    help="time vit_patch_embed: N images of 3 x 224 x 224, 16 x 16 patches, CLS "
                         "row and positions, into (N, 197, D) tokens")
    ap.add_argument("--encoder-layers", type=int, default=0,
                    help="time vit_encoder: this many blocks with Q/K/V/O biases, LN affine "
                         "terms and the final LayerNorm, instead of one block")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f32"],
                    help="f32: time the fp32 path of the block (3xTF32 products)")
    ap.add_argument("--cls-only", action="store_true",
                    help="the last block computes the CLS rows alone: vit_block_cls (with "
                         "--encoder-layers 0) or vit_encoder_cls")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the Ti, L/16@384 and H/14@448 block timings added after the headline")
    ap.add_argument("--other-steps", type=int, default=50,
                    help="timed steps per other block configuration")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank, world, local = dist_setup()
    name = args.config
    c = dict(CONFIGS[name])
    if args.n_seq:
        c["N"] = args.n_seq
    H, eps = c["H"], c["eps"]
    dev = torch.device("cuda", torch.cuda.current_device())
    f32 = args.dtype == "f32"
    if f32 and (args.patch_embed or args.cls_only or args.encoder_layers):
        ap.error("--dtype f32 times the single block only")
    inp = make_config_inputs(name, seed=rank, dtype=torch.float32 if f32 else torch.bfloat16, N=c["N"])
    d = inp.to(device=dev)
    out = torch.empty_like(d.x)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    L = args.encoder_layers

    if args.patch_embed:
        g = torch.Generator().manual_seed(rank)
        K = 3 * 16 * 16
        pim = torch.randn(c["N"], 3, 224, 224, generator=g).to(torch.bfloat16).to(dev)
        pw = (torch.randn(K, c["D"], generator=g) / K ** 0.5).to(torch.bfloat16).to(dev)
        pb = (torch.randn(c["D"], generator=g) * 0.02).to(torch.bfloat16).to(dev)
        pcls = (torch.randn(c["D"], generator=g) * 0.02).to(torch.bfloat16).to(dev)
        ppos = (torch.randn(197, c["D"], generator=g) * 0.02).to(torch.bfloat16).to(dev)

        def step():
            api.vit_patch_embed(pim, 16, pw, b=pb, cls=pcls, pos=ppos, out=out, stream=stream)
    elif args.cls_only:
        ex, elayers, elnf_g, elnf_b = make_encoder_inputs(c["N"], c["T"], c["D"], c["F"], max(L, 1), seed=rank,
                                                          dtype=torch.bfloat16, device=dev)
        out = torch.empty((c["N"], c["D"]), dtype=torch.bfloat16, device=dev)
        if L == 0:
            def step():
                api.vit_block_cls(ex, elayers[0], H, eps, out=out, stream=stream)
        else:
            def step():
                api.vit_encoder(ex, elayers, H, eps, lnf_g=elnf_g, lnf_b=elnf_b, out=out, stream=stream,
                                cls_only=True)
    elif L > 0:
        ex, elayers, elnf_g, elnf_b = make_encoder_inputs(c["N"], c["T"], c["D"], c["F"], L, seed=rank,
                                                          dtype=torch.bfloat16, device=dev)

        def step():
            api.vit_encoder(ex, elayers, H, eps, lnf_g=elnf_g, lnf_b=elnf_b, out=out, stream=stream)
    else:
        def step():
            api.vit_block(d.x, *d.weights(), H, eps, out=out, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[local] \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else None
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.2)
    K = args.steps

    def timed_pass(per_kernel_events):
        # K steps, each bracketed by events on the launching stream; L2 flushed between
        # steps outside the events. With per_kernel_events the library also brackets
        # each of its launches with a pair of events on the same stream.
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        api.timing_reset()
        api.timing_enable(per_kernel_events)
        barrier(world)
        torch.cuda.synchronize()
        n0 = api.launch_count()
        for k in range(K):
            flush.zero_()
            starts[k].record(stream)
            step()
            ends[k].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        n = api.launch_count() - n0
        api.timing_enable(False)
        return sum(s.elapsed_time(e) for s, e in zip(starts, ends)), n

    # The headline pass runs the steps as a user does, without per-kernel events: an
    # event between two launches serialises them (the next launch no longer overlaps the
    # previous kernel's drain), which adds microseconds per launch. A second pass of the
    # same K steps with events around every launch gives the per-kernel durations that
    # the roofline uses (each slightly inflated by its own events: a conservative figure).
    t0 = time.time()
    step_ms_sum, launches = timed_pass(False)
    t1 = time.time()
    kernel_pass_ms, _ = timed_pass(True)
    per_kernel = api.timing_collect()
    single_block = L == 0 and not args.patch_embed and not args.cls_only
    others = None
    prepared = None
    if (single_block and not f32 and world == 1 and not args.n_seq and name == "vit_b16"
            and not args.no_other_configs):
        others = time_other_configs(args.other_steps, args.warmup, flush, stream, sampler)
        prepared = time_prepared(inp, c, args.other_steps, args.warmup, flush, stream)
    time.sleep(0.1)
    sampler.stop()
    total_ms = reduce_max(step_ms_sum, world)
    kernel_pass_total = reduce_max(kernel_pass_ms, world)
    tokens = c["N"] * c["T"]
    value = world * tokens * K / (total_ms / 1e3)
    ms_per_step = total_ms / K

    # end to end through the host-buffer entry points (pinned host memory), the weights
    # copied to the device once beforehand (vit_weights_create, outside the timed region)
    # as a serving process holds its model, so each step moves its x in and its out back:
    #  - value: vit_block_w_host_async, successive batches issued on a ring of three
    #    streams, each with its own pinned x and out, so that one batch's copies overlap
    #    the blocks of its neighbours; timed from the first call to the last result landed
    #  - per_call: vit_block_w_host, one synchronous call per batch (each call chunks its
    #    batch to overlap its own copies)
    #  - weights_copied_every_call: vit_block_host, which copies the weights in as well
    e2e = None
    if args.e2e_steps > 0 and single_block:
        pinned = [t.pin_memory() for t in [inp.x] + inp.weights()]
        hout = torch.empty_like(pinned[0]).pin_memory()
        wts = api.VitWeights(dict(zip(("w_q", "w_k", "w_v", "w_o", "w_mlp1", "w_mlp2"), pinned[1:])), H,
                             device=dev.index)
        ring = 3
        xs = [pinned[0]] + [torch.roll(inp.x, r, 0).pin_memory() for r in range(1, ring)]
        houts = [hout] + [torch.empty_like(hout).pin_memory() for _ in range(1, ring)]
        rstreams = [torch.cuda.Stream(device=dev) for _ in range(ring)]

        def streamed(n):
            for i in range(n):
                api.vit_block_w_host_async(xs[i % ring], wts, eps, houts[i % ring], rstreams[i % ring])
            for rs in rstreams:
                rs.synchronize()

        def timed(call):
            call()
            barrier(world)
            te = time.perf_counter()
            for _ in range(args.e2e_steps):
                call()
            return reduce_max(time.perf_counter() - te, world)

        streamed(2 * ring)
        barrier(world)
        te = time.perf_counter()
        streamed(args.e2e_steps)
        e2e_a_s = reduce_max(time.perf_counter() - te, world)
        e2e_s = timed(lambda: api.vit_block_w_host(pinned[0], wts, eps, out=hout))
        e2e_w_s = timed(lambda: api.vit_block_host(*pinned, H, eps, out=hout, device=dev.index))
        wts.close()
        xb = pinned[0].numel() * pinned[0].element_size()
        wb = sum(t.numel() * t.element_size() for t in pinned[1:])
        d2h = hout.numel() * hout.element_size()
        e2e = {"value": world * tokens * args.e2e_steps / e2e_a_s, "unit": UNIT,
               "h2d_bytes_per_step": xb, "d2h_bytes_per_step": d2h,
               "steps": args.e2e_steps,
               "ms_per_step": e2e_a_s * 1e3 / args.e2e_steps,
               "api": "vit_block_w_host_async (C ABI, pinned host x and out, one batch per call, successive "
                      "calls on a ring of %d streams; weights prepared on the device once, outside the timed "
                      "region; timed from the first call to the last output landed)" % ring,
               "per_call": {
                   "value": world * tokens * args.e2e_steps / e2e_s, "unit": UNIT,
                   "ms_per_step": e2e_s * 1e3 / args.e2e_steps,
                   "h2d_bytes_per_step": xb, "d2h_bytes_per_step": d2h,
                   "api": "vit_block_w_host (C ABI, pinned host x and out, one synchronous call per batch)"},
               "weights_copied_every_call": {
                   "value": world * tokens * args.e2e_steps / e2e_w_s, "unit": UNIT,
                   "ms_per_step": e2e_w_s * 1e3 / args.e2e_steps,
                   "h2d_bytes_per_step": xb + wb, "d2h_bytes_per_step": d2h,
                   "api": "vit_block_host (C ABI, pinned host buffers, one synchronous call per batch)"}}

    if rank != 0:
        return 0

    peaks, peak_src = load_peaks()
    work = kernel_work(c, f32)
    per_kernel = {k: v for k, v in per_kernel.items() if v[1] > 0}
    dom = max(per_kernel, key=lambda k: per_kernel[k][0])
    kms, kn = per_kernel[dom]
    bound, amount, _unit = work[dom]
    avg_s = kms / kn / 1e3
    # the committed DRAM counters were taken on the bf16 path's kernels
    traffic = None if f32 else load_traffic().get(dom)
    tc_scale = TF32X3_OF_BF16 if f32 else 1.0   # contraction peak of this path's dtype
    if bound == "tensor":
        peak = peaks["bf16_tflops"] * tc_scale
        achieved = amount / avg_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak}
    elif bound == "alu":
        peak = FP32_ALU_TFLOPS
        achieved = amount / avg_s / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak}
    else:
        peak = peaks["hbm_gbs"]
        achieved = amount / avg_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak}
    roof.update({"traffic": traffic, "kernel": dom, "launches": kn,
                 "avg_launch_us": avg_s * 1e6,
                 "algorithmic_per_launch": amount,
                 "peak_source": ("%s (%s)" % (peak_src, "bf16 burst" if not f32 else
                                              "bf16 burst x 1.1 / 2.25 TF32/BF16 nominal / 3 products")
                                 if bound == "tensor" else
                                 "%s (copy)" % peak_src if bound == "hbm" else
                                 "152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz"),
                 "frac_of_sustained": (achieved / (peaks["bf16_tflops_sustained"] * tc_scale)
                                       if bound == "tensor" else None)})
    if args.patch_embed:
        step_flops = 2 * c["N"] * 196 * 768 * c["D"]
    elif args.cls_only:
        step_flops = max(L - 1, 0) * flops_per_step(c) + cls_flops_per_step(c)
    else:
        step_flops = max(L, 1) * flops_per_step(c)
    if args.patch_embed:
        metric = PATCH_METRIC
        workload = ("patch embedding of %d images 3 x 224 x 224 (16 x 16 patches, CLS row, positions) into "
                    "(%d, 197, %d) tokens" % (c["N"], c["N"], c["D"]))
    elif args.cls_only and L == 0:
        metric = CLS_METRIC
        workload = ("CLS-only block (row 0 of each sequence; Q/K/V/O and MLP biases, LN gains) of %s"
                    % workload_name(name, c))
    elif args.cls_only:
        metric = ENCODER_CLS_METRIC % L
        workload = ("%d-block encoder with a CLS-only last block (Q/K/V/O and MLP biases, LN gains, final "
                    "LayerNorm of the CLS rows) of %s" % (L, workload_name(name, c)))
    elif L > 0:
        metric = ENCODER_METRIC % L
        workload = ("%d-block encoder (Q/K/V/O and MLP biases, LN gains, final LayerNorm) of %s"
                    % (L, workload_name(name, c)))
    else:
        metric, workload = (METRIC_F32 if f32 else METRIC), workload_name(name, c)
    step_tflops = step_flops / (ms_per_step / 1e3) / 1e12
    kernels = {k: {"avg_us": 1e3 * v[0] / v[1] if v[1] else None, "launches": v[1],
                   "share": v[0] / sum(x[0] for x in per_kernel.values())}
               for k, v in per_kernel.items()}
    line = {
        "metric": metric,
        "value": value, "unit": UNIT,
        "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32" if f32 else "bf16", "data": "synthetic",
        "config": {"workload": workload,
                   "tokens_per_step_per_gpu": tokens,
                   "inputs": "seeded synthetic: x ~ N(0,1), weights ~ N(0, 1/fan_in), %s" % args.dtype,
                   "l2": "512 MiB written between timed steps (flush); per-step working set "
                         "about 0.9 GB, larger than L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tflops": step_tflops,
        "frac_of_peak": step_tflops / (peaks["bf16_tflops"] * (TF32X3_OF_BF16 if f32 else 1.0)),
        "roofline": roof,
        "kernels": kernels,
        "kernel_pass_ms_per_step": kernel_pass_total / K,
        "gpu_launches": launches,
        "e2e": e2e,
        "clocks": sampler.summary(t0, t1),
    }
    if others is not None:
        line["configs"] = others
    if prepared:
        line["prepared_weights"] = dict(prepared, note=(
            "the headline block on prepared weights (vit_block_w): plain, and with both "
            "LayerNorms folded into the QKV and W1 products (column terms prepared once)"))
    if world == 1 and not args.no_cpu_baseline and single_block:
        line["cpu_baseline"] = cpu_baseline(name, c)
    if args.n_seq:
        line["config"]["note"] = "N overridden on the command line (not the headline workload)"
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
