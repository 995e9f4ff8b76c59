#!/usr/bin/env python3
"""Benchmark of the weight-only quantized linear hot path on GB300.

Workload (one "step"): the full-depth sweep of an LFM3-class hybrid decoder's
linear layers - 16 layers with the FFN (w1, w3: 2048 -> 8192, w2: 8192 -> 2048)
and 6 of them with the attention set (q 2048 -> 2048, k, v 2048 -> 512,
gate 2048 -> 2048, o 2048 -> 2048), MLX affine 4-bit group 64 by default:

  1. decode at R = 1 stream row through all 16 layers (fused q/k/v/gate, o, fused
     w1 + w3 + SwiGLU, w2): the headline "decode qmv HBM GB/s";
  2. the same decode pass at R = 16 rows;
  3. prefill of one 8192-row prompt through the same layers with one M = 8192
     pgemm per linear (SwiGLU between w1/w3 and w2): "pgemm TFLOP/s".

Decode passes are captured once as CUDA graphs (the kernels are a few
microseconds long, so host launch time would otherwise dominate); prefill is
launched directly.  Inputs are seeded synthetic data with the pages' shapes and
distributions; every decode pass reads 502.5 MB of distinct weights, far more than
the 129 MB L2, so no L2 flush is needed between iterations.

Reported beside the step (timed after it): the decode pass with the steps between
the linears (QK norm + partial RoPE + KV store, post-add / next-norm) and those
kernels alone (`decode_post_ops`), and the end-to-end R = 1 pass from pinned host
memory (`e2e`).  `--case window` prints the window-cost table (qlinear_mv_rows vs
qlinear_pgemm for 1..256 rows); `--case pgemm/ffn/mv` time one kernel on one shape
(for profiler captures).

Output: one JSON line (rank 0).  --impl reference times the float64 CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "decode qmv HBM GB/s (% of peak); pgemm TFLOP/s (% of bf16 TC peak)"
D_MODEL, D_FF, D_KV = 2048, 8192, 512
N_LAYERS, N_ATTN = 16, 6
ATTN_LAYERS = [0, 3, 6, 9, 12, 15]  # the 6 attention layers among the 16
PROMPT = 8192

# DRAM traffic per launch of the dominant kernels from one ncu capture, keyed to the
# hash of the kernel source it was taken on; reported as null once the source changes.
NCU_TRAFFIC = {"dc65b8344a25c24c": 45327360 + 212923904}  # pgemm M=8192 N=8192 K=2048, 4-bit (device code as captured)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--bits", type=int, default=4, choices=[4, 6, 8])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", default=None, choices=["pgemm", "ffn", "mv", "window"],
                    help="run only one kernel (for profiler captures): warm-up launches, then --steps launches")
    ap.add_argument("--m", type=int, default=PROMPT, help="--case pgemm: rows of X")
    ap.add_argument("--n", type=int, default=D_FF, help="--case: output channels")
    ap.add_argument("--k", type=int, default=D_MODEL, help="--case: input channels")
    ap.add_argument("--rows", type=int, default=1, help="--case ffn/mv: activation rows")
    ap.add_argument("--copies", type=int, default=1,
                    help="--case ffn/mv: distinct weight copies cycled through (> L2 with enough copies)")
    return ap.parse_args()


def source_hash(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "weight_only_bit_mlx_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm": p["hbm_gbs"], "bf16": p["bf16_tflops"], "bf16_sus": p["bf16_tflops_sustained"],
                "src": "measured"}
    except Exception:  # noqa: BLE001 - the recipe's fallback figures
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sus": 1700.0, "src": "fallback"}


def layer_shapes():
    """(name, n, k) of every linear of the sweep, in execution order."""
    out = []
    for layer in range(N_LAYERS):
        if layer in ATTN_LAYERS:
            out += [(f"L{layer}.q", D_MODEL, D_MODEL), (f"L{layer}.k", D_KV, D_MODEL),
                    (f"L{layer}.v", D_KV, D_MODEL), (f"L{layer}.g", D_MODEL, D_MODEL),
                    (f"L{layer}.o", D_MODEL, D_MODEL)]
        out += [(f"L{layer}.w1", D_FF, D_MODEL), (f"L{layer}.w3", D_FF, D_MODEL), (f"L{layer}.w2", D_MODEL, D_FF)]
    return out


def weight_bytes(n, k, bits):
    return n * k * bits // 8 + 2 * n * (k // 64) * 2


def decode_bytes(bits, rows):
    """Algorithmic bytes of one decode pass: packed weights + scales + biases +
    activations read + outputs written, per launch."""
    total = 0
    for layer in range(N_LAYERS):
        if layer in ATTN_LAYERS:
            nq = 2 * D_MODEL + 2 * D_KV
            total += sum(weight_bytes(n, D_MODEL, bits) for n in (D_MODEL, D_KV, D_KV, D_MODEL))
            total += rows * D_MODEL * 2 + rows * nq * 4                      # fused q/k/v/gate
            total += weight_bytes(D_MODEL, D_MODEL, bits) + rows * D_MODEL * 2 + rows * D_MODEL * 4  # o
        total += 2 * weight_bytes(D_FF, D_MODEL, bits) + rows * D_MODEL * 2 + rows * D_FF * 2   # w1+w3 -> h
        total += weight_bytes(D_MODEL, D_FF, bits) + rows * D_FF * 2 + rows * D_MODEL * 4       # w2
    return total


def prefill_flops():
    return sum(2 * PROMPT * n * k for _, n, k in layer_shapes())


def workload_config(bits, world):
    """The `config` object both arms report: the workload the metric is quoted on."""
    return {"workload": f"full-depth sweep: 16 layers (FFN 2048->8192->2048) + 6 attention sets "
                        f"(q,g,o 2048->2048; k,v 2048->512), MLX affine {bits}-bit g64; decode R=1 "
                        f"(value) and R=16, prefill M={PROMPT} pgemm",
            "rows": 1, "prompt_rows": PROMPT, "bits": bits,
            "l2": "no flush: every decode pass streams 502.5 MB of distinct weights (> 129 MB L2)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def max_over_ranks_of(v, world, device):
    """The largest of v over all ranks: a replicated job ends when its slowest rank does."""
    if world == 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, steps, max_ms, world):
    """Whole-job throughput of `world` replicas (weak scaling): every rank processes
    units_per_rank per step, and the job takes the slowest rank's time max_ms."""
    return world * units_per_rank * steps / (max_ms * 1e-3)


# ------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while it runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9 and f[1].replace(".", "").isdigit():
                    rows.append(f)
        except OSError:
            pass
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = np.array([float(r[1]) for r in rows])
        power = np.array([float(r[3]) if r[3].replace(".", "").isdigit() else 0.0 for r in rows])
        loaded = sm[power >= np.median(power)] if len(rows) > 4 else sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower().startswith("active")})
        return {"sm_mhz": float(np.median(loaded)), "sm_max_mhz": float(max(float(r[2]) for r in rows)),
                "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------------------------------
def cpu_baseline_sample(bits, target_s=10.0):
    """The float64 oracle, as it stands, on the host cores: decode of the FFN of one
    layer (w1, w3, SwiGLU, w2) at R = 1, repeated for about target_s seconds."""
    from oracle import qlinear_oracle as orc
    from weight_only_bit_mlx_gb300 import synth
    w1 = synth.make_weight(D_FF, D_MODEL, bits, config_id=4, tensor_id=1)
    w3 = synth.make_weight(D_FF, D_MODEL, bits, config_id=4, tensor_id=3)
    w2 = synth.make_weight(D_MODEL, D_FF, bits, config_id=4, tensor_id=2)
    x = synth.make_x(1, D_MODEL, config_id=4)
    per = (2 * weight_bytes(D_FF, D_MODEL, bits) + D_MODEL * 2 + D_FF * 2
           + weight_bytes(D_MODEL, D_FF, bits) + D_FF * 2 + D_MODEL * 4)
    reps, t0 = 0, time.perf_counter()
    while True:
        _, _, _, _, h = orc.ffn_swiglu(x, w1, w3)
        hb = synth.f32_to_bf16_bits(h.astype(np.float32))
        orc.qlinear_w(hb, w2)
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return {"value": per * reps / el / 1e9, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{reps} x one layer's FFN decode (w1+w3+SwiGLU+w2, 2048->8192->2048, {bits}-bit, R=1) "
                      f"in {el:.1f} s; numpy float64 (BLAS on all cores, unpack/dequant single-threaded)"}


def run_reference(args):
    """--impl reference: the float64 oracle on the host cores, a bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import qlinear_oracle as orc
    from weight_only_bit_mlx_gb300 import synth
    bits = args.bits
    w1 = synth.make_weight(D_FF, D_MODEL, bits, config_id=4, tensor_id=1)
    w3 = synth.make_weight(D_FF, D_MODEL, bits, config_id=4, tensor_id=3)
    w2 = synth.make_weight(D_MODEL, D_FF, bits, config_id=4, tensor_id=2)
    x = synth.make_x(1, D_MODEL, config_id=4)
    per = (2 * weight_bytes(D_FF, D_MODEL, bits) + D_MODEL * 2 + D_FF * 2
           + weight_bytes(D_MODEL, D_FF, bits) + D_FF * 2 + D_MODEL * 4)

    def step():
        _, _, _, _, h = orc.ffn_swiglu(x, w1, w3)
        orc.qlinear_w(synth.f32_to_bf16_bits(h.astype(np.float32)), w2)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = per * args.steps / el / 1e9
    sample = f"per step: one layer's FFN decode (w1+w3+SwiGLU+w2, {bits}-bit, R=1) by the float64 oracle"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(workload_config(bits, 1), sample=sample),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from weight_only_bit_mlx_gb300 import qlinear as q
    from weight_only_bit_mlx_gb300 import synth

    bits = args.bits
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)

    def dev_weight(n, k, tid):
        # seeded synthetic weight drawn on the device (same recipe as synth.make_weight:
        # uniform words, scale ~ U(0.005, 0.02), bias ~ U(-0.1, 0.1), rounded to bf16)
        wq = torch.randint(-2**31, 2**31 - 1, (n, k * bits // 32), generator=gen, dtype=torch.int32, device=dev)
        s = (torch.rand(n, k // 64, generator=gen, device=dev, dtype=torch.float32) * 0.015 + 0.005)
        b = (torch.rand(n, k // 64, generator=gen, device=dev, dtype=torch.float32) * 0.2 - 0.1)
        return q.QWeight(wq, s.to(torch.bfloat16), b.to(torch.bfloat16), k, bits)

    W = {}
    for name, n, k in layer_shapes():
        W[name] = dev_weight(n, k, name)
    torch.cuda.synchronize()

    def rnd_bf16(*shape):
        return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)

    # decode activations and outputs (per R)
    bufs = {}
    for R in (1, 16):
        bufs[R] = {
            "x": rnd_bf16(R, D_MODEL), "attn": rnd_bf16(R, D_MODEL),
            "q": torch.empty(R, D_MODEL, device=dev), "k": torch.empty(R, D_KV, device=dev),
            "v": torch.empty(R, D_KV, device=dev), "g": torch.empty(R, D_MODEL, device=dev),
            "o": torch.empty(R, D_MODEL, device=dev), "h": torch.empty(R, D_FF, dtype=torch.bfloat16, device=dev),
            "y": torch.empty(R, D_MODEL, device=dev),
        }
    launches = {"decode": 0, "prefill": 0}

    def decode_pass(R, count=False):
        b = bufs[R]
        n = 0
        for layer in range(N_LAYERS):
            if layer in ATTN_LAYERS:
                p = f"L{layer}."
                q.qattn_proj_mv(W[p + "q"], W[p + "k"], W[p + "v"], W[p + "g"], b["x"],
                                outs=(b["q"], b["k"], b["v"], b["g"]))
                q.qlinear_mv_rows(W[p + "o"], b["attn"], b["o"])
                n += 2
            q.qffn_swiglu_mv(W[f"L{layer}.w1"], W[f"L{layer}.w3"], b["x"], b["h"])
            q.qlinear_mv_rows(W[f"L{layer}.w2"], b["h"], b["y"])
            n += 2
        return n

    # ---- the steps after the projections (QK norm + partial RoPE + KV store, post-add /
    #      next-norm): head_dim 64 (32 q heads, 8 kv heads), rotary on the first 32 dims,
    #      base 1e6, eps 1e-5, KV rings of 1024 slots per stream
    HD, ROT, RING = 64, 32, 1024
    post = {}
    for R in (1, 16):
        post[R] = {
            "q_out": torch.empty(R, D_MODEL, dtype=torch.bfloat16, device=dev),
            "k_ring": torch.zeros(R, RING, D_KV, dtype=torch.bfloat16, device=dev),
            "v_ring": torch.zeros(R, RING, D_KV, dtype=torch.bfloat16, device=dev),
            "pos": torch.randint(0, 1 << 20, (R,), generator=gen, device=dev, dtype=torch.int32),
            "resid": rnd_bf16(R, D_MODEL),
        }
    qn_w = (torch.rand(HD, generator=gen, device=dev) + 0.5).to(torch.bfloat16)
    kn_w = (torch.rand(HD, generator=gen, device=dev) + 0.5).to(torch.bfloat16)
    gammas = [(torch.rand(D_MODEL, generator=gen, device=dev) + 0.5).to(torch.bfloat16) for _ in range(2)]

    def qknorm(R):
        b, pp = bufs[R], post[R]
        q.qattn_qknorm_rope_kv(b["q"], b["k"], b["v"], D_MODEL // HD, D_KV // HD, HD, ROT, 1e6, 1e-5, qn_w, kn_w,
                               pp["pos"], pp["k_ring"], pp["v_ring"], q_out=pp["q_out"])

    def resid_norm(R, y, gi):
        # the normed output becomes the next linear's activation x
        q.qresid_rmsnorm(y, post[R]["resid"], gammas[gi], 1e-5, out=bufs[R]["x"])

    def decode_layer_pass(R, fused=False):
        """The decode pass with the steps between the linears: per attention layer
        q/k/v/gate -> QK norm + RoPE + KV store -> o -> post-add / next-norm; per layer
        w1 + w3 + SwiGLU -> w2 -> post-add / next-norm (attention itself excluded: o
        reads a fixed attention output)."""
        b = bufs[R]
        n = 0
        for layer in range(N_LAYERS):
            p = f"L{layer}."
            if layer in ATTN_LAYERS:
                q.qattn_proj_mv(W[p + "q"], W[p + "k"], W[p + "v"], W[p + "g"], b["x"],
                                outs=(b["q"], b["k"], b["v"], b["g"]))
                qknorm(R)
                if fused:  # the post-add / next-norm as the matvec's epilogue
                    q.qlinear_mv_resid_norm(W[p + "o"], b["attn"], post[R]["resid"], gammas[0], 1e-5, out=b["x"])
                    n += 3
                else:
                    q.qlinear_mv_rows(W[p + "o"], b["attn"], b["o"])
                    resid_norm(R, b["o"], 0)
                    n += 4
            q.qffn_swiglu_mv(W[p + "w1"], W[p + "w3"], b["x"], b["h"])
            if fused:
                q.qlinear_mv_resid_norm(W[p + "w2"], b["h"], post[R]["resid"], gammas[1], 1e-5, out=b["x"])
                n += 2
            else:
                q.qlinear_mv_rows(W[p + "w2"], b["h"], b["y"])
                resid_norm(R, b["y"], 1)
                n += 3
        return n

    # prefill buffers
    X = rnd_bf16(PROMPT, D_MODEL)
    Pa = torch.empty(PROMPT, D_FF, device=dev)
    Pc = torch.empty(PROMPT, D_FF, device=dev)
    Ph = torch.empty(PROMPT, D_FF, dtype=torch.bfloat16, device=dev)
    Pout = torch.empty(PROMPT, D_MODEL, device=dev)
    Pq = torch.empty(PROMPT, D_MODEL, device=dev)
    Pkv = torch.empty(PROMPT, D_KV, device=dev)
    Patt = rnd_bf16(PROMPT, D_MODEL)
    stream = torch.cuda.current_stream()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    gemm_events = []  # (start, stop, flops) of every pgemm call of the timed steps

    def pgemm(w, Xin, Y, timed):
        if timed:
            e0, e1 = ev(), ev()
            e0.record(stream)
            q.qlinear_pgemm(w, Xin, Y)
            e1.record(stream)
            gemm_events.append((e0, e1, 2 * Xin.shape[0] * w.n * w.k, (int(Xin.shape[0]), w.n, w.k)))
        else:
            q.qlinear_pgemm(w, Xin, Y)

    def prefill_pass(timed=False):
        n = 0
        for layer in range(N_LAYERS):
            p = f"L{layer}."
            if layer in ATTN_LAYERS:
                pgemm(W[p + "q"], X, Pq, timed)
                pgemm(W[p + "k"], X, Pkv, timed)
                pgemm(W[p + "v"], X, Pkv, timed)
                pgemm(W[p + "g"], X, Pq, timed)
                pgemm(W[p + "o"], Patt, Pout, timed)
                n += 10
            pgemm(W[p + "w1"], X, Pa, timed)
            pgemm(W[p + "w3"], X, Pc, timed)
            q.qswiglu(Pa, Pc, Ph)
            pgemm(W[p + "w2"], Ph, Pout, timed)
            n += 7
        return n

    # warm-up (also sizes the library's scratch before any capture)
    for _ in range(max(1, args.warmup)):
        decode_pass(1)
        decode_pass(16)
        prefill_pass()
    torch.cuda.synchronize()

    graphs = {}
    for R in (1, 16):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            launches[f"decode{R}"] = decode_pass(R)
        graphs[R] = g
    for R in (1, 16):
        for fused in (False, True):
            key = f"layer{R}" + ("f" if fused else "")
            decode_layer_pass(R, fused)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                launches[key] = decode_layer_pass(R, fused)
            graphs[key] = g
    for _ in range(args.warmup):
        graphs[1].replay()
        graphs[16].replay()
        for key in ("layer1", "layer16", "layer1f", "layer16f"):
            graphs[key].replay()
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK

    # ---------------- timed region
    marks = []
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_start = ev()
        t_start.record(stream)
        n_launch = 0
        for _ in range(args.steps):
            e = [ev() for _ in range(4)]
            e[0].record(stream)
            graphs[1].replay()
            e[1].record(stream)
            graphs[16].replay()
            e[2].record(stream)
            n_launch += launches["decode1"] + launches["decode16"]
            n_launch += prefill_pass(timed=True)
            e[3].record(stream)
            marks.append(e)
        t_stop = ev()
        t_stop.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    clocks = clk.summary()
    status = q.qlinear_last_error()

    total_ms = t_start.elapsed_time(t_stop)
    d1_ms = sum(m[0].elapsed_time(m[1]) for m in marks)
    d16_ms = sum(m[1].elapsed_time(m[2]) for m in marks)
    pf_ms = sum(m[2].elapsed_time(m[3]) for m in marks)
    gemm_ms = sum(a.elapsed_time(b) for a, b, _, _ in gemm_events)
    gemm_flops = sum(f for _, _, f, _ in gemm_events)
    # the roofline kernel: the M = 8192, N = 8192, K = 2048 launches (w1, w3 of every layer)
    ffn_ev = [(a, b, f) for a, b, f, shape in gemm_events if shape == (PROMPT, D_FF, D_MODEL)]
    ffn_ms = sum(a.elapsed_time(b) for a, b, _ in ffn_ev)
    ffn_flops = sum(f for _, _, f in ffn_ev)

    def max_over_ranks(v):
        return max_over_ranks_of(v, world, dev)

    total_ms, d1_ms, d16_ms, pf_ms, gemm_ms, ffn_ms = (max_over_ranks(v) for v in (total_ms, d1_ms, d16_ms, pf_ms,
                                                                                 gemm_ms, ffn_ms))

    # ---------------- the decode pass with the steps between the linears, and those steps alone
    layer_ms = {}
    for key in ("layer1", "layer16", "layer1f", "layer16f"):
        e0, e1 = ev(), ev()
        e0.record(stream)
        for _ in range(args.steps):
            graphs[key].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        layer_ms[key] = max_over_ranks(e0.elapsed_time(e1)) / args.steps

    def time_kernel(fn, reps=200):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(20):
                fn()
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = ev(), ev()
        e0.record(stream)
        for _ in range(reps // 20):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3  # us per launch (back to back, in a graph)

    post_lines = {}
    for R in (1, 16):
        qk_us = time_kernel(lambda: qknorm(R))
        rn_us = time_kernel(lambda: resid_norm(R, bufs[R]["y"], 1))
        qk_bytes = R * ((D_MODEL + 2 * D_KV) * 4 + (D_MODEL + 2 * D_KV) * 2 + 4) + 2 * HD * 2
        rn_bytes = R * D_MODEL * (4 + 2 + 2 + 2) + D_MODEL * 2
        post_lines[f"r{R}"] = {"qattn_qknorm_rope_kv_us": qk_us, "qattn_qknorm_rope_kv_GB/s": qk_bytes / qk_us / 1e3,
                               "qresid_rmsnorm_us": rn_us, "qresid_rmsnorm_GB/s": rn_bytes / rn_us / 1e3,
                               "layer_pass_ms": layer_ms[f"layer{R}"], "layer_pass_launches": launches[f"layer{R}"],
                               "layer_pass_tok_s_modelled": R / (layer_ms[f"layer{R}"] * 1e-3),
                               "layer_pass_fused_ms": layer_ms[f"layer{R}f"],
                               "layer_pass_fused_launches": launches[f"layer{R}f"],
                               "layer_pass_fused_tok_s_modelled": R / (layer_ms[f"layer{R}f"] * 1e-3)}
    assert q.qlinear_last_error() == q.QL_OK

    # ---------------- end to end: host buffers in pinned memory, copies inside the timed region
    xh = torch.empty(1, D_MODEL, dtype=torch.bfloat16).pin_memory()
    xh.copy_(bufs[1]["x"].cpu())
    yh = torch.empty(1, D_MODEL, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    e0.record(stream)
    for _ in range(args.steps):
        bufs[1]["x"].copy_(xh, non_blocking=True)
        graphs[1].replay()
        yh.copy_(bufs[1]["y"], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1))

    pk = peaks()
    d1_bytes = decode_bytes(bits, 1)
    d16_bytes = decode_bytes(bits, 16)
    value = job_throughput(d1_bytes, args.steps, d1_ms, world) / 1e9
    d16_gbs = job_throughput(d16_bytes, args.steps, d16_ms, world) / 1e9
    pf_tflops = job_throughput(prefill_flops(), args.steps, pf_ms, world) / 1e12
    gemm_tflops = gemm_flops / (gemm_ms * 1e-3) / 1e12  # per GPU, all GEMM launches of the pass
    ffn_tflops = ffn_flops / (ffn_ms * 1e-3) / 1e12      # per GPU, the roofline kernel's launches
    src = source_hash(["pgemm.cu", "common.cuh", "sync.cuh"])
    traffic = NCU_TRAFFIC.get(src)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16xq%d->f32" % bits, "data": "synthetic",
        "config": workload_config(bits, world),
        "decode_r1": {"GB/s": value / world, "frac_of_hbm": value / world / pk["hbm"],
                      "ms_per_pass": d1_ms / args.steps, "bytes_per_pass": d1_bytes,
                      "tok_s_modelled": 1.0 / (d1_ms / args.steps * 1e-3)},
        "decode_post_ops": dict(post_lines, what="QK norm + partial RoPE + KV store after q/k/v/gate and "
                                "post-add / next-norm after o and w2 (head_dim 64, rotary 32, 1024-slot rings); "
                                "layer_pass = the decode pass with them between the linears (graph, timed "
                                "after the main region); layer_pass_fused = the same with the post-add / next-norm "
                                "as the o / w2 matvec's epilogue (qlinear_mv_resid_norm); per-kernel times are back-to-back launches, "
                                "bytes = algorithmic reads + writes (latency-bound at these sizes)"),
        "decode_r16": {"GB/s": d16_gbs / world, "frac_of_hbm": d16_gbs / world / pk["hbm"],
                       "ms_per_pass": d16_ms / args.steps, "bytes_per_pass": d16_bytes,
                       "tok_s_modelled": 16.0 / (d16_ms / args.steps * 1e-3)},
        "prefill": {"TFLOP/s": pf_tflops / world, "ms_per_pass": pf_ms / args.steps,
                    "flops_per_pass": prefill_flops(), "includes": "pgemm (row-sum pre-pass + GEMM) and SwiGLU",
                    "tok_s_modelled": PROMPT / (gemm_ms / args.steps * 1e-3)},
        "tok_s_note": "modelled from the linear layers only: decode R / (decode pass time), prefill "
                      "prompt rows / (sum of the pass's pgemm times); attention, norms and sampling excluded",
        "roofline": {"bound": "tensor", "kernel": "qlinear_pgemm (row-sum pre-pass + tcgen05 GEMM), "
                                                  f"M={PROMPT} N={D_FF} K={D_MODEL} launches (w1, w3)",
                     "achieved": ffn_tflops, "peak": pk["bf16_sus"], "unit": "TFLOP/s",
                     "frac": ffn_tflops / pk["bf16_sus"], "traffic": traffic,
                     "traffic_unit": "bytes per launch (DRAM read + write, one ncu capture of this shape)",
                     "algorithmic_bytes_per_launch": PROMPT * D_MODEL * 2 + weight_bytes(D_FF, D_MODEL, bits)
                     + PROMPT * D_FF * 4,
                     "all_gemm_launches_TFLOP/s": gemm_tflops,
                     "peak_source": f"{pk['src']} bf16 sustained"},
        "roofline_decode": {"bound": "hbm", "kernel": "decode pass R=1 (qattn_proj_mv, qlinear_mv_rows, "
                                                      "qffn_swiglu_mv)",
                            "achieved": value / world, "peak": pk["hbm"], "unit": "GB/s",
                            "frac": value / world / pk["hbm"], "traffic": None,
                            "traffic_note": "per-launch DRAM bytes of the FFN decode kernel equal its algorithmic "
                                            "bytes (ncu: 18.91 MB read for 18.87 MB); no capture of the whole pass",
                            "peak_source": f"{pk['src']} copy bandwidth"},
        "e2e": {"value": job_throughput(d1_bytes, args.steps, e2e_ms, world) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": D_MODEL * 2, "d2h_bytes_per_step": D_MODEL * 4,
                "what": "decode pass R=1 with x copied from pinned host memory and the last output copied back"},
        "gpu_launches": n_launch,
        "clocks": clocks,
        "status": status,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(bits)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_case(args):
    """One kernel on one shape: --warmup launches, then --steps timed launches."""
    import torch
    from weight_only_bit_mlx_gb300 import qlinear as q
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    bits, n, k = args.bits, args.n, args.k

    def w():
        wq = torch.randint(-2**31, 2**31 - 1, (n, k * bits // 32), generator=gen, dtype=torch.int32, device=dev)
        s = (torch.rand(n, k // 64, generator=gen, device=dev) * 0.015 + 0.005).to(torch.bfloat16)
        b = (torch.rand(n, k // 64, generator=gen, device=dev) * 0.2 - 0.1).to(torch.bfloat16)
        return q.QWeight(wq, s, b, k, bits)

    if args.case == "window":
        return window_table(args, q, w, gen, dev)
    if args.case == "pgemm":
        wt = w()
        X = torch.randn(args.m, k, generator=gen, device=dev).to(torch.bfloat16)
        Y = torch.empty(args.m, n, device=dev)
        fn, unit, work = (lambda: q.qlinear_pgemm(wt, X, Y)), "TFLOP/s", 2.0 * args.m * n * k
    elif args.case == "ffn":
        pairs = [(w(), w()) for _ in range(args.copies)]
        x = torch.randn(args.rows, k, generator=gen, device=dev).to(torch.bfloat16)
        h = torch.empty(args.rows, n, dtype=torch.bfloat16, device=dev)
        it = [0]

        def fn():
            w1, w3 = pairs[it[0] % len(pairs)]
            it[0] += 1
            q.qffn_swiglu_mv(w1, w3, x, h)
        unit = "GB/s"
        work = 2 * weight_bytes(n, k, bits) + args.rows * (k * 2 + n * 2)
    else:
        ws = [w() for _ in range(args.copies)]
        x = torch.randn(args.rows, k, generator=gen, device=dev).to(torch.bfloat16)
        y = torch.empty(args.rows, n, device=dev)
        it = [0]

        def fn():
            wt = ws[it[0] % len(ws)]
            it[0] += 1
            q.qlinear_mv_rows(wt, x, y)
        unit = "GB/s"
        work = weight_bytes(n, k, bits) + args.rows * (k * 2 + n * 4)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / max(1, args.steps)
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    print(json.dumps({"case": args.case, "bits": bits, "m": args.m, "n": n, "k": k, "rows": args.rows,
                      "copies": args.copies,
                      "us_per_launch": ms * 1e3, unit: work / (ms * 1e-3) / scale,
                      "status": q.qlinear_last_error()}), flush=True)


def interp_cost(points, rows):
    """Per-call cost of a window of `rows` rows from costs measured at a few window
    sizes (TensorFold PR #1696, later revision, "What it adds": windows are timed at a
    handful of sizes at load and the rest interpolated).  points: [(rows_i, us_i)] with
    distinct rows_i.  Between two measured sizes the cost is the straight line through
    them; below the smallest size it is the smallest size's cost; above the largest it
    follows the last segment (a single measured size is a constant).  Returns None when
    no size was measured."""
    pts = sorted((int(r), float(c)) for r, c in points if c is not None)
    if not pts:
        return None
    if rows <= pts[0][0] or len(pts) == 1:
        return pts[0][1]
    for (r0, c0), (r1, c1) in zip(pts, pts[1:]):
        if rows <= r1:
            return c0 + (c1 - c0) * (rows - r0) / (r1 - r0)
    (r0, c0), (r1, c1) = pts[-2], pts[-1]
    return c0 + (c1 - c0) * (rows - r0) / (r1 - r0)


def window_choice(table, max_rows, mv_max_rows=16):
    """For every window size 1..max_rows, the cheaper call by interpolated cost
    (qlinear_mv_rows only up to mv_max_rows rows), merged into runs:
    [{"rows": [lo, hi], "call": name}, ...]."""
    mv = [(t["rows"], t["mv_rows_us"]) for t in table if t["mv_rows_us"] is not None]
    pg = [(t["rows"], t["pgemm_us"]) for t in table]
    runs = []
    for R in range(1, max_rows + 1):
        c_mv = interp_cost(mv, R) if R <= mv_max_rows else None
        c_pg = interp_cost(pg, R)
        call = "qlinear_mv_rows" if c_mv is not None and (c_pg is None or c_mv <= c_pg) else "qlinear_pgemm"
        if runs and runs[-1]["call"] == call:
            runs[-1]["rows"][1] = R
        else:
            runs.append({"rows": [R, R], "call": call})
    return runs


def window_table(args, q, make_w, gen, dev):
    """Cost of one window of R rows through qlinear_mv_rows (R <= 16) and through
    qlinear_pgemm (any R), with enough distinct weight copies cycled to exceed L2, so
    every call streams its weights from HBM.  Prints the table and, per R, which call
    is cheaper (a window of more than 16 rows can only take the GEMM)."""
    import torch
    n, k = args.n, args.k
    props = torch.cuda.get_device_properties(dev)
    wbytes = weight_bytes(n, k, args.bits)
    copies = max(2, int(2 * props.L2_cache_size // wbytes) + 1)
    ws = [make_w() for _ in range(copies)]
    it = [0]

    def timed(fn, reps=60):
        for _ in range(copies):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3  # us per call

    rows_list = [1, 2, 4, 8, 16, 32, 64, 128, 256]
    table = []
    for R in rows_list:
        X = torch.randn(R, k, generator=gen, device=dev).to(torch.bfloat16)
        Y = torch.empty(R, n, device=dev)

        def nxt():
            wt = ws[it[0] % copies]
            it[0] += 1
            return wt
        mv = timed(lambda: q.qlinear_mv_rows(nxt(), X, Y)) if R <= 16 else None
        pg = timed(lambda: q.qlinear_pgemm(nxt(), X, Y))
        best = "qlinear_mv_rows" if mv is not None and mv <= pg else "qlinear_pgemm"
        table.append({"rows": R, "mv_rows_us": mv, "pgemm_us": pg, "cheaper": best,
                      "us_per_row": min(x for x in (mv, pg) if x is not None) / R})
    print(json.dumps({"case": "window", "bits": args.bits, "n": n, "k": k, "weight_copies": copies,
                      "weight_bytes": wbytes, "table": table,
                      "interpolation": "cost(R) for R between two measured sizes is the linear interpolation "
                                       "of their per-call costs",
                      "choice": window_choice(table, rows_list[-1]),
                      "status": q.qlinear_last_error()}), flush=True)


def main():
    args = parse()
    if args.case is not None:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    sys.path.insert(0, ROOT)
    main()
