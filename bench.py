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
import re
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
# rows from which the library converts the codes once per prompt-GEMM call (one more launch)
PRE_ROWS = 2048
NCU_TRAFFIC = {"6f7a3378bb41c6e9": 121433088 + 229151488}  # pgemm M=8192 N=8192 K=2048, 4-bit (device code as captured)


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
    """Hash of the sources' code: comments and whitespace removed, so that the key of a
    DRAM capture outlives edits that leave the device code as it was."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "weight_only_bit_mlx_gb300", "csrc", n)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
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
def sweep_weight_bytes(bits):
    """Packed codes + scales + biases of every linear of the sweep (one decode pass reads
    each once)."""
    return sum(weight_bytes(n, k, bits) for _, n, k in layer_shapes())


def _oracle_layer_inputs(bits):
    from weight_only_bit_mlx_gb300 import synth
    mk = synth.make_weight
    ffn = {"w1": mk(D_FF, D_MODEL, bits, config_id=4, tensor_id=1), "w3": mk(D_FF, D_MODEL, bits, config_id=4, tensor_id=3),
           "w2": mk(D_MODEL, D_FF, bits, config_id=4, tensor_id=2)}
    attn = {t: mk(n, D_MODEL, bits, config_id=4, tensor_id=10 + i)
            for i, (t, n) in enumerate((("q", D_MODEL), ("k", D_KV), ("v", D_KV), ("g", D_MODEL), ("o", D_MODEL)))}
    x = synth.make_x(1, D_MODEL, config_id=4)
    return ffn, attn, x


def _oracle_ffn_layer(ffn, x):
    from oracle import qlinear_oracle as orc
    from weight_only_bit_mlx_gb300 import synth
    _, _, _, _, h = orc.ffn_swiglu(x, ffn["w1"], ffn["w3"])
    orc.qlinear_w(synth.f32_to_bf16_bits(h.astype(np.float32)), ffn["w2"])


def _oracle_attn_set(attn, x):
    from oracle import qlinear_oracle as orc
    for t in ("q", "k", "v", "g", "o"):
        orc.qlinear_w(x, attn[t])


def ffn_layer_bytes(bits, rows=1):
    return (2 * weight_bytes(D_FF, D_MODEL, bits) + rows * (D_MODEL * 2 + D_FF * 2)
            + weight_bytes(D_MODEL, D_FF, bits) + rows * (D_FF * 2 + D_MODEL * 4))


def attn_set_bytes(bits, rows=1):
    nq = 2 * D_MODEL + 2 * D_KV
    return (sum(weight_bytes(n, D_MODEL, bits) for n in (D_MODEL, D_KV, D_KV, D_MODEL)) + rows * (D_MODEL * 2 + nq * 4)
            + weight_bytes(D_MODEL, D_MODEL, bits) + rows * (D_MODEL * 2 + D_MODEL * 4))


def _timed(fn, min_s):
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_s:
            return el / reps, reps


def cpu_baselines(bits, budget_s=16.0):
    """The float64 oracle, as it stands, on the host cores, for each workload (configs
    0-3 on their own shapes; the full-depth sweep scaled from one layer of each kind).
    About budget_s seconds of CPU work in all."""
    from oracle import qlinear_oracle as orc
    from weight_only_bit_mlx_gb300 import synth
    cores = os.cpu_count()
    kind = "oracle"
    note = "numpy float64 (BLAS on all cores, unpack/dequant single-threaded)"
    out = {}
    per = budget_s / 5
    # config 0: one 2048 -> 2048 qmv, R = 1
    w0 = synth.make_weight(D_MODEL, D_MODEL, bits, config_id=0, tensor_id=0)
    x0 = synth.make_x(1, D_MODEL, config_id=0)
    t, reps = _timed(lambda: orc.qlinear_w(x0, w0), per)
    b0 = weight_bytes(D_MODEL, D_MODEL, bits) + D_MODEL * 2 + D_MODEL * 4
    out["c0_qmv"] = {"value": b0 / t / 1e9, "unit": "GB/s", "cores": cores, "kind": kind,
                     "sample": f"{reps} x qmv 2048->2048 {bits}-bit R=1; {note}"}
    ffn, attn, x = _oracle_layer_inputs(bits)
    t_f, reps = _timed(lambda: _oracle_ffn_layer(ffn, x), per)
    out["c1_ffn_decode"] = {"value": ffn_layer_bytes(bits) / t_f / 1e9, "unit": "GB/s", "cores": cores, "kind": kind,
                            "sample": f"{reps} x one layer's FFN decode (w1+w3+SwiGLU+w2, 2048->8192->2048, "
                                      f"{bits}-bit, R=1); {note}"}
    t_a, reps = _timed(lambda: _oracle_attn_set(attn, x), per)
    out["c2_attn_decode"] = {"value": attn_set_bytes(bits) / t_a / 1e9, "unit": "GB/s", "cores": cores, "kind": kind,
                             "sample": f"{reps} x one layer's attention projections (q, k, v, gate, o; {bits}-bit, "
                                       f"R=1); {note}"}
    pass_s = N_LAYERS * t_f + N_ATTN * t_a
    out["sweep_decode_r1"] = {"value": decode_bytes(bits, 1) / pass_s / 1e9, "unit": "GB/s", "cores": cores,
                              "kind": kind,
                              "sample": f"full-depth decode pass R=1 scaled from one layer of each kind: 16 x "
                                        f"{t_f * 1e3:.0f} ms (FFN) + 6 x {t_a * 1e3:.0f} ms (attention set); {note}"}
    # config 3: the 1024-row prompt GEMM, 2048 -> 8192
    w3 = synth.make_weight(D_FF, D_MODEL, bits, config_id=3, tensor_id=0)
    X3 = synth.make_x(1024, D_MODEL, config_id=3)
    t3, reps = _timed(lambda: orc.pgemm(X3, w3), per)
    f3 = 2.0 * 1024 * D_FF * D_MODEL
    out["c3_pgemm"] = {"value": f3 / t3 / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": kind,
                       "sample": f"{reps} x pgemm X[1024, 2048] x W 2048->8192 {bits}-bit ({f3 / t3 / 1e9:.1f} "
                                 f"GFLOP/s); the M=8192 prefill would take {prefill_flops() / (f3 / t3):.0f} s at "
                                 f"this rate; {note}"}
    return out


def run_reference(args):
    """--impl reference: the float64 oracle on the host cores.  Each step is a bounded
    sample of the workload: one layer's FFN decode and one layer's attention projections
    at R = 1; the throughput is the full-depth decode pass's bytes over the pass time
    those imply (16 FFN layers + 6 attention sets), the metric of the GPU arm's `value`."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    bits = args.bits
    ffn, attn, x = _oracle_layer_inputs(bits)
    for _ in range(args.warmup):
        _oracle_ffn_layer(ffn, x)
        _oracle_attn_set(attn, x)
    t_f = t_a = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_ffn_layer(ffn, x)
        t1 = time.perf_counter()
        _oracle_attn_set(attn, x)
        t2 = time.perf_counter()
        t_f += t1 - t0
        t_a += t2 - t1
    pass_s = (N_LAYERS * t_f + N_ATTN * t_a) / args.steps
    value = decode_bytes(bits, 1) / pass_s / 1e9
    sample = (f"per step: one layer's FFN decode and one layer's attention projections ({bits}-bit, R=1) by the "
              f"float64 oracle; the full-depth pass time scaled from them (16 x FFN + 6 x attention)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": (t_f + t_a) / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(workload_config(bits, 1), sample=sample),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


class Sweep:
    """The full-depth sweep's weights and buffers at one code width, on one device, with
    the passes of the workload: decode at R rows, the 8192-row prefill as one M = 8192
    pgemm per linear, and the same prefill in windows of `win` rows."""

    HD, ROT, RING = 64, 32, 1024  # head_dim, rotary dims, KV ring slots per stream

    def __init__(self, q, bits, gen, dev, with_post=True):
        import torch
        self.q, self.bits, self.gen, self.dev = q, bits, gen, dev
        self.W = {name: self._weight(n, k) for name, n, k in layer_shapes()}

        def rnd(*shape):
            return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
        self.rnd = rnd
        self.bufs = {}
        for R in (1, 16):
            self.bufs[R] = {
                "x": rnd(R, D_MODEL), "attn": rnd(R, D_MODEL),
                "q": torch.empty(R, D_MODEL, device=dev), "k": torch.empty(R, D_KV, device=dev),
                "v": torch.empty(R, D_KV, device=dev), "g": torch.empty(R, D_MODEL, device=dev),
                "o": torch.empty(R, D_MODEL, device=dev), "h": torch.empty(R, D_FF, dtype=torch.bfloat16, device=dev),
                "y": torch.empty(R, D_MODEL, device=dev),
            }
        # prefill buffers
        self.X = rnd(PROMPT, D_MODEL)
        self.Pa = torch.empty(PROMPT, D_FF, device=dev)
        self.Pc = torch.empty(PROMPT, D_FF, device=dev)
        self.Ph = torch.empty(PROMPT, D_FF, dtype=torch.bfloat16, device=dev)
        self.Pout = torch.empty(PROMPT, D_MODEL, device=dev)
        self.Pq = torch.empty(PROMPT, D_MODEL, device=dev)
        self.Pg = torch.empty(PROMPT, D_MODEL, device=dev)
        self.Pkv = torch.empty(PROMPT, D_KV, device=dev)
        self.Pv = torch.empty(PROMPT, D_KV, device=dev)
        self.Patt = rnd(PROMPT, D_MODEL)
        self.Presid = rnd(PROMPT, D_MODEL)      # the residual stream of the prompt rows
        self.Pnorm = torch.empty(PROMPT, D_MODEL, dtype=torch.bfloat16, device=dev)  # next layer's input
        self.pgamma = (torch.rand(D_MODEL, generator=gen, device=dev) + 0.5).to(torch.bfloat16)
        self.gemm_events = []  # (start, stop, flops, (m, n, k)) of the timed pgemm calls
        if with_post:
            self._post_buffers()

    def _weight(self, n, k):
        # seeded synthetic weight drawn on the device (same recipe as synth.make_weight:
        # uniform words, scale ~ U(0.005, 0.02), bias ~ U(-0.1, 0.1), rounded to bf16)
        import torch
        gen, dev, bits = self.gen, self.dev, self.bits
        wq = torch.randint(-2**31, 2**31 - 1, (n, k * bits // 32), generator=gen, dtype=torch.int32, device=dev)
        s = (torch.rand(n, k // 64, generator=gen, device=dev, dtype=torch.float32) * 0.015 + 0.005)
        b = (torch.rand(n, k // 64, generator=gen, device=dev, dtype=torch.float32) * 0.2 - 0.1)
        return self.q.QWeight(wq, s.to(torch.bfloat16), b.to(torch.bfloat16), k, bits)

    def decode_pass(self, R):
        q, W, b = self.q, self.W, self.bufs[R]
        n = 0
        for layer in range(N_LAYERS):
            p = f"L{layer}."
            if layer in ATTN_LAYERS:
                q.qattn_proj_mv(W[p + "q"], W[p + "k"], W[p + "v"], W[p + "g"], b["x"],
                                outs=(b["q"], b["k"], b["v"], b["g"]))
                q.qlinear_mv_rows(W[p + "o"], b["attn"], b["o"])
                n += 2
            q.qffn_swiglu_mv(W[p + "w1"], W[p + "w3"], b["x"], b["h"])
            q.qlinear_mv_rows(W[p + "w2"], b["h"], b["y"])
            n += 2
        return n

    # ---- the steps after the projections (QK norm + partial RoPE + KV store, post-add /
    #      next-norm): head_dim 64 (32 q heads, 8 kv heads), rotary on the first 32 dims,
    #      base 1e6, eps 1e-5, KV rings of 1024 slots per stream
    def _post_buffers(self):
        import torch
        gen, dev, rnd = self.gen, self.dev, self.rnd
        self.post = {}
        for R in (1, 16):
            self.post[R] = {
                "q_out": torch.empty(R, D_MODEL, dtype=torch.bfloat16, device=dev),
                "k_ring": torch.zeros(R, self.RING, D_KV, dtype=torch.bfloat16, device=dev),
                "v_ring": torch.zeros(R, self.RING, D_KV, dtype=torch.bfloat16, device=dev),
                "pos": torch.randint(0, 1 << 20, (R,), generator=gen, device=dev, dtype=torch.int32),
                "resid": rnd(R, D_MODEL),
            }
        self.qn_w = (torch.rand(self.HD, generator=gen, device=dev) + 0.5).to(torch.bfloat16)
        self.kn_w = (torch.rand(self.HD, generator=gen, device=dev) + 0.5).to(torch.bfloat16)
        self.gammas = [(torch.rand(D_MODEL, generator=gen, device=dev) + 0.5).to(torch.bfloat16) for _ in range(2)]

    def qknorm(self, R):
        b, pp = self.bufs[R], self.post[R]
        self.q.qattn_qknorm_rope_kv(b["q"], b["k"], b["v"], D_MODEL // self.HD, D_KV // self.HD, self.HD, self.ROT,
                                    1e6, 1e-5, self.qn_w, self.kn_w, pp["pos"], pp["k_ring"], pp["v_ring"],
                                    q_out=pp["q_out"])

    def resid_norm(self, R, y, gi):
        # the normed output becomes the next linear's activation x
        self.q.qresid_rmsnorm(y, self.post[R]["resid"], self.gammas[gi], 1e-5, out=self.bufs[R]["x"])

    def decode_layer_pass(self, R, fused=False):
        """The decode pass with the steps between the linears: per attention layer
        q/k/v/gate -> QK norm + RoPE + KV store -> o -> post-add / next-norm; per layer
        w1 + w3 + SwiGLU -> w2 -> post-add / next-norm (attention itself excluded: o
        reads a fixed attention output)."""
        q, W, b = self.q, self.W, self.bufs[R]
        n = 0
        for layer in range(N_LAYERS):
            p = f"L{layer}."
            if layer in ATTN_LAYERS:
                q.qattn_proj_mv(W[p + "q"], W[p + "k"], W[p + "v"], W[p + "g"], b["x"],
                                outs=(b["q"], b["k"], b["v"], b["g"]))
                self.qknorm(R)
                if fused:  # the post-add / next-norm as the matvec's epilogue
                    q.qlinear_mv_resid_norm(W[p + "o"], b["attn"], self.post[R]["resid"], self.gammas[0], 1e-5,
                                            out=b["x"])
                    n += 3
                else:
                    q.qlinear_mv_rows(W[p + "o"], b["attn"], b["o"])
                    self.resid_norm(R, b["o"], 0)
                    n += 4
            q.qffn_swiglu_mv(W[p + "w1"], W[p + "w3"], b["x"], b["h"])
            if fused:
                q.qlinear_mv_resid_norm(W[p + "w2"], b["h"], self.post[R]["resid"], self.gammas[1], 1e-5, out=b["x"])
                n += 2
            else:
                q.qlinear_mv_rows(W[p + "w2"], b["h"], b["y"])
                self.resid_norm(R, b["y"], 1)
                n += 3
        return n

    def _pgemm(self, w, Xin, Y, timed):
        import torch
        if timed == "calls":
            st = torch.cuda.current_stream()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            self.q.qlinear_pgemm(w, Xin, Y)
            e1.record(st)
            self.gemm_events.append((e0, e1, 2 * Xin.shape[0] * w.n * w.k, (int(Xin.shape[0]), w.n, w.k)))
        else:
            self.q.qlinear_pgemm(w, Xin, Y)

    def _timed_call(self, fn, timed, flops, tag):
        import torch
        if timed != "calls":
            fn()
            return
        st = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        fn()
        e1.record(st)
        self.gemm_events.append((e0, e1, flops, tag))

    def prefill_pass(self, timed=None, lo=0, hi=PROMPT, fused=False, post=None):
        """Rows lo..hi-1 of the prompt through every linear: one pgemm per linear, the
        SwiGLU as the up projection's epilogue (fused) or as a kernel of its own, and
        with post="fused" / "unfused" the post-add / next-norm after o and w2 (as the
        GEMM's epilogue plus the norm, or the plain GEMM plus qresid_rmsnorm).
        The weights that read the same X (q, k, v, gate; w1, w3) go through one
        qlinear_pgemm_multi each.  timed="pairs": CUDA events around each layer's (w1, w3)
        call only (the roofline kernel's launches, as the layer runs them); timed="calls":
        every GEMM as a qlinear_pgemm call of its own, with events around each.  An event between two calls ends the programmatic
        overlap between them (a call's code conversion can then no longer run in the
        previous GEMM's last tiles), so the pass itself is timed with "pairs" at most.
        Returns the number of launches."""
        import torch
        W, n, q = self.W, 0, self.q
        # launches of one prompt-GEMM call: the row-sum pre-pass and the GEMM, plus the
        # once-per-call code conversion from PRE_ROWS rows on
        pg = 3 if hi - lo >= PRE_ROWS else 2
        X, Patt = self.X[lo:hi], self.Patt[lo:hi]
        Pa, Pc, Ph = self.Pa[lo:hi], self.Pc[lo:hi], self.Ph[lo:hi]
        Pq, Pkv, Pout = self.Pq[lo:hi], self.Pkv[lo:hi], self.Pout[lo:hi]
        Pg, Pv = self.Pg[lo:hi], self.Pv[lo:hi]
        R, Rn = self.Presid[lo:hi], self.Pnorm[lo:hi]

        def down(w, Xin):  # o or w2, then the post-add / next-norm if asked for
            nonlocal n
            if post == "fused":
                q.qlinear_pgemm_resid_norm(w, Xin, R, self.pgamma, 1e-5, out=Rn)
                n += pg + 1
            else:
                self._pgemm(w, Xin, Pout, timed)
                n += pg
                if post == "unfused":
                    q.qresid_rmsnorm(Pout, R, self.pgamma, 1e-5, out=Rn)
                    n += 1

        def multi(ws, outs):
            # the weights that read X: one qlinear_pgemm_multi (the row sums of X formed
            # once), or call by call when every call is timed alone
            nonlocal n
            if timed == "calls":
                for w, out in zip(ws, outs):
                    self._pgemm(w, X, out, timed)
                n += len(ws) * pg
            else:
                q.qlinear_pgemm_multi(ws, X, outs)
                n += len(ws) * (pg - 1) + 1

        for layer in range(N_LAYERS):
            p = f"L{layer}."
            if layer in ATTN_LAYERS:
                multi([W[p + "q"], W[p + "k"], W[p + "v"], W[p + "g"]], [Pq, Pkv, Pv, Pg])
                down(W[p + "o"], Patt)
            if timed == "pairs" and not fused:
                st = torch.cuda.current_stream()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                multi([W[p + "w1"], W[p + "w3"]], [Pa, Pc])
                e1.record(st)
                rows = X.shape[0]
                self.gemm_events.append((e0, e1, 2 * rows * W[p + "w1"].n * W[p + "w1"].k
                                         + 2 * rows * W[p + "w3"].n * W[p + "w3"].k, "ffn_pair"))
                q.qswiglu(Pa, Pc, Ph)
                n += 1
            elif not fused:
                multi([W[p + "w1"], W[p + "w3"]], [Pa, Pc])
                q.qswiglu(Pa, Pc, Ph)
                n += 1
            else:
                self._pgemm(W[p + "w1"], X, Pa, timed)
                self._timed_call(lambda: q.qlinear_pgemm_swiglu(W[p + "w3"], X, Pa, Ph), timed,
                                 2 * X.shape[0] * W[p + "w3"].n * W[p + "w3"].k, "swiglu")
                n += 2 * pg
            down(W[p + "w2"], Ph)
        return n

    def prefill_windows_pass(self, win):
        """The 8192-row prompt in windows of `win` rows, each window through all the
        layers before the next (every window streams every weight again)."""
        n = 0
        for lo in range(0, PROMPT, win):
            n += self.prefill_pass(lo=lo, hi=min(PROMPT, lo + win))
        return n

    def gemm_summary(self, shape=None):
        """(ms, flops) summed over the timed pgemm calls (of one shape, or one tag such as
        "swiglu" for the up projections with the SwiGLU epilogue, if given)."""
        ev = [(a, b, f) for a, b, f, sh in self.gemm_events if shape is None or sh == shape]
        return sum(a.elapsed_time(b) for a, b, _ in ev), sum(f for _, _, f in ev)


def graph_of(fn):
    """Capture fn() once into a CUDA graph; returns (graph, fn's return value)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ret = fn()
    return g, ret


def width_line(q, bits, gen, dev, steps, pk):
    """Decode R = 1 / R = 16 and the M = 8192 prompt GEMM at another code width (the
    same shapes), measured the way the main step measures them."""
    import torch
    sw = Sweep(q, bits, gen, dev, with_post=False)
    sw.decode_pass(1)
    sw.decode_pass(16)
    sw.prefill_pass()
    torch.cuda.synchronize()
    g1, n1 = graph_of(lambda: sw.decode_pass(1))
    g16, _ = graph_of(lambda: sw.decode_pass(16))
    for _ in range(3):
        g1.replay()
        g16.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    ms = {}
    for key, g in (("r1", g1), ("r16", g16)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(steps):
            g.replay()
        e1.record(st)
        torch.cuda.synchronize()
        ms[key] = e0.elapsed_time(e1) / steps
    for _ in range(max(1, steps // 4)):
        sw.prefill_pass(timed="pairs")
    torch.cuda.synchronize()
    gemm_ms, gemm_flops = sw.gemm_summary("ffn_pair")
    tf = gemm_flops / (gemm_ms * 1e-3) / 1e12
    status = q.qlinear_last_error()
    out = {"bits": bits,
           "decode_r1": {"GB/s": decode_bytes(bits, 1) / (ms["r1"] * 1e-3) / 1e9, "ms_per_pass": ms["r1"],
                         "frac_of_hbm": decode_bytes(bits, 1) / (ms["r1"] * 1e-3) / 1e9 / pk["hbm"]},
           "decode_r16": {"GB/s": decode_bytes(bits, 16) / (ms["r16"] * 1e-3) / 1e9, "ms_per_pass": ms["r16"],
                          "frac_of_hbm": decode_bytes(bits, 16) / (ms["r16"] * 1e-3) / 1e9 / pk["hbm"]},
           "pgemm_m8192_n8192_k2048": {"TFLOP/s": tf, "frac_of_sustained": tf / pk["bf16_sus"],
                                       "frac_of_burst": tf / pk["bf16"]},
           "status": status}
    del sw, g1, g16
    torch.cuda.empty_cache()
    return out


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

    bits = args.bits
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    sw = Sweep(q, bits, gen, dev)
    torch.cuda.synchronize()
    launches = {}

    # warm-up (also sizes the library's scratch before any capture); `pre` counts this
    # library's launches before the timed region (the skip count of a launch-list capture)
    pre = 0
    for _ in range(max(1, args.warmup)):
        pre += sw.decode_pass(1) + sw.decode_pass(16) + sw.prefill_pass()
    torch.cuda.synchronize()

    graphs = {}
    for R in (1, 16):
        graphs[R], launches[f"decode{R}"] = graph_of(lambda: sw.decode_pass(R))
    for R in (1, 16):
        for fused in (False, True):
            key = f"layer{R}" + ("f" if fused else "")
            pre += sw.decode_layer_pass(R, fused)
            graphs[key], launches[key] = graph_of(lambda: sw.decode_layer_pass(R, fused))
    # the prompt in windows of 128 rows (north of 10,000 launches: one graph)
    WIN = 128
    graphs["win"], launches["win"] = graph_of(lambda: sw.prefill_windows_pass(WIN))
    for _ in range(args.warmup):
        graphs[1].replay()
        graphs[16].replay()
        pre += launches["decode1"] + launches["decode16"]
        for key in ("layer1", "layer16", "layer1f", "layer16f"):
            graphs[key].replay()
            pre += launches[key]
    graphs["win"].replay()
    pre += launches["win"]
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK

    def ev():
        return torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()

    # ---------------- timed region: K steps of (decode R=1, decode R=16, prefill as one
    #                  M=8192 pgemm per linear, prefill in windows of 128 rows)
    marks = []
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_start = ev()
        t_start.record(stream)
        n_launch = 0
        for _ in range(args.steps):
            e = [ev() for _ in range(5)]
            e[0].record(stream)
            graphs[1].replay()
            e[1].record(stream)
            graphs[16].replay()
            e[2].record(stream)
            n_launch += launches["decode1"] + launches["decode16"]
            n_launch += sw.prefill_pass(timed="pairs")
            e[3].record(stream)
            graphs["win"].replay()
            n_launch += launches["win"]
            e[4].record(stream)
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
    win_ms = sum(m[3].elapsed_time(m[4]) for m in marks)
    # the roofline kernel: the M = 8192, N = 8192, K = 2048 launches (w1, w3 of every layer),
    # timed in pairs
    ffn_ms, ffn_flops = sw.gemm_summary("ffn_pair")

    def max_over_ranks(v):
        return max_over_ranks_of(v, world, dev)

    total_ms, d1_ms, d16_ms, pf_ms, win_ms, ffn_ms = (
        max_over_ranks(v) for v in (total_ms, d1_ms, d16_ms, pf_ms, win_ms, ffn_ms))

    # every GEMM call of one prefill pass timed alone (events around each call), after
    # the timed region
    sw.gemm_events = []
    sw.prefill_pass(timed="calls")
    torch.cuda.synchronize()
    gemm_ms, gemm_flops = sw.gemm_summary()
    gemm_ms = max_over_ranks(gemm_ms)

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
        g, _ = graph_of(lambda: [fn() for _ in range(20)])
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
        qk_us = time_kernel(lambda: sw.qknorm(R))
        rn_us = time_kernel(lambda: sw.resid_norm(R, sw.bufs[R]["y"], 1))
        qk_bytes = R * ((D_MODEL + 2 * D_KV) * 4 + (D_MODEL + 2 * D_KV) * 2 + 4) + 2 * Sweep.HD * 2
        rn_bytes = R * D_MODEL * (4 + 2 + 2 + 2) + D_MODEL * 2
        post_lines[f"r{R}"] = {"qattn_qknorm_rope_kv_us": qk_us, "qattn_qknorm_rope_kv_GB/s": qk_bytes / qk_us / 1e3,
                               "qresid_rmsnorm_us": rn_us, "qresid_rmsnorm_GB/s": rn_bytes / rn_us / 1e3,
                               "layer_pass_ms": layer_ms[f"layer{R}"], "layer_pass_launches": launches[f"layer{R}"],
                               "layer_pass_tok_s_modelled": R / (layer_ms[f"layer{R}"] * 1e-3),
                               "layer_pass_fused_ms": layer_ms[f"layer{R}f"],
                               "layer_pass_fused_launches": launches[f"layer{R}f"],
                               "layer_pass_fused_tok_s_modelled": R / (layer_ms[f"layer{R}f"] * 1e-3)}
    assert q.qlinear_last_error() == q.QL_OK

    # ---------------- the prefill pass with the SwiGLU as a kernel of its own, and with the
    #                  post-add / next-norm after o and w2 (unfused, and as the GEMM's epilogue)
    def time_pass(**kw):
        sw.prefill_pass(**kw)
        torch.cuda.synchronize()
        e0, e1 = ev(), ev()
        e0.record(stream)
        sw.prefill_pass(**kw)
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1))
    pf_variants = {"swiglu_epilogue_ms": time_pass(fused=True),
                   "post_unfused_ms": time_pass(post="unfused"),
                   "post_fused_ms": time_pass(post="fused")}
    sw.gemm_events = []
    sw.prefill_pass(fused=True, timed="calls")  # the up projections with the SwiGLU epilogue, call by call
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK

    # ---------------- end to end: host buffers in pinned memory, copies inside the timed region
    xh = torch.empty(1, D_MODEL, dtype=torch.bfloat16).pin_memory()
    xh.copy_(sw.bufs[1]["x"].cpu())
    yh = torch.empty(1, D_MODEL, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    e0.record(stream)
    for _ in range(args.steps):
        sw.bufs[1]["x"].copy_(xh, non_blocking=True)
        graphs[1].replay()
        yh.copy_(sw.bufs[1]["y"], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1))

    pk = peaks()
    d1_bytes = decode_bytes(bits, 1)
    d16_bytes = decode_bytes(bits, 16)
    value = job_throughput(d1_bytes, args.steps, d1_ms, world) / 1e9
    d16_gbs = job_throughput(d16_bytes, args.steps, d16_ms, world) / 1e9
    pf_tflops = job_throughput(prefill_flops(), args.steps, pf_ms, world) / 1e12
    win_tflops = job_throughput(prefill_flops(), args.steps, win_ms, world) / 1e12
    win_wbytes = (PROMPT // WIN) * sweep_weight_bytes(bits)
    gemm_tflops = gemm_flops / (gemm_ms * 1e-3) / 1e12  # per GPU, all GEMM launches of the pass
    sw_ms, sw_flops = sw.gemm_summary("swiglu")  # the up projections of the pass with the SwiGLU epilogue
    sw_tflops = sw_flops / (sw_ms * 1e-3) / 1e12 if sw_ms > 0 else None
    ffn_tflops = ffn_flops / (ffn_ms * 1e-3) / 1e12      # per GPU, the roofline kernel's launches
    src = source_hash(["pgemm.cu", "common.cuh", "sync.cuh"])
    traffic = NCU_TRAFFIC.get(src)
    del graphs
    # the same sweep at the other code widths (decode and the prompt GEMM)
    widths = {}
    if rank == 0 or world > 1:
        for b2 in (4, 6, 8):
            if b2 != bits:
                widths[str(b2)] = width_line(q, b2, gen, dev, args.steps, pk)
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
                                "as the o / w2 matvec's epilogue (qlinear_mv_resid_norm); per-kernel times are "
                                "back-to-back launches, bytes = algorithmic reads + writes (latency-bound at these "
                                "sizes)"),
        "decode_r16": {"GB/s": d16_gbs / world, "frac_of_hbm": d16_gbs / world / pk["hbm"],
                       "ms_per_pass": d16_ms / args.steps, "bytes_per_pass": d16_bytes,
                       "tok_s_modelled": 16.0 / (d16_ms / args.steps * 1e-3)},
        "prefill": {"TFLOP/s": pf_tflops / world, "ms_per_pass": pf_ms / args.steps,
                    "flops_per_pass": prefill_flops(),
                    "includes": "prompt GEMMs (q/k/v/gate and w1/w3 each as one qlinear_pgemm_multi, o and w2 as "
                                "qlinear_pgemm) and SwiGLU (qswiglu): the faster composition as measured; the up "
                                "projection with the SwiGLU as its epilogue is timed beside it",
                    "swiglu_epilogue_TFLOP/s": sw_tflops,
                    "tok_s_modelled": PROMPT / (pf_ms / args.steps * 1e-3),
                    "variants_ms_per_pass": dict(pf_variants, swiglu_separate_ms=pf_ms / args.steps,
                                                 what="one pass each after the timed region: the up projection with "
                                                      "the SwiGLU as its epilogue (qlinear_pgemm_swiglu); the "
                                                      "post-add / next-norm after o and w2 as qlinear_pgemm + "
                                                      "qresid_rmsnorm, and as qlinear_pgemm_resid_norm (the GEMM's "
                                                      "epilogue + the norm)")},
        "prefill_windows": {"window_rows": WIN, "windows": PROMPT // WIN,
                            "TFLOP/s": win_tflops / world, "ms_per_pass": win_ms / args.steps,
                            "launches_per_pass": launches["win"],
                            "us_per_pgemm_call": win_ms / args.steps * 1e3 / ((PROMPT // WIN) * len(layer_shapes())),
                            "weight_stream_GB/s": win_wbytes / (win_ms / args.steps * 1e-3) / 1e9 / world,
                            "weight_stream_frac_of_hbm": win_wbytes / (win_ms / args.steps * 1e-3) / 1e9 / world
                            / pk["hbm"],
                            "vs_one_m8192_pass": (win_ms / args.steps) / (pf_ms / args.steps),
                            "what": "the 8192-row prompt in 64 windows of 128 rows, each window through all 16 "
                                    "layers (78 pgemm + 16 SwiGLU per window, one CUDA graph) before the next: "
                                    "every window streams every weight again (64 x the sweep's weight bytes)"},
        "tok_s_note": "modelled from the linear layers only: decode R / (decode pass time), prefill "
                      "prompt rows / (prefill pass time); attention, norms and sampling excluded",
        "roofline": {"bound": "tensor", "kernel": "qlinear_pgemm_multi(w1, w3): one row-sum pre-pass, then per "
                                                  "weight the code conversion and the tcgen05 GEMM, timed together; "
                                                  f"M={PROMPT} N={D_FF} K={D_MODEL}",
                     "achieved": ffn_tflops, "peak": pk["bf16_sus"], "unit": "TFLOP/s",
                     "frac": ffn_tflops / pk["bf16_sus"], "frac_of_burst": ffn_tflops / pk["bf16"],
                     "traffic": traffic,
                     "traffic_unit": "bytes per launch (DRAM read + write, one ncu capture of this shape)",
                     "algorithmic_bytes_per_launch": PROMPT * D_MODEL * 2 + weight_bytes(D_FF, D_MODEL, bits)
                     + PROMPT * D_FF * 4,
                     "timing": "CUDA events around each layer's qlinear_pgemm_multi(w1, w3) call in the timed "
                               "prefill passes, as the layer runs it: the w3 code conversion runs in the w1 GEMM's "
                               "last tiles",
                     "all_gemm_launches_TFLOP/s": gemm_tflops,
                     "all_gemm_launches_timing": "one prefill pass after the timed region, CUDA events around "
                                                 "every call (which ends the overlap between calls)",
                     "peak_source": f"{pk['src']} bf16 sustained (the launches run back to back inside a "
                                    "seconds-long step); frac_of_burst against the burst figure"},
        "roofline_decode": {"bound": "hbm", "kernel": "decode pass R=1 (qattn_proj_mv, qlinear_mv_rows, "
                                                      "qffn_swiglu_mv)",
                            "achieved": value / world, "peak": pk["hbm"], "unit": "GB/s",
                            "frac": value / world / pk["hbm"], "traffic": None,
                            "traffic_note": "per-launch DRAM bytes of the FFN decode kernel equal its algorithmic "
                                            "bytes (ncu); no capture of the whole pass",
                            "peak_source": f"{pk['src']} copy bandwidth"},
        "widths": widths,
        "e2e": {"value": job_throughput(d1_bytes, args.steps, e2e_ms, world) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": D_MODEL * 2, "d2h_bytes_per_step": D_MODEL * 4,
                "what": "decode pass R=1 with x copied from pinned host memory and the last output copied back"},
        "gpu_launches": n_launch,
        "launches_before_timed_region": pre,
        "clocks": clocks,
        "status": status,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baselines(bits)
        line["cpu_baseline"] = base["sweep_decode_r1"]
        line["cpu_baselines"] = base
        line["roofline"]["cpu_baseline"] = base["c3_pgemm"]
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
