"""Benchmark: one dense-8B-shaped MLP training step through the FP8 path.

Workload (per GPU, per step), all BF16 inputs resident in HBM:
  X [8192 x 4096], H [8192 x 12288], W_gate, W_up [12288 x 4096],
  W_down [4096 x 12288], dY_gate, dY_up [8192 x 12288], dY_down [8192 x 4096]
  1. weight quantizers (128x128 blocks + transposed copies) on W_gate, W_up, W_down
  2. activation quantizers (1x128 row + 128x1 column copies) on X and H
  3. FProp  gate/up: X W^T, down: H W_down^T                     (BF16 out)
  4. gradient quantizers on dY_gate, dY_up, dY_down
  5. DGrad  dY W                                                 (BF16 out)
  6. WGrad  dY^T X (gate, up), dY_down^T H (down)                (FP32 out)
  = 17 kernel launches and 9 GEMMs of 2*8192*12288*4096 = 824.6 GFLOP each.

value  = GEMM FLOPs of the step / wall time of the whole step (quantizers
         included), TFLOP/s, inputs resident; every step touches ~1.07 GB of
         inputs, several times the 129 MB L2.
e2e    = the same through host buffers: each step copies its BF16 inputs from
         pinned host memory and reads the three FP32 weight gradients back
         (copy streams overlap one step's copies with the neighbouring steps'
         compute; every copy is inside the timed region).
roofline = the dominant kernel (the FProp/DGrad GEMM kernel) against the FP8
         dense peak: the measured burst BF16 cuBLAS peak x 2 (the nominal
         FP8/BF16 ratio), because the timed region lasts well under a second
         at full clock; the sustained figure (measured at a lower clock under
         the power cap) is reported beside it.

--impl reference times the CPU oracle (oracle/) on a bounded sample of the same
workload on the host cores.  Multi-GPU (torchrun): independent replicas, one
per rank, no collective on the data path (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-scaled FP8 GEMM TFLOP/s (% dense FP8 peak); quantizer GB/s (% HBM)"
N_TOK, C, D = 8192, 4096, 12288
GEMM_FLOP = 2.0 * N_TOK * C * D
GEMMS_PER_STEP = 9
ACT_BYTES_PER_ELT = 2 + 2 * (1 + 4 / 128)      # BF16 in, two FP8 copies + FP32 scales
W_BYTES_PER_ELT = 2 + 2 + 2 * 4 / (128 * 128)  # BF16 in, codes + transposed codes, scales
CONFIG = {
    "workload": "dense-8B MLP layer training step, 128-block FP8 recipe: N=8192 tokens, hidden 4096, "
                "intermediate 12288; quantize X, H, W_gate/up/down, dY; FProp/DGrad/WGrad x3",
    "tokens": N_TOK, "hidden": C, "intermediate": D,
    "l2": "inputs larger than L2: ~1.07 GB of BF16 inputs read every step (L2 129 MB)",
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm": float(p["hbm_gbs"]), "bf16": float(p["bf16_tflops"]),
                "bf16_sust": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "src": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sust": 1700.0, "src": "fallback"}


def _profile_traffic(kernel_key: str, source: str):
    """Per-launch DRAM bytes recorded by the committed ncu summary, if the kernel
    source has not changed since it was captured (else None)."""
    prof = os.path.join(ROOT, "profiles", f"{kernel_key}.md")
    if not os.path.exists(prof):
        return None
    txt = open(prof).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s*\(source sha256 ([0-9a-f]+)\)", txt)
    if not m:
        return None
    sha = hashlib.sha256(open(source, "rb").read()).hexdigest()
    return float(m.group(1)) if sha.startswith(m.group(2)) else None


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        pass

    def result(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- ours

def _rank_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _max_over_ranks(values, dev, world):
    """Each value's maximum over the ranks of the process group (the slowest replica
    sets the job's time); the values themselves when running alone."""
    import torch

    t = torch.tensor(values, dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t]


def _inputs_host(seed: int):
    """The step's BF16 inputs as numpy uint16 arrays (synthetic, seeded)."""
    import synth

    return {
        "x": synth.activation(N_TOK, C, seed=seed, stream="x"),
        "h": synth.activation(N_TOK, D, seed=seed, stream="h"),
        "w_gate": synth.weight(D, C, seed=seed, stream="w_gate"),
        "w_up": synth.weight(D, C, seed=seed, stream="w_up"),
        "w_down": synth.weight(C, D, seed=seed, stream="w_down"),
        "dy_gate": synth.gradient(N_TOK, D, seed=seed, stream="dy_gate"),
        "dy_up": synth.gradient(N_TOK, D, seed=seed, stream="dy_up"),
        "dy_down": synth.gradient(N_TOK, C, seed=seed, stream="dy_down"),
    }


class Step:
    """Preallocated buffers and the 17-launch step."""

    def __init__(self, dev, inputs):
        import torch

        import rollout_x128_act_gb300 as jq

        self.jq = jq
        self.t = {k: torch.empty(v.shape, dtype=torch.bfloat16, device=dev) for k, v in inputs.items()}
        e = lambda *s, dt=torch.uint8: torch.empty(s, dtype=dt, device=dev)  # noqa: E731
        f32 = torch.float32
        self.act = {}
        for name, (n, c) in (("x", (N_TOK, C)), ("h", (N_TOK, D)), ("dy_gate", (N_TOK, D)), ("dy_up", (N_TOK, D)),
                             ("dy_down", (N_TOK, C))):
            cap = jq.jetq_colcopy_capacity(n, 1)
            self.act[name] = dict(q_row=e(n, c), s_row=e(c // 128, n, dt=f32), q_col=e(c, cap),
                                  s_col=e(cap // 128, c, dt=f32), cap=cap)
        self.w = {}
        for name, (d, c) in (("w_gate", (D, C)), ("w_up", (D, C)), ("w_down", (C, D))):
            self.w[name] = (e(d, c), e(d // 128, c // 128, dt=f32), e(c, d), e(c // 128, d // 128, dt=f32))
        bf = torch.bfloat16
        self.y = {"gate": e(N_TOK, D, dt=bf), "up": e(N_TOK, D, dt=bf), "down": e(N_TOK, C, dt=bf)}
        self.dx = {"gate": e(N_TOK, C, dt=bf), "up": e(N_TOK, C, dt=bf), "down": e(N_TOK, D, dt=bf)}
        self.dw = {"gate": e(D, C, dt=f32), "up": e(D, C, dt=f32), "down": e(C, D, dt=f32)}
        self.gemm_events = []

    def load(self, inputs, non_blocking=False):
        import numpy as np
        import torch

        for k, v in inputs.items():
            src = v if isinstance(v, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(v).view(np.int16))
            self.t[k].view(torch.int16).copy_(src.view(torch.int16) if isinstance(v, torch.Tensor) else src,
                                              non_blocking=non_blocking)

    def run(self, stream=None, time_gemms=False, inputs=None, dw=None):
        """The step on `inputs` (device BF16 tensors, default self.t), weight gradients into
        `dw` (default self.dw)."""
        import torch

        jq = self.jq
        t_in = self.t if inputs is None else inputs
        dw_out = self.dw if dw is None else dw
        launches = 0
        for name in ("w_gate", "w_up", "w_down"):
            q, s, qT, sT = self.w[name]
            jq.jetq_quant_w_128x128(t_in[name], q, s, qT, sT, stream)
            launches += 1

        def qa(name):
            a = self.act[name]
            jq.jetq_quant_act_1x128(t_in[name], a["q_row"], a["s_row"], a["q_col"], a["s_col"], a["cap"],
                                    None, 0, stream)

        def timed(fn):
            if time_gemms:
                s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                st = stream or torch.cuda.current_stream()
                s0.record(st)
                fn()
                s1.record(st)
                self.gemm_events.append((s0, s1))
            else:
                fn()

        qa("x")
        qa("h")
        launches += 2
        X, H = self.act["x"], self.act["h"]
        for g, (a, w) in (("gate", (X, "w_gate")), ("up", (X, "w_up")), ("down", (H, "w_down"))):
            q, s, _, _ = self.w[w]
            n, c = a["q_row"].shape
            timed(lambda a=a, q=q, s=s, g=g, n=n, c=c: jq.jetq_gemm_fprop(
                jq.RECIPE_BLOCK128, a["q_row"], a["s_row"], q, s, n, q.shape[0], c, self.y[g], jq.PATH_TRAIN, stream))
            launches += 1
        for name in ("dy_gate", "dy_up", "dy_down"):
            qa(name)
            launches += 1
        for g, w in (("gate", "w_gate"), ("up", "w_up"), ("down", "w_down")):
            a = self.act["dy_" + g]
            _, _, qT, sT = self.w[w]
            n, d = a["q_row"].shape
            timed(lambda a=a, qT=qT, sT=sT, g=g, n=n, d=d: jq.jetq_gemm_dgrad(
                jq.RECIPE_BLOCK128, a["q_row"], a["s_row"], qT, sT, n, d, qT.shape[0], self.dx[g], stream))
            launches += 1
        for g, xa in (("gate", X), ("up", X), ("down", H)):
            a = self.act["dy_" + g]
            d, c = a["q_col"].shape[0], xa["q_col"].shape[0]
            timed(lambda a=a, xa=xa, g=g, d=d, c=c: jq.jetq_gemm_wgrad(
                jq.RECIPE_BLOCK128, a["q_col"], a["s_col"], xa["q_col"], xa["s_col"], N_TOK, a["cap"], d, c,
                dw_out[g], False, stream))
            launches += 1
        return launches


# --------------------------------------------------------------------------- other configurations

def _dev_inputs(dev, seed):
    """Seeded device-side generator for the secondary measurements (speed only;
    same distributions as synth/: N(0,1) + 0.1% x50 activations, N(0,0.02)
    weights, N(0,1e-3) gradients, BF16 by round-to-nearest)."""
    import torch

    g = torch.Generator(device=dev)
    g.manual_seed(seed)

    def act(r, c):
        x = torch.randn(r, c, generator=g, device=dev)
        k = int(round(0.001 * r * c))
        idx = torch.randint(0, r * c, (k,), generator=g, device=dev)
        x.view(-1)[idx] *= 50.0
        return x.to(torch.bfloat16)

    def weight(r, c):
        return (torch.randn(r, c, generator=g, device=dev) * 0.02).to(torch.bfloat16)

    def grad(r, c):
        return (torch.randn(r, c, generator=g, device=dev) * 1e-3).to(torch.bfloat16)

    return act, weight, grad


def _time(fn, iters, warm=3):
    import torch

    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters  # ms


def measure_decode(dev, peaks):
    """Rollout decode FProp (DECODE path) against the dense-8B weights: N tokens
    x 4096 vs W_up 12288x4096 and N x 12288 vs W_down 4096x12288.  Eight weight
    copies (402 MB) rotate so each call streams its weight from HBM."""
    import torch

    import rollout_x128_act_gb300 as jq

    act, weight, _ = _dev_inputs(dev, 7)
    out = {}
    for name, (d, c) in (("up", (D, C)), ("down", (C, D))):
        ws = [jq.quant_weight(weight(d, c), transposed=False) for _ in range(8)]
        x = act(256, c)
        for n in (1, 8, 64, 256):
            a = jq.quant_act(x[:n], col=False)
            y = torch.empty((n, d), dtype=torch.bfloat16, device=dev)
            # the split-K decode's partial sums (allocated once, as a rollout engine would)
            work = torch.empty(max(jq.jetq_decode_workspace_bytes(n, d, c), 16), dtype=torch.uint8, device=dev)
            i = [0]

            def call():
                q, s, _, _ = ws[i[0] % 8]
                i[0] += 1
                jq.jetq_gemm_fprop_ws(jq.RECIPE_BLOCK128, a["q_row"], a["s_row"], q, s, n, d, c, y, work,
                                      jq.PATH_DECODE)

            ms = _time(call, 40)
            # CUDA-graph replay of 8 calls (one per weight copy), as a decode step replays
            st = torch.cuda.Stream()
            st.wait_stream(torch.cuda.current_stream())
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(st):
                for _ in range(2):
                    call()
                torch.cuda.synchronize()
                with torch.cuda.graph(graph, stream=st):
                    for _ in range(8):
                        call()
            ms_graph = _time(graph.replay, 10) / 8
            byts = d * c + (d // 128) * (c // 128) * 4 + n * c * (1 + 4 / 128) + n * d * 2
            flops = 2.0 * n * d * c
            t_roof = max(byts / (peaks["hbm"] * 1e9), flops / (2.0 * peaks["bf16"] * 1e12))
            out[f"{name}_n{n}"] = {
                "us": round(ms * 1e3, 2), "us_graph": round(ms_graph * 1e3, 2),
                "gbs": round(byts / (ms * 1e-3) / 1e9, 1),
                "frac_of_roofline": round(t_roof / (ms * 1e-3), 3),
                "frac_of_roofline_graph": round(t_roof / (ms_graph * 1e-3), 3),
            }
        del ws
    return out


def measure_mxfp8(dev):
    """MXFP8 recipe on the dense-8B gate shapes: quantizer GB/s and the three GEMMs."""
    import torch

    import rollout_x128_act_gb300 as jq

    act, weight, grad = _dev_inputs(dev, 8)
    x, w, dy = act(N_TOK, C), weight(D, C), grad(N_TOK, D)
    ms_q = _time(lambda: jq.quant_mx(dy), 10)
    gx, gw, gdy = jq.quant_mx(x), jq.quant_mx(w), jq.quant_mx(dy)
    y = torch.empty((N_TOK, D), dtype=torch.bfloat16, device=dev)
    dx = torch.empty((N_TOK, C), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((D, C), dtype=torch.float32, device=dev)
    R = jq.RECIPE_MXFP8
    t = {
        "fprop": _time(lambda: jq.jetq_gemm_fprop(R, gx["q_row"], gx["e8_row"], gw["q_row"], gw["e8_row"], N_TOK, D,
                                                  C, y, jq.PATH_TRAIN), 10),
        "dgrad": _time(lambda: jq.jetq_gemm_dgrad(R, gdy["q_row"], gdy["e8_row"], gw["q_col"], gw["e8_col"], N_TOK, D,
                                                  C, dx), 10),
        "wgrad": _time(lambda: jq.jetq_gemm_wgrad(R, gdy["q_col"], gdy["e8_col"], gx["q_col"], gx["e8_col"], N_TOK,
                                                  gx["ldq_col"], D, C, dw), 10),
    }
    res = {k: {"ms": round(v, 4), "tflops": round(GEMM_FLOP / (v * 1e-3) / 1e12, 1)} for k, v in t.items()}
    res["quant_mx_dy_gbs"] = round(N_TOK * D * ACT_BYTES_PER_ELT / (ms_q * 1e-3) / 1e9, 1)
    return res


def measure_pow2(dev):
    """The dense-8B training step in the 128-block recipe with power-of-two scales
    (E8M0 atoms, block-scaled MMA): 3 weight + 5 activation/gradient quantizations
    and the 9 GEMMs, timed as one step, plus the gate-shape GEMMs alone."""
    import torch

    import rollout_x128_act_gb300 as jq

    act, weight, grad = _dev_inputs(dev, 10)
    x, h = act(N_TOK, C), act(N_TOK, D)
    ws = {"gate": weight(D, C), "up": weight(D, C), "down": weight(C, D)}
    dys = {"gate": grad(N_TOK, D), "up": grad(N_TOK, D), "down": grad(N_TOK, C)}
    R = jq.RECIPE_BLOCK128_POW2
    bf = torch.bfloat16
    y = {"gate": torch.empty((N_TOK, D), dtype=bf, device=dev), "up": torch.empty((N_TOK, D), dtype=bf, device=dev),
         "down": torch.empty((N_TOK, C), dtype=bf, device=dev)}
    dx = {"gate": torch.empty((N_TOK, C), dtype=bf, device=dev), "up": torch.empty((N_TOK, C), dtype=bf, device=dev),
          "down": torch.empty((N_TOK, D), dtype=bf, device=dev)}
    dw = {g: torch.empty(tuple(ws[g].shape), dtype=torch.float32, device=dev) for g in ws}

    def step():
        qw = {g: jq.quant_weight_pow2(ws[g]) for g in ws}
        ax, ah = jq.quant_act_pow2(x), jq.quant_act_pow2(h)
        a_in = {"gate": ax, "up": ax, "down": ah}
        for g in ("gate", "up", "down"):
            a, (q, e, _, _) = a_in[g], qw[g]
            jq.jetq_gemm_fprop(R, a["q_row"], a["e8_row"], q, e, N_TOK, q.shape[0], q.shape[1], y[g], jq.PATH_TRAIN)
        ady = {g: jq.quant_act_pow2(dys[g]) for g in dys}
        for g in ("gate", "up", "down"):
            a, (_, _, qT, eT) = ady[g], qw[g]
            jq.jetq_gemm_dgrad(R, a["q_row"], a["e8_row"], qT, eT, N_TOK, qT.shape[1], qT.shape[0], dx[g])
        for g in ("gate", "up", "down"):
            a, xa = ady[g], a_in[g]
            jq.jetq_gemm_wgrad(R, a["q_col"], a["e8_col"], xa["q_col"], xa["e8_col"], N_TOK, a["ldq_col"],
                               a["q_col"].shape[0], xa["q_col"].shape[0], dw[g])

    ms_step = _time(step, 10)
    gx, gdy = jq.quant_act_pow2(x), jq.quant_act_pow2(dys["gate"])
    q, e, qT, eT = jq.quant_weight_pow2(ws["gate"])
    t = {
        "fprop": _time(lambda: jq.jetq_gemm_fprop(R, gx["q_row"], gx["e8_row"], q, e, N_TOK, D, C, y["gate"],
                                                  jq.PATH_TRAIN), 10),
        "dgrad": _time(lambda: jq.jetq_gemm_dgrad(R, gdy["q_row"], gdy["e8_row"], qT, eT, N_TOK, D, C, dx["gate"]),
                       10),
        "wgrad": _time(lambda: jq.jetq_gemm_wgrad(R, gdy["q_col"], gdy["e8_col"], gx["q_col"], gx["e8_col"], N_TOK,
                                                  gx["ldq_col"], D, C, dw["gate"]), 10),
    }
    res = {"step_ms": round(ms_step, 4), "step_tflops": round(9 * GEMM_FLOP / (ms_step * 1e-3) / 1e12, 1)}
    res.update({k: {"ms": round(v, 4), "tflops": round(GEMM_FLOP / (v * 1e-3) / 1e12, 1)} for k, v in t.items()})
    return res


def measure_f3_kernels(dev):
    """Re-quantized column copy and BF16 dequantizer on the 8192 x 12288 activation
    (HBM-bound; algorithmic bytes: 1 + 4/128 read and 1 + 4/128 written per element for
    the re-quantizer, 1 + 4/128 read and 2 written for the dequantizer)."""
    import torch

    import rollout_x128_act_gb300 as jq

    act, _, _ = _dev_inputs(dev, 11)
    h = act(N_TOK, D)
    a = jq.quant_act(h, col=False)
    g = jq.requant_col(a["q_row"], a["s_row"])
    out = torch.empty((N_TOK, D), dtype=torch.bfloat16, device=dev)
    ms_r = _time(lambda: jq.jetq_requant_col_from_row(a["q_row"], a["s_row"], g["q_col"], g["s_col"],
                                                      g["ldq_col"]), 20)
    ms_d = _time(lambda: jq.jetq_dequant_bf16(a["q_row"], a["s_row"], jq.SCALES_ROWGROUPS_1X128, out), 20)
    n = N_TOK * D
    return {"requant_col_gbs": round(n * 2 * (1 + 4 / 128) / (ms_r * 1e-3) / 1e9, 1), "requant_col_us": round(ms_r * 1e3, 1),
            "dequant_bf16_gbs": round(n * (3 + 4 / 128) / (ms_d * 1e-3) / 1e9, 1), "dequant_bf16_us": round(ms_d * 1e3, 1)}


def measure_fused_producers(dev):
    """The 1x128 quantizer fused with its producer, dense-8B MLP shapes, row + column
    copies.  RMSNorm over X 8192 x 4096 (four input buffers in rotation, 256 MB, so no
    launch finds its input in L2 from the launch before; the statistics pass and the
    quantizer each read X, the second read mostly from L2); SwiGLU over gate and up
    8192 x 12288 (400 MB).  Algorithmic bytes per element: the producer's inputs once
    (2 for RMSNorm, 4 for SwiGLU) + 2 * (1 + 4/128) written.  The plain quantizer on the
    same X is timed beside them."""
    import torch

    import rollout_x128_act_gb300 as jq

    act, _, _ = _dev_inputs(dev, 12)
    xs = [act(N_TOK, C) for _ in range(4)]
    w = (1.0 + 0.1 * act(1, C).float().clamp(-3, 3)).to(torch.bfloat16).view(-1)
    o = jq.quant_act_rmsnorm(xs[0], w)
    it = [0]

    def rms():
        it[0] += 1
        jq.jetq_quant_act_1x128_rmsnorm(xs[it[0] % 4], w, 1e-6, o["rstd"], o["q_row"], o["s_row"], o["q_col"],
                                        o["s_col"], o["ldq_col"])

    def plain():
        it[0] += 1
        jq.jetq_quant_act_1x128(xs[it[0] % 4], o["q_row"], o["s_row"], o["q_col"], o["s_col"], o["ldq_col"])

    ms_rms, ms_plain = _time(rms, 40), _time(plain, 40)
    del xs
    gate, up = act(N_TOK, D), act(N_TOK, D)
    s = jq.quant_act_swiglu(gate, up)
    ms_sw = _time(lambda: jq.jetq_quant_act_1x128_swiglu(gate, up, s["q_row"], s["s_row"], s["q_col"], s["s_col"],
                                                         s["ldq_col"]), 20)
    out_b = 2 * (1 + 4 / 128)
    nx, nh = N_TOK * C, N_TOK * D
    return {"rmsnorm_quant_gbs": round(nx * (2 + out_b) / (ms_rms * 1e-3) / 1e9, 1),
            "rmsnorm_quant_us": round(ms_rms * 1e3, 1),
            "plain_quant_same_x_us": round(ms_plain * 1e3, 1),
            "swiglu_quant_gbs": round(nh * (4 + out_b) / (ms_sw * 1e-3) / 1e9, 1),
            "swiglu_quant_us": round(ms_sw * 1e3, 1)}


def measure_nvfp4(dev):
    """NVFP4 quantizer (per-token scope: two reads of each row) and BF16 dequantizer on
    the 30B-A3B routed activations, 131072 rows x hidden 2048 (512 MB of BF16).
    Algorithmic bytes per element: quantizer 2 + 1/2 + 1/16 (+ 4 per row), dequantizer
    1/2 + 1/16 + 2."""
    import torch

    import rollout_x128_act_gb300 as jq

    act, _, _ = _dev_inputs(dev, 13)
    R, Cn = 131072, 2048
    x = act(R, Cn)
    o = jq.quant_nvfp4(x)
    out = torch.empty((R, Cn), dtype=torch.bfloat16, device=dev)
    ms_q = _time(lambda: jq.jetq_quant_nvfp4(x, o["q"], o["sb"], o["sg"]), 20)
    ms_d = _time(lambda: jq.jetq_dequant_nvfp4_bf16(o["q"], o["sb"], o["sg"], True, out), 20)
    n = R * Cn
    res = {"quant_gbs": round((n * (2 + 0.5 + 1 / 16) + 4 * R) / (ms_q * 1e-3) / 1e9, 1),
           "quant_us": round(ms_q * 1e3, 1),
           "dequant_gbs": round(n * (0.5 + 1 / 16 + 2) / (ms_d * 1e-3) / 1e9, 1), "dequant_us": round(ms_d * 1e3, 1)}
    del out
    # NVFP4 FProp (block-scaled FP4 MMA, per-token x tensor scope scales in the epilogue):
    # the dense-8B gate projection, 8192 tokens x 4096 -> 12288, BF16 out
    xa = act(N_TOK, C)
    wq = act(D, C)
    ga = jq.quant_nvfp4(xa)
    ga["atoms"] = jq.nvfp4_atoms(ga["sb"], C)
    gw = jq.quant_nvfp4(wq, scope_amax=jq.amax_bf16(wq))
    gw["atoms"] = jq.nvfp4_atoms(gw["sb"], C)
    y = torch.empty((N_TOK, D), dtype=torch.bfloat16, device=dev)
    ms_g = _time(lambda: jq.jetq_gemm_nvfp4(ga["q"], ga["atoms"], ga["sg"], True, gw["q"], gw["atoms"], gw["sg"],
                                            N_TOK, D, C, y), 20)
    if jq.jetq_check_device_error() != 0:
        raise RuntimeError("device error word set by the NVFP4 GEMM")
    res["gemm"] = {"shape": f"{N_TOK}x{D}x{C}", "ms": round(ms_g, 4),
                   "tflops": round(GEMM_FLOP / (ms_g * 1e-3) / 1e12, 1),
                   "note": "FP4 dense nominal 13.5 PFLOP/s (3 x FP8); scope scales applied in the epilogue"}
    return res


def measure_rollout_step(dev, peaks):
    """On-policy FP8 weight sync plus one rollout decode step of 128 concurrent
    sequences through the dense-8B MLP (quantize, gate/up FProp, quantize, down
    FProp), replayed from a CUDA graph: step latency, weight-stream GB/s, and the
    payload copy's time and byte identity."""
    import torch

    import rollout_x128_act_gb300 as jq

    act, weight, _ = _dev_inputs(dev, 12)
    n = 128
    trainer = {"gate": jq.quant_weight(weight(D, C), transposed=False)[:2],
               "up": jq.quant_weight(weight(D, C), transposed=False)[:2],
               "down": jq.quant_weight(weight(C, D), transposed=False)[:2]}
    rollout = {k: (torch.empty_like(q), torch.empty_like(s)) for k, (q, s) in trainer.items()}

    def sync():
        for k in trainer:
            rollout[k][0].copy_(trainer[k][0], non_blocking=True)
            rollout[k][1].copy_(trainer[k][1], non_blocking=True)

    ms_sync = _time(sync, 10)
    payload = sum(q.numel() + s.numel() * 4 for q, s in trainer.values())
    identical = all(torch.equal(rollout[k][0], trainer[k][0]) and torch.equal(rollout[k][1], trainer[k][1])
                    for k in trainer)
    x, h = act(n, C), act(n, D)
    ax, ah = jq.quant_act(x, col=False), jq.quant_act(h, col=False)
    y = {"gate": torch.empty((n, D), dtype=torch.bfloat16, device=dev),
         "up": torch.empty((n, D), dtype=torch.bfloat16, device=dev),
         "down": torch.empty((n, C), dtype=torch.bfloat16, device=dev)}

    def step():
        jq.jetq_quant_act_1x128(x, ax["q_row"], ax["s_row"], None, None, 0)
        for k in ("gate", "up"):
            q, s = rollout[k]
            jq.jetq_gemm_fprop(jq.RECIPE_BLOCK128, ax["q_row"], ax["s_row"], q, s, n, D, C, y[k], jq.PATH_DECODE)
        jq.jetq_quant_act_1x128(h, ah["q_row"], ah["s_row"], None, None, 0)
        q, s = rollout["down"]
        jq.jetq_gemm_fprop(jq.RECIPE_BLOCK128, ah["q_row"], ah["s_row"], q, s, n, C, D, y["down"], jq.PATH_DECODE)

    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            step()
    ms_step = _time(graph.replay, 20)
    return {"concurrent": n, "step_us_graph": round(ms_step * 1e3, 2),
            "weight_gbs": round(payload / (ms_step * 1e-3) / 1e9, 1),
            "frac_of_hbm": round(payload / (ms_step * 1e-3) / 1e9 / peaks["hbm"], 3),
            "sync_payload_bytes": int(payload), "sync_us": round(ms_sync * 1e3, 1),
            "sync_gbs": round(2 * payload / (ms_sync * 1e-3) / 1e9, 1), "sync_byte_identical": bool(identical)}


def measure_moe(dev):
    """MoE grouped GEMMs, 30B-A3B shapes: 128 experts, 16384 tokens top-8 with
    Zipf(1.2) load (131072 routed rows), hidden 2048, expert intermediate 768
    (gate/up fused 1536); FProp/DGrad/WGrad of the gate/up projection, both recipes."""
    import torch

    import rollout_x128_act_gb300 as jq
    import synth

    E, Cm, Dm = 128, 2048, 1536
    off, _ = synth.zipf_topk_routing(16384, E, 8, 1.2, seed=0)
    R = int(off[-1])
    seg = torch.tensor(off, dtype=torch.int64, device=dev)
    act, weight, grad = _dev_inputs(dev, 9)
    x, dy = act(R, Cm), grad(R, Dm)
    wst = weight(E * Dm, Cm)
    flops = 2.0 * R * Dm * Cm
    res = {"routed_rows": R, "expert_rows_min": int((off[1:] - off[:-1]).min()),
           "expert_rows_max": int((off[1:] - off[:-1]).max())}
    # 128-block recipe
    ax, ady = jq.quant_act(x, seg_offsets=seg), jq.quant_act(dy, seg_offsets=seg)
    qs = [jq.quant_weight(wst[e * Dm:(e + 1) * Dm]) for e in range(E)]
    qw, sw = torch.stack([q[0] for q in qs]), torch.stack([q[1] for q in qs])
    qwt, swt = torch.stack([q[2] for q in qs]), torch.stack([q[3] for q in qs])
    del qs
    P = ax["ldq_col"]
    y = torch.empty((R, Dm), dtype=torch.bfloat16, device=dev)
    dx = torch.empty((R, Cm), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((E, Dm, Cm), dtype=torch.float32, device=dev)
    B = jq.RECIPE_BLOCK128
    t = {
        "b128_fprop": _time(lambda: jq.grouped(jq.GEMM_FPROP, ax["q_row"], ax["s_row"], qw, sw, seg, n=Dm, k=Cm,
                                               out=y), 10),
        "b128_dgrad": _time(lambda: jq.grouped(jq.GEMM_DGRAD, ady["q_row"], ady["s_row"], qwt, swt, seg, n=Cm, k=Dm,
                                               out=dx), 10),
        "b128_wgrad": _time(lambda: jq.grouped(jq.GEMM_WGRAD, ady["q_col"], ady["s_col"], ax["q_col"], ax["s_col"],
                                               seg, n=Cm, k=P, out=dw), 5),
    }
    del ax, ady, qw, sw, qwt, swt
    # MXFP8 recipe
    gx, gdy = jq.quant_mx(x, seg_offsets=seg), jq.quant_mx(dy, seg_offsets=seg)
    gws = [jq.quant_mx(wst[e * Dm:(e + 1) * Dm]) for e in range(E)]
    qw, ew = torch.stack([g["q_row"] for g in gws]), torch.cat([g["e8_row"] for g in gws])
    qwc, ewc = torch.stack([g["q_col"] for g in gws]), torch.cat([g["e8_col"] for g in gws])
    del gws
    M = jq.RECIPE_MXFP8
    t.update({
        "mx_fprop": _time(lambda: jq.grouped(jq.GEMM_FPROP, gx["q_row"], gx["e8_row"], qw, ew, seg, n=Dm, k=Cm,
                                             out=y, recipe=M), 10),
        "mx_dgrad": _time(lambda: jq.grouped(jq.GEMM_DGRAD, gdy["q_row"], gdy["e8_row"], qwc, ewc, seg, n=Cm, k=Dm,
                                             out=dx, recipe=M), 10),
        "mx_wgrad": _time(lambda: jq.grouped(jq.GEMM_WGRAD, gdy["q_col"], gdy["e8_col"], gx["q_col"], gx["e8_col"],
                                             seg, n=Cm, k=P, out=dw, recipe=M), 5),
    })
    for k, v in t.items():
        res[k] = {"ms": round(v, 4), "tflops": round(flops / (v * 1e-3) / 1e12, 1)}
    del B
    return res


def quant_bytes_per_step():
    act_elts = N_TOK * C * 2 + N_TOK * D * 3  # X, dY_down ; H, dY_gate, dY_up
    w_elts = 3 * D * C
    return act_elts * ACT_BYTES_PER_ELT + w_elts * W_BYTES_PER_ELT


def step_error() -> bool:
    import rollout_x128_act_gb300 as jq

    return jq.jetq_check_device_error() != 0


def run_ours(args):
    import numpy as np
    import torch

    rank, world, local = _rank_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__

    __graft_entry__.build()
    inputs = _inputs_host(seed=rank)
    step = Step(dev, inputs)
    step.load(inputs)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # ---- warm-up
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    if step.jq.jetq_check_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    # ---- timed: inputs resident, per-GEMM events for the roofline
    barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        ev0.record(stream)
        launches = 0
        for _ in range(args.steps):
            launches += step.run(time_gemms=True)
        ev1.record(stream)
        torch.cuda.synchronize()
    clocks = clk.result()
    barrier()
    ms_total = ev0.elapsed_time(ev1)
    if step.jq.jetq_check_device_error() != 0:
        raise RuntimeError("device error word set during the timed steps")
    gemm_ms = [a.elapsed_time(b) for a, b in step.gemm_events]
    step.gemm_events.clear()

    # ---- e2e: pinned host inputs in, weight gradients out, every step.  Two device
    # buffer sets: step i+1's inputs are copied in (and step i-1's gradients out) on
    # copy streams while step i computes; events order every buffer's reuse, and the
    # timed region spans every step's copies.
    pinned = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).pin_memory() for k, v in inputs.items()}
    h2d = sum(v.numel() * 2 for v in pinned.values())
    d2h = sum(t.numel() * 4 for t in step.dw.values())
    t_sets = [step.t, {k: torch.empty_like(v) for k, v in step.t.items()}]
    dw_sets = [step.dw, {g: torch.empty_like(t) for g, t in step.dw.items()}]
    dw_host = [{g: torch.empty(t.shape, dtype=t.dtype).pin_memory() for g, t in step.dw.items()} for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_steps(n):
        comp_done, d2h_done = [None, None], [None, None]
        start = torch.cuda.Event()
        start.record(stream)
        h2d_s.wait_event(start)
        for i in range(n):
            b = i % 2
            if comp_done[b] is not None:
                h2d_s.wait_event(comp_done[b])  # the step that last read set b has finished
            with torch.cuda.stream(h2d_s):
                for k, v in pinned.items():
                    t_sets[b][k].view(torch.int16).copy_(v, non_blocking=True)
            loaded = torch.cuda.Event()
            loaded.record(h2d_s)
            stream.wait_event(loaded)
            if d2h_done[b] is not None:
                stream.wait_event(d2h_done[b])  # set b's previous gradients have left
            step.run(inputs=t_sets[b], dw=dw_sets[b])
            done = torch.cuda.Event()
            done.record(stream)
            comp_done[b] = done
            d2h_s.wait_event(done)
            with torch.cuda.stream(d2h_s):
                for g, t in dw_sets[b].items():
                    dw_host[b][g].copy_(t, non_blocking=True)
            out = torch.cuda.Event()
            out.record(d2h_s)
            d2h_done[b] = out
        for ev in d2h_done:
            if ev is not None:
                stream.wait_event(ev)

    e2e_steps(max(2, args.warmup // 2))
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = e0.elapsed_time(e1)
    if step.jq.jetq_check_device_error() != 0:
        raise RuntimeError("device error word set during the e2e steps")

    # ---- reduce over ranks (max time)
    ms_total, ms_e2e = _max_over_ranks([ms_total, ms_e2e], dev, world)
    flops = GEMM_FLOP * GEMMS_PER_STEP * args.steps * world
    value = flops / (ms_total * 1e-3) / 1e12
    e2e = flops / (ms_e2e * 1e-3) / 1e12

    peaks = _peaks()
    # the timed region is a fraction of a second at full clock: the burst peak applies
    fp8_peak = 2.0 * peaks["bf16"]
    fp8_peak_sust = 2.0 * peaks["bf16_sust"]
    # per GEMM kind: [fprop x3, dgrad x3, wgrad x3] per step
    per = {"fprop": [], "dgrad": [], "wgrad": []}
    kinds = ["fprop"] * 3 + ["dgrad"] * 3 + ["wgrad"] * 3
    for i, ms in enumerate(gemm_ms):
        per[kinds[i % 9]].append(ms)
    blk = per["fprop"] + per["dgrad"]
    avg_blk = statistics.mean(blk)
    avg_wg = statistics.mean(per["wgrad"])
    gemm_only_ms = sum(gemm_ms) / args.steps
    achieved = GEMM_FLOP / (avg_blk * 1e-3) / 1e12
    gemm_src = os.path.join(ROOT, "rollout_x128_act_gb300", "csrc", "gemm.cu")
    traffic = _profile_traffic("gemm_block128_dense8b", gemm_src)
    step_ms = ms_total / args.steps
    quant_ms = max(step_ms - gemm_only_ms, 1e-9)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic (seeded SplitMix64 normals; 0.1% x50 outliers in activations)",
        "config": CONFIG,
        "roofline": {
            "kernel": "k_gemm_b128<256,8,4,2,block-scaled B> (FProp/DGrad, training shape)",
            "bound": "tensor",
            "achieved": round(achieved, 1),
            "peak": round(fp8_peak, 1),
            "unit": "TFLOP/s",
            "frac": round(achieved / fp8_peak, 4),
            "traffic": traffic,
            "peak_note": f"FP8 dense = 2 x {peaks['src']} burst BF16 cuBLAS ({peaks['bf16']} TFLOP/s), the nominal "
                         f"FP8/BF16 ratio; the timed region lasts {ms_total:.0f} ms at the sampled clock "
                         f"(frac of measured)",
            "frac_of_sustained": round(achieved / fp8_peak_sust, 4),
        },
        "gemm": {
            "fprop_dgrad_ms": round(avg_blk, 4), "wgrad_ms": round(avg_wg, 4),
            "fprop_dgrad_tflops": round(achieved, 1),
            "wgrad_tflops": round(GEMM_FLOP / (avg_wg * 1e-3) / 1e12, 1),
            "gemm_only_tflops": round(GEMM_FLOP * GEMMS_PER_STEP / (gemm_only_ms * 1e-3) / 1e12, 1),
            "wgrad_frac_of_fp8_peak": round(GEMM_FLOP / (avg_wg * 1e-3) / 1e12 / fp8_peak, 4),
        },
        "quantizers": {
            "bytes_per_step": quant_bytes_per_step(),
            "ms_per_step_est": round(quant_ms, 4),
            "gbs_est": round(quant_bytes_per_step() / (quant_ms * 1e-3) / 1e9, 1),
            "hbm_peak_gbs": peaks["hbm"],
            "note": "step time minus the event-timed GEMMs; per-kernel figures in profiles/",
        },
        "e2e": {"value": round(e2e, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if rank == 0:
        if not args.no_extras:
            del step, pinned, dw_host, t_sets, dw_sets
            torch.cuda.empty_cache()
            peaks_now = _peaks()
            line["decode"] = measure_decode(dev, peaks_now)
            line["mxfp8"] = measure_mxfp8(dev)
            line["block128_pow2"] = measure_pow2(dev)
            line["requant_dequant"] = measure_f3_kernels(dev)
            line["fused_producers"] = measure_fused_producers(dev)
            line["nvfp4"] = measure_nvfp4(dev)
            line["rollout_step"] = measure_rollout_step(dev, peaks_now)
            line["moe"] = measure_moe(dev)
            if step_error():
                raise RuntimeError("device error word set during the secondary measurements")
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.cpu_sample_rows)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# --------------------------------------------------------------------------- oracle

_SAMPLE_CACHE = {}


def _oracle_sample(rows: int, band: int = 1024, seed: int = 0, threads: int | None = None):
    """The oracle on a slice of the workload, its calls spread over the host cores
    (ctypes releases the GIL around each C call): quantize `rows` tokens of X (row
    and column copies, 128-token slices per task) and the first `band` output rows
    of W_up (128x128 blocks, one 128-row band per task), dequantize, FP64 FProp of
    those tokens against that band.  Returns (seconds, flops, threads)."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle
    import synth

    threads = threads or os.cpu_count() or 1
    key = (seed, rows, band)
    if key not in _SAMPLE_CACHE:
        _SAMPLE_CACHE[key] = (synth.activation(N_TOK, C, seed=seed, stream="x")[:rows].copy(),
                              synth.weight(D, C, seed=seed, stream="w_up")[:band].copy())
    x, w = _SAMPLE_CACHE[key]

    def weight_band(r0):
        q, s_, _, _ = oracle.quant_blocks(w[r0:r0 + 128])
        return oracle.dequant_blocks(q, s_)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        W = np.concatenate(list(ex.map(weight_band, range(0, band, 128))))

        def token_slice(r0):
            xs = x[r0:r0 + 128]
            qx, sx = oracle.quant_rowgroups(xs)
            oracle.quant_colgroups(xs)
            return oracle.fprop(oracle.dequant_rowgroups(qx, sx), W)[0].shape

        list(ex.map(token_slice, range(0, rows, 128)))
    return time.perf_counter() - t0, 2.0 * rows * band * C, threads


def cpu_baseline(rows: int):
    secs, flops, threads = _oracle_sample(rows)
    return {"value": round(flops / secs / 1e12, 8), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} tokens of the step on {threads} host threads (os.cpu_count() = {os.cpu_count()}): "
                      f"1x128 + 128x1 quantization of X[{rows}x4096] in 128-token slices, 128x128 quantization of "
                      f"W_up[0:1024] in 128-row bands, FP64 FProp {rows}x1024x4096 ({secs:.1f} s wall)"}


def run_reference(args):
    rank, world, _ = _rank_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    for _ in range(args.warmup):
        _oracle_sample(args.ref_rows)
    total_s, total_f, threads = 0.0, 0.0, 1
    for _ in range(args.steps):
        s, f, threads = _oracle_sample(args.ref_rows)
        total_s += s
        total_f += f
    v = total_f / total_s / 1e12
    sample = f"each step: {args.ref_rows} tokens of X quantized (row + column copies), W_up[0:1024] quantized " \
             f"(128x128 blocks), FP64 FProp {args.ref_rows}x1024x4096; the C oracle on {threads} host threads " \
             f"(os.cpu_count() = {os.cpu_count()})"
    line = {
        "metric": METRIC, "value": round(v, 8), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * total_s / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": CONFIG,
        "impl": "reference",
        "cpu_baseline": {"value": round(v, 8), "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 8), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PROFILE_CASES = {
    # name: (description, inputs are all larger than the 129 MB L2)
    "gemm_fprop": "FProp 4096 x 12288 x 4096 (training shape, BF16 out)",
    "gemm_wgrad": "WGrad 12288 x 4096 x K=4096 (training shape, FP32 out)",
    "decode": "FProp 8 tokens x 12288 x 12288 (decode shape, 151 MB of FP8 weight)",
    "quant_act": "activation quantizer, X 8192 x 12288 BF16 (row + column copies)",
    "quant_w": "weight quantizer, W 12288 x 12288 BF16 (+ transposed copy)",
    "quant_mx": "MXFP8 quantizer, X 8192 x 12288 BF16 (row + column copies)",
    "gemm_mx_fprop": "MXFP8 FProp 4096 x 12288 x 4096 (BF16 out)",
    "grouped_fprop": "grouped FProp, 32 experts x 1536 x 2048, 16384 routed rows (Zipf 1.2), BF16 out",
    "requant_col": "column copy re-quantized from the row copy of H 8192 x 12288",
    "dequant_bf16": "BF16 dequantization of the row copy of H 8192 x 12288",
    "quant_rmsnorm": "RMSNorm statistics + fused RMSNorm quantizer, X 32768 x 4096 BF16 (row + column copies)",
    "quant_swiglu": "fused SwiGLU quantizer, gate and up 8192 x 12288 BF16 (row + column copies)",
    "quant_nvfp4": "NVFP4 quantizer, per-token scope, 131072 routed rows x 2048 BF16",
    "gemm_nvfp4": "NVFP4 FProp 4096 x 12288 x 4096 (per-token x tensor scope, BF16 out)",
    "decode_narrow": "FProp 128 tokens x W_down 4096 x 12288 (narrow 32-row weight tiles, BF16 out)",
    "gemm_mx_dgrad": "MXFP8 DGrad 4096 x 4096 x 12288 (BF16 out)",
    "gemm_mx_wgrad": "MXFP8 WGrad 12288 x 4096 x K=4096 (FP32 out)",
    "grouped_wgrad": "grouped WGrad, 32 experts x 1536 x 2048, 16384 routed rows (Zipf 1.2), FP32 out",
    "quant_act_pow2": "power-of-two 1x128 row + 128x1 column copies, X 8192 x 12288 BF16",
    "quant_w_pow2": "power-of-two 128x128 weight blocks + transposed copy, W 12288 x 12288 BF16",
    "amax_bf16": "max |x| over 131072 x 2048 BF16 (NVFP4 tensor scope)",
    "dequant_nvfp4": "BF16 dequantization of the NVFP4 copy of 131072 x 2048 (per-token scope)",
    "decode_split": "split-K FProp 8 tokens x W_down 4096 x 12288 with a workspace (4 weight copies rotate: 201 MB)",
    "grouped_mx_fprop": "MXFP8 grouped FProp, 32 experts x 1536 x 2048, 16384 routed rows (Zipf 1.2), BF16 out",
}


def run_case(name: str, launches: int = 5):
    """A few launches of one kernel on a mid-size case, for ncu captures."""
    import torch

    import __graft_entry__
    import rollout_x128_act_gb300 as jq
    import synth

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)

    def bf16(a):
        import numpy as np

        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    if name in ("gemm_fprop", "gemm_wgrad", "decode"):
        n, c, d = {"gemm_fprop": (4096, 4096, 12288), "gemm_wgrad": (4096, 4096, 12288),
                   "decode": (8, 12288, 12288)}[name]
        x = bf16(synth.activation(n, c, seed=0, stream="x"))
        w = bf16(synth.weight(d, c, seed=0, stream="w_up"))
        ax = jq.quant_act(x, col=(name == "gemm_wgrad"))
        qw, sw, _, _ = jq.quant_weight(w, transposed=False)
        if name == "gemm_wgrad":
            dy = bf16(synth.gradient(n, d, seed=0, stream="dy_up"))
            ady = jq.quant_act(dy, row=False)
            out = torch.empty((d, c), dtype=torch.float32, device=dev)
            fn = lambda: jq.wgrad(ady["q_col"], ady["s_col"], ax["q_col"], ax["s_col"], n, dw=out)  # noqa: E731
        else:
            path = jq.PATH_DECODE if name == "decode" else jq.PATH_TRAIN
            out = torch.empty((n, d), dtype=torch.bfloat16, device=dev)
            fn = lambda: jq.jetq_gemm_fprop(jq.RECIPE_BLOCK128, ax["q_row"], ax["s_row"], qw, sw, n, d, c,  # noqa
                                            out, path)
    elif name == "decode_split":
        n, c, d = 8, 12288, 4096
        ax = jq.quant_act(bf16(synth.activation(n, c, seed=0, stream="h")), col=False)
        wq = [jq.quant_weight(bf16(synth.weight(d, c, seed=i, stream="w_down")), transposed=False) for i in range(4)]
        out = torch.empty((n, d), dtype=torch.bfloat16, device=dev)
        work = torch.empty(jq.jetq_decode_workspace_bytes(n, d, c), dtype=torch.uint8, device=dev)
        turn = [0]

        def fn():
            qw, sw, _, _ = wq[turn[0] % 4]
            turn[0] += 1
            jq.jetq_gemm_fprop_ws(jq.RECIPE_BLOCK128, ax["q_row"], ax["s_row"], qw, sw, n, d, c, out, work,
                                  jq.PATH_DECODE)
    elif name == "gemm_mx_fprop":
        n, c, d = 4096, 4096, 12288
        gx = jq.quant_mx(bf16(synth.activation(n, c, seed=0, stream="x")), col=False)
        gw = jq.quant_mx(bf16(synth.weight(d, c, seed=0, stream="w_up")), col=False)
        out = torch.empty((n, d), dtype=torch.bfloat16, device=dev)
        fn = lambda: jq.jetq_gemm_fprop(jq.RECIPE_MXFP8, gx["q_row"], gx["e8_row"], gw["q_row"], gw["e8_row"],  # noqa
                                        n, d, c, out, jq.PATH_TRAIN)
    elif name == "grouped_fprop":
        E, c, d = 32, 2048, 1536
        off, _ = synth.zipf_topk_routing(2048, E, 8, 1.2, seed=0)
        R = int(off[-1])
        seg = torch.tensor(off, dtype=torch.int64, device=dev)
        ax = jq.quant_act(bf16(synth.activation(R, c, seed=0, stream="x")), col=False)
        ws = bf16(synth.weight(E * d, c, seed=0, stream="w_gate"))
        qs = [jq.quant_weight(ws[e * d:(e + 1) * d], transposed=False) for e in range(E)]
        qw, sw = torch.stack([q[0] for q in qs]), torch.stack([q[1] for q in qs])
        out = torch.empty((R, d), dtype=torch.bfloat16, device=dev)
        fn = lambda: jq.grouped(jq.GEMM_FPROP, ax["q_row"], ax["s_row"], qw, sw, seg, n=d, k=c, out=out)  # noqa
    elif name == "grouped_mx_fprop":
        E, c, d = 32, 2048, 1536
        off, _ = synth.zipf_topk_routing(2048, E, 8, 1.2, seed=0)
        R = int(off[-1])
        seg = torch.tensor(off, dtype=torch.int64, device=dev)
        gx = jq.quant_mx(bf16(synth.activation(R, c, seed=0, stream="x")), col=False, seg_offsets=seg)
        ws = bf16(synth.weight(E * d, c, seed=0, stream="w_gate"))
        gws = [jq.quant_mx(ws[e * d:(e + 1) * d], col=False) for e in range(E)]
        qw, ew = torch.stack([g["q_row"] for g in gws]), torch.cat([g["e8_row"] for g in gws])
        out = torch.empty((R, d), dtype=torch.bfloat16, device=dev)
        fn = lambda: jq.grouped(jq.GEMM_FPROP, gx["q_row"], gx["e8_row"], qw, ew, seg, n=d, k=c, out=out,  # noqa
                                recipe=jq.RECIPE_MXFP8)
    elif name in ("requant_col", "dequant_bf16"):
        a = jq.quant_act(bf16(synth.activation(8192, 12288, seed=0, stream="h")), col=False)
        if name == "requant_col":
            gcol = jq.requant_col(a["q_row"], a["s_row"])
            fn = lambda: jq.jetq_requant_col_from_row(a["q_row"], a["s_row"], gcol["q_col"], gcol["s_col"],  # noqa
                                                      gcol["ldq_col"])
        else:
            out = torch.empty((8192, 12288), dtype=torch.bfloat16, device=dev)
            fn = lambda: jq.jetq_dequant_bf16(a["q_row"], a["s_row"], jq.SCALES_ROWGROUPS_1X128, out)  # noqa
    elif name == "quant_rmsnorm":
        x = bf16(synth.activation(32768, 4096, seed=0, stream="x"))
        w = bf16(synth.bf16_bits(1.0 + 0.1 * synth.normal(4096, seed=0, stream=synth.STREAM["x"])))
        fn = lambda: jq.quant_act_rmsnorm(x, w)  # noqa: E731
    elif name == "quant_swiglu":
        gate = bf16(synth.activation(8192, 12288, seed=0, stream="h"))
        up = bf16(synth.activation(8192, 12288, seed=1, stream="h"))
        fn = lambda: jq.quant_act_swiglu(gate, up)  # noqa: E731
    elif name == "quant_nvfp4":
        x = bf16(synth.activation(131072, 2048, seed=0, stream="x"))
        fn = lambda: jq.quant_nvfp4(x)  # noqa: E731
    elif name == "decode_narrow":
        n, c, d = 128, 12288, 4096
        ax = jq.quant_act(bf16(synth.activation(n, c, seed=0, stream="h")), col=False)
        qw, sw, _, _ = jq.quant_weight(bf16(synth.weight(d, c, seed=0, stream="w_down")), transposed=False)
        out = torch.empty((n, d), dtype=torch.bfloat16, device=dev)
        fn = lambda: jq.jetq_gemm_fprop(jq.RECIPE_BLOCK128, ax["q_row"], ax["s_row"], qw, sw, n, d, c, out,  # noqa
                                        jq.PATH_DECODE)
    elif name in ("gemm_mx_dgrad", "gemm_mx_wgrad"):
        n, c, d = 4096, 4096, 12288
        gdy = jq.quant_mx(bf16(synth.gradient(n, d, seed=0, stream="dy_up")))
        if name == "gemm_mx_dgrad":
            gw = jq.quant_mx(bf16(synth.weight(d, c, seed=0, stream="w_up")))
            out = torch.empty((n, c), dtype=torch.bfloat16, device=dev)
            fn = lambda: jq.jetq_gemm_dgrad(jq.RECIPE_MXFP8, gdy["q_row"], gdy["e8_row"], gw["q_col"],  # noqa
                                            gw["e8_col"], n, d, c, out)
        else:
            gx = jq.quant_mx(bf16(synth.activation(n, c, seed=0, stream="x")))
            out = torch.empty((d, c), dtype=torch.float32, device=dev)
            fn = lambda: jq.jetq_gemm_wgrad(jq.RECIPE_MXFP8, gdy["q_col"], gdy["e8_col"], gx["q_col"],  # noqa
                                            gx["e8_col"], n, gx["ldq_col"], d, c, out)
    elif name == "grouped_wgrad":
        E, c, d = 32, 2048, 1536
        off, _ = synth.zipf_topk_routing(2048, E, 8, 1.2, seed=0)
        R = int(off[-1])
        seg = torch.tensor(off, dtype=torch.int64, device=dev)
        ax = jq.quant_act(bf16(synth.activation(R, c, seed=0, stream="x")), row=False, seg_offsets=seg)
        ady = jq.quant_act(bf16(synth.gradient(R, d, seed=0, stream="dy_gate")), row=False, seg_offsets=seg)
        P = int(sum((int(off[e + 1] - off[e]) + 127) // 128 * 128 for e in range(E)))
        out = torch.empty((E, d, c), dtype=torch.float32, device=dev)
        fn = lambda: jq.grouped(jq.GEMM_WGRAD, ady["q_col"], ady["s_col"], ax["q_col"], ax["s_col"], seg, n=c,  # noqa
                                k=P, out=out)
    elif name == "quant_act_pow2":
        x = bf16(synth.activation(8192, 12288, seed=0, stream="h"))
        fn = lambda: jq.quant_act_pow2(x)  # noqa: E731
    elif name == "quant_w_pow2":
        w = bf16(synth.weight(12288, 12288, seed=0, stream="w"))
        fn = lambda: jq.quant_weight_pow2(w)  # noqa: E731
    elif name == "amax_bf16":
        x = bf16(synth.activation(131072, 2048, seed=0, stream="x"))
        fn = lambda: jq.amax_bf16(x)  # noqa: E731
    elif name == "dequant_nvfp4":
        o = jq.quant_nvfp4(bf16(synth.activation(131072, 2048, seed=0, stream="x")))
        fn = lambda: jq.dequant_nvfp4_bf16(o["q"], o["sb"], o["sg"])  # noqa: E731
    elif name == "gemm_nvfp4":
        n, c, d = 4096, 4096, 12288
        ga = jq.quant_nvfp4(bf16(synth.activation(n, c, seed=0, stream="x")))
        ga["atoms"] = jq.nvfp4_atoms(ga["sb"], c)
        wd = bf16(synth.weight(d, c, seed=0, stream="w_up"))
        gw = jq.quant_nvfp4(wd, scope_amax=jq.amax_bf16(wd))
        gw["atoms"] = jq.nvfp4_atoms(gw["sb"], c)
        fn = lambda: jq.nvfp4_fprop(ga, gw, c, out_dtype=torch.bfloat16)  # noqa: E731
    elif name == "quant_mx":
        x = bf16(synth.activation(8192, 12288, seed=0, stream="h"))
        fn = lambda: jq.quant_mx(x)  # noqa: E731
    elif name == "quant_act":
        x = bf16(synth.activation(8192, 12288, seed=0, stream="h"))
        fn = lambda: jq.quant_act(x)  # noqa: E731
    elif name == "quant_w":
        w = bf16(synth.weight(12288, 12288, seed=0, stream="w"))
        fn = lambda: jq.quant_weight(w)  # noqa: E731
    else:
        raise SystemExit(f"unknown case {name}; one of {sorted(PROFILE_CASES)}")
    torch.cuda.synchronize()
    for _ in range(launches):
        fn()
    torch.cuda.synchronize()
    if jq.jetq_check_device_error() != 0:
        raise RuntimeError("device error word set")
    print(f"case {name}: {PROFILE_CASES[name]}: {launches} launches ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample-rows", type=int, default=8192)
    ap.add_argument("--ref-rows", type=int, default=1024)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the decode / MXFP8 / MoE measurements")
    ap.add_argument("--case", default=None, help="profiling case: " + ", ".join(sorted(PROFILE_CASES)))
    args = ap.parse_args()
    if args.case:
        run_case(args.case)
        return
    args.warmup = max(3, args.warmup)  # timing rule: at least 3 warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
