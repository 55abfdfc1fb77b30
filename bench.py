"""Benchmark of the quantized decode linear layer on GB300.

Default workload: INT8 W8A8 skinny GEMM at the 27B-class decode shapes
(N,K) in {(17408,5120), (5120,17408), (10240,5120)} x M in {1,2,4,8,16} tokens.
One step = one call of each of those 15 (shape, M) cases (per-token INT8 activation
quantisation + skinny GEMM each).  Metric: achieved HBM GB/s = algorithmic bytes
(weights + weight scales + activations + outputs) / device time, plus µs per call.

Weights rotate over 6 copies per shape (>= 1 GB in total), so every call streams its
weights from HBM (no call finds them in the 129 MB L2).  Activations are small and stay
wherever the previous write left them, as in a decode step.

--config selects the other workloads (c0: INT8 M=1 N=512 K=1024; c2: FP8 128x128 block;
c3: MXFP4 MoE E=256 H=4096 I=2048 top-8; c4: tcgen05 FP8/MXFP4 M=64..256;
n2: FP8 E4M3 per-channel scales; n4: BF16 unquantised weights).
--impl reference times the CPU oracle on a bounded row sample of the same workload.
Under torchrun each rank runs an independent replica (the layer needs no exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# the CPU oracle's numpy calls run single-threaded; its parallel mode splits the output rows
# over a thread pool of its own (set before numpy loads its BLAS)
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "µs/call and achieved HBM GB/s (% of GB300 roofline) for quantized decode GEMV"
C1_SHAPES = [(17408, 5120), (5120, 17408), (10240, 5120)]
C1_MS = [1, 2, 4, 8, 16]
C2_SHAPES = [(17408, 5120), (5120, 17408)]
C2_MS = [1, 4, 8, 16]
C3_MS = list(range(1, 10))
C4_MS = [64, 128, 256]
ROTATE = 6  # weight copies per shape (>= 3 x 44.6 MB between reuses)


# one name per workload, used by both arms
WORKLOADS = {
    "c0": "INT8 W8A8 GEMV M=1 N=512 K=1024",
    "c1": "INT8 W8A8 skinny GEMM, 27B-class decode shapes (N,K) in {(17408,5120),(5120,17408),(10240,5120)} "
          "x M in {1,2,4,8,16}",
    "c2": "FP8 E4M3 128x128 UE8M0 block-scaled GEMV, bf16 activations, (N,K) in {(17408,5120),(5120,17408)} "
          "x M in {1,4,8,16}",
    "c3": "MXFP4 MoE decode: 256 experts, hidden 4096, intermediate 2048, top-8, M in 1..9",
    "c4": "tcgen05 block-scaled GEMM, 1x128 E4M3 activations, FP8 128x128 and MXFP4 weights, "
          "(N,K)=(17408,5120), M in {64,128,256}",
    "n3": "MXFP4 MoE decode with clamped SwiGLU (alpha 1, limit 10): 256 experts, hidden 4096, "
          "intermediate 2048, top-8, M in 1..9",
    "n1": "INT8 W8A8 for more than 16 tokens (M = 32: the persistent skinny kernel with four 8-token MMA tiles; "
          "M > 32: per-token quantisation + tcgen05 kind::f16 MMAs on exact f16 images), "
          "27B-class shapes (N,K) in {(17408,5120),(5120,17408),(10240,5120)} x M in {32,64,128,256}",
    "n5": "Grouped MXFP4 MoE on the tcgen05 path with 1x128 E4M3 activations: 256 experts, hidden 4096, "
          "intermediate 2048, top-8, M in {32,64,128,256}",
    "n2": "FP8 E4M3 per-channel-scaled decode GEMV, bf16 activations, (N,K) in "
          "{(17408,5120),(5120,17408),(10240,5120)} x M in {1,4,16}",
    "n4": "BF16 dense decode GEMV (unquantised weights), (N,K) in {(17408,5120),(5120,17408)} x M in {1,4,16}",
}
# the arithmetic type of each workload's weights
DTYPES = {"c0": "int8", "c1": "int8", "c2": "fp8", "c3": "fp4", "c4": "fp8/fp4", "n1": "int8", "n2": "fp8", "n3": "fp4", "n4": "bf16", "n5": "fp4/fp8"}


# ----------------------------------------------------------------------------- bytes / flops
def bytes_int8(M, N, K):
    return N * K + 4 * N + 2 * M * K + 2 * M * N


def bytes_fp8(M, N, K):
    return N * K + (-(-N // 128)) * (-(-K // 128)) + 2 * M * K + 2 * M * N


def bytes_fp8c(M, N, K, per_channel=True):
    return N * K + (4 * N if per_channel else 4) + 2 * M * K + 2 * M * N


def bytes_bf16(M, N, K):
    return 2 * N * K + 2 * M * K + 2 * M * N


def bytes_mxfp4(M, N, K):
    return N * K // 2 + N * K // 32 + 2 * M * K + 2 * M * N


def bytes_moe_expert(H, I):
    return 2 * I * H // 2 + 2 * I * H // 32 + H * I // 2 + H * I // 32


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# the sources that define each configuration's kernels (device code and the host code that
# plans their launches): a committed traffic figure holds while these files are unchanged
_SKINNY_SRC = ("skinny.cuh", "skinny2.cuh", "skinny2_kernel.cuh", "kernels_skinny2.cu", "kernels_skinny.cu",
               "kernels_quant.cu", "kernels_moe.cu", "route.cuh", "tc_ptx.cuh", "common.cuh", "internal.h", "api.cu")
_TC_SRC = ("gemm_tcgen05.cu", "gemm_tcgen05.h", "kernels_quant.cu", "quant_e4m3.cuh", "tc_ptx.cuh", "common.cuh",
           "internal.h", "api.cu")
_I8_SRC = ("gemm_i8_tcgen05.cu", "gemm_i8_tcgen05.h", "kernels_quant.cu", "tc_ptx.cuh", "common.cuh", "internal.h",
           "api.cu")
KERNEL_SOURCES = {"c0": _SKINNY_SRC, "c1": _SKINNY_SRC, "c2": _SKINNY_SRC, "c3": _SKINNY_SRC, "c4": _TC_SRC,
                  "n1": tuple(dict.fromkeys(_I8_SRC + _SKINNY_SRC)), "n2": _SKINNY_SRC, "n3": _SKINNY_SRC, "n4": _SKINNY_SRC,
                  "n5": _TC_SRC + ("kernels_moe_grouped.cu", "route.cuh", "kernels_moe.cu")}


def kernel_source_hash(config):
    h = hashlib.sha1()
    for f in KERNEL_SOURCES[config]:
        h.update(open(os.path.join(ROOT, "skinny_gemm_dequant_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:12]


def load_traffic(config):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, or None if
    the summary is missing or the kernels changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(config)
    if not d or d.get("source_hash") != kernel_source_hash(config):
        return None
    return d.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- workloads (GPU)
def static_cfg(name):
    """The `config` object of a workload: the same for both arms (it describes the work, not
    the device)."""
    if name in ("c0", "c1", "n1"):
        shapes = [(512, 1024)] if name == "c0" else C1_SHAPES
        Ms = {"c0": [1], "c1": C1_MS, "n1": N1_MS}[name]
        return {"workload": WORKLOADS[name], "shapes": [list(x) for x in shapes], "M": Ms}
    if name in ("c3", "n3", "n5"):
        return {"workload": WORKLOADS[name], "bytes": "unique touched experts x 13369344 B + x + logits + y"}
    return {"workload": WORKLOADS[name]}


def arm_config(name, ws):
    return dict(static_cfg(name), parallelism=f"replicas x{ws}",
                l2="weights rotate over 6 copies per shape (inputs larger than L2)")


class Workload:
    """A list of calls; each call(i) enqueues one layer call on the current stream."""

    def __init__(self, name, calls, launches_per_step, cfg):
        self.name, self.calls, self.launches_per_step, self.cfg = name, calls, launches_per_step, cfg

    @property
    def bytes_per_step(self):
        return sum(c["bytes"] for c in self.calls)


def dev_bf16(bits, torch):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def build_c1(ql, torch, shapes=C1_SHAPES, Ms=C1_MS, name="c1"):
    calls = []
    weights = {}
    for (N, K) in shapes:
        c = synth.int8_case(1, N, K, seed=0)
        w0 = torch.from_numpy(c["w"]).cuda()
        weights[(N, K)] = ([w0] + [w0.clone() for _ in range(ROTATE - 1)], torch.from_numpy(c["w_s"]).cuda(),
                           {"i": 0})
    for M in Ms:  # shapes inner; each use of a shape takes the next weight copy
        for (N, K) in shapes:
            ws, sc, state = weights[(N, K)]
            x = dev_bf16(synth.int8_case(M, 1, K, seed=1)["x"], torch)
            y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")

            def call(ws=ws, sc=sc, x=x, y=y, state=state):
                w = ws[state["i"] % ROTATE]
                state["i"] += 1
                ql.qlinear_int8_w8a8(x, w, sc, out=y)

            calls.append({"fn": call, "M": M, "N": N, "K": K, "bytes": bytes_int8(M, N, K), "flops": 2 * M * N * K,
                          "x": x, "y": y, "kind": "int8"})
    return Workload(name, calls, len(calls), static_cfg(name))  # one fused launch per call


def build_c0(ql, torch):
    return build_c1(ql, torch, shapes=[(512, 1024)], Ms=[1], name="c0")


def build_c2(ql, torch):
    calls = []
    weights = {}
    for (N, K) in C2_SHAPES:
        c = synth.fp8_block_case(1, N, K, seed=0)
        w0 = torch.from_numpy(c["w"]).cuda()
        weights[(N, K)] = ([w0] + [w0.clone() for _ in range(ROTATE - 1)], torch.from_numpy(c["s"]).cuda(),
                           {"i": 0})
    for M in C2_MS:
        for (N, K) in C2_SHAPES:
            ws, sc, state = weights[(N, K)]
            x = dev_bf16(synth.fp8_block_case(M, 1, K, seed=1)["x"], torch)
            y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")

            def call(ws=ws, sc=sc, x=x, y=y, state=state):
                w = ws[state["i"] % ROTATE]
                state["i"] += 1
                ql.qlinear_fp8_block(x, w, sc, out=y)

            calls.append({"fn": call, "M": M, "N": N, "K": K, "bytes": bytes_fp8(M, N, K), "flops": 2 * M * N * K,
                          "x": x, "y": y, "kind": "fp8"})
    return Workload("c2", calls, len(calls), static_cfg("c2"))


def build_c3(ql, torch, limit=None, name="c3", Ms=None):
    from oracle import qlinear_oracle as Q  # only to count the experts each routing touches
    E, H, I, topk = 256, 4096, 2048, 8
    w = synth.moe_weights_only(E, H, I, seed=0)
    dev = [torch.from_numpy(w[k]).cuda() for k in ("w13", "s13", "w2", "s2")]
    calls = []
    grouped = Ms is not None  # batches above 16 tokens: the grouped tcgen05 path
    for M in (Ms or C3_MS):
        sets = []
        for r in range(ROTATE):  # different routings per rotation: different experts, cold L2
            t = synth.moe_tokens(M, E, H, seed=100 + 10 * M + r)
            ids, _ = Q.route_topk(t["logits"], topk)
            sets.append((dev_bf16(t["x"], torch), dev_bf16(t["logits"], torch), len(np.unique(ids))))
        y = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
        state = {"i": 0}

        def call(sets=sets, y=y, state=state):
            x, lg, _ = sets[state["i"] % ROTATE]
            state["i"] += 1
            ql.moe_mxfp4_grouped(x, *dev, router_logits=lg, topk=topk, swiglu_limit=limit, out=y)

        uniq = float(np.mean([s[2] for s in sets]))
        b = uniq * bytes_moe_expert(H, I) + 2 * M * H * 2 + 2 * M * E
        calls.append({"fn": call, "M": M, "N": H, "K": I, "bytes": b, "flops": 2 * M * topk * 3 * H * I,
                      "x": sets[0][0], "y": y, "kind": "moe_tcgen05" if grouped else "moe",
                      "inputs": [t for st in sets for t in st[:2]],  # every rotation's x and logits
                      "unique_experts": uniq})
    cfg = static_cfg(name)
    # skinny path: gate_up (with routing), down, combine, twice for 9..16 tokens (two calls of 8
    # and M - 8 tokens); grouped path: routing, dispatch, quantise-and-scatter, gate_up GEMM,
    # h quantisation, down GEMM, combine
    launches = sum(7 if grouped else (6 if c["M"] > 8 else 3) for c in calls)
    return Workload(name, calls, launches, cfg)


N5_MS = [32, 64, 128, 256]


def build_n5(ql, torch):
    """Grouped MoE for larger batches on the tcgen05 path (a NEXT row)."""
    return build_c3(ql, torch, name="n5", Ms=N5_MS)


def build_n3(ql, torch):
    """The MoE workload with the clamped SwiGLU (alpha 1, limit 10) as the expert activation."""
    return build_c3(ql, torch, limit=10.0, name="n3")


def build_c4(ql, torch):
    calls = []
    N, K = 17408, 5120
    cf = synth.fp8_block_case(1, N, K, seed=0)
    cm = synth.mxfp4_dense_case(1, N, K, seed=0)
    lds = -(-(K // 32) // 16) * 16
    sm = np.zeros((N, lds), np.uint8)
    sm[:, : K // 32] = cm["s"]
    fw = torch.from_numpy(cf["w"]).cuda()
    mw = torch.from_numpy(cm["w"]).cuda()
    fws = [fw] + [fw.clone() for _ in range(ROTATE - 1)]
    mws = [mw] + [mw.clone() for _ in range(ROTATE - 1)]
    fs = torch.from_numpy(cf["s"]).cuda()
    ms = torch.from_numpy(sm).cuda()
    rot = {"fp8": {"i": 0}, "mxfp4": {"i": 0}}
    for M in C4_MS:
        x = dev_bf16(synth.fp8_block_case(M, 1, K, seed=1)["x"], torch)
        for kind in ("fp8", "mxfp4"):
            y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            state = rot[kind]
            if kind == "fp8":
                def call(x=x, y=y, state=state):
                    w = fws[state["i"] % ROTATE]
                    state["i"] += 1
                    ql.qlinear_fp8_block(x, w, fs, act_mode=ql.ACT_E4M3_1X128, out=y)
                b = bytes_fp8(M, N, K)
            else:
                def call(x=x, y=y, state=state):
                    w = mws[state["i"] % ROTATE]
                    state["i"] += 1
                    ql.qlinear_mxfp4(x, w, ms, act_mode=ql.ACT_E4M3_1X128, out=y)
                b = bytes_mxfp4(M, N, K)
            calls.append({"fn": call, "M": M, "N": N, "K": K, "bytes": b, "flops": 2 * M * N * K, "x": x, "y": y,
                          "kind": kind + "_tcgen05"})
    return Workload("c4", calls, 2 * len(calls), static_cfg("c4"))


N4_MS = [1, 4, 16]


def build_n4(ql, torch):
    """BF16 dense decode GEMV (a NEXT row: unquantised weights on the same skinny kernel)."""
    calls = []
    weights = {}
    for (N, K) in C2_SHAPES:
        c = synth.bf16_dense_case(1, N, K, seed=0)
        w0 = torch.from_numpy(c["w"].view(np.int16)).cuda().view(torch.bfloat16)
        weights[(N, K)] = ([w0] + [w0.clone() for _ in range(ROTATE - 1)], {"i": 0})
    for M in N4_MS:
        for (N, K) in C2_SHAPES:
            ws, state = weights[(N, K)]
            x = dev_bf16(synth.bf16_dense_case(M, 1, K, seed=1)["x"], torch)
            y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")

            def call(ws=ws, x=x, y=y, state=state):
                w = ws[state["i"] % ROTATE]
                state["i"] += 1
                ql.qlinear_bf16(x, w, out=y)

            calls.append({"fn": call, "M": M, "N": N, "K": K, "bytes": bytes_bf16(M, N, K), "flops": 2 * M * N * K,
                          "x": x, "y": y, "kind": "bf16"})
    return Workload("n4", calls, len(calls), static_cfg("n4"))


N1_MS = [32, 64, 128, 256]


def build_n1(ql, torch):
    """INT8 W8A8 for M > 16 (a NEXT row): the tcgen05 GEMM, two launches per call."""
    w = build_c1(ql, torch, shapes=C1_SHAPES, Ms=N1_MS, name="n1")
    # M <= 32: one skinny launch; above: quantisation + GEMM
    w.launches_per_step = sum(1 if c["M"] <= 32 else 2 for c in w.calls)
    for c in w.calls:
        c["kind"] = "int8_skinny" if c["M"] <= 32 else "int8_tcgen05"
    return w


N2_SHAPES = C1_SHAPES
N2_MS = [1, 4, 16]


def build_n2(ql, torch):
    """FP8 weights with one fp32 scale per output channel (a NEXT row: e4m3fn codes, the scale
    applied once at the end), on the 27B-class decode shapes the pages time the emulated FP8
    GEMV on."""
    calls = []
    weights = {}
    for (N, K) in N2_SHAPES:
        c = synth.fp8_channel_case(1, N, K, seed=0)
        w0 = torch.from_numpy(c["w"]).cuda()
        weights[(N, K)] = ([w0] + [w0.clone() for _ in range(ROTATE - 1)], torch.from_numpy(c["w_s"]).cuda(),
                           {"i": 0})
    for M in N2_MS:
        for (N, K) in N2_SHAPES:
            ws, sc, state = weights[(N, K)]
            x = dev_bf16(synth.fp8_channel_case(M, 1, K, seed=1)["x"], torch)
            y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")

            def call(ws=ws, sc=sc, x=x, y=y, state=state):
                w = ws[state["i"] % ROTATE]
                state["i"] += 1
                ql.qlinear_fp8(x, w, sc, "e4m3", out=y)

            calls.append({"fn": call, "M": M, "N": N, "K": K, "bytes": bytes_fp8c(M, N, K), "flops": 2 * M * N * K,
                          "x": x, "y": y, "kind": "fp8_channel"})
    return Workload("n2", calls, len(calls), static_cfg("n2"))


BUILDERS = {"c0": build_c0, "c1": build_c1, "c2": build_c2, "c3": build_c3, "c4": build_c4, "n1": build_n1, "n2": build_n2,
            "n3": build_n3, "n5": build_n5,
            "n4": build_n4}

_SKINNY = ("skinny2_kernel (one launch per call: activation preparation + weight-streaming GEMM); "
           "achieved = the step's algorithmic bytes / the step's device time")
_MOE = ("MoE launches per call (gate_up with the routing fused in, down, combine); the step's touched-expert "
        "bytes / the step's device time")
KERNEL_DESC = {"c0": _SKINNY, "c1": _SKINNY, "c2": _SKINNY, "n2": _SKINNY, "n4": _SKINNY,
               "c3": _MOE, "n3": _MOE,
               "n5": "grouped MoE launches per call (routing, dispatch, activation quantisation, two grouped "
                     "tcgen05 GEMMs, h quantisation, combine); the step's touched-expert bytes / device time",
               "c4": "tcgen05 block-scaled GEMM + its activation-quantisation launch; the step's bytes / device time",
               "n1": "INT8 for M = 32..256: skinny2_kernel (M = 32) or the tcgen05 GEMM + its per-token quantisation "
                     "launch (M > 32); the step's bytes / device time"}


# ----------------------------------------------------------------------------- timing
def capture(torch, body):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()
    return g


def step_graphs(wl, torch):
    """ROTATE graphs of one step each, captured in order: replaying them cyclically keeps every
    use of a weight set on a different copy than the previous use."""
    def body():
        for c in wl.calls:
            c["fn"]()
    return [capture(torch, body) for _ in range(ROTATE)]


def time_steps(graphs, steps, torch):
    st = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for i in range(steps):
        graphs[i % len(graphs)].replay()
    b.record(st)
    b.synchronize()
    return a.elapsed_time(b)  # ms


def time_per_call(wl, torch, uses=32, reps=8):
    """µs per call: a graph of `uses` back-to-back calls of one case (rotating weight copies),
    replayed `reps` times between two events."""
    st = torch.cuda.current_stream()
    out = []
    for c in wl.calls:
        def body(c=c):
            for _ in range(uses):
                c["fn"]()
        g = capture(torch, body)
        g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(reps):
            g.replay()
        b.record(st)
        b.synchronize()
        out.append(a.elapsed_time(b) * 1e3 / (uses * reps))
        del g
    return out


def rehome(torch, tensors):
    """Re-point bf16 device tensors, in place (Tensor.set_), at consecutive 128-byte aligned views
    of one device buffer, which is returned: the calls keep using the same tensor objects, and a
    single copy then moves all of them."""
    uniq = list({id(t): t for t in tensors}.values())
    sizes = [-(-t.numel() // 64) * 64 for t in uniq]
    arena = torch.zeros(sum(sizes), dtype=torch.bfloat16, device="cuda")
    off = 0
    for t, n in zip(uniq, sizes):
        assert t.dtype == torch.bfloat16 and t.is_contiguous()
        arena[off:off + t.numel()].copy_(t.reshape(-1))
        t.set_(arena.untyped_storage(), off, t.size(), t.stride())
        off += n
    return arena


def time_e2e(wl, steps, torch):
    """Through the public API with host buffers: every step copies all of its activations from
    pinned host memory in one copy, runs its calls, and copies all of its outputs back to pinned
    host memory in one copy, inside the timed region (captured in CUDA graphs, replayed).  The
    activations and outputs of the step's calls live in one device buffer each (rehome)."""
    st = torch.cuda.current_stream()
    hx = wl.x_arena.cpu().pin_memory()
    hy = torch.empty(wl.y_arena.shape, dtype=wl.y_arena.dtype).pin_memory()

    def body():
        wl.x_arena.copy_(hx, non_blocking=True)
        for c in wl.calls:
            c["fn"]()
        hy.copy_(wl.y_arena, non_blocking=True)
    graphs = [capture(torch, body) for _ in range(ROTATE)]
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for i in range(steps):
        graphs[i % len(graphs)].replay()
    b.record(st)
    b.synchronize()
    return a.elapsed_time(b), hx.numel() * hx.element_size(), hy.numel() * hy.element_size()


# ----------------------------------------------------------------------------- CPU oracle
_CASES = {}


def _case(key, fn):
    if key not in _CASES:
        _CASES[key] = fn()
    return _CASES[key]


def _chunks(n, parts, align=1):
    """[lo, hi) ranges covering range(n) in `parts` pieces whose bounds are multiples of align."""
    units = -(-n // align)
    edges = [min(n, align * (units * i // parts)) for i in range(parts + 1)]
    return [(a, b) for a, b in zip(edges[:-1], edges[1:]) if b > a]


def oracle_jobs(config, rows_per_call, parts):
    """The oracle's work on a bounded row sample of the workload, as independent jobs: each
    call's sampled output rows (MoE: intermediate columns) are cut into `parts` ranges, and a
    job runs the oracle on one range.  Returns (jobs, algorithmic bytes of the sampled work,
    description).  Inputs are generated here, outside any timing."""
    from oracle import formats as F
    from oracle import qlinear_oracle as Q
    jobs = []
    done = 0.0
    if config in ("c0", "c1", "n1"):
        shapes, Ms = {"c0": ([(512, 1024)], [1]), "c1": (C1_SHAPES, C1_MS), "n1": (C1_SHAPES, N1_MS)}[config]
        for (N, K) in shapes:
            c = _case(("int8", N, K, max(Ms)), lambda: synth.int8_case(max(Ms), N, K, seed=0))
            R = min(rows_per_call, N)
            for M in Ms:
                for a, b in _chunks(R, parts):
                    jobs.append(lambda c=c, M=M, a=a, b=b: Q.int8_w8a8(c["x"][:M], c["w"][a:b], c["w_s"][a:b]))
                done += bytes_int8(M, R, K)
        desc = f"INT8 oracle on the first {rows_per_call} output rows of each of the {len(shapes) * len(Ms)} calls"
    elif config in ("c2", "c4"):
        shapes, Ms = (C2_SHAPES, C2_MS) if config == "c2" else ([(17408, 5120)], [64])
        for (N, K) in shapes:
            c = _case(("fp8", N, K, max(Ms)), lambda: synth.fp8_block_case(max(Ms), N, K, seed=0))
            xv = F.bf16_to_f64(c["x"])
            R = min(rows_per_call, N)
            for M in Ms:
                for a, b in _chunks(R, parts, 128):  # whole 128-row scale blocks per job
                    if config == "c2":
                        jobs.append(lambda c=c, xv=xv, M=M, a=a, b=b, K=K:
                                    Q.fp8_block(xv[:M], c["w"][a:b], c["s"][a // 128:-(-b // 128)], K))
                    else:
                        jobs.append(lambda c=c, M=M, a=a, b=b, K=K:
                                    Q.fp8_block_act_quant(c["x"][:M], c["w"][a:b], c["s"][a // 128:-(-b // 128)], K))
                done += bytes_fp8(M, R, K)
        desc = (f"FP8 block oracle on the first {rows_per_call} output rows of each of the 8 calls" if config == "c2"
                else f"FP8 1x128-activation oracle on {rows_per_call} rows at M=64")
    elif config in ("c3", "n3", "n5"):
        E, H, I = 256, 4096, 2048
        wsub = _case(("moe8",), lambda: synth.moe_weights_only(8, H, I, seed=0))
        grouped = config == "n5"
        for M in ((32, 256) if grouped else (1, 9)):
            tk = _case(("tok", M), lambda: synth.moe_tokens(M, E, H, seed=0))
            C = min(rows_per_call, I)
            ids, _ = Q.route_topk(tk["logits"], 8)
            ids = np.asarray(ids) % 8  # 8 stand-in experts carry the sampled work
            for a, b in _chunks(C, parts):
                rows = np.concatenate([np.arange(a, b), I + np.arange(a, b)])
                w13, s13 = wsub["w13"][:, rows], wsub["s13"][:, rows]
                if grouped:
                    jobs.append(lambda tk=tk, ids=ids, w13=w13, s13=s13, n=b - a:
                                (Q.route_topk(tk["logits"], 8),
                                 Q.moe_gate_up_act_quant(tk["x"], ids, w13, s13, n)))
                else:
                    jobs.append(lambda tk=tk, ids=ids, w13=w13, s13=s13, n=b - a:
                                (Q.route_topk(tk["logits"], 8),
                                 Q.moe_gate_up(tk["x"], ids, w13, s13, n, limit=10.0 if config == "n3" else None)))
            done += len(np.unique(ids)) * 2 * C * (H // 2 + H // 32)
        desc = (f"{'grouped-MoE' if grouped else 'MoE'} oracle routing + {'quantised ' if grouped else ''}gate_up on "
                f"{rows_per_call} intermediate rows for M={'32 and M=256' if grouped else '1 and M=9'} (routing "
                "repeated in every job)")
    elif config == "n2":
        for (N, K) in N2_SHAPES:
            c = _case(("fp8c", N, K), lambda: synth.fp8_channel_case(16, N, K, seed=0))
            R = min(rows_per_call, N)
            for M in N2_MS:
                for a, b in _chunks(R, parts):
                    jobs.append(lambda c=c, M=M, a=a, b=b, K=K:
                                Q.fp8_channel(c["x"][:M], c["w"][a:b], "e4m3", c["w_s"][a:b], K))
                done += bytes_fp8c(M, R, K)
        desc = f"FP8 per-channel oracle on the first {rows_per_call} output rows of each of the 9 calls"
    elif config == "n4":
        for (N, K) in C2_SHAPES:
            c = _case(("bf16", N, K), lambda: synth.bf16_dense_case(16, N, K, seed=0))
            R = min(rows_per_call, N)
            for M in N4_MS:
                for a, b in _chunks(R, parts):
                    jobs.append(lambda c=c, M=M, a=a, b=b, K=K: Q.bf16_linear(c["x"][:M], c["w"][a:b], K))
                done += bytes_bf16(M, R, K)
        desc = f"BF16 oracle on the first {rows_per_call} output rows of each of the 6 calls"
    else:
        raise ValueError(config)
    return jobs, done, desc


def time_jobs(jobs, threads):
    """Seconds to run every job: in order on this thread, or spread over a thread pool (numpy
    releases the interpreter lock inside its array loops, so the jobs run in parallel)."""
    from concurrent.futures import ThreadPoolExecutor
    t = time.perf_counter()
    if threads <= 1:
        for j in jobs:
            j()
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda j: j(), jobs))
    return time.perf_counter() - t


def host_cores():
    return len(os.sched_getaffinity(0))


def cpu_baseline(config, budget_s=15.0):
    """Oracle throughput in the metric's unit on a bounded sample: single-threaded, then with
    the sampled rows split over one thread per host core (identical results: every output's
    sum is computed by one job).  `value` is the all-cores figure."""
    cores = host_cores()
    rows = 64
    jobs, b, desc = oracle_jobs(config, rows, 1)
    sec = time_jobs(jobs, 1)
    # grow the sample until it takes a few seconds single-threaded, within the budget
    while sec < budget_s / 4 and rows < 4096:
        rows *= 4
        jobs, b, desc = oracle_jobs(config, rows, 1)
        sec = time_jobs(jobs, 1)
    pjobs, _, _ = oracle_jobs(config, rows, cores)
    psec = time_jobs(pjobs, cores)
    return {"value": b / psec / 1e9, "unit": "GB/s", "cores": cores, "threads": cores, "kind": "oracle",
            "sample": desc + f"; rows split over {cores} threads",
            "seconds": round(psec, 3), "single_thread_value": b / sec / 1e9, "single_thread_seconds": round(sec, 3)}


# ----------------------------------------------------------------------------- main
def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(values, op="max"):
    return max(values) if op == "max" else sum(values)


def max_over_ranks(ms, dist=None, device="cpu"):
    """The slowest rank's timed region in ms (every rank gets it): the job is done when its last
    replica is.  `dist` is torch.distributed with a process group (nccl: device "cuda", gloo: "cpu")."""
    if dist is None:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step, steps, ms_max, world):
    """GB/s of the whole job: the bytes all replicas processed / the slowest replica's time."""
    return world * bytes_per_rank_step * steps / (ms_max * 1e-3) / 1e9


def run_reference(args, ws, rank):
    if rank != 0:
        return
    # the oracle as it stands, its sampled rows split over one thread per host core; the sample
    # grows (64 rows a call, x4, up to 4096) until a step takes its share of about 90 s for the
    # whole run, so the per-call work that does not scale with the rows (the activation
    # quantisation of every call) does not dominate a short step
    cores = host_cores()
    per_step = min(5.0, max(0.25, 90.0 / max(1, args.steps + args.warmup)))
    rows = 64
    jobs, bb, desc = oracle_jobs(args.config, rows, cores)
    while rows < 4096 and time_jobs(jobs, cores) < per_step / 4:
        rows *= 4
        jobs, bb, desc = oracle_jobs(args.config, rows, cores)
    for _ in range(args.warmup):
        time_jobs(jobs, cores)
    t = 0.0
    b = 0.0
    for _ in range(args.steps):
        t += time_jobs(jobs, cores)
        b += bb
    val = b / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPES[args.config],
            "data": "synthetic", "config": arm_config(args.config, ws),
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "threads": cores, "kind": "oracle",
                             "sample": desc + f" ({rows} rows per call per step, split over {cores} threads)"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c1", choices=sorted(BUILDERS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true", help="a few steps, no clocks/e2e/baseline (for ncu)")
    args = ap.parse_args()
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        if args.steps is None:
            args.steps = 20
        return run_reference(args, ws, rank)

    import torch
    if args.steps is None:
        args.steps = {"c0": 20000, "c1": 4000, "c2": 4000, "c3": 2000, "c4": 2000, "n1": 2000, "n2": 3000, "n3": 2000, "n5": 200,
                      "n4": 2000}[args.config]
    torch.cuda.set_device(local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    import skinny_gemm_dequant_gb300 as ql
    wl = BUILDERS[args.config](ql, torch)
    # the step's activations and outputs in one device buffer each (one copy per step end to end)
    wl.x_arena = rehome(torch, [t for c in wl.calls for t in c.get("inputs", [c["x"]])])
    wl.y_arena = rehome(torch, [c["y"] for c in wl.calls])
    for c in wl.calls:  # sizes the shared workspace before any capture
        c["fn"]()
    torch.cuda.synchronize()
    if args.profile:  # plain launches, no graphs (for ncu launch lists)
        for _ in range(args.warmup + args.steps):
            for c in wl.calls:
                c["fn"]()
        torch.cuda.synchronize()
        return
    graphs = step_graphs(wl, torch)
    for i in range(max(args.warmup, 3)):
        graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()

    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms_total = time_steps(graphs, args.steps, torch)
    torch.cuda.synchronize()
    ms_total = max_over_ranks(ms_total, pg, "cuda")
    ms_step = ms_total / args.steps
    peaks = load_peaks()
    value = job_throughput(wl.bytes_per_step, args.steps, ms_total, ws)  # GB/s, all ranks

    per_call = time_per_call(wl, torch)
    calls = []
    for c, us in zip(wl.calls, per_call):
        gbs = c["bytes"] / (us * 1e-6) / 1e9
        e = {"kind": c["kind"], "M": c["M"], "N": c["N"], "K": c["K"], "us": round(us, 3), "GBps": round(gbs, 1),
             "hbm_frac": round(gbs / peaks["hbm_gbs"], 4)}
        if "unique_experts" in c:
            e["unique_experts"] = c["unique_experts"]
        calls.append(e)
    tot_b = sum(c["bytes"] for c in wl.calls)
    tot_us = sum(per_call)
    # achieved: the step's algorithmic bytes over the step's device time (the timed region);
    # the per-call graphs (32 identical calls back to back) give frac_per_call beside it
    achieved = tot_b / (ms_step * 1e-3) / 1e9
    per_call_gbs = tot_b / (tot_us * 1e-6) / 1e9
    traffic = load_traffic(args.config)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                "frac_per_call": round(per_call_gbs / peaks["hbm_gbs"], 4),
                "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, copy)",
                "kernel": KERNEL_DESC[args.config],
                "algorithmic_bytes_per_step": tot_b}
    if args.config in ("c4", "n1"):
        fl = sum(c["flops"] for c in wl.calls)
        roofline["tensor_tflops"] = round(fl / (ms_step * 1e-3) / 1e12, 1)

    e2e_steps = max(3, min(args.steps // 10, 400))
    e2e_ms, h2d, d2h = time_e2e(wl, e2e_steps, torch)
    e2e_val = ws * wl.bytes_per_step / (e2e_ms / e2e_steps * 1e-3) / 1e9

    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": DTYPES[args.config], "data": "synthetic",
            "config": arm_config(args.config, ws),
            "us_per_call_mean": round(ms_step * 1e3 / len(wl.calls), 3),
            "calls": calls, "roofline": roofline,
            "e2e": {"value": round(e2e_val, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps},
            "gpu_launches": wl.launches_per_step * args.steps,
            "clocks": clk.summary()}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.config)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
