"""Benchmark of the decode-time MoE layer on GB300.

Workload (the 128-expert decode layer): H=2048, I=768, E=128, top_k=8,
BS=16, FP8 E4M3 experts with 128x128 fp32 block scales, bf16 activations
~N(0,1), router logits N(0,1) drawn fresh for every step; M=8 rows is the
headline, M in {1, 2, 4, 8} is reported as a sweep.  A step is one whole
layer call (top-k softmax -> align -> grouped gate+up -> grouped down ->
blend).  Steps rotate over 16 copies of the expert weights (16 x 604 MB), so
no step finds its weights in the 129 MB L2.

Timed regions (CUDA events on the launching stream, after W warm-up steps,
synchronize on both sides):
  * value:    K steps captured in one CUDA graph, replayed once;
  * roofline: the layer's dominant kernel alone (the tensor-core expert kernel
              on the FP8 decode shapes): K launches of moe_decode_experts in one
              CUDA graph, each on routing and alignment tables prepared in its
              own workspace beforehand, so only that kernel runs in the timed
              region; algorithmic bytes / mean duration per launch; DRAM
              traffic per launch from the committed ncu summary of the same
              kernel source, else null;
  * e2e:      K steps through the public API with host buffers: x and logits
              copied in from pinned memory, the output copied back, per step.
The CPU baseline is the oracle on a bounded sample of the same workload, on one
host core and on all of them (threads over the rows of the layer calls).

The line also carries `align_grid`: µs per moe_align call over the alignment
stress grid (n = 8·{1, 64, 1024, 4096}, E in {64, 256, 1024}, BS in {16, 64, 128},
uniform ids); `nvfp4_decode`: the NVFP4 layer with its FP8 shared expert at
M in {1, 8, 32} on the tensor-core kernel (the default) and on the fused CUDA-core
kernel, and at M=64 (the staged kernels);
`nvfp4_gate_up_tier`: the layer with NVFP4 gate and up and FP8 down at M=8;
`prefill`: M in {512, 2048} rows of the verify shape on the tensor cores.

The line also carries `router_logits`: the router matrix-vector product ahead of the
top-k (bf16 x times bf16 router weights) at the decode and verify widths, timed over
weight copies that keep it out of L2; and `hidden_in`: the headline decode layer given
x alone, its logits computed from router weights inside the layer call; and
`gated_shared`: the NVFP4 layer with an FP8 shared expert, ungated and gated.

The same line carries `verify_batch`: the M=128 verify batch (H=4096,
I=1536, E=256, top_k=8, BS=64, router logits with a Zipf(s=1.1) per-expert
bias, fresh noise every step) on the tensor-core path, K graph-replayed steps
over 2 weight copies of 4.8 GB, with its weight-stream GB/s against the
measured HBM peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
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

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
METRIC = ("MoE decode layer µs/tokens·s⁻¹ and weight-stream HBM GB/s "
          "(% peak), M=1..128")
N_COPIES = 16
NOMINAL_HBM_GBS = 8000.0
SEED = 1001


# The layer's dominant kernel on each path: its source file and the ncu
# summary that holds its DRAM traffic on the decode workload.
KERNELS = {
    "fused": ("decode_layer_kernel (one cooperative launch per layer call)", "decode_fused.cu",
              "decode_layer_kernel_fp8_decode.md"),
    "tc": ("verify_ffn_kernel (tcgen05; after moe_topk_softmax and moe_align)", "verify_tc.cu",
           "verify_ffn_kernel_fp8_decode.md"),
    "f4": ("nvfp4_ffn_kernel (tcgen05 kind::f16; after moe_topk_softmax and moe_align)",
           "nvfp4_tc.cu", "nvfp4_ffn_kernel_nvfp4_decode.md"),
}


def kernel_source_digest(src_name: str) -> str:
    """sha256 of a kernel's source file (ties a profile to a build)."""
    import hashlib
    src = os.path.join(HERE, "expert_routing_alignment_gb300", "csrc", src_name)
    with open(src, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def profiled_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of the path's layer kernel for `workload` from the
    committed ncu summary, if it was taken on the current kernel source."""
    _, src_name, prof = KERNELS[kernel]
    path = os.path.join(HERE, "profiles", prof)
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel source sha256") != kernel_source_digest(src_name):
        return None
    key = f"traffic bytes per launch ({workload})"
    return int(fields[key]) if key in fields else None


def measured_peaks() -> dict:
    path = os.path.join(HERE, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), source="measured")
    return dict(hbm_gbs=6800.0, source="fallback")


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["unsampled"], samples=0)
        return dict(sm_mhz=statistics.median(sm), sm_max_mhz=max(mx), reasons=sorted(reasons),
                    samples=len(sm))


# --------------------------------------------------------------------------
# workload
# --------------------------------------------------------------------------

def build_workload(M: int, steps: int, device: str, path: int = 0):
    import synth
    import expert_routing_alignment_gb300 as moe
    shape = synth.decode_fp8(M)
    base = synth.make_experts(shape.E, shape.H, shape.I, shape.fmt, SEED, device)
    copies = [base] + [_clone_experts(base) for _ in range(N_COPIES - 1)]
    x = synth.make_x(M, shape.H, SEED + 2, device)
    # fresh routing for every step: logits [steps, M, E]
    logits = torch.stack([synth.make_logits(M, shape.E, SEED + 100 + s, device)
                          for s in range(steps)])
    layers = [moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS,
                            routed=moe.Experts.from_synth(c), path=path) for c in copies]
    return shape, base, copies, layers, x, logits


def _clone_experts(d):
    import synth
    c = lambda p: synth.ProjData(p.fmt, p.rows, p.cols, p.codes.clone(), p.scale.clone(),
                                 None if p.glob is None else p.glob.clone())
    return synth.ExpertData(d.E, d.H, d.I, d.fmt, c(d.gate), c(d.up), c(d.down))


def active_expert_counts(logits: torch.Tensor, k: int) -> list:
    """Distinct experts each step routes to, read from the same logits."""
    ids = torch.topk(logits, k, dim=-1).indices
    return [int(torch.unique(ids[s]).numel()) for s in range(logits.shape[0])]


def layer_bytes(shape, base, n_active: int) -> int:
    per_expert = base.bytes_per_expert()
    n = shape.M * shape.top_k
    mt = shape.n + min(shape.n, shape.E) * (shape.BS - 1)
    tables = 4 * (mt + n + shape.E)
    return (n_active * per_expert + shape.M * shape.H * 2 * 2 + shape.M * shape.E * 4 + tables)


def expert_kernel_bytes(shape, base, n_active: int) -> int:
    """Algorithmic bytes of one launch of the expert kernel: the layer's bytes
    without the router logits (the routing and alignment ran before it)."""
    return layer_bytes(shape, base, n_active) - shape.M * shape.E * 4


def run_verify(moe, stream, K: int, W: int, peaks: dict) -> dict:
    """The M=128 verify batch: K steps in one CUDA graph, fresh logits each."""
    import synth
    shape = synth.verify_fp8(128)
    base = synth.make_experts(shape.E, shape.H, shape.I, shape.fmt, SEED + 4, "cuda")
    copies = [base, _clone_experts(base)]
    x = synth.make_x(shape.M, shape.H, SEED + 6, "cuda")
    logits = torch.stack([synth.make_logits(shape.M, shape.E, SEED + 300 + s, "cuda",
                                            shape.zipf_s, shape.zipf_scale) for s in range(K)])
    layers = [moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS,
                            routed=moe.Experts.from_synth(c)) for c in copies]
    ws = moe.alloc_workspace(layers[0], shape.M)
    out = torch.empty(shape.M, shape.H, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(stream):
        for s in range(W):
            moe.moe_decode_layer(layers[s % 2], x, out, ws, router_logits=logits[s % K])
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for s in range(K):
            moe.moe_decode_layer(layers[s % 2], x, out, ws, router_logits=logits[s])
    g.replay()
    stream.synchronize()
    times = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    ms = float(np.median(times))
    n_act = active_expert_counts(logits, shape.top_k)
    ids = torch.topk(logits, shape.top_k, dim=-1).indices
    max_rows = max(int(torch.bincount(ids[s].flatten(), minlength=shape.E).max())
                   for s in range(K))
    nbytes = float(np.mean([layer_bytes(shape, base, a) for a in n_act]))
    us = 1e3 * ms / K
    gbs = nbytes / (us * 1e-6) / 1e9
    launches = moe.moe_decode_layer_launches(layers[0], shape.M)
    res = dict(workload=shape.name, M=shape.M, H=shape.H, I=shape.I, E=shape.E,
               top_k=shape.top_k, BS=shape.BS, steps=K, us_per_layer=round(us, 3),
               tokens_per_s=round(shape.M / (us * 1e-6), 1), weight_stream_gbs=round(gbs, 1),
               pct_of_measured_hbm=round(100 * gbs / peaks["hbm_gbs"], 1),
               mean_active_experts=round(float(np.mean(n_act)), 2), max_rows_per_expert=max_rows,
               algorithmic_bytes_per_layer=int(nbytes), launches_per_layer=launches,
               path=("tensor cores: verify_ffn_kernel (tcgen05 kind::f8f6f4, TMEM accumulators)"
                     if launches == 3 else f"{launches} launches"),
               l2="2 weight copies of 4.8 GB; each step streams ~1.2 GB")
    del g, copies, layers, base, ws
    torch.cuda.empty_cache()
    return res


def run_router(moe, stream, peaks: dict) -> list:
    """The router logits (bf16 x times bf16 router weights) at the decode and
    verify widths: 64 calls in one CUDA graph, rotating over enough weight
    copies (256 MB in all) that no call finds its weights in L2."""
    res = []
    for M, H, E in ((8, 2048, 128), (128, 4096, 256)):
        g = torch.Generator(device="cuda").manual_seed(SEED + 7)
        x = torch.randn(M, H, generator=g, device="cuda").to(torch.bfloat16)
        per = E * H * 2
        n_w = max(2, (256 << 20) // per)
        Ws = (torch.randn(E, H, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
        Ws = Ws.unsqueeze(0).repeat(n_w, 1, 1).contiguous()
        out = torch.empty(M, E, dtype=torch.float32, device="cuda")
        calls = 64
        with torch.cuda.stream(stream):
            for i in range(8):
                moe.moe_router_logits(x, Ws[i % n_w], out)
        stream.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(calls):
                moe.moe_router_logits(x, Ws[(i * 7) % n_w], out)
        times = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                gr.replay()
                b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        us = 1e3 * float(np.median(times)) / calls
        nbytes = per + M * H * 2 + M * E * 4
        gbs = nbytes / (us * 1e-6) / 1e9
        res.append(dict(M=M, H=H, E=E, us_per_call=round(us, 3), bytes_per_call=nbytes,
                        gbs=round(gbs, 1), pct_of_measured_hbm=round(100 * gbs / peaks["hbm_gbs"], 1),
                        kernel="router_logits_kernel (k split over 256 threads, fixed-order sums)"))
        del gr, Ws
        torch.cuda.empty_cache()
    return res


def run_gated_shared(moe, stream, M: int, K: int, W: int, peaks: dict) -> dict:
    """The NVFP4 layer with an FP8 shared expert of inter 512 (M rows, fresh
    logits every step), its shared term ungated and gated by
    sigmoid(x . gate_w): K steps in one CUDA graph over 4 weight copies of
    340 MB."""
    import synth
    shape = synth.decode_nvfp4(M)
    base = synth.make_experts(shape.E, shape.H, shape.I, shape.fmt, SEED + 8, "cuda")
    sh = synth.make_experts(1, shape.H, shape.shared_I, synth.FMT_FP8, SEED + 9, "cuda")
    copies = [base] + [_clone_experts(base) for _ in range(3)]
    gate = synth.make_shared_gate(shape.H, SEED + 10, "cuda")
    x = synth.make_x(M, shape.H, SEED + 11, "cuda")
    logits = torch.stack([synth.make_logits(M, shape.E, SEED + 700 + s, "cuda")
                          for s in range(K)])
    shared = moe.Experts.from_synth(sh)
    res = dict(workload=shape.name, M=M, steps=K)
    for name, g in (("ungated", None), ("gated", gate)):
        layers = [moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS,
                                routed=moe.Experts.from_synth(c), shared=shared, shared_gate=g)
                  for c in copies]
        ws = moe.alloc_workspace(layers[0], M)
        out = torch.empty(M, shape.H, dtype=torch.bfloat16, device="cuda")
        with torch.cuda.stream(stream):
            for s in range(W):
                moe.moe_decode_layer(layers[s % 4], x, out, ws, router_logits=logits[s % K])
        stream.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for s in range(K):
                moe.moe_decode_layer(layers[s % 4], x, out, ws, router_logits=logits[s])
        gr.replay()
        stream.synchronize()
        times = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                gr.replay()
                b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        us = 1e3 * float(np.median(times)) / K
        res[f"us_per_layer_{name}"] = round(us, 3)
        res[f"launches_{name}"] = moe.moe_decode_layer_launches(layers[0], M)
        del gr, layers, ws
    n_act = active_expert_counts(logits, shape.top_k)
    nbytes = float(np.mean([layer_bytes(shape, base, a) for a in n_act])) + \
        sh.bytes_per_expert()
    res["algorithmic_bytes_per_layer"] = int(nbytes)
    res["weight_stream_gbs_gated"] = round(nbytes / (res["us_per_layer_gated"] * 1e-6) / 1e9, 1)
    res["pct_of_measured_hbm_gated"] = round(
        100 * res["weight_stream_gbs_gated"] / peaks["hbm_gbs"], 1)
    del copies, base, sh
    torch.cuda.empty_cache()
    return res


def run_hidden_in(moe, stream, M: int, K: int, W: int, path: int) -> dict:
    """The decode layer given x alone: the layer computes its logits from its
    router weights (one launch more).  K steps in one CUDA graph over the 16
    weight copies (each with its own router weights) and fresh x every step."""
    import synth
    shape, base, copies, layers, _, _ = build_workload(M, 1, "cuda", path)
    ws_r = [synth.make_router_weight(shape.E, shape.H, SEED + 500 + i, "cuda")
            for i in range(N_COPIES)]
    layers = [moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS, routed=lay.routed,
                            path=path, router_weight=w) for lay, w in zip(layers, ws_r)]
    xs = torch.stack([synth.make_x(M, shape.H, SEED + 600 + s, "cuda") for s in range(K)])
    ws = moe.alloc_workspace(layers[0], M)
    out = torch.empty(M, shape.H, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(stream):
        for s in range(W):
            moe.moe_decode_layer(layers[s % N_COPIES], xs[s % K], out, ws)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for s in range(K):
            moe.moe_decode_layer(layers[s % N_COPIES], xs[s], out, ws)
    g.replay()
    stream.synchronize()
    times = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    us = 1e3 * float(np.median(times)) / K
    res = dict(workload=shape.name, M=M, steps=K, us_per_layer=round(us, 3),
               tokens_per_s=round(M / (us * 1e-6), 1),
               launches_per_layer=moe.moe_decode_layer_launches(layers[0], M, 2),
               input="x alone; logits from bf16 router weights [E, H], one set per weight copy")
    del g, copies, layers, base, ws
    torch.cuda.empty_cache()
    return res


def _graph_ms(stream, K: int, body) -> float:
    """Median over 3 replays of a CUDA graph of body(s) for s < K, in ms per
    step (one untimed replay first)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for s in range(K):
            body(s)
    g.replay()
    stream.synchronize()
    times = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) / K)
    del g
    return float(np.median(times))


def run_nvfp4_decode(moe, stream, K: int, W: int, peaks: dict) -> dict:
    """The NVFP4 layer with its FP8 shared expert (inter 512) at M in {1, 8, 32}
    and 64: K graph-replayed steps over 4 weight copies of 340 MB, fresh
    logits every step, ungated.  M <= 32 runs both on the NVFP4 tensor-core
    kernel (the shared expert inside it) and on the fused CUDA-core kernel,
    each row naming its path and whether the layer's default takes it; M=64
    the staged CUDA-core kernels."""
    import synth
    shape0 = synth.decode_nvfp4(1)
    base = synth.make_experts(shape0.E, shape0.H, shape0.I, shape0.fmt, SEED + 8, "cuda")
    sh = synth.make_experts(1, shape0.H, shape0.shared_I, synth.FMT_FP8, SEED + 9, "cuda")
    copies = [base] + [_clone_experts(base) for _ in range(3)]
    shared = moe.Experts.from_synth(sh)

    def layers_for(path):
        return [moe.LayerDesc(top_k=shape0.top_k, block_size=shape0.BS,
                              routed=moe.Experts.from_synth(c), shared=shared, path=path)
                for c in copies]

    by_path = {"tc": layers_for(moe.PATH_TC), "fused": layers_for(moe.PATH_SIMT),
               "auto": layers_for(moe.PATH_AUTO)}
    rows = []
    for M in (1, 8, 32, 64):
        shape = synth.decode_nvfp4(M)
        x = synth.make_x(M, shape.H, SEED + 11, "cuda")
        logits = torch.stack([synth.make_logits(M, shape.E, SEED + 800 + s, "cuda")
                              for s in range(K)])
        n_act = active_expert_counts(logits, shape.top_k)
        nbytes = float(np.mean([layer_bytes(shape, base, a) for a in n_act])) + \
            sh.bytes_per_expert()
        auto_launches = moe.moe_decode_layer_launches(by_path["auto"][0], M)
        for name in (("tc", "fused") if M <= 32 else ("auto",)):
            layers = by_path[name]
            ws = moe.alloc_workspace(layers[0], M)
            out = torch.empty(M, shape.H, dtype=torch.bfloat16, device="cuda")
            with torch.cuda.stream(stream):
                for s in range(W):
                    moe.moe_decode_layer(layers[s % 4], x, out, ws, router_logits=logits[s % K])
            stream.synchronize()
            ms = _graph_ms(stream, K, lambda s: moe.moe_decode_layer(
                layers[s % 4], x, out, ws, router_logits=logits[s]))
            us = 1e3 * ms
            gbs = nbytes / (us * 1e-6) / 1e9
            launches = moe.moe_decode_layer_launches(layers[0], M)
            half = {}
            if name == "tc":
                # the expert half alone on the tables the last call left: the
                # x-table launch and the tensor-core kernel (weights rotate)
                ms_e = _graph_ms(stream, K, lambda s: moe.moe_decode_experts(
                    layers[s % 4], x, out, ws))
                e_bytes = nbytes - M * shape.E * 4
                half = dict(expert_half_us=round(1e3 * ms_e, 3),
                            expert_half_pct_of_measured_hbm=round(
                                100 * e_bytes / (ms_e * 1e-3) / 1e9 / peaks["hbm_gbs"], 1),
                            kernel_traffic_bytes_per_launch=profiled_traffic(shape.name, "f4"))
            rows.append(dict(M=M, path=name if name != "auto" else "staged",
                             default=name == "auto" or launches == auto_launches,
                             us_per_layer=round(us, 3), tokens_per_s=round(M / (us * 1e-6), 1),
                             weight_stream_gbs=round(gbs, 1),
                             pct_of_measured_hbm=round(100 * gbs / peaks["hbm_gbs"], 1),
                             launches_per_layer=launches,
                             mean_active_experts=round(float(np.mean(n_act)), 2),
                             algorithmic_bytes_per_layer=int(nbytes), **half))
            del ws
    del copies, by_path, base, sh
    torch.cuda.empty_cache()
    return dict(workload="decode_h2048_i768_e128_k8_nvfp4_shared512", steps=K, rows=rows)


def run_nvfp4_gate_up(moe, stream, M: int, K: int, W: int, peaks: dict) -> dict:
    """The nvfp4-gate-up tier (NVFP4 gate and up, FP8 down, FP8 shared expert
    of inter 512) at M rows: K graph-replayed steps over 4 weight copies,
    fresh logits every step (the staged CUDA-core kernels)."""
    import synth
    shape = synth.decode_nvfp4_gate_up(M)
    base = synth.make_experts(shape.E, shape.H, shape.I, shape.fmt, SEED + 20, "cuda")
    sh = synth.make_experts(1, shape.H, shape.shared_I, synth.FMT_FP8, SEED + 21, "cuda")
    copies = [base] + [_clone_experts(base) for _ in range(3)]
    shared = moe.Experts.from_synth(sh)
    layers = [moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS,
                            routed=moe.Experts.from_synth(c), shared=shared) for c in copies]
    x = synth.make_x(M, shape.H, SEED + 22, "cuda")
    logits = torch.stack([synth.make_logits(M, shape.E, SEED + 900 + s, "cuda")
                          for s in range(K)])
    ws = moe.alloc_workspace(layers[0], M)
    out = torch.empty(M, shape.H, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(stream):
        for s in range(W):
            moe.moe_decode_layer(layers[s % 4], x, out, ws, router_logits=logits[s % K])
    stream.synchronize()
    ms = _graph_ms(stream, K, lambda s: moe.moe_decode_layer(layers[s % 4], x, out, ws,
                                                             router_logits=logits[s]))
    n_act = active_expert_counts(logits, shape.top_k)
    nbytes = float(np.mean([layer_bytes(shape, base, a) for a in n_act])) + sh.bytes_per_expert()
    us = 1e3 * ms
    gbs = nbytes / (us * 1e-6) / 1e9
    res = dict(workload=shape.name, M=M, steps=K, us_per_layer=round(us, 3),
               tokens_per_s=round(M / (us * 1e-6), 1), weight_stream_gbs=round(gbs, 1),
               pct_of_measured_hbm=round(100 * gbs / peaks["hbm_gbs"], 1),
               launches_per_layer=moe.moe_decode_layer_launches(layers[0], M),
               algorithmic_bytes_per_layer=int(nbytes))
    del copies, layers, base, sh, ws
    torch.cuda.empty_cache()
    return res


def run_prefill(moe, stream, M: int, K: int, W: int, peaks: dict) -> dict:
    """A prefill-sized batch on the tensor-core path: M rows of the verify
    shape (H=4096, I=1536, E=256, k=8, BS=64, uniform N(0,1) logits, fresh
    every step), K graph-replayed steps over 2 weight copies of 4.8 GB.
    Reported as tokens/s, effective TFLOP/s (2 n 3 H I per layer, the
    products the layer asks for) and weight-stream GB/s."""
    import synth
    shape = synth.LayerShape(f"prefill_h4096_i1536_e256_k8_fp8_m{M}", M, 4096, 1536, 256, 8, 64,
                             synth.FMT_FP8)
    base = synth.make_experts(shape.E, shape.H, shape.I, shape.fmt, SEED + 30, "cuda")
    copies = [base, _clone_experts(base)]
    layers = [moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS,
                            routed=moe.Experts.from_synth(c)) for c in copies]
    x = synth.make_x(M, shape.H, SEED + 31, "cuda")
    logits = torch.stack([synth.make_logits(M, shape.E, SEED + 1000 + s, "cuda")
                          for s in range(K)])
    ws = moe.alloc_workspace(layers[0], M)
    out = torch.empty(M, shape.H, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(stream):
        for s in range(W):
            moe.moe_decode_layer(layers[s % 2], x, out, ws, router_logits=logits[s % K])
    stream.synchronize()
    ms = _graph_ms(stream, K, lambda s: moe.moe_decode_layer(layers[s % 2], x, out, ws,
                                                             router_logits=logits[s]))
    n_act = active_expert_counts(logits, shape.top_k)
    nbytes = float(np.mean([layer_bytes(shape, base, a) for a in n_act]))
    us = 1e3 * ms
    flops = 2.0 * shape.n * 3 * shape.H * shape.I
    res = dict(workload=shape.name, M=M, steps=K, us_per_layer=round(us, 3),
               tokens_per_s=round(M / (us * 1e-6), 1),
               effective_tflops=round(flops / (us * 1e-6) / 1e12, 1),
               weight_stream_gbs=round(nbytes / (us * 1e-6) / 1e9, 1),
               mean_active_experts=round(float(np.mean(n_act)), 2),
               launches_per_layer=moe.moe_decode_layer_launches(layers[0], M),
               path="tensor cores: verify_ffn_kernel")
    del copies, layers, base, ws
    torch.cuda.empty_cache()
    return res


def run_align_grid(moe, stream) -> list:
    """µs per moe_align call over the alignment stress grid (uniform int64
    ids): 32 calls in one CUDA graph, rotating over 4 id sets."""
    import synth
    res = []
    for M in (1, 64, 1024, 4096):
        n = 8 * M
        for E in (64, 256, 1024):
            for BS in (16, 64, 128):
                ids = [torch.from_numpy(synth.align_ids(n, E, "uniform", SEED + 40 + j)).cuda()
                       for j in range(4)]
                outs = [moe.alloc_align_outputs(n, E, BS) for _ in range(4)]
                for j in range(4):
                    moe.moe_align(ids[j], E, BS, out=outs[j], stream=stream)
                stream.synchronize()
                ms = _graph_ms(stream, 32, lambda s: moe.moe_align(ids[s % 4], E, BS,
                                                                   out=outs[s % 4],
                                                                   stream=stream))
                res.append(dict(n=n, E=E, BS=BS, us_per_align=round(1e3 * ms, 3)))
    return res


# --------------------------------------------------------------------------
# timed regions
# --------------------------------------------------------------------------

def time_graph(moe, layers, x, logits, out, ws, K: int, W: int, stream,
               busy: bool = False) -> float:
    """Milliseconds for K layer calls replayed from one CUDA graph."""
    with torch.cuda.stream(stream):
        for s in range(W):
            moe.moe_decode_layer(layers[s % N_COPIES], x, out, ws, router_logits=logits[s % K])
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for s in range(K):
            moe.moe_decode_layer(layers[s % N_COPIES], x, out, ws, router_logits=logits[s])
    t0 = time.perf_counter()
    g.replay()                        # one untimed replay (first-touch of the graph)
    stream.synchronize()
    # untimed replays before and after keep the GPU loaded for ~0.5 s around
    # the timed one, so that sampled clocks describe the timed region
    once = max(time.perf_counter() - t0, 1e-4)
    pad = int(min(2000, max(1, 0.25 / once)))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if torch.distributed.is_initialized():
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(pad if busy else 0):
            g.replay()
        start.record(stream)
        g.replay()
        end.record(stream)
        for _ in range(pad if busy else 0):
            g.replay()
    end.synchronize()
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def time_expert_kernel(moe, layers, x, logits, out, K: int, W: int, stream):
    """Mean duration (ms) of one launch of the layer's expert kernel alone.

    Each of the N_COPIES weight copies gets its own workspace, and one layer
    call on it (untimed) leaves that step's routing and alignment tables
    there; then K launches of moe_decode_experts (the expert half of the layer:
    one kernel on the tensor-core and fused paths) run back to back from one
    CUDA graph, launch s on copy s % N_COPIES with its tables, and the graph is
    timed with events on the launching stream."""
    M = x.shape[0]
    n = min(N_COPIES, K)
    wss = [moe.alloc_workspace(layers[c], M) for c in range(n)]
    with torch.cuda.stream(stream):
        for c in range(n):
            moe.moe_decode_layer(layers[c], x, out, wss[c], router_logits=logits[c % K])
        for s in range(W):
            moe.moe_decode_experts(layers[s % n], x, out, wss[s % n])
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for s in range(K):
            moe.moe_decode_experts(layers[s % n], x, out, wss[s % n])
    g.replay()
    stream.synchronize()
    times = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) / K)
    del g, wss
    return float(np.median(times))


def time_e2e(moe, shape, layer, x_host, logits_host, out_host, ws, K: int, W: int, stream):
    """K steps through the public API from pinned host buffers."""
    x_dev = torch.empty(shape.M, shape.H, dtype=torch.bfloat16, device="cuda")
    lg_dev = torch.empty(shape.M, shape.E, dtype=torch.float32, device="cuda")
    out_dev = torch.empty(shape.M, shape.H, dtype=torch.bfloat16, device="cuda")

    def step(s):
        x_dev.copy_(x_host, non_blocking=True)
        lg_dev.copy_(logits_host[s % logits_host.shape[0]], non_blocking=True)
        moe.moe_decode_layer(layer, x_dev, out_dev, ws, router_logits=lg_dev)
        out_host.copy_(out_dev, non_blocking=True)

    with torch.cuda.stream(stream):
        for s in range(W):
            step(s)
    stream.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for s in range(K):
            step(s)
        end.record(stream)
    end.synchronize()
    h2d = x_dev.numel() * 2 + lg_dev.numel() * 4
    d2h = out_dev.numel() * 2
    return start.elapsed_time(end), h2d, d2h


def oracle_experts(d):
    """synth expert data -> the oracle's host structures (each projection in
    its own format)."""
    import oracle
    P = lambda p: oracle.Proj(oracle.FMT_FP8_B128 if p.fmt == "fp8" else oracle.FMT_NVFP4_G16,
                              p.rows, p.cols, p.codes.cpu().numpy(), p.scale.cpu().numpy(),
                              None if p.glob is None else p.glob.cpu().numpy())
    return oracle.Experts(d.E, d.H, d.I, P(d.gate), P(d.up), P(d.down))


def _oracle_rows(X, xb, lg, M: int, top_k: int, BS: int, threads: int, budget_s: float,
                 max_calls: int):
    """Whole layer calls of M rows on the oracle, `threads` host threads at a
    time, for about budget_s seconds (at least one call).  A call's rows go to
    the threads one row each (a row's output depends only on its own x and
    logits, so each is the oracle's layer on that row alone); ctypes drops
    the interpreter lock during the C call, so the threads run in parallel.
    Returns (calls, seconds)."""
    import concurrent.futures as cf
    import oracle
    t0 = time.perf_counter()
    calls = 0
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        while True:
            lgc = lg[calls % len(lg)]
            if threads == 1:
                oracle.moe_layer(X, None, xb, M, top_k, BS, logits=lgc)
            else:
                list(ex.map(lambda r: oracle.moe_layer(X, None, xb[r:r + 1], 1, top_k, BS,
                                                       logits=lgc[r:r + 1]), range(M)))
            calls += 1
            if time.perf_counter() - t0 > budget_s or calls >= max_calls:
                break
    return calls, time.perf_counter() - t0


def cpu_baseline(shape, base, x, logits, budget_s: float = 8.0) -> dict:
    """The oracle on the host cores: whole layer calls of the workload at M
    rows, as many as fit in the time budget, on all host cores (threads over
    the rows) and on one core."""
    X = oracle_experts(base)
    xb = x.cpu().view(torch.int16).numpy().view(np.uint16)
    lg = logits.cpu().numpy()
    threads = max(1, min(os.cpu_count() or 1, shape.M))
    calls, dt = _oracle_rows(X, xb, lg, shape.M, shape.top_k, shape.BS, threads, budget_s,
                             1 << 20)
    calls1, dt1 = _oracle_rows(X, xb, lg, shape.M, shape.top_k, shape.BS, 1, budget_s, 1 << 20)
    return dict(value=shape.M * calls / dt, unit="tokens/s", cores=threads, kind="oracle",
                host_cpus=os.cpu_count(),
                sample=f"{calls} whole layer calls of {shape.name} ({shape.M} rows each, one "
                       f"row per thread on {threads} threads), C oracle in double, {dt:.1f} s",
                single_thread=dict(value=shape.M * calls1 / dt1, unit="tokens/s", cores=1,
                                   sample=f"{calls1} whole layer calls on one thread, "
                                          f"{dt1:.1f} s"))


def workload_config(shape, world: int) -> dict:
    """The `config` object of the headline line (both arms carry the same)."""
    return dict(workload=shape.name, M=shape.M, H=shape.H, I=shape.I, E=shape.E,
                top_k=shape.top_k, BS=shape.BS, weights="fp8_e4m3 128x128 fp32 block scales",
                routing="fresh N(0,1) logits every step",
                l2="inputs larger than L2: steps rotate over 16 weight copies of 604 MB",
                parallelism=f"replicas x{world}")


# --------------------------------------------------------------------------
# arms
# --------------------------------------------------------------------------

def run_reference(args, rank: int, world: int):
    """The oracle as the reference arm: each step is one whole layer call of the
    headline workload (all M rows) on the host cores, one row per thread."""
    if rank != 0:
        return
    import synth
    M = args.m
    shape = synth.decode_fp8(M)
    base = synth.make_experts(shape.E, shape.H, shape.I, shape.fmt, SEED, "cpu")
    X = oracle_experts(base)
    x = synth.make_x(M, shape.H, SEED + 2, "cpu")
    xb = x.contiguous().view(torch.int16).numpy().view(np.uint16)
    threads = max(1, min(os.cpu_count() or 1, M))
    lg_w = np.stack([synth.make_logits(M, shape.E, SEED + 100 + s, "cpu").numpy()
                     for s in range(args.warmup)])
    _oracle_rows(X, xb, lg_w, M, shape.top_k, shape.BS, threads, 0.0, args.warmup)
    lgs = np.stack([synth.make_logits(M, shape.E, SEED + 100 + s, "cpu").numpy()
                    for s in range(args.steps)])
    calls, dt = _oracle_rows(X, xb, lgs, M, shape.top_k, shape.BS, threads, float("inf"),
                             args.steps)
    value = M * calls / dt
    line = dict(
        impl="reference", metric=METRIC, value=value, unit="tokens/s", n_gpus=world,
        steps=args.steps, warmup=args.warmup, ms_per_step=1e3 * dt / args.steps,
        higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
        config=workload_config(shape, world),
        cpu_baseline=dict(value=value, unit="tokens/s", cores=threads, kind="oracle",
                          host_cpus=os.cpu_count(),
                          sample=f"each step: one whole layer call of {shape.name} ({M} rows, "
                                 f"one row per thread on {threads} threads), C oracle in "
                                 f"double"),
        e2e=dict(value=value, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def run_profile_verify(args):
    """A small case of the verify-batch kernel for ncu: the verify shape with
    E=64 experts (1.2 GB of weights, ~40 active per step, ~0.75 GB streamed
    per layer, above the L2), W+K direct layer calls, no graph."""
    import dataclasses
    import synth
    import expert_routing_alignment_gb300 as moe
    moe.load()
    shape = dataclasses.replace(synth.verify_fp8(128), E=64,
                                name="verify_h4096_i1536_e64_k8_fp8_zipf_m128")
    base = synth.make_experts(shape.E, shape.H, shape.I, shape.fmt, SEED + 4, "cuda")
    x = synth.make_x(shape.M, shape.H, SEED + 6, "cuda")
    layer = moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS, routed=moe.Experts.from_synth(base))
    ws = moe.alloc_workspace(layer, shape.M)
    out = torch.empty(shape.M, shape.H, dtype=torch.bfloat16, device="cuda")
    for s in range(args.warmup + args.steps):
        lg = synth.make_logits(shape.M, shape.E, SEED + 300 + s, "cuda", shape.zipf_s,
                               shape.zipf_scale)
        moe.moe_decode_layer(layer, x, out, ws, router_logits=lg)
    torch.cuda.synchronize()
    print(json.dumps(dict(profile_verify=shape.name, steps=args.warmup + args.steps)), flush=True)


def run_profile_nvfp4(args):
    """Profiler workload for the NVFP4 tensor-core kernel: the NVFP4 layer
    with its FP8 shared expert at M = args.m rows, W + K eager calls rotating
    over 2 weight copies (680 MB, beyond L2)."""
    import expert_routing_alignment_gb300 as moe
    import synth
    moe.load()
    shape = synth.decode_nvfp4(args.m)
    base = synth.make_experts(shape.E, shape.H, shape.I, shape.fmt, SEED + 8, "cuda")
    sh = synth.make_experts(1, shape.H, shape.shared_I, synth.FMT_FP8, SEED + 9, "cuda")
    copies = [base, _clone_experts(base)]
    shared = moe.Experts.from_synth(sh)
    layers = [moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS, path=moe.PATH_TC,
                            routed=moe.Experts.from_synth(c), shared=shared) for c in copies]
    x = synth.make_x(args.m, shape.H, SEED + 11, "cuda")
    ws = moe.alloc_workspace(layers[0], args.m)
    out = torch.empty(args.m, shape.H, dtype=torch.bfloat16, device="cuda")
    n = args.warmup + args.steps
    for s in range(n):
        logits = synth.make_logits(args.m, shape.E, SEED + 800 + s, "cuda")
        moe.moe_decode_layer(layers[s % 2], x, out, ws, router_logits=logits)
    torch.cuda.synchronize()
    print(json.dumps(dict(profile_nvfp4=True, M=args.m, calls=n)), flush=True)


def run_profile_router(args):
    """The router logits kernel for ncu: W+K direct calls at the decode width
    (M=8, H=2048, E=128) and then at the verify width (M=128, H=4096, E=256)."""
    import synth
    import expert_routing_alignment_gb300 as moe
    moe.load()
    for M, H, E in ((8, 2048, 128), (128, 4096, 256)):
        x = synth.make_x(M, H, SEED + 12, "cuda")
        Wr = synth.make_router_weight(E, H, SEED + 13, "cuda")
        out = torch.empty(M, E, dtype=torch.float32, device="cuda")
        for _ in range(args.warmup + args.steps):
            moe.moe_router_logits(x, Wr, out)
    torch.cuda.synchronize()
    print(json.dumps(dict(profile_router=True, calls=2 * (args.warmup + args.steps))), flush=True)


def run_gpu(args, rank: int, world: int):
    import expert_routing_alignment_gb300 as moe
    moe.load()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    K, W = args.steps, args.warmup
    peaks = measured_peaks()
    results = {}
    sweep = []
    for M in args.sweep:
        shape, base, copies, layers, x, logits = build_workload(M, K, "cuda", args.path)
        ws = moe.alloc_workspace(layers[0], M)
        out = torch.empty(M, shape.H, dtype=torch.bfloat16, device="cuda")
        head = M == args.m and not args.profile
        sampler = ClockSampler(local)
        if head:
            sampler.__enter__()
        ms = time_graph(moe, layers, x, logits, out, ws, K, W, stream, busy=head)
        if head:
            sampler.__exit__(None, None, None)
        n_act = active_expert_counts(logits, shape.top_k)
        nbytes = float(np.mean([layer_bytes(shape, base, a) for a in n_act]))
        us = 1e3 * ms / K
        gbs = nbytes / (us * 1e-6) / 1e9
        sweep.append(dict(M=M, us_per_layer=round(us, 3), tokens_per_s=round(M / (us * 1e-6), 1),
                          weight_stream_gbs=round(gbs, 1),
                          pct_of_measured_hbm=round(100 * gbs / peaks["hbm_gbs"], 1),
                          pct_of_8tbs=round(100 * gbs / NOMINAL_HBM_GBS, 1),
                          mean_active_experts=round(float(np.mean(n_act)), 2)))
        if head:
            dk_ms = time_expert_kernel(moe, layers, x, logits, out, K, W, stream)
            n_kern = min(N_COPIES, K)
            kbytes = float(np.mean([expert_kernel_bytes(shape, base, a)
                                    for a in active_expert_counts(logits[:n_kern],
                                                                  shape.top_k)]))
            launches = moe.moe_decode_layer_launches(layers[0], M)
            x_host = x.cpu().pin_memory()
            lg_host = logits.cpu().pin_memory()
            out_host = torch.empty(M, shape.H, dtype=torch.bfloat16).pin_memory()
            e2e_ms, h2d, d2h = time_e2e(moe, shape, layers[0], x_host, lg_host, out_host, ws,
                                        K, W, stream)
            results = dict(shape=shape, base=base, x=x, logits=logits, ms=ms, us=us, gbs=gbs,
                           nbytes=nbytes, dk_ms=dk_ms, kbytes=kbytes, launches=launches,
                           e2e_ms=e2e_ms,
                           kernel="fused" if launches == 1 else "tc",
                           h2d=h2d, d2h=d2h, clocks=sampler.summary())
        del copies, layers, base, ws
        torch.cuda.empty_cache()

    if args.profile:
        if rank == 0:
            print(json.dumps(dict(profile=True, sweep=sweep)), flush=True)
        return
    verify = None if args.no_verify else run_verify(moe, stream, min(K, 16), 3, peaks)
    router = None if args.no_verify else run_router(moe, stream, peaks)
    hidden_in = None if args.no_verify else run_hidden_in(moe, stream, args.m, K, W, args.path)
    gated = None if args.no_verify else run_gated_shared(moe, stream, 8, min(K, 16), 3, peaks)
    nvfp4 = None if args.no_verify else run_nvfp4_decode(moe, stream, min(K, 16), 3, peaks)
    align_grid = None if args.no_verify else run_align_grid(moe, stream)
    gate_up_tier = None if args.no_verify else run_nvfp4_gate_up(moe, stream, 8, min(K, 16), 3,
                                                                   peaks)
    prefill = None if args.no_verify else [run_prefill(moe, stream, m, 8, 3, peaks)
                                           for m in (512, 2048)]
    # max over ranks
    ms_t = torch.tensor([results["ms"]], device="cuda")
    if world > 1:
        torch.distributed.all_reduce(ms_t, op=torch.distributed.ReduceOp.MAX)
    ms_max = float(ms_t.item())
    if rank != 0:
        return
    r = results
    shape = r["shape"]
    value = world * shape.M * K / (ms_max * 1e-3)
    dk_achieved = r["kbytes"] / (r["dk_ms"] * 1e-3) / 1e9
    line = dict(
        metric=METRIC, value=value, unit="tokens/s", n_gpus=world, steps=K, warmup=W,
        ms_per_step=ms_max / K, higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype=("fp8_e4m3 weights, f16 x f16 -> f32 mma" if r["kernel"] == "fused" else
               "fp8_e4m3 weights x e4m3 activation terms -> f32 (tcgen05 kind::f8f6f4)"),
        data="synthetic",
        config=workload_config(shape, world),
        us_per_layer=round(r["us"], 3), weight_stream_gbs=round(r["gbs"], 1),
        pct_of_measured_hbm=round(100 * r["gbs"] / peaks["hbm_gbs"], 1),
        pct_of_8tbs=round(100 * r["gbs"] / NOMINAL_HBM_GBS, 1),
        algorithmic_bytes_per_layer=int(r["nbytes"]),
        sweep=sweep,
        verify_batch=verify,
        router_logits=router,
        hidden_in=hidden_in,
        gated_shared=gated,
        nvfp4_decode=nvfp4,
        nvfp4_gate_up_tier=gate_up_tier,
        prefill=prefill,
        align_grid=align_grid,
        roofline=dict(bound="hbm",
                      kernel=KERNELS[r["kernel"]][0],
                      achieved=round(dk_achieved, 1),
                      peak=peaks["hbm_gbs"], peak_source=f"{peaks['source']} copy bandwidth",
                      unit="GB/s", frac=round(dk_achieved / peaks["hbm_gbs"], 4),
                      bytes_per_launch=int(r["kbytes"]), us_per_launch=round(1e3 * r["dk_ms"], 3),
                      timed="the kernel alone: K launches of moe_decode_experts from one CUDA "
                            "graph on prepared tables, CUDA events on the launching stream",
                      traffic=profiled_traffic(shape.name, r["kernel"])),
        e2e=dict(value=shape.M * K / (r["e2e_ms"] * 1e-3), unit="tokens/s",
                 h2d_bytes_per_step=r["h2d"], d2h_bytes_per_step=r["d2h"]),
        gpu_launches=r["launches"] * K,
        clocks=r["clocks"])
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(shape, r["base"], r["x"], r["logits"])
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--m", type=int, default=8, help="rows of the headline workload")
    ap.add_argument("--sweep", type=int, nargs="*", default=[1, 2, 4, 8])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-verify", action="store_true",
                    help="skip the M=128 verify-batch measurement")
    ap.add_argument("--profile-verify", action="store_true",
                    help="only run a small case of the verify-batch kernel (for ncu)")
    ap.add_argument("--profile-nvfp4", action="store_true",
                    help="profiler workload: the NVFP4 layer (tensor-core kernel) at --m rows")
    ap.add_argument("--profile-router", action="store_true",
                    help="only run the router logits kernel at two widths (for ncu)")
    ap.add_argument("--path", type=int, default=0,
                    help="MOE_PATH_* of the decode workloads (0 auto: tensor cores for FP8; "
                         "1: the CUDA cores' fused kernel)")
    ap.add_argument("--copies", type=int, default=16,
                    help="weight copies the steps rotate over (16 keeps weights out of L2)")
    ap.add_argument("--profile", action="store_true",
                    help="only the graph region, without the clock window, the dominant-kernel "
                         "region, e2e and the CPU baseline (for profiler runs)")
    args = ap.parse_args()
    if args.m not in args.sweep:
        args.sweep.append(args.m)
    global N_COPIES
    N_COPIES = max(1, args.copies)
    args.warmup = max(args.warmup, 3)
    sys.path.insert(0, HERE)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("nccl" if args.impl == "gb300" else "gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.profile_verify:
            run_profile_verify(args)
        elif args.profile_router:
            run_profile_router(args)
        elif args.profile_nvfp4:
            run_profile_nvfp4(args)
        else:
            run_gpu(args, rank, world)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
