"""Shared test helpers: hand synthetic data to the oracle, and an independent
float64 PyTorch restatement of the layer built from library routines (torch's
float8 decoding, matmul, silu, topk, softmax) that pins the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

E2M1_TABLE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                       -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def oracle_proj(p: synth.ProjData) -> oracle.Proj:
    fmt = oracle.FMT_FP8_B128 if p.fmt == synth.FMT_FP8 else oracle.FMT_NVFP4_G16
    return oracle.Proj(fmt, p.rows, p.cols, p.codes.cpu().numpy(), p.scale.cpu().numpy(),
                       None if p.glob is None else p.glob.cpu().numpy())


def oracle_experts(d: synth.ExpertData) -> oracle.Experts:
    return oracle.Experts(d.E, d.H, d.I, oracle_proj(d.gate), oracle_proj(d.up),
                          oracle_proj(d.down))


def subset_experts(d: synth.ExpertData, ids) -> synth.ExpertData:
    """The experts `ids` (in that order) as a smaller expert set on the CPU."""
    idx = torch.as_tensor(list(ids), dtype=torch.long)

    def sub(p: synth.ProjData) -> synth.ProjData:
        i = idx.to(p.codes.device)
        return synth.ProjData(p.fmt, p.rows, p.cols, p.codes[i].cpu(), p.scale[i].cpu(),
                              None if p.glob is None else p.glob[i].cpu())

    return synth.ExpertData(len(idx), d.H, d.I, d.fmt, sub(d.gate), sub(d.up), sub(d.down))


# --------------------------------------------------------------------------
# torch float64 restatement (library routines)
# --------------------------------------------------------------------------

def torch_dequant(p: synth.ProjData, e: int) -> torch.Tensor:
    if p.fmt == synth.FMT_FP8:
        q = p.codes[e].cpu().view(torch.float8_e4m3fn).to(torch.float64)
        s = p.scale[e].cpu().to(torch.float64)
        s = s.repeat_interleave(128, 0).repeat_interleave(128, 1)
        return q * s[: q.shape[0], : q.shape[1]]
    packed = p.codes[e].cpu().numpy()
    codes = np.empty((packed.shape[0], packed.shape[1] * 2), np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    v = torch.from_numpy(E2M1_TABLE[codes])
    s16 = p.scale[e].cpu().view(torch.float8_e4m3fn).to(torch.float64)
    return v * s16.repeat_interleave(16, 1) * float(p.glob[e])


def torch_ffn(d: synth.ExpertData, e: int, x: torch.Tensor) -> torch.Tensor:
    """down(silu(gate x) * up x) for float64 rows x [m, H]."""
    g = x @ torch_dequant(d.gate, e).T
    u = x @ torch_dequant(d.up, e).T
    h = torch.nn.functional.silu(g) * u
    return h @ torch_dequant(d.down, e).T


def torch_route(logits: torch.Tensor, k: int):
    p = torch.softmax(logits.to(torch.float64), dim=-1)
    vals, ids = torch.topk(logits.to(torch.float64), k, dim=-1)
    w = torch.gather(p, 1, ids)
    return ids, w / w.sum(dim=-1, keepdim=True)


def torch_layer(inp: synth.LayerInputs, ids=None, w=None, gate=None) -> torch.Tensor:
    """out[t] = sum_j w[t, j] * FFN_{ids[t, j]}(x[t]) + g[t] * shared(x[t]),
    float64; g[t] = torch.sigmoid(x[t] . gate) for a bf16 gate weight [H],
    else 1."""
    x = inp.x.cpu().to(torch.float64)
    if ids is None:
        ids, w = torch_route(inp.logits.cpu(), inp.shape.top_k)
    out = torch.zeros(x.shape[0], inp.shape.H, dtype=torch.float64)
    for t in range(x.shape[0]):
        for j in range(ids.shape[1]):
            out[t] += float(w[t, j]) * torch_ffn(inp.experts, int(ids[t, j]), x[t: t + 1])[0]
    if inp.shared is not None:
        sh = torch_ffn(inp.shared, 0, x)
        if gate is not None:
            sh = torch.sigmoid(x @ gate.cpu().to(torch.float64))[:, None] * sh
        out += sh
    return out


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


# --------------------------------------------------------------------------
# running the GPU path and the oracle on the same inputs
# --------------------------------------------------------------------------

# Tolerances.  Layer output (bf16): the workload statement's relative L2
# 1e-3 and max-abs 2e-2, comparing the bf16 outputs of both sides.
# Intermediates (fp32 on the GPU against double): fp32 accumulation of K <=
# 4096 exact products has a typical relative error ~ sqrt(K) * 2^-24 < 4e-6;
# 1e-5 relative L2 leaves 2.5x margin.
LAYER_REL_L2 = 1e-3
LAYER_MAX_ABS = 2e-2
STAGE_REL_L2 = 1e-5
TOPK_W_ABS = 2e-6


def gpu_layer(moe, inp: synth.LayerInputs, path: int = 0, use_logits: bool = True,
              ids=None, w=None, err=None):
    """Run moe_decode_layer on device inputs; returns (out bf16 [M, H], view)."""
    s = inp.shape
    routed = moe.Experts.from_synth(inp.experts)
    shared = moe.Experts.from_synth(inp.shared) if inp.shared is not None else None
    layer = moe.LayerDesc(top_k=s.top_k, block_size=s.BS, routed=routed, shared=shared, path=path)
    ws = moe.alloc_workspace(layer, s.M)
    out = torch.empty(s.M, s.H, dtype=torch.bfloat16, device="cuda")
    if use_logits:
        moe.moe_decode_layer(layer, inp.x, out, ws, router_logits=inp.logits, err_word=err)
    else:
        moe.moe_decode_layer(layer, inp.x, out, ws, topk_ids=ids, topk_w=w, err_word=err)
    torch.cuda.synchronize()
    return out, moe.workspace_view(layer, s.M, ws), (layer, ws)


def oracle_layer(inp: synth.LayerInputs, ids=None, w=None):
    """The oracle's layer output for the same inputs (host copies)."""
    s = inp.shape
    X = oracle_experts(inp.experts.to("cpu"))
    S = oracle_experts(inp.shared.to("cpu")) if inp.shared is not None else None
    xb = synth.bf16_bits(inp.x)
    if ids is None:
        return oracle.moe_layer(X, S, xb, s.M, s.top_k, s.BS, logits=inp.logits.cpu().numpy())
    return oracle.moe_layer(X, S, xb, s.M, s.top_k, s.BS, ids=ids, w=w)


def compare_bf16(got: torch.Tensor, ref_bits: np.ndarray):
    g = synth.bf16_bits(got).astype(np.uint16)
    gf = oracle.bf16_bits_to_f64(g)
    rf = oracle.bf16_bits_to_f64(ref_bits)
    return rel_l2(gf, rf), float(np.abs(gf - rf).max())
