"""The gated shared expert on the GPU against the oracle: the blend's gate
sigmoid(x[t] . gate_w) on the shared term, alone (moe_blend) and in the whole
layer on the fused and staged CUDA-core paths (NVFP4 routed experts with an
FP8 shared expert, and FP8 routed experts with one)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu

# a gate is sigmoid of an fp32 dot of at most 8192 exact products: its
# error is far below 1e-6 for arguments of unit size
GATE_ABS = 1e-6


@pytest.fixture(scope="module")
def moe():
    import expert_routing_alignment_gb300 as m
    m.load()
    return m


def test_blend_gated_matches_oracle(moe):
    M, k, E, Hd = 8, 8, 128, 2048
    g = torch.Generator(device="cuda").manual_seed(11)
    logits = torch.randn(M, E, generator=g, device="cuda")
    ids, w = moe.moe_topk_softmax(logits, k)
    t = moe.moe_align(ids, E, 16)
    y = torch.randn(t["max_total"], Hd, generator=g, device="cuda")
    y_sh = torch.randn(M, Hd, generator=g, device="cuda")
    x = synth.make_x(M, Hd, 12, device="cuda")
    gate = synth.make_shared_gate(Hd, 13, device="cuda")
    out = torch.empty(M, Hd, dtype=torch.bfloat16, device="cuda")
    moe.moe_blend(y, w, t["token_to_perm"], y_sh, out, k, x=x, shared_gate=gate)
    torch.cuda.synchronize()
    tables = oracle.align(ids.cpu().numpy().ravel(), E, 16)
    g_ref = oracle.shared_gate(synth.bf16_bits(x), synth.bf16_bits(gate))
    assert 0.02 < g_ref.min() and g_ref.max() < 0.98   # the gate is not saturated
    _, ob = oracle.blend(y.cpu().numpy().astype(np.float64), w.cpu().numpy().astype(np.float64),
                         tables["token_to_perm"], y_sh.cpu().numpy().astype(np.float64), M, k,
                         Hd, gate=g_ref)
    diff = np.abs(synth.bf16_bits(out).astype(np.int32) - ob.astype(np.int32))
    assert diff.max() <= 1 and (diff > 0).mean() < 0.01
    # ungated differs (the gate is really applied)
    out_u = torch.empty_like(out)
    moe.moe_blend(y, w, t["token_to_perm"], y_sh, out_u, k)
    torch.cuda.synchronize()
    assert not torch.equal(out.view(torch.int16), out_u.view(torch.int16))


def test_blend_gate_needs_the_shared_term(moe):
    y = torch.zeros(16, 256, device="cuda")
    w = torch.ones(2, 1, device="cuda")
    ttp = torch.zeros(2, dtype=torch.int32, device="cuda")
    x = torch.zeros(2, 256, dtype=torch.bfloat16, device="cuda")
    gate = torch.zeros(256, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(2, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as exc:
        moe.moe_blend(y, w, ttp, None, out, 1, x=x, shared_gate=gate)
    assert exc.value.status == moe.MOE_EINVAL


def _fp8_shared(M):
    return synth.LayerShape(f"decode_h2048_i768_e128_k8_fp8_shared512_m{M}", M, 2048, 768, 128,
                            8, 16, synth.FMT_FP8, shared_I=512)


GATED = [(synth.decode_nvfp4(1), 0), (synth.decode_nvfp4(8), 0), (synth.decode_nvfp4(32), 0),
         (synth.decode_nvfp4(8), 3), (synth.decode_nvfp4(32), 3), (_fp8_shared(8), 0),
         (_fp8_shared(8), 3)]


@pytest.mark.parametrize("shape,path", GATED, ids=lambda v: getattr(v, "name", str(v)))
def test_gated_layer_matches_oracle(moe, shape, path):
    inp = synth.make_layer(shape, 1000, device="cuda")
    gate = synth.make_shared_gate(shape.H, 77, device="cuda")
    routed = moe.Experts.from_synth(inp.experts)
    shared = moe.Experts.from_synth(inp.shared)
    layer = moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS, routed=routed, shared=shared,
                          path=path, shared_gate=gate)
    ws = moe.alloc_workspace(layer, shape.M)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(shape.M, shape.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_decode_layer(layer, inp.x, out, ws, router_logits=inp.logits, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    X = H.oracle_experts(inp.experts.to("cpu"))
    S = H.oracle_experts(inp.shared.to("cpu"))
    _, ref_b, bad = oracle.moe_layer(X, S, synth.bf16_bits(inp.x), shape.M, shape.top_k,
                                     shape.BS, logits=inp.logits.cpu().numpy(),
                                     shared_gate_bits=synth.bf16_bits(gate))
    assert bad == 0
    rl2, mx = H.compare_bf16(out, ref_b)
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS, (rl2, mx)
    if moe.moe_decode_layer_launches(layer, shape.M) == 1:   # fused: the gates in the workspace
        g_ref = oracle.shared_gate(synth.bf16_bits(inp.x), synth.bf16_bits(gate))
        g = moe.workspace_view(layer, shape.M, ws)["shared_gate"].cpu().numpy()
        np.testing.assert_allclose(g, g_ref, rtol=0, atol=GATE_ABS)
    # the ungated layer differs from the gated one
    plain = moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS, routed=routed, shared=shared,
                          path=path)
    out_u = torch.empty_like(out)
    moe.moe_decode_layer(plain, inp.x, out_u, ws, router_logits=inp.logits)
    torch.cuda.synchronize()
    assert H.compare_bf16(out_u, ref_b)[0] > 10 * H.LAYER_REL_L2
