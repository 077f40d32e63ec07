"""The router logits on the GPU against the oracle (the matrix-vector product
ahead of the top-k): tiny, decode and verify widths and an odd shape, within
a bound derived from fp32 accumulation; run-to-run bit equality; a row's
logits the same bits for every batch width (the kernel takes 1 to 8 expert
rows per block by M); and the top-k taken on the GPU's logits equals the
oracle's top-k of the same fp32 logits."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import helpers as H_

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import expert_routing_alignment_gb300 as m
    m.load()
    return m


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


SHAPES = [(4, 256, 8), (1, 2048, 128), (8, 2048, 128), (128, 4096, 256), (3, 264, 33),
          (17, 8192, 64), (200, 1024, 157), (2, 16384, 16), (1, 8, 1), (5, 16, 3)]


@pytest.mark.parametrize("M,H,E", SHAPES, ids=lambda v: str(v))
def test_router_logits_match_oracle(moe, M, H, E):
    g = torch.Generator(device="cuda").manual_seed(M * 1000 + E)
    x = torch.randn(M, H, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(E, H, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    got = moe.moe_router_logits(x, W)
    torch.cuda.synchronize()
    ref = oracle.router_logits(_bits(x), _bits(W))
    # every product of two bf16 values is exact in fp32; the sum of H of them
    # in fp32 errs by at most H * 2^-24 of the sum of magnitudes (a loose,
    # order-free bound); 2^-14 of it is far above what the fixed order gives
    mag = (x.double().abs() @ W.double().abs().T).cpu().numpy()
    err = np.abs(got.cpu().numpy().astype(np.float64) - ref)
    assert (err <= mag * 2.0 ** -14).all(), float((err / np.maximum(mag, 1e-30)).max())
    # run to run identical
    again = moe.moe_router_logits(x, W)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int32), again.view(torch.int32))


def test_router_rows_invariant_across_batch_widths(moe):
    H, E = 4096, 256
    g = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn(128, H, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(E, H, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    full = moe.moe_router_logits(x, W)
    for M in (1, 5, 8, 40):
        part = moe.moe_router_logits(x[:M].contiguous(), W)
        torch.cuda.synchronize()
        assert torch.equal(part.view(torch.int32), full[:M].view(torch.int32)), M


def test_router_then_topk_equals_oracle_topk_of_the_same_logits(moe):
    M, H, E, k = 8, 2048, 128, 8
    g = torch.Generator(device="cuda").manual_seed(7)
    x = torch.randn(M, H, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(E, H, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    lg = moe.moe_router_logits(x, W)
    ids, w = moe.moe_topk_softmax(lg, k)
    torch.cuda.synchronize()
    rid, rw = oracle.topk_softmax(lg.cpu().numpy(), k)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, atol=2e-6)


def test_router_rejects_unsupported_shapes(moe):
    x = torch.zeros(2, 100, dtype=torch.bfloat16, device="cuda")   # hidden % 8 != 0
    W = torch.zeros(4, 100, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as exc:
        moe.moe_router_logits(x, W)
    assert exc.value.status == moe.MOE_EUNSUPPORTED


HIDDEN_IN = [(synth.decode_fp8(1), 0), (synth.decode_fp8(8), 0), (synth.decode_fp8(8), 1),
             (synth.decode_fp8(8), 3),
             (synth.decode_nvfp4(8), 0), (synth.verify_fp8(128), 0)]


@pytest.mark.parametrize("shape,path", HIDDEN_IN, ids=lambda v: getattr(v, "name", str(v)))
def test_layer_hidden_in_equals_logits_in(moe, shape, path):
    """x alone (the layer computes its logits from its router weights) gives
    the same output bits as passing moe_router_logits' logits, on the
    tensor-core, fused and staged paths; the workspace keeps those logits."""
    inp = synth.make_layer(shape, 1000, device="cuda")
    W = synth.make_router_weight(shape.E, shape.H, 2024, device="cuda")
    routed = moe.Experts.from_synth(inp.experts)
    shared = moe.Experts.from_synth(inp.shared) if inp.shared is not None else None
    layer = moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS, routed=routed, shared=shared,
                          path=path, router_weight=W)
    ws = moe.alloc_workspace(layer, shape.M)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_h = torch.empty(shape.M, shape.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_decode_layer(layer, inp.x, out_h, ws, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    view = moe.workspace_view(layer, shape.M, ws)
    lg = moe.moe_router_logits(inp.x, W)
    torch.cuda.synchronize()
    assert torch.equal(view["router_logits"].view(torch.int32), lg.view(torch.int32))
    out_l = torch.empty_like(out_h)
    ws2 = moe.alloc_workspace(layer, shape.M)
    moe.moe_decode_layer(layer, inp.x, out_l, ws2, router_logits=lg)
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int16), out_l.view(torch.int16))


def test_layer_hidden_in_matches_oracle_chain(moe):
    """The whole hidden-in chain against the oracle's: oracle router logits
    (double), its top-k on them, its layer; the GPU's ids equal the oracle's
    and the output is within the layer tolerance."""
    shape = synth.decode_fp8(8)
    inp = synth.make_layer(shape, 1000, device="cuda")
    W = synth.make_router_weight(shape.E, shape.H, 2024, device="cuda")
    routed = moe.Experts.from_synth(inp.experts)
    layer = moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS, routed=routed, router_weight=W)
    ws = moe.alloc_workspace(layer, shape.M)
    out = torch.empty(shape.M, shape.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_decode_layer(layer, inp.x, out, ws)
    torch.cuda.synchronize()
    view = moe.workspace_view(layer, shape.M, ws)
    ref_lg = oracle.router_logits(_bits(inp.x), _bits(W))
    rid, _ = oracle.topk_softmax(ref_lg, shape.top_k)
    np.testing.assert_array_equal(view["topk_ids"].cpu().numpy(), rid.ravel())
    X = H_.oracle_experts(inp.experts.to("cpu"))
    _, ref_b, bad = oracle.moe_layer(X, None, _bits(inp.x), shape.M, shape.top_k, shape.BS,
                                     logits=ref_lg)
    assert bad == 0
    rl2, mx = H_.compare_bf16(out, ref_b)
    assert rl2 < H_.LAYER_REL_L2 and mx < H_.LAYER_MAX_ABS, (rl2, mx)
