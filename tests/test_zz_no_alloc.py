"""moe_decode_layer_noalloc: the decode layer for callers that cannot allocate
device memory when they run it (code inside another framework's captured
graph, plugins whose host forbids allocation after start-up, runtimes with a
fixed device budget).  It takes its workspace from the library's fixed device
array instead of a caller buffer; its output must match moe_decode_layer's on
the same inputs, call after call.

Both calls run the same kernels on the same inputs, so the output must be
the same bits, not merely within the layer tolerance: a stale counter or a
misplaced region of the shared array would show as a few changed values.

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test before it; it also passes alone in a fresh
process."""
from __future__ import annotations

import pytest
import torch

import synth
from tests.helpers import LAYER_MAX_ABS, LAYER_REL_L2, compare_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import expert_routing_alignment_gb300 as m
    m.load()
    return m


def _layer(moe, inp, path=0):
    s = inp.shape
    routed = moe.Experts.from_synth(inp.experts)
    shared = moe.Experts.from_synth(inp.shared) if inp.shared is not None else None
    return moe.LayerDesc(top_k=s.top_k, block_size=s.BS, routed=routed, shared=shared, path=path)


@pytest.mark.parametrize("shape", [synth.tiny(), synth.decode_fp8(8), synth.decode_fp8(1),
                                   synth.decode_nvfp4(8)], ids=lambda s: s.name)
def test_noalloc_matches_decode_layer_two_calls_in_a_row(moe, shape):
    inp = synth.make_layer(shape, 4242, device="cuda")
    layer = _layer(moe, inp)
    ws = moe.alloc_workspace(layer, shape.M)
    ref = torch.empty(shape.M, shape.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_decode_layer(layer, inp.x, ref, ws, router_logits=inp.logits)
    ref_bits = synth.bf16_bits(ref)
    for call in range(2):
        out = torch.full((shape.M, shape.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.moe_decode_layer_noalloc(layer, inp.x, out, router_logits=inp.logits, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, call
        rel, mx = compare_bf16(out, ref_bits)
        assert rel <= LAYER_REL_L2 and mx <= LAYER_MAX_ABS, (call, rel, mx)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), call


@pytest.mark.parametrize("path", [0, 1], ids=["auto", "simt"])
def test_noalloc_alternating_rows_share_the_array(moe, path):
    # M = 8, then 1, then 8 again through the one shared array: each call's
    # output is the bits of moe_decode_layer on a fresh workspace
    outs = {}
    for M in (8, 1, 8):
        shape = synth.decode_fp8(M)
        inp = synth.make_layer(shape, 9000 + M, device="cuda")
        layer = _layer(moe, inp, path)
        if M not in outs:
            ws = moe.alloc_workspace(layer, M)
            ref = torch.empty(M, shape.H, dtype=torch.bfloat16, device="cuda")
            moe.moe_decode_layer(layer, inp.x, ref, ws, router_logits=inp.logits)
            outs[M] = ref
        out = torch.full((M, shape.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.moe_decode_layer_noalloc(layer, inp.x, out, router_logits=inp.logits, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, M
        assert torch.equal(out.view(torch.int16), outs[M].view(torch.int16)), M


def test_noalloc_given_ids_matches_decode_layer(moe):
    shape = synth.decode_fp8(4)
    inp = synth.make_layer(shape, 77, device="cuda")
    layer = _layer(moe, inp)
    ids, w = moe.moe_topk_softmax(inp.logits, shape.top_k)
    ws = moe.alloc_workspace(layer, shape.M)
    ref = torch.empty(shape.M, shape.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_decode_layer(layer, inp.x, ref, ws, topk_ids=ids, topk_w=w)
    for _ in range(2):
        out = torch.empty_like(ref)
        moe.moe_decode_layer_noalloc(layer, inp.x, out, topk_ids=ids, topk_w=w)
        torch.cuda.synchronize()
        rel, mx = compare_bf16(out, synth.bf16_bits(ref))
        assert rel <= LAYER_REL_L2 and mx <= LAYER_MAX_ABS
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_noalloc_rejects_a_workspace_beyond_its_array(moe):
    # the verify batch (M=128, H=4096, I=1536, E=256, BS=64) needs far more
    # than the array: rejected on the host, nothing launched, output untouched
    # (the weights are never read: small stand-in tables give the pointers)
    shape = synth.verify_fp8(128)
    E, H, I = shape.E, shape.H, shape.I
    f8 = lambda: torch.zeros(256, dtype=torch.uint8, device="cuda")
    sc = lambda: torch.ones(64, device="cuda")
    ex = moe.Experts(moe.FMT_FP8_B128, E, H, I, gate=(f8(), sc(), None), up=(f8(), sc(), None),
                     down=(f8(), sc(), None))
    layer = moe.LayerDesc(top_k=shape.top_k, block_size=shape.BS, routed=ex)
    assert moe.workspace_bytes(layer, shape.M) > moe.NOALLOC_SCRATCH_BYTES
    x = torch.zeros(shape.M, H, dtype=torch.bfloat16, device="cuda")
    logits = torch.zeros(shape.M, E, device="cuda")
    out = torch.full((shape.M, H), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as exc:
        moe.moe_decode_layer_noalloc(layer, x, out, router_logits=logits)
    assert exc.value.status == moe.MOE_EUNSUPPORTED
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
