"""The decode MoE layer on the GPU against the oracle.

Stages are checked in isolation (each fed the same inputs as the oracle's
function), then the whole layer on every workload: the tiny layer, the
128-expert FP8 decode layer at M = 1, 2, 4, 8, the NVFP4 layer with an FP8
shared expert at M = 1, 8, 32, and the M = 128 verify batch (sampled rows).
Row invariance, determinism, CUDA-graph replay and out-of-range ids too."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import expert_routing_alignment_gb300 as m
    m.load()
    return m


_CACHE = {}


def layer_inputs(shape: synth.LayerShape, seed: int = 1000) -> synth.LayerInputs:
    key = (shape, seed)
    if key not in _CACHE:
        _CACHE.clear()
        _CACHE[key] = synth.make_layer(shape, seed, device="cuda")
    return _CACHE[key]


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------

@pytest.mark.parametrize("M,E,k", [(4, 8, 2), (8, 128, 8), (32, 128, 8), (128, 256, 8),
                                   (3, 1024, 32), (5, 33, 1)])
def test_topk_softmax_matches_oracle(moe, M, E, k):
    lg = synth.make_logits(M, E, seed=M * E, device="cuda")
    ids, w = moe.moe_topk_softmax(lg, k)
    torch.cuda.synchronize()
    rid, rw = oracle.topk_softmax(lg.cpu().numpy(), k)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=0, atol=H.TOPK_W_ABS)


def test_topk_ties_take_lower_id(moe):
    lg = torch.randint(-2, 3, (64, 40), generator=torch.Generator().manual_seed(2)).float()
    ids, w = moe.moe_topk_softmax(lg.cuda(), 6)
    torch.cuda.synchronize()
    rid, rw = oracle.topk_softmax(lg.numpy(), 6)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=0, atol=H.TOPK_W_ABS)


# --------------------------------------------------------------------------
# grouped stages in isolation
# --------------------------------------------------------------------------

STAGE_SHAPES = [synth.tiny(), synth.decode_fp8(8), synth.decode_nvfp4(8)]


@pytest.mark.parametrize("shape", STAGE_SHAPES, ids=lambda s: s.name)
def test_grouped_stages_match_oracle(moe, shape):
    inp = layer_inputs(shape)
    s = shape
    routed = moe.Experts.from_synth(inp.experts)
    shared = moe.Experts.from_synth(inp.shared) if inp.shared is not None else None
    ids, w = moe.moe_topk_softmax(inp.logits, s.top_k)
    t = moe.moe_align(ids, s.E, s.BS)
    I, Hd = s.I, s.H
    h = torch.zeros(t["max_total"], I, device="cuda")
    y = torch.zeros(t["max_total"], Hd, device="cuda")
    h_sh = torch.zeros(s.M, s.shared_I, device="cuda") if shared else None
    y_sh = torch.zeros(s.M, Hd, device="cuda") if shared else None
    moe.moe_grouped_gate_up(routed, shared, inp.x, s.top_k, t, h, h_sh, path=moe.PATH_SIMT)
    moe.moe_grouped_down(routed, shared, h, h_sh, s.M, s.top_k, t, y, y_sh, path=moe.PATH_SIMT)
    out = torch.empty(s.M, Hd, dtype=torch.bfloat16, device="cuda")
    moe.moe_blend(y, w, t["token_to_perm"], y_sh, out, s.top_k)
    torch.cuda.synchronize()

    tables = oracle.align(ids.cpu().numpy().ravel(), s.E, s.BS)
    assert (t["sorted_token_ids"].cpu().numpy()[: t["max_total"]]
            == tables["sorted_token_ids"]).all()
    X = H.oracle_experts(inp.experts.to("cpu"))
    S = H.oracle_experts(inp.shared.to("cpu")) if shared else None
    real = tables["sorted_token_ids"] < s.n

    # gate + up on the same x and tables
    h_ref, hs_ref = oracle.grouped_gate_up(X, S, synth.bf16_bits(inp.x), s.M, s.top_k, tables)
    h_gpu = h.cpu().numpy().astype(np.float64)
    assert H.rel_l2(h_gpu[real], h_ref[real]) < H.STAGE_REL_L2
    if shared:
        assert H.rel_l2(h_sh.cpu().numpy(), hs_ref) < H.STAGE_REL_L2

    # down on the GPU's own h
    hs_gpu = h_sh.cpu().numpy().astype(np.float64) if shared else None
    y_ref, ys_ref = oracle.grouped_down(X, S, h_gpu, hs_gpu, s.M, s.top_k, tables)
    y_gpu = y.cpu().numpy().astype(np.float64)
    assert H.rel_l2(y_gpu[real], y_ref[real]) < H.STAGE_REL_L2
    if shared:
        assert H.rel_l2(y_sh.cpu().numpy(), ys_ref) < H.STAGE_REL_L2

    # blend on the GPU's own y and weights: equal bf16 bits except where the
    # fp32 and double sums fall on two sides of a rounding boundary (1 ulp)
    ys_gpu = y_sh.cpu().numpy().astype(np.float64) if shared else None
    _, ob = oracle.blend(y_gpu, w.cpu().numpy().astype(np.float64), tables["token_to_perm"],
                         ys_gpu, s.M, s.top_k, Hd)
    gb = synth.bf16_bits(out).astype(np.int32)
    diff = np.abs(gb - ob.astype(np.int32))
    assert diff.max() <= 1 and (diff > 0).mean() < 0.01


# --------------------------------------------------------------------------
# the whole layer
# --------------------------------------------------------------------------

LAYER_SHAPES = ([synth.tiny()] + [synth.decode_fp8(M) for M in (1, 2, 4, 8)]
                + [synth.decode_nvfp4(M) for M in (1, 8, 32)])
# "auto" takes the tensor cores for the FP8 shapes, "fused" (MOE_PATH_SIMT)
# keeps every shape on the CUDA cores' one-launch kernel, "staged" forces the
# five CUDA-core launches.
PATHS = {"auto": 0, "fused": 1, "staged": 3}
TC_Y_REL_L2 = 5e-4   # y from h carried as three E4M3 terms (see test_tc_gpu)


@pytest.mark.parametrize("path", list(PATHS), ids=str)
@pytest.mark.parametrize("shape", LAYER_SHAPES, ids=lambda s: s.name)
def test_layer_matches_oracle(moe, shape, path):
    inp = layer_inputs(shape)
    out, view, (layer, _) = H.gpu_layer(moe, inp, path=PATHS[path])
    if path == "fused":
        assert moe.moe_decode_layer_launches(layer, shape.M) == 1
    _, ref_b, bad = H.oracle_layer(inp)
    assert bad == 0
    rl2, mx = H.compare_bf16(out, ref_b)
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS, (rl2, mx)
    # the layer's own tables equal the oracle's
    rid, rw = oracle.topk_softmax(inp.logits.cpu().numpy(), shape.top_k)
    np.testing.assert_array_equal(view["topk_ids"].cpu().numpy(), rid.ravel())
    np.testing.assert_allclose(view["topk_w"].cpu().numpy(), rw.ravel(), atol=H.TOPK_W_ABS)
    tables = oracle.align(rid.ravel(), shape.E, shape.BS)
    for key in ("sorted_token_ids", "expert_offsets", "token_to_perm", "sorted_expert_ids",
                "active_experts"):
        np.testing.assert_array_equal(view[key].cpu().numpy(), tables[key], err_msg=key)
    assert int(view["active_count"].item()) == int(tables["active_count"][0])
    assert int(view["num_tokens_post_padded"].item()) == int(tables["num_tokens_post_padded"][0])
    if shape.M <= 8:
        # the intermediates in the workspace: h against the oracle on the same
        # x, y against the oracle's down of the layer's own h
        X = H.oracle_experts(inp.experts.to("cpu"))
        S = H.oracle_experts(inp.shared.to("cpu")) if inp.shared is not None else None
        real = tables["sorted_token_ids"] < shape.n
        h_ref, hs_ref = oracle.grouped_gate_up(X, S, synth.bf16_bits(inp.x), shape.M,
                                               shape.top_k, tables)
        h_gpu = view["h"].cpu().numpy().astype(np.float64)
        assert H.rel_l2(h_gpu[real], h_ref[real]) < H.STAGE_REL_L2
        hs_gpu = view["h_shared"].cpu().numpy().astype(np.float64) if S else None
        if S:
            assert H.rel_l2(hs_gpu, hs_ref) < H.STAGE_REL_L2
        y_ref, ys_ref = oracle.grouped_down(X, S, h_gpu, hs_gpu, shape.M, shape.top_k, tables)
        y_gpu = view["y"].cpu().numpy().astype(np.float64)
        y_tol = TC_Y_REL_L2 if "tc_h_terms" in view else H.STAGE_REL_L2
        assert H.rel_l2(y_gpu[real], y_ref[real]) < y_tol
        if S:
            assert H.rel_l2(view["y_shared"].cpu().numpy(), ys_ref) < H.STAGE_REL_L2


def test_verify_batch_sampled_rows(moe):
    """M = 128, H = 4096, I = 1536, E = 256, k = 8, BS = 64 with a Zipf(1.1)
    router bias: the full batch on the GPU, the oracle on 6 sampled rows
    (each row's output depends on that row only)."""
    shape = synth.verify_fp8(128)
    inp = layer_inputs(shape)
    out, view, _ = H.gpu_layer(moe, inp)
    counts = np.bincount(view["topk_ids"].cpu().numpy(), minlength=shape.E)
    assert counts.max() >= 30, counts.max()           # the skew the workload asks for
    rows = [0, 17, 63, 64, 101, 127]
    lg = inp.logits[rows].cpu().numpy()
    rid, rw = oracle.topk_softmax(lg, shape.top_k)
    uniq = sorted(set(rid.ravel().tolist()))
    remap = {e: i for i, e in enumerate(uniq)}
    sub = H.subset_experts(inp.experts, uniq)
    X = H.oracle_experts(sub)
    ids_sub = np.vectorize(remap.get)(rid).astype(np.int32)
    _, ref_b, _ = oracle.moe_layer(X, None, synth.bf16_bits(inp.x[rows]), len(rows),
                                   shape.top_k, shape.BS, ids=ids_sub, w=rw)
    rl2, mx = H.compare_bf16(out[rows], ref_b)
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS, (rl2, mx)


@pytest.mark.parametrize("path", list(PATHS), ids=str)
@pytest.mark.parametrize("shape", [synth.decode_nvfp4(32), synth.decode_fp8(8),
                                   synth.decode_fp8(16)], ids=lambda s: s.name)
def test_row_invariance(moe, shape, path):
    """Row 0's output bits are the same whether the batch has 1 or M rows (on
    the tensor cores, M = 1..16 share the decode kernel)."""
    inp = layer_inputs(shape)
    out_m, _, _ = H.gpu_layer(moe, inp, path=PATHS[path])
    one = synth.LayerInputs(
        synth.LayerShape(shape.name + "_row0", 1, shape.H, shape.I, shape.E, shape.top_k,
                         shape.BS, shape.fmt, shape.shared_I),
        inp.x[:1].contiguous(), inp.logits[:1].contiguous(), inp.experts, inp.shared)
    out_1, _, _ = H.gpu_layer(moe, one, path=PATHS[path])
    assert torch.equal(out_m[:1].view(torch.int16), out_1.view(torch.int16))


def test_layer_deterministic_and_graph_replayable(moe):
    shape = synth.decode_fp8(8)
    inp = layer_inputs(shape)
    out_a, _, (layer, ws) = H.gpu_layer(moe, inp)
    out_b, _, _ = H.gpu_layer(moe, inp)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))

    logits = inp.logits.clone()
    out = torch.empty_like(out_a)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        moe.moe_decode_layer(layer, inp.x, out, ws, router_logits=logits)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_decode_layer(layer, inp.x, out, ws, router_logits=logits)
    for seed in (5, 6):
        logits.copy_(synth.make_logits(shape.M, shape.E, seed, device="cuda"))
        g.replay()
        torch.cuda.synchronize()
        eager = torch.empty_like(out)
        moe.moe_decode_layer(layer, inp.x, eager, ws, router_logits=logits)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


@pytest.mark.parametrize("path", list(PATHS), ids=str)
def test_layer_given_ids_with_out_of_range_id(moe, path):
    shape = synth.tiny(M=4)
    inp = layer_inputs(shape)
    ids, w = oracle.topk_softmax(inp.logits.cpu().numpy(), shape.top_k)
    ids[1, 1] = shape.E + 3                        # out of range: skipped, flagged
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, view, _ = H.gpu_layer(moe, inp, path=PATHS[path], use_logits=False,
                               ids=torch.from_numpy(ids).cuda(),
                               w=torch.from_numpy(w.astype(np.float32)).cuda(), err=err)
    assert int(err.item()) == moe.MOE_ERR_BAD_ID
    _, ref_b, bad = H.oracle_layer(inp, ids=ids, w=w)
    assert bad == 1
    rl2, mx = H.compare_bf16(out, ref_b)
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS
    tables = oracle.align(ids.ravel(), shape.E, shape.BS)
    np.testing.assert_array_equal(view["token_to_perm"].cpu().numpy(), tables["token_to_perm"])
    np.testing.assert_array_equal(view["sorted_token_ids"].cpu().numpy(),
                                  tables["sorted_token_ids"])


def test_fused_and_staged_paths_agree(moe):
    """The fused pair and the five launches compute the same layer: equal
    tables, outputs within the layer tolerance of each other."""
    shape = synth.decode_nvfp4(8)
    inp = layer_inputs(shape)
    out_f, vf, _ = H.gpu_layer(moe, inp, path=PATHS["fused"])
    out_s, vs, _ = H.gpu_layer(moe, inp, path=PATHS["staged"])
    for key in ("sorted_token_ids", "expert_offsets", "token_to_perm", "topk_ids"):
        assert torch.equal(vf[key], vs[key]), key
    rl2, mx = H.compare_bf16(out_f, synth.bf16_bits(out_s))
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS


@pytest.mark.parametrize("path", [0, 1], ids=["auto", "simt"])
def test_one_workspace_serves_alternating_rows(moe, path):
    """A workspace sized for M=8 serves calls at M=8, then M=1, then M=8: each
    output is the bits of the same call on a fresh zeroed workspace (the
    counters that persist between calls sit where M does not move them)."""
    shape8 = synth.decode_fp8(8)
    ex = synth.make_experts(shape8.E, shape8.H, shape8.I, shape8.fmt, 3100, "cuda")
    layer = moe.LayerDesc(top_k=shape8.top_k, block_size=shape8.BS,
                          routed=moe.Experts.from_synth(ex), path=path)
    shared_ws = moe.alloc_workspace(layer, 8)
    for call, M in enumerate((8, 1, 8, 1)):
        x = synth.make_x(M, shape8.H, 3200 + call, "cuda")
        lg = synth.make_logits(M, shape8.E, 3300 + call, "cuda")
        fresh = torch.empty(M, shape8.H, dtype=torch.bfloat16, device="cuda")
        moe.moe_decode_layer(layer, x, fresh, moe.alloc_workspace(layer, M), router_logits=lg)
        out = torch.full((M, shape8.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.moe_decode_layer(layer, x, out, shared_ws, router_logits=lg, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, (call, M)
        assert torch.equal(out.view(torch.int16), fresh.view(torch.int16)), (call, M)


@pytest.mark.parametrize("path", [0, 1, 3], ids=["auto", "simt", "staged"])
@pytest.mark.parametrize("M", [4, 32], ids=["m4", "m32"])
def test_decode_experts_on_tables_in_the_workspace(moe, path, M):
    """moe_decode_experts runs the expert half of the layer on the routing and
    alignment tables an earlier moe_decode_layer call left in the workspace:
    again on the same x it gives the same bits, and on another x the bits of
    moe_decode_layer on that x with the same logits."""
    shape = synth.LayerShape(f"decode_h2048_i768_e128_k8_fp8_m{M}", M, 2048, 768, 128, 8, 16,
                             synth.FMT_FP8)
    inp = synth.make_layer(shape, 5150, device="cuda")
    out, view, (layer, ws) = H.gpu_layer(moe, inp, path=path)
    again = torch.full_like(out, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_decode_experts(layer, inp.x, again, ws, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(again.view(torch.int16), out.view(torch.int16))
    x2 = synth.make_x(M, shape.H, 5151, "cuda")
    ref2 = torch.empty_like(out)
    moe.moe_decode_layer(layer, x2, ref2, moe.alloc_workspace(layer, M), router_logits=inp.logits)
    third = torch.full_like(out, float("nan"))
    moe.moe_decode_experts(layer, x2, third, ws, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(third.view(torch.int16), ref2.view(torch.int16))


@pytest.mark.parametrize("path", [0, 2, 1, 3], ids=["auto", "tc", "simt", "staged"])
@pytest.mark.parametrize("M", [1, 8, 32])
def test_nvfp4_gate_up_tier_matches_oracle(moe, M, path):
    """The nvfp4-gate-up tier (NVFP4 gate and up, FP8 down, FP8 shared expert)
    runs on the NVFP4 tensor-core kernel (default and MOE_PATH_TC: its down
    projection as E4M3 items) or on the staged CUDA-core kernels (each
    projection in its own format): the layer output within the layer
    tolerance of the oracle, h and y within the stage tolerance of the
    oracle's stages, and row 0 the same bits at M rows as alone."""
    shape = synth.decode_nvfp4_gate_up(M)
    inp = layer_inputs(shape)
    out, view, (layer, _) = H.gpu_layer(moe, inp, path=path)
    assert moe.moe_decode_layer_launches(layer, M) == (3 if path in (0, 2) else 5)
    _, ref_b, bad = H.oracle_layer(inp)
    assert bad == 0
    rl2, mx = H.compare_bf16(out, ref_b)
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS, (rl2, mx)
    tables = oracle.align(view["topk_ids"].cpu().numpy(), shape.E, shape.BS)
    real = tables["sorted_token_ids"] < shape.n
    X = H.oracle_experts(inp.experts.to("cpu"))
    S = H.oracle_experts(inp.shared.to("cpu"))
    h_ref, hs_ref = oracle.grouped_gate_up(X, S, synth.bf16_bits(inp.x), M, shape.top_k, tables)
    h_gpu = view["h"].cpu().numpy().astype(np.float64)
    assert H.rel_l2(h_gpu[real], h_ref[real]) < H.STAGE_REL_L2
    hs_gpu = view["h_shared"].cpu().numpy().astype(np.float64)
    assert H.rel_l2(hs_gpu, hs_ref) < H.STAGE_REL_L2
    y_ref, ys_ref = oracle.grouped_down(X, S, h_gpu, hs_gpu, M, shape.top_k, tables)
    assert H.rel_l2(view["y"].cpu().numpy().astype(np.float64)[real], y_ref[real]) < H.STAGE_REL_L2
    assert H.rel_l2(view["y_shared"].cpu().numpy(), ys_ref) < H.STAGE_REL_L2
    one = synth.LayerInputs(
        synth.LayerShape(shape.name + "_row0", 1, shape.H, shape.I, shape.E, shape.top_k,
                         shape.BS, shape.fmt, shape.shared_I),
        inp.x[:1].contiguous(), inp.logits[:1].contiguous(), inp.experts, inp.shared)
    out_1, _, _ = H.gpu_layer(moe, one, path=path)
    assert torch.equal(out[:1].view(torch.int16), out_1.view(torch.int16))


@pytest.mark.parametrize("M", [256, 1024])
def test_prefill_batch_sampled_rows(moe, M):
    """Prefill-sized batches (M > 128, FP8 experts of the verify shape: H=4096,
    I=1536, E=256, k=8, BS=64) run on the tensor-core path: the alignment's
    tables bit-exact, and sampled rows within the layer tolerance of the
    oracle (each row's output depends on that row only)."""
    shape = synth.LayerShape(f"prefill_h4096_i1536_e256_k8_fp8_m{M}", M, 4096, 1536, 256, 8, 64,
                             synth.FMT_FP8)
    inp = layer_inputs(shape)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, view, (layer, _) = H.gpu_layer(moe, inp, err=err)
    assert moe.moe_decode_layer_launches(layer, M) == 3
    assert int(err.item()) == 0
    rid, rw = oracle.topk_softmax(inp.logits.cpu().numpy(), shape.top_k)
    np.testing.assert_array_equal(view["topk_ids"].cpu().numpy(), rid.ravel())
    tables = oracle.align(rid.ravel(), shape.E, shape.BS)
    for key in ("sorted_token_ids", "expert_offsets", "token_to_perm", "sorted_expert_ids",
                "active_experts"):
        np.testing.assert_array_equal(view[key].cpu().numpy(), tables[key], err_msg=key)
    rows = [0, 1, M // 3, M // 2 + 7, M - 1]
    uniq = sorted(set(rid[rows].ravel().tolist()))
    remap = {e: i for i, e in enumerate(uniq)}
    X = H.oracle_experts(H.subset_experts(inp.experts, uniq))
    ids_sub = np.vectorize(remap.get)(rid[rows]).astype(np.int32)
    _, ref_b, _ = oracle.moe_layer(X, None, synth.bf16_bits(inp.x[rows]), len(rows),
                                   shape.top_k, shape.BS, ids=ids_sub, w=rw[rows])
    rl2, mx = H.compare_bf16(out[rows], ref_b)
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS, (rl2, mx)
