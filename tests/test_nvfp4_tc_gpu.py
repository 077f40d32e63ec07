"""The NVFP4 tensor-core expert kernel of the decode MoE layer against the
oracle (NVFP4 routed experts, M <= 32, with or without the FP8 shared expert).

The kernel decodes each E2M1 code times its E4M3 scale exactly to f16 in
tensor memory, multiplies it by an f16 x table by token (x times a power of
two per token, exact for bf16 x) and by h carried as two f16 terms (hi + lo,
22 significant bits under a power-of-two scale per (row, 128-column block)),
promotes every 128-wide k block to fp32 and applies the fp32 globals once per
item.  Checked here: the layer output within the workload's tolerance; h
against the oracle's gate+up on the same x and y against the oracle's down of
the layer's own h; the x table exact; the h terms within their bound; the
gates; row-invariant output bits across M (16 and 32 token columns);
one workspace serving alternating M (some on the CUDA cores); CUDA-graph
replay; the expert half alone through moe_decode_experts."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu

AUTO, TC = 0, 2

# h: exact weights (E2M1 x E4M3 in f16) and x (bf16 in f16 under a power of
# two), fp32 promotion of each 128-wide k block: the CUDA-core path's
# accumulation error.  y: h as hi + lo f16 terms is within 2^-22 of the
# (row, block) maximum, far below the fp32 accumulation error of the down.
F4_H_REL_L2 = H.STAGE_REL_L2
F4_Y_REL_L2 = H.STAGE_REL_L2
GATE_ABS = 1e-6


@pytest.fixture(scope="module")
def moe():
    import expert_routing_alignment_gb300 as m
    m.load()
    return m


def _shape(M, shared=True):
    return synth.LayerShape(
        f"decode_h2048_i768_e128_k8_nvfp4{'_shared512' if shared else ''}_m{M}", M, 2048, 768,
        128, 8, 16, synth.FMT_NVFP4, shared_I=512 if shared else None)


def _run(moe, inp, path=TC, gate=None, ws=None, M=None, err=None):
    s = inp.shape
    routed = moe.Experts.from_synth(inp.experts)
    shared = moe.Experts.from_synth(inp.shared) if inp.shared is not None else None
    layer = moe.LayerDesc(top_k=s.top_k, block_size=s.BS, routed=routed, shared=shared,
                          path=path, shared_gate=gate)
    if ws is None:
        ws = moe.alloc_workspace(layer, s.M)
    out = torch.full((s.M, s.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_decode_layer(layer, inp.x, out, ws, router_logits=inp.logits, err_word=err)
    torch.cuda.synchronize()
    return out, layer, ws


@pytest.mark.parametrize("shared", [True, False], ids=["shared", "no_shared"])
@pytest.mark.parametrize("M", [1, 8, 16, 17, 32])
def test_nvfp4_tc_layer_matches_oracle(moe, M, shared):
    shape = _shape(M, shared)
    inp = synth.make_layer(shape, 2000 + M, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, layer, ws = _run(moe, inp, err=err)
    assert moe.moe_decode_layer_launches(layer, M) == 3
    assert int(err.item()) == 0
    _, ref_b, bad = H.oracle_layer(inp)
    assert bad == 0
    rl2, mx = H.compare_bf16(out, ref_b)
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS, (rl2, mx)

    view = moe.workspace_view(layer, M, ws)
    rid, _ = oracle.topk_softmax(inp.logits.cpu().numpy(), shape.top_k)
    np.testing.assert_array_equal(view["topk_ids"].cpu().numpy(), rid.ravel())
    tables = oracle.align(rid.ravel(), shape.E, shape.BS)
    for key in ("sorted_token_ids", "expert_offsets", "token_to_perm", "sorted_expert_ids",
                "active_experts"):
        np.testing.assert_array_equal(view[key].cpu().numpy(), tables[key], err_msg=key)
    real = tables["sorted_token_ids"] < shape.n
    X = H.oracle_experts(inp.experts.to("cpu"))
    S = H.oracle_experts(inp.shared.to("cpu")) if shared else None
    h_ref, hs_ref = oracle.grouped_gate_up(X, S, synth.bf16_bits(inp.x), M, shape.top_k, tables)
    h_gpu = view["h"].cpu().numpy().astype(np.float64)
    assert H.rel_l2(h_gpu[real], h_ref[real]) < F4_H_REL_L2
    hs_gpu = view["h_shared"].cpu().numpy().astype(np.float64) if shared else None
    if shared:
        assert H.rel_l2(hs_gpu, hs_ref) < H.STAGE_REL_L2
    y_ref, ys_ref = oracle.grouped_down(X, S, h_gpu, hs_gpu, M, shape.top_k, tables)
    y_gpu = view["y"].cpu().numpy().astype(np.float64)
    assert H.rel_l2(y_gpu[real], y_ref[real]) < F4_Y_REL_L2
    if shared:
        assert H.rel_l2(view["y_shared"].cpu().numpy(), ys_ref) < H.STAGE_REL_L2


@pytest.mark.parametrize("M", [8, 20], ids=["16_columns", "32_columns"])
def test_nvfp4_tc_tables(moe, M):
    """The x table holds each token's x times its power of two exactly; the
    active table is {run offset, expert, slot count, 0}; the h terms give h
    back within 2^-21 of each (row, 128-column block) maximum."""
    shape = _shape(M)
    inp = synth.make_layer(shape, 777, device="cuda")
    _, layer, ws = _run(moe, inp)
    view = moe.workspace_view(layer, M, ws)
    nt = 16 if M <= 16 else 32
    table = view["tc_x_table"].to(torch.float64)             # [H/128][2][nt][64]
    assert table.shape == (shape.H // 128, 2, nt, 64)
    xt = table.permute(2, 0, 1, 3).reshape(nt, shape.H)[:M]
    xs = view["tc_x_scale"][:M].to(torch.float64)
    assert torch.all(xs > 0)
    assert torch.equal(xt * xs[:, None], inp.x.to(torch.float64))
    # each token's scale puts its largest |x| in [2^14, 2^15)
    amax = xt.abs().amax(dim=1)
    assert torch.all((amax >= 2.0 ** 14) & (amax < 2.0 ** 15))

    tables = oracle.align(view["topk_ids"].cpu().numpy(), shape.E, shape.BS)
    A = int(tables["active_count"][0])
    act = tables["active_experts"][:A]
    items = view["tc_items"][:A].cpu().numpy()
    np.testing.assert_array_equal(items[:, 1], act)
    np.testing.assert_array_equal(items[:, 0], tables["expert_offsets"][act])
    counts = np.bincount(view["topk_ids"].cpu().numpy(), minlength=shape.E)
    np.testing.assert_array_equal(items[:, 2], counts[act])
    np.testing.assert_array_equal(items[:, 3], 0)

    real = torch.as_tensor(np.nonzero(tables["sorted_token_ids"] < shape.n)[0], device="cuda")
    h = view["h"][real].to(torch.float64)                    # [rows][I]
    hq = view["tc_h_terms"][:, real].to(torch.float64)       # [2][rows][I]
    hsc = view["tc_h_scale"][real].to(torch.float64)         # [rows][I/128]
    back = (hq[0] + hq[1]) * hsc.repeat_interleave(128, dim=1)
    blk = h.abs().view(h.shape[0], -1, 128).amax(dim=2).repeat_interleave(128, dim=1)
    assert torch.all((back - h).abs() <= blk * 2.0 ** -21)
    # the hi term is h's f16 rounding under the scale, lo the rest's
    hi_f = (h / hsc.repeat_interleave(128, dim=1)).to(torch.float16).to(torch.float64)
    assert torch.equal(hq[0], hi_f)


@pytest.mark.parametrize("pair", [(32, 1), (17, 1), (16, 1), (16, 5), (32, 17)],
                         ids=lambda p: f"m{p[0]}_vs_m{p[1]}")
def test_nvfp4_tc_row_invariance(moe, pair):
    """The first rows' output bits are the same in a batch of M rows as in a
    batch of fewer (16 and 32 token columns alike)."""
    big, small = pair
    inp = synth.make_layer(_shape(big), 4100, device="cuda")
    out_b, _, _ = _run(moe, inp)
    few = synth.LayerInputs(_shape(small), inp.x[:small].contiguous(),
                            inp.logits[:small].contiguous(), inp.experts, inp.shared)
    out_s, _, _ = _run(moe, few)
    assert torch.equal(out_b[:small].view(torch.int16), out_s.view(torch.int16))


@pytest.mark.parametrize("M", [1, 8, 32])
def test_nvfp4_tc_gated_shared_expert(moe, M):
    """A gated shared expert: the kernel computes each token's gate
    sigmoid(x[t] . gate_w) into the workspace and blends g[t] * y_sh[t]."""
    shape = _shape(M)
    inp = synth.make_layer(shape, 1000, device="cuda")
    gate = synth.make_shared_gate(shape.H, 77, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, layer, ws = _run(moe, inp, gate=gate, err=err)
    assert int(err.item()) == 0
    X = H.oracle_experts(inp.experts.to("cpu"))
    S = H.oracle_experts(inp.shared.to("cpu"))
    _, ref_b, bad = oracle.moe_layer(X, S, synth.bf16_bits(inp.x), M, shape.top_k, shape.BS,
                                     logits=inp.logits.cpu().numpy(),
                                     shared_gate_bits=synth.bf16_bits(gate))
    assert bad == 0
    rl2, mx = H.compare_bf16(out, ref_b)
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS, (rl2, mx)
    g_ref = oracle.shared_gate(synth.bf16_bits(inp.x), synth.bf16_bits(gate))
    g = moe.workspace_view(layer, M, ws)["shared_gate"].cpu().numpy()
    np.testing.assert_allclose(g, g_ref, rtol=0, atol=GATE_ABS)


@pytest.mark.parametrize("gated", [False, True], ids=["plain", "gated"])
def test_nvfp4_one_workspace_serves_alternating_rows(moe, gated):
    """A workspace sized for M = 40 serves calls at 8, 1, 32, 40 (the CUDA
    cores), 17 and 8: each output is the bits of the same call on a fresh
    zeroed workspace (the token flags and counters keep their place)."""
    base = synth.make_layer(_shape(40), 3100, device="cuda")
    gate = synth.make_shared_gate(2048, 78, device="cuda") if gated else None
    routed = moe.Experts.from_synth(base.experts)
    shared = moe.Experts.from_synth(base.shared)
    layer = moe.LayerDesc(top_k=8, block_size=16, routed=routed, shared=shared,
                          shared_gate=gate)
    shared_ws = moe.alloc_workspace(layer, 40)
    for call, M in enumerate((8, 1, 32, 40, 17, 8)):
        x = synth.make_x(M, 2048, 3200 + call, "cuda")
        lg = synth.make_logits(M, 128, 3300 + call, "cuda")
        fresh = torch.empty(M, 2048, dtype=torch.bfloat16, device="cuda")
        moe.moe_decode_layer(layer, x, fresh, moe.alloc_workspace(layer, M), router_logits=lg)
        out = torch.full((M, 2048), float("nan"), dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.moe_decode_layer(layer, x, out, shared_ws, router_logits=lg, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, (call, M)
        assert torch.equal(out.view(torch.int16), fresh.view(torch.int16)), (call, M)


def test_nvfp4_tc_graph_replay(moe):
    """The layer captured once in a CUDA graph and replayed on new logits
    gives the bits of an eager call on the same logits."""
    shape = _shape(8)
    inp = synth.make_layer(shape, 1000, device="cuda")
    out_a, layer, ws = _run(moe, inp)
    out_b, _, _ = _run(moe, inp, ws=ws)
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
    eager_ws = moe.alloc_workspace(layer, shape.M)
    for seed in (5, 6, 7):
        logits.copy_(synth.make_logits(shape.M, shape.E, seed, device="cuda"))
        g.replay()
        torch.cuda.synchronize()
        eager = torch.empty_like(out)
        moe.moe_decode_layer(layer, inp.x, eager, eager_ws, router_logits=logits)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16)), seed


@pytest.mark.parametrize("M", [4, 32])
def test_nvfp4_tc_decode_experts(moe, M):
    """moe_decode_experts on the tables an earlier call left: the same bits
    on the same x, and on another x the bits of a whole layer call on it."""
    shape = _shape(M)
    inp = synth.make_layer(shape, 5150, device="cuda")
    out, layer, ws = _run(moe, inp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    again = torch.full_like(out, float("nan"))
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


def test_nvfp4_tc_new_scales_under_the_same_codes(moe):
    """Two expert sets that share their code tensors but not their scale
    tensors, run one after the other on one workspace: each output matches
    the oracle of its own scales (the kernel's tensor maps are keyed by every
    address they hold, scales included)."""
    shape = _shape(4, shared=False)
    inp = synth.make_layer(shape, 6100, device="cuda")
    other = synth.make_experts(shape.E, shape.H, shape.I, shape.fmt, 6200, "cuda")

    def with_scales(src, scales_from):
        def proj(p, q):
            return synth.ProjData(p.fmt, p.rows, p.cols, p.codes, q.scale.clone(), p.glob)
        return synth.ExpertData(src.E, src.H, src.I, src.fmt, proj(src.gate, scales_from.gate),
                                proj(src.up, scales_from.up), proj(src.down, scales_from.down))

    ws = None
    for ex in (inp.experts, with_scales(inp.experts, other)):
        cur = synth.LayerInputs(shape, inp.x, inp.logits, ex, None)
        out, _, ws = _run(moe, cur, ws=ws)
        _, ref_b, _ = H.oracle_layer(cur)
        rl2, mx = H.compare_bf16(out, ref_b)
        assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS, (rl2, mx)
