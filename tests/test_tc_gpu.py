"""The tensor-core (tcgen05) expert path of the decode MoE layer against the
oracle, in both its forms: up to 16 rows the gate+up MMAs take the 16 token
columns of a per-token x-term table (no grid barrier before the first
copies), above that the item's own rows of x terms by sorted position.

The path multiplies the E4M3 weight codes by E4M3 splits of the activations
(x = t0 + t1 exactly, h = t0 + t1 + t2 to 12 significant bits, each with a
power-of-two scale) and promotes every 128-wide k block to fp32 times its
block scale.  Checked here: the layer output within the workload's tolerance
on the tiny, decode and verify shapes; h against the oracle's gate+up on the
same x; y against the oracle's down of the layer's own h; the split of x exact
and the split of h within its bound; ragged row tiles (16/17 rows, a full
64-row tile plus one row, two tiles of one expert); run-to-run bit equality and
CUDA-graph replay."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu

TC = 2
STAGED = 3

# h: exact x and weight codes, fp32 promotion of each 128-wide k block; the
# same fp32 accumulation error as the CUDA-core path (see helpers).
TC_H_REL_L2 = H.STAGE_REL_L2
# y: its input h is carried as three E4M3 terms, at most 2^-12 relative plus
# 2^-10 of the (row, block) scale per element, so y's relative L2 error is at
# most about 2.4e-4; 5e-4 leaves 2x margin.
TC_Y_REL_L2 = 5e-4


@pytest.fixture(scope="module")
def moe():
    import expert_routing_alignment_gb300 as m
    m.load()
    return m


def _shape(name, M, H_, I, E, k, BS):
    return synth.LayerShape(name, M, H_, I, E, k, BS, synth.FMT_FP8)


SHAPES = [synth.tiny(), synth.decode_fp8(1), synth.decode_fp8(8), synth.decode_fp8(16),
          _shape("decode_h4096_i1536_e64_k8_fp8_m5", 5, 4096, 1536, 64, 8, 16),
          _shape("decode_h2048_i768_e128_k8_fp8_m17", 17, 2048, 768, 128, 8, 16),
          _shape("decode_h2048_i768_e128_k8_fp8_m64", 64, 2048, 768, 128, 8, 16)]


def _tables_and_real(view, shape):
    tables = oracle.align(view["topk_ids"].cpu().numpy(), shape.E, shape.BS)
    return tables, tables["sorted_token_ids"] < shape.n


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_tc_layer_matches_oracle(moe, shape):
    inp = synth.make_layer(shape, 1000, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, view, (layer, _) = H.gpu_layer(moe, inp, path=TC, err=err)
    assert moe.moe_decode_layer_launches(layer, shape.M) == 3
    assert int(err.item()) == 0
    _, ref_b, bad = H.oracle_layer(inp)
    assert bad == 0
    rl2, mx = H.compare_bf16(out, ref_b)
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS, (rl2, mx)

    # the kernel's own routing and alignment tables equal the oracle's
    rid, rw = oracle.topk_softmax(inp.logits.cpu().numpy(), shape.top_k)
    np.testing.assert_array_equal(view["topk_ids"].cpu().numpy(), rid.ravel())
    np.testing.assert_allclose(view["topk_w"].cpu().numpy(), rw.ravel(), atol=H.TOPK_W_ABS)
    tables, real = _tables_and_real(view, shape)
    for key in ("sorted_token_ids", "expert_offsets", "token_to_perm", "sorted_expert_ids",
                "active_experts"):
        np.testing.assert_array_equal(view[key].cpu().numpy(), tables[key], err_msg=key)
    assert int(view["active_count"].item()) == int(tables["active_count"][0])
    assert int(view["num_tokens_post_padded"].item()) == int(tables["num_tokens_post_padded"][0])
    X = H.oracle_experts(inp.experts.to("cpu"))
    h_ref, _ = oracle.grouped_gate_up(X, None, synth.bf16_bits(inp.x), shape.M, shape.top_k,
                                      tables)
    h_gpu = view["h"].cpu().numpy().astype(np.float64)
    assert H.rel_l2(h_gpu[real], h_ref[real]) < TC_H_REL_L2
    y_ref, _ = oracle.grouped_down(X, None, h_gpu, None, shape.M, shape.top_k, tables)
    y_gpu = view["y"].cpu().numpy().astype(np.float64)
    assert H.rel_l2(y_gpu[real], y_ref[real]) < TC_Y_REL_L2


def _e4m3(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.float8_e4m3fn).to(torch.float64)


@pytest.mark.parametrize("M", [8, 32], ids=["token_form", "row_form"])
def test_tc_x_terms_exact_and_h_terms_bounded(moe, M):
    shape = _shape(f"decode_h2048_i768_e128_k8_fp8_m{M}", M, 2048, 768, 128, 8, 16)
    inp = synth.make_layer(shape, 321, device="cuda")
    _, view, _ = H.gpu_layer(moe, inp, path=TC)
    tables, real = _tables_and_real(view, shape)
    pos = np.nonzero(real)[0]
    tok = tables["sorted_token_ids"][pos] // shape.top_k
    pos_t = torch.as_tensor(pos, device="cuda")
    # the active table the alignment wrote for the tensor-core kernels:
    # {run offset, expert, slot count, 0} per active expert
    A = int(tables["active_count"][0])
    act = tables["active_experts"][:A]
    items = view["tc_items"][:A].cpu().numpy()
    np.testing.assert_array_equal(items[:, 1], act)
    np.testing.assert_array_equal(items[:, 0], tables["expert_offsets"][act])
    counts = np.bincount(view["topk_ids"].cpu().numpy(), minlength=shape.E)
    np.testing.assert_array_equal(items[:, 2], counts[act])
    if M > 16:
        _check_x_terms(view, inp, pos_t, tok)
    else:   # the token table: token t's terms are x[t] times its scale
        table = view["tc_x_table"]                       # [H/128][2][16][128]
        xq = table.permute(1, 2, 0, 3).reshape(2, 16, shape.H)[:, :M]
        _check_x_terms(dict(tc_x_terms=xq, tc_x_scale=view["tc_x_scale"][:M]), inp,
                       torch.arange(M, device="cuda"), np.arange(M))
    _check_h_terms(view, shape, pos_t, len(pos))


def _check_x_terms(view, inp, pos_t, tok):
    # x: (t0 + t1) * xs == x exactly where |x| * 2^s >= 2^-2, and within 2^-10
    # of the scale elsewhere; the row maximum lands in [128, 256)
    xq = view["tc_x_terms"][:, pos_t]
    xs = view["tc_x_scale"][pos_t].to(torch.float64)[:, None]
    rec = (_e4m3(xq[0]) + _e4m3(xq[1])) * xs
    x = inp.x[torch.as_tensor(tok, device="cuda")].to(torch.float64)
    scaled = x.abs() / xs
    big = scaled >= 0.25
    assert bool((rec[big] == x[big]).all())
    assert bool(((rec - x).abs() <= xs * 2.0 ** -10).all())
    mx = scaled.amax(dim=1)
    assert bool(((mx >= 128) & (mx < 256)).all())


def _check_h_terms(view, shape, pos_t, npos):
    # h: |sum of three terms * hs - h| <= 2^-12 |h| + 2^-10 hs per (row, block)
    I = shape.I
    hq = view["tc_h_terms"][:, pos_t]
    hs = view["tc_h_scale"][pos_t].to(torch.float64).repeat_interleave(128, dim=1)
    rec = (_e4m3(hq[0]) + _e4m3(hq[1]) + _e4m3(hq[2])) * hs
    h = view["h"][pos_t].to(torch.float64)
    assert rec.shape == h.shape == (npos, I)
    assert bool(((rec - h).abs() <= h.abs() * 2.0 ** -12 + hs * 2.0 ** -10).all())
    bmax = (h.abs() / hs).reshape(npos, I // 128, 128).amax(dim=2)
    assert bool(((bmax >= 128) & (bmax < 256)).all())


@pytest.mark.parametrize("rows", [(1,), (16,), (7, 9), (16, 17), (64, 1), (65, 63), (128,)],
                         ids=str)
def test_tc_row_tile_edges(moe, rows):
    """Given ids (top_k = 1): expert 3 takes rows[0] tokens, expert 5 the next
    rows[1], and so on -- item boundaries at 16-row MMA steps and 64-row tiles
    (M <= 16: the token form's 16-row items)."""
    M = sum(rows)
    shape = _shape(f"tc_edges_m{M}", M, 256, 512, 8, 1, 16)
    inp = synth.make_layer(shape, 55, device="cuda")
    ids = np.concatenate([np.full(r, e, np.int32) for r, e in zip(rows, (3, 5, 6))])[:, None]
    w = np.ones((M, 1), np.float32)
    ids_t = torch.as_tensor(ids, device="cuda")
    w_t = torch.as_tensor(w, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, view, _ = H.gpu_layer(moe, inp, path=TC, use_logits=False, ids=ids_t, w=w_t, err=err)
    assert int(err.item()) == 0
    _, ref_b, bad = H.oracle_layer(inp, ids=ids, w=w.astype(np.float64))
    assert bad == 0
    rl2, mx = H.compare_bf16(out, ref_b)
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS, (rl2, mx)


def test_tc_repeated_expert_in_a_token(moe):
    """Given ids that list one expert twice in every token (top_k = 2, M = 16):
    the expert's run holds 32 rows, two 16-row items of the token form, each
    row taking its token's column."""
    M = 16
    shape = _shape("tc_repeat_m16", M, 2048, 768, 16, 2, 16)
    inp = synth.make_layer(shape, 57, device="cuda")
    ids = np.full((M, 2), 3, np.int32)
    ids[::3, 1] = 7
    w = np.full((M, 2), 0.5, np.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, view, _ = H.gpu_layer(moe, inp, path=TC, use_logits=False,
                               ids=torch.as_tensor(ids, device="cuda"),
                               w=torch.as_tensor(w, device="cuda"), err=err)
    assert int(err.item()) == 0
    _, ref_b, bad = H.oracle_layer(inp, ids=ids, w=w.astype(np.float64))
    assert bad == 0
    rl2, mx = H.compare_bf16(out, ref_b)
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS, (rl2, mx)


@pytest.mark.parametrize("M", [8, 32], ids=["token_form", "row_form"])
def test_tc_deterministic_and_graph_replayable(moe, M):
    shape = _shape(f"decode_h2048_i768_e128_k8_fp8_m{M}", M, 2048, 768, 128, 8, 16)
    inp = synth.make_layer(shape, 9, device="cuda")
    out1, _, (layer, ws) = H.gpu_layer(moe, inp, path=TC)
    out2 = torch.empty_like(out1)
    moe.moe_decode_layer(layer, inp.x, out2, ws, router_logits=inp.logits)
    torch.cuda.synchronize()
    assert bool((out1.view(torch.int16) == out2.view(torch.int16)).all())
    # one captured graph, replayed on fresh logits, equals direct calls
    lg = inp.logits.clone()
    out3 = torch.empty_like(out1)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        moe.moe_decode_layer(layer, inp.x, out3, ws, router_logits=lg)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        moe.moe_decode_layer(layer, inp.x, out3, ws, router_logits=lg)
    lg.copy_(synth.make_logits(shape.M, shape.E, 77, device="cuda"))
    with torch.cuda.stream(st):
        g.replay()
    st.synchronize()
    ref = torch.empty_like(out1)
    moe.moe_decode_layer(layer, inp.x, ref, ws, router_logits=lg)
    torch.cuda.synchronize()
    assert bool((out3.view(torch.int16) == ref.view(torch.int16)).all())


def test_tc_verify_batch_matches_staged_path(moe):
    """The M = 128 verify batch (E = 256, H = 4096, I = 1536, BS = 64, Zipf
    bias) takes the tensor-core path by default; its output agrees with the
    CUDA-core staged path's within the layer tolerance on every row (the
    oracle checks sampled rows in test_layer_gpu)."""
    shape = synth.verify_fp8(128)
    inp = synth.make_layer(shape, 1000, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_tc, view, (layer, _) = H.gpu_layer(moe, inp, err=err)
    assert moe.moe_decode_layer_launches(layer, shape.M) == 3
    assert int(err.item()) == 0
    assert "tc_x_terms" in view
    out_st, _, _ = H.gpu_layer(moe, inp, path=STAGED)
    rl2, mx = H.compare_bf16(out_tc, synth.bf16_bits(out_st))
    assert rl2 < H.LAYER_REL_L2 and mx < H.LAYER_MAX_ABS, (rl2, mx)


@pytest.mark.parametrize("M,m", [(8, 1), (8, 4), (4, 1), (4, 3), (5, 2), (16, 1), (16, 5),
                                 (64, 17), (64, 1), (128, 33)], ids=str)
def test_tc_row_invariance(moe, M, m):
    """On the tensor-core path the first m rows' output bits are the same
    whether the batch has m or M rows, across the token form (M <= 16) and
    the row form alike: each row has its own x scale (its token's), every MMA
    column is one row or one token, and promotion, SiLU, the h scales and the
    blend are per row."""
    shape = _shape(f"decode_h2048_i768_e128_k8_fp8_m{M}", M, 2048, 768, 128, 8, 16)
    inp = synth.make_layer(shape, 1000, device="cuda")
    out_m, _, _ = H.gpu_layer(moe, inp, path=TC)
    few = synth.LayerInputs(
        synth.LayerShape(shape.name + f"_rows{m}", m, shape.H, shape.I, shape.E, shape.top_k,
                         shape.BS, shape.fmt),
        inp.x[:m].contiguous(), inp.logits[:m].contiguous(), inp.experts)
    out_1, _, _ = H.gpu_layer(moe, few, path=TC)
    assert torch.equal(out_m[:m].view(torch.int16), out_1.view(torch.int16))
