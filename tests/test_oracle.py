"""Pins of the CPU oracle against what the pages and mathematics fix (CPU only).

Every oracle function is checked against something other than itself:
published format tables (tests/golden), library routines (torch's float8
decoding, float64 matmul, softmax, topk), brute force on every tiny routing,
the worst-case-size closed form, invariants, and special cases that reduce to
a dense FFN or a single token.
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import helpers

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                a, b = line.split()
                rows.append((int(a, 0), float(b)))
    return rows


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def test_e2m1_matches_ocp_table():
    for code, val in _golden("e2m1_ocp_mx.txt"):
        got = oracle.e2m1_value(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code


def test_e4m3_special_values_match_ocp():
    for code, val in _golden("e4m3_ocp_fp8.txt"):
        got = oracle.e4m3_value(code)
        if math.isnan(val):
            assert math.isnan(got), code
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], c


def test_bf16_rne_matches_torch_on_float32_values():
    g = torch.Generator().manual_seed(5)
    v = torch.cat([torch.randn(4000, generator=g) * 10.0 ** torch.randint(-30, 30, (4000,),
                                                                           generator=g),
                   torch.tensor([0.0, -0.0, 1e-40, -3e-39, 3.3e38, -3.4e38, float("inf")])])
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round_array(v.to(torch.float64).numpy())
    np.testing.assert_array_equal(got, ref)


def test_bf16_rne_closed_form_cases():
    # ties go to the even neighbour; a hair above a tie rounds up (single
    # rounding from double); overflow past the largest finite value -> inf
    assert oracle.bf16_rne(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.bf16_rne(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert oracle.bf16_rne(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.bf16_rne(-(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 0xBF81
    assert oracle.bf16_rne(2.0 ** 128) == 0x7F80
    assert oracle.bf16_rne((2 - 2.0 ** -7) * 2.0 ** 127) == 0x7F7F
    assert oracle.bf16_rne(2.0 ** -133) == 0x0001          # smallest subnormal
    assert oracle.bf16_rne(2.0 ** -134) == 0x0000          # tie -> even (zero)


def test_dequant_fp8_matches_torch():
    g = torch.Generator().manual_seed(11)
    w = torch.randn(256, 384, generator=g) * 0.02
    codes, scale = synth.encode_fp8_b128(w)
    p = synth.ProjData(synth.FMT_FP8, 256, 384, codes[None], scale[None])
    got = oracle.dequant(helpers.oracle_proj(p), 0)
    ref = helpers.torch_dequant(p, 0).numpy()
    np.testing.assert_array_equal(got, ref)
    # the block scale is per 128x128 block: perturbing one block's scale
    # changes exactly that block
    s2 = scale.clone()
    s2[1, 2] *= 2
    p2 = synth.ProjData(synth.FMT_FP8, 256, 384, codes[None], s2[None])
    d = oracle.dequant(helpers.oracle_proj(p2), 0) != got
    mask = np.zeros_like(d)
    mask[128:256, 256:384] = codes.numpy()[128:256, 256:384] != 0
    np.testing.assert_array_equal(d, mask)


def test_dequant_nvfp4_matches_table_and_torch():
    g = torch.Generator().manual_seed(12)
    packed = torch.randint(0, 256, (2, 32, 64), generator=g, dtype=torch.int32).to(torch.uint8)
    # scales: finite positive E4M3 codes
    s16 = torch.randint(0x08, 0x78, (2, 32, 8), generator=g, dtype=torch.int32).to(torch.uint8)
    glob = torch.tensor([0.5, 3.0e-4])
    p = synth.ProjData(synth.FMT_NVFP4, 32, 128, packed, s16, glob)
    for e in range(2):
        got = oracle.dequant(helpers.oracle_proj(p), e)
        ref = helpers.torch_dequant(p, e).numpy()
        np.testing.assert_allclose(got, ref, rtol=1e-7, atol=0)
    # element order: even element in the low nibble
    single = torch.zeros((1, 1, 16), dtype=torch.uint8)
    single[0, 0, 0] = 0x72          # element 0 -> code 2 (1.0), element 1 -> code 7 (6.0)
    p1 = synth.ProjData(synth.FMT_NVFP4, 1, 32, single, torch.full((1, 1, 2), 0x38,
                                                                    dtype=torch.uint8),
                        torch.tensor([1.0]))
    row = oracle.dequant(helpers.oracle_proj(p1), 0)[0]
    assert row[0] == 1.0 and row[1] == 6.0 and not row[2:].any()


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------

def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_router_logits_match_torch_matmul():
    """The router's logits equal a float64 matmul of the bf16 values (library
    routine), for several shapes including the decode and verify widths."""
    g = torch.Generator().manual_seed(3)
    for M, H, E in [(1, 64, 8), (4, 256, 8), (8, 2048, 128), (3, 4096, 256)]:
        x = torch.randn(M, H, generator=g).to(torch.bfloat16)
        W = (torch.randn(E, H, generator=g) * 0.02).to(torch.bfloat16)
        got = oracle.router_logits(_bits(x), _bits(W))
        ref = (x.double() @ W.double().T).numpy()
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_router_logits_closed_form():
    """Exact cases: one-hot rows pick out a weight column; small-integer
    operands give exact integer dot products; the order of the rows and of
    the experts is kept (a transposed operand would fail)."""
    M, H, E = 3, 40, 5
    x = np.zeros((M, H), np.float32)
    x[0, 7] = 1.0
    x[1, 0] = 2.0
    x[2] = np.arange(H) % 5 - 2
    W = (np.arange(E * H).reshape(E, H) % 7 - 3).astype(np.float32)
    xb = _bits(torch.from_numpy(x).to(torch.bfloat16))
    Wb = _bits(torch.from_numpy(W).to(torch.bfloat16))
    got = oracle.router_logits(xb, Wb)
    np.testing.assert_array_equal(got[0], W[:, 7])
    np.testing.assert_array_equal(got[1], 2.0 * W[:, 0])
    want2 = [sum(int(x[2, c]) * int(W[e, c]) for c in range(H)) for e in range(E)]
    np.testing.assert_array_equal(got[2], np.array(want2, np.float64))


def test_topk_softmax_matches_torch():
    g = torch.Generator().manual_seed(3)
    lg = torch.randn(64, 128, generator=g)
    ids, w = oracle.topk_softmax(lg.numpy(), 8)
    rid, rw = helpers.torch_route(lg, 8)
    np.testing.assert_array_equal(ids, rid.numpy())
    np.testing.assert_allclose(w, rw.numpy(), rtol=1e-13, atol=0)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-12)


def test_topk_ties_take_lower_id_brute_force():
    rng = np.random.default_rng(4)
    for _ in range(200):
        E = int(rng.integers(2, 9))
        k = int(rng.integers(1, E + 1))
        lg = rng.integers(-2, 3, size=(1, E)).astype(np.float32)   # many ties
        ids, w = oracle.topk_softmax(lg, k)
        ref = sorted(range(E), key=lambda e: (-lg[0, e], e))[:k]
        assert list(ids[0]) == ref
        p = np.exp(lg[0].astype(np.float64) - lg[0].max())
        np.testing.assert_allclose(w[0], p[ref] / p[ref].sum(), rtol=1e-14)


# --------------------------------------------------------------------------
# alignment
# --------------------------------------------------------------------------

def brute_align(ids, E, BS):
    """A differently written reference: Python's stable sort of the slots by
    expert, then the tables read off the sorted order."""
    n = len(ids)
    valid = [i for i in range(n) if 0 <= ids[i] < E]
    order = sorted(valid, key=lambda i: (ids[i], i))
    counts = [sum(1 for i in valid if ids[i] == e) for e in range(E)]
    padded = [-(-c // BS) * BS for c in counts]
    offsets = [sum(padded[:e]) for e in range(E + 1)]
    total = offsets[E]
    max_total = -(-min(n * BS, n + E * (BS - 1)) // BS) * BS
    sti = [n] * max_total
    ttp = [-1] * n
    for e in range(E):
        run = [i for i in order if ids[i] == e]
        for r, i in enumerate(run):
            sti[offsets[e] + r] = i
            ttp[i] = offsets[e] + r
    sei = []
    for b in range(max_total // BS):
        owner = -1
        for e in range(E):
            if offsets[e] <= b * BS < offsets[e] + padded[e]:
                owner = e
        sei.append(owner)
    cap = min(n, E)
    act = [e for e in range(E) if counts[e] > 0]
    return dict(sorted_token_ids=sti, sorted_expert_ids=sei, expert_offsets=offsets,
                token_to_perm=ttp, active_experts=act + [-1] * (cap - len(act)),
                active_count=len(act), num_tokens_post_padded=total)


def _check_same(got, ref):
    for key in ("sorted_token_ids", "sorted_expert_ids", "expert_offsets", "token_to_perm",
                "active_experts"):
        assert list(got[key]) == list(ref[key]), key
    assert int(got["active_count"][0]) == ref["active_count"]
    assert int(got["num_tokens_post_padded"][0]) == ref["num_tokens_post_padded"]


def test_align_every_routing_of_three_tokens_brute_force():
    E = 4
    for M in (1, 2, 3):
        for k in (1, 2):
            per_token = list(itertools.permutations(range(E), k))
            for routing in itertools.product(per_token, repeat=M):
                ids = [e for tok in routing for e in tok]
                for BS in (1, 2, 3, 4, 16):
                    _check_same(oracle.align(np.array(ids), E, BS), brute_align(ids, E, BS))


def test_align_arbitrary_ids_with_repeats_brute_force():
    E = 4
    for n in range(0, 5):
        for ids in itertools.product(range(E), repeat=n):
            for BS in (1, 3, 4):
                _check_same(oracle.align(np.array(ids, dtype=np.int64), E, BS),
                            brute_align(list(ids), E, BS))


def test_align_out_of_range_ids_skipped():
    ids = [3, -1, 0, 7, 3, 2**40]
    got = oracle.align(np.array(ids, dtype=np.int64), 4, 2)
    _check_same(got, brute_align(ids, 4, 2))
    assert got["bad"] == 3
    assert list(got["token_to_perm"][[1, 3, 5]]) == [-1, -1, -1]


def check_align_invariants(ids, E, BS, t):
    n = len(ids)
    max_total = -(-min(n * BS, n + E * (BS - 1)) // BS) * BS
    assert t["max_total"] == max_total
    assert t["sorted_token_ids"].size == max_total
    off = t["expert_offsets"].astype(np.int64)
    counts = np.bincount(ids, minlength=E)
    total = int(sum(-(-c // BS) * BS for c in counts))
    assert off[E] == total == int(t["num_tokens_post_padded"][0]) <= max_total
    assert (off % BS == 0).all() and (np.diff(off) >= 0).all()
    sti = t["sorted_token_ids"]
    real = sti[sti < n]
    # every slot exactly once, every other position the sentinel
    assert sorted(real.tolist()) == list(range(n))
    assert ((sti == n) | (sti < n)).all()
    for e in np.nonzero(counts)[0]:
        run = sti[off[e]: off[e] + counts[e]]
        assert (ids[run] == e).all()                  # contiguous run of expert e
        assert (np.diff(run) > 0).all()               # ascending: the stable order
        assert (sti[off[e] + counts[e]: off[e + 1]] == n).all()
    ttp = t["token_to_perm"]
    assert (sti[ttp] == np.arange(n)).all()           # inverse on real entries
    act = t["active_experts"]
    cnt = int(t["active_count"][0])
    assert act[:cnt].tolist() == np.nonzero(counts)[0].tolist()
    assert (act[cnt:] == -1).all() and act.size == min(n, E)
    sei = t["sorted_expert_ids"]
    for b in range(sei.size):
        e = sei[b]
        if b * BS >= total:
            assert e == -1
        else:
            assert off[e] <= b * BS < off[e + 1]


@pytest.mark.parametrize("M,E,BS,dist", [
    (1, 64, 16, "uniform"), (64, 256, 64, "zipf"), (64, 1024, 128, "uniform"),
    (1024, 256, 16, "zipf"), (1024, 64, 128, "one"), (4096, 1024, 64, "uniform"),
    (4096, 1024, 128, "zipf"),
])
def test_align_invariants_stress_shapes(M, E, BS, dist):
    ids = synth.align_ids(8 * M, E, dist, seed=M + E + BS)
    check_align_invariants(ids, E, BS, oracle.align(ids, E, BS))


@pytest.mark.parametrize("e", [0, 63])
def test_align_all_one_expert(e):
    n, E, BS = 8 * 64, 64, 16
    t = oracle.align(np.full(n, e, dtype=np.int64), E, BS)
    assert int(t["num_tokens_post_padded"][0]) == -(-n // BS) * BS
    assert int(t["active_count"][0]) == 1 and t["active_experts"][0] == e
    assert t["sorted_token_ids"][:n].tolist() == list(range(n))
    assert t["expert_offsets"][: e + 1].tolist() == [0] * (e + 1)


def test_align_sizes_closed_form():
    for n in (0, 1, 8, 64, 1000, 32768):
        for E in (1, 4, 64, 1024):
            for BS in (1, 16, 64, 128):
                mt, mb, cap = oracle.align_sizes(n, E, BS)
                # min(n*BS, n+E*(BS-1)) = n + min(n, E)*(BS-1), already rounded
                assert mt == n + min(n, E) * (BS - 1) or mt == -(-(n + min(n, E) * (BS - 1))
                                                            // BS) * BS
                assert mt % BS == 0 and mb * BS == mt and cap == min(n, E)


# --------------------------------------------------------------------------
# expert FFN and layer
# --------------------------------------------------------------------------

def _small_inputs(fmt, shared, M=4, H=256, I=256, E=8, k=2, seed=21):
    shape = synth.LayerShape("t", M, H, I, E, k, 16, fmt, shared_I=128 if shared else None)
    return synth.make_layer(shape, seed)


# (the nvfp4-gate-up tier: NVFP4 gate and up, FP8 down, with an FP8 shared expert)
FMT_CASES = [(synth.FMT_FP8, False), (synth.FMT_NVFP4, True), (synth.FMT_NVFP4_GATE_UP, True)]


@pytest.mark.parametrize("fmt,shared", FMT_CASES)
def test_grouped_stages_match_torch(fmt, shared):
    inp = _small_inputs(fmt, shared)
    s = inp.shape
    X = helpers.oracle_experts(inp.experts)
    S = helpers.oracle_experts(inp.shared) if shared else None
    ids, w = oracle.topk_softmax(inp.logits.numpy(), s.top_k)
    t = oracle.align(ids.ravel(), s.E, s.BS)
    xb = synth.bf16_bits(inp.x)
    h, h_sh = oracle.grouped_gate_up(X, S, xb, s.M, s.top_k, t)
    y, y_sh = oracle.grouped_down(X, S, h, h_sh, s.M, s.top_k, t)
    x64 = inp.x.to(torch.float64)
    for p in range(t["max_total"]):
        slot = int(t["sorted_token_ids"][p])
        if slot >= s.n:
            continue
        e = int(ids.ravel()[slot])
        xt = x64[slot // s.top_k: slot // s.top_k + 1]
        g = xt @ helpers.torch_dequant(inp.experts.gate, e).T
        u = xt @ helpers.torch_dequant(inp.experts.up, e).T
        href = (torch.nn.functional.silu(g) * u)[0]
        np.testing.assert_allclose(h[p], href.numpy(), rtol=1e-10, atol=1e-12)
        yref = helpers.torch_ffn(inp.experts, e, xt)[0]
        np.testing.assert_allclose(y[p], yref.numpy(), rtol=1e-10, atol=1e-12)
    if shared:
        np.testing.assert_allclose(y_sh, helpers.torch_ffn(inp.shared, 0, x64).numpy(),
                                   rtol=1e-10, atol=1e-12)
    out_d, out_b = oracle.blend(y, w, t["token_to_perm"], y_sh, s.M, s.top_k, s.H)
    ref = helpers.torch_layer(inp)
    np.testing.assert_allclose(out_d, ref.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_array_equal(out_b, oracle.bf16_round_array(out_d))


@pytest.mark.parametrize("fmt,shared", FMT_CASES)
def test_layer_matches_torch(fmt, shared):
    inp = _small_inputs(fmt, shared, M=5, seed=33)
    s = inp.shape
    X = helpers.oracle_experts(inp.experts)
    S = helpers.oracle_experts(inp.shared) if shared else None
    out_d, out_b, bad = oracle.moe_layer(X, S, synth.bf16_bits(inp.x), s.M, s.top_k, s.BS,
                                         logits=inp.logits.numpy())
    assert bad == 0
    np.testing.assert_allclose(out_d, helpers.torch_layer(inp).numpy(), rtol=1e-10, atol=1e-12)


def test_layer_tiny_workload_matches_torch():
    inp = synth.make_layer(synth.tiny(), 1000)
    s = inp.shape
    out_d, _, _ = oracle.moe_layer(helpers.oracle_experts(inp.experts), None,
                                   synth.bf16_bits(inp.x), s.M, s.top_k, s.BS,
                                   logits=inp.logits.numpy())
    np.testing.assert_allclose(out_d, helpers.torch_layer(inp).numpy(), rtol=1e-10, atol=1e-12)


def test_layer_single_expert_is_dense_swiglu():
    # E = 1, k = 1: every token goes to expert 0 with weight 1 -> a dense
    # SwiGLU FFN, written here with torch.nn.functional.linear/silu
    inp = _small_inputs(synth.FMT_FP8, False, M=6, E=1, k=1, seed=44)
    s = inp.shape
    out_d, _, _ = oracle.moe_layer(helpers.oracle_experts(inp.experts), None,
                                   synth.bf16_bits(inp.x), s.M, 1, s.BS,
                                   logits=inp.logits.numpy())
    x = inp.x.to(torch.float64)
    F = torch.nn.functional
    wg, wu, wd = (helpers.torch_dequant(p, 0) for p in
                  (inp.experts.gate, inp.experts.up, inp.experts.down))
    ref = F.linear(F.silu(F.linear(x, wg)) * F.linear(x, wu), wd)
    np.testing.assert_allclose(out_d, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_layer_one_token_closed_form_without_sort():
    # M = 1: out = sum_j w_j * down_j(silu(gate_j x) * up_j x); given ids and
    # weights directly (no router), in numpy einsum form
    inp = _small_inputs(synth.FMT_NVFP4, False, M=1, E=8, k=3, seed=55)
    s = inp.shape
    ids = np.array([[6, 1, 3]], np.int32)
    w = np.array([[0.5, 0.3, 0.2]])
    out_d, _, _ = oracle.moe_layer(helpers.oracle_experts(inp.experts), None,
                                   synth.bf16_bits(inp.x), 1, 3, s.BS, ids=ids, w=w)
    x = inp.x.to(torch.float64).numpy()[0]
    ref = np.zeros(s.H)
    for j, e in enumerate(ids[0]):
        wg, wu, wd = (helpers.torch_dequant(p, int(e)).numpy() for p in
                      (inp.experts.gate, inp.experts.up, inp.experts.down))
        g = np.einsum("oi,i->o", wg, x)
        u = np.einsum("oi,i->o", wu, x)
        ref += w[0, j] * np.einsum("co,o->c", wd, g / (1 + np.exp(-g)) * u)
    np.testing.assert_allclose(out_d[0], ref, rtol=1e-10, atol=1e-12)


def test_blend_skips_bad_slots_and_is_weighted_sum():
    y = np.arange(12, dtype=np.float64).reshape(4, 3)
    w = np.array([[0.25, 0.75], [1.0, 0.5]])
    ttp = np.array([2, 0, -1, 3], np.int32)
    y_sh = np.ones((2, 3))
    out, _ = oracle.blend(y, w, ttp, y_sh, 2, 2, 3)
    np.testing.assert_array_equal(out[0], 0.25 * y[2] + 0.75 * y[0] + 1)
    np.testing.assert_array_equal(out[1], 0.5 * y[3] + 1)


# ---- the shared expert's gate: sigmoid(x . gate_w), on the shared term only ----

def test_shared_gate_special_values_and_symmetry():
    rng = np.random.default_rng(5)
    H = 64
    x = synth.bf16_bits(torch.tensor(rng.standard_normal((3, H)), dtype=torch.bfloat16))
    zero = np.zeros(H, np.uint16)
    np.testing.assert_array_equal(oracle.shared_gate(x, zero), [0.5, 0.5, 0.5])
    ones = synth.bf16_bits(torch.ones(1, H, dtype=torch.bfloat16))
    g1 = synth.bf16_bits(torch.ones(H, dtype=torch.bfloat16))
    assert oracle.shared_gate(ones, g1)[0] == 1.0                   # sigmoid(64)
    assert 0.0 < oracle.shared_gate(ones, g1 | 0x8000)[0] < 1e-27   # sigmoid(-64)
    g = synth.bf16_bits(torch.tensor(rng.standard_normal(H) / 8, dtype=torch.bfloat16))
    np.testing.assert_allclose(oracle.shared_gate(x, g) + oracle.shared_gate(x, g ^ 0x8000),
                               1.0, rtol=0, atol=1e-15)


def test_shared_gate_matches_library_sigmoid_of_the_dot():
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(6)
    M, H = 5, 256
    xt = torch.tensor(rng.standard_normal((M, H)), dtype=torch.bfloat16)
    gt = torch.tensor(rng.standard_normal(H) / 16, dtype=torch.bfloat16)
    z = (xt.to(torch.float64) @ gt.to(torch.float64)).numpy()
    np.testing.assert_allclose(oracle.shared_gate(synth.bf16_bits(xt), synth.bf16_bits(gt)),
                               special.expit(z), rtol=1e-14, atol=0)


def test_blend_gate_scales_only_the_shared_term():
    # the worked blend above with gates 0.5 and 0.25 on the shared term
    y = np.arange(12, dtype=np.float64).reshape(4, 3)
    w = np.array([[0.25, 0.75], [1.0, 0.5]])
    ttp = np.array([2, 0, -1, 3], np.int32)
    y_sh = np.ones((2, 3))
    out, _ = oracle.blend(y, w, ttp, y_sh, 2, 2, 3, gate=np.array([0.5, 0.25]))
    np.testing.assert_array_equal(out[0], 0.25 * y[2] + 0.75 * y[0] + 0.5)
    np.testing.assert_array_equal(out[1], 0.5 * y[3] + 0.25)
    ungated, _ = oracle.blend(y, w, ttp, y_sh, 2, 2, 3)
    ones, _ = oracle.blend(y, w, ttp, y_sh, 2, 2, 3, gate=np.ones(2))
    np.testing.assert_array_equal(ungated, ones)


@pytest.mark.parametrize("fmt", [synth.FMT_FP8, synth.FMT_NVFP4])
def test_layer_gated_shared_expert_matches_torch(fmt):
    inp = _small_inputs(fmt, True, M=5, seed=66)
    s = inp.shape
    gate = synth.make_shared_gate(s.H, 67)
    X = helpers.oracle_experts(inp.experts)
    S = helpers.oracle_experts(inp.shared)
    out_d, _, bad = oracle.moe_layer(X, S, synth.bf16_bits(inp.x), s.M, s.top_k, s.BS,
                                     logits=inp.logits.numpy(),
                                     shared_gate_bits=synth.bf16_bits(gate))
    assert bad == 0
    ref = helpers.torch_layer(inp, gate=gate).numpy()
    np.testing.assert_allclose(out_d, ref, rtol=1e-10, atol=1e-12)
    # and the gate matters: the ungated layer differs
    plain, _, _ = oracle.moe_layer(X, S, synth.bf16_bits(inp.x), s.M, s.top_k, s.BS,
                                   logits=inp.logits.numpy())
    assert np.abs(plain - out_d).max() > 1e-3
