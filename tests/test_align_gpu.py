"""moe_align on the GPU against the oracle: bit-exact tables over the whole
alignment stress grid (n = 8*M for M in {1, 64, 1024, 4096}, E in {64, 256,
1024}, BS in {16, 64, 128}; uniform, Zipf(1.2) and one-expert ids), every
routing of up to three tokens on four experts, int32 ids, out-of-range ids
and the empty input."""
from __future__ import annotations

import itertools

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

KEYS = ("sorted_token_ids", "sorted_expert_ids", "expert_offsets", "token_to_perm",
        "active_experts", "active_count", "num_tokens_post_padded")


@pytest.fixture(scope="module")
def moe():
    import expert_routing_alignment_gb300 as m
    m.load()
    return m


def run_gpu(moe, ids: np.ndarray, E: int, BS: int, dtype=torch.int64):
    dev_ids = torch.from_numpy(ids.astype(np.int64)).to(dtype).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = moe.moe_align(dev_ids, E, BS, err_word=err)
    torch.cuda.synchronize()
    got = {k: out[k].cpu().numpy() for k in KEYS}
    got["sorted_token_ids"] = got["sorted_token_ids"][: out["max_total"]]
    got["sorted_expert_ids"] = got["sorted_expert_ids"][: out["max_blocks"]]
    got["active_experts"] = got["active_experts"][: out["cap"]]
    got["token_to_perm"] = got["token_to_perm"][: ids.size]
    return got, int(err.item())


def assert_tables_equal(got, ref):
    for k in KEYS:
        np.testing.assert_array_equal(got[k], np.asarray(ref[k]).ravel(), err_msg=k)


GRID = [(M, E, BS, dist) for M in (1, 64, 1024, 4096) for E in (64, 256, 1024)
        for BS in (16, 64, 128) for dist in ("uniform", "zipf", "one0", "oneL")]


@pytest.mark.parametrize("M,E,BS,dist", GRID)
def test_align_stress_grid_bit_exact(moe, M, E, BS, dist):
    n = 8 * M
    if dist.startswith("one"):
        ids = synth.align_ids(n, E, "one", 0, expert=0 if dist == "one0" else E - 1)
    else:
        ids = synth.align_ids(n, E, dist, seed=1000 + M * 7 + E + BS)
    got, err = run_gpu(moe, ids, E, BS)
    assert err == 0
    assert_tables_equal(got, oracle.align(ids, E, BS))


def test_align_every_routing_of_three_tokens(moe):
    E = 4
    for M in (1, 2, 3):
        for k in (1, 2):
            per_token = list(itertools.permutations(range(E), k))
            for routing in itertools.product(per_token, repeat=M):
                ids = np.array([e for tok in routing for e in tok], np.int64)
                for BS in (1, 3, 16):
                    got, _ = run_gpu(moe, ids, E, BS, torch.int32)
                    assert_tables_equal(got, oracle.align(ids, E, BS))


@pytest.mark.parametrize("n", [1, 31, 32, 33, 255, 257, 513, 4095, 4097, 16385, 32767, 32769,
                               65536])
def test_align_ragged_sizes_int32(moe, n):
    ids = synth.align_ids(n, 256, "zipf", seed=n)
    got, _ = run_gpu(moe, ids, 256, 64, torch.int32)
    assert_tables_equal(got, oracle.align(ids, 256, 64))


def test_align_out_of_range_ids(moe):
    rng = np.random.default_rng(9)
    ids = rng.integers(0, 64, size=1000).astype(np.int64)
    ids[[3, 500, 999]] = [-1, 64, 1 << 40]
    got, err = run_gpu(moe, ids, 64, 16)
    assert err & moe.MOE_ERR_BAD_ID
    ref = oracle.align(ids, 64, 16)
    assert ref["bad"] == 3
    assert_tables_equal(got, ref)


def test_align_empty_input(moe):
    got, err = run_gpu(moe, np.zeros(0, np.int64), 16, 16)
    assert err == 0
    assert got["expert_offsets"].tolist() == [0] * 17
    assert int(got["active_count"][0]) == 0 and int(got["num_tokens_post_padded"][0]) == 0


def test_align_repeatable_and_graph_replayable(moe):
    n, E, BS = 8 * 64, 128, 16
    ids_dev = torch.zeros(n, dtype=torch.int32, device="cuda")
    out = moe.alloc_align_outputs(n, E, BS)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        moe.moe_align(ids_dev, E, BS, out=out)   # warm-up (sets kernel attributes)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_align(ids_dev, E, BS, out=out)
    for seed in range(3):
        ids = synth.align_ids(n, E, "zipf", seed=seed)
        ids_dev.copy_(torch.from_numpy(ids.astype(np.int32)))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.align(ids, E, BS)
        np.testing.assert_array_equal(out["sorted_token_ids"].cpu().numpy(),
                                      ref["sorted_token_ids"])
        np.testing.assert_array_equal(out["token_to_perm"].cpu().numpy(), ref["token_to_perm"])
