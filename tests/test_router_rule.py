"""The router kernel's reduction rule, checked on the host.

Each thread of the router kernel holds RE x 8 fp32 partial sums, one per
(expert row, x row), and RE depends on the batch width.  A warp ends them
with a reduce-scatter butterfly: at xor distance 16, 8, 4, 2, 1 a lane that
still holds more than one sum keeps half of them (the upper half where its
lane bit is set) and adds its partner's copy; once one sum is left the steps
are a plain butterfly.  The claim the kernel relies on for row invariance:
every sum comes out bit for bit as a plain xor butterfly gives it, whatever
the number of sums per lane.  This restates the rule in numpy float32 (IEEE
round-to-nearest adds, as on the GPU) and checks it."""
from __future__ import annotations

import numpy as np
import pytest


def plain_butterfly(v: np.ndarray) -> np.ndarray:
    """v [32 lanes, N] -> lane 0's sums after xor steps 16..1, [N]."""
    v = v.copy()
    for m in (16, 8, 4, 2, 1):
        v = (v + v[np.arange(32) ^ m]).astype(np.float32)
    return v[0]


def reduce_scatter(v: np.ndarray) -> np.ndarray:
    """The kernel's rule; returns every sum from the lane that ends with it."""
    N = v.shape[1]
    acc = v.copy()
    idx = np.zeros(32, np.int64)
    cnt = N
    lanes = np.arange(32)
    for m in (16, 8, 4, 2, 1):
        partner = acc[lanes ^ m].copy()
        if cnt > 1:
            half = cnt // 2
            up = (lanes & m) != 0
            new = acc.copy()
            for i in range(half):
                send_p = np.where(up[lanes ^ m], partner[:, i], partner[:, i + half])
                keep = np.where(up, acc[:, i + half], acc[:, i])
                new[:, i] = (keep + send_p).astype(np.float32)
            acc = new
            idx = idx + np.where(up, half, 0)
            cnt = half
        else:
            acc[:, 0] = (acc[:, 0] + partner[:, 0]).astype(np.float32)
    out = np.full(N, np.nan, np.float32)
    for lane in range(32):
        for i in range(min(cnt, N)):
            o = idx[lane] + i
            if np.isnan(out[o]):
                out[o] = acc[lane, i]
            else:   # lanes holding the same sum hold the same bits
                assert out[o].tobytes() == acc[lane, i].tobytes()
    assert not np.isnan(out).any()
    return out


@pytest.mark.parametrize("RE", [1, 2, 4, 8])
def test_reduce_scatter_equals_plain_butterfly(RE):
    rng = np.random.default_rng(RE)
    N = RE * 8
    for _ in range(200):
        # magnitudes spread over many binades so that the add order shows
        v = (rng.standard_normal((32, N)) * 2.0 ** rng.integers(-20, 20, (32, N)))
        v = v.astype(np.float32)
        got = reduce_scatter(v)
        want = plain_butterfly(v)
        assert got.tobytes() == want.tobytes()


def test_a_different_pairing_order_would_differ():
    """Negative control: the pairing order matters (xor 1 first gives other
    bits), so the equality above is not trivial."""
    rng = np.random.default_rng(0)
    differs = False
    for _ in range(50):
        v = (rng.standard_normal((32, 8)) * 2.0 ** rng.integers(-20, 20, (32, 8)))
        v = v.astype(np.float32)
        w = v.copy()
        for m in (1, 2, 4, 8, 16):
            w = (w + w[np.arange(32) ^ m]).astype(np.float32)
        differs |= w[0].tobytes() != plain_butterfly(v).tobytes()
    assert differs
