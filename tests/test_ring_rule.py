"""The placement rule of the tensor-core kernel's two rings, checked on the host.

The kernel keeps its copy stages in a ring of shared-memory bytes and its
accumulators in a ring of TMEM columns.  Ranges of varying length are placed
in order (at the head, or at 0 when the range does not fit before the end)
and freed oldest first.  Before placing a range the kernel retires stages:

  * on a wrap, every in-flight stage lying in the skipped end [head, end);
  * then the oldest stage while it overlaps the new range (or while the
    record ring is full).

The claim the kernel relies on: after this, the new range overlaps no
in-flight range at all, although only the oldest one was compared.  This is
the rule restated on the host and checked against every in-flight range over
random sequences of the stage sizes the kernel uses (a check of the rule,
not of the device code)."""
from __future__ import annotations

import random

import pytest

KB = 1024
RECORDS = 8


def place_all(sizes, ring, records=RECORDS):
    """Run the rule over `sizes`; return the first overlap found, or None."""
    head, tail, rec = 0, 0, {}
    for s, size in enumerate(sizes):
        wrap = head + size > ring
        at = 0 if wrap else head
        while tail < s:
            tp, tl = rec[tail]
            busy = (s - tail >= records or (wrap and tp >= head)
                    or (at < tp + tl and tp < at + size))
            if not busy:
                break
            tail += 1
        for j in range(tail, s):   # every in-flight range, not only the oldest
            p, l = rec[j]
            if at < p + l and p < at + size:
                return s, j
        rec[s] = (at, size)
        head = at + size
    return None


def test_wrap_without_retiring_the_skipped_end_would_overlap():
    # the case the wrap step exists for: the oldest stage sits in the skipped
    # end, a newer one at the start of the ring
    ring = 214 * KB
    sizes = [88 * KB, 88 * KB, 40 * KB, 80 * KB, 72 * KB, 80 * KB]
    assert place_all(sizes, ring) is None


@pytest.mark.parametrize("ring,sizes", [
    # shared-memory stages (bytes): one or two k blocks of two 16 KB weight
    # tiles plus 2 or 3 activation terms of 16..64 rows
    (214 * KB, [36, 38, 40, 44, 48, 56, 72, 76, 80, 88]),
    (221 * KB, [36, 40, 48, 56, 72, 80, 88]),
    # TMEM accumulators (columns): 2 tiles x terms x rows, per stage
    (512, [64, 96, 128, 192, 256, 384]),
])
def test_no_overlap_over_random_sequences(ring, sizes):
    unit = KB if ring > 512 else 1
    rng = random.Random(12345)
    for _ in range(4000):
        seq = [rng.choice(sizes) * unit for _ in range(60)]
        assert place_all(seq, ring) is None


def test_overlap_scan_catches_the_rule_without_the_wrap_step():
    """Without retiring the skipped end on a wrap, the oldest-only comparison
    lets a new range overlap a newer in-flight one; the overlap scan finds it."""
    def naive(sizes, ring):
        head, tail, rec = 0, 0, {}
        for s, size in enumerate(sizes):
            at = head if head + size <= ring else 0
            while tail < s:
                tp, tl = rec[tail]
                if not (s - tail >= RECORDS or (at < tp + tl and tp < at + size)):
                    break
                tail += 1
            for j in range(tail, s):
                p, l = rec[j]
                if at < p + l and p < at + size:
                    return s, j
            rec[s] = (at, size)
            head = at + size
        return None

    rng = random.Random(1)
    sizes = [36, 40, 48, 56, 72, 80, 88]
    found = any(naive([rng.choice(sizes) * KB for _ in range(60)], 214 * KB) is not None
                for _ in range(2000))
    assert found
