"""Host-side model of the GEMM's stream-K partition and partial-sum slots (no GPU).

The GEMM (w12_gemm.cu) splits T units (row block x 64 columns, or row-block pair x 64
columns) over G places: place b takes units [b*T/G, (b+1)*T/G), and the place holding unit i
is ((i+1)*G - 1) / T.  A row split between places gets one slot per (place c, row r) at
index c + r (pairs: 2*(c + r) + pipeline), out of RB + G slots (pairs: 2*((RB+1)/2 + G)).
The last part of a row, or the after-grid sum, adds the slots of places cf..cl.  These
checks restate those formulas and test what the fix-up relies on, over many shapes:
the place formula inverts the ranges, the parts of a row are exactly the places whose
ranges meet it, and no two partial (place, row) pairs share a slot or leave the slot array.
"""
import random

import pytest

K_MIN_ITERS = 4


def place_of_unit(i, G, T):
    return ((i + 1) * G - 1) // T


def partition_places(T, sms, per_sm):
    return max(1, min((T + K_MIN_ITERS - 1) // K_MIN_ITERS, sms * per_sm))


def shapes():
    rng = random.Random(12)
    out = [(40, 80, 152, False), (40, 272, 152, True), (272, 80, 152, True), (1, 1, 152, False),
           (9, 732, 152, True), (11, 625, 152, True), (56, 80, 304, False), (3, 1024, 152, True)]
    for _ in range(300):
        out.append((rng.randint(1, 400), rng.randint(1, 1024), rng.choice([132, 148, 152, 304]), rng.random() < 0.5))
    return out


@pytest.mark.parametrize("RB,KC,places,wide", shapes())
def test_partition_and_slots(RB, KC, places, wide):
    rows = (RB + 1) // 2 if wide else RB
    T = rows * KC
    G = partition_places(T, places, 1)
    ranges = [(b * T // G, (b + 1) * T // G) for b in range(G)]
    # the ranges tile [0, T) in order, none empty (G <= T)
    assert ranges[0][0] == 0 and ranges[-1][1] == T
    assert all(ranges[b][1] == ranges[b + 1][0] for b in range(G - 1))
    assert all(lo < hi for lo, hi in ranges)
    # the place formula inverts the ranges (spot-checked at every range edge)
    for b, (lo, hi) in enumerate(ranges):
        for i in {lo, hi - 1, (lo + hi) // 2}:
            assert place_of_unit(i, G, T) == b
    n_slots = 2 * ((RB + 1) // 2 + G) if wide else RB + G
    used = set()
    for r in range(rows):
        cf, cl = place_of_unit(r * KC, G, T), place_of_unit((r + 1) * KC - 1, G, T)
        meet = [b for b, (lo, hi) in enumerate(ranges) if lo < (r + 1) * KC and hi > r * KC]
        assert meet == list(range(cf, cl + 1))
        # a row held by one place is stored directly: the GEMM's test (its segment starts at
        # or before the row and reaches its last chunk) agrees with cf == cl
        whole = ranges[cf][0] <= r * KC and ranges[cf][1] >= (r + 1) * KC
        assert whole == (cf == cl)
        if cf == cl:
            continue
        for c in range(cf, cl + 1):
            for p in (0, 1) if wide else (0,):
                slot = 2 * (c + r) + p if wide else c + r
                assert 0 <= slot < n_slots
                assert slot not in used
                used.add(slot)
