"""The backward stores its sink-gradient partials under a key-tile number
that does not depend on the order of the device-built work list: tile t of
sequence b is numbered b + (cu[b] + 128 t) // 128. The partial array has one
slot per possible tile, ceil(total / 128) + nseq, so the numbering must be
one-to-one into that range for every packing. Checked here over random
packings with empty, length-1, tile-multiple and ragged sequences."""

import numpy as np

TILE = 128


def numbers(lengths):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    out = []
    for b, L in enumerate(lengths):
        for t in range((L + TILE - 1) // TILE):
            out.append(b + (cu[b] + TILE * t) // TILE)
    return out, int(cu[-1])


def test_numbers_are_unique_and_below_capacity():
    rng = np.random.default_rng(0)
    for trial in range(2000):
        nseq = int(rng.integers(0, 40))
        kind = trial % 4
        if kind == 0:
            lengths = rng.integers(0, 600, nseq)
        elif kind == 1:
            lengths = rng.choice([0, 1, 127, 128, 129, 255, 256, 257], nseq)
        elif kind == 2:
            lengths = TILE * rng.integers(0, 5, nseq)
        else:
            lengths = rng.integers(0, 3, nseq)
        got, total = numbers([int(x) for x in lengths])
        capacity = (total + TILE - 1) // TILE + nseq
        assert len(set(got)) == len(got)
        assert all(0 <= x < capacity for x in got)
        assert got == sorted(got)  # increasing in (sequence, tile) order
