"""Pins for the oracle's schedule tables (per-expert counts, exclusive prefix
sums, token->slot permutation, tile list).

The schedule is built from the router's top-k ids with no token dropping
(clip "Mixture-of-Kittens: Cursor open-sources an MoE training megakernel",
key point 4). Pins: counts from numpy's bincount, offsets from cumsum, the
permutation from numpy's stable argsort (a library routine), bijection and
segment invariants.
"""
import numpy as np
import pytest

import oracle


def _cases():
    rng = np.random.default_rng(0)
    yield "uniform", np.stack([rng.permutation(8)[:2] for _ in range(256)]).astype(np.int32), 8
    yield "skewed", np.stack([rng.choice(64, 8, replace=False, p=_zipf(64)) for _ in range(333)]
                             ).astype(np.int32), 64
    ids = np.stack([[0, 1] for _ in range(300)]).astype(np.int32)  # two hot experts, rest empty
    yield "two_hot", ids, 16
    yield "single_token", np.array([[3, 0, 5]], np.int32), 6
    yield "empty", np.zeros((0, 4), np.int32), 8


def _zipf(E, s=1.2):
    p = np.arange(1, E + 1, dtype=np.float64) ** -s
    return p / p.sum()


@pytest.mark.parametrize("name,ids,E", list(_cases()), ids=[c[0] for c in _cases()])
@pytest.mark.parametrize("tile_m,pad_m", [(128, 128), (32, 32), (128, 512), (32, 64)])
def test_schedule_invariants(name, ids, E, tile_m, pad_m):
    N, k = ids.shape
    A = N * k
    s = oracle.build_schedule(ids, E, tile_m, pad_m)
    counts, offsets, pad = s["counts"], s["offsets"], s["pad_offsets"]
    np.testing.assert_array_equal(counts, np.bincount(ids.ravel(), minlength=E))
    assert counts.sum() == A and offsets[E] == A
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    padded = (counts + pad_m - 1) // pad_m * pad_m
    np.testing.assert_array_equal(pad, np.concatenate([[0], np.cumsum(padded)]))
    assert np.all(pad % pad_m == 0)

    # Permutation: the stable sort of assignments by expert, placed at each
    # expert's padded segment start.
    order = np.argsort(ids.ravel(), kind="stable")
    expect_slot = np.empty(A, np.int64)
    for r, a in enumerate(order):
        e = ids.ravel()[a]
        expect_slot[a] = pad[e] + (r - offsets[e])
    np.testing.assert_array_equal(s["slot_of"].ravel(), expect_slot)

    # Inverse map and bijection onto the used rows.
    src = s["src_of_row"]
    assert src.shape[0] == pad[E]
    seen = np.zeros(pad[E], bool)
    seen[s["slot_of"].ravel()] = True
    assert seen.sum() == A
    np.testing.assert_array_equal(src[s["slot_of"].ravel()], np.arange(A))
    assert np.all(src[~seen] == -1)

    # Tile list: consecutive tile_m-row tiles, each inside one segment.
    tiles = s["tiles"]
    assert s["n_tiles"] == pad[E] // tile_m
    if s["n_tiles"]:
        np.testing.assert_array_equal(tiles[:, 1], np.arange(s["n_tiles"]) * tile_m)
        for e, r0, valid in tiles:
            assert pad[e] <= r0 < pad[e + 1]
            assert valid == max(0, min(tile_m, pad[e] + counts[e] - r0))
            rows = src[r0:r0 + tile_m]
            assert np.all(rows[:valid] >= 0) and np.all(rows[valid:] == -1)
            assert np.all(ids.ravel()[rows[:valid]] == e)


def test_slots_stable_by_token():
    ids = np.array([[2, 0], [0, 2], [1, 2], [2, 1]], np.int32)
    s = oracle.build_schedule(ids, 3, 4)
    # expert 0 segment [0,4): tokens 0,1 ; expert 1 [4,8): tokens 2,3 ; expert 2 [8,12): 0,1,2,3
    np.testing.assert_array_equal(s["slot_of"], [[8, 0], [1, 9], [4, 10], [11, 5]])
    np.testing.assert_array_equal(s["tiles"], [[0, 0, 2], [1, 4, 2], [2, 8, 4]])


def test_out_of_range_expert_is_rejected():
    with pytest.raises(oracle.OracleError):
        oracle.build_schedule(np.array([[0, 9]], np.int32), 4)
