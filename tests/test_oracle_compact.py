"""Pins of the oracle's compaction and exit scatter (no GPU)."""
import itertools

import numpy as np

import oracle


def _check_partition(mask, res):
    """The stable split is the unique pair of strictly increasing lists whose
    union is [0, n), with mask 0 on one and mask 1 on the other."""
    n = len(mask)
    c, e = list(res["cont_rows"]), list(res["exit_rows"])
    assert res["counts"][0] == len(c) and res["counts"][1] == len(e) and len(c) + len(e) == n
    assert all(x < y for x, y in zip(c, c[1:])) and all(x < y for x, y in zip(e, e[1:]))
    assert sorted(c + e) == list(range(n))
    assert all(mask[r] == 0 for r in c) and all(mask[r] != 0 for r in e)


def test_all_masks_up_to_12_rows():
    for n in range(0, 13):
        for bits in itertools.product((0, 1), repeat=n) if n <= 10 else (
                tuple(int(b) for b in np.random.default_rng(n).integers(0, 2, n)) for _ in range(300)):
            mask = np.array(bits, dtype=np.uint8)
            _check_partition(mask, oracle.stable_partition(mask))


def test_worked_example_and_position_carry():
    mask = np.array([0, 1, 1, 0, 1], dtype=np.uint8)
    res = oracle.stable_partition(mask, pos_in=np.array([40, 41, 42, 43, 44]))
    assert list(res["cont_rows"]) == [0, 3] and list(res["exit_rows"]) == [1, 2, 4]
    assert list(res["cont_pos"]) == [40, 43] and list(res["exit_pos"]) == [41, 42, 44]
    assert list(res["counts"]) == [2, 3]


def test_nonzero_bytes_count_as_exit():
    res = oracle.stable_partition(np.array([0, 7, 255, 0], dtype=np.uint8))
    assert list(res["exit_rows"]) == [1, 2]


def test_random_masks_at_workload_sizes():
    rng = np.random.default_rng(7)
    for n in (8, 32, 64, 4095, 4096, 4097):
        for frac in (0.0, 0.3, 1.0):
            mask = (rng.random(n) < frac).astype(np.uint8)
            _check_partition(mask, oracle.stable_partition(mask))


def test_gather_builds_the_compacted_buffer():
    h = np.arange(20, dtype=float).reshape(5, 4)
    g = oracle.gather_rows(h, [0, 3])
    np.testing.assert_array_equal(g, h[[0, 3]])
    assert oracle.gather_rows(h, []).shape == (0, 4)


def test_scatter_after_compact_restores_exiting_rows():
    rng = np.random.default_rng(3)
    n, d = 33, 16
    h = rng.standard_normal((n, d))
    mask = (rng.random(n) < 0.4).astype(np.uint8)
    res = oracle.stable_partition(mask)
    out = np.full((n, d), -7.0)
    got = oracle.exit_scatter(out, h, res["exit_rows"], res["exit_pos"])
    for r in range(n):
        np.testing.assert_array_equal(got[r], h[r] if mask[r] else out[r])


def test_scatter_worked_example_with_original_slots():
    # Local rows 1 and 2 of a compacted batch came from original slots 5 and 0.
    h_src = np.array([[1.0, 1.0], [2.0, 3.0], [4.0, 5.0]])
    out = np.zeros((6, 2))
    got = oracle.exit_scatter(out, h_src, exit_rows=[1, 2], exit_pos=[5, 0])
    np.testing.assert_array_equal(got[5], [2.0, 3.0])
    np.testing.assert_array_equal(got[0], [4.0, 5.0])
    assert np.all(got[1:5] == 0.0)


def test_exit_projection_is_rmsnorm_then_scatter():
    # RMSNorm of (3, 4): mean square 12.5 -> (3, 4) / sqrt(12.5) = (3 sqrt2/5, 4 sqrt2/5).
    got = oracle.exit_scatter(np.zeros((2, 2)), np.array([[3.0, 4.0]]), [0], [1],
                              gamma=np.array([1.0, 2.0]), eps=0.0)
    s2 = np.sqrt(2.0)
    np.testing.assert_allclose(got[1], [3 * s2 / 5, 8 * s2 / 5], atol=1e-15)
    assert np.all(got[0] == 0.0)
