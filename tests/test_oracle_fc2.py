"""Pins for the oracle's FlashComm2 token reorganisation (vllm-ascend SP/FlashComm notes §4.4).

The page prints a worked example (global_tp=4, otp_size=2); the fixture in
tests/golden/fc2_reorganize_tp4_otp2.json restates it. Beyond it: the reorganisation is a
permutation of the input rows' feature slices (nothing lost or repeated), every output row of a
rank holds one token's features from all members of its ODP group, and the ranks of an OTP group
(same position in their ODP groups) hold the same tokens.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fc2_reorganize_tp4_otp2.json")


def _labelled_input(G: int, N: int, F: int) -> np.ndarray:
    """x[r][t][f] = a unique id of (rank r's feature f of token t)."""
    r, t, f = np.meshgrid(np.arange(G), np.arange(N), np.arange(F), indexing="ij")
    return (r * 1_000_000 + t * 1000 + f).astype(np.int64)


def test_batch_ids_match_the_page():
    gold = json.load(open(GOLDEN))
    assert oracle.fc2_batch_ids(gold["global_tp"], gold["otp_size"]) == gold["batch_ids"]


def test_worked_example_of_the_page():
    gold = json.load(open(GOLDEN))
    G, P = gold["global_tp"], gold["otp_size"]
    letters = gold["feature_slices"]
    # one token per segment T0..T3, one element per feature slice: the element names its block
    x = np.array([[[10 * seg + r] for seg in range(G)] for r in range(G)], np.int64)  # [G][N=4][1]
    y = oracle.fc2_reorganize(x, P)
    assert y.shape == (G, G // (G // P), G // P)
    for r, rows in gold["output"].items():
        got = []
        for row in y[int(r)]:
            seg = {int(v) // 10 for v in row}
            assert len(seg) == 1  # one token per output row
            got.append(f"T{seg.pop()}" + "".join(letters[int(v) % 10] for v in row))
        assert got == rows


@pytest.mark.parametrize("G,P,N,F", [(4, 2, 8, 3), (8, 2, 16, 2), (8, 4, 8, 5), (4, 1, 4, 2),
                                     (4, 4, 12, 1), (16, 4, 32, 1), (2, 1, 6, 4)])
def test_reorganisation_is_a_permutation_with_the_group_structure(G, P, N, F):
    D = G // P
    x = _labelled_input(G, N, F)
    y = oracle.fc2_reorganize(x, P)
    assert y.shape == (G, N // D, F * D)
    assert np.array_equal(np.sort(y.ravel()), np.sort(x.ravel()))
    tokens = (y // 1000) % 1000
    ranks = y // 1_000_000
    feats = y % 1000
    for r in range(G):
        g = r // D
        # every output row is one token, with member m's slice in feature block m, in order
        assert np.all(tokens[r] == tokens[r][:, :1])
        for m in range(D):
            assert np.all(ranks[r][:, m * F:(m + 1) * F] == g * D + m)
            assert np.array_equal(feats[r][:, m * F:(m + 1) * F], np.tile(np.arange(F), (N // D, 1)))
    # the ranks of one OTP group {j, j+D, ...} hold the same tokens in the same order
    for j in range(D):
        for g in range(1, P):
            assert np.array_equal(tokens[j][:, 0], tokens[g * D + j][:, 0])
    # and the D ranks of an ODP group hold disjoint tokens covering all N
    for g in range(P):
        seen = np.concatenate([tokens[g * D + j][:, 0] for j in range(D)])
        assert np.array_equal(np.sort(seen), np.arange(N))


def test_otp_equal_global_tp_is_identity():
    x = _labelled_input(4, 8, 3)
    assert np.array_equal(oracle.fc2_reorganize(x, 4), x)
