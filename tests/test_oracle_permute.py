"""Pins for the oracle histogram and permutation: counting identities and a
library stable sort."""
import numpy as np

from oracle.layer import bias_update
from oracle.permute import histogram, permute
from conftest import read_golden


def _random_idx(T, E, K, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)


def test_histogram_matches_bincount_and_total():
    idx = _random_idx(300, 16, 4, 0)
    c = histogram(idx, 16)
    assert c.sum() == 300 * 4
    assert np.array_equal(c, np.bincount(idx.ravel(), minlength=16))


def test_permutation_is_stable_sort():
    T, E, K = 257, 24, 5
    idx = _random_idx(T, E, K, 1)
    offsets, sorted_token, row_of = permute(idx, E)
    assert offsets[0] == 0 and offsets[-1] == T * K and np.all(np.diff(offsets) >= 0)
    order = np.argsort(idx.ravel(), kind="stable")      # library stable sort of the expert keys
    assert np.array_equal(sorted_token, order // K)
    inv = np.empty(T * K, np.int64)
    inv[order] = np.arange(T * K)
    assert np.array_equal(row_of.ravel(), inv)
    for t in range(T):
        for k in range(K):
            r = row_of[t, k]
            assert sorted_token[r] == t and offsets[idx[t, k]] <= r < offsets[idx[t, k] + 1]


def test_empty_experts_and_single_hot_expert():
    idx = np.zeros((10, 1), np.int32) + 3
    offsets, sorted_token, row_of = permute(idx, 8)
    assert list(offsets) == [0, 0, 0, 0, 10, 10, 10, 10, 10]
    assert list(sorted_token) == list(range(10))


def test_bias_update_golden():
    g = read_golden("bias_update_example.txt")
    T, K = int(g["T"][0][0]), int(g["K"][0][0])
    gamma = float(g["gamma"][0][0])
    counts = np.array([int(v) for v in g["counts"][0]])
    before = np.array([float(v) for v in g["bias_before"][0]], np.float32)
    after = np.array([float(v) for v in g["bias_after"][0]], np.float32)
    assert np.array_equal(bias_update(before, counts, T, K, gamma), after)


def test_bias_update_sign_follows_load():
    rng = np.random.default_rng(2)
    E, T, K = 64, 1000, 6
    counts = rng.multinomial(T * K, np.ones(E) / E)
    b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    nb = bias_update(b, counts, T, K, 1e-3)
    mean = T * K / E
    assert np.all(nb[counts > mean] < b[counts > mean])
    assert np.all(nb[counts < mean] > b[counts < mean])
    assert np.array_equal(bias_update(b, counts, T, K, 0.0), b)
    even = np.full(8, 5)
    b8 = b[:8]
    assert np.array_equal(bias_update(b8, even, 8, 5, 1e-3), b8)
