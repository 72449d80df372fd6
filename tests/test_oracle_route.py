"""Pins for the oracle router: hand-worked example, brute force over all
group and expert subsets, special cases that reduce to a plain sort, and the
invariants the aux-loss-free scheme fixes."""
import itertools

import numpy as np
import pytest

from conftest import read_golden
from oracle import route


def _golden_case(tag):
    g = read_golden("route_example.txt")
    s = np.array([[float(v) for v in g["s"][0]]])
    bias = np.array([float(v) for v in g[f"{tag}_bias"][0]])
    gk = int(g[f"{tag}_gk"][0][0])
    idx = [int(v) for v in g[f"{tag}_idx"][0]]
    gate = [float(v) for v in g[f"{tag}_gate"][0]]
    return s, bias, gk, idx, gate


@pytest.mark.parametrize("tag", ["caseA", "caseB", "caseC"])
def test_golden_routing(tag):
    s, bias, gk, idx, gate = _golden_case(tag)
    got_idx, got_gate, _ = route.select(s, bias, G=4, M=2, K=3, gk=gk)
    assert list(got_idx[0]) == idx
    np.testing.assert_allclose(got_gate[0], gate, rtol=0, atol=1e-12)


def _brute(sb, s, G, M, K, gk):
    """Best M groups by score (sum of top-gk), then best K experts inside, by full enumeration."""
    E = sb.shape[0]
    n = E // G
    score = [sum(sorted(sb[g * n:(g + 1) * n], reverse=True)[:gk]) for g in range(G)]
    best_groups = max(itertools.combinations(range(G), M), key=lambda c: sum(score[g] for g in c))
    cand = [e for g in best_groups for e in range(g * n, (g + 1) * n)]
    best = max(itertools.combinations(cand, K), key=lambda c: sum(sb[e] for e in c))
    gates = {e: s[e] / sum(s[j] for j in best) for e in best}
    return set(best), gates


@pytest.mark.parametrize("E,G,M,K,gk", [(8, 4, 2, 3, 1), (8, 4, 2, 3, 2), (12, 3, 2, 4, 2),
                                        (16, 4, 2, 4, 2), (16, 8, 3, 5, 2), (16, 4, 4, 6, 3)])
def test_brute_force(E, G, M, K, gk):
    rng = np.random.default_rng(E * 100 + K)
    x = rng.standard_normal((40, 32))
    Wr = rng.standard_normal((E, 32)) / np.sqrt(32)
    bias = rng.uniform(-0.1, 0.1, E)
    s = route.affinity(x, Wr)
    idx, gate, info = route.select(s, bias, G, M, K, gk)
    for t in range(40):
        sb = s[t] + bias
        want, wg = _brute(sb, s[t], G, M, K, gk)
        assert set(idx[t]) == want
        for k, e in enumerate(idx[t]):
            assert abs(gate[t, k] - wg[e]) < 1e-12
        assert np.all(np.diff(sb[idx[t]]) <= 0)            # listed by descending biased affinity


def test_all_groups_reduces_to_plain_topk():
    rng = np.random.default_rng(5)
    s = route.affinity(rng.standard_normal((64, 16)), rng.standard_normal((32, 16)) / 4)
    bias = rng.uniform(-0.1, 0.1, 32)
    idx, gate, _ = route.select(s, bias, G=4, M=4, K=6, gk=2)
    want = np.argsort(-(s + bias), axis=1, kind="stable")[:, :6]
    assert np.array_equal(idx, want)
    # zero bias: plain top-K of the affinity itself
    idx0, _, _ = route.select(s, np.zeros(32), G=4, M=4, K=6, gk=2)
    assert np.array_equal(idx0, np.argsort(-s, axis=1, kind="stable")[:, :6])


def test_all_experts_gates_are_normalised_affinity():
    rng = np.random.default_rng(6)
    s = route.affinity(rng.standard_normal((10, 8)), rng.standard_normal((8, 8)))
    idx, gate, _ = route.select(s, np.zeros(8), G=2, M=2, K=8, gk=1)
    full = np.zeros_like(s)
    np.put_along_axis(full, idx, gate, axis=1)
    np.testing.assert_allclose(full, s / s.sum(1, keepdims=True), rtol=0, atol=1e-15)


def test_invariants_on_workload_shape():
    rng = np.random.default_rng(7)
    E, G, M, K = 64, 8, 3, 6
    s = route.affinity(rng.standard_normal((500, 64)), rng.standard_normal((E, 64)) / 8)
    bias = rng.uniform(-0.1, 0.1, E)
    idx, gate, _ = route.select(s, bias, G, M, K, gk=2)
    for t in range(500):
        assert len(set(idx[t])) == K
        assert len(set(idx[t] // (E // G))) <= M
    np.testing.assert_allclose(gate.sum(1), 1.0, rtol=0, atol=1e-12)
    assert np.all(gate > 0)


def test_bias_changes_choice_not_gate_formula():
    rng = np.random.default_rng(8)
    E, G, M, K = 16, 4, 2, 4
    s = route.affinity(rng.standard_normal((300, 16)), rng.standard_normal((E, 16)) / 4)
    b0 = np.zeros(E)
    idx0, gate0, _ = route.select(s, b0, G, M, K, gk=2)
    # a bias small enough to keep every choice leaves every gate bit-identical
    tiny = rng.uniform(-1e-12, 1e-12, E)
    idx1, gate1, info1 = route.select(s, tiny, G, M, K, gk=2)
    same = np.all(np.sort(idx0, 1) == np.sort(idx1, 1), axis=1)
    assert same.mean() > 0.99
    for t in np.nonzero(same)[0]:
        g0 = dict(zip(idx0[t], gate0[t]))
        g1 = dict(zip(idx1[t], gate1[t]))
        assert all(g0[e] == g1[e] for e in g0)
    # a large bias on one expert makes it chosen by every token; gates stay s_e / sum over chosen
    big = np.zeros(E)
    big[5] = 10.0
    idx2, gate2, _ = route.select(s, big, G, M, K, gk=2)
    assert np.all(np.any(idx2 == 5, axis=1))
    assert not np.all(np.any(idx0 == 5, axis=1))
    chosen = np.take_along_axis(s, idx2, 1)
    np.testing.assert_allclose(gate2, chosen / chosen.sum(1, keepdims=True), rtol=0, atol=1e-15)


def test_sigmoid_closed_form():
    s = route.affinity(np.zeros((1, 4)), np.ones((3, 4)), logit_offset=np.array([0.0, np.log(3.0), -np.log(3.0)]))
    np.testing.assert_allclose(s[0], [0.5, 0.75, 0.25], rtol=0, atol=1e-15)


def test_near_tie_flags():
    s = np.array([[0.5, 0.5, 0.2, 0.1]])
    _, _, info = route.select(s, np.zeros(4), G=2, M=2, K=1, gk=1)
    assert route.near_tie(info)[0]
