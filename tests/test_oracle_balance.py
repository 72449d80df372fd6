"""Pins for the oracle's sequence-wise balance statistics (closed forms of
balanced and collapsed routing, brute-force loops on a tiny case)."""
import numpy as np

from oracle.balance import balance_loss, balance_stats


def test_perfectly_balanced_routing_gives_alpha():
    # uniform affinities, every expert chosen equally often: f_i = 1, P_i = 1/E, L = alpha
    E, K, L = 8, 2, 16
    s = np.full((L, E), 0.3)
    idx = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(L)])
    f, P = balance_stats(s, idx, L)
    assert np.allclose(f, 1.0) and np.allclose(P, 1.0 / E)
    assert np.allclose(balance_loss(s, idx, L, 1e-4), 1e-4)


def test_collapsed_routing_gives_e_over_k():
    # every token picks experts {0, 1}, which hold all the affinity: f = E/K on them, P = 1/K
    E, K, L = 8, 2, 10
    s = np.zeros((L, E)) + 1e-300
    s[:, :2] = 0.5
    idx = np.tile([0, 1], (L, 1))
    loss = balance_loss(s, idx, L, 1.0)
    assert np.allclose(loss, E / K * (0.5 + 0.5))


def test_brute_force_two_sequences():
    rng = np.random.default_rng(3)
    T, E, K, L = 12, 6, 3, 6
    s = rng.uniform(0.01, 1.0, (T, E))
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)])
    loss = balance_loss(s, idx, L, 0.01)
    for q in range(2):
        tot = 0.0
        for i in range(E):
            cnt = sum(1 for t in range(q * L, (q + 1) * L) for k in range(K) if idx[t, k] == i)
            p = sum(s[t, i] / sum(s[t, j] for j in range(E)) for t in range(q * L, (q + 1) * L)) / L
            tot += E / (K * L) * cnt * p
        assert abs(loss[q] - 0.01 * tot) <= 1e-12 * abs(tot)
