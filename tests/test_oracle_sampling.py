"""Pins of the oracle's sampler (CPU): the generator against its published reference vector,
the special cases that reduce to greedy, the top-k / top-p sets on hand examples, and the
empirical distribution of many draws against the renormalised probabilities."""
import os

import numpy as np
import pytest

from oracle import sampling as smp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_mix_reproduces_the_published_splitmix64_vector():
    with open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt")) as f:
        want = [int(l) for l in f if l.strip() and not l.startswith("#")]
    got = [smp.mix(1234567 + (i + 1) * smp.GAMMA) for i in range(5)]
    assert got == want


def test_uniform_is_a_function_of_seed_and_counter_in_unit_interval():
    us = [smp.uniform(99, c) for c in range(2000)]
    assert all(0.0 <= u < 1.0 for u in us)
    assert smp.uniform(99, 17) == smp.uniform(99, 17)
    assert smp.uniform(99, 17) != smp.uniform(100, 17)
    assert all(float(np.float32(u)) == u for u in us)        # 24 bits: exact in float32
    assert abs(np.mean(us) - 0.5) < 0.02


def test_greedy_cases():
    rng = np.random.default_rng(0)
    logits = rng.normal(0, 3, 1000).astype(np.float32)
    am = int(np.argmax(logits))
    assert smp.sample(logits, 0.0, 20, 0.9, 1, 5)[0] == am          # temperature 0
    for c in range(50):
        assert smp.sample(logits, 0.8, 1, 0.9, 7, c)[0] == am       # top-k 1
        assert smp.sample(logits, 0.8, 20, 1e-6, 7, c)[0] == am     # top-p -> 0
    tied = np.zeros(16, np.float32)
    assert smp.sample(tied, 0.0, 4, 0.5, 1, 1)[0] == 0               # lowest index on ties


def test_top_k_keeps_lowest_indices_on_ties():
    logits = np.array([1, 5, 3, 5, 5, 2], np.float32)
    _, kept, _ = smp.sample(logits, 1.0, 2, 1.0, 3, 0)
    assert kept == [1, 3]
    _, kept, _ = smp.sample(logits, 1.0, 4, 1.0, 3, 0)
    assert kept == [1, 3, 4, 2]


def test_top_p_prefix_on_a_hand_example():
    # probabilities 0.5, 0.3, 0.15, 0.05 at temperature 1
    logits = np.log(np.array([0.5, 0.3, 0.15, 0.05])).astype(np.float32)
    assert smp.sample(logits, 1.0, 4, 0.7, 0, 0)[1] == [0, 1]
    assert smp.sample(logits, 1.0, 4, 0.85, 0, 0)[1] == [0, 1, 2]
    assert smp.sample(logits, 1.0, 4, 0.99, 0, 0)[1] == [0, 1, 2, 3]
    assert smp.sample(logits, 1.0, 4, 0.4, 0, 0)[1] == [0]


@pytest.mark.parametrize("T,k,p", [(1.0, 6, 1.0), (0.7, 6, 0.8), (2.0, 10, 0.95)])
def test_empirical_distribution_matches_renormalised_probabilities(T, k, p):
    logits = np.array([2.0, 1.5, 1.4, 0.3, 0.2, -0.5, -1.0, -3.0, 0.9, 1.1], np.float32)
    n = 40000
    counts = np.zeros(logits.size)
    for c in range(n):
        counts[smp.sample(logits, T, k, p, 2024, c)[0]] += 1
    order = sorted(range(logits.size), key=lambda i: (-logits[i], i))[:k]
    w = np.exp((logits[order].astype(np.float64) - logits[order[0]]) / T)
    cum = np.cumsum(w)
    m = int(np.flatnonzero(cum >= p * cum[-1])[0]) if p < 1 else k - 1
    prob = np.zeros(logits.size)
    prob[order[: m + 1]] = w[: m + 1] / cum[m]
    assert np.all(counts[prob == 0] == 0)
    sigma = np.sqrt(n * prob * (1 - prob)) + 1
    assert np.all(np.abs(counts - n * prob) <= 5 * sigma)
