"""Pins of the oracle's batch-aware routing (reading R8 of the batch-aware
routing named in "SM120 FP4 Kernel Research Campaign", key finding 6 and
section 6).  Checked against hand-derived selections, the reduction to plain
top-k, and brute-force properties of the definition (CPU only)."""
import itertools

import numpy as np
import pytest

from oracle import nvfp4_moe_oracle as O
from nvfp4_block_scaled_07_gb300 import workloads as W


def test_hand_worked_batch():
    # token 0 prefers expert 0, token 1 expert 5, token 2 expert 1 (k_primary = 1),
    # so S = {0, 1, 5}; each token then takes its 3 best members of S.
    logits = np.array([[5, 4, 3, 2, 1, 0],
                       [0, 1, 2, 3, 4, 5],
                       [1, 5, 0, 4, 2, 3]], np.float32)
    idx, w = O.route_batch_aware(logits, None, 3, 1, "sigmoid")
    assert idx.tolist() == [[0, 1, 5], [5, 1, 0], [1, 5, 0]]
    # plain top-3 would touch all six experts
    std, _ = O.route_topk(logits, None, 3, "sigmoid")
    assert std.tolist() == [[0, 1, 2], [5, 4, 3], [1, 3, 5]]
    sig = 1 / (1 + np.exp(-np.array([5.0, 4.0, 0.0])))
    assert np.allclose(w[0], sig / sig.sum(), rtol=1e-15)


def test_hand_worked_fallback_outside_active_set():
    # one token, k_primary = 1: S = {1}; the other two slots go to its best outside S
    idx, _ = O.route_batch_aware(np.array([[1, 3, 2, 0]], np.float32), None, 3, 1, "softmax")
    assert idx.tolist() == [[1, 2, 0]]


def test_hand_worked_ties_and_bias():
    # bias creates ties in v = logit + bias; ties go to the lower index everywhere
    logits = np.array([[1.0, 0.5, 1.0, 0.0], [0.0, 1.0, 0.0, 1.0]], np.float32)
    bias = np.array([0.0, 0.5, 0.0, 0.0], np.float32)
    # v = [[1, 1, 1, 0], [0, 1.5, 0, 1]]: primaries (k_primary=1) are 0 and 1; S = {0, 1}
    idx, _ = O.route_batch_aware(logits, bias, 2, 1, "sigmoid")
    assert idx.tolist() == [[0, 1], [1, 0]]


@pytest.mark.parametrize("score", ["softmax", "sigmoid"])
def test_k_primary_equal_k_is_plain_topk(score):
    lg = np.random.default_rng(1).standard_normal((50, 32)).astype(np.float32)
    a = O.route_batch_aware(lg, None, 6, 6, score)
    b = O.route_topk(lg, None, 6, score)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_single_token_is_plain_topk():
    # with one token S is its own top-k_primary, so the fallback completes its plain top-k
    lg = np.random.default_rng(2).standard_normal((1, 64)).astype(np.float32)
    for k0 in (1, 3, 8):
        assert np.array_equal(O.route_batch_aware(lg, None, 8, k0, "sigmoid")[0], O.route_topk(lg, None, 8, "sigmoid")[0])


def _rank_key(v, e):
    return (-float(v[e]), e)


@pytest.mark.parametrize("T,E,k,k0", [(40, 64, 8, 1), (40, 64, 8, 2), (128, 256, 8, 4), (7, 16, 4, 1)])
def test_brute_force_properties(T, E, k, k0):
    lg = np.random.default_rng(T * E + k0).standard_normal((T, E)).astype(np.float32)
    bias = W.zipf_bias(E, 1.1)
    v = (lg + bias).astype(np.float32)
    idx, w = O.route_batch_aware(lg, bias, k, k0, "sigmoid")
    # the active set, from scratch: every token's k0 best by (value desc, index asc)
    S = set()
    for t in range(T):
        S.update(sorted(range(E), key=lambda e: _rank_key(v[t], e))[:k0])
    for t in range(T):
        chosen = [int(e) for e in idx[t]]
        assert len(set(chosen)) == k
        # the primaries come first, in rank order
        assert chosen[:k0] == sorted(range(E), key=lambda e: _rank_key(v[t], e))[:k0]
        if len(S) >= k:
            assert set(chosen) <= S
            # no unchosen member of S outranks a chosen one
            worst = max(_rank_key(v[t], e) for e in chosen)
            assert all(_rank_key(v[t], e) > worst for e in S - set(chosen))
        # slots follow the rank order: members of S first, then value, then index
        key = [((e not in S),) + _rank_key(v[t], e) for e in chosen]
        assert key == sorted(key)
    if len(S) >= k:
        assert set(np.unique(idx).tolist()) <= S
    # fewer (or as many) active experts than plain top-k
    std, _ = O.route_topk(lg, bias, k, "sigmoid")
    assert len(np.unique(idx)) <= len(np.unique(std))
    sig = 1 / (1 + np.exp(-np.take_along_axis(v, idx, 1).astype(np.float64)))
    assert np.allclose(w, sig / sig.sum(1, keepdims=True), rtol=1e-14)


def test_exhaustive_tiny_batches():
    """Every selection of a tiny batch against an enumeration of all k-subsets:
    the chosen set is the subset that maximises (members of S, then values)."""
    rng = np.random.default_rng(3)
    for _ in range(30):
        T, E, k, k0 = 3, 5, 3, int(rng.integers(1, 3))
        lg = rng.integers(-2, 3, size=(T, E)).astype(np.float32)   # many ties
        idx, _ = O.route_batch_aware(lg, None, k, k0, "sigmoid")
        S = set()
        for t in range(T):
            S.update(sorted(range(E), key=lambda e: (-lg[t, e], e))[:k0])
        for t in range(T):
            best = min(itertools.combinations(range(E), k),
                       key=lambda c: sorted(((e not in S), -lg[t, e], e) for e in c))
            assert sorted(idx[t].tolist()) == sorted(best)
