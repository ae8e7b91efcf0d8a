"""Pins of the oracle's sigmoid top-k routing and its expert grouping.

Routing is checked against a brute-force lexicographic sort (numpy) and
scipy's logistic function; the grouping against the invariants that define it.
"""
import numpy as np
import pytest
from scipy.special import expit

from mxfp4_latent_moe_gb300 import synth


def _brute_topk(logits, k):
    T, E = logits.shape
    ids = np.empty((T, k), np.int64)
    for t in range(T):
        ids[t] = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))[:k]
    return ids


@pytest.mark.parametrize("T,E,k", [(64, 896, 16), (50, 32, 4), (7, 33, 5), (5, 16, 16), (3, 1, 1)])
def test_route_ids_equal_brute_force_sort(orc, T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    logits = rng.normal(0, 1, (T, E)).astype(np.float32)
    ids, w = orc.route_topk(logits, k)
    assert np.array_equal(ids, _brute_topk(logits, k))
    sel = np.take_along_axis(logits, ids, axis=1).astype(np.float64)
    s = expit(sel)
    ref = s / s.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w, ref, rtol=1e-7, atol=0)
    np.testing.assert_allclose(w.astype(np.float64).sum(axis=1), 1.0, rtol=0, atol=1e-6)


def test_route_ties_go_to_lower_id_and_signed_zero_ties(orc):
    E, k = 64, 16
    logits = np.zeros((4, E), np.float32)
    logits[0, :] = 1.0                       # all equal: ids 0..15
    logits[1, ::2] = -0.0                    # -0 == +0
    logits[1, 40] = 2.0
    logits[2, :] = np.where(np.arange(E) % 3 == 0, 30.0, -30.0)  # saturating sigmoid
    logits[3, :] = np.arange(E)[::-1] % 7    # many repeated values
    ids, w = orc.route_topk(logits, k)
    assert list(ids[0]) == list(range(16))
    assert ids[1, 0] == 40 and list(ids[1, 1:]) == list(range(15))
    assert list(ids[2]) == [i for i in range(E) if i % 3 == 0][:16]
    assert np.array_equal(ids, _brute_topk(logits, k))
    np.testing.assert_allclose(w[0], 1.0 / 16, rtol=1e-7)


def test_route_k_equals_e_and_single_expert(orc):
    logits = np.array([[0.3]], np.float32)
    ids, w = orc.route_topk(logits, 1)
    assert ids[0, 0] == 0 and w[0, 0] == 1.0


def test_skewed_workload_is_dominated_by_top_ranked_experts(orc):
    wl = synth.shape("skew_small", T=2048, d=128, E=896, k=16, I=128, skew=True)
    x, logits = synth.make_activations(wl, seed=0)
    ids, _ = orc.route_topk(logits.numpy(), 16)
    counts = np.bincount(ids.ravel(), minlength=896)
    touched = int((counts > 0).sum())
    assert touched < 300                                # far fewer than 896
    assert counts.max() == 2048                          # some expert takes every token
    uni = synth.shape("uni_small", T=2048, d=128, E=896, k=16, I=128)
    _, logits_u = synth.make_activations(uni, seed=0)
    ids_u, _ = orc.route_topk(logits_u.numpy(), 16)
    assert (np.bincount(ids_u.ravel(), minlength=896) > 0).sum() > 850


def _check_grouping(ids, E, pad_m, out):
    T, k = ids.shape
    counts, offsets = out["counts"], out["offsets"]
    s2r, r2s = out["slot_to_row"], out["row_to_slot"]
    assert counts.sum() == T * k
    assert np.array_equal(counts, np.bincount(ids.ravel(), minlength=E))
    assert offsets[0] == 0
    assert np.all(offsets % pad_m == 0)
    assert np.all(np.diff(offsets) == (counts + pad_m - 1) // pad_m * pad_m)
    # slot -> row -> slot is the identity; padding rows hold -1
    assert np.array_equal(r2s[s2r], np.arange(T * k))
    assert (r2s == -1).sum() == offsets[E] - T * k
    for e in range(E):
        rows = np.arange(offsets[e], offsets[e] + counts[e])
        slots = r2s[rows]
        assert np.all(ids.ravel()[slots] == e)
        assert np.all(np.diff(slots // k) > 0)          # ascending token order
        assert np.all(r2s[offsets[e] + counts[e]: offsets[e + 1]] == -1)


@pytest.mark.parametrize("pad_m", [1, 16, 128])
def test_permute_invariants_random(orc, pad_m):
    rng = np.random.default_rng(pad_m)
    T, E, k = 300, 40, 6
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    _check_grouping(ids, E, pad_m, orc.permute(ids, E, pad_m))


def test_permute_empty_experts_and_one_hot_expert(orc):
    T, E, k = 200, 64, 4
    rng = np.random.default_rng(9)
    ids = np.stack([np.concatenate([[0], 1 + rng.permutation(10)[: k - 1]]) for _ in range(T)]).astype(np.int32)
    out = orc.permute(ids, E, 128)
    _check_grouping(ids, E, 128, out)
    assert out["counts"][0] == T                 # every token on expert 0
    assert np.all(out["counts"][11:] == 0)       # empty experts take no rows
    assert np.all(np.diff(out["offsets"])[11:] == 0)


def test_permute_rejects_bad_ids(orc):
    with pytest.raises(ValueError):
        orc.permute(np.array([[0, 0]], np.int32), 4, 1)      # repeated expert
    with pytest.raises(ValueError):
        orc.permute(np.array([[0, 4]], np.int32), 4, 1)      # out of range
    with pytest.raises(ValueError):
        orc.permute(np.array([[0, 1]], np.int32), 4, 128, rows_capacity=200)


def test_permute_zero_tokens(orc):
    out = orc.permute(np.zeros((0, 4), np.int32), 8, 16)
    assert out["offsets"][-1] == 0 and out["counts"].sum() == 0
