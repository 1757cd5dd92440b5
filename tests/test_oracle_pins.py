"""Pins for the CPU oracle: each test ties it to something other than itself.

Sources: values the pages print (the worked dispatch/combine example, Table 1,
Figure 2), closed forms, special cases that reduce to simpler formulas,
invariants of the method, and brute force on tiny inputs.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from moe_decode_layer_fp32_gb300 import synth

LN3 = math.log(3.0)


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# SiLU closed forms
# ---------------------------------------------------------------------------


def test_silu_closed_forms():
    assert O.silu(0.0) == 0.0
    # sigmoid(ln 3) = 3/4
    assert O.silu(LN3) == pytest.approx(0.75 * LN3, rel=1e-15)
    # sigmoid(-ln 3) = 1/4
    assert O.silu(-LN3) == pytest.approx(-0.25 * LN3, rel=1e-15)
    z = np.linspace(-8, 8, 33)
    # SiLU(-z) = SiLU(z) - z
    np.testing.assert_allclose(O.silu(-z), O.silu(z) - z, atol=1e-14)
    # large z: SiLU(z) -> z
    assert O.silu(60.0) == pytest.approx(60.0, rel=1e-15)


def test_bf16_decode_exact():
    vals = torch.tensor([1.0, -2.5, 0.0078125, 3.0e38, -1.0e-30], dtype=torch.float32)
    b = vals.to(torch.bfloat16)
    dec = O.to_f64(b)
    np.testing.assert_array_equal(dec, b.to(torch.float32).double().numpy())
    assert O.to_f64(torch.tensor([1.0], dtype=torch.bfloat16))[0] == 1.0


# ---------------------------------------------------------------------------
# The pages' worked 4-token / 4-expert top-2 example
# ---------------------------------------------------------------------------


def worked_example(golden):
    T = n = d = 4
    wr = np.full((n, d), -10.0)
    name = {"E1": 0, "E2": 1, "E3": 2, "E4": 3}
    for t, tok in enumerate(["T1", "T2", "T3", "T4"]):
        for ex, w in golden["choices"][tok]:
            wr[name[ex], t] = math.log(w)
    x = np.eye(T, d)
    return x, wr


def test_worked_example_routing(golden_dir):
    gd = load(golden_dir, "dispatch_combine_4tok_4exp_top2.json")
    x, wr = worked_example(gd)
    idx, p, _ = O.route(x, wr, k=2)
    np.testing.assert_array_equal(idx, np.array(gd["expected_idx"]))
    np.testing.assert_allclose(p, np.array(gd["expected_w"]), rtol=1e-12)


def test_worked_example_dispatch(golden_dir):
    gd = load(golden_dir, "dispatch_combine_4tok_4exp_top2.json")
    idx = np.array(gd["expected_idx"], np.int32)
    w = np.array(gd["expected_w"])
    D = O.dispatch(idx, w, n=4, g=1)
    np.testing.assert_array_equal(D["exp_count"], gd["expected_exp_count"])
    np.testing.assert_array_equal(D["exp_off"], gd["expected_exp_off"])
    np.testing.assert_array_equal(D["asg_tok"], gd["expected_asg_tok"])
    np.testing.assert_array_equal(D["asg_slot"], gd["expected_asg_slot"])
    np.testing.assert_array_equal(D["tok_asg"], gd["expected_tok_asg"])
    D2 = O.dispatch(idx, w, n=4, g=2)
    dg = gd["departments_g2"]
    np.testing.assert_array_equal(D2["dept_tok"], dg["expected_dept_tok"])
    np.testing.assert_array_equal(D2["dept_off"], dg["expected_dept_off"])
    np.testing.assert_allclose(D2["dept_w"], dg["expected_dept_w"], rtol=1e-15)


def test_worked_example_combine(golden_dir):
    gd = load(golden_dir, "dispatch_combine_4tok_4exp_top2.json")
    x, wr = worked_example(gd)
    n, I, d = 4, 2, 4
    wg = np.full((n, I, d), LN3)
    wu = np.zeros((n, I, d))
    wd = np.zeros((n, I, d))
    for e in range(n):
        for i in range(I):
            for t in range(d):
                wu[e, i, t] = (e + 1) * (i + 1) * (t + 1)
            wd[e, i, (e + i) % 4] = 1.0
    idx, p, _ = O.route(x, wr, k=2)
    y = O.vanilla_layer(x, idx, p, wg, wu, wd)
    expected = 0.75 * LN3 * np.array(gd["expected_y_over_three_quarters_ln3"])
    np.testing.assert_allclose(y, expected, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# Routing: brute force and special cases
# ---------------------------------------------------------------------------


def test_topk_matches_rank_definition():
    rng = np.random.default_rng(7)
    for trial in range(200):
        n = int(rng.choice([4, 8, 16]))
        k = int(rng.integers(1, n + 1))
        T = int(rng.integers(1, 6))
        d = int(rng.choice([8, 16]))
        x = rng.standard_normal((T, d))
        wr = rng.standard_normal((n, d)) * 0.3
        if trial % 3 == 0:                     # force exact ties
            wr[n // 2] = wr[0]
            if n > 3:
                wr[n - 1] = wr[1]
        bias = rng.standard_normal(n) * 0.1 if trial % 2 else None
        idx, p, info = O.route(x, wr, k, bias=bias)
        key = info["key32"]
        for t in range(T):
            for r, e in enumerate(idx[t]):
                # rank of e = number of experts strictly ahead of it
                ahead = sum(1 for f in range(n)
                            if key[t, f] > key[t, e] or (key[t, f] == key[t, e] and f < e))
                assert ahead == r
            assert p[t].sum() == pytest.approx(1.0, abs=1e-14)       # I4


def test_topk_softmax_uses_unbiased_logits():
    # bias moves the selection but not the weights
    x = np.array([[1.0, 0.0]])
    wr = np.array([[2.0, 0.0], [1.0, 0.0], [0.5, 0.0]])
    bias = np.array([-5.0, 0.0, 0.0], np.float32)
    idx, p, _ = O.route(x, wr, 2, bias=bias)
    assert list(idx[0]) == [1, 2]
    e1, e2 = math.exp(1.0), math.exp(0.5)
    np.testing.assert_allclose(p[0], [e1 / (e1 + e2), e2 / (e1 + e2)], rtol=1e-14)


def test_equal_logits_give_uniform_weights():
    x = np.ones((3, 8))
    wr = np.zeros((16, 8))
    idx, p, _ = O.route(x, wr, 4, scale=2.0)
    np.testing.assert_array_equal(idx, np.tile(np.arange(4), (3, 1)))   # I5
    np.testing.assert_allclose(p, np.full((3, 4), 0.5), rtol=1e-15)    # scale/k


def test_k_equals_n_routes_everything():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 8))
    wr = rng.standard_normal((5, 8))
    idx, p, _ = O.route(x, wr, 5)
    for t in range(2):
        assert sorted(idx[t]) == list(range(5))
        l = wr @ x[t]
        np.testing.assert_allclose(p[t], np.exp(l[idx[t]]) / np.exp(l).sum(), rtol=1e-13)


# ---------------------------------------------------------------------------
# Group-limited top-k ([DeaMoE] §3.3 k_dept; strict coverage of its Table 4)
# ---------------------------------------------------------------------------


def _rand_router(rng, T, d, n, ties=False):
    x = rng.standard_normal((T, d))
    wr = rng.standard_normal((n, d)) * 0.3
    if ties:
        wr[n // 2] = wr[0]
        wr[n - 1] = wr[1]
    return x, wr


def test_grouped_all_departments_is_plain_topk():
    # k_dept = m keeps every department: plain top-k, weights included
    rng = np.random.default_rng(11)
    for trial in range(60):
        g = int(rng.choice([1, 2, 4]))
        n = g * int(rng.integers(2, 6))
        k = int(rng.integers(1, n + 1))
        x, wr = _rand_router(rng, 3, 8, n, ties=trial % 3 == 0)
        bias = rng.standard_normal(n) * 0.1 if trial % 2 else None
        i0, p0, _ = O.route(x, wr, k, bias=bias, scale=1.5)
        i1, p1, _ = O.route_grouped(x, wr, k, g, n // g, bias=bias, scale=1.5)
        np.testing.assert_array_equal(i1, i0)
        np.testing.assert_array_equal(p1, p0)


def test_grouped_single_expert_departments_is_plain_topk():
    # g = 1: the k_dept >= k best departments are the k_dept best experts
    rng = np.random.default_rng(12)
    for trial in range(40):
        n = int(rng.integers(4, 12))
        k = int(rng.integers(1, n + 1))
        k_dept = int(rng.integers(k, n + 1))
        x, wr = _rand_router(rng, 2, 8, n, ties=trial % 2 == 0)
        for strict in (False, True):
            i0, p0, _ = O.route(x, wr, k)
            # strict needs k >= k_dept, and k <= k_dept * g = k_dept
            i1, p1, _ = O.route_grouped(x, wr, k, 1, k if strict else k_dept, strict=strict)
            np.testing.assert_array_equal(i1, i0)
            np.testing.assert_array_equal(p1, p0)


def _keys32(x, wr, bias):
    b = np.zeros(wr.shape[0], np.float32) if bias is None else np.asarray(bias, np.float32)
    return (np.asarray(x, np.float64) @ np.asarray(wr, np.float64).T).astype(np.float32) + b


@pytest.mark.parametrize("strict", [False, True])
def test_grouped_matches_bruteforce(strict):
    # Distinct keys (continuous random inputs).  Kept departments: the k_dept-
    # subset with the largest summed department score (score = best key).
    # Soft: the k-subset of the kept departments' experts with the largest key
    # sum.  Strict: the same, over the k-subsets that cover every kept
    # department.  Order: descending key.
    rng = np.random.default_rng(13 + strict)
    for trial in range(80):
        g = int(rng.choice([2, 3]))
        m = int(rng.integers(2, 5))
        n = g * m
        k_dept = int(rng.integers(1, m + 1))
        k = int(rng.integers(k_dept if strict else 1, k_dept * g + 1))
        x, wr = _rand_router(rng, 2, 6, n)
        bias = rng.standard_normal(n) * 0.2 if trial % 2 else None
        idx, p, _ = O.route_grouped(x, wr, k, g, k_dept, bias=bias, strict=strict)
        key = _keys32(x, wr, bias)
        for t in range(2):
            score = [key[t, j * g:(j + 1) * g].max() for j in range(m)]
            kept = max(itertools.combinations(range(m), k_dept), key=lambda c: sum(score[j] for j in c))
            pool = [e for e in range(n) if e // g in kept]
            subsets = [c for c in itertools.combinations(pool, k)
                       if not strict or {e // g for e in c} == set(kept)]
            best = max(subsets, key=lambda c: sum(float(key[t, e]) for e in c))
            assert sorted(idx[t]) == sorted(best)
            assert all(key[t, a] > key[t, b] for a, b in zip(idx[t], idx[t][1:]))
            l = np.asarray(x[t], np.float64) @ np.asarray(wr, np.float64).T
            ex = np.exp(l[idx[t]])
            np.testing.assert_allclose(p[t], ex / ex.sum(), rtol=1e-13)


def test_grouped_hand_example():
    # Logits of one token over 8 experts in 4 departments of 2 (x = e_0, so the
    # router's first column gives the logits).
    #   logits  [5, 1 | 4.9, 0 | 4.8, 4.7 | 0, 0]
    #   department scores 5, 4.9, 4.8, 0 -> k_dept = 2 keeps departments 0, 1
    #   plain top-3: 0, 2, 4; group-limited top-3 (soft): 0, 2, 1
    l = np.array([5.0, 1.0, 4.9, 0.0, 4.8, 4.7, 0.0, 0.0])
    wr = np.zeros((8, 4))
    wr[:, 0] = l
    x = np.array([[1.0, 0.0, 0.0, 0.0]])
    assert list(O.route(x, wr, 3)[0][0]) == [0, 2, 4]
    idx, p, info = O.route_grouped(x, wr, 3, 2, 2)
    assert list(idx[0]) == [0, 2, 1]
    assert list(info["kept"][0]) == [0, 1]
    ex = np.exp(np.array([5.0, 4.9, 1.0]))
    np.testing.assert_allclose(p[0], ex / ex.sum(), rtol=1e-14)
    # Strict, k = 3, k_dept = 3: departments 0, 1, 2 kept.  Soft picks 0, 2, 4
    # (3 departments): already covered, strict leaves it.
    assert list(O.route_grouped(x, wr, 3, 2, 3, strict=True)[0][0]) == [0, 2, 4]
    # logits [5, 4.9 | 4.8, 4.7 | 1, 0 | 0.5, 0.2], k = 3, k_dept = 3: kept 0, 1, 2;
    # soft picks 0, 1, 2 (departments 0, 1); strict swaps the lowest-ranked
    # expert of a doubly covered department (1) for department 2's leader (4).
    wr[:, 0] = [5.0, 4.9, 4.8, 4.7, 1.0, 0.0, 0.5, 0.2]
    assert list(O.route_grouped(x, wr, 3, 2, 3)[0][0]) == [0, 1, 2]
    idx, p, _ = O.route_grouped(x, wr, 3, 2, 3, strict=True)
    assert list(idx[0]) == [0, 2, 4]
    ex = np.exp(np.array([5.0, 4.8, 1.0]))
    np.testing.assert_allclose(p[0], ex / ex.sum(), rtol=1e-14)


def test_grouped_coverage_invariants():
    rng = np.random.default_rng(14)
    for trial in range(60):
        g = int(rng.choice([2, 4, 8]))
        m = int(rng.integers(2, 9))
        n = g * m
        k_dept = int(rng.integers(1, m + 1))
        k = int(rng.integers(k_dept, min(k_dept * g, 16) + 1))
        x, wr = _rand_router(rng, 4, 8, n, ties=trial % 4 == 0)
        bias = rng.standard_normal(n) * 0.1 if trial % 2 else None
        soft, ps, info = O.route_grouped(x, wr, k, g, k_dept, bias=bias, scale=2.0)
        strict, pt, _ = O.route_grouped(x, wr, k, g, k_dept, bias=bias, scale=2.0, strict=True)
        for t in range(4):
            kept = set(info["kept"][t])
            assert len(set(soft[t])) == k and len(set(strict[t])) == k
            assert {e // g for e in soft[t]} <= kept
            assert {e // g for e in strict[t]} == kept
            if len({e // g for e in soft[t]}) == k_dept:
                np.testing.assert_array_equal(strict[t], soft[t])
            assert ps[t].sum() == pytest.approx(2.0, abs=1e-13)
            assert pt[t].sum() == pytest.approx(2.0, abs=1e-13)


def test_grouped_rejects_bad_arguments():
    x, wr = np.ones((1, 4)), np.ones((8, 4))
    for args in [(3, 3, 1), (3, 2, 0), (3, 2, 5), (5, 2, 2), (9, 8, 1)]:
        with pytest.raises(ValueError):
            O.route_grouped(x, wr, *args)
    with pytest.raises(ValueError):
        O.route_grouped(x, wr, 1, 2, 2, strict=True)


# ---------------------------------------------------------------------------
# Router-bias load balancing (DeepSeekMoE guide, auxiliary-loss-free section)
# ---------------------------------------------------------------------------


def test_bias_sign_rule_hand_example():
    # 8 tokens over 4 experts: target 2; expert 0 is over (-gamma), expert 1
    # under (+gamma), experts 2 and 3 on target (unchanged); dyadic values so
    # that every result is exact
    b = O.bias_update([3, 1, 2, 2], np.array([0.5, -0.25, 0.0, 1.0], np.float32), 0.125)
    np.testing.assert_array_equal(b, np.array([0.375, -0.125, 0.0, 1.0], np.float32))
    # a target that is not an integer: 1 token over 3 experts (target 1/3)
    b = O.bias_update([1, 0, 0], np.zeros(3, np.float32), 0.5)
    np.testing.assert_array_equal(b, np.array([-0.5, 0.5, 0.5], np.float32))


def test_bias_proportional_rule_hand_example():
    b = O.bias_update([4, 0, 2, 2], np.zeros(4, np.float32), 0.125, rule=O.BIAS_PROPORTIONAL)
    np.testing.assert_array_equal(b, np.array([-0.25, 0.25, 0.0, 0.0], np.float32))
    # target 1/3: deltas gamma * (1/3 - 1), gamma / 3, gamma / 3 with gamma = 0.75
    b = O.bias_update([1, 0, 0], np.zeros(3, np.float32), 0.75, rule=O.BIAS_PROPORTIONAL)
    np.testing.assert_allclose(b, [-0.5, 0.25, 0.25], rtol=2 ** -23)


def test_bias_update_invariants():
    rng = np.random.default_rng(21)
    for trial in range(50):
        n = int(rng.integers(1, 300))
        c = rng.integers(0, 40, n)
        b = (rng.standard_normal(n) * 0.1).astype(np.float32)
        gamma = float(rng.uniform(1e-4, 1e-2))
        # proportional: the deltas sum to zero, so the bias sum is kept
        bp = O.bias_update(c, b, gamma, rule=O.BIAS_PROPORTIONAL)
        assert abs(float(bp.astype(np.float64).sum() - b.astype(np.float64).sum())) \
            <= n * 2 ** -23 * (np.abs(b).max() + gamma * c.max() + 1)
        # sign: every bias moves by exactly 0 or +-gamma (before fp32 rounding)
        bs = O.bias_update(c, b, gamma)
        mean = c.sum() / n
        for i in range(n):
            bi = float(b[i])
            want = bi - gamma if c[i] > mean else bi + gamma if c[i] < mean else bi
            assert bs[i] == np.float32(want)
    # balanced load: nothing moves under either rule, the ratio is 1
    for rule in (O.BIAS_SIGN, O.BIAS_PROPORTIONAL):
        b = np.arange(8, dtype=np.float32)
        np.testing.assert_array_equal(O.bias_update([5] * 8, b, 0.1, rule=rule), b)
        np.testing.assert_array_equal(O.bias_update([0] * 8, b, 0.1, rule=rule), b)
    assert O.imbalance_ratio([5] * 8) == 1.0


def test_imbalance_ratio_closed_forms():
    assert O.imbalance_ratio([3, 1, 2, 2]) == 1.5
    assert O.imbalance_ratio([0, 0, 7, 0, 0]) == 5.0        # one expert takes all: n
    assert O.imbalance_ratio([0, 0, 0]) == 0.0               # nothing routed
    rng = np.random.default_rng(22)
    for _ in range(20):
        c = rng.integers(0, 50, int(rng.integers(1, 64)))
        if c.sum():
            r = O.imbalance_ratio(c)
            assert 1.0 <= r <= len(c)


def test_sign_rule_reduces_imbalance():
    # The guide's claim: the per-step sign update balances the load.  A router
    # skewed towards the low expert ids (a logit offset from 1.5 down to -1.5)
    # starts near 2.3x the mean load on its busiest expert; after 150 steps of
    # 256 tokens the ratio is near the sampling noise of a balanced router.
    rng = np.random.default_rng(0)
    n, k, T, d = 16, 2, 256, 16
    wr = np.concatenate([rng.standard_normal((n, d)) * 0.5, np.linspace(1.5, -1.5, n)[:, None]], 1)
    b = np.zeros(n, np.float32)
    hist = []
    for step in range(150):
        x = np.concatenate([rng.standard_normal((T, d)), np.ones((T, 1))], 1)
        idx, _, _ = O.route(x, wr, k, bias=b)
        c = np.bincount(idx.reshape(-1), minlength=n)
        hist.append(O.imbalance_ratio(c))
        b = O.bias_update(c, b, 0.02)
    assert hist[0] > 2.0
    assert np.mean(hist[-20:]) < 1.5
    # the bias ends up lowest where the skew was strongest
    assert b[0] < b[-1]


# ---------------------------------------------------------------------------
# Dense brute force vs the gathered per-token evaluation
# ---------------------------------------------------------------------------


def dense_layer(x, gate_matrix, wg, wu, wd):
    """All experts on all tokens, masked afterwards by the gate matrix."""
    G = np.einsum("eid,td->eti", wg, x)
    U = np.einsum("eid,td->eti", wu, x)
    H = G / (1.0 + np.exp(-G)) * U
    Y = np.einsum("eti,eid->etd", H, wd)
    return np.einsum("te,etd->td", gate_matrix, Y)


def test_vanilla_matches_dense_bruteforce():
    rng = np.random.default_rng(11)
    for trial in range(200):
        d = int(rng.choice([8, 16]))
        n = int(rng.choice([4, 8]))
        k = int(rng.integers(1, 4))
        T = int(rng.integers(1, 9))
        I = 4
        x = rng.standard_normal((T, d))
        wr = rng.standard_normal((n, d)) * 0.5
        wg, wu, wd = (rng.standard_normal((n, I, d)) * 0.3 for _ in range(3))
        idx, p, _ = O.route(x, wr, k)
        Gm = np.zeros((T, n))
        for t in range(T):
            for s in range(k):
                Gm[t, idx[t, s]] = p[t, s]
        y = O.vanilla_layer(x, idx, p, wg, wu, wd)
        np.testing.assert_allclose(y, dense_layer(x, Gm, wg, wu, wd), rtol=1e-11, atol=1e-12)


def test_shared_expert_added_with_weight_one():
    rng = np.random.default_rng(5)
    T, d, n, I, k = 3, 8, 4, 4, 2
    x = rng.standard_normal((T, d))
    wr = rng.standard_normal((n, d))
    wg, wu, wd = (rng.standard_normal((n, I, d)) for _ in range(3))
    sg, su, sd = (rng.standard_normal((6, d)) for _ in range(3))
    idx, p, _ = O.route(x, wr, k)
    y0 = O.vanilla_layer(x, idx, p, wg, wu, wd)
    y1 = O.vanilla_layer(x, idx, p, wg, wu, wd, shared=(sg, su, sd))
    # the shared expert is the only expert of a 1-expert, top-1 layer (weight 1)
    ys = O.vanilla_layer(x, np.zeros((T, 1), np.int32), np.ones((T, 1)),
                         sg[None], su[None], sd[None])
    np.testing.assert_allclose(y1 - y0, ys, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# DeaMoE form C invariants
# ---------------------------------------------------------------------------


def rand_formc(rng, T=5, d=16, n=8, g=4, I_sh=8, I_pr=4, k=3):
    x = rng.standard_normal((T, d))
    wr = rng.standard_normal((n, d)) * 0.5
    m = n // g
    dept = [rng.standard_normal((m, I_sh, d)) * 0.3 for _ in range(3)]
    priv = [rng.standard_normal((n, I_pr, d)) * 0.3 for _ in range(3)]
    return x, wr, dept, priv


def test_formc_g1_no_private_is_vanilla():
    rng = np.random.default_rng(21)
    x, wr, dept, _ = rand_formc(rng, n=8, g=1, I_sh=8)
    idx, p, _ = O.route(x, wr, 3)
    y_dea = O.deamoe_layer_c(x, idx, p, 1, *dept)
    y_van = O.vanilla_layer(x, idx, p, *dept)
    np.testing.assert_array_equal(y_dea, y_van)                           # I1


def test_formc_zero_private_reduces_to_department_ffn():
    """Zero private weights: y_t = sum_j omega_{t,j} FFN_j(x_t), the two-stage
    grouping of DeaMoE §3.2 applied to the department backbones."""
    rng = np.random.default_rng(22)
    for g in (2, 4):
        x, wr, dept, priv = rand_formc(rng, g=g)
        zero = [np.zeros_like(w) for w in priv]
        idx, p, _ = O.route(x, wr, 3)
        y = O.deamoe_layer_c(x, idx, p, g, *dept, *zero)
        D = O.dispatch(idx, p, n=8, g=g)
        ref = np.zeros_like(y)
        m = 8 // g
        for j in range(m):
            for pos in range(D["dept_off"][j], D["dept_off"][j + 1]):
                t = D["dept_tok"][pos]
                ref[t] += D["dept_w"][pos] * O.swiglu_expert(x[t], dept[0][j], dept[1][j], dept[2][j])
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)          # I2


def test_formc_equals_vanilla_with_materialised_weights():
    rng = np.random.default_rng(23)
    g, n = 4, 8
    x, wr, dept, priv = rand_formc(rng, g=g, n=n)
    idx, p, _ = O.route(x, wr, 3)
    y = O.deamoe_layer_c(x, idx, p, g, *dept, *priv)
    # materialise: expert e = rows of department e//g (np.repeat) over its private rows
    mats = [np.concatenate([np.repeat(dept[a], g, axis=0), priv[a]], axis=1) for a in range(3)]
    y_ref = O.vanilla_layer(x, idx, p, *mats)
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)            # I3


def test_layer_token_permutation_equivariance():
    rng = np.random.default_rng(24)
    x, wr, dept, priv = rand_formc(rng, T=6)
    perm = rng.permutation(6)
    idx, p, _ = O.route(x, wr, 3)
    y = O.deamoe_layer_c(x, idx, p, 4, *dept, *priv)
    idx2, p2, _ = O.route(x[perm], wr, 3)
    y2 = O.deamoe_layer_c(x[perm], idx2, p2, 4, *dept, *priv)
    np.testing.assert_allclose(y2, y[perm], rtol=1e-13, atol=1e-13)        # I6


def test_dispatch_lists_are_a_partition():
    rng = np.random.default_rng(25)
    for trial in range(100):
        n, g = 16, int(rng.choice([1, 2, 4, 8]))
        T, k = int(rng.integers(1, 20)), int(rng.integers(1, 6))
        idx = np.stack([rng.permutation(n)[:k] for _ in range(T)]).astype(np.int32)
        p = rng.random((T, k))
        D = O.dispatch(idx, p, n, g)
        # every (token, slot) appears once, grouped by expert, tokens ascending
        seen = set()
        for e in range(n):
            toks = D["asg_tok"][D["exp_off"][e]:D["exp_off"][e + 1]]
            assert list(toks) == sorted(toks)
            for pos in range(D["exp_off"][e], D["exp_off"][e + 1]):
                t, s = int(D["asg_tok"][pos]), int(D["asg_slot"][pos])
                assert idx[t, s] == e and D["tok_asg"][t, s] == pos
                seen.add((t, s))
        assert len(seen) == T * k
        if g > 1:
            for j in range(n // g):
                toks = list(D["dept_tok"][D["dept_off"][j]:D["dept_off"][j + 1]])
                want = sorted({t for t in range(T) for s in range(k) if idx[t, s] // g == j})
                assert toks == want


# ---------------------------------------------------------------------------
# DeaMoE form P (eq. 4)
# ---------------------------------------------------------------------------


def test_formp_zero_A_gives_zero():
    rng = np.random.default_rng(31)
    h, r = 6, 4
    W = [rng.standard_normal((r, h)) for _ in range(3)]
    Z = np.zeros((r, r))
    out = O.deamoe_expert_p(rng.standard_normal(h), *W, Z, Z, Z)
    np.testing.assert_array_equal(out, np.zeros(h))


def test_formp_identity_A_closed_form():
    """Identity init (DeaMoE §3.4): with A = I each expert reduces to
    W_d^T SiLU(SiLU(SiLU(W_g x)) * SiLU(W_u x))."""
    rng = np.random.default_rng(32)
    h, r = 6, 4
    wg, wu, wd = (rng.standard_normal((r, h)) for _ in range(3))
    x = rng.standard_normal(h)
    Id = np.eye(r)
    out = O.deamoe_expert_p(x, wg, wu, wd, Id, Id, Id)
    s = lambda z: z / (1 + np.exp(-z))
    ref = wd.T @ s(s(s(wg @ x)) * s(wu @ x))
    np.testing.assert_allclose(out, ref, rtol=1e-14)


def test_formp_hand_example():
    """h = r = 2, worked by hand so every SiLU argument is 0 or ln 3:
    W_g x = [ln3, 0] -> sigma -> [3/4 ln3, 0] -> A_g (4/3) -> [ln3, 0] -> SiLU -> [3/4 ln3, 0];
    W_u x = [0, ln3] -> sigma -> [0, 3/4 ln3] -> A_u (swap) -> [3/4 ln3, 0];
    product [9/16 ln3^2, 0] -> A_d^T -> [ln3, 0] -> sigma -> [3/4 ln3, 0];
    W_d^T [3/4 ln3, 0] = 3/4 ln3 * W_d[0, :] = [3/2 ln3, -3/4 ln3]."""
    x = np.array([LN3, 0.0])
    wg = np.array([[1.0, 0.0], [0.0, 1.0]])
    ag = np.array([[4.0 / 3.0, 0.0], [0.0, 1.0]])
    wu = np.array([[0.0, 1.0], [1.0, 0.0]])
    au = np.array([[0.0, 1.0], [1.0, 0.0]])
    c = 1.0 / (0.5625 * LN3)
    ad = np.array([[c, 0.0], [7.0, 1.0]])      # A_d^T [a, 0] = [c a, 0]; A_d [a, 0] would not be
    wd = np.array([[2.0, -1.0], [5.0, 7.0]])   # W_d^T picks row 0; W_d would not
    out = O.deamoe_expert_p(x, wg, wu, wd, ag, au, ad)
    np.testing.assert_allclose(out, [1.5 * LN3, -0.75 * LN3], rtol=1e-14)


def test_formp_layer_combines_per_eq3():
    rng = np.random.default_rng(33)
    T, h, r, n, g, k = 3, 6, 4, 8, 4, 2
    x = rng.standard_normal((T, h))
    wr = rng.standard_normal((n, h))
    W = [rng.standard_normal((n // g, r, h)) for _ in range(3)]
    A = [rng.standard_normal((n, r, r)) * 0.5 for _ in range(3)]
    idx, p, _ = O.route(x, wr, k)
    y = O.deamoe_layer_p(x, idx, p, g, *W, *A)
    # Two-stage reading (DeaMoE §3.2): O^j = W_d^T sum_i p_i Z^{j,i}
    ref = np.zeros_like(y)
    s = lambda z: z / (1 + np.exp(-z))
    for t in range(T):
        by_dept = {}
        for q in range(k):
            e = idx[t, q]
            j = e // g
            Xg, Xu = s(W[0][j] @ x[t]), s(W[1][j] @ x[t])
            Y = s(A[0][e] @ Xg) * (A[1][e] @ Xu)
            by_dept[j] = by_dept.get(j, 0) + p[t, q] * s(A[2][e].T @ Y)
        for j, Zs in by_dept.items():
            ref[t] += W[2][j].T @ Zs
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# Table 1 and Figure 2
# ---------------------------------------------------------------------------


def test_table1_ratios(golden_dir):
    gd = load(golden_dir, "table1_fig2.json")
    for name, r in gd["rows"].items():
        fl, pa = O.table1_ratios(r["h"], r["r"], r["n_base"], r["k_base"], r["m"], r["n"],
                                 r["k_dept"], r["k"])
        assert round(pa, 3) == pytest.approx(r["params"], abs=1e-3 + 1e-9), name
        if r["flops"] is not None:
            assert round(fl, 3) == pytest.approx(r["flops"], abs=1e-3 + 1e-9), name


def test_figure2_dsv3_loading_bounds(golden_dir):
    gd = load(golden_dir, "table1_fig2.json")
    r = gd["rows"]["DeepSeek-V3"]
    f = gd["figure2_dsv3"]
    for with_router in (False, True):
        ratios = [100 * O.loading_ratio_formp(r["h"], r["r"], r["n_base"], r["k_base"], r["n"],
                                              r["m"], r["k"], T, with_router)
                  for T in range(f["batch_range"][0], f["batch_range"][1] + 1)]
        assert min(ratios) == pytest.approx(f["min_percent"], abs=f["tolerance_pp"])
        assert max(ratios) == pytest.approx(f["max_percent"], abs=f["tolerance_pp"])
    # the non-monotonic shape the figure describes: falls, then rises toward 1
    rt = [O.loading_ratio_formp(7168, 2048, 256, 8, 864, 8, 10, T) for T in (1, 16, 512)]
    assert rt[1] < rt[0] and rt[1] < rt[2] and rt[2] < 1.0


def test_expected_active_counts_monte_carlo():
    """E[A_e], E[A_d] closed forms against the oracle's dispatch counts for
    uniform k-of-n routing (10^4 trials)."""
    rng = np.random.default_rng(41)
    n, k, g, T = 64, 8, 8, 4
    trials = 10000
    Ae = np.empty(trials)
    Ad = np.empty(trials)
    for i in range(trials):
        idx = np.stack([rng.choice(n, k, replace=False) for _ in range(T)]).astype(np.int32)
        occupied = np.zeros(n, bool)
        occupied[idx.ravel()] = True
        Ae[i] = occupied.sum()
        Ad[i] = len(set(int(e) // g for e in idx.ravel()))
    # 4-sigma bands on the sample means
    assert abs(Ae.mean() - O.expected_active_experts(n, k, T)) < 4 * Ae.std() / math.sqrt(trials)
    assert abs(Ad.mean() - O.expected_active_depts(n, k, g, T)) < 4 * Ad.std() / math.sqrt(trials)
    # and the oracle's dispatch agrees with the direct count on a sample
    for i in range(50):
        idx = np.stack([rng.choice(n, k, replace=False) for _ in range(T)]).astype(np.int32)
        D = O.dispatch(idx, np.ones((T, k)), n, g)
        assert len(D["active_experts"]) == len(set(idx.ravel()))
        assert len(D["active_depts"]) == len(set(int(e) // g for e in idx.ravel()))


def test_unique_bytes_matches_touched_tensors():
    """The closed-form byte count equals the bytes of the weight slices the
    literal evaluation touches (router + shared + active units)."""
    shape = synth.TINY_DEAMOE
    L = synth.make_layer(shape, seed=0)
    x = synth.hidden(4, shape.d, seed=0)
    idx, p, _ = O.route(x, L["router"], shape.k)
    D = O.dispatch(idx, p, shape.n, shape.g)
    touched = L["router"].numel() * L["router"].element_size()
    for j in D["active_depts"]:
        touched += sum(L[key][int(j)].numel() * L[key].element_size() for key in ("dgate", "dup", "ddown"))
    for e in D["active_experts"]:
        touched += sum(L[key][int(e)].numel() * L[key].element_size() for key in ("pgate", "pup", "pdown"))
    U = O.unique_bytes_deamoe_c(shape.d, shape.n, shape.I_sh, shape.I_pr, 0,
                                len(D["active_depts"]), len(D["active_experts"]), 4)
    assert U == touched
    # vanilla with a shared expert, bf16
    Uv = O.unique_bytes_vanilla(2048, 128, 768, 256, 10, 2)
    assert Uv == 4 * 2048 * 128 + 2 * 3 * 2048 * (10 * 768 + 256)


def test_unique_bytes_formp_matches_touched_tensors():
    """Form P: the closed-form byte count equals the bytes of the tensors one
    literal evaluation of eq. (4) touches -- the fp32 router, the three
    [r, h] department matrices of every department a token reaches and the
    three [r, r] A-matrices of every selected expert ([DeaMoE] §3.1, §3.3)."""
    shape = synth.TINY_FORMP
    L = synth.make_layer(shape, seed=2)
    for T, k_dept in ((1, 2), (5, 2), (9, 0)):
        x = synth.hidden(T, shape.d, seed=T)
        if k_dept:
            idx, p, _ = O.route_grouped(x, L["router"], shape.k, shape.g, k_dept)
        else:
            idx, p, _ = O.route(x, L["router"], shape.k)
        depts = sorted({int(e) // shape.g for e in idx.ravel()})
        experts = sorted({int(e) for e in idx.ravel()})
        touched = L["router"].numel() * L["router"].element_size()
        for j in depts:
            touched += sum(L[key][j].numel() * L[key].element_size() for key in ("dgate", "dup", "ddown"))
        for e in experts:
            touched += sum(L[key][e].numel() * L[key].element_size() for key in ("agate", "aup", "adown"))
        D = O.dispatch(idx, p, shape.n, shape.g)
        assert list(D["active_depts"]) == depts and list(D["active_experts"]) == experts
        U = O.unique_bytes_deamoe_p(shape.d, shape.n, shape.I_sh, len(D["active_depts"]),
                                    len(D["active_experts"]), 2)
        assert U == touched, (T, k_dept, U, touched)
    # a department reached by several experts of one token is read once: one
    # token, every selected expert in department 0 (k_dept = 1)
    idx = np.arange(shape.k, dtype=np.int32)[None, :]
    D = O.dispatch(idx, np.ones((1, shape.k)), shape.n, shape.g)
    assert len(D["active_depts"]) == 1
    assert O.unique_bytes_deamoe_p(shape.d, shape.n, shape.I_sh, 1, shape.k, 2) == (
        4 * shape.d * shape.n + 2 * 3 * shape.I_sh * (shape.d + shape.k * shape.I_sh))


# ---------------------------------------------------------------------------
# FP8 (E4M3) weights with per-row scales
# ---------------------------------------------------------------------------


def test_e4m3_decode_hand_values():
    # worked from the layout: sign | 4 exponent bits (bias 7) | 3 mantissa bits
    codes = np.array([0x00, 0x80, 0x38, 0xB8, 0x7E, 0xFE, 0x01, 0x07, 0x08, 0x3C, 0x40, 0x30],
                     np.uint8)
    want = [0.0, -0.0, 1.0, -1.0, 448.0, -448.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.5, 2.0, 0.5]
    got = O.e4m3_bits_to_f64(codes)
    np.testing.assert_array_equal(got, want)
    assert np.signbit(got[1]) and not np.signbit(got[0])
    assert np.isnan(O.e4m3_bits_to_f64(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_decode_matches_library_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = O.e4m3_bits_to_f64(codes.numpy())
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(lib))
    ok = ~np.isnan(lib)
    np.testing.assert_array_equal(mine[ok], lib[ok])


def test_dequant_rows_scales_each_row():
    codes = np.array([[[0x38, 0x40], [0xB8, 0x30]]], np.uint8)      # 1, 2 / -1, 0.5
    scale = np.array([[0.25, 3.0]], np.float32)
    np.testing.assert_array_equal(O.dequant_rows_e4m3(codes, scale),
                                  [[[0.25, 0.5], [-3.0, 1.5]]])


def test_e4m3_row_quantisation_error_bound():
    """Round to nearest even with 3 mantissa bits: a weight stored as row scale
    times an E4M3 code is within 2^-4 of itself (relative) in the normal range,
    and within half the smallest subnormal step (2^-10 times the scale) below."""
    g = torch.Generator().manual_seed(5)
    w = torch.randn((64, 512), generator=g) * 0.02
    codes, scale = synth.quantize_rows_e4m3(w)
    back = O.dequant_rows_e4m3(codes, scale)
    wd = w.double().numpy()
    bound = np.maximum(2.0 ** -4 * np.abs(wd), 2.0 ** -10 * scale.double().numpy()[:, None])
    assert (np.abs(back - wd) <= bound * (1 + 1e-12)).all()
    # the row maximum is represented exactly (it maps to 448)
    np.testing.assert_allclose(np.abs(back).max(axis=1), np.abs(wd).max(axis=1), rtol=1e-7)
