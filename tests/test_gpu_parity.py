"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Routing indices and dispatch lists must match bit-exactly (certified fp32
near-ties excepted, see helpers.compare_routing; the lists of a step with one
are compared with the oracle's lists of the device's own routing); outputs
must match within the output tolerance, max|y - y_ref| / max|y_ref| <= 2e-2
for bf16 weights and 1e-4 for fp32 weights, and within the kernels' own
accuracy, 1e-4, for every weight storage (helpers.KERNEL_TOL).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from moe_decode_layer_fp32_gb300 import synth
from oracle import moe_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return H.ensure_built()


def route_on_gpu(B, x, wr, bias, k, scale=1.0):
    T = x.shape[0]
    n = wr.shape[0]
    ws = B.new_workspace(T, n, k, 1)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    B.moe_route_topk(x, wr, bias, k, scale, idx, w, ws)
    torch.cuda.synchronize()
    return ws, idx.cpu().numpy(), w.cpu().numpy()


# ---------------------------------------------------------------------------
# Routing
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("shape", [synth.TINY_VANILLA, synth.VANILLA_128E, synth.DEAMOE_7B,
                                   synth.DSV3_VANILLA, synth.ZIPF_DEAMOE],
                         ids=lambda s: s.name)
def test_route_topk_matches_oracle(B, shape):
    ties_total = 0
    for T in sorted(set(shape.batches) | {1}):
        for seed in (0, 1):
            wr = synth.router(shape.d, shape.n, seed, DEV)
            bias = (synth.zipf_bias(shape.n, shape.zipf_g, shape.zipf, seed).to(DEV)
                    if shape.zipf > 0 else None)
            x = synth.hidden(T, shape.d, seed + 100 * T, DEV)
            _, gi, gw = route_on_gpu(B, x, wr, bias, shape.k)
            oi, op, info = O.route(x, wr, shape.k, bias=bias)
            ties_total += len(H.compare_routing(gi, gw, oi, op, info, x, wr))
    assert ties_total <= 1


def test_route_worked_example(B, golden_dir):
    gd = json.load(open(os.path.join(golden_dir, "dispatch_combine_4tok_4exp_top2.json")))
    n = d_min = 8   # the device needs d % 8 == 0: pad the 4-wide example with zero columns
    wr = torch.full((4, d_min), 0.0)
    wr[:, :4] = -10.0
    name = {"E1": 0, "E2": 1, "E3": 2, "E4": 3}
    for t, tok in enumerate(["T1", "T2", "T3", "T4"]):
        for ex, w in gd["choices"][tok]:
            wr[name[ex], t] = math.log(w)
    x = torch.zeros((4, d_min))
    x[:, :4] = torch.eye(4)
    ws, gi, gw = route_on_gpu(B, x.to(DEV), wr.to(DEV), None, 2)
    np.testing.assert_array_equal(gi, gd["expected_idx"])
    np.testing.assert_allclose(gw, gd["expected_w"], rtol=1e-6)
    # and the device dispatch of that routing reproduces the page's groups
    for g in (1, 2):
        ws = B.new_workspace(4, 4, 2, g)
        B.moe_dispatch(torch.tensor(gi, device=DEV), torch.tensor(gw, device=DEV), 4, g, ws)
        dev = H.dispatch_lists(B, ws, 4, 4, 2, g)
        np.testing.assert_array_equal(dev["exp_off"], gd["expected_exp_off"])
        np.testing.assert_array_equal(dev["asg_tok"], gd["expected_asg_tok"])
        np.testing.assert_array_equal(dev["tok_asg"], gd["expected_tok_asg"])
        if g == 2:
            dg = gd["departments_g2"]
            np.testing.assert_array_equal(dev["dept_tok"], dg["expected_dept_tok"])
            np.testing.assert_array_equal(dev["dept_off"], dg["expected_dept_off"])
            np.testing.assert_allclose(dev["dept_w"], dg["expected_dept_w"], rtol=1e-6)


def test_route_ties_go_to_lower_index(B):
    T, d, n, k = 3, 16, 40, 5
    x = torch.ones((T, d), device=DEV)
    wr = torch.zeros((n, d), device=DEV)
    _, gi, gw = route_on_gpu(B, x, wr, None, k, scale=2.5)
    np.testing.assert_array_equal(gi, np.tile(np.arange(k), (T, 1)))
    np.testing.assert_allclose(gw, np.full((T, k), 2.5 / k), rtol=1e-6)


def test_route_k_equals_n_and_bias(B):
    T, d, n = 5, 64, 8
    x = synth.hidden(T, d, 3, DEV)
    wr = synth.router(d, n, 3, DEV)
    bias = torch.linspace(-1, 1, n, device=DEV)
    _, gi, gw = route_on_gpu(B, x, wr, bias, n)
    oi, op, info = O.route(x, wr, n, bias=bias)
    H.compare_routing(gi, gw, oi, op, info, x, wr)


# ---------------------------------------------------------------------------
# Group-limited top-k ([DeaMoE] §3.3 k_dept; strict coverage of its Table 4)
# ---------------------------------------------------------------------------


def grouped_on_gpu(B, x, wr, bias, k, g, k_dept, strict, scale=1.0):
    T = x.shape[0]
    n = wr.shape[0]
    ws = B.new_workspace(T, n, k, 1)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    B.moe_route_topk_grouped(x, wr, bias, k, g, k_dept, strict, scale, idx, w, ws)
    torch.cuda.synchronize()
    st, _, _ = B.moe_read_status(ws)
    assert st == 0
    return idx.cpu().numpy(), w.cpu().numpy()


# (d, n, g, k, k_dept): the DeaMoE-7B router with 2, 4 and all 8 departments,
# the 256-expert router in 16 departments, one expert per department, and the
# widest router (1024 experts) in 8 departments of 128
GROUPED_CASES = [(2048, 64, 8, 8, 2), (2048, 64, 8, 8, 4), (2048, 64, 8, 8, 8), (7168, 256, 16, 8, 4),
                 (512, 32, 1, 6, 6), (256, 1024, 128, 32, 3), (256, 48, 3, 5, 4)]


@pytest.mark.parametrize("case", GROUPED_CASES, ids=lambda c: "d%d-n%d-g%d-k%d-kd%d" % c)
@pytest.mark.parametrize("strict", [False, True], ids=["soft", "strict"])
def test_route_grouped_matches_oracle(B, case, strict):
    d, n, g, k, k_dept = case
    ties = 0
    for T in (1, 5, 33, 128):
        for seed in (0, 1):
            wr = synth.router(d, n, seed, DEV)
            bias = synth.zipf_bias(n, g, 1.1, seed).to(DEV) if seed else None
            x = synth.hidden(T, d, seed + 100 * T, DEV)
            gi, gw = grouped_on_gpu(B, x, wr, bias, k, g, k_dept, strict, scale=1.25)
            oi, op, info = O.route_grouped(x, wr, k, g, k_dept, bias=bias, scale=1.25, strict=strict)
            ties += len(H.compare_grouped_routing(gi, gw, oi, op, info, x, wr, g, k_dept, strict))
    assert ties <= 1


@pytest.mark.parametrize("strict", [False, True], ids=["soft", "strict"])
def test_route_grouped_exact_ties(B, strict):
    # equal logits; a bias that is constant within departments and repeats
    # across them: every decision is a tie broken by index
    T, d, n, g = 4, 16, 64, 8
    x = torch.ones((T, d), device=DEV)
    wr = torch.zeros((n, d), device=DEV)
    for bias in (None, torch.tensor([float((e // g) % 3) for e in range(n)], device=DEV)):
        for k, k_dept in ((8, 2), (5, 5), (16, 3)):
            gi, gw = grouped_on_gpu(B, x, wr, bias, k, g, k_dept, strict)
            oi, op, _ = O.route_grouped(x, wr, k, g, k_dept, bias=bias, strict=strict)
            np.testing.assert_array_equal(gi, oi)
            np.testing.assert_allclose(gw, op, rtol=1e-6)


@pytest.mark.parametrize("strict", [False, True], ids=["soft", "strict"])
def test_route_grouped_wide_router_ties_and_bits(B, strict):
    """More than 512 experts (20-21 keys per lane of the selecting warp), one or
    two tokens: every tie is broken by index as in the oracle, and a token's
    indices and weights do not depend on the other tokens of its step."""
    d, n, g = 16, 640, 80
    for T in (1, 2):
        x = torch.ones((T, d), device=DEV)
        wr = torch.zeros((n, d), device=DEV)
        for bias in (None, torch.tensor([float((e // g) % 3) for e in range(n)], device=DEV)):
            for k, k_dept in ((8, 2), (5, 5), (20, 3)):
                gi, gw = grouped_on_gpu(B, x, wr, bias, k, g, k_dept, strict)
                oi, op, _ = O.route_grouped(x, wr, k, g, k_dept, bias=bias, strict=strict)
                np.testing.assert_array_equal(gi, oi)
                np.testing.assert_allclose(gw, op, rtol=1e-6)
    d, n, g, k, k_dept = 1024, 672, 84, 10, 4
    wr = synth.router(d, n, 5, DEV)
    bias = synth.zipf_bias(n, g, 1.1, 5).to(DEV)
    x3 = synth.hidden(3, d, 5, DEV)
    i1, w1 = grouped_on_gpu(B, x3[:1].contiguous(), wr, bias, k, g, k_dept, strict)
    i3, w3 = grouped_on_gpu(B, x3, wr, bias, k, g, k_dept, strict)
    np.testing.assert_array_equal(i1[0], i3[0])
    assert np.array_equal(w1[0].view(np.uint32), w3[0].view(np.uint32))


def test_route_grouped_hand_example(B):
    # the oracle pin's example: logits [5, 1 | 4.9, 0 | 4.8, 4.7 | 0, 0] and
    # [5, 4.9 | 4.8, 4.7 | 1, 0 | 0.5, 0.2] (x = e_0, d padded to 8)
    x = torch.zeros((2, 8), device=DEV)
    x[:, 0] = 1.0
    wr = torch.zeros((8, 8), device=DEV)
    wr[:, 0] = torch.tensor([5.0, 1.0, 4.9, 0.0, 4.8, 4.7, 0.0, 0.0])
    assert grouped_on_gpu(B, x, wr, None, 3, 2, 2, False)[0][0].tolist() == [0, 2, 1]
    wr[:, 0] = torch.tensor([5.0, 4.9, 4.8, 4.7, 1.0, 0.0, 0.5, 0.2])
    assert grouped_on_gpu(B, x, wr, None, 3, 2, 3, False)[0][0].tolist() == [0, 1, 2]
    gi, gw = grouped_on_gpu(B, x, wr, None, 3, 2, 3, True)
    assert gi[0].tolist() == [0, 2, 4]
    ex = np.exp(np.array([5.0, 4.8, 1.0]))
    np.testing.assert_allclose(gw[0], ex / ex.sum(), rtol=1e-6)


def test_route_grouped_rejects_bad_arguments(B):
    x = torch.zeros((2, 8), device=DEV)
    wr = torch.zeros((8, 8), device=DEV)
    ws = B.new_workspace(2, 8, 4, 1)
    idx = torch.empty((2, 4), dtype=torch.int32, device=DEV)
    w = torch.empty((2, 4), dtype=torch.float32, device=DEV)
    for g, k_dept, strict in ((3, 1, False), (2, 0, False), (2, 5, False), (2, 1, False), (1, 3, True)):
        with pytest.raises(RuntimeError):
            B.moe_route_topk_grouped(x, wr, None, 4, g, k_dept, strict, 1.0, idx, w, ws)


# ---------------------------------------------------------------------------
# Router-bias update and imbalance ratio (DeepSeekMoE guide, auxiliary-loss-
# free section): fp64 arithmetic on both sides, so the fp32 results agree
# bit for bit
# ---------------------------------------------------------------------------


def bias_update_on_gpu(B, counts, bias, gamma, rule):
    c = torch.tensor(np.asarray(counts, np.int32), device=DEV)
    b = torch.tensor(np.asarray(bias, np.float32), device=DEV)
    r = torch.full((1,), -1.0, device=DEV)
    B.moe_bias_update(c, gamma, rule, b, r)
    torch.cuda.synchronize()
    return b.cpu().numpy(), float(r.item())


@pytest.mark.parametrize("n", [1, 7, 64, 256, 1000, 1024])
@pytest.mark.parametrize("rule", [0, 1], ids=["sign", "proportional"])
def test_bias_update_matches_oracle(B, n, rule):
    rng = np.random.default_rng(n + 17 * rule)
    for trial in range(4):
        if trial == 0:
            counts = np.zeros(n, np.int32)                       # nothing routed
        elif trial == 1:
            counts = np.full(n, 3, np.int32)                     # on target everywhere
        else:
            counts = rng.zipf(1.3, n).clip(max=5000).astype(np.int32)
        bias = (rng.standard_normal(n) * 0.05).astype(np.float32)
        gamma = float(np.float32(rng.uniform(1e-4, 1e-2)))
        gb, gr = bias_update_on_gpu(B, counts, bias, gamma, rule)
        np.testing.assert_array_equal(gb, O.bias_update(counts, bias, gamma, rule=rule))
        assert gr == float(np.float32(O.imbalance_ratio(counts)))


def test_bias_update_hand_example(B):
    gb, gr = bias_update_on_gpu(B, [3, 1, 2, 2], [0.5, -0.25, 0.0, 1.0], 0.125, 0)
    np.testing.assert_array_equal(gb, np.array([0.375, -0.125, 0.0, 1.0], np.float32))
    assert gr == 1.5


def test_bias_update_after_layer_forward(B):
    # the layer leaves its expert loads in the workspace; the update reads them
    # there (no host round trip) and matches the oracle's routing of the step
    shape = synth.DEAMOE_7B
    L = synth.make_layer(shape, 4, DEV)
    L["bias"] = (torch.randn(shape.n, generator=torch.Generator().manual_seed(4)) * 0.01).to(DEV)
    for T in (1, 16, 64):
        x = synth.hidden(T, shape.d, 40 + T, DEV)
        ws, gi, gw, _ = H.run_layer_forward(B, shape, L, x)
        counts = B.workspace_counts(ws, T, shape.n, shape.k, shape.g)
        b = L["bias"].clone()
        r = torch.empty(1, device=DEV)
        B.moe_bias_update(counts, 1e-3, 0, b, r)
        torch.cuda.synchronize()
        oi, op, info = O.route(x, L["router"], shape.k, bias=L["bias"])
        assert not H.compare_routing(gi.cpu().numpy(), gw.cpu().numpy(), oi, op, info, x, L["router"])
        oc = np.bincount(oi.reshape(-1), minlength=shape.n)
        np.testing.assert_array_equal(counts.cpu().numpy(), oc)
        np.testing.assert_array_equal(b.cpu().numpy(),
                                      O.bias_update(oc, L["bias"].cpu().numpy(), float(np.float32(1e-3))))
        assert r.item() == float(np.float32(O.imbalance_ratio(oc)))


def test_bias_update_rejects_bad_arguments(B):
    c = torch.zeros(8, dtype=torch.int32, device=DEV)
    b = torch.zeros(8, device=DEV)
    for gamma, rule, bias, imb in ((0.1, 2, b, None), (-1.0, 0, b, None), (float("inf"), 0, b, None),
                                   (float("nan"), 1, b, None), (0.1, 0, None, None)):
        with pytest.raises(RuntimeError):
            B.moe_bias_update(c, gamma, rule, bias, imb)
    with pytest.raises(RuntimeError):
        B.moe_bias_update(torch.zeros(1025, dtype=torch.int32, device=DEV), 0.1, 0, None,
                          torch.zeros(1, device=DEV))


# ---------------------------------------------------------------------------
# Dispatch (fed the oracle's routing: bit-exact lists)
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("T,n,k,g", [(1, 128, 8, 1), (4, 16, 2, 4), (16, 64, 8, 8), (33, 64, 8, 8),
                                     (64, 256, 8, 16), (128, 64, 8, 8), (128, 1024, 32, 2),
                                     (7, 16, 16, 4), (128, 8, 8, 1)])
def test_dispatch_bit_exact(B, T, n, k, g):
    rng = np.random.default_rng(T * 1000 + n + k + g)
    idx = np.stack([rng.permutation(n)[:k] for _ in range(T)]).astype(np.int32)
    p = rng.random((T, k)).astype(np.float32)
    ref = O.dispatch(idx, p.astype(np.float64), n, g)
    ws = B.new_workspace(T, n, k, g)
    B.moe_dispatch(torch.tensor(idx, device=DEV), torch.tensor(p, device=DEV), n, g, ws)
    dev = H.dispatch_lists(B, ws, T, n, k, g)
    assert dev["status"] == 0
    H.assert_dispatch_equal(dev, ref, g)


def test_dispatch_flags_bad_routing_without_faulting(B):
    T, n, k = 4, 16, 2
    ws = B.new_workspace(T, n, k, 1)
    idx = torch.tensor([[0, 1], [2, 99], [3, 4], [5, 6]], dtype=torch.int32, device=DEV)
    w = torch.ones((T, k), device=DEV)
    B.moe_dispatch(idx, w, n, 1, ws)
    st, A_e, _ = B.moe_read_status(ws)
    assert st == -6 and A_e == 0
    # a repeated expert is flagged too
    ws = B.new_workspace(T, n, k, 1)
    idx = torch.tensor([[0, 0], [1, 2], [3, 4], [5, 6]], dtype=torch.int32, device=DEV)
    B.moe_dispatch(idx, w, n, 1, ws)
    assert B.moe_read_status(ws)[0] == -6


# ---------------------------------------------------------------------------
# FFN + combine, against the oracle's per-token evaluation
# ---------------------------------------------------------------------------


def check_layer(B, shape, T, seed, sample=None, modes=("layer", "rows", "accum")):
    L = synth.make_layer(shape, seed, DEV)
    x = synth.hidden(T, shape.d, seed + 7 * T, DEV)
    tol = H.TOL[shape.dtype]
    g = shape.g if shape.I_sh > 0 else 1
    results = {}
    # whole-layer path first: its routing is the one compared with the oracle
    ws, gi, gw, y = H.run_layer_forward(B, shape, L, x)
    torch.cuda.synchronize()
    st, A_e, A_d = B.moe_read_status(ws)
    assert st == 0
    oi, op, info = O.route(x, L["router"], shape.k, bias=L["bias"])
    ties = H.compare_routing(gi.cpu().numpy(), gw.cpu().numpy(), oi, op, info, x, L["router"])
    tokens = [t for t in (range(T) if sample is None else sample) if t not in ties]
    y_ref = H.oracle_layer(shape, L, x, oi, op, tokens)
    if "layer" in modes:
        results["layer"] = H.rel_err(y.cpu().numpy()[tokens], y_ref)
    # dispatch lists of the fused path vs the oracle's lists of the oracle's
    # routing; after a certified near-tie (where the device's choice is the
    # other correct one) vs the oracle's lists of the device's own routing
    dev = H.dispatch_lists(B, ws, T, shape.n, shape.k, g)
    if not ties:
        ref = O.dispatch(oi, op, shape.n, g)
        H.assert_dispatch_equal(dev, ref, g, w_rtol=1e-5)
    else:
        ref = O.dispatch(gi.cpu().numpy(), gw.cpu().numpy().astype(np.float64), shape.n, g)
        H.assert_dispatch_equal(dev, ref, g, w_rtol=1e-7)
    assert A_e == len(ref["active_experts"])
    if g > 1:
        assert A_d == len(ref["active_depts"])
    # step-by-step path: FFN in ROWS mode + combine, and FFN in ACCUM mode
    sh = H.shared_of(L)
    for mode in [m for m in modes if m != "layer"]:
        if mode == "rows":
            rows = torch.empty((B.moe_rows_count(T, shape.n, shape.k, g, sh is not None), shape.d),
                               device=DEV)
            out = rows
            code = B.MOE_OUT_ROWS
        else:
            out = torch.zeros((T, shape.d), device=DEV)
            code = B.MOE_OUT_ACCUM
        if shape.I_sh > 0:
            priv = (L["pgate"], L["pup"], L["pdown"]) if shape.I_pr > 0 else None
            B.deamoe_ffn(x, shape.k, shape.g, (L["dgate"], L["dup"], L["ddown"]), priv, sh, ws,
                         code, out)
        else:
            B.moe_ffn_vanilla(x, shape.k, L["gate"], L["up"], L["down"], sh, ws, code, out)
        if mode == "rows":
            y2 = torch.empty((T, shape.d), device=DEV)
            B.moe_combine(rows, T, shape.n, shape.k, g, sh is not None, ws, y2)
        else:
            y2 = out
        torch.cuda.synchronize()
        results[mode] = H.rel_err(y2.cpu().numpy()[tokens], y_ref)
    for mode, err in results.items():
        assert err <= tol, f"{shape.name} T={T} {mode}: rel err {err:.3g} > {tol}"
        assert err <= H.KERNEL_TOL, f"{shape.name} T={T} {mode}: rel err {err:.3g} > {H.KERNEL_TOL}"
    return results


@pytest.mark.parametrize("shape", [synth.TINY_VANILLA, synth.TINY_DEAMOE], ids=lambda s: s.name)
def test_tiny_fp32_layers(B, shape):
    for T in (1, 4, 16):
        check_layer(B, shape, T, seed=0)


@pytest.mark.parametrize("T", [1, 4, 16])
def test_vanilla_128_experts(B, T):
    check_layer(B, synth.VANILLA_128E, T, seed=0)


@pytest.mark.parametrize("T", [1, 4, 8, 16])
def test_deamoe_7b_and_vanilla_twin(B, T):
    check_layer(B, synth.DEAMOE_7B, T, seed=1)
    check_layer(B, synth.VANILLA_7B, T, seed=1, modes=("layer",))


@pytest.mark.parametrize("T", [1, 8, 64])
def test_dsv3_shaped_layers_sampled(B, T):
    sample = [0] if T == 1 else [0, T - 1]
    check_layer(B, synth.DSV3_DEAMOE, T, seed=0, sample=sample, modes=("layer", "accum"))
    check_layer(B, synth.DSV3_VANILLA, T, seed=0, sample=sample, modes=("layer",))


@pytest.mark.parametrize("T", [1, 2, 32, 128])
def test_zipf_skew_layers(B, T):
    sample = None if T <= 32 else list(range(0, T, 16))
    check_layer(B, synth.ZIPF_DEAMOE, T, seed=2, sample=sample)
    check_layer(B, synth.ZIPF_VANILLA, T, seed=2, sample=sample, modes=("layer",))


def test_edge_shapes(B):
    # ragged intermediate (not a multiple of the stage rows), k = 1, tiny hidden
    s1 = synth.LayerShape("ragged", d=64, n=8, k=1, dtype="bf16", I=48, batches=(3,))
    check_layer(B, s1, 3, seed=5)
    # k = n: every token uses every expert (units with many tokens, several groups)
    s2 = synth.LayerShape("k-eq-n", d=128, n=4, k=4, dtype="f32", I=32, I_s=16, batches=(9,))
    check_layer(B, s2, 9, seed=6)
    # DeaMoE without private rows, and with a shared expert
    s3 = synth.LayerShape("dea-no-priv", d=256, n=16, k=4, dtype="f32", g=4, I_sh=64, I_pr=0,
                          I_s=32, batches=(5,))
    check_layer(B, s3, 5, seed=7)
    # max batch on a small layer
    s4 = synth.LayerShape("t128", d=128, n=32, k=8, dtype="bf16", g=8, I_sh=64, I_pr=16,
                          batches=(128,))
    check_layer(B, s4, 128, seed=8)


# One token on the whole-layer path: its top-k ranks the candidates in one
# pass instead of k warp rounds; the order and the bits must not change.
ONE_TOKEN_SHAPES = [
    synth.LayerShape("one-vanilla", d=256, n=64, k=6, dtype="bf16", I=64, batches=(1,)),
    synth.LayerShape("one-deamoe", d=256, n=64, k=6, dtype="bf16", g=8, I_sh=64, I_pr=32,
                     batches=(1,)),
]


def dyadic_router(d, n):
    """Router whose logit for the all-ones token is exactly level(e) / 8 in
    fp32 and fp64 alike (dyadic entries, power-of-two d): 16 levels of 4
    experts each (37 is prime to 64), so the keys hold exact ties."""
    c = torch.tensor([((e * 37) % n) // 4 / 8.0 for e in range(n)], dtype=torch.float32)
    return (c[:, None] / d).expand(n, d).contiguous().to(DEV)


@pytest.mark.parametrize("shape", ONE_TOKEN_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("with_bias", [False, True], ids=["no-bias", "bias"])
def test_one_token_layer_exact_ties(B, shape, with_bias):
    L = synth.make_layer(shape, 11, DEV)
    L["router"] = dyadic_router(shape.d, shape.n)
    L["bias"] = (torch.tensor([((e * 13) % 5 - 2) / 4 for e in range(shape.n)], device=DEV)
                 if with_bias else None)
    x = torch.ones((1, shape.d), device=DEV)
    ws, gi, gw, y = H.run_layer_forward(B, shape, L, x)
    torch.cuda.synchronize()
    assert B.moe_read_status(ws)[0] == 0
    oi, op, info = O.route(x, L["router"], shape.k, bias=L["bias"])
    gi, gw = gi.cpu().numpy(), gw.cpu().numpy()
    # the oracle orders equal keys by expert index; so must the device
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_allclose(gw, op, rtol=1e-6)
    # the last selected key is shared with experts left out: a tie was cut
    key = info["key32"][0]
    last = key[oi[0, -1]]
    assert np.count_nonzero(key == last) > np.count_nonzero(key[oi[0]] == last)
    y_ref = H.oracle_layer(shape, L, x, oi, op)
    assert H.rel_err(y.cpu().numpy(), y_ref) <= H.TOL[shape.dtype]
    # the routing kernel's warp top-k (the multi-token selection) gives the same bits
    _, ri, rw = route_on_gpu(B, x, L["router"], L["bias"], shape.k)
    np.testing.assert_array_equal(gi, ri)
    assert np.array_equal(gw.view(np.uint32), rw.view(np.uint32))


@pytest.mark.parametrize("T", [1, 3])
def test_layer_flags_masked_experts_in_the_selection(B, T):
    """Experts masked by a -inf selection bias rank after every finite key,
    lowest index first; selecting one sets the routing status (no fault)."""
    shape = ONE_TOKEN_SHAPES[0]
    L = synth.make_layer(shape, 12, DEV)
    bias = torch.full((shape.n,), float("-inf"), device=DEV)
    bias[[5, 17, 40, 63]] = 0.0
    L["bias"] = bias
    x = synth.hidden(T, shape.d, 12, DEV)
    ws, gi, gw, y = H.run_layer_forward(B, shape, L, x)
    torch.cuda.synchronize()
    assert B.moe_read_status(ws)[0] == -6
    gi = gi.cpu().numpy()
    for t in range(T):
        assert sorted(gi[t, :4].tolist()) == [5, 17, 40, 63]
        assert gi[t, 4:].tolist() == [0, 1]
    _, ri, _ = route_on_gpu(B, x, L["router"], L["bias"], shape.k)
    np.testing.assert_array_equal(gi, ri)


def test_invariant_one_expert_per_dept_no_private_is_vanilla(B):
    """DeaMoE with one expert per department and no private rows is the
    vanilla layer: the two device paths agree."""
    T, d, n, k, I = 6, 256, 16, 2, 64
    van = synth.LayerShape("v", d=d, n=n, k=k, dtype="bf16", I=I)
    dea = synth.LayerShape("d", d=d, n=n, k=k, dtype="bf16", g=1, I_sh=I, I_pr=0)
    L = synth.make_layer(van, 9, DEV)
    Ld = {"shape": dea, "router": L["router"], "bias": None, "dgate": L["gate"], "dup": L["up"],
          "ddown": L["down"], "sgate": None, "sup": None, "sdown": None}
    x = synth.hidden(T, d, 9, DEV)
    _, gi_v, _, y_v = H.run_layer_forward(B, van, L, x)
    _, gi_d, _, y_d = H.run_layer_forward(B, dea, Ld, x)
    torch.cuda.synchronize()
    assert torch.equal(gi_v, gi_d)
    assert H.rel_err(y_d.cpu().numpy(), y_v.cpu().numpy()) < 1e-6


def test_invariant_zero_private_is_department_ffn(B):
    """Zero private weights: y_t = sum_j omega_{t,j} FFN_j(x_t)."""
    T = 6
    dea = synth.LayerShape("d", d=256, n=16, k=3, dtype="f32", g=4, I_sh=64, I_pr=16)
    Ld = synth.make_layer(dea, 10, DEV)
    for key in ("pgate", "pup", "pdown"):
        Ld[key].zero_()
    x = synth.hidden(T, dea.d, 10, DEV)
    _, gi, gw, y = H.run_layer_forward(B, dea, Ld, x)
    torch.cuda.synchronize()
    oi, op, info = O.route(x, Ld["router"], dea.k)
    assert not H.compare_routing(gi.cpu().numpy(), gw.cpu().numpy(), oi, op, info, x, Ld["router"])
    D = O.dispatch(oi, op, dea.n, dea.g)
    ref = np.zeros((T, dea.d))
    for j in range(dea.m):
        for pos in range(D["dept_off"][j], D["dept_off"][j + 1]):
            t = D["dept_tok"][pos]
            ref[t] += D["dept_w"][pos] * O.swiglu_expert(x[t], Ld["dgate"][j], Ld["dup"][j], Ld["ddown"][j])
    assert H.rel_err(y.cpu().numpy(), ref) <= H.TOL["f32"]


def test_one_workspace_for_routing_calls_and_smaller_steps(B):
    """A DeaMoE workspace sized for 128 tokens: after a full layer step, the
    routing calls (plain and group-limited) on it run their top-k (their
    counters are the layer's, kept at zero) and leave the department lists
    alone; then layer steps with fewer tokens on the same buffer match the
    oracle."""
    shape = synth.ZIPF_DEAMOE
    L = synth.make_layer(shape, 12, DEV)
    Tm = 128
    ws = B.new_workspace(Tm, shape.n, shape.k, shape.g)
    lay = B.moe_workspace_layout(Tm, shape.n, shape.k, shape.g)
    x = synth.hidden(Tm, shape.d, 12, DEV)
    idx = torch.empty((Tm, shape.k), dtype=torch.int32, device=DEV)
    w = torch.empty((Tm, shape.k), device=DEV)
    y = torch.empty((Tm, shape.d), device=DEV)
    priv = (L["pgate"], L["pup"], L["pdown"])
    dept = (L["dgate"], L["dup"], L["ddown"])
    B.deamoe_layer_forward(x, shape.k, 1.0, L["router"], L["bias"], shape.g, dept, priv, None, ws, idx, w, y)
    torch.cuda.synchronize()
    lo, hi = lay["dept_count"], lay["total"]
    dept_bytes = ws[lo:hi].clone()
    for T in (Tm, 16, 1):
        xt = x[:T].contiguous()
        for grouped in (False, True):
            gi = torch.empty((T, shape.k), dtype=torch.int32, device=DEV)
            gw = torch.empty((T, shape.k), device=DEV)
            if grouped:
                B.moe_route_topk_grouped(xt, L["router"], L["bias"], shape.k, shape.g, 4, False, 1.0, gi, gw, ws)
                oi, op, info = O.route_grouped(xt, L["router"], shape.k, shape.g, 4, bias=L["bias"])
                torch.cuda.synchronize()
                assert len(H.compare_grouped_routing(gi.cpu().numpy(), gw.cpu().numpy(), oi, op, info, xt,
                                                     L["router"], shape.g, 4, False)) <= 1
            else:
                B.moe_route_topk(xt, L["router"], L["bias"], shape.k, 1.0, gi, gw, ws)
                oi, op, info = O.route(xt, L["router"], shape.k, bias=L["bias"])
                torch.cuda.synchronize()
                assert len(H.compare_routing(gi.cpu().numpy(), gw.cpu().numpy(), oi, op, info, xt,
                                             L["router"])) <= 1
    assert torch.equal(ws[lo:hi], dept_bytes)
    assert B.moe_read_status(ws)[0] == 0
    # smaller layer steps on the same buffer
    for T in (16, 3):
        xt = x[:T].contiguous()
        it = torch.empty((T, shape.k), dtype=torch.int32, device=DEV)
        wt = torch.empty((T, shape.k), device=DEV)
        yt = torch.empty((T, shape.d), device=DEV)
        B.deamoe_layer_forward(xt, shape.k, 1.0, L["router"], L["bias"], shape.g, dept, priv, None, ws, it, wt, yt)
        torch.cuda.synchronize()
        oi, op, info = O.route(xt, L["router"], shape.k, bias=L["bias"])
        assert not H.compare_routing(it.cpu().numpy(), wt.cpu().numpy(), oi, op, info, xt, L["router"])
        ref = H.oracle_layer(shape, L, xt, oi, op)
        assert H.rel_err(yt.cpu().numpy(), ref) <= H.TOL[shape.dtype]


def test_layer_with_host_activations_through_the_abi(B):
    """moe_input_from_host -> layer -> moe_output_to_host: both copies are
    exact, and the layer matches the same layer on device buffers (to the
    rounding of its fp32 atomics), for each batch size of the default workload."""
    shape = synth.VANILLA_128E
    L = synth.make_layer(shape, 3, DEV)
    for T in (1, 4, 16):
        x = synth.hidden(T, shape.d, 3 + T, DEV)
        _, _, _, y_dev = H.run_layer_forward(B, shape, L, x)
        x_host = x.cpu().pin_memory()
        y_host = torch.full((T, shape.d), float("nan")).pin_memory()
        x_in = torch.full_like(x, float("nan"))
        B.moe_input_from_host(x_in, x_host)
        _, _, _, y = H.run_layer_forward(B, shape, L, x_in)
        B.moe_output_to_host(y_host, y)
        torch.cuda.synchronize()
        assert torch.equal(x_in, x)
        assert torch.equal(y_host, y.cpu())
        assert H.rel_err(y_host.numpy(), y_dev.cpu().numpy()) <= 1e-6
    with pytest.raises(ValueError):
        B.moe_input_from_host(x_in, x_host[:, :8].contiguous())


def test_repeated_calls_reuse_workspace(B):
    shape = synth.VANILLA_128E
    L = synth.make_layer(shape, 3, DEV)
    ws = B.new_workspace(16, shape.n, shape.k, 1)
    outs = []
    for rep in range(3):
        x = synth.hidden(16, shape.d, 3, DEV)
        idx = torch.empty((16, shape.k), dtype=torch.int32, device=DEV)
        w = torch.empty((16, shape.k), device=DEV)
        y = torch.empty((16, shape.d), device=DEV)
        B.moe_layer_forward(x, shape.k, 1.0, L["router"], None, L["gate"], L["up"], L["down"],
                            None, ws, idx, w, y)
        outs.append(y.cpu().numpy())
    assert B.moe_read_status(ws)[0] == 0
    for o in outs[1:]:
        assert H.rel_err(o, outs[0]) < 1e-6
