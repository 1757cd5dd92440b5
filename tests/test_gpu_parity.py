"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Routing indices and dispatch lists must match bit-exactly (certified fp32
near-ties excepted, see helpers.compare_routing); outputs must match within
the benchmark spec's tolerance: max|y - y_ref| / max|y_ref| <= 2e-2 for bf16
weights and 1e-4 for fp32 weights.
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
    # dispatch lists of the fused path vs the oracle's lists
    ref = O.dispatch(oi, op, shape.n, g)
    if not ties:
        dev = H.dispatch_lists(B, ws, T, shape.n, shape.k, g)
        H.assert_dispatch_equal(dev, ref, g, w_rtol=1e-5)
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
