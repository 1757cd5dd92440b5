"""Shared glue for the parity tests: build inputs, run the CUDA path through
the C ABI, run the oracle on the same inputs, compare."""

from __future__ import annotations

import numpy as np
import torch

from moe_decode_layer_fp32_gb300 import synth
from oracle import moe_oracle as O

# Output tolerances: max|y - y_ref| / max|y_ref| per output tensor.
TOL = {"bf16": 2e-2, "f32": 1e-4}
# The kernels' own accuracy, checked beside TOL: they compute in fp32 on the
# exactly decoded weights (the tensor-core kernel on bf16 hi + lo parts of the
# activations and of H, exact to about 2^-17), so every output lands within
# 1e-4 of the oracle whatever the weight storage.  A dropped intermediate row,
# token or department term moves the output by about 1e-2 and fails it.
KERNEL_TOL = 1e-4


def ensure_built():
    from moe_decode_layer_fp32_gb300 import build_native
    build_native.build()
    from moe_decode_layer_fp32_gb300 import binding
    return binding


def rel_err(y, y_ref) -> float:
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    den = np.abs(y_ref).max()
    return float(np.abs(y - y_ref).max() / (den if den > 0 else 1.0))


def near_tie_bound(x, w_router) -> np.ndarray:
    """Per-token scale of the fp32 summation error of a logit:
    2^-20 * max_e sum_c |x_c| |W_r[e, c]|."""
    ax = np.abs(O.to_f64(x))
    aw = np.abs(O.to_f64(w_router))
    return (ax @ aw.T).max(axis=1) * 2.0 ** -20


def compare_routing(g_idx, g_w, o_idx, o_p, info, x, w_router, w_rtol=1e-5):
    """Indices bit-exact, except tokens whose oracle key gap at a swapped
    position is within the fp32 summation error (certified near-ties, where
    either order is a correct fp32 decision).  Returns those token ids."""
    g_idx = np.asarray(g_idx)
    g_w = np.asarray(g_w, np.float64)
    eps = near_tie_bound(x, w_router)
    key = info["key64"]
    ties = []
    for t in range(g_idx.shape[0]):
        if np.array_equal(g_idx[t], o_idx[t]):
            np.testing.assert_allclose(g_w[t], o_p[t], rtol=w_rtol, atol=1e-7,
                                       err_msg=f"routing weights of token {t}")
            continue
        # every expert the device placed must be within eps of the oracle's key at that rank
        ok = all(abs(key[t, int(g_idx[t, r])] - key[t, int(o_idx[t, r])]) <= eps[t]
                 for r in range(g_idx.shape[1]))
        assert ok, (f"token {t}: device {g_idx[t].tolist()} vs oracle {o_idx[t].tolist()} "
                    f"with gaps above the fp32 bound {eps[t]:.3g}")
        ties.append(t)
    return ties


def compare_grouped_routing(g_idx, g_w, o_idx, o_p, info, x, w_router, g, k_dept, strict,
                            w_rtol=1e-5):
    """Group-limited routing: indices bit-exact, except tokens where the
    oracle shows a near-tie (a department-score gap at the k_dept boundary or
    a key gap inside the kept departments within twice the fp32 summation
    error) and the device's selection is still a valid one: k distinct
    experts, at most (strict: exactly) k_dept departments, keys descending
    within the error.  Returns those token ids."""
    g_idx = np.asarray(g_idx)
    g_w = np.asarray(g_w, np.float64)
    eps = near_tie_bound(x, w_router)
    key, dscore = info["key64"], info["dscore64"]
    k = g_idx.shape[1]
    ties = []
    for t in range(g_idx.shape[0]):
        if np.array_equal(g_idx[t], o_idx[t]):
            np.testing.assert_allclose(g_w[t], o_p[t], rtol=w_rtol, atol=1e-7,
                                       err_msg=f"routing weights of token {t}")
            continue
        ds = np.sort(dscore[t])[::-1]
        near = k_dept < len(ds) and ds[k_dept - 1] - ds[k_dept] <= 2 * eps[t]
        pool = np.sort([key[t, e] for e in range(key.shape[1]) if e // g in set(info["kept"][t])])
        near = near or (np.diff(pool).min() if len(pool) > 1 else np.inf) <= 2 * eps[t]
        sel = [int(e) for e in g_idx[t]]
        deps = {e // g for e in sel}
        valid = (len(set(sel)) == k and (len(deps) == k_dept if strict else len(deps) <= k_dept)
                 and all(key[t, a] >= key[t, b] - 2 * eps[t] for a, b in zip(sel, sel[1:])))
        assert near and valid, (f"token {t}: device {sel} vs oracle {o_idx[t].tolist()} "
                                f"(near-tie {near}, valid {valid})")
        ties.append(t)
    return ties


def dispatch_lists(binding, ws, T, n, k, g):
    """Read every dispatch list out of a device workspace (host numpy)."""
    L = binding.moe_workspace_layout(T, n, k, g)
    raw = ws.cpu()

    def arr(name, count, dtype):
        off = L[name]
        return raw[off: off + 4 * count].view(dtype).numpy().copy()

    out = {
        "status": arr("status", 1, torch.int32)[0],
        "A_e": arr("counts", 2, torch.int32)[0],
        "A_d": arr("counts", 2, torch.int32)[1],
        "exp_count": arr("exp_count", n, torch.int32),
        "exp_off": arr("exp_off", n + 1, torch.int32),
        "asg_tok": arr("asg_tok", T * k, torch.int32),
        "asg_slot": arr("asg_slot", T * k, torch.int32),
        "asg_w": arr("asg_w", T * k, torch.float32),
        "tok_asg": arr("tok_asg", T * k, torch.int32).reshape(T, k),
    }
    out["active_experts"] = arr("act_exp", n, torch.int32)[: out["A_e"]]
    out["exp_units"] = arr("exp_units", 4 * n, torch.int32).reshape(n, 4)[: out["A_e"]]
    if g > 1:
        m = n // g
        D = int(arr("dept_off", m + 1, torch.int32)[m])
        out.update({
            "dept_count": arr("dept_count", m, torch.int32),
            "dept_off": arr("dept_off", m + 1, torch.int32),
            "dept_tok": arr("dept_tok", D, torch.int32),
            "dept_w": arr("dept_w", D, torch.float32),
            "tok_dpos": arr("tok_dpos", T * m, torch.int32).reshape(T, m),
        })
        out["active_depts"] = arr("act_dept", m, torch.int32)[: out["A_d"]]
        out["dept_units"] = arr("dept_units", 4 * m, torch.int32).reshape(m, 4)[: out["A_d"]]
    return out


def unit_records(active, off, count, group=4):
    """Expected FFN work records: {unit, first entry, entries, inclusive
    prefix of ceil(entries / group)} per active unit, ascending."""
    rec, run = [], 0
    for u in active:
        c = int(count[u])
        run += -(-c // group)
        rec.append([int(u), int(off[u]), c, run])
    return np.array(rec, np.int32).reshape(-1, 4)


def assert_dispatch_equal(dev, ref, g, w_rtol=1e-7):
    """Index lists bit-exact; weights within w_rtol (1e-7 when the device was
    fed the oracle's fp32 weights, looser when it computed them itself)."""
    for key in ("exp_count", "exp_off", "asg_tok", "asg_slot", "tok_asg", "active_experts"):
        np.testing.assert_array_equal(dev[key], ref[key], err_msg=key)
    np.testing.assert_allclose(dev["asg_w"], ref["asg_w"], rtol=w_rtol, err_msg="asg_w")
    np.testing.assert_array_equal(
        dev["exp_units"], unit_records(ref["active_experts"], ref["exp_off"], ref["exp_count"]),
        err_msg="exp_units")
    if g > 1:
        for key in ("dept_count", "dept_off", "dept_tok", "tok_dpos", "active_depts"):
            np.testing.assert_array_equal(dev[key], ref[key], err_msg=key)
        np.testing.assert_array_equal(
            dev["dept_units"],
            unit_records(ref["active_depts"], ref["dept_off"], ref["dept_count"]),
            err_msg="dept_units")
        np.testing.assert_allclose(dev["dept_w"], ref["dept_w"], rtol=max(w_rtol, 1e-6),
                                   err_msg="dept_w")


def layer_tensors(shape: synth.LayerShape, seed: int, device: str):
    return synth.make_layer(shape, seed, device)


def shared_of(L):
    return None if L["sgate"] is None else (L["sgate"], L["sup"], L["sdown"])


def oracle_layer(shape, L, x, idx, p, tokens=None):
    """Oracle output for `tokens` (all by default) given the routing."""
    tokens = list(range(x.shape[0])) if tokens is None else list(tokens)
    xs = x[tokens]
    idx_s, p_s = idx[tokens], p[tokens]
    sh = shared_of(L)
    if shape.I_sh > 0:
        priv = (L["pgate"], L["pup"], L["pdown"]) if shape.I_pr > 0 else (None, None, None)
        return O.deamoe_layer_c(xs, idx_s, p_s, shape.g, L["dgate"], L["dup"], L["ddown"],
                                *priv, shared=sh)
    return O.vanilla_layer(xs, idx_s, p_s, L["gate"], L["up"], L["down"], shared=sh)


def fp8_scales(shape, L):
    """Row scales of an FP8 layer in the order of the *_fp8 calls (None otherwise)."""
    if shape.dtype != "fp8":
        return None
    keys = ("dgate", "dup", "ddown", "pgate", "pup", "pdown") if shape.I_sh > 0 else ("gate", "up", "down")
    return [L.get(k + "_sc") for k in keys + ("sgate", "sup", "sdown")]


def run_layer_forward(binding, shape, L, x, scale=1.0):
    """Whole-layer path (fused route+dispatch, FFN as its dependent)."""
    T = x.shape[0]
    g = shape.g if shape.I_sh > 0 else 1
    ws = binding.new_workspace(T, shape.n, shape.k, g)
    idx = torch.empty((T, shape.k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, shape.k), dtype=torch.float32, device=x.device)
    y = torch.empty((T, shape.d), dtype=torch.float32, device=x.device)
    sc = fp8_scales(shape, L)
    if shape.I_sh > 0:
        priv = (L["pgate"], L["pup"], L["pdown"]) if shape.I_pr > 0 else None
        binding.deamoe_layer_forward(x, shape.k, scale, L["router"], L["bias"], shape.g,
                                     (L["dgate"], L["dup"], L["ddown"]), priv, shared_of(L),
                                     ws, idx, w, y, scales=sc)
    else:
        binding.moe_layer_forward(x, shape.k, scale, L["router"], L["bias"], L["gate"], L["up"],
                                  L["down"], shared_of(L), ws, idx, w, y, scales=sc)
    return ws, idx, w, y
