"""FP8 (E4M3, one fp32 scale per row) expert weights on the GPU, through the
C ABI, against the oracle on the exactly decoded weights.

The device decodes each code exactly and applies the row scale in fp32, so
outputs stay within 1e-4 of the fp64 oracle (the 2e-2 output bound for
reduced-precision weights is checked as well); routing is unchanged (fp32
router) and compared as everywhere else.
"""

import numpy as np
import pytest
import torch

from moe_decode_layer_fp32_gb300 import synth
from oracle import moe_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu

DEV = "cuda"

TINY_VAN_FP8 = synth.LayerShape("tiny-vanilla-fp8-shared", d=256, n=16, k=2, dtype="fp8", I=64, I_s=32)
TINY_DEA_FP8 = synth.LayerShape("tiny-deamoe-fp8-shared", d=256, n=16, k=3, dtype="fp8", g=4, I_sh=64,
                                I_pr=16, I_s=32)
WEIGHT_KEYS = ("gate", "up", "down", "dgate", "dup", "ddown", "pgate", "pup", "pdown", "sgate", "sup", "sdown")


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return H.ensure_built()


@pytest.fixture
def threshold(B):
    prev = B.moe_set_tc_min_tokens(0)

    def set_(v):
        B.moe_set_tc_min_tokens(v)
    yield set_
    B.moe_set_tc_min_tokens(prev)


# Small enough for the oracle, with every weight block a multiple of 128 rows
# so that the tensor-core kernel takes each class, shared expert included.
TC_DEA_FP8 = synth.LayerShape("tc-deamoe-fp8-shared", d=256, n=16, k=4, dtype="fp8", g=4, I_sh=256, I_pr=128,
                              I_s=128)
TC_VAN_FP8 = synth.LayerShape("tc-vanilla-fp8-shared", d=384, n=16, k=4, dtype="fp8", I=128, I_s=128)


def scales_of(shape, L):
    sc = lambda key: L.get(key + "_sc")                                       # noqa: E731
    if shape.I_sh > 0:
        return [sc(k) for k in ("dgate", "dup", "ddown", "pgate", "pup", "pdown", "sgate", "sup", "sdown")]
    return [sc(k) for k in ("gate", "up", "down", "sgate", "sup", "sdown")]


def decoded(L):
    """The layer with every FP8 weight tensor decoded exactly (fp64, host)."""
    D = dict(L)
    for key in WEIGHT_KEYS:
        if L.get(key) is not None:
            D[key] = O.dequant_rows_e4m3(L[key], L[key + "_sc"])
    return D


def run_layer(B, shape, L, x):
    T = x.shape[0]
    g = shape.g if shape.I_sh > 0 else 1
    ws = B.new_workspace(T, shape.n, shape.k, g)
    idx = torch.empty((T, shape.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, shape.k), device=DEV)
    y = torch.full((T, shape.d), float("nan"), device=DEV)
    sh = H.shared_of(L)
    if shape.I_sh > 0:
        priv = (L["pgate"], L["pup"], L["pdown"]) if shape.I_pr > 0 else None
        B.deamoe_layer_forward(x, shape.k, 1.0, L["router"], L["bias"], shape.g, (L["dgate"], L["dup"], L["ddown"]),
                               priv, sh, ws, idx, w, y, scales=scales_of(shape, L))
    else:
        B.moe_layer_forward(x, shape.k, 1.0, L["router"], L["bias"], L["gate"], L["up"], L["down"], sh, ws, idx, w,
                            y, scales=scales_of(shape, L))
    torch.cuda.synchronize()
    return ws, idx.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()


def check_fp8_layer(B, shape, T, seed, sample=None, L=None):
    L = synth.make_layer(shape, seed, DEV) if L is None else L
    x = synth.hidden(T, shape.d, seed + 3 * T, DEV)
    ws, gi, gw, y = run_layer(B, shape, L, x)
    assert B.moe_read_status(ws)[0] == 0
    oi, op, info = O.route(x, L["router"], shape.k, bias=L["bias"])
    ties = H.compare_routing(gi, gw, oi, op, info, x, L["router"])
    tokens = [t for t in (range(T) if sample is None else sample) if t not in ties]
    ref = H.oracle_layer(shape, decoded(L), x, oi, op, tokens)
    err = H.rel_err(y[tokens], ref)
    assert err <= H.TOL["bf16"]
    assert err <= 1e-4, err
    return len(ties)


@pytest.mark.parametrize("T", [1, 4, 16, 64])
def test_vanilla_128e_fp8_layer(B, T):
    sample = None if T <= 16 else [0, 1, 32, 63]
    assert check_fp8_layer(B, synth.VANILLA_128E_FP8, T, seed=21, sample=sample) <= 1


@pytest.mark.parametrize("T", [1, 4, 8, 16, 33])
def test_deamoe_7b_fp8_layer(B, T):
    sample = None if T <= 16 else [0, 16, 32]
    assert check_fp8_layer(B, synth.DEAMOE_7B_FP8, T, seed=22, sample=sample) <= 1


@pytest.mark.parametrize("shape", [TINY_VAN_FP8, TINY_DEA_FP8], ids=lambda s: s.name)
@pytest.mark.parametrize("T", [3, 40])
def test_fp8_with_shared_expert(B, shape, T):
    assert check_fp8_layer(B, shape, T, seed=23) <= 1


@pytest.mark.parametrize("mode", ["rows", "accum"])
def test_fp8_ffn_step_on_the_oracle_dispatch(B, mode):
    """The FFN step alone on the oracle's routing: ROWS (+ combine) and ACCUM."""
    shape = TINY_DEA_FP8
    T = 7
    L = synth.make_layer(shape, 24, DEV)
    x = synth.hidden(T, shape.d, 24, DEV)
    oi, op, _ = O.route(x, L["router"], shape.k)
    ws = B.new_workspace(T, shape.n, shape.k, shape.g)
    B.moe_dispatch(torch.tensor(oi, device=DEV), torch.tensor(op, dtype=torch.float32, device=DEV), shape.n,
                   shape.g, ws)
    dept = (L["dgate"], L["dup"], L["ddown"])
    priv = (L["pgate"], L["pup"], L["pdown"])
    sh = H.shared_of(L)
    y = torch.zeros((T, shape.d), device=DEV)
    if mode == "rows":
        rows = torch.empty((B.moe_rows_count(T, shape.n, shape.k, shape.g, True), shape.d), device=DEV)
        B.deamoe_ffn(x, shape.k, shape.g, dept, priv, sh, ws, B.MOE_OUT_ROWS, rows, scales=scales_of(shape, L))
        B.moe_combine(rows, T, shape.n, shape.k, shape.g, True, ws, y)
    else:
        B.deamoe_ffn(x, shape.k, shape.g, dept, priv, sh, ws, B.MOE_OUT_ACCUM, y, scales=scales_of(shape, L))
    torch.cuda.synchronize()
    ref = H.oracle_layer(shape, decoded(L), x, oi, op)
    assert H.rel_err(y.cpu().numpy(), ref) <= 1e-4


@pytest.mark.parametrize("mode", ["tc", "cc"])
@pytest.mark.parametrize("shape,T", [(synth.DEAMOE_7B_FP8, 4), (synth.DEAMOE_7B_FP8, 16), (synth.DEAMOE_7B_FP8, 33),
                                     (synth.VANILLA_128E_FP8, 16)], ids=lambda v: getattr(v, "name", v))
def test_fp8_each_path(B, threshold, mode, shape, T):
    """The E4M3 tensor-core kernel (converter warps, row scales in the
    epilogue) forced on every unit, and the CUDA-core stream alone, on the
    7B-class FP8 layers: both within 1e-4 of the oracle on the decoded
    weights.  T = 33 gives departments three groups of 16 tokens, the last
    one ragged."""
    threshold(1 if mode == "tc" else 10 ** 6)
    sample = None if T <= 16 else [0, 16, 32]
    assert check_fp8_layer(B, shape, T, seed=27, sample=sample) <= 1


@pytest.mark.parametrize("shape", [TC_DEA_FP8, TC_VAN_FP8], ids=lambda s: s.name)
@pytest.mark.parametrize("T", [1, 5, 17, 33])
def test_fp8_tc_small_layers(B, threshold, shape, T):
    """Shared expert, departments and expert blocks on the tensor cores with
    one token, a partial group, and several groups with a ragged tail."""
    threshold(1)
    assert check_fp8_layer(B, shape, T, seed=28) <= 1


E4M3_SUBNORMAL = [0x00, 0x80] + list(range(0x01, 0x08)) + list(range(0x81, 0x88))
E4M3_ALL = [c for c in range(256) if c not in (0x7F, 0xFF)]          # every code but the two NaNs


@pytest.mark.parametrize("mode", ["tc", "cc"])
@pytest.mark.parametrize("pool", ["subnormal", "all"])
def test_fp8_every_code(B, threshold, mode, pool):
    """Weights drawn from a set of E4M3 codes, decoded by each path and
    compared with the oracle's exact decode: the zeros and subnormals alone
    (a path that flushed or mis-scaled them would be off by the whole output)
    and every finite code."""
    threshold(1 if mode == "tc" else 10 ** 6)
    shape = TC_VAN_FP8
    L = synth.make_layer(shape, 30, DEV)
    rng = np.random.default_rng(30 if pool == "all" else 31)
    codes = np.array(E4M3_SUBNORMAL if pool == "subnormal" else E4M3_ALL, np.uint8)
    for key in ("gate", "up", "down", "sgate", "sup", "sdown"):
        draw = rng.choice(codes, size=tuple(L[key].shape))
        L[key] = torch.tensor(draw, dtype=torch.uint8, device=DEV).view(torch.float8_e4m3fn)
        if pool == "subnormal":
            L[key + "_sc"] = L[key + "_sc"] * 256.0
    for T in (3, 17):
        assert check_fp8_layer(B, shape, T, seed=30, L=L) <= 1


@pytest.mark.parametrize("mode", ["rows", "accum"])
def test_fp8_tc_ffn_step_on_the_oracle_dispatch(B, threshold, mode):
    """The FFN step alone on the tensor cores with the oracle's routing:
    ROWS (each row unweighted, then the combine) and ACCUM."""
    threshold(1)
    shape = TC_DEA_FP8
    T = 21
    L = synth.make_layer(shape, 29, DEV)
    x = synth.hidden(T, shape.d, 29, DEV)
    oi, op, _ = O.route(x, L["router"], shape.k)
    ws = B.new_workspace(T, shape.n, shape.k, shape.g)
    B.moe_dispatch(torch.tensor(oi, device=DEV), torch.tensor(op, dtype=torch.float32, device=DEV), shape.n,
                   shape.g, ws)
    dept = (L["dgate"], L["dup"], L["ddown"])
    priv = (L["pgate"], L["pup"], L["pdown"])
    sh = H.shared_of(L)
    y = torch.zeros((T, shape.d), device=DEV)
    if mode == "rows":
        rows = torch.empty((B.moe_rows_count(T, shape.n, shape.k, shape.g, True), shape.d), device=DEV)
        B.deamoe_ffn(x, shape.k, shape.g, dept, priv, sh, ws, B.MOE_OUT_ROWS, rows, scales=scales_of(shape, L))
        B.moe_combine(rows, T, shape.n, shape.k, shape.g, True, ws, y)
    else:
        B.deamoe_ffn(x, shape.k, shape.g, dept, priv, sh, ws, B.MOE_OUT_ACCUM, y, scales=scales_of(shape, L))
    torch.cuda.synchronize()
    assert B.moe_read_status(ws)[0] == 0
    ref = H.oracle_layer(shape, decoded(L), x, oi, op)
    assert H.rel_err(y.cpu().numpy(), ref) <= 1e-4


def test_fp8_rejects_bad_arguments(B):
    shape = synth.VANILLA_128E_FP8
    L = synth.make_layer(shape, 25, DEV)
    T = 2
    x = synth.hidden(T, shape.d, 25, DEV)
    ws = B.new_workspace(T, shape.n, shape.k, 1)
    idx = torch.empty((T, shape.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, shape.k), device=DEV)
    y = torch.empty((T, shape.d), device=DEV)
    lib = B.lib()
    # the bf16 / fp32 call with the FP8 dtype code: no scales to read, refused
    rc = lib.moe_layer_forward(B._ptr(x), T, shape.d, shape.n, shape.k, 1.0, B._ptr(L["router"]), None, shape.I,
                               B.MOE_DTYPE_FP8_E4M3, B._ptr(L["gate"]), B._ptr(L["up"]), B._ptr(L["down"]), 0,
                               None, None, None, B._ptr(ws), ws.numel(), B._ptr(idx), B._ptr(w), B._ptr(y),
                               B._stream())
    assert rc == -1
    # a missing scale tensor
    sc = scales_of(shape, L)
    sc[1] = None
    with pytest.raises(RuntimeError):
        B.moe_layer_forward(x, shape.k, 1.0, L["router"], None, L["gate"], L["up"], L["down"], None, ws, idx, w, y,
                            scales=sc)
    with pytest.raises(ValueError):
        B.moe_layer_forward(x, shape.k, 1.0, L["router"], None, L["gate"], L["up"], L["down"], None, ws, idx, w, y)


def test_fp8_unique_bytes_count_codes_and_scales(B):
    d, n, I = 2048, 128, 768
    assert B.moe_unique_weight_bytes_vanilla(d, n, I, 0, B.MOE_DTYPE_FP8_E4M3, 8) == 4 * d * n + 8 * I * 3 * (d + 4)
    bf = B.moe_unique_weight_bytes_vanilla(d, n, I, 0, B.MOE_DTYPE_BF16, 8) - 4 * d * n
    fp = B.moe_unique_weight_bytes_vanilla(d, n, I, 0, B.MOE_DTYPE_FP8_E4M3, 8) - 4 * d * n
    assert abs(fp / bf - 0.5) < 0.002
    np.testing.assert_equal(fp, 8 * I * 3 * (d + 4))


@pytest.mark.parametrize("shape", [synth.VANILLA_128E_FP8, synth.DEAMOE_7B_FP8], ids=lambda s: s.name)
def test_fp8_model_change_stays_within_its_tolerance(B, shape):
    """FP8 storage is a change of the model, not a rounding of the
    computation: against the same draws stored in bf16 the layer output moves
    by up to a few percent of max|y| (E4M3 rounds each weight by up to 2^-4
    relative).  Its own tolerance here: 0.1 of max|y|."""
    import dataclasses
    T = 8
    L = synth.make_layer(shape, 26, DEV)
    Lb = synth.make_layer(dataclasses.replace(shape, dtype="bf16"), 26, DEV)
    x = synth.hidden(T, shape.d, 26, DEV)
    _, gi, gw, y = run_layer(B, shape, L, x)
    oi, op, info = O.route(x, L["router"], shape.k)
    ties = H.compare_routing(gi, gw, oi, op, info, x, L["router"])
    tokens = [t for t in range(T) if t not in ties]
    ref_bf16 = H.oracle_layer(shape, Lb, x, oi, op, tokens)
    err = H.rel_err(y[tokens], ref_bf16)
    assert err <= 0.1, err
