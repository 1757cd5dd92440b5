"""Failure detection of the FFN kernels' bounded waits, without a GPU fault.

With the library's test hook set, the weight producers issue no copy, so the
first wait of every consumer on a weight stage can never be satisfied and runs
out after a short limit (1 µs here instead of two seconds).  Each kernel must
then record MOE_ERR_TIMEOUT in the workspace status word and return with
nothing in flight; the context stays usable, and the same step run again with
the hook off matches the oracle.
"""

import numpy as np
import pytest
import torch

from moe_decode_layer_fp32_gb300 import synth
from oracle import moe_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu

DEV = "cuda"
MOE_ERR_TIMEOUT = -5      # include/moe_decode.h
STALL_NS = 1000


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return H.ensure_built()


def scales_of(shape, L):
    """FP8 row scales in the order of the *_fp8 calls (None for bf16 layers)."""
    if shape.dtype != "fp8":
        return None
    keys = ("dgate", "dup", "ddown", "pgate", "pup", "pdown") if shape.I_sh > 0 else ("gate", "up", "down")
    return [L[k + "_sc"] for k in keys] + [None, None, None]


def decoded(shape, L):
    """The layer with its FP8 weights decoded exactly (the oracle's weights)."""
    if shape.dtype != "fp8":
        return L
    D = dict(L)
    for key in ("gate", "up", "down", "dgate", "dup", "ddown", "pgate", "pup", "pdown"):
        if L.get(key) is not None:
            D[key] = O.dequant_rows_e4m3(L[key], L[key + "_sc"])
    return D


def layer_once(B, shape, L, x, ws):
    T = x.shape[0]
    idx = torch.empty((T, shape.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, shape.k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, shape.d), dtype=torch.float32, device=DEV)
    sc = scales_of(shape, L)
    if shape.I_sh > 0:
        B.deamoe_layer_forward(x, shape.k, 1.0, L["router"], L["bias"], shape.g,
                               (L["dgate"], L["dup"], L["ddown"]), (L["pgate"], L["pup"], L["pdown"]),
                               None, ws, idx, w, y, scales=sc)
    else:
        B.moe_layer_forward(x, shape.k, 1.0, L["router"], L["bias"], L["gate"], L["up"], L["down"], None,
                            ws, idx, w, y, scales=sc)
    torch.cuda.synchronize()
    return idx, w, y


# (layer, T, tensor-core threshold): the CUDA-core kernel alone with routing
# in its CTAs; the tensor-core kernel alone with routing in its CTAs; both
# kernels on the routing kernel's dispatch (units of >= 4 tokens on tcgen05);
# the same three with E4M3 weights (the tensor-core kernel's converter warps
# and its two landing barriers per code slot)
CASES = [(synth.VANILLA_128E, 4, 0, "ffn_stream_kernel"),
         (synth.DEAMOE_7B, 16, 0, "ffn_tc_kernel"),
         (synth.DEAMOE_7B, 16, 4, "both"),
         (synth.VANILLA_128E_FP8, 4, 0, "ffn_stream_kernel-fp8"),
         (synth.DEAMOE_7B_FP8, 16, 0, "ffn_tc_kernel-fp8"),
         (synth.DEAMOE_7B_FP8, 16, 4, "both-fp8")]


@pytest.mark.parametrize("shape,T,thr,kernels", CASES, ids=[c[3] for c in CASES])
def test_wait_runs_out_and_reports_timeout(B, shape, T, thr, kernels):
    L = synth.make_layer(shape, 21, DEV)
    x = synth.hidden(T, shape.d, 21 + T, DEV)
    g = shape.g if shape.I_sh > 0 else 1
    ws = B.new_workspace(T, shape.n, shape.k, g)
    prev_thr = B.moe_set_tc_min_tokens(thr)
    try:
        prev = B.moe_test_stall_weight_copies(STALL_NS)
        try:
            idx, w, _ = layer_once(B, shape, L, x, ws)
        finally:
            B.moe_test_stall_weight_copies(prev)
        assert prev == 0
        st, _, _ = B.moe_read_status(ws)
        assert st == MOE_ERR_TIMEOUT, f"{kernels}: device status {st}"
        # the routing of the stalled step still ran
        oi, op, info = O.route(x, L["router"], shape.k, bias=L["bias"])
        H.compare_routing(idx.cpu().numpy(), w.cpu().numpy(), oi, op, info, x, L["router"])
        # the context is usable: the same step on a cleared workspace is correct
        B.moe_workspace_init(ws)
        idx, w, y = layer_once(B, shape, L, x, ws)
        assert B.moe_read_status(ws)[0] == 0
        ties = H.compare_routing(idx.cpu().numpy(), w.cpu().numpy(), oi, op, info, x, L["router"])
        tokens = [t for t in range(T) if t not in ties]
        ref = H.oracle_layer(shape, decoded(shape, L), x, oi, op, tokens)
        assert H.rel_err(y.cpu().numpy()[tokens], ref) <= H.KERNEL_TOL
    finally:
        B.moe_set_tc_min_tokens(prev_thr)


def test_stall_hook_rejects_a_negative_limit(B):
    with pytest.raises(RuntimeError):
        B.moe_test_stall_weight_copies(-1)
    assert B.moe_test_stall_weight_copies(0) == 0
