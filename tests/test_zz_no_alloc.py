"""moe_route_topk_noalloc: the router step on the library's fixed device
scratch (no workspace, no allocation), checked through the C ABI against
moe_route_topk with a workspace on the same inputs, for two calls in a row.
Collected last so that it also runs after every other test in one process."""

import pytest
import torch

from moe_decode_layer_fp32_gb300 import synth
from tests import helpers as H

MAX_LOGITS = 64 * 1024   # T * n the fixed scratch holds
MOE_ERR_INVALID_ARG = -1  # include/moe_decode.h
MOE_ERR_UNSUPPORTED = -2


@pytest.fixture(scope="module")
def B():
    return H.ensure_built()


@pytest.mark.parametrize("T,n,k", [(128, 1024, 8), (65, 1024, 4), (128, 513, 2)])
def test_rejects_steps_beyond_the_scratch(B, T, n, k):
    """Host-side check only: nothing is looked up or launched."""
    assert T * n > MAX_LOGITS
    rc = B.lib().moe_route_topk_noalloc(None, None, None, T, 256, n, k, 1.0, None, None, None, None)
    assert rc == MOE_ERR_UNSUPPORTED
    msg = B.lib().moe_last_error().decode()
    assert "fixed scratch" in msg and str(T * n) in msg


def test_rejects_invalid_sizes(B):
    rc = B.lib().moe_route_topk_noalloc(None, None, None, 0, 256, 16, 2, 1.0, None, None, None, None)
    assert rc == MOE_ERR_INVALID_ARG


CASES = [
    # (d, n, k, T, with_bias, scale)
    (2048, 128, 8, 16, False, 1.0),      # vanilla 128-expert decode step
    (7168, 256, 8, 64, True, 2.5),       # DeepSeek-V3-shaped router with selection bias
    (256, 1024, 8, 64, False, 1.0),      # T * n exactly at the scratch limit
    (512, 16, 2, 1, False, 1.0),         # single token
]


@pytest.mark.gpu
@pytest.mark.parametrize("d,n,k,T,with_bias,scale", CASES)
def test_noalloc_matches_workspace_entry_point(B, d, n, k, T, with_bias, scale):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = "cuda"
    seed = 11 + T
    x = synth.hidden(T, d, seed, dev)
    wr = synth.router(d, n, seed, dev)
    bias = synth.zipf_bias(n, 1, 1.1, seed).to(dev) if with_bias else None

    ws = B.new_workspace(T, n, k)
    idx_ref = torch.empty(T, k, dtype=torch.int32, device=dev)
    w_ref = torch.empty(T, k, dtype=torch.float32, device=dev)
    B.moe_route_topk(x, wr, bias, k, scale, idx_ref, w_ref, ws)
    torch.cuda.synchronize()
    st_ref, _, _ = B.moe_read_status(ws)
    assert st_ref == 0

    for call in range(2):
        idx = torch.full((T, k), -7, dtype=torch.int32, device=dev)
        w = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev)
        status = torch.full((1,), 12345, dtype=torch.int32, device=dev)
        B.moe_route_topk_noalloc(x, wr, bias, k, scale, idx, w, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        assert torch.equal(idx.cpu(), idx_ref.cpu()), f"call {call}: expert indices differ"
        # the same routing kernel on the same inputs: the weights agree bit for bit
        assert torch.equal(w.cpu(), w_ref.cpu()), f"call {call}: routing weights differ"
