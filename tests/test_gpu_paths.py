"""Both FFN paths against the oracle: the tcgen05 tensor-core kernel forced on
every unit (threshold 1 token) and the CUDA-core stream alone (threshold above
every batch), on the same layers.  The default split is covered by
test_gpu_parity.py."""

import numpy as np
import pytest
import torch

from moe_decode_layer_fp32_gb300 import synth
from tests import helpers as H
from tests.test_gpu_parity import check_layer

pytestmark = pytest.mark.gpu

DEV = "cuda"


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


SMALL_TC = synth.LayerShape("tc-small", d=256, n=16, k=4, dtype="bf16", g=4, I_sh=256, I_pr=128,
                            I_s=128, batches=(5,))


@pytest.mark.parametrize("mode", ["tc", "cc"])
def test_small_layer_each_path(B, threshold, mode):
    threshold(1 if mode == "tc" else 10 ** 6)
    for T in (1, 5, 33):
        check_layer(B, SMALL_TC, T, seed=3)
        van = synth.LayerShape("tc-small-v", d=384, n=16, k=4, dtype="bf16", I=128, I_s=128)
        check_layer(B, van, T, seed=4)


def test_tc_matches_cc_on_device(B, threshold):
    """Same layer, same routing: tensor-core and CUDA-core outputs agree
    closely (the hi/lo bf16 split keeps the activations near fp32)."""
    shape = synth.DEAMOE_7B
    L = synth.make_layer(shape, 5, DEV)
    x = synth.hidden(16, shape.d, 5, DEV)
    outs = {}
    for mode, v in (("tc", 1), ("cc", 10 ** 6)):
        threshold(v)
        _, _, _, y = H.run_layer_forward(B, shape, L, x)
        torch.cuda.synchronize()
        outs[mode] = y.cpu().numpy()
    assert H.rel_err(outs["tc"], outs["cc"]) < 1e-4


@pytest.mark.parametrize("mode", ["tc", "cc"])
@pytest.mark.parametrize("T", [1, 4, 16])
def test_vanilla_128e_each_path(B, threshold, mode, T):
    threshold(1 if mode == "tc" else 10 ** 6)
    check_layer(B, synth.VANILLA_128E, T, seed=0)


@pytest.mark.parametrize("mode", ["tc", "cc"])
@pytest.mark.parametrize("T", [8, 16])
def test_deamoe_7b_each_path(B, threshold, mode, T):
    threshold(1 if mode == "tc" else 10 ** 6)
    check_layer(B, synth.DEAMOE_7B, T, seed=1)


@pytest.mark.parametrize("T", [32, 64])
def test_dsv3_tc_sampled(B, threshold, T):
    threshold(0)
    check_layer(B, synth.DSV3_DEAMOE, T, seed=0, sample=[0, T // 2, T - 1],
                modes=("layer", "accum"))
    check_layer(B, synth.DSV3_VANILLA, T, seed=0, sample=[0, T - 1], modes=("layer",))


@pytest.mark.parametrize("T", [64, 128])
def test_zipf_large_batch_tc(B, threshold, T):
    threshold(0)
    check_layer(B, synth.ZIPF_DEAMOE, T, seed=2, sample=list(range(0, T, 9)))


def expected_auto_choice(shape, T, exp_count, dept_count, sms):
    """Host restatement of the whole-layer kernel choice: 0 the CUDA-core
    kernel alone (the step is not eligible for the tensor-core kernel, or not
    expected to gain from it), 1 CUDA cores and 2 tensor cores as chosen on the
    device (rows wider than 4096), 2 the tensor-core kernel alone."""
    classes = []
    if shape.I_sh > 0:
        classes.append((shape.I_sh, dept_count))
        if shape.I_pr > 0:
            classes.append((shape.I_pr, exp_count))
    else:
        classes.append((shape.I, exp_count))
    if shape.I_s > 0:
        classes.append((shape.I_s, [T]))
    if shape.dtype not in ("bf16", "fp8") or shape.d % 128 or any(r % 128 for r, _ in classes):
        return 0
    wide = shape.d > 4096
    if T <= 4 and not wide:
        return 0
    # launched only when some class expects more than one CUDA-core group
    # (4 tokens) per unit
    expect = []
    if shape.I_sh > 0:
        miss = 1.0
        for i in range(shape.k):
            miss *= max(shape.n - shape.g - i, 0) / (shape.n - i)
        expect.append(T * (1 - miss))
    if shape.I_sh == 0 or shape.I_pr > 0:
        expect.append(T * shape.k / shape.n)
    if shape.I_s > 0:
        expect.append(T)
    if max(expect) <= 4 and not wide:
        return 0
    if not wide and T <= 32:
        # launched for rows up to 4096 wide and up to 32 tokens: the
        # tensor-core kernel alone, with the routing inside its CTAs
        return 2
    rows_cc = sum(r * sum(-(-int(c) // 4) for c in cnt) for r, cnt in classes)
    tiles = sum(r // 128 * sum(-(-int(c) // 32) for c in cnt) for r, cnt in classes)
    tc_rows = -(-tiles // sms) * 128
    cc_weight = 4 if wide else 3
    return 2 if tiles > 0 and tc_rows * sms * 3 < rows_cc * cc_weight else 1


@pytest.mark.parametrize("shape,T", [(synth.VANILLA_128E, 16), (synth.VANILLA_128E, 4),
                                     (synth.DEAMOE_7B, 16), (synth.DEAMOE_7B, 8),
                                     (synth.DEAMOE_7B, 4), (synth.ZIPF_DEAMOE, 64),
                                     (synth.DSV3_DEAMOE, 32), (synth.DSV3_VANILLA, 1),
                                     (synth.DEAMOE_7B_FP8, 16), (synth.DEAMOE_7B_FP8, 4)])
def test_auto_choice_matches_cost_model(B, threshold, shape, T):
    """Default mode: the FFN kernels pick one path per call on the device;
    the choice they record equals the cost model evaluated on the host from
    the same dispatch counts, and the output stays at parity (checked by
    test_gpu_parity in the same mode)."""
    threshold(0)
    L = synth.make_layer(shape, 7, DEV)
    x = synth.hidden(T, shape.d, 7, DEV)
    ws, _, _, _ = H.run_layer_forward(B, shape, L, x)
    torch.cuda.synchronize()
    g = shape.g if shape.I_sh > 0 else 1
    lists = H.dispatch_lists(B, ws, T, shape.n, shape.k, g)
    lay = B.moe_workspace_layout(T, shape.n, shape.k, g)
    got = int(ws.cpu()[lay["sync"] + 4: lay["sync"] + 8].view(torch.int32)[0])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    want = expected_auto_choice(shape, T, lists["exp_count"], lists.get("dept_count", []), sms)
    assert got == want
    if (shape, T) == (synth.DEAMOE_7B, 16):
        assert want == 2          # dense department backbones: tensor cores
    if (shape, T) == (synth.VANILLA_128E, 16):
        assert want == 0          # ~1 token per expert expected: tensor cores not launched
    if (shape, T) == (synth.DEAMOE_7B_FP8, 16):
        assert want == 2          # E4M3 weights take the same choice as bf16
