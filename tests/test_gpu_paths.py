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
