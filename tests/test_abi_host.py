"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every declared entry point, and rejects bad arguments before
launching anything."""

import ctypes as C
import os
import re

import pytest

from tests.helpers import ensure_built
from oracle import moe_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    return ensure_built()


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, re.M):
            if m.group(1) not in ("defined",):
                names.append(m.group(1))
    return names


def test_library_exports_every_declared_symbol(B):
    L = B.lib()
    names = declared_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(L, name), f"{name} declared in include/ but not exported"
    # and the binding covers every declared entry point
    assert set(names) == set(B.exported_symbols())


def test_version_and_error_string(B):
    assert B.lib().moe_version() >= 100
    assert isinstance(B.lib().moe_last_error(), bytes)


# memory order of the workspace arrays (the header lists them in this order)
WS_ORDER = ("status", "counts", "sync", "logits", "exp_count", "exp_off", "asg_tok", "asg_slot", "asg_w",
            "tok_asg", "act_exp", "exp_units", "xb", "dept_count", "dept_off", "dept_tok", "dept_w",
            "tok_dpos", "act_dept", "dept_units")
WS_SHARED = WS_ORDER[:WS_ORDER.index("dept_count")]


def test_workspace_layout_is_ordered_and_aligned(B):
    for (T, n, k, g) in [(1, 16, 2, 1), (4, 16, 2, 4), (16, 128, 8, 1), (128, 64, 8, 8), (64, 256, 8, 16)]:
        L = B.moe_workspace_layout(T, n, k, g)
        offs = [L[f] for f in WS_ORDER]
        assert offs == sorted(offs)
        assert all(o % 256 == 0 for o in offs)
        assert L["total"] == B.moe_workspace_bytes(T, n, k, g)
        # documented fixed positions (moe_read_status reads status and counts)
        assert (L["status"], L["counts"], L["sync"]) == (0, 256, 512)
        assert L["logits"] >= L["sync"] + 18 * 4
        assert L["total"] >= L["dept_units"]


def test_workspace_serves_smaller_steps_and_routing_views(B):
    """A workspace sized for (T_max, n, k, g) holds every smaller step's layout,
    and the g = 1 layout a routing call uses has the same offsets as the
    department workspace for every array it has (the counters above all)."""
    for (T, n, k, g) in [(128, 64, 8, 8), (64, 256, 8, 16), (32, 16, 2, 4), (128, 1024, 32, 2)]:
        big = B.moe_workspace_layout(T, n, k, g)
        for t in (1, 3, 16, T):
            if t > T:
                continue
            small = B.moe_workspace_layout(t, n, k, g)
            assert small["total"] <= big["total"]
            view = B.moe_workspace_layout(t, n, k, 1)
            assert {f: view[f] for f in WS_SHARED} == {f: small[f] for f in WS_SHARED}
            assert view["total"] <= small["total"]
            assert (small["status"], small["counts"], small["sync"]) == (0, 256, 512)


@pytest.mark.parametrize("args", [(0, 16, 2, 1), (129, 16, 2, 1), (4, 16, 0, 1), (4, 16, 17, 1),
                                  (4, 16, 33, 64), (4, 16, 2, 3), (4, 2048, 2, 1)])
def test_workspace_rejects_bad_sizes(B, args):
    assert B.lib().moe_workspace_bytes(*args) == 0
    L = B.WsLayout()
    assert B.lib().moe_workspace_layout(*args, C.byref(L)) == -1


def test_calls_reject_null_and_small_workspace(B):
    lib = B.lib()
    # null workspace
    rc = lib.moe_route_topk(None, None, None, 4, 256, 16, 2, 1.0, None, None, None, 0, None)
    assert rc == -1 and b"workspace" in lib.moe_last_error()
    # workspace too small (a fake aligned address; nothing is launched)
    fake = 1 << 20
    rc = lib.moe_dispatch(fake, fake, 4, 16, 2, 1, fake, 64, None)
    assert rc == -3
    # bad hidden size
    need = lib.moe_workspace_bytes(4, 16, 2, 1)
    rc = lib.moe_route_topk(fake, fake, None, 4, 12, 16, 2, 1.0, fake, fake, fake, need, None)
    assert rc == -1 and b"d=12" in lib.moe_last_error()
    # misaligned weights
    rc = lib.moe_ffn_vanilla(fake, 4, 256, 16, 2, 64, 1, fake + 2, fake, fake, 0, None, None, None,
                             fake, need, 1, fake, None)
    assert rc == -1 and b"unaligned" in lib.moe_last_error()
    # intermediate not a multiple of 16
    rc = lib.moe_ffn_vanilla(fake, 4, 256, 16, 2, 40, 1, fake, fake, fake, 0, None, None, None,
                             fake, need, 1, fake, None)
    assert rc == -1
    # unsupported dtype / out mode
    rc = lib.moe_ffn_vanilla(fake, 4, 256, 16, 2, 64, 7, fake, fake, fake, 0, None, None, None,
                             fake, need, 1, fake, None)
    assert rc == -2
    rc = lib.moe_ffn_vanilla(fake, 4, 256, 16, 2, 64, 1, fake, fake, fake, 0, None, None, None,
                             fake, need, 5, fake, None)
    assert rc == -1
    # hidden size wider than the streaming kernel covers
    rc = lib.moe_ffn_vanilla(fake, 4, 8192, 16, 2, 64, 1, fake, fake, fake, 0, None, None, None,
                             fake, need, 1, fake, None)
    assert rc == -2
    # DeaMoE needs g >= 1 and n % g == 0
    need4 = lib.moe_workspace_bytes(4, 16, 2, 4)
    rc = lib.deamoe_ffn(fake, 4, 256, 16, 2, 0, 64, 16, 1, fake, fake, fake, fake, fake, fake, 0,
                        None, None, None, fake, need4, 1, fake, None)
    assert rc == -1
    rc = lib.deamoe_ffn(fake, 4, 256, 16, 2, 3, 64, 16, 1, fake, fake, fake, fake, fake, fake, 0,
                        None, None, None, fake, need4, 1, fake, None)
    assert rc == -1


def test_rows_count(B):
    assert B.moe_rows_count(4, 16, 2, 1, False) == 8
    assert B.moe_rows_count(4, 16, 2, 1, True) == 12
    assert B.moe_rows_count(4, 16, 2, 4, False) == 8 + 8      # T*min(k,m) = 4*2
    assert B.moe_rows_count(16, 64, 8, 8, True) == 128 + 128 + 16


def test_unique_bytes_match_oracle_formula(B):
    for (d, n, I, I_s, A_e) in [(2048, 128, 768, 0, 8), (7168, 256, 2048, 2048, 77), (256, 16, 576, 0, 3)]:
        for code, bw in ((0, 4), (1, 2)):
            assert B.moe_unique_weight_bytes_vanilla(d, n, I, I_s, code, A_e) == \
                O.unique_bytes_vanilla(d, n, I, I_s, A_e, bw)
    for (d, n, I_sh, I_pr, I_s, A_d, A_e) in [(2048, 64, 1024, 128, 0, 6, 8), (7168, 256, 1792, 256, 2048, 16, 200)]:
        assert B.moe_unique_weight_bytes_deamoe(d, n, I_sh, I_pr, I_s, 1, A_d, A_e) == \
            O.unique_bytes_deamoe_c(d, n, I_sh, I_pr, I_s, A_d, A_e, 2)
    assert B.moe_unique_weight_bytes_vanilla(2048, 128, 768, 0, 9, 8) == -1


def test_unique_bytes_formp_match_oracle_formula(B):
    """The library's form-P count (bf16 weights) equals the oracle's, whose
    closed form is pinned to the bytes of the tensors an evaluation touches."""
    for (d, n, r, A_d, A_e) in [(256, 16, 64, 2, 4), (1024, 672, 384, 4, 10), (1024, 672, 384, 8, 383),
                                (7168, 864, 2048, 5, 10), (7168, 864, 2048, 8, 416), (2048, 64, 1024, 0, 0)]:
        assert B.moe_unique_weight_bytes_formp(d, n, r, A_d, A_e) == \
            O.unique_bytes_deamoe_p(d, n, r, A_d, A_e, 2)
    lib = B.lib()
    for bad in ((0, 16, 64, 1, 1), (256, 16, 0, 1, 1), (256, 16, 64, -1, 1), (256, 16, 64, 1, 17)):
        assert lib.moe_unique_weight_bytes_formp(*bad) == -1


# ---------------------------------------------------------------------------
# Host checks of the NEXT-row entry points (nothing is launched)
# ---------------------------------------------------------------------------

FAKE = 1 << 20          # an aligned address that is never dereferenced


def test_grouped_routing_rejects_bad_group_arguments(B):
    lib = B.lib()
    need = lib.moe_workspace_bytes(4, 16, 4, 1)
    args = lambda g, kd, strict, k=4: (FAKE, FAKE, None, 4, 256, 16, k, g, kd, strict, 1.0, FAKE, FAKE,  # noqa: E731
                                       FAKE, need, None)
    for g, kd, strict, k in ((3, 1, 0, 4), (4, 0, 0, 4), (4, 5, 0, 4), (4, 1, 0, 5), (1, 5, 1, 4)):
        assert lib.moe_route_topk_grouped(*args(g, kd, strict, k)) == -1


def test_host_activation_copies_reject_bad_arguments(B):
    lib = B.lib()
    for fn in (lib.moe_input_from_host, lib.moe_output_to_host):
        assert fn(None, FAKE, 4, 256, None) == -1
        assert fn(FAKE, None, 4, 256, None) == -1
        assert fn(FAKE, FAKE, 0, 256, None) == -1
        assert fn(FAKE, FAKE, 4, 0, None) == -1
        assert b"T=4, d=0" in lib.moe_last_error()
    import torch
    with pytest.raises(ValueError):   # shapes that differ
        B.moe_output_to_host(torch.zeros(2, 8), torch.zeros(2, 4))


def test_bias_update_rejects_bad_arguments_on_the_host(B):
    lib = B.lib()
    assert lib.moe_bias_update(FAKE, 0, 0.1, 0, FAKE, None, None) == -1
    assert lib.moe_bias_update(FAKE, 1025, 0.1, 0, FAKE, None, None) == -1
    assert lib.moe_bias_update(None, 8, 0.1, 0, FAKE, None, None) == -1
    assert lib.moe_bias_update(FAKE, 8, 0.1, 0, None, None, None) == -1
    assert lib.moe_bias_update(FAKE, 8, 0.1, 7, FAKE, None, None) == -1
    assert lib.moe_bias_update(FAKE, 8, -0.5, 0, FAKE, None, None) == -1
    assert lib.moe_bias_update(FAKE, 8, float("nan"), 1, FAKE, None, None) == -1
    assert lib.moe_bias_update(FAKE, 8, float("inf"), 1, FAKE, None, None) == -1


def test_formp_workspace_and_argument_checks(B):
    lib = B.lib()
    T, n, k, g, r = 4, 16, 4, 4, 64
    base = lib.moe_workspace_bytes(T, n, k, g)
    total = lib.moe_formp_workspace_bytes(T, n, k, g, r)
    # G and U per department entry (T * min(k, m)), A_d^T Y per assignment, fp32
    assert total >= base + 4 * r * (2 * T * min(k, n // g) + T * k)
    assert lib.moe_formp_workspace_bytes(T, n, k, 1, r) == 0        # no departments
    assert lib.moe_formp_workspace_bytes(T, n, k, g, 40) == 0       # r % 16
    w = (FAKE,) * 6

    def call(k_dept=0, dtype=1, rr=r, ws_bytes=total, weights=w, d=256):
        return lib.deamoe_p_layer_forward(FAKE, T, d, n, k, 1.0, FAKE, None, g, k_dept, rr, dtype, *weights,
                                          FAKE, ws_bytes, FAKE, FAKE, FAKE, None)
    assert call(k_dept=-1) == -1
    assert call(k_dept=5) == -1                      # more departments than m = 4
    assert call(dtype=0) == -2                       # fp32 weights
    assert call(ws_bytes=total - 256) == -3
    assert call(weights=(FAKE, None, FAKE, FAKE, FAKE, FAKE)) == -1
    assert call(d=8192) == -2                        # wider than the passes take
    big = lib.moe_formp_workspace_bytes(T, n, k, g, 4096)
    assert call(rr=4096, ws_bytes=big) == -2         # r above 2048


def test_fp8_calls_need_their_row_scales(B):
    lib = B.lib()
    T, d, n, k, I = 2, 256, 16, 2, 64
    need = lib.moe_workspace_bytes(T, n, k, 1)
    # the bf16 / fp32 call with the FP8 code: refused before any launch
    rc = lib.moe_layer_forward(FAKE, T, d, n, k, 1.0, FAKE, None, I, B.MOE_DTYPE_FP8_E4M3, FAKE, FAKE, FAKE, 0,
                               None, None, None, FAKE, need, FAKE, FAKE, FAKE, None)
    assert rc == -1 and b"row scales" in lib.moe_last_error()
    # the FP8 call without scales, or with a missing one
    rc = lib.moe_layer_forward_fp8(FAKE, T, d, n, k, 1.0, FAKE, None, I, FAKE, FAKE, FAKE, 0, None, None, None,
                                   None, FAKE, need, FAKE, FAKE, FAKE, None)
    assert rc == -1
    sc = (C.c_void_p * 6)(FAKE, None, FAKE, None, None, None)
    rc = lib.moe_layer_forward_fp8(FAKE, T, d, n, k, 1.0, FAKE, None, I, FAKE, FAKE, FAKE, 0, None, None, None,
                                   sc, FAKE, need, FAKE, FAKE, FAKE, None)
    assert rc == -1 and b"set 0" in lib.moe_last_error()
    # FP8 bytes: codes plus three fp32 scales per row
    assert lib.moe_unique_weight_bytes_vanilla(d, n, I, 0, B.MOE_DTYPE_FP8_E4M3, 3) == 4 * d * n + 3 * I * 3 * (d + 4)
