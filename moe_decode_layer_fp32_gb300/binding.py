"""ctypes binding of ``libmoe_gb300.so``: argument marshalling only.

Every function has the name of the C entry point it calls (see
``include/moe_decode.h``).  Tensors are passed as device pointers, sizes are
read from their shapes, and the stream is torch's current CUDA stream.  No
step of the layer runs here; a missing library raises instead of falling back.
"""

from __future__ import annotations

import ctypes as C
import os

import torch

LIB_PATH = os.environ.get("MOE_GB300_LIB") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "libmoe_gb300.so")

MOE_OK = 0
MOE_DTYPE_F32 = 0
MOE_DTYPE_BF16 = 1
MOE_DTYPE_FP8_E4M3 = 2
MOE_OUT_ROWS = 0
MOE_OUT_ACCUM = 1

ERRORS = {-1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_WORKSPACE",
          -4: "MOE_ERR_CUDA", -5: "MOE_ERR_TIMEOUT", -6: "MOE_ERR_DEVICE"}

WS_FIELDS = ("total", "status", "counts", "logits", "exp_count", "exp_off", "asg_tok",
             "asg_slot", "asg_w", "tok_asg", "act_exp", "dept_count", "dept_off", "dept_tok",
             "dept_w", "tok_dpos", "act_dept", "exp_units", "dept_units", "sync", "xb")


class WsLayout(C.Structure):
    _fields_ = [(f, C.c_size_t) for f in WS_FIELDS]


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {ERRORS.get(code, code)}: {msg}")
        self.code = code


_lib = None

_P, _I, _F, _SZ, _I64 = C.c_void_p, C.c_int, C.c_float, C.c_size_t, C.c_int64

_SIGS = {
    "moe_version": (_I, []),
    "moe_set_tc_min_tokens": (_I, [_I]),
    "moe_test_stall_weight_copies": (C.c_int64, [C.c_int64]),
    "moe_last_error": (C.c_char_p, []),
    "moe_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "moe_workspace_layout": (_I, [_I, _I, _I, _I, C.POINTER(WsLayout)]),
    "moe_workspace_init": (_I, [_P, _SZ, _P]),
    "moe_read_status": (_I, [_P, _SZ, C.POINTER(C.c_int32), C.POINTER(C.c_int32), _P]),
    "moe_input_from_host": (_I, [_P, _P, _I, _I, _P]),
    "moe_output_to_host": (_I, [_P, _P, _I, _I, _P]),
    "moe_route_topk": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _SZ, _P]),
    "moe_route_topk_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P]),
    "moe_bias_update": (_I, [_P, _I, _F, _I, _P, _P, _P]),
    "moe_ffn_vanilla_fp8": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P, _SZ, _I, _P, _P]),
    "deamoe_ffn_fp8": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P,
                            _SZ, _I, _P, _P]),
    "moe_layer_forward_fp8": (_I, [_P, _I, _I, _I, _I, _F, _P, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P,
                                   _SZ, _P, _P, _P, _P]),
    "deamoe_layer_forward_fp8": (_I, [_P, _I, _I, _I, _I, _F, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                                      _I, _P, _P, _P, _P, _P, _SZ, _P, _P, _P, _P]),
    "moe_formp_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "deamoe_p_layer_forward": (_I, [_P, _I, _I, _I, _I, _F, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P,
                                    _P, _P, _P, _SZ, _P, _P, _P, _P]),
    "moe_unique_weight_bytes_formp": (C.c_int64, [_I, _I, _I, _I, _I]),
    "deamoe_p_ffn": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "moe_route_topk_grouped": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _SZ, _P]),
    "moe_dispatch": (_I, [_P, _P, _I, _I, _I, _I, _P, _SZ, _P]),
    "moe_rows_count": (_I64, [_I, _I, _I, _I, _I]),
    "moe_ffn_vanilla": (_I, [_P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P,
                             _P, _SZ, _I, _P, _P]),
    "deamoe_ffn": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I,
                        _P, _P, _P, _P, _SZ, _I, _P, _P]),
    "moe_combine": (_I, [_P, _I, _I, _I, _I, _I, _I, _P, _SZ, _P, _P]),
    "moe_layer_forward": (_I, [_P, _I, _I, _I, _I, _F, _P, _P, _I, _I, _P, _P, _P, _I,
                               _P, _P, _P, _P, _SZ, _P, _P, _P, _P]),
    "deamoe_layer_forward": (_I, [_P, _I, _I, _I, _I, _F, _P, _P, _I, _I, _I, _I, _P, _P,
                                  _P, _P, _P, _P, _I, _P, _P, _P, _P, _SZ, _P, _P, _P, _P]),
    "moe_unique_weight_bytes_vanilla": (_I64, [_I, _I, _I, _I, _I, _I]),
    "moe_unique_weight_bytes_deamoe": (_I64, [_I, _I, _I, _I, _I, _I, _I, _I]),
}


def lib() -> C.CDLL:
    """Load the native library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"native library not built: {LIB_PATH} "
                              "(run __graft_entry__.build())")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return tuple(_SIGS)


def _check(fn: str, rc: int):
    if rc != MOE_OK:
        raise MoeError(fn, rc, lib().moe_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _dtype_code(t) -> int:
    if t.dtype == torch.bfloat16:
        return MOE_DTYPE_BF16
    if t.dtype == torch.float32:
        return MOE_DTYPE_F32
    if t.dtype == torch.float8_e4m3fn:
        return MOE_DTYPE_FP8_E4M3
    raise ValueError(f"unsupported weight dtype {t.dtype}")


def _scales(scales, count: int):
    """Host array of device pointers to the FP8 row scales (None entries for
    absent classes)."""
    if scales is None or len(scales) != count:
        raise ValueError(f"FP8 weights need {count} row-scale tensors (None where a class is absent)")
    return (C.c_void_p * count)(*[_ptr(t) for t in scales])


def moe_set_tc_min_tokens(min_tokens: int) -> int:
    r = lib().moe_set_tc_min_tokens(min_tokens)
    if r < 0:
        raise MoeError("moe_set_tc_min_tokens", r, lib().moe_last_error().decode())
    return r


def moe_test_stall_weight_copies(wait_ns: int) -> int:
    """Test hook: FFN steps launched while wait_ns > 0 issue no weight copy
    and give up their waits after wait_ns ns (MOE_ERR_TIMEOUT in the
    workspace status).  Returns the previous setting."""
    r = lib().moe_test_stall_weight_copies(int(wait_ns))
    if r < 0:
        raise MoeError("moe_test_stall_weight_copies", r, lib().moe_last_error().decode())
    return int(r)


# ---------------------------------------------------------------- workspace


def moe_workspace_bytes(T: int, n: int, k: int, experts_per_dept: int = 1) -> int:
    b = lib().moe_workspace_bytes(T, n, k, experts_per_dept)
    if b == 0:
        raise MoeError("moe_workspace_bytes", -1, "invalid sizes")
    return b


def moe_workspace_layout(T: int, n: int, k: int, experts_per_dept: int = 1) -> dict:
    L = WsLayout()
    _check("moe_workspace_layout", lib().moe_workspace_layout(T, n, k, experts_per_dept, C.byref(L)))
    return {f: getattr(L, f) for f in WS_FIELDS}


def new_workspace(T: int, n: int, k: int, experts_per_dept: int = 1, device="cuda") -> torch.Tensor:
    """Allocate (torch) and zero (library kernel) a workspace."""
    ws = torch.empty(moe_workspace_bytes(T, n, k, experts_per_dept), dtype=torch.uint8, device=device)
    moe_workspace_init(ws)
    return ws


def moe_workspace_init(ws: torch.Tensor):
    _check("moe_workspace_init", lib().moe_workspace_init(_ptr(ws), ws.numel(), _stream()))


def moe_read_status(ws: torch.Tensor):
    """(status, A_e, A_d) -- synchronises the current stream."""
    st = (C.c_int32 * 1)()
    cnt = (C.c_int32 * 2)()
    _check("moe_read_status", lib().moe_read_status(_ptr(ws), ws.numel(), st, cnt, _stream()))
    return int(st[0]), int(cnt[0]), int(cnt[1])


def _host_ptr(t):
    if t.is_cuda:
        raise ValueError("expected a host (CPU) tensor")
    if not t.is_contiguous() or t.dtype != torch.float32:
        raise ValueError("expected a contiguous float32 host tensor")
    return t.data_ptr()


def moe_input_from_host(x, x_host):
    """Enqueue the copy of host activations x_host [T, d] into device x [T, d]."""
    if x.shape != x_host.shape or x.dim() != 2 or x.dtype != torch.float32:
        raise ValueError("x and x_host must both be float32 [T, d]")
    T, d = x.shape
    _check("moe_input_from_host", lib().moe_input_from_host(_ptr(x), _host_ptr(x_host), T, d, _stream()))


def moe_output_to_host(y_host, y):
    """Enqueue the copy of the device output y [T, d] into host y_host [T, d]."""
    if y.shape != y_host.shape or y.dim() != 2 or y.dtype != torch.float32:
        raise ValueError("y and y_host must both be float32 [T, d]")
    T, d = y.shape
    _check("moe_output_to_host", lib().moe_output_to_host(_host_ptr(y_host), _ptr(y), T, d, _stream()))


# ---------------------------------------------------------------- steps


def moe_route_topk(x, w_router, bias, k: int, scale: float, topk_idx, topk_w, ws):
    T, d = x.shape
    n = w_router.shape[0]
    _check("moe_route_topk", lib().moe_route_topk(
        _ptr(x), _ptr(w_router), _ptr(bias), T, d, n, k, scale, _ptr(topk_idx), _ptr(topk_w),
        _ptr(ws), ws.numel(), _stream()))


def moe_route_topk_noalloc(x, w_router, bias, k: int, scale: float, topk_idx, topk_w, status=None):
    """``status``: int32 CUDA tensor of one element, or None."""
    T, d = x.shape
    n = w_router.shape[0]
    _check("moe_route_topk_noalloc", lib().moe_route_topk_noalloc(
        _ptr(x), _ptr(w_router), _ptr(bias), T, d, n, k, scale, _ptr(topk_idx), _ptr(topk_w),
        _ptr(status), _stream()))


def moe_route_topk_grouped(x, w_router, bias, k: int, experts_per_dept: int, k_dept: int, strict: bool,
                           scale: float, topk_idx, topk_w, ws):
    T, d = x.shape
    n = w_router.shape[0]
    _check("moe_route_topk_grouped", lib().moe_route_topk_grouped(
        _ptr(x), _ptr(w_router), _ptr(bias), T, d, n, k, experts_per_dept, k_dept, int(bool(strict)), scale,
        _ptr(topk_idx), _ptr(topk_w), _ptr(ws), ws.numel(), _stream()))


MOE_BIAS_SIGN = 0
MOE_BIAS_PROPORTIONAL = 1


def moe_bias_update(counts, gamma: float, rule: int, bias=None, imbalance=None):
    """``counts``: int32 CUDA tensor [n]; ``bias`` float32 [n] (updated in
    place) and/or ``imbalance`` float32 [1]."""
    _check("moe_bias_update", lib().moe_bias_update(
        _ptr(counts), counts.numel(), gamma, rule, _ptr(bias), _ptr(imbalance), _stream()))


def workspace_counts(ws, T: int, n: int, k: int, experts_per_dept: int):
    """The workspace's per-expert token counts (int32 [n]) as a view of ws."""
    off = moe_workspace_layout(T, n, k, experts_per_dept)["exp_count"]
    return ws[off: off + 4 * n].view(torch.int32)


def moe_dispatch(topk_idx, topk_w, n: int, experts_per_dept: int, ws):
    T, k = topk_idx.shape
    _check("moe_dispatch", lib().moe_dispatch(
        _ptr(topk_idx), _ptr(topk_w), T, n, k, experts_per_dept, _ptr(ws), ws.numel(), _stream()))


def moe_rows_count(T: int, n: int, k: int, experts_per_dept: int, has_shared: bool) -> int:
    r = lib().moe_rows_count(T, n, k, experts_per_dept, 1 if has_shared else 0)
    if r < 0:
        raise MoeError("moe_rows_count", -1, "invalid sizes")
    return r


def moe_ffn_vanilla(x, k: int, w_gate, w_up, w_down, shared, ws, out_mode: int, out, scales=None):
    """``shared`` = (s_gate, s_up, s_down) or None; FP8 weights: ``scales`` =
    the row scales (gate, up, down of the experts, then of the shared expert)."""
    T, d = x.shape
    n, I, _ = w_gate.shape
    sg, su, sd = shared if shared is not None else (None, None, None)
    I_s = sg.shape[0] if sg is not None else 0
    if _dtype_code(w_gate) == MOE_DTYPE_FP8_E4M3:
        _check("moe_ffn_vanilla_fp8", lib().moe_ffn_vanilla_fp8(
            _ptr(x), T, d, n, k, I, _ptr(w_gate), _ptr(w_up), _ptr(w_down), I_s, _ptr(sg), _ptr(su),
            _ptr(sd), _scales(scales, 6), _ptr(ws), ws.numel(), out_mode, _ptr(out), _stream()))
        return
    _check("moe_ffn_vanilla", lib().moe_ffn_vanilla(
        _ptr(x), T, d, n, k, I, _dtype_code(w_gate), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
        I_s, _ptr(sg), _ptr(su), _ptr(sd), _ptr(ws), ws.numel(), out_mode, _ptr(out), _stream()))


def deamoe_ffn(x, k: int, experts_per_dept: int, dept, priv, shared, ws, out_mode: int, out, scales=None):
    """``dept`` = (gate, up, down) [m, I_sh, d]; ``priv`` = (gate, up, down)
    [n, I_pr, d] or None; ``shared`` = (gate, up, down) [I_s, d] or None; FP8
    weights: ``scales`` = 9 row-scale tensors (departments, private, shared)."""
    T, d = x.shape
    m, I_sh, _ = dept[0].shape
    n = m * experts_per_dept
    pg, pu, pd = priv if priv is not None else (None, None, None)
    I_pr = pg.shape[1] if pg is not None else 0
    sg, su, sd = shared if shared is not None else (None, None, None)
    I_s = sg.shape[0] if sg is not None else 0
    if _dtype_code(dept[0]) == MOE_DTYPE_FP8_E4M3:
        _check("deamoe_ffn_fp8", lib().deamoe_ffn_fp8(
            _ptr(x), T, d, n, k, experts_per_dept, I_sh, I_pr, _ptr(dept[0]), _ptr(dept[1]), _ptr(dept[2]),
            _ptr(pg), _ptr(pu), _ptr(pd), I_s, _ptr(sg), _ptr(su), _ptr(sd), _scales(scales, 9), _ptr(ws),
            ws.numel(), out_mode, _ptr(out), _stream()))
        return
    _check("deamoe_ffn", lib().deamoe_ffn(
        _ptr(x), T, d, n, k, experts_per_dept, I_sh, I_pr, _dtype_code(dept[0]),
        _ptr(dept[0]), _ptr(dept[1]), _ptr(dept[2]), _ptr(pg), _ptr(pu), _ptr(pd),
        I_s, _ptr(sg), _ptr(su), _ptr(sd), _ptr(ws), ws.numel(), out_mode, _ptr(out), _stream()))


def moe_combine(rows, T: int, n: int, k: int, experts_per_dept: int, has_shared: bool, ws, y):
    d = rows.shape[1]
    _check("moe_combine", lib().moe_combine(
        _ptr(rows), T, d, n, k, experts_per_dept, 1 if has_shared else 0, _ptr(ws), ws.numel(),
        _ptr(y), _stream()))


def moe_layer_forward(x, k: int, scale: float, w_router, bias, w_gate, w_up, w_down, shared,
                      ws, topk_idx, topk_w, y, scales=None):
    T, d = x.shape
    n, I, _ = w_gate.shape
    sg, su, sd = shared if shared is not None else (None, None, None)
    I_s = sg.shape[0] if sg is not None else 0
    if _dtype_code(w_gate) == MOE_DTYPE_FP8_E4M3:
        _check("moe_layer_forward_fp8", lib().moe_layer_forward_fp8(
            _ptr(x), T, d, n, k, scale, _ptr(w_router), _ptr(bias), I, _ptr(w_gate), _ptr(w_up),
            _ptr(w_down), I_s, _ptr(sg), _ptr(su), _ptr(sd), _scales(scales, 6), _ptr(ws), ws.numel(),
            _ptr(topk_idx), _ptr(topk_w), _ptr(y), _stream()))
        return
    _check("moe_layer_forward", lib().moe_layer_forward(
        _ptr(x), T, d, n, k, scale, _ptr(w_router), _ptr(bias), I, _dtype_code(w_gate),
        _ptr(w_gate), _ptr(w_up), _ptr(w_down), I_s, _ptr(sg), _ptr(su), _ptr(sd),
        _ptr(ws), ws.numel(), _ptr(topk_idx), _ptr(topk_w), _ptr(y), _stream()))


def deamoe_layer_forward(x, k: int, scale: float, w_router, bias, experts_per_dept: int, dept,
                         priv, shared, ws, topk_idx, topk_w, y, scales=None):
    T, d = x.shape
    n = w_router.shape[0]
    I_sh = dept[0].shape[1]
    pg, pu, pd = priv if priv is not None else (None, None, None)
    I_pr = pg.shape[1] if pg is not None else 0
    sg, su, sd = shared if shared is not None else (None, None, None)
    I_s = sg.shape[0] if sg is not None else 0
    if _dtype_code(dept[0]) == MOE_DTYPE_FP8_E4M3:
        _check("deamoe_layer_forward_fp8", lib().deamoe_layer_forward_fp8(
            _ptr(x), T, d, n, k, scale, _ptr(w_router), _ptr(bias), experts_per_dept, I_sh, I_pr,
            _ptr(dept[0]), _ptr(dept[1]), _ptr(dept[2]), _ptr(pg), _ptr(pu), _ptr(pd), I_s, _ptr(sg),
            _ptr(su), _ptr(sd), _scales(scales, 9), _ptr(ws), ws.numel(), _ptr(topk_idx), _ptr(topk_w),
            _ptr(y), _stream()))
        return
    _check("deamoe_layer_forward", lib().deamoe_layer_forward(
        _ptr(x), T, d, n, k, scale, _ptr(w_router), _ptr(bias), experts_per_dept, I_sh, I_pr,
        _dtype_code(dept[0]), _ptr(dept[0]), _ptr(dept[1]), _ptr(dept[2]), _ptr(pg), _ptr(pu),
        _ptr(pd), I_s, _ptr(sg), _ptr(su), _ptr(sd), _ptr(ws), ws.numel(), _ptr(topk_idx),
        _ptr(topk_w), _ptr(y), _stream()))


def moe_formp_workspace_bytes(T: int, n: int, k: int, experts_per_dept: int, r: int) -> int:
    return int(lib().moe_formp_workspace_bytes(T, n, k, experts_per_dept, r))


def new_formp_workspace(T: int, n: int, k: int, experts_per_dept: int, r: int, device="cuda") -> torch.Tensor:
    """Allocate (torch) and zero (library kernel) a form-P workspace."""
    nbytes = moe_formp_workspace_bytes(T, n, k, experts_per_dept, r)
    if nbytes == 0:
        raise MoeError("moe_formp_workspace_bytes", -1, "invalid sizes")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    moe_workspace_init(ws)
    return ws


def deamoe_p_layer_forward(x, k: int, scale: float, w_router, bias, experts_per_dept: int, k_dept: int,
                           dept, amat, ws, topk_idx, topk_w, y):
    """``dept`` = (gate, up, down) [m, r, d]; ``amat`` = (A_g, A_u, A_d) [n, r, r]."""
    T, d = x.shape
    n = w_router.shape[0]
    r = dept[0].shape[1]
    _check("deamoe_p_layer_forward", lib().deamoe_p_layer_forward(
        _ptr(x), T, d, n, k, scale, _ptr(w_router), _ptr(bias), experts_per_dept, k_dept, r,
        _dtype_code(dept[0]), _ptr(dept[0]), _ptr(dept[1]), _ptr(dept[2]), _ptr(amat[0]), _ptr(amat[1]),
        _ptr(amat[2]), _ptr(ws), ws.numel(), _ptr(topk_idx), _ptr(topk_w), _ptr(y), _stream()))


def deamoe_p_ffn(x, k: int, experts_per_dept: int, dept, amat, topk_idx, ws, y):
    T, d = x.shape
    n = amat[0].shape[0]
    r = dept[0].shape[1]
    _check("deamoe_p_ffn", lib().deamoe_p_ffn(
        _ptr(x), T, d, n, k, experts_per_dept, r, _dtype_code(dept[0]), _ptr(dept[0]), _ptr(dept[1]),
        _ptr(dept[2]), _ptr(amat[0]), _ptr(amat[1]), _ptr(amat[2]), _ptr(topk_idx), _ptr(ws), ws.numel(),
        _ptr(y), _stream()))


def moe_unique_weight_bytes_formp(d, n, r, A_d, A_e) -> int:
    return int(lib().moe_unique_weight_bytes_formp(d, n, r, A_d, A_e))


def moe_unique_weight_bytes_vanilla(d, n, I, I_s, dtype_code, A_e) -> int:
    return int(lib().moe_unique_weight_bytes_vanilla(d, n, I, I_s, dtype_code, A_e))


def moe_unique_weight_bytes_deamoe(d, n, I_sh, I_pr, I_s, dtype_code, A_d, A_e) -> int:
    return int(lib().moe_unique_weight_bytes_deamoe(d, n, I_sh, I_pr, I_s, dtype_code, A_d, A_e))
