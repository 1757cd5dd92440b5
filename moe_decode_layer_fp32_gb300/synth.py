"""Seeded synthetic inputs for the MoE / DeaMoE decode layer.

This module is the one place both the CUDA path (tests, bench) and the CPU oracle
take their inputs from. It holds none of the layer's arithmetic: it draws random
numbers, rounds them to the storage dtype and builds the Zipf router bias used by
the skewed-routing sweep. Nothing here routes, multiplies or combines.

Recipe (all values seeded; no dataset is involved):

* hidden states ``x ~ N(0, 1)``, fp32, shape ``[T, d]``;
* every weight ``~ N(0, 0.02)``, drawn in fp32 and rounded to nearest-even into
  the storage dtype (bf16 or fp32);
* the router is drawn as a ``[d, n]`` array and stored transposed, ``[n, d]``,
  so that row ``e`` is expert ``e``'s router vector;
* projection weights are stored ``[unit, rows, d]``: gate and up rows are the
  rows of ``W_gate`` / ``W_up`` (shape ``[I, d]``), and the down tensor holds
  the paper's ``W_down`` with shape ``[I, d]``, applied transposed
  (DeaMoE: Efficient MoE Structure for Fast Small-Batch Decoding, §2.1).

Every tensor has its own stream: the generator is seeded with a 63-bit mix of
``(seed, tensor id)``, so adding a tensor never changes the others.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

# ---------------------------------------------------------------------------
# Workload shapes (the layer sizes of the pages' Table 1 models and of the
# synthetic sweeps built on them).
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class LayerShape:
    """Shapes of one decode layer (vanilla MoE or DeaMoE form C)."""

    name: str
    d: int                 # hidden size (h in the DeaMoE paper)
    n: int                 # routed experts
    k: int                 # experts per token
    dtype: str             # weight storage: "bf16", "f32" or "fp8" (E4M3 + fp32 row scales)
    # vanilla
    I: int = 0             # vanilla expert intermediate
    # DeaMoE form C
    g: int = 1             # experts per department (m = n // g)
    I_sh: int = 0          # department shared intermediate
    I_pr: int = 0          # per-expert private intermediate
    # always-on shared expert (DeepSeekMoE style); 0 = none
    I_s: int = 0
    batches: tuple = field(default_factory=tuple)
    zipf: float = 0.0      # >0: router bias makes popularity Zipf(s)
    zipf_g: int = 0        # department size used to build that bias
    # DeaMoE in the paper's parameterisation (eq. 4): departments of width
    # r = I_sh and per-expert r x r matrices A_g, A_u, A_d
    form_p: bool = False
    k_dept: int = 0        # group-limited routing: departments per token (0 = plain top-k)

    @property
    def m(self) -> int:
        return self.n // self.g


# Tiny correctness layer, fp32 weights: 16 experts in 4 departments of 4,
# shared intermediate 512 + private 64; the vanilla twin has intermediate 576.
TINY_DEAMOE = LayerShape("tiny-deamoe-fp32", d=256, n=16, k=2, dtype="f32",
                         g=4, I_sh=512, I_pr=64, batches=(4,))
TINY_VANILLA = LayerShape("tiny-vanilla-fp32", d=256, n=16, k=2, dtype="f32",
                          I=576, batches=(4,))
# Vanilla decode layer: d=2048, 128 experts, intermediate 768, top-8, bf16.
VANILLA_128E = LayerShape("vanilla-d2048-e128-i768-top8-bf16", d=2048, n=128, k=8,
                          dtype="bf16", I=768, batches=(1, 4, 16))
# DeaMoE ~7B-class layer and its budget-matched vanilla twin.
DEAMOE_7B = LayerShape("deamoe-d2048-e64-dept8x8-ish1024-ipr128-top8-bf16", d=2048,
                       n=64, k=8, dtype="bf16", g=8, I_sh=1024, I_pr=128,
                       batches=(1, 4, 8, 16))
VANILLA_7B = LayerShape("vanilla-d2048-e64-i1152-top8-bf16", d=2048, n=64, k=8,
                        dtype="bf16", I=1152, batches=(1, 4, 8, 16))
# DeepSeek-V3-shaped layer (+1 shared expert) and its DeaMoE variant.
DSV3_VANILLA = LayerShape("vanilla-d7168-e256-i2048-top8-shared2048-bf16", d=7168,
                          n=256, k=8, dtype="bf16", I=2048, I_s=2048,
                          batches=(1, 8, 32, 64))
DSV3_DEAMOE = LayerShape("deamoe-d7168-e256-dept16x16-ish1792-ipr256-top8-shared2048-bf16",
                         d=7168, n=256, k=8, dtype="bf16", g=16, I_sh=1792,
                         I_pr=256, I_s=2048, batches=(1, 8, 32, 64))
# Skewed-routing sweep on the 7B shapes, Zipf(1.1) popularity.
ZIPF_DEAMOE = LayerShape("deamoe-7b-zipf1.1", d=2048, n=64, k=8, dtype="bf16", g=8,
                         I_sh=1024, I_pr=128, zipf=1.1, zipf_g=8,
                         batches=(1, 2, 4, 8, 16, 32, 64, 128))
ZIPF_VANILLA = LayerShape("vanilla-7b-zipf1.1", d=2048, n=64, k=8, dtype="bf16",
                          I=1152, zipf=1.1, zipf_g=8,
                          batches=(1, 2, 4, 8, 16, 32, 64, 128))

# DeaMoE form P at the budget-matched Table 1 shapes (h, r, m departments, n
# experts, k_dept, k): the 7B-class model (1024, 384, 8, 672, 4, 10) and the
# DeepSeek-V3 match (7168, 2048, 8, 864, 5, 10), plus a tiny correctness case.
TINY_FORMP = LayerShape("tiny-deamoe-p-h256-r64-dept4x4-top4-kdept2-bf16", d=256, n=16, k=4,
                        dtype="bf16", g=4, I_sh=64, form_p=True, k_dept=2, batches=(1, 5, 33))
FORMP_7B = LayerShape("deamoe-p-h1024-r384-dept8x84-top10-kdept4-bf16", d=1024, n=672, k=10,
                      dtype="bf16", g=84, I_sh=384, form_p=True, k_dept=4,
                      batches=(1, 4, 16, 64))
FORMP_DSV3 = LayerShape("deamoe-p-h7168-r2048-dept8x108-top10-kdept5-bf16", d=7168, n=864,
                        k=10, dtype="bf16", g=108, I_sh=2048, form_p=True, k_dept=5,
                        batches=(1, 4, 16, 64))
# FP8 (E4M3, one fp32 scale per row) storage of the two 2048-wide layers.
VANILLA_128E_FP8 = LayerShape("vanilla-d2048-e128-i768-top8-fp8", d=2048, n=128, k=8,
                              dtype="fp8", I=768, batches=(1, 4, 16))
DEAMOE_7B_FP8 = LayerShape("deamoe-d2048-e64-dept8x8-ish1024-ipr128-top8-fp8", d=2048,
                           n=64, k=8, dtype="fp8", g=8, I_sh=1024, I_pr=128,
                           batches=(1, 4, 8, 16))
# The DeepSeek-V3 routed experts alone (the baseline of Figure 2).
DSV3_ROUTED = LayerShape("vanilla-d7168-e256-i2048-top8-bf16", d=7168, n=256, k=8,
                         dtype="bf16", I=2048, batches=(1, 4, 16, 64))

ALL_SHAPES = (TINY_DEAMOE, TINY_VANILLA, VANILLA_128E, DEAMOE_7B, VANILLA_7B,
              DSV3_VANILLA, DSV3_DEAMOE, ZIPF_DEAMOE, ZIPF_VANILLA, TINY_FORMP, FORMP_7B,
              FORMP_DSV3, DSV3_ROUTED, VANILLA_128E_FP8, DEAMOE_7B_FP8)

WEIGHT_STD = 0.02

# Tensor ids: fixed small integers so every tensor has an independent stream.
TID_X = 1
TID_ROUTER = 2
TID_ZIPF = 3
TID_GATE, TID_UP, TID_DOWN = 10, 11, 12            # vanilla experts
TID_DGATE, TID_DUP, TID_DDOWN = 20, 21, 22         # department backbone
TID_PGATE, TID_PUP, TID_PDOWN = 30, 31, 32         # private columns
TID_SGATE, TID_SUP, TID_SDOWN = 40, 41, 42         # shared expert
TID_AGATE, TID_AUP, TID_ADOWN = 50, 51, 52         # form-P expert matrices


def stream_seed(seed: int, tensor_id: int, salt: int = 0) -> int:
    """A 63-bit seed for one tensor (splitmix64 finaliser over the triple)."""
    z = (seed * 0x9E3779B97F4A7C15 + tensor_id * 0xBF58476D1CE4E5B9
         + salt * 0x94D049BB133111EB + 0x632BE59BD9B4E019) & 0xFFFFFFFFFFFFFFFF
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    z ^= z >> 31
    return z & 0x7FFFFFFFFFFFFFFF


def _gen(device) -> torch.Generator:
    return torch.Generator(device=device)


def normal(shape, seed: int, tensor_id: int, std: float = 1.0, device="cpu",
           dtype: torch.dtype = torch.float32, salt: int = 0) -> torch.Tensor:
    """``N(0, std)`` drawn in fp32 on ``device``, then rounded to ``dtype``."""
    g = _gen(device)
    g.manual_seed(stream_seed(seed, tensor_id, salt))
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t if dtype == torch.float32 else t.to(dtype)


def storage_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32, "fp8": torch.float8_e4m3fn}[name]


E4M3_MAX = 448.0


def quantize_rows_e4m3(w: torch.Tensor):
    """Storage of fp32 weights ``[..., rows, d]`` as FP8 E4M3 codes with one
    fp32 scale per row: ``scale = max|row| / 448`` (1 for an all-zero row),
    codes = the row divided by its scale, rounded to nearest even E4M3.
    Returns ``(codes, scales)``."""
    amax = w.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (w / scale.unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX)
    return q.to(torch.float8_e4m3fn), scale.to(torch.float32)


def hidden(T: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    """Hidden states of one decode step, ``[T, d]`` fp32, ``N(0, 1)``."""
    return normal((T, d), seed, TID_X, 1.0, device)


def router(d: int, n: int, seed: int, device="cpu") -> torch.Tensor:
    """Router weights ``[n, d]`` fp32: drawn as ``[d, n]``, stored transposed."""
    w = normal((d, n), seed, TID_ROUTER, WEIGHT_STD, device)
    return w.t().contiguous()


def zipf_bias(n: int, g: int, s: float, seed: int) -> torch.Tensor:
    """Router bias ``[n]`` (fp32, host) that makes popularity roughly Zipf(s).

    Departments get a seeded rank permutation ``pi_d`` and the experts inside
    department ``j`` another permutation ``pi_j``.  With
    ``p_dept(j) ~ (1 + pi_d(j))**-s`` and ``p_in(i|j) ~ (1 + pi_j(i))**-s``
    (each normalised), expert ``e = j*g + i`` gets
    ``b_e = ln p_dept(j) + ln p_in(i|j)``.  The calibration is approximate:
    top-k over Gaussian logits plus this bias is not exactly proportional.
    """
    m = n // g
    gen = torch.Generator().manual_seed(stream_seed(seed, TID_ZIPF))
    pi_d = torch.randperm(m, generator=gen)
    w_d = torch.tensor([(1.0 + float(pi_d[j])) ** (-s) for j in range(m)], dtype=torch.float64)
    w_d /= w_d.sum()
    bias = torch.empty(n, dtype=torch.float64)
    for j in range(m):
        pi_j = torch.randperm(g, generator=gen)
        w_i = torch.tensor([(1.0 + float(pi_j[i])) ** (-s) for i in range(g)], dtype=torch.float64)
        w_i /= w_i.sum()
        for i in range(g):
            bias[j * g + i] = math.log(float(w_d[j])) + math.log(float(w_i[i]))
    return bias.to(torch.float32)


def proj(units: int, rows: int, d: int, seed: int, tensor_id: int, dtype: str,
         device="cpu") -> torch.Tensor:
    """One projection tensor ``[units, rows, d]`` in the storage dtype.

    Each unit is drawn from its own stream (salt = unit index), so a single
    unit can be regenerated without drawing the others.
    """
    out = torch.empty((units, rows, d), dtype=storage_dtype(dtype), device=device)
    for u in range(units):
        out[u].copy_(normal((rows, d), seed, tensor_id, WEIGHT_STD, device,
                            storage_dtype(dtype), salt=u + 1))
    return out


def near_identity(units: int, r: int, seed: int, tensor_id: int, dtype: str,
                  device="cpu") -> torch.Tensor:
    """``[units, r, r]`` matrices ``I + N(0, 0.02)`` in the storage dtype: the
    identity start of the form-P expert matrices (DeaMoE §3.4) with a
    perturbation standing in for training.  Drawn in fp32, rounded once."""
    out = torch.empty((units, r, r), dtype=storage_dtype(dtype), device=device)
    for u in range(units):
        out[u].copy_(near_identity_unit(u, r, seed, tensor_id, dtype, device))
    return out


def near_identity_unit(u: int, r: int, seed: int, tensor_id: int, dtype: str, device="cpu") -> torch.Tensor:
    """Unit ``u`` of ``near_identity`` alone (its own stream, salt = u + 1)."""
    a = normal((r, r), seed, tensor_id, WEIGHT_STD, device, salt=u + 1)
    a += torch.eye(r, dtype=torch.float32, device=device)
    return a.to(storage_dtype(dtype))


def proj_fp8(units: int, rows: int, d: int, seed: int, tensor_id: int, device="cpu"):
    """``proj`` in FP8 storage: the same fp32 draws, quantised per row.
    Returns ``(codes [units, rows, d], scales [units, rows])``."""
    codes = torch.empty((units, rows, d), dtype=torch.float8_e4m3fn, device=device)
    scales = torch.empty((units, rows), dtype=torch.float32, device=device)
    for u in range(units):
        w = normal((rows, d), seed, tensor_id, WEIGHT_STD, device, salt=u + 1)
        codes[u], scales[u] = quantize_rows_e4m3(w)
    return codes, scales


def make_layer(shape: LayerShape, seed: int, device="cpu", with_router: bool = True) -> dict:
    """All weights of one layer as a dict of tensors on ``device``.

    Keys: ``router`` [n,d] f32, ``bias`` [n] f32 or None; vanilla: ``gate``,
    ``up``, ``down`` [n,I,d]; DeaMoE: ``dgate``, ``dup``, ``ddown`` [m,I_sh,d]
    and ``pgate``, ``pup``, ``pdown`` [n,I_pr,d]; shared expert: ``sgate``,
    ``sup``, ``sdown`` [I_s,d] (or None); form P: the department tensors
    with r = I_sh and ``agate``, ``aup``, ``adown`` [n,r,r].  FP8 layers hold
    E4M3 codes under those keys and the row scales under ``<key>_sc``.
    """
    s = shape
    L: dict = {"shape": s}

    def put(key, units, rows, tid, squeeze=False):
        if s.dtype == "fp8":
            codes, scales = proj_fp8(units, rows, s.d, seed, tid, device)
            L[key], L[key + "_sc"] = (codes[0], scales[0]) if squeeze else (codes, scales)
        else:
            w = proj(units, rows, s.d, seed, tid, s.dtype, device)
            L[key] = w[0] if squeeze else w

    if with_router:
        L["router"] = router(s.d, s.n, seed, device)
        L["bias"] = (zipf_bias(s.n, s.zipf_g, s.zipf, seed).to(device)
                     if s.zipf > 0 else None)
    if s.I > 0:
        put("gate", s.n, s.I, TID_GATE)
        put("up", s.n, s.I, TID_UP)
        put("down", s.n, s.I, TID_DOWN)
    if s.I_sh > 0:
        put("dgate", s.m, s.I_sh, TID_DGATE)
        put("dup", s.m, s.I_sh, TID_DUP)
        put("ddown", s.m, s.I_sh, TID_DDOWN)
    if s.form_p:
        L["agate"] = near_identity(s.n, s.I_sh, seed, TID_AGATE, s.dtype, device)
        L["aup"] = near_identity(s.n, s.I_sh, seed, TID_AUP, s.dtype, device)
        L["adown"] = near_identity(s.n, s.I_sh, seed, TID_ADOWN, s.dtype, device)
    if s.I_pr > 0:
        put("pgate", s.n, s.I_pr, TID_PGATE)
        put("pup", s.n, s.I_pr, TID_PUP)
        put("pdown", s.n, s.I_pr, TID_PDOWN)
    if s.I_s > 0:
        put("sgate", 1, s.I_s, TID_SGATE, squeeze=True)
        put("sup", 1, s.I_s, TID_SUP, squeeze=True)
        put("sdown", 1, s.I_s, TID_SDOWN, squeeze=True)
    else:
        L["sgate"] = L["sup"] = L["sdown"] = None
    return L
