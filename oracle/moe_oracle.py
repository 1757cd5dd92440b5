"""Plain CPU oracle for the MoE / DeaMoE small-batch decode layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may call it.  It shares no code, table or helper with the CUDA
path; both sides take their inputs from ``moe_decode_layer_fp32_gb300.synth``.

Everything is fp64 numpy, written as the plain definition of what the layer
computes, per token and per selected expert, with no department reuse, no
blocking and no fusion.  Weights arrive in their storage dtype (bf16 or fp32)
and are decoded exactly.

Sources (cited by title and section):

* [DeaMoE] "DeaMoE: Efficient MoE Structure for Fast Small-Batch Decoding"
  (arXiv 2608.14385v1): §2.1 eqs. (1)-(3) (SwiGLU expert, top-k router,
  weighted combine), §3.1 eq. (4) (department structure, "form P"), §3.2
  (two-stage routing), §3.3 with Table 1 and Figure 2 (budget matching and the
  expected-loading curve), §3.4 (SiLU at all three interfaces, identity init).
* [DSMoE] "DeepSeekMoE Guide: Fine-Grained Experts & Dynamic Routing",
  section "Mathematical Formulation of the DeepSeekMoE Forward Pass" (shared
  expert with weight 1; routing bias used for selection only; softmax over
  the selected affinities).
* [DSMoE-ALF] the same guide, section "Algorithmic Mechanics: Auxiliary-Loss-Free
  Dynamic Load Balancing" (step 4 of its routing loop: the sign update of the
  router bias; its part 2: the proportional update; its part 3: the imbalance
  ratio).
* [MoE-inf] "MoE inference engineering, clearly explained", sections "How a
  batch becomes expert-specific matrices" (dispatch / combine) and "Local MoE
  execution pipeline" (permutation with an inverse map).

Readings where the pages are silent:

* R1 routing decision: keys are fp32 (the router is fp32); the oracle rounds
  its fp64 logit to fp32, adds the fp32 bias in fp32, and orders by key
  descending, equal keys -> lower expert index first.
* R2 routing weights: ``p = scale * softmax(logits[selected])`` over the k
  selected *unbiased* logits, in fp64.
* R3 form C (the shapes every measured layer uses): expert i of department
  j = i // g is a SwiGLU FFN whose intermediate is department j's shared rows
  followed by expert i's private rows.
* R4 the shared expert has weight 1 and no gate; the layer output excludes the
  residual ``u_t`` of the [DSMoE] formula.
* R5 form P (eq. 4) uses sigma = SiLU at all three interfaces ([DeaMoE] §3.4).
* R6 expert e belongs to department floor(e / g).
* R7 group-limited top-k: a department's score is its best expert key.
* R8 strict coverage: the replaced expert is the lowest-ranked one whose
  department keeps another selected expert (otherwise the coverage would not
  grow), and the uncovered departments are among the k_dept kept ones.
* R9 bias update: the target load of an expert is the batch's mean load,
  (sum of the expert token counts) / n; the bias is fp32 state, updated once
  per call from fp64 arithmetic rounded to fp32 once.  With no routed token
  the imbalance ratio (0 / 0) is reported as 0 and no bias moves.
* R10 FP8 weights: E4M3 codes with one fp32 scale per weight row (a row of a
  gate, up or down matrix, i.e. one intermediate index of a unit); the pages
  give the format's size only.
"""

from __future__ import annotations

from math import comb

import numpy as np

# ---------------------------------------------------------------------------
# Scalars and decoding
# ---------------------------------------------------------------------------


def bf16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns: the top half of an fp32 word."""
    u32 = u16.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def e4m3_bits_to_f64(u8: np.ndarray) -> np.ndarray:
    """Exact value of FP8 E4M3 codes (the "fn" layout: 1 sign bit, 4 exponent
    bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN).
    Normal: (-1)^s 2^(e-7) (1 + m/8); subnormal (e = 0): (-1)^s 2^-6 (m/8)."""
    b = np.asarray(u8, dtype=np.uint8).astype(np.int64)
    sgn = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64)))
    out = sgn * mag
    return np.where((b & 0x7F) == 0x7F, np.nan, out)


def dequant_rows_e4m3(codes, row_scale) -> np.ndarray:
    """FP8 weights with one fp32 scale per row (R10): ``w[..., r, c] =
    row_scale[..., r] * e4m3(codes[..., r, c])``, exactly, in fp64."""
    try:
        import torch
        if isinstance(codes, torch.Tensor):
            codes = codes.detach().cpu().contiguous().view(torch.uint8).numpy()
        if isinstance(row_scale, torch.Tensor):
            row_scale = row_scale.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    vals = e4m3_bits_to_f64(codes)
    return vals * np.asarray(row_scale, np.float64)[..., None]


def to_f64(w) -> np.ndarray:
    """Decode a weight tensor (torch bf16/fp32 or numpy) to fp64, exactly."""
    try:
        import torch
        if isinstance(w, torch.Tensor):
            w = w.detach().cpu().contiguous()
            if w.dtype == torch.bfloat16:
                return bf16_bits_to_f64(w.view(torch.int16).numpy().view(np.uint16))
            return w.numpy().astype(np.float64)
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    return np.asarray(w, dtype=np.float64)


def silu(z):
    """SiLU(z) = z * sigmoid(z) = z / (1 + e^-z)  ([DeaMoE] §2.1 gate projection)."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


# ---------------------------------------------------------------------------
# Router: [DeaMoE] §2.1 eqs. (2)-(3); [DSMoE] routing-bias formulation
# ---------------------------------------------------------------------------


def router_logits(x, w_router) -> np.ndarray:
    """``l[t, e] = <x_t, W_r[e, :]>`` in fp64: the ``W_r x`` of eq. (2)."""
    return to_f64(x) @ to_f64(w_router).T


def route(x, w_router, k: int, bias=None, scale: float = 1.0):
    """Top-k routing of eq. (2) with the weights of eq. (3).

    Returns ``(idx [T,k] int32, p [T,k] float64, info)``.  ``idx[t, 0]`` is the
    best expert.  ``info`` holds the fp64 logits, the fp32 keys and, per token,
    the fp64 gap between the k-th and (k+1)-th key and the smallest gap between
    adjacent selected keys (used to certify near-ties when comparing with a
    device that sums in a different order).
    """
    l64 = router_logits(x, w_router)
    T, n = l64.shape
    if not 1 <= k <= n:
        raise ValueError("need 1 <= k <= n")
    b32 = np.zeros(n, np.float32) if bias is None else to_f64(bias).astype(np.float32)
    key32 = (l64.astype(np.float32) + b32[None, :]).astype(np.float32)   # R1
    key64 = l64 + b32.astype(np.float64)[None, :]
    idx = np.empty((T, k), np.int32)
    p = np.empty((T, k), np.float64)
    gap_boundary = np.full(T, np.inf)
    gap_adjacent = np.full(T, np.inf)
    for t in range(T):
        order = sorted(range(n), key=lambda e: (-float(key32[t, e]), e))
        sel = order[:k]
        idx[t] = sel
        ls = l64[t, sel]                                   # unbiased affinities (R2)
        ex = np.exp(ls - ls.max())
        p[t] = scale * ex / ex.sum()
        ks = [key64[t, e] for e in order]
        if k < n:
            gap_boundary[t] = ks[k - 1] - ks[k]
        if k > 1:
            gap_adjacent[t] = min(ks[i] - ks[i + 1] for i in range(k - 1))
    info = {"logits": l64, "key32": key32, "key64": key64,
            "gap_boundary": gap_boundary, "gap_adjacent": gap_adjacent}
    return idx, p, info


def route_grouped(x, w_router, k: int, g: int, k_dept: int, bias=None, scale: float = 1.0,
                  strict: bool = False):
    """Group-limited top-k of [DeaMoE] §3.3 ("we use group top-k routing to cap
    the activated FLOPs per token associated with department matrices"), with
    the strict-coverage variant of its appendix ablation.

    Per token, with the fp32 keys of ``route`` (R1):

    1. department j's score is its best expert key, ``max_{e in j} key[e]``
       (R7: the pages do not define the score);
    2. the k_dept departments with the best scores are kept (score descending,
       equal scores -> lower department first);
    3. the top-k of the experts of the kept departments, as in ``route``;
    4. strict only (R8): while the selection covers fewer than k_dept
       departments, the best expert (largest key, lower index on ties) of the
       best-scored uncovered kept department replaces the lowest-ranked
       selected expert among those whose department holds another selected
       expert; the selection is then re-ordered by key;
    5. weights: ``scale * softmax`` over the selected unbiased logits (R2).

    Returns ``(idx [T,k] int32, p [T,k] float64, info)`` like ``route``; info
    adds the kept departments ``kept [T,k_dept]`` and the fp64 department
    scores ``dscore64``.
    """
    l64 = router_logits(x, w_router)
    T, n = l64.shape
    if g < 1 or n % g:
        raise ValueError("need g >= 1 dividing n")
    m = n // g
    if not 1 <= k_dept <= m or not 1 <= k <= k_dept * g:
        raise ValueError("need 1 <= k_dept <= n/g and 1 <= k <= k_dept * g")
    if strict and k < k_dept:
        raise ValueError("strict coverage needs k >= k_dept")
    b32 = np.zeros(n, np.float32) if bias is None else to_f64(bias).astype(np.float32)
    key32 = (l64.astype(np.float32) + b32[None, :]).astype(np.float32)
    key64 = l64 + b32.astype(np.float64)[None, :]
    idx = np.empty((T, k), np.int32)
    p = np.empty((T, k), np.float64)
    kept_all = np.empty((T, k_dept), np.int32)
    dscore64 = np.empty((T, m))
    for t in range(T):
        rank = lambda e: (-float(key32[t, e]), e)                      # noqa: E731
        score = [max(float(key32[t, e]) for e in range(j * g, (j + 1) * g)) for j in range(m)]
        dscore64[t] = [max(key64[t, e] for e in range(j * g, (j + 1) * g)) for j in range(m)]
        kept = sorted(range(m), key=lambda j: (-score[j], j))[:k_dept]
        kept_all[t] = kept
        cand = [e for j in kept for e in range(j * g, (j + 1) * g)]
        sel = sorted(cand, key=rank)[:k]
        if strict:
            while len({e // g for e in sel}) < k_dept:
                covered = {e // g for e in sel}
                j_new = min((j for j in kept if j not in covered), key=lambda j: (-score[j], j))
                e_new = min(range(j_new * g, (j_new + 1) * g), key=rank)
                shared = [e for e in sel if sum(1 for f in sel if f // g == e // g) > 1]
                e_out = max(shared, key=rank)                           # lowest ranked
                sel = sorted([e for e in sel if e != e_out] + [e_new], key=rank)
        idx[t] = sel
        ls = l64[t, sel]
        ex = np.exp(ls - ls.max())
        p[t] = scale * ex / ex.sum()
    info = {"logits": l64, "key32": key32, "key64": key64, "kept": kept_all, "dscore64": dscore64}
    return idx, p, info


# ---------------------------------------------------------------------------
# Router-bias load balancing: [DSMoE-ALF]
# ---------------------------------------------------------------------------

BIAS_SIGN = 0           # b_i -/+ gamma when expert i is over / under its target
BIAS_PROPORTIONAL = 1   # b_i + gamma * (target - tokens_i)


def bias_update(counts, bias, gamma: float, rule: int = BIAS_SIGN) -> np.ndarray:
    """One gradient-free update of the selection-only router bias from the
    tokens each expert received ([DSMoE-ALF] step 4 and part 2).

    ``counts[i]`` is the number of tokens routed to expert i in the batch,
    ``bias`` the fp32 bias before the update.  The target is the mean load
    sum(counts) / n (R9).  Sign rule: an expert above its target loses gamma,
    one below it gains gamma, one exactly on it keeps its bias.  Proportional
    rule: ``b_i + gamma * (target - counts_i)``.  Returns the new fp32 bias.
    """
    c = [int(v) for v in np.asarray(counts).reshape(-1)]
    b = np.asarray(bias, np.float32).reshape(-1)
    n = len(c)
    if b.shape[0] != n:
        raise ValueError("counts and bias differ in length")
    total = sum(c)
    out = np.empty(n, np.float32)
    for i in range(n):
        bi = float(b[i])
        if rule == BIAS_SIGN:
            # compare counts_i with total / n exactly: counts_i * n vs total
            if c[i] * n > total:
                bi = bi - float(gamma)
            elif c[i] * n < total:
                bi = bi + float(gamma)
        elif rule == BIAS_PROPORTIONAL:
            bi = bi + float(gamma) * (total / n - c[i])
        else:
            raise ValueError("unknown rule")
        out[i] = np.float32(bi)
    return out


def imbalance_ratio(counts) -> float:
    """[DSMoE-ALF] part 3: max_j tokens_j / ((1/n) sum_j tokens_j); 0 when no
    token was routed (R9)."""
    c = [int(v) for v in np.asarray(counts).reshape(-1)]
    total = sum(c)
    if total == 0:
        return 0.0
    return max(c) / (total / len(c))


# ---------------------------------------------------------------------------
# Dispatch lists: [MoE-inf] "How a batch becomes expert-specific matrices";
# departments X^j of [DeaMoE] §3.2.
# ---------------------------------------------------------------------------


def dispatch(idx, p, n: int, g: int = 1) -> dict:
    """Group the T*k assignments by expert and the tokens by department.

    Canonical order: ascending expert (department) id, then ascending token
    id.  A token appears once in X^j even when it picked several experts of
    department j; its department weight is the sum of those experts' routing
    weights, added in slot order.
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    assign = []                                  # (expert, token, slot, weight)
    for t in range(T):
        if len(set(int(e) for e in idx[t])) != k:
            raise ValueError(f"token {t} selects an expert twice")
        for s in range(k):
            e = int(idx[t, s])
            if not 0 <= e < n:
                raise ValueError("expert index out of range")
            assign.append((e, t, s, float(p[t, s])))
    assign.sort(key=lambda a: (a[0], a[1]))
    exp_count = np.zeros(n, np.int32)
    for a in assign:
        exp_count[a[0]] += 1
    exp_off = np.zeros(n + 1, np.int32)
    exp_off[1:] = np.cumsum(exp_count)
    asg_tok = np.array([a[1] for a in assign], np.int32)
    asg_slot = np.array([a[2] for a in assign], np.int32)
    asg_w = np.array([a[3] for a in assign], np.float64)
    tok_asg = np.empty((T, k), np.int32)
    for pos, a in enumerate(assign):
        tok_asg[a[1], a[2]] = pos
    active_experts = np.array([e for e in range(n) if exp_count[e] > 0], np.int32)

    out = {"exp_count": exp_count, "exp_off": exp_off, "asg_tok": asg_tok,
           "asg_slot": asg_slot, "asg_w": asg_w, "tok_asg": tok_asg,
           "active_experts": active_experts}
    if g > 1:
        if n % g:
            raise ValueError("n must be a multiple of g")
        m = n // g
        dept_tok, dept_w, dept_count = [], [], np.zeros(m, np.int32)
        tok_dpos = np.full((T, m), -1, np.int32)
        for j in range(m):
            for t in range(T):
                slots = [s for s in range(k) if int(idx[t, s]) // g == j]   # R6
                if not slots:
                    continue
                w = 0.0
                for s in slots:
                    w += float(p[t, s])
                tok_dpos[t, j] = len(dept_tok)
                dept_tok.append(t)
                dept_w.append(w)
                dept_count[j] += 1
        dept_off = np.zeros(m + 1, np.int32)
        dept_off[1:] = np.cumsum(dept_count)
        out.update({"dept_count": dept_count, "dept_off": dept_off,
                    "dept_tok": np.array(dept_tok, np.int32),
                    "dept_w": np.array(dept_w, np.float64), "tok_dpos": tok_dpos,
                    "active_depts": np.array([j for j in range(m) if dept_count[j] > 0],
                                             np.int32)})
    return out


# ---------------------------------------------------------------------------
# Experts
# ---------------------------------------------------------------------------


def swiglu_expert(x_t, w_gate, w_up, w_down) -> np.ndarray:
    """Eq. (1): ``MoE_i(x) = d_i(g_i(x) * u_i(x))`` with
    ``g_i(x) = SiLU(W_gate x)``, ``u_i(x) = W_up x`` and
    ``d_i(v) = (W_down)^T v``; every W has shape ``[I, d]`` (hffn x h)."""
    x_t = to_f64(x_t)
    g = to_f64(w_gate) @ x_t
    u = to_f64(w_up) @ x_t
    return to_f64(w_down).T @ (silu(g) * u)


class Units:
    """Lazy fp64 access to one projection tensor ``[units, rows, d]``."""

    def __init__(self, tensor):
        self.t = tensor
        self.cache: dict = {}

    def __call__(self, u: int) -> np.ndarray:
        if u not in self.cache:
            self.cache[u] = to_f64(self.t[u])
        return self.cache[u]


def vanilla_layer(x, idx, p, gate, up, down, shared=None) -> np.ndarray:
    """Eq. (3) plus an optional always-on shared expert ([DSMoE]):
    ``y_t = sum_s p[t,s] * MoE_{idx[t,s]}(x_t) + FFN_shared(x_t)``.

    ``gate``/``up``/``down`` are ``[n, I, d]`` tensors; ``shared`` is
    ``(gate, up, down)`` with ``[I_s, d]`` each, or None.
    """
    xs = to_f64(x)
    T, d = xs.shape
    G, U, D = Units(gate), Units(up), Units(down)
    sh = None if shared is None else tuple(to_f64(w) for w in shared)
    y = np.zeros((T, d))
    for t in range(T):
        for s in range(idx.shape[1]):
            e = int(idx[t, s])
            y[t] += p[t, s] * swiglu_expert(xs[t], G(e), U(e), D(e))
        if sh is not None:
            y[t] += swiglu_expert(xs[t], *sh)                         # R4
    return y


def deamoe_expert_c(e: int, g: int, dept, priv):
    """Form C (R3): expert e's projections are department floor(e/g)'s shared
    rows stacked on top of expert e's private rows."""
    j = e // g
    w = []
    for a in range(3):
        parts = [dept[a](j)]
        if priv is not None:
            parts.append(priv[a](e))
        w.append(np.concatenate(parts, axis=0))
    return w


def deamoe_layer_c(x, idx, p, g: int, dgate, dup, ddown, pgate=None, pup=None,
                   pdown=None, shared=None) -> np.ndarray:
    """DeaMoE form C layer evaluated literally with eqs. (1) and (3): each
    selected expert is run on its own token with its materialised weights.
    No department reuse (that is the two-stage fast path, not the definition)."""
    xs = to_f64(x)
    T, d = xs.shape
    dept = (Units(dgate), Units(dup), Units(ddown))
    priv = None if pgate is None else (Units(pgate), Units(pup), Units(pdown))
    sh = None if shared is None else tuple(to_f64(w) for w in shared)
    y = np.zeros((T, d))
    for t in range(T):
        for s in range(idx.shape[1]):
            e = int(idx[t, s])
            wg, wu, wd = deamoe_expert_c(e, g, dept, priv)
            y[t] += p[t, s] * swiglu_expert(xs[t], wg, wu, wd)
        if sh is not None:
            y[t] += swiglu_expert(xs[t], *sh)
    return y


def deamoe_expert_p(x_t, wg, wu, wd, ag, au, ad) -> np.ndarray:
    """Form P, eq. (4) of [DeaMoE] §3.1 with sigma = SiLU (R5):
    ``g^ = SiLU(A_g SiLU(W_g x))``, ``u^ = A_u SiLU(W_u x)``,
    ``d^(v) = W_d^T SiLU(A_d^T v)`` and ``DeaMoE_i(x) = d^(g^ * u^)``.
    ``W_*`` are the department's ``[r, h]`` matrices, ``A_*`` expert i's
    ``[r, r]`` private matrices."""
    x_t = to_f64(x_t)
    gh = silu(to_f64(ag) @ silu(to_f64(wg) @ x_t))
    uh = to_f64(au) @ silu(to_f64(wu) @ x_t)
    z = silu(to_f64(ad).T @ (gh * uh))
    return to_f64(wd).T @ z


def deamoe_layer_p(x, idx, p, g: int, dgate, dup, ddown, agate, aup, adown) -> np.ndarray:
    """Form P layer: eq. (3) over eq. (4) experts, per token and expert."""
    xs = to_f64(x)
    T, d = xs.shape
    y = np.zeros((T, d))
    for t in range(T):
        for s in range(idx.shape[1]):
            e = int(idx[t, s])
            j = e // g
            y[t] += p[t, s] * deamoe_expert_p(xs[t], dgate[j], dup[j], ddown[j],
                                              agate[e], aup[e], adown[e])
    return y


# ---------------------------------------------------------------------------
# Byte accounting ([DeaMoE] §3.3, Figure 2) and budget matching (Table 1)
# ---------------------------------------------------------------------------


def unique_bytes_vanilla(d, n, I, I_s, A_e, bw) -> int:
    """Weights one vanilla step must read: the fp32 router, the shared expert
    and every active expert's three ``[I, d]`` matrices."""
    return 4 * d * n + bw * 3 * d * (A_e * I + I_s)


def unique_bytes_deamoe_c(d, n, I_sh, I_pr, I_s, A_d, A_e, bw) -> int:
    """Form C: each active department's backbone once, plus each active
    expert's private rows, the shared expert and the fp32 router."""
    return 4 * d * n + bw * 3 * d * (A_d * I_sh + A_e * I_pr + I_s)


def unique_bytes_deamoe_p(h, n, r, A_d, A_e, bw) -> int:
    """Form P: each active department's ``3 h r`` backbone once and each active
    expert's three ``r x r`` A-matrices, plus the fp32 router."""
    return 4 * h * n + bw * (A_d * 3 * h * r + A_e * 3 * r * r)


def expected_active_experts(n, k, T) -> float:
    """Expected distinct experts hit by T tokens that each pick k of n
    uniformly without replacement: ``n (1 - (1 - k/n)^T)``."""
    return n * (1.0 - (1.0 - k / n) ** T)


def expected_active_depts(n, k, g, T) -> float:
    """Expected distinct departments (m = n/g) hit under the same model: a
    token misses department j with probability ``C(n-g, k) / C(n, k)``."""
    m = n // g
    return m * (1.0 - (comb(n - g, k) / comb(n, k)) ** T)


def loading_ratio_formp(h, r, n_base, k_base, n, m, k, T, with_router=False) -> float:
    """Expected weight loaded per step, DeaMoE form P over its baseline
    (the quantity plotted in Figure 2), in element counts."""
    g = n // m
    base = expected_active_experts(n_base, k_base, T) * 3 * h * r
    dea = (expected_active_depts(n, k, g, T) * 3 * h * r
           + expected_active_experts(n, k, T) * 3 * r * r)
    if with_router:
        base += h * n_base
        dea += h * n
    return dea / base


def table1_ratios(h, r, n_base, k_base, m, n, k_dept, k) -> tuple:
    """(FLOPs ratio, params ratio) of a budget-matched DeaMoE config over its
    baseline, router included ([DeaMoE] §3.3, Table 1)."""
    params_base = n_base * 3 * h * r + h * n_base
    params_dea = m * 3 * h * r + n * 3 * r * r + h * n
    flops_base = k_base * 3 * h * r + h * n_base
    flops_dea = k_dept * 3 * h * r + k * 3 * r * r + h * n
    return flops_dea / flops_base, params_dea / params_base
