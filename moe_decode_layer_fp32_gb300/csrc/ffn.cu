// Expert FFN of the decode layer as one weight-streaming pass (CUDA-core path).
//
// What it computes: for every active unit u (the shared expert, a department
// backbone, or an expert's own rows) and its gathered tokens X_u,
//     Y_u = W_down^T ( SiLU(W_gate X_u) * (W_up X_u) ),
// the SwiGLU expert of "DeaMoE: Efficient MoE Structure for Fast Small-Batch
// Decoding" §2.1 eq. (1), with W_down stored in the paper's [hffn, h] shape.
// A department backbone runs once over its token set X^j and its rows are
// scaled by the department token weight, which is the two-stage routing of
// DeaMoE §3.2 specialised to form C (shared rows are common to every expert
// of the department, so by linearity sum_i p_i W^T h = W^T h * sum_i p_i).
//
// How: the intermediate rows of all active units form one row space that is
// split evenly over CPS CTAs per SM.  In each CTA a producer warp streams the
// CTA's rows (gate, up, then down; every row is contiguous) from HBM into a
// shared-memory ring with bulk copies (cp.async.bulk + mbarrier transaction
// counts).  Consumer warps own fixed 8-column chunks of the hidden dimension:
// gate/up dot products use packed fp32x2 FMAs, are reduced across the warp and
// then across warps with shared atomics; the SwiGLU is applied in shared
// memory; the down projection accumulates each thread's columns in registers.
// The CTA's partial output is added into the output with vector atomics.
#include <cuda_bf16.h>

#include "../../include/moe_decode.h"
#include "kernels.h"
#include "local_route.cuh"
#include "stream_core.cuh"

namespace moe {

namespace {

constexpr int kStageBytes = 16384;   // one ring slot
#ifndef MOE_ROUTE_PDL
#define MOE_ROUTE_PDL 1
#endif
constexpr int kRingBytesPerSM = 10 * kStageBytes;  // weights in flight per SM
constexpr int kSegMax = 256;         // rows per segment (gate/up/h buffers)


// Shared-memory carve-up (after the ring).  The unit table is sized at launch.
template <int NS>
struct FfnSmem {
    uint64_t full[NS];
    uint64_t empty[NS];
    float gu[2][kSegMax * kMT];       // gate / up pre-activations of the segment
    float h[kSegMax * kMT];           // SwiGLU output (times the token weight)
    int cls_units[3];
    int cls_groups[3];
    int cls_off[3];                   // offset of the class's records in `units`
    int cls_cost[3];                  // cost units of the class (see cost_units)
    // per unit: {weight index, first token entry, tokens, inclusive group prefix}
    int4 units[1];
};

// A segment: rows [row0, row0+nrows) of one token group of one unit.
struct Seg {
    int cls, q, grp, row0, nrows;
};

// Next segment of [r, r_end) in the class / unit / group / row order.
template <int NS>
__device__ __forceinline__ bool next_seg(const FfnArgs& a, const FfnSmem<NS>& sm, long long& r,
                                         long long r_end, Seg& s) {
    if (r >= r_end) return false;
    long long base = 0;
    int c = 0;
    while (c < a.ncls - 1 && r >= base + (long long)a.cls[c].rows * sm.cls_groups[c]) {
        base += (long long)a.cls[c].rows * sm.cls_groups[c];
        ++c;
    }
    const int rows = a.cls[c].rows;
    const int rel = (int)(r - base);       // row spaces stay far below 2^31
    const int vg = rel / rows;
    const int rin = rel - vg * rows;
    const int4* u = sm.units + sm.cls_off[c];
    int lo = 0, hi = sm.cls_units[c] - 1;  // first q whose group prefix exceeds vg
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (u[mid].w > vg) hi = mid; else lo = mid + 1;
    }
    s.cls = c;
    s.q = lo;
    s.grp = vg - (lo > 0 ? u[lo - 1].w : 0);
    s.row0 = rin;
    long long n = rows - rin;
    if (n > r_end - r) n = r_end - r;
    if (n > kSegMax) n = kSegMax;
    s.nrows = (int)n;
    r += n;
    return true;
}

// Work-balanced split of the row space.  A row costs what its token group's
// code path costs: groups of one or two tokens run the narrow register tiles,
// groups of three or four the wide one, which was measured about 1.5x slower
// per row (the weight stream is the same; the per-token dot products,
// reductions and accumulations are not).  Each token group also costs
// kSegCost once, at its first row: a CTA whose range starts a new group pays
// a segment switch (activation loads, the SwiGLU barrier, a drained ring).
// A unit of t tokens costs rows * cost_units(t) + groups * kSegCost; every
// class keeps the exclusive prefix of its units' costs (cpre) next to the
// unit records.
// One warp: exclusive prefix of the records' unit costs into cpre; returns
// the class total (on every lane).
__device__ __forceinline__ int class_cost_prefix_warp(const int4* u, int nu, int rows, int* cpre) {
    const int lane = threadIdx.x & 31;
    int carry = 0;
    for (int b = 0; b < nu; b += 32) {
        const int q = b + lane;
        const int c = q < nu ? unit_cost(u[q].z, rows) : 0;
        int inc = c;
        __syncwarp();
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += t;
        }
        if (q < nu) cpre[q] = carry + inc - c;
        carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    return carry;
}

template <int NS>
__device__ __forceinline__ long long split_total_cost(const FfnArgs& a, const FfnSmem<NS>& sm) {
    long long tot = 0;
    for (int c = 0; c < a.ncls; ++c) tot += sm.cls_cost[c];
    return tot;
}

// Row-space position whose cost prefix is C (rounded down to a whole row).
// 32-bit arithmetic throughout (the caller keeps the total cost below 2^31).
template <int NS>
__device__ __forceinline__ int split_row_at(const FfnArgs& a, const FfnSmem<NS>& sm, const int* cpre_all,
                                            int C) {
    int row_base = 0;
    for (int c = 0; c < a.ncls; ++c) {
        const int rows = a.cls[c].rows;
        const int nu = sm.cls_units[c];
        const int4* u = sm.units + sm.cls_off[c];
        const int* cpre = cpre_all + sm.cls_off[c];
        const int cc = sm.cls_cost[c];
        if (C < cc || c == a.ncls - 1) {
            if (nu == 0) return row_base;
            if (C >= cc) return row_base + rows * sm.cls_groups[c];
            int lo = 0, hi = nu - 1;    // last q with cpre[q] <= C
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (cpre[mid] <= C) lo = mid; else hi = mid - 1;
            }
            const int t = u[lo].z;
            const int G = (t + kMT - 1) / kMT;
            const int Cq = C - cpre[lo];
            const int full = rows * group_cost(kMT) + kSegCost;   // every group but the last is full
            const int g = min(Cq / full, G - 1);
            const int mg = min(kMT, t - g * kMT);
            const int i = min(max(Cq - g * full - kSegCost, 0) / group_cost(mg), rows);
            const int gpre = lo > 0 ? u[lo - 1].w : 0;
            return row_base + (gpre + g) * rows + i;
        }
        C -= cc;
        row_base += rows * sm.cls_groups[c];
    }
    return row_base;
}

// Tokens of a group: token id, weight and output row (ROWS or ACCUM mode).
__device__ __forceinline__ int group_tokens(const FfnArgs& a, const int4 rec, int kind, int grp,
                                            int (&tok)[kMT], float (&wt)[kMT], int (&orow)[kMT]) {
    const int first = grp * kMT;
    const int mg = min(kMT, rec.z - first);
#pragma unroll
    for (int i = 0; i < kMT; ++i) {
        tok[i] = 0;
        wt[i] = 0.0f;
        orow[i] = 0;
        if (i < mg) {
            const int p = rec.y + first + i;
            int t;
            float w;
            int row;
            if (kind == kUnitShared) {
                t = p;
                w = 1.0f;
                row = a.rows_shared_base + p;
            } else if (kind == kUnitDept) {
                t = a.ws.dept_tok[p];
                w = a.ws.dept_w[p];
                row = a.rows_dept_base + p;
            } else {
                t = a.ws.asg_tok[p];
                w = a.ws.asg_w[p];
                row = p;
            }
            // a token id outside [0, T) (a workspace the dispatch did not
            // write for this step) is reported, never used as an address
            if ((unsigned)t >= (unsigned)a.T) {
                set_status(a.ws.status, kDevErrRouting);
                t = 0;
                w = 0.0f;
            }
            tok[i] = t;
            wt[i] = w;
            orow[i] = a.out_mode == MOE_OUT_ACCUM ? t : row;
        }
    }
    return mg;
}


// ONE: a one-token step on the in-CTA routing path
// (the host launches it only then).  CTA 0 builds the workspace lists as
// usual; the other CTAs take the unit records straight from the selection
// (local_tables_one_token), every CTA streams an equal share of the rows, and
// the consumers run the one-token register tile only.  A separate
// instantiation, so that the general kernel's code is not touched by it.
template <typename WT, int NCW, int CH, int RMAX, int CPS, bool ONE>
__global__ void __launch_bounds__((NCW + 1) * 32, CPS) ffn_stream_kernel(FfnArgs a) {
    using K = Ffn<WT, NCW, CH, RMAX>;
    constexpr int NS = kRingBytesPerSM / kStageBytes / CPS;   // ring slots per CTA
    constexpr int kNT = (NCW + 1) * 32;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char* ring = smem_raw;
    FfnSmem<NS>& sm = *reinterpret_cast<FfnSmem<NS>*>(smem_raw + (size_t)NS * kStageBytes);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], NCW);
        }
        mbar_init_fence();
    }
    for (int i = tid; i < 2 * kSegMax * kMT; i += kNT) (&sm.gu[0][0])[i] = 0.0f;
    // after the unit records: their cost prefixes, then the local routing state
    int cap = 0;
    for (int c = 0; c < a.ncls; ++c) cap += class_capacity(a.cls[c], a.n, a.g);
    int* cpre = reinterpret_cast<int*>(sm.units + cap);
    LocalRoute lr = {};
    if (a.local_route) {
        lr = local_route_at(reinterpret_cast<unsigned char*>(sm.units + cap) + align16(4 * (size_t)cap), a.T,
                            a.n, a.k, a.g, NCW + 1);
        for (int i = tid; i < a.n * lr.W; i += kNT) lr.emask[i] = 0u;
        if (tid == 0) {
            int off = 0;
            for (int c = 0; c < a.ncls; ++c) {
                sm.cls_off[c] = off;
                off += class_capacity(a.cls[c], a.n, a.g);
            }
        }
        __syncthreads();
    }

    // The next layer's routing grid (a programmatic dependent) may take SMs
    // as this grid's CTAs finish; it waits for this grid's completion.
    if (MOE_ROUTE_PDL) pdl_allow_dependents();
    // Everything below reads what the routing / dispatch kernel wrote.
    pdl_wait_primary();
    // The tensor-core kernel ran first and took the step: nothing to do.
    if (a.tc_first && *reinterpret_cast<volatile uint32_t*>(a.ws.sync + 1) == 2u) return;

    // ---- unit table: built here from the router logits (whole-layer path),
    // the dispatch's per-unit records (one coalesced load), or, when units
    // with more than max_tokens tokens go to the tensor-core kernel, the
    // records of the remaining units with their own group prefix ----
    if (a.local_route) {
        const bool writer = blockIdx.x == 0;
        local_topk<kNT>(a, lr, writer);
        const UnitTableView view = {sm.units, sm.cls_off, sm.cls_units, sm.cls_groups, sm.cls_cost, cpre};
        if constexpr (ONE) {
            if (!writer) local_tables_one_token<kNT>(a, view, lr);
            else local_tables<kNT, kMT, true>(a, view, lr, writer);
        } else {
            local_tables<kNT, kMT, true>(a, view, lr, writer);
        }
    } else if (a.max_tokens >= a.T) {
        int off = 0;
        for (int c = 0; c < a.ncls; ++c) {
            const UnitClass& uc = a.cls[c];
            const int cap = class_capacity(uc, a.n, a.g);
            if (uc.kind == kUnitShared) {
                if (tid == 0) sm.units[off] = make_int4(0, 0, a.T, (a.T + kMT - 1) / kMT);
            } else {
                const int4* src = uc.kind == kUnitDept ? a.ws.dept_units : a.ws.exp_units;
                for (int q = tid; q < cap; q += kNT) sm.units[off + q] = src[q];
            }
            if (tid == 0) {
                sm.cls_units[c] = uc.kind == kUnitShared ? 1
                                  : uc.kind == kUnitDept ? a.ws.counts[1] : a.ws.counts[0];
                sm.cls_off[c] = off;
            }
            off += cap;
        }
        __syncthreads();
        if (warp < a.ncls) {
            const int nu = sm.cls_units[warp];
            const int tot = class_cost_prefix_warp(sm.units + sm.cls_off[warp], nu, a.cls[warp].rows,
                                                   cpre + sm.cls_off[warp]);
            if (lane == 0) {
                sm.cls_groups[warp] = nu > 0 ? sm.units[sm.cls_off[warp] + nu - 1].w : 0;
                sm.cls_cost[warp] = tot;
            }
        }
        __syncthreads();
    } else {
        if (warp == 0) {
            int off = 0;
            for (int c = 0; c < a.ncls; ++c) {
                const UnitClass& uc = a.cls[c];
                int kept, groups;
                if (uc.kind == kUnitShared) {
                    const bool keep = a.T <= a.max_tokens;
                    kept = keep ? 1 : 0;
                    groups = keep ? (a.T + kMT - 1) / kMT : 0;
                    if (lane == 0 && keep) sm.units[off] = make_int4(0, 0, a.T, groups);
                } else {
                    const int4* src = uc.kind == kUnitDept ? a.ws.dept_units : a.ws.exp_units;
                    const int A = uc.kind == kUnitDept ? a.ws.counts[1] : a.ws.counts[0];
                    kept = filter_units_warp(src, A, 1, a.max_tokens, kMT, sm.units + off, &groups);
                }
                __syncwarp();
                const int tot = class_cost_prefix_warp(sm.units + off, kept, uc.rows, cpre + off);
                if (lane == 0) {
                    sm.cls_units[c] = kept;
                    sm.cls_groups[c] = groups;
                    sm.cls_off[c] = off;
                    sm.cls_cost[c] = tot;
                }
                off += class_capacity(uc, a.n, a.g);
            }
        }
        __syncthreads();
    }
    long long R = 0;
    for (int c = 0; c < a.ncls; ++c) R += (long long)a.cls[c].rows * sm.cls_groups[c];
    if (a.tc_first) {
        // the tensor-core kernel ran first and kept the step (its choice
        // was read right after the PDL wait, see the unit-table code)
    } else if (a.auto_tc) {
        // the tensor-core kernel takes the whole step when it is the faster one
        __shared__ int s_tc;
        if (tid == 0) s_tc = prefer_tc(a) ? 1 : 0;
        __syncthreads();
        if (s_tc) R = 0;
        if (blockIdx.x == 0 && tid == 0) a.ws.sync[1] = 1u + (uint32_t)s_tc;
    } else if (blockIdx.x == 0 && tid == 0) {
        a.ws.sync[1] = 0u;
    }
    // CTA's share: equal work (cost units, see cost_units), or equal rows
    // when the cost total would not fit the 32-bit split search
    long long r_begin = grid_share(R, blockIdx.x, gridDim.x, a.grid_magic);
    long long r_end = grid_share(R, blockIdx.x + 1, gridDim.x, a.grid_magic);
    if constexpr (ONE) {
        // one token: every row costs the same, so the equal split above stands
    } else if (R > 0) {
        __shared__ long long s_split[2];
        const long long tot = split_total_cost(a, sm);
        if (tot > 0 && tot < (1ll << 31)) {
            if (tid == 0 || tid == 32) {
                const unsigned b = blockIdx.x + (tid ? 1u : 0u);
                s_split[tid ? 1 : 0] =
                    b == gridDim.x ? R
                                   : split_row_at(a, sm, cpre, (int)grid_share(tot, b, gridDim.x, a.grid_magic));
            }
            __syncthreads();
            r_begin = s_split[0];
            r_end = s_split[1];
        }
    }

    const int row_bytes = a.d * K::kBw;
    const int rps = min(RMAX, kStageBytes / row_bytes);   // rows per stage
    const int nchunks = a.d / 8;

    if (warp == NCW) {
        // ===================== producer =====================
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            uint32_t it = 0;
            long long r = r_begin;
            Seg s;
            bool ok = true;
            auto issue = [&](const char* src, int nr) -> bool {
                const int slot = it % NS;
                const uint32_t par = ((it / NS) & 1u) ^ 1u;
                if (!mbar_wait_bounded(&sm.empty[slot], par)) return false;
                const uint32_t bytes = (uint32_t)nr * row_bytes;
                mbar_arrive_expect_tx(&sm.full[slot], bytes);
                bulk_load(ring + (size_t)slot * kStageBytes, src, bytes, &sm.full[slot], pol);
                ++it;
                return true;
            };
            while (ok && !a.stall_copies && next_seg(a, sm, r, r_end, s)) {
                const UnitClass& uc = a.cls[s.cls];
                const size_t ubase = ((size_t)sm.units[sm.cls_off[s.cls] + s.q].x * uc.rows + s.row0) *
                                     (size_t)row_bytes;
                const char* g = static_cast<const char*>(uc.w_gate) + ubase;
                const char* u = static_cast<const char*>(uc.w_up) + ubase;
                const char* dn = static_cast<const char*>(uc.w_down) + ubase;
                for (int rb = 0; ok && rb < s.nrows; rb += rps) {
                    const int nr = min(rps, s.nrows - rb);
                    ok = issue(g + (size_t)rb * row_bytes, nr) &&
                         issue(u + (size_t)rb * row_bytes, nr);
                }
                for (int rb = 0; ok && rb < s.nrows; rb += rps)
                    ok = issue(dn + (size_t)rb * row_bytes, min(rps, s.nrows - rb));
            }
            if (!ok) set_status(a.ws.status, kDevErrTimeout);
            // Drain: every issued copy must land before the CTA may exit.
            const uint32_t first = it > (uint32_t)NS ? it - NS : 0u;
            for (uint32_t i = first; i < it; ++i)
                mbar_wait_bounded(&sm.full[i % NS], (i / NS) & 1u);
        }
        return;
    }

    // ===================== consumers =====================
    int coff[CH];
    bool cval[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
        const int c = tid + j * K::kNC;
        cval[j] = c < nchunks;
        coff[j] = c * 8 * K::kBw;
    }
    uint32_t it = 0;
    long long r = r_begin;
    Seg s;
    bool ok = true;
    bool aborted = false;
    // Down-projection accumulators.  A one-token step keeps them across its
    // segments (every unit adds into the same output row, the routing weight
    // is already in h) and adds them into the output once, at the end.
    float2 yacc[CH][kMT][4];
#pragma unroll
    for (int j = 0; j < CH; ++j)
#pragma unroll
        for (int m = 0; m < kMT; ++m)
#pragma unroll
            for (int e = 0; e < 4; ++e) yacc[j][m][e] = make_float2(0.0f, 0.0f);
    auto wait_full = [&](int slot, uint32_t i) -> bool {
        if (!ok) return false;
        if (!mbar_wait_bounded(&sm.full[slot], (i / NS) & 1u, ffn_wait_limit(a))) {
            ok = false;
            set_status(a.ws.status, kDevErrTimeout);
        }
        return ok;
    };
    auto release = [&](int slot) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
    };

    while (next_seg(a, sm, r, r_end, s)) {
        int tok[kMT], orow[kMT];
        float wt[kMT];
        const int4 rec = sm.units[sm.cls_off[s.cls] + s.q];
        const int mg = a.local_route ? group_tokens_local(lr, rec, a.cls[s.cls].kind, s.grp, tok, wt, orow)
                                     : group_tokens(a, rec, a.cls[s.cls].kind, s.grp, tok, wt, orow);

        // ---- phase A: gate / up dot products ----
        {
            float2 xr[CH][kMT][4];
#pragma unroll
            for (int j = 0; j < CH; ++j) {
#pragma unroll
                for (int m = 0; m < kMT; ++m) {
                    if (cval[j] && m < mg) {
                        const float4* xp = reinterpret_cast<const float4*>(
                            a.x + (size_t)tok[m] * a.d + (tid + j * K::kNC) * 8);
                        const float4 lo = __ldg(xp), hi = __ldg(xp + 1);
                        xr[j][m][0] = make_float2(lo.x, lo.y);
                        xr[j][m][1] = make_float2(lo.z, lo.w);
                        xr[j][m][2] = make_float2(hi.x, hi.y);
                        xr[j][m][3] = make_float2(hi.z, hi.w);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) xr[j][m][e] = make_float2(0.0f, 0.0f);
                    }
                }
            }
            for (int rb = 0; rb < s.nrows; rb += rps) {
                const int nr = min(rps, s.nrows - rb);
#pragma unroll 1
                for (int mat = 0; mat < 2; ++mat) {
                    const int slot = it % NS;
                    if (wait_full(slot, it)) {
                        const char* st = reinterpret_cast<const char*>(ring + (size_t)slot * kStageBytes);
                        float* gr = &sm.gu[mat][rb * kMT];
                        if (ONE || mg == 1)
                            K::template gu_any<1>(st, nr, row_bytes, coff, cval, xr, gr, mg, lane);
                        else if (mg == 2)
                            K::template gu_any<2>(st, nr, row_bytes, coff, cval, xr, gr, mg, lane);
                        else
                            K::template gu_any<4>(st, nr, row_bytes, coff, cval, xr, gr, mg, lane);
                        release(slot);
                    }
                    ++it;
                }
            }
        }
        // every consumer leaves the barrier with the same abort decision
        if (named_bar_or(1, K::kNC, !ok)) {
            aborted = true;
            break;
        }

        // ---- SwiGLU: h = SiLU(g) * u (times the token's weight when accumulating) ----
        for (int i = tid; i < s.nrows * kMT; i += K::kNC) {
            const int m = i & (kMT - 1);
            float hv = 0.0f;
            if (m < mg) {
                if constexpr (K::kBw == 1) {
                    // FP8 rows: the gate and up dot products and the down row
                    // carry the rows' scales
                    const UnitClass& uc = a.cls[s.cls];
                    const size_t ri = (size_t)rec.x * uc.rows + s.row0 + i / kMT;
                    hv = silu_f(__ldg(uc.sc_gate + ri) * sm.gu[0][i]) * (__ldg(uc.sc_up + ri) * sm.gu[1][i]) *
                         __ldg(uc.sc_down + ri);
                } else {
                    hv = silu_f(sm.gu[0][i]) * sm.gu[1][i];
                }
                if (a.out_mode == MOE_OUT_ACCUM)
                    hv *= m == 0 ? wt[0] : m == 1 ? wt[1] : m == 2 ? wt[2] : wt[3];
            }
            sm.h[i] = hv;
            sm.gu[0][i] = 0.0f;
            sm.gu[1][i] = 0.0f;
        }
        named_bar_sync(1, K::kNC);

        // ---- phase B: down projection into per-thread column accumulators ----
        if constexpr (!ONE) {
#pragma unroll
            for (int j = 0; j < CH; ++j)
#pragma unroll
                for (int m = 0; m < kMT; ++m)
#pragma unroll
                    for (int e = 0; e < 4; ++e) yacc[j][m][e] = make_float2(0.0f, 0.0f);
        }
        for (int rb = 0; rb < s.nrows; rb += rps) {
            const int nr = min(rps, s.nrows - rb);
            const int slot = it % NS;
            if (wait_full(slot, it)) {
                const char* st = reinterpret_cast<const char*>(ring + (size_t)slot * kStageBytes);
                const float* hr = &sm.h[rb * kMT];
                if (ONE || mg == 1)
                    K::template down_any<1>(st, nr, row_bytes, coff, cval, hr, yacc);
                else if (mg == 2)
                    K::template down_any<2>(st, nr, row_bytes, coff, cval, hr, yacc);
                else
                    K::template down_any<4>(st, nr, row_bytes, coff, cval, hr, yacc);
                release(slot);
            }
            ++it;
        }
        if (named_bar_or(1, K::kNC, !ok)) {
            aborted = true;
            break;
        }
        // ---- add this CTA's partial rows into the output (one token: once,
        // after the loop) ----
#pragma unroll
        for (int j = 0; j < (ONE ? 0 : CH); ++j) {
            if (cval[j]) {
                const int col = (tid + j * K::kNC) * 8;
#pragma unroll
                for (int m = 0; m < kMT; ++m) {
                    if (m < mg) {
                        float4* dst = reinterpret_cast<float4*>(a.out + (size_t)orow[m] * a.d + col);
                        atomicAdd(dst, make_float4(yacc[j][m][0].x, yacc[j][m][0].y,
                                                   yacc[j][m][1].x, yacc[j][m][1].y));
                        atomicAdd(dst + 1, make_float4(yacc[j][m][2].x, yacc[j][m][2].y,
                                                       yacc[j][m][3].x, yacc[j][m][3].y));
                    }
                }
            }
        }
    }
    if constexpr (ONE) {
        // One token: the CTA's partial output row goes through shared memory
        // (the ring, idle once every stage was consumed) and is added into
        // the output by one bulk reduction.  Every CTA adds into the same row,
        // and hundreds of CTAs' per-element atomics on it queue at L2 for
        // microseconds; a bulk reduction per CTA does not.
        if (!aborted && r_begin < r_end && (size_t)a.d * 4 <= (size_t)NS * kStageBytes) {
            float* stg = reinterpret_cast<float*>(ring);
#pragma unroll
            for (int j = 0; j < CH; ++j) {
                if (cval[j]) {
                    float4* p = reinterpret_cast<float4*>(stg + (tid + j * K::kNC) * 8);
                    p[0] = make_float4(yacc[j][0][0].x, yacc[j][0][0].y, yacc[j][0][1].x, yacc[j][0][1].y);
                    p[1] = make_float4(yacc[j][0][2].x, yacc[j][0][2].y, yacc[j][0][3].x, yacc[j][0][3].y);
                }
            }
            fence_async_smem();
            named_bar_sync(1, K::kNC);
            if (tid == 0) {
                bulk_reduce_add_f32(a.out, stg, (uint32_t)a.d * 4u);
                bulk_commit();
                bulk_wait_all();
            }
        } else if (!aborted && r_begin < r_end) {
#pragma unroll
            for (int j = 0; j < CH; ++j) {
                if (cval[j]) {
                    float4* dst = reinterpret_cast<float4*>(a.out + (tid + j * K::kNC) * 8);
                    atomicAdd(dst, make_float4(yacc[j][0][0].x, yacc[j][0][0].y, yacc[j][0][1].x, yacc[j][0][1].y));
                    atomicAdd(dst + 1, make_float4(yacc[j][0][2].x, yacc[j][0][2].y, yacc[j][0][3].x, yacc[j][0][3].y));
                }
            }
        }
    }
}

// Launch shape of one instantiation: weight type, consumer warps, 8-column
// chunks per thread, rows per stage, CTAs per SM.
template <typename WT, int NCW, int CH, int RMAX, int CPS>
struct FfnCfg {};

// Dynamic shared memory of a launch: ring, fixed carve-up, one unit record
// per possible unit of every class, and the routing state of the local path.
template <typename WT, int NCW, int CH, int RMAX, int CPS>
constexpr int cps_of(FfnCfg<WT, NCW, CH, RMAX, CPS>) { return CPS; }
template <typename WT, int NCW, int CH, int RMAX, int CPS>
constexpr int threads_of(FfnCfg<WT, NCW, CH, RMAX, CPS>) { return (NCW + 1) * 32; }

template <typename WT, int NCW, int CH, int RMAX, int CPS>
size_t ffn_smem(const FfnArgs& a, FfnCfg<WT, NCW, CH, RMAX, CPS>) {
    constexpr int NS = kRingBytesPerSM / kStageBytes / CPS;
    int units = 0;
    for (int c = 0; c < a.ncls; ++c) units += class_capacity(a.cls[c], a.n, a.g);
    return (size_t)NS * kStageBytes + sizeof(FfnSmem<NS>) + (size_t)units * sizeof(int4) +
           align16(4 * (size_t)units) + (a.local_route ? local_route_bytes(a.T, a.n, a.k, a.g, NCW + 1) : 0);
}

// Largest dynamic shared memory per CTA that still lets `cps` CTAs share an SM.
size_t smem_per_cta_limit(int cps) {
    static int cache[64][3] = {};   // per device: per-SM, reserved per block, opt-in maximum
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int* c = cache[dev];
    if (c[0] == 0) {
        cudaDeviceGetAttribute(&c[1], cudaDevAttrReservedSharedMemoryPerBlock, dev);
        cudaDeviceGetAttribute(&c[2], cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&c[0], cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    }
    const long long lim = (long long)c[0] / cps - c[1];
    return (size_t)(lim < c[2] ? (lim > 0 ? lim : 0) : c[2]);
}

template <typename WT, int NCW, int CH, int RMAX, int CPS>
cudaError_t launch_ffn_t(const FfnArgs& a, cudaStream_t s, FfnCfg<WT, NCW, CH, RMAX, CPS> cfg_tag) {
    const unsigned grid = (unsigned)(device_sm_count() * CPS);
    auto kern = a.local_route && a.T == 1 ? ffn_stream_kernel<WT, NCW, CH, RMAX, CPS, true>
                                          : ffn_stream_kernel<WT, NCW, CH, RMAX, CPS, false>;
    const size_t smem = ffn_smem(a, cfg_tag);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    FfnArgs args = a;
    args.grid_magic = grid_magic_of(grid);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3((NCW + 1) * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

// ---- combine: y[t] = sum of the token's rows with their weights, fixed order ----
__global__ void combine_kernel(CombineArgs a) {
    const int t = blockIdx.y;
    const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
    if (c4 * 4 >= a.d) return;
    const float4* rows = reinterpret_cast<const float4*>(a.rows);
    const int d4 = a.d / 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < a.k; ++s) {
        const int p = a.ws.tok_asg[t * a.k + s];
        const float w = a.ws.asg_w[p];
        const float4 v = rows[(size_t)p * d4 + c4];
        acc.x = fmaf(w, v.x, acc.x); acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z); acc.w = fmaf(w, v.w, acc.w);
    }
    for (int j = 0; j < a.m; ++j) {
        const int p = a.ws.tok_dpos[t * a.m + j];
        if (p < 0) continue;
        const float w = a.ws.dept_w[p];
        const float4 v = rows[(size_t)(a.rows_dept_base + p) * d4 + c4];
        acc.x = fmaf(w, v.x, acc.x); acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z); acc.w = fmaf(w, v.w, acc.w);
    }
    if (a.has_shared) {
        const float4 v = rows[(size_t)(a.rows_shared_base + t) * d4 + c4];
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    reinterpret_cast<float4*>(a.y)[(size_t)t * d4 + c4] = acc;
}

__global__ void split_x_kernel(const float* x, long long elems, __nv_bfloat16* xb) {
    split_activations(x, elems, xb, blockIdx.x * (long long)blockDim.x + threadIdx.x,
                      (long long)gridDim.x * blockDim.x);
}

__global__ void split_terms_kernel(const float* x, int T, int d, uint8_t* xq) {
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, nw = (gridDim.x * blockDim.x) >> 5;
    for (int t = gw; t < T; t += nw) split_e4m3_terms_warp(x, T, d, t, xq, lane);
}

__global__ void zero_kernel(uint4* p, size_t n16) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16;
         i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

// Launch shape of the bf16 kernel for d <= 2048: consumer warps, 8-column
// chunks per thread, rows per stage, CTAs per SM.
#ifndef MOE_CC_NCW
#define MOE_CC_NCW 8
#endif
#ifndef MOE_CC_CH
#define MOE_CC_CH 1
#endif
#ifndef MOE_CC_RMAX
#define MOE_CC_RMAX 4
#endif
#ifndef MOE_CC_CPS
#define MOE_CC_CPS 2
#endif

// Calls f with the launch shape for this dtype and hidden size: consumer
// warps x chunks per thread x 8 must cover d; RMAX is the most rows one 16 KB
// stage holds at that width.
template <class F>
auto with_ffn_cfg(const FfnArgs& a, F f) {
    if (a.dtype == MOE_DTYPE_BF16) {
        if (a.d <= 2048) return f(FfnCfg<__nv_bfloat16, MOE_CC_NCW, MOE_CC_CH, MOE_CC_RMAX, MOE_CC_CPS>{});
        return f(FfnCfg<__nv_bfloat16, 15, 2, 1, 1>{});
    }
    if (a.dtype == MOE_DTYPE_FP8_E4M3) {
        if (a.d <= 2048) return f(FfnCfg<__nv_fp8_e4m3, 8, 1, 4, 2>{});
        return f(FfnCfg<__nv_fp8_e4m3, 15, 2, 2, 1>{});
    }
    if (a.d <= 1024) return f(FfnCfg<float, 4, 1, 8, 1>{});
    return f(FfnCfg<float, 15, 2, 1, 1>{});
}

cudaError_t launch_ffn(const FfnArgs& a, cudaStream_t s) {
    return with_ffn_cfg(a, [&](auto cfg) { return launch_ffn_t(a, s, cfg); });
}

bool ffn_local_route_fits(const FfnArgs& a) {
    FfnArgs b = a;
    b.local_route = 1;
    const int m = a.g > 1 ? a.n / a.g : 0;
    return with_ffn_cfg(b, [&](auto cfg) {
        // one thread per unit: the experts, then the departments from the next warp on
        // (and the top-k's lane-held candidates: n <= 256)
        return a.n <= 256 && ((a.n + 31) / 32) * 32 + m <= threads_of(cfg) &&
               ffn_smem(b, cfg) <= smem_per_cta_limit(cps_of(cfg));
    });
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
    const int d4 = a.d / 4;
    const int threads = d4 < 256 ? ((d4 + 31) / 32) * 32 : 256;
    dim3 grid((d4 + threads - 1) / threads, a.T);
    combine_kernel<<<grid, threads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t s) {
    const size_t n16 = bytes / 16;
    if (n16 == 0) return cudaSuccess;
    const int threads = 256;
    const size_t want = (n16 + threads - 1) / threads;
    const int blocks = (int)(want < 4096 ? want : 4096);
    zero_kernel<<<blocks, threads, 0, s>>>(reinterpret_cast<uint4*>(p), n16);
    return cudaGetLastError();
}

}  // namespace moe

namespace moe {
cudaError_t launch_split_terms(const float* x, int T, int d, __nv_bfloat16* xb, cudaStream_t s) {
    const int threads = 128;                  // a warp per token
    split_terms_kernel<<<(T + 3) / 4, threads, 0, s>>>(x, T, d, reinterpret_cast<uint8_t*>(xb));
    return cudaGetLastError();
}

cudaError_t launch_split_x(const float* x, long long elems, __nv_bfloat16* xb, cudaStream_t s) {
    const long long n8 = elems / 8;
    const int threads = 256;
    const long long want = (n8 + threads - 1) / threads;
    split_x_kernel<<<(int)(want < 1024 ? (want > 0 ? want : 1) : 1024), threads, 0, s>>>(x, elems, xb);
    return cudaGetLastError();
}
}  // namespace moe
