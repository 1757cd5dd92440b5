// Routing inside the FFN CTAs (whole-layer path), shared by the CUDA-core and
// tensor-core FFN kernels: the top-k of every token from the router logits,
// the unit records and the per-unit token lists, all in shared memory, built
// by every CTA.  Routing as in "DeaMoE: Efficient MoE Structure for Fast
// Small-Batch Decoding" §2.1 eqs. (2)-(3) with the selection-only bias of
// "DeepSeekMoE Guide: Fine-Grained Experts & Dynamic Routing"; the lists
// group the assignments per expert and the tokens per department (DeaMoE
// §3.2), as "MoE inference engineering, clearly explained" describes ("How a
// batch becomes expert-specific matrices").
#pragma once

#include "kernels.h"

namespace moe {

namespace {

// ---- cost model of the CUDA-core row split --------------------------------
// A row costs what its token group's code path costs: groups of one or two
// tokens run the narrow register tiles, groups of three or four the wide one,
// which was measured about 1.5x slower per row (the weight stream is the
// same; the per-token dot products, reductions and accumulations are not).
// Each token group also costs kSegCost once, at its first row: a CTA whose
// range starts a new group pays a segment switch (activation loads, the
// SwiGLU barrier, a drained ring).  A unit of t tokens costs
// rows * cost_units(t) + groups * kSegCost.
#ifndef MOE_COST_NARROW
#define MOE_COST_NARROW 2
#endif
#ifndef MOE_COST_WIDE
#define MOE_COST_WIDE 3
#endif
#ifndef MOE_COST_SEG
#define MOE_COST_SEG 24
#endif
constexpr int kCostNarrow = MOE_COST_NARROW;
constexpr int kCostWide = MOE_COST_WIDE;
constexpr int kSegCost = MOE_COST_SEG;

__device__ __forceinline__ int group_cost(int mg) { return mg > 2 ? kCostWide : kCostNarrow; }
__device__ __forceinline__ int cost_units(int t) {
    constexpr int G = kGroupTokens;
    return (t / G) * group_cost(G) + (t % G ? group_cost(t % G) : 0);
}
// Cost of a unit of t tokens whose rows are `rows` long.
__device__ __forceinline__ int unit_cost(int t, int rows) {
    return rows * cost_units(t) + ((t + kGroupTokens - 1) / kGroupTokens) * kSegCost;
}


// Where a kernel keeps its unit table: per class the offset of its records,
// their count, group total and (CUDA-core split) cost total; the records
// {unit, first entry, tokens, inclusive group prefix}; the cost prefixes.
struct UnitTableView {
    int4* units;
    int* cls_off;
    int* cls_units;
    int* cls_groups;
    int* cls_cost;   // null without a cost model
    int* cpre;       // null without a cost model
};

// ---- routing inside the CTA (whole-layer path) ------------------------------
// Every CTA takes the top-k of every token from the router logits and builds
// its own unit records and per-unit token lists in shared memory, so that no
// single block serialises the dispatch and nothing is read back from global
// memory.  Order and content match the dispatch kernel's: ascending unit id,
// then ascending token id; a department's token set X^j is the union of its
// experts' sets, with weight omega = sum of the token's routing weights on
// that department's experts, in slot order.  Units sit one per thread (the
// experts, then the departments from the next warp boundary on), so the host
// takes this path only when roundup32(n) + m fits the block.
struct LocalRoute {
    uint32_t* emask;   // [n][W]: bit t of row e = token t chose expert e
    uint32_t* dmask;   // [m][W]: union over the department's experts
    int16_t* idx;      // [T*k] selected experts
    int16_t* didx;     // [T*k] their departments
    float* w;          // [T*k] routing weights
    int* off;          // [n + m] first list entry of each expert, then each department
    int16_t* etok;     // [T*k] expert lists (ascending expert, then token): token
    float* ew;         //       and routing weight
    int16_t* dtok;     // [T*min(k, m)] department lists: token
    float* dw;         //       and department weight omega
    int4* wtot;        // per warp: totals of the unit scan
    int* tcg;          // [2] tensor-core group totals (experts, departments)
    int W, m;
};

__host__ __device__ __forceinline__ size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

// Bytes of the local routing state for a block of nwarps warps.
__host__ __device__ __forceinline__ size_t local_route_bytes(int T, int n, int k, int g, int nwarps) {
    const size_t W = (size_t)(T + 31) / 32;
    const size_t m = g > 1 ? (size_t)(n / g) : 0;
    const size_t TK = (size_t)T * k;
    const size_t DK = m ? (size_t)T * ((size_t)k < m ? (size_t)k : m) : 0;
    return align16(4 * n * W) + align16(4 * m * W) + align16(2 * TK) * 2 + align16(4 * TK) +
           align16(4 * (n + m)) + align16(2 * TK) + align16(4 * TK) + align16(2 * DK) + align16(4 * DK) +
           align16(16 * (size_t)nwarps) + 16;
}

__device__ __forceinline__ LocalRoute local_route_at(unsigned char* p, int T, int n, int k, int g,
                                                     int nwarps) {
    LocalRoute lr;
    lr.W = (T + 31) >> 5;
    lr.m = g > 1 ? n / g : 0;
    const size_t TK = (size_t)T * k;
    const size_t DK = lr.m ? (size_t)T * (k < lr.m ? k : lr.m) : 0;
    auto take = [&](size_t bytes) {
        unsigned char* q = p;
        p += align16(bytes);
        return q;
    };
    lr.emask = reinterpret_cast<uint32_t*>(take(4 * (size_t)n * lr.W));
    lr.dmask = reinterpret_cast<uint32_t*>(take(4 * (size_t)lr.m * lr.W));
    lr.idx = reinterpret_cast<int16_t*>(take(2 * TK));
    lr.didx = reinterpret_cast<int16_t*>(take(2 * TK));
    lr.w = reinterpret_cast<float*>(take(4 * TK));
    lr.off = reinterpret_cast<int*>(take(4 * (size_t)(n + lr.m)));
    lr.etok = reinterpret_cast<int16_t*>(take(2 * TK));
    lr.ew = reinterpret_cast<float*>(take(4 * TK));
    lr.dtok = reinterpret_cast<int16_t*>(take(2 * DK));
    lr.dw = reinterpret_cast<float*>(take(4 * DK));
    lr.wtot = reinterpret_cast<int4*>(take(16 * (size_t)nwarps));
    lr.tcg = reinterpret_cast<int*>(take(16));
    return lr;
}

// Rank of token t among the tokens of a mask row (ascending).
__device__ __forceinline__ int row_rank(const uint32_t* row, int t) {
    int r = __popc(row[t >> 5] & ((1u << (t & 31)) - 1u));
    for (int w = 0; w < (t >> 5); ++w) r += __popc(row[w]);
    return r;
}

// Top-k of every token, one warp per token: selections into shared memory,
// the expert bitmasks (zeroed by the caller) and department ids; CTA 0 also
// stores them as the routing outputs.  Ends with a barrier.
template <int J, int NT>
__device__ void local_topk_rows(const FfnArgs& a, const LocalRoute& lr, bool writer) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int t = warp; t < a.T; t += NT / 32) {
        int e;
        float w;
        const bool bad =
            topk_select_warp<J>(a.ws.logits + (size_t)t * a.n, a.bias, a.n, a.k, a.scale, e, w);
        if (lane < a.k) {
            lr.idx[t * a.k + lane] = (int16_t)e;
            lr.didx[t * a.k + lane] = (int16_t)(a.g > 1 ? e / a.g : e);
            lr.w[t * a.k + lane] = w;
            atomicOr(&lr.emask[e * lr.W + (t >> 5)], 1u << (t & 31));
            if (writer) {
                a.topk_idx[(size_t)t * a.k + lane] = e;
                a.topk_w[(size_t)t * a.k + lane] = w;
            }
        }
        if (bad && writer && lane == 0) set_status(a.ws.status, kDevErrRouting);
    }
    __syncthreads();
}

template <int NT>
__device__ __forceinline__ void local_topk(const FfnArgs& a, const LocalRoute& lr, bool writer) {
    const int J = (a.n + 31) / 32;
    if (J <= 1) local_topk_rows<1, NT>(a, lr, writer);
    else if (J <= 2) local_topk_rows<2, NT>(a, lr, writer);
    else if (J <= 4) local_topk_rows<4, NT>(a, lr, writer);
    else local_topk_rows<8, NT>(a, lr, writer);
}

// Inclusive warp scan of four counters.
__device__ __forceinline__ int4 warp_inclusive_scan4(int4 v) {
    const int lane = threadIdx.x & 31;
    __syncwarp();
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int tx = __shfl_up_sync(0xffffffffu, v.x, o);
        const int ty = __shfl_up_sync(0xffffffffu, v.y, o);
        const int tz = __shfl_up_sync(0xffffffffu, v.z, o);
        const int tw = __shfl_up_sync(0xffffffffu, v.w, o);
        if (lane >= o) {
            v.x += tx;
            v.y += ty;
            v.z += tz;
            v.w += tw;
        }
    }
    return v;
}

// After the top-k (every thread of the CTA; ends with a barrier): unit
// counts, records (groups of GSZ tokens) and, with COST, the cost prefixes of
// the CUDA-core split for every class, then the per-unit token lists.  Expert u sits on thread u, department j on thread roundup32(n) + j,
// so each kind's prefix sums are warp scans plus the totals of its earlier
// warps.  CTA 0 (`writer`) also stores the dispatch in the workspace in the
// layout moe_dispatch writes.
template <int NT, int GSZ, bool COST>
__device__ void local_tables(const FfnArgs& a, const UnitTableView& sm, const LocalRoute& lr,
                             bool writer) {
    int* cpre = sm.cpre;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = a.n, m = lr.m, W = lr.W;
    const int n_pad = (n + 31) & ~31;
    const bool isx = tid < n;
    const bool isd = m > 0 && tid >= n_pad && tid < n_pad + m;
    const int u = isx ? tid : tid - n_pad;
    int cnt = 0;
    if (isx) {
        for (int w = 0; w < W; ++w) cnt += __popc(lr.emask[u * W + w]);
    } else if (isd) {
        for (int w = 0; w < W; ++w) {
            uint32_t v = 0u;
            for (int e = u * a.g; e < (u + 1) * a.g; ++e) v |= lr.emask[e * W + w];
            lr.dmask[u * W + w] = v;
            cnt += __popc(v);
        }
    }
    // tokens, active units, groups of GSZ tokens, and the cost units of the
    // CUDA-core split (COST) or else the groups of kGroupTokens that the
    // workspace records carry
    const int4 mine = make_int4(cnt, cnt > 0 ? 1 : 0, (cnt + GSZ - 1) / GSZ,
                                COST ? cost_units(cnt) : (cnt + kGroupTokens - 1) / kGroupTokens);
    const int4 inc = warp_inclusive_scan4(mine);
    if (lane == 31) lr.wtot[warp] = inc;
    if (tid < 2) lr.tcg[tid] = 0;
    __syncthreads();
    int4 pre = make_int4(inc.x - mine.x, inc.y - mine.y, inc.z - mine.z, inc.w - mine.w);
    for (int w2 = isd ? n_pad / 32 : 0; w2 < warp; ++w2) {
        const int4 t = lr.wtot[w2];
        pre.x += t.x;
        pre.y += t.y;
        pre.z += t.z;
        pre.w += t.w;
    }
    if (isx || isd) {
        lr.off[isx ? u : n + u] = pre.x;
        if (cnt > 0) {
            const int4 r = make_int4(u, pre.x, cnt, pre.z + mine.z);
            for (int c = 0; c < a.ncls; ++c) {
                const int kind = a.cls[c].kind;
                if ((isx && kind == kUnitExpert) || (isd && kind == kUnitDept)) {
                    sm.units[sm.cls_off[c] + pre.y] = r;
                    if (COST) cpre[sm.cls_off[c] + pre.y] = a.cls[c].rows * pre.w + kSegCost * pre.z;
                }
            }
            if (writer) {
                (isd ? a.ws.act_dept : a.ws.act_exp)[pre.y] = u;
                (isd ? a.ws.dept_units : a.ws.exp_units)[pre.y] =
                    GSZ == kGroupTokens ? r : make_int4(u, pre.x, cnt, pre.w + mine.w);
                atomicAdd(&lr.tcg[isd ? 1 : 0], (cnt + kTcGroupTokens - 1) / kTcGroupTokens);
            }
        }
        if (writer) {
            (isd ? a.ws.dept_count : a.ws.exp_count)[u] = cnt;
            (isd ? a.ws.dept_off : a.ws.exp_off)[u] = pre.x;
        }
        // the last unit of each kind holds the kind's totals
        if (u == (isd ? m : n) - 1) {
            const int4 tot = make_int4(pre.x + mine.x, pre.y + mine.y, pre.z + mine.z, pre.w + mine.w);
            for (int c = 0; c < a.ncls; ++c) {
                const int kind = a.cls[c].kind;
                if ((isx && kind == kUnitExpert) || (isd && kind == kUnitDept)) {
                    sm.cls_units[c] = tot.y;
                    sm.cls_groups[c] = tot.z;
                    if (COST) sm.cls_cost[c] = a.cls[c].rows * tot.w + kSegCost * tot.z;
                }
            }
            if (writer) {
                (isd ? a.ws.dept_off : a.ws.exp_off)[isd ? m : n] = tot.x;
                a.ws.counts[isd ? 1 : 0] = tot.y;
            }
        }
    }
    if (tid == 0) {
        for (int c = 0; c < a.ncls; ++c)
            if (a.cls[c].kind == kUnitShared) {
                const int G = (a.T + GSZ - 1) / GSZ;
                sm.units[sm.cls_off[c]] = make_int4(0, 0, a.T, G);
                sm.cls_units[c] = 1;
                sm.cls_groups[c] = G;
                if (COST) {
                    cpre[sm.cls_off[c]] = 0;
                    sm.cls_cost[c] = unit_cost(a.T, a.cls[c].rows);
                }
            }
        if (writer && m == 0) {
            a.ws.counts[1] = 0;
            a.ws.counts[3] = 0;
        }
    }
    __syncthreads();
    if (writer && tid == 0) {
        a.ws.counts[2] = lr.tcg[0];
        if (m > 0) a.ws.counts[3] = lr.tcg[1];
    }
    // token lists: expert lists from every assignment, department lists from
    // the first slot of each token on each department
    const int TK = a.T * a.k;
    for (int i = tid; i < TK; i += NT) {
        const int t = i / a.k, sl = i - t * a.k;
        const int e = lr.idx[i];
        const float wv = lr.w[i];
        const int pos = lr.off[e] + row_rank(lr.emask + e * W, t);
        lr.etok[pos] = (int16_t)t;
        lr.ew[pos] = wv;
        if (writer) {
            a.ws.asg_tok[pos] = t;
            a.ws.asg_slot[pos] = sl;
            a.ws.asg_w[pos] = wv;
            a.ws.tok_asg[i] = pos;
        }
        if (m > 0) {
            const int j = lr.didx[i];
            bool first = true;
            float om = 0.0f;   // omega: the token's weights on department j, slot order
            for (int q = 0; q < a.k; ++q)
                if (lr.didx[t * a.k + q] == j) {
                    if (q < sl) first = false;
                    om += lr.w[t * a.k + q];
                }
            if (first) {
                const int pd = lr.off[n + j] + row_rank(lr.dmask + j * W, t);
                lr.dtok[pd] = (int16_t)t;
                lr.dw[pd] = om;
                if (writer) {
                    a.ws.dept_tok[pd] = t;
                    a.ws.dept_w[pd] = om;
                    a.ws.tok_dpos[t * m + j] = pd;
                }
            }
        }
    }
    if (writer && m > 0)
        for (int i = tid; i < a.T * m; i += NT) {
            const int t = i / m, j = i - t * m;
            if (!((lr.dmask[j * W + (t >> 5)] >> (t & 31)) & 1u)) a.ws.tok_dpos[i] = -1;
        }
    __syncthreads();
}

// One token (after the top-k; every thread of the CTA; ends with a barrier):
// every unit then holds exactly that token, so the unit records follow from
// the selection itself, with no masks, counts or scans.  The order is the
// general tables' (ascending expert id, then ascending department id: a
// unit's place is the number of selected ids below its own), so that a CTA
// built either way splits the same row sequence; one group per unit; a
// department's omega is the token's weights on its experts summed in slot
// order.  No cost prefixes: the caller splits the rows evenly.
template <int NT>
__device__ void local_tables_one_token(const FfnArgs& a, const UnitTableView& sm, const LocalRoute& lr) {
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x, k = a.k;
        const bool act = lane < k;
        const int e = act ? lr.idx[lane] : 0;
        const int dj = act ? lr.didx[lane] : 0;
        const float w = act ? lr.w[lane] : 0.0f;
        const bool dept = lr.m > 0;
        // the lane-dependent loads above may leave the warp diverged; the
        // shuffle loops below run at full speed only on a converged warp
        __syncwarp();
        int p = 0;              // experts selected below e
        uint32_t same = 0u;     // slots on department dj
        float om = 0.0f;
        for (int r = 0; r < k; ++r) {
            const int er = __shfl_sync(0xffffffffu, e, r);
            const int dr = __shfl_sync(0xffffffffu, dj, r);
            const float wr = __shfl_sync(0xffffffffu, w, r);
            p += er < e ? 1 : 0;
            // selects, not a branch: the warp stays converged for the next
            // round's shuffles (adding +0 leaves omega's bits unchanged)
            const bool sd = dr == dj;
            same |= sd ? 1u << r : 0u;
            om += sd ? wr : 0.0f;
        }
        // one lane per selected department: its first slot
        const bool first = dept && act && (same & ((1u << lane) - 1u)) == 0u;
        const uint32_t fm = __ballot_sync(0xffffffffu, first);
        int q = 0;              // departments selected below dj
        for (int r = 0; r < k; ++r) {
            const int dr = __shfl_sync(0xffffffffu, dj, r);
            q += ((fm >> r) & 1u) && dr < dj ? 1 : 0;
        }
        if (act) {
            lr.etok[p] = 0;
            lr.ew[p] = w;
        }
        if (first) {
            lr.dtok[q] = 0;
            lr.dw[q] = om;
        }
        for (int c = 0; c < a.ncls; ++c) {
            const int kind = a.cls[c].kind;
            int4* u = sm.units + sm.cls_off[c];
            int nu = 0;
            if (kind == kUnitExpert) {
                if (act) u[p] = make_int4(e, p, 1, p + 1);
                nu = k;
            } else if (kind == kUnitDept) {
                if (first) u[q] = make_int4(dj, q, 1, q + 1);
                nu = __popc(fm);
            } else {
                if (lane == 0) u[0] = make_int4(0, 0, 1, 1);
                nu = 1;
            }
            if (lane == 0) {
                sm.cls_units[c] = nu;
                sm.cls_groups[c] = nu;
            }
        }
    }
    __syncthreads();
}

// Tokens of group `grp` of a unit from the shared-memory lists, with their
// weights (ACCUM mode: the output row is the token).
template <int MT>
__device__ __forceinline__ int group_tokens_local(const LocalRoute& lr, const int4 rec, int kind, int grp,
                                                  int (&tok)[MT], float (&wt)[MT], int (&orow)[MT]) {
    const int first = grp * MT;
    const int mg = min(MT, rec.z - first);
    const int p0 = rec.y + first;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
        int t = 0;
        float w = 0.0f;
        if (i < mg) {
            if (kind == kUnitShared) {
                t = first + i;
                w = 1.0f;
            } else if (kind == kUnitDept) {
                t = lr.dtok[p0 + i];
                w = lr.dw[p0 + i];
            } else {
                t = lr.etok[p0 + i];
                w = lr.ew[p0 + i];
            }
        }
        tok[i] = t;
        wt[i] = w;
        orow[i] = t;
    }
    return mg;
}

// Token and weight of entry `entry` of a unit's list (its first entry is
// the record's .y): the shared expert's entries are its tokens.
__device__ __forceinline__ void local_entry(const LocalRoute& lr, int kind, int entry, int& t, float& w) {
    if (kind == kUnitShared) {
        t = entry;
        w = 1.0f;
    } else if (kind == kUnitDept) {
        t = lr.dtok[entry];
        w = lr.dw[entry];
    } else {
        t = lr.etok[entry];
        w = lr.ew[entry];
    }
}

}  // namespace

}  // namespace moe
