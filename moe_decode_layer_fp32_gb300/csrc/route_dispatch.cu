// Router GEMV + warp top-k + routing weights, and the device-side dispatch that
// turns (topk_idx, topk_w) into expert / department index lists.
//
// Routing follows "DeaMoE: Efficient MoE Structure for Fast Small-Batch
// Decoding" §2.1 eqs. (2)-(3) (S(x) = TopK(W_r x, k), weights = softmax over the
// selected logits, scaled) and the selection-only bias of "DeepSeekMoE Guide:
// Fine-Grained Experts & Dynamic Routing" (routing-bias formulation).  Dispatch
// builds the grouping of "MoE inference engineering, clearly explained" ("How a
// batch becomes expert-specific matrices": assignments grouped by expert, token
// ids kept, inverse map for the combine) and the department token sets X^j of
// DeaMoE §3.2.
#include <climits>

#include "kernels.h"

namespace moe {

namespace {

constexpr int kRouteThreads = 512;
#ifndef MOE_ROUTE_PDL
#define MOE_ROUTE_PDL 1
#endif
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kDispatchThreads = 512;
constexpr int kMaskWords = (kMaxT + 31) / 32;
constexpr int kStagedAssignments = 1024;   // T*k staged in shared memory for the fused dispatch

struct DispatchSmem {
    uint32_t emask[kMaxN * kMaskWords];       // expert -> token bitmask
    uint32_t dmask[(kMaxN / 2) * kMaskWords]; // department -> token bitmask
    int cnt[kMaxN];                           // tokens per unit -> offsets
    int act[kMaxN];                           // active flag -> active position
    int grp[kMaxN];                           // register groups -> group prefix
    int3 warp_tmp[32];
    int err;
    int tc_groups;
};

// Rank of token t among the tokens set in a mask row (tokens ascending).
__device__ __forceinline__ int mask_rank(const uint32_t* row, int t) {
    int r = __popc(row[t >> 5] & ((1u << (t & 31)) - 1u));
    for (int w = 0; w < (t >> 5); ++w) r += __popc(row[w]);
    return r;
}

// Counts of `units` mask rows -> offsets, active lists and the FFN unit records.
// Also writes the total of ceil(count / kTcGroupTokens) (tensor-core token groups).
template <int NT>
__device__ void unit_lists(const uint32_t* mask, int units, int W, int32_t* count_out,
                           int32_t* off_out, int32_t* act_out, int4* rec_out, int32_t* n_active,
                           int32_t* tc_groups_out, DispatchSmem& sm) {
    const int tid = threadIdx.x;
    int tcg = 0;
    for (int u = tid; u < units; u += NT) {
        int c = 0;
        for (int w = 0; w < W; ++w) c += __popc(mask[u * W + w]);
        sm.cnt[u] = c;
        sm.act[u] = c > 0 ? 1 : 0;
        sm.grp[u] = (c + kGroupTokens - 1) / kGroupTokens;
        tcg += (c + kTcGroupTokens - 1) / kTcGroupTokens;
        count_out[u] = c;
    }
    tcg = warp_sum_int(tcg);
    if ((tid & 31) == 0 && tcg) atomicAdd(&sm.tc_groups, tcg);   // zeroed by the caller
    __syncthreads();
    const int3 tot = block_exclusive_scan3<NT>(sm.cnt, sm.act, sm.grp, units, sm.warp_tmp);
    for (int u = tid; u < units; u += NT) {
        off_out[u] = sm.cnt[u];
        const int next_act = u + 1 < units ? sm.act[u + 1] : tot.y;
        if (next_act != sm.act[u]) {  // active
            const int next_grp = u + 1 < units ? sm.grp[u + 1] : tot.z;
            const int next_off = u + 1 < units ? sm.cnt[u + 1] : tot.x;
            act_out[sm.act[u]] = u;
            rec_out[sm.act[u]] = make_int4(u, sm.cnt[u], next_off - sm.cnt[u], next_grp);
        }
    }
    if (tid == 0) {
        off_out[units] = tot.x;
        *n_active = tot.y;
        *tc_groups_out = sm.tc_groups;
    }
}

// Builds every dispatch list in the workspace.  One block, NT threads.
// Order: ascending expert (department) id, then ascending token id.
template <int NT>
__device__ void dispatch_block(const int32_t* idx, const float* wts, int T, int n, int k,
                               int g, const WsPtrs& ws, DispatchSmem& sm) {
    const int tid = threadIdx.x;
    const int W = (T + 31) >> 5;
    const int TK = T * k;
    for (int i = tid; i < n * W; i += NT) sm.emask[i] = 0u;
    if (tid == 0) {
        sm.err = 0;
        sm.tc_groups = 0;
    }
    __syncthreads();
    for (int a = tid; a < TK; a += NT) {
        const int t = a / k;
        const int e = idx[a];
        if (e < 0 || e >= n) {
            sm.err = 1;
            continue;
        }
        const uint32_t bit = 1u << (t & 31);
        const uint32_t old = atomicOr(&sm.emask[e * W + (t >> 5)], bit);
        if (old & bit) sm.err = 1;  // the token chose this expert twice
    }
    __syncthreads();
    if (sm.err) {
        if (tid == 0) {
            set_status(ws.status, kDevErrRouting);
            ws.counts[0] = 0;
            ws.counts[1] = 0;
            ws.counts[2] = 0;
            ws.counts[3] = 0;
        }
        return;
    }
    // ---- experts ----
    unit_lists<NT>(sm.emask, n, W, ws.exp_count, ws.exp_off, ws.act_exp, ws.exp_units,
                   &ws.counts[0], &ws.counts[2], sm);
    for (int a = tid; a < TK; a += NT) {
        const int t = a / k;
        const int e = idx[a];
        const int pos = sm.cnt[e] + mask_rank(&sm.emask[e * W], t);
        ws.asg_tok[pos] = t;
        ws.asg_slot[pos] = a - t * k;
        ws.asg_w[pos] = wts[a];
        ws.tok_asg[a] = pos;
    }
    __syncthreads();
    if (g <= 1) {
        if (tid == 0) {
            ws.counts[1] = 0;
            ws.counts[3] = 0;
        }
        return;
    }
    // ---- departments: X^j = tokens that chose any expert of department j ----
    const int m = n / g;
    if (tid == 0) sm.tc_groups = 0;   // ordered before its use by the barrier below
    for (int i = tid; i < m * W; i += NT) {
        const int j = i / W, w = i - (i / W) * W;
        uint32_t v = 0u;
        for (int e = j * g; e < (j + 1) * g; ++e) v |= sm.emask[e * W + w];
        sm.dmask[i] = v;
    }
    __syncthreads();
    unit_lists<NT>(sm.dmask, m, W, ws.dept_count, ws.dept_off, ws.act_dept, ws.dept_units,
                   &ws.counts[1], &ws.counts[3], sm);
    for (int i = tid; i < m * T; i += NT) {
        const int j = i / T, t = i - (i / T) * T;
        const uint32_t* row = &sm.dmask[j * W];
        if ((row[t >> 5] >> (t & 31)) & 1u) {
            const int pos = sm.cnt[j] + mask_rank(row, t);
            float s = 0.0f;  // department weight: routing weights of its experts, slot order
            for (int q = 0; q < k; ++q) {
                const int e = idx[t * k + q];
                if (e / g == j) s += wts[t * k + q];
            }
            ws.dept_tok[pos] = t;
            ws.dept_w[pos] = s;
            ws.tok_dpos[t * m + j] = pos;
        } else {
            ws.tok_dpos[t * m + j] = -1;
        }
    }
}

// Top-k of one token by one warp, written to the routing outputs (and to
// the shared-memory copy the fused dispatch reads, when given).
// GROUPED: the selection is group-limited (k_dept departments of g experts
// at most; strict: exactly k_dept).
template <int J, bool GROUPED, bool SMEM = false>
__device__ void topk_warp(const float* logits_row, const float* bias, int n, int k, float scale,
                          int g, int k_dept, bool strict, int32_t* idx_out, float* w_out,
                          int32_t* status, int32_t* idx_sm, float* w_sm) {
    const int lane = threadIdx.x & 31;
    int e;
    float wv;
    const bool bad = GROUPED
                         ? topk_select_warp_grouped<J, SMEM>(logits_row, bias, n, k, g, k_dept, strict, scale, e, wv)
                         : topk_select_warp<J, SMEM>(logits_row, bias, n, k, scale, e, wv);
    if (lane < k) {
        idx_out[lane] = e;
        w_out[lane] = wv;
        if (idx_sm) {
            idx_sm[lane] = e;
            w_sm[lane] = wv;
        }
    }
    if (bad && lane == 0) set_status(status, kDevErrRouting);
}

// Top-k of tokens [t0, t1), one warp per token.  For the group-limited
// selection from 16 keys a lane on, `lsm` (when given) holds the tokens'
// logits in shared memory, row t - t0: a warp's loads from L2 there come
// one round trip after another.
template <int J, bool GROUPED>
__device__ __forceinline__ void topk_rows(const RouteArgs& a, int warp, int t0, int t1, int32_t* idx_sm,
                                          float* w_sm, const float* lsm) {
    for (int t = t0 + warp; t < t1; t += kRouteWarps) {
        int32_t* io = a.topk_idx + (size_t)t * a.k;
        float* wo = a.topk_w + (size_t)t * a.k;
        int32_t* is = idx_sm ? idx_sm + t * a.k : nullptr;
        float* ws_ = idx_sm ? w_sm + t * a.k : nullptr;
        if constexpr (GROUPED && J >= 16) {
            if (lsm) {
                topk_warp<J, GROUPED, true>(lsm + (size_t)(t - t0) * a.n, a.bias, a.n, a.k, a.scale, a.route_g,
                                            a.k_dept, a.strict != 0, io, wo, a.ws.status, is, ws_);
                continue;
            }
        }
        topk_warp<J, GROUPED>(a.ws.logits + (size_t)t * a.n, a.bias, a.n, a.k, a.scale, a.route_g, a.k_dept,
                              a.strict != 0, io, wo, a.ws.status, is, ws_);
    }
}

template <bool GROUPED>
__device__ __forceinline__ void topk_any(const RouteArgs& a, int warp, int t0, int t1, int32_t* idx_sm,
                                         float* w_sm, const float* lsm) {
    const int J = (a.n + 31) / 32;
    if (J <= 1) topk_rows<1, GROUPED>(a, warp, t0, t1, idx_sm, w_sm, nullptr);
    else if (J <= 2) topk_rows<2, GROUPED>(a, warp, t0, t1, idx_sm, w_sm, nullptr);
    else if (J <= 4) topk_rows<4, GROUPED>(a, warp, t0, t1, idx_sm, w_sm, nullptr);
    else if (J <= 8) topk_rows<8, GROUPED>(a, warp, t0, t1, idx_sm, w_sm, nullptr);
    else if (J <= 16) topk_rows<16, GROUPED>(a, warp, t0, t1, idx_sm, w_sm, lsm);
    else topk_rows<32, GROUPED>(a, warp, t0, t1, idx_sm, w_sm, lsm);
}

// Router logits: block (expert group, token block) computes the logits of EB
// experts for 8 tokens; each thread holds RCH float4 chunks of each router
// row, all loaded up front so the rows arrive in one memory round trip, and
// every activation chunk it loads serves the EB experts.  Blocks of one
// expert group are adjacent so that its router rows are read from HBM once
// and then from L2.  Unless only the logits are wanted, the last block to
// finish picks the top-k, one warp per token, and on the whole-layer path
// builds the dispatch lists.  Beyond two token blocks (more tokens than one
// block's warps take in one round) the top-k is split: the last block of
// each token block to finish (a per-token-block counter) picks that block's
// tokens, and the last token block to finish builds the dispatch.
template <int RCH, int EB, bool GROUPED>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteArgs a) {
    __shared__ DispatchSmem sm;
    __shared__ int32_t s_idx[kStagedAssignments];   // top-k results for the fused dispatch
    __shared__ float s_w[kStagedAssignments];
    __shared__ float red[kRouteWarps][8 * EB];
    __shared__ int s_last;
    // Let the FFN grid (launched as a programmatic dependent) start its prologue.
    pdl_allow_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tblocks = (a.T + 7) >> 3;
    const int eg = blockIdx.x / tblocks;
    const int d4 = a.d >> 2;
    // One expert per block: its router row is a layer constant, loaded before
    // the wait below so that the round trip overlaps the previous kernel's
    // last blocks (this grid's blocks take SMs as that kernel's blocks exit).
    float4 w[EB == 1 ? RCH : 1];
    if constexpr (EB == 1) {
        const float4* wr = reinterpret_cast<const float4*>(a.w_router + (size_t)eg * a.d);
#pragma unroll
        for (int i = 0; i < RCH; ++i) {
            const int c = tid + i * kRouteThreads;
            w[i] = c < d4 ? __ldg(wr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    // This grid is itself a programmatic dependent of the kernel before it
    // in the stream (an FFN step of the previous layer, say): its blocks may
    // be resident early, and everything else they read or write waits for
    // that kernel's completion here.
    pdl_wait_primary();

    if (a.split_x == 1)
        split_activations(a.x, (long long)a.T * a.d, a.ws.xb, blockIdx.x * (long long)kRouteThreads + tid,
                          (long long)gridDim.x * kRouteThreads);
    if (a.split_x == 2) {
        // a warp per token
        const int gw = (blockIdx.x * kRouteThreads + tid) >> 5, nw = (gridDim.x * kRouteThreads) >> 5;
        for (int t = gw; t < a.T; t += nw)
            split_e4m3_terms_warp(a.x, a.T, a.d, t, reinterpret_cast<uint8_t*>(a.ws.xb), tid & 31);
    }
    if (a.y_zero) {
        float4* y4 = reinterpret_cast<float4*>(a.y_zero);
        const long long n4 = a.y_elems >> 2;
        for (long long i = blockIdx.x * (long long)kRouteThreads + tid; i < n4;
             i += (long long)gridDim.x * kRouteThreads)
            y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    const int groups = a.n / EB;
    const int tb = blockIdx.x - eg * tblocks;
    const int t0 = tb * 8;
    {
        float acc[8 * EB];
#pragma unroll
        for (int q = 0; q < 8 * EB; ++q) acc[q] = 0.f;
        if constexpr (EB == 1) {
            // one expert: its router chunks were loaded before the wait,
            // then the tokens' activations chunk by chunk
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (t0 + q < a.T) {
                    const float4* xr = reinterpret_cast<const float4*>(a.x + (size_t)(t0 + q) * a.d);
#pragma unroll
                    for (int i = 0; i < RCH; ++i) {
                        const int c = tid + i * kRouteThreads;
                        if (c < d4) {
                            const float4 xv = __ldg(xr + c);
                            acc[q] = fmaf(w[i].x, xv.x, acc[q]);
                            acc[q] = fmaf(w[i].y, xv.y, acc[q]);
                            acc[q] = fmaf(w[i].z, xv.z, acc[q]);
                            acc[q] = fmaf(w[i].w, xv.w, acc[q]);
                        }
                    }
                }
            }
        } else {
            // several experts: chunk by chunk, the EB router chunks and the 8
            // tokens' activation chunks of a step are loaded together, so a
            // wide row costs one round trip per chunk, not per token; per
            // logit the sum runs over the chunks in the same order
#pragma unroll
            for (int i = 0; i < RCH; ++i) {
                const int c = tid + i * kRouteThreads;
                if (c < d4) {
                    float4 wv[EB], xv[8];
#pragma unroll
                    for (int ee = 0; ee < EB; ++ee)
                        wv[ee] = __ldg(reinterpret_cast<const float4*>(a.w_router + (size_t)(eg * EB + ee) * a.d) + c);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        xv[q] = t0 + q < a.T ? __ldg(reinterpret_cast<const float4*>(a.x + (size_t)(t0 + q) * a.d) + c)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
#pragma unroll
                        for (int ee = 0; ee < EB; ++ee) {
                            float& r = acc[ee * 8 + q];
                            r = fmaf(wv[ee].x, xv[q].x, r);
                            r = fmaf(wv[ee].y, xv[q].y, r);
                            r = fmaf(wv[ee].z, xv[q].z, r);
                            r = fmaf(wv[ee].w, xv[q].w, r);
                        }
                }
            }
        }
        int vi;
        const float v = warp_reduce_spread<8 * EB>(acc, lane, vi);
        if ((lane & (32 / (8 * EB) - 1)) == 0) red[warp][vi] = v;
        __syncthreads();
        if (tid < 8 * EB && t0 + (tid & 7) < a.T) {
            float s = 0.f;
#pragma unroll
            for (int w_ = 0; w_ < kRouteWarps; ++w_) s += red[w_][tid];
            a.ws.logits[(size_t)(t0 + (tid & 7)) * a.n + eg * EB + (tid >> 3)] = s;
        }
        __syncthreads();
    }
    if (a.logits_only) return;
    // Count this block in (on its token block when the top-k is split).  The
    // counter add is a GPU-scope release/acquire: it publishes the block's
    // logits (ordered before it by the CTA barrier above) and lets the last
    // block to arrive see every counted block's logits (ordered for its
    // other threads by the barrier below).
    const bool split = tblocks > 2;
    const int ctr = split ? 2 + tb : 2;
    const uint32_t arrivals = (uint32_t)(split ? groups : groups * tblocks);
    if (tid == 0) s_last = atomic_add_acq_rel_gpu(&a.ws.sync[ctr], 1u) == arrivals - 1;
    __syncthreads();
    if (!s_last) return;
    // the fused dispatch reads the top-k results from shared memory when one
    // block picked them all and they fit
    const bool staged = a.fuse_dispatch && !split && a.T * a.k <= kStagedAssignments;
    // Wide group-limited routers: the block first copies the tokens' logits into shared
    // memory (the dispatch's, free until the dispatch starts) in one parallel
    // round trip, so the selecting warps read them from there.
    const int tt0 = split ? t0 : 0, tt1 = split ? min(t0 + 8, a.T) : a.T;
    const float* lsm = nullptr;
    if (GROUPED && a.n > 512 && (tt1 - tt0) * a.n <= kMaxN * kMaskWords) {
        float* st = reinterpret_cast<float*>(sm.emask);
        const float* src = a.ws.logits + (size_t)tt0 * a.n;
        for (int i = tid; i < (tt1 - tt0) * a.n; i += kRouteThreads) st[i] = __ldcg(src + i);
        __syncthreads();
        lsm = st;
    }
    topk_any<GROUPED>(a, warp, tt0, tt1, staged ? s_idx : nullptr, s_w, lsm);
    if (tid == 0) a.ws.sync[ctr] = 0u;  // ready for the next call
    if (!a.fuse_dispatch) return;
    // With a split top-k the last token block to finish builds the dispatch;
    // same ordering argument, one level up, for the other blocks' outputs.
    __syncthreads();
    if (tid == 0) s_last = !split || atomic_add_acq_rel_gpu(&a.ws.sync[0], 1u) == (uint32_t)tblocks - 1;
    __syncthreads();
    if (!s_last) return;
    if (tid == 0) a.ws.sync[0] = 0u;
    dispatch_block<kRouteThreads>(staged ? s_idx : a.topk_idx, staged ? s_w : a.topk_w, a.T, a.n, a.k,
                                  a.g, a.ws, sm);
}

__global__ void __launch_bounds__(kDispatchThreads) dispatch_kernel(DispatchArgs a) {
    __shared__ DispatchSmem sm;
    dispatch_block<kDispatchThreads>(a.topk_idx, a.topk_w, a.T, a.n, a.k, a.g, a.ws, sm);
}

}  // namespace

// The group-limited selection is its own instantiation, which leaves the
// plain kernel's registers as they are.
template <int EB, bool GROUPED>
cudaError_t launch_route_eb(const RouteArgs& a, int rch, int blocks, cudaStream_t s) {
    auto kern = rch <= 1 ? route_kernel<1, EB, GROUPED> : rch <= 2 ? route_kernel<2, EB, GROUPED>
                                                                   : route_kernel<4, EB, GROUPED>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kRouteThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = MOE_ROUTE_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
    // float4 chunks of a router row per thread: ceil(d / 4 / threads)
    const int rch = (a.d / 4 + kRouteThreads - 1) / kRouteThreads;
    const int tblocks = (a.T + 7) / 8;
    // from four token blocks on, 4 experts per block so that each activation
    // chunk serves 4; below, one expert per block for parallelism, unless
    // that would take more than one wave of blocks (a 512-thread block holds
    // its SM's registers alone): from 256 experts on, 4 per block
    const int eb = a.n % 4 == 0 && (tblocks >= 4 || a.n >= 256) ? 4 : 1;
    const bool grouped = a.k_dept > 0 && !a.logits_only;
    if (eb == 4) return grouped ? launch_route_eb<4, true>(a, rch, a.n / 4 * tblocks, s)
                                : launch_route_eb<4, false>(a, rch, a.n / 4 * tblocks, s);
    return grouped ? launch_route_eb<1, true>(a, rch, a.n * tblocks, s)
                   : launch_route_eb<1, false>(a, rch, a.n * tblocks, s);
}

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s) {
    dispatch_kernel<<<1, kDispatchThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
