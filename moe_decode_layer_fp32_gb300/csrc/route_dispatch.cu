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

constexpr int kRouteWarps = 4;
constexpr int kRouteThreads = kRouteWarps * 32;
constexpr int kDispatchThreads = 256;
constexpr int kMaskWords = (kMaxT + 31) / 32;

struct DispatchSmem {
    uint32_t emask[kMaxN * kMaskWords];       // expert -> token bitmask
    uint32_t dmask[(kMaxN / 2) * kMaskWords]; // department -> token bitmask
    int cnt[kMaxN + 1];
    int act[kMaxN + 1];
    int warp_tmp[32];
    int err;
};

// Rank of token t among the tokens set in a mask row (tokens ascending).
__device__ __forceinline__ int mask_rank(const uint32_t* row, int t) {
    int r = __popc(row[t >> 5] & ((1u << (t & 31)) - 1u));
    for (int w = 0; w < (t >> 5); ++w) r += __popc(row[w]);
    return r;
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
    if (tid == 0) sm.err = 0;
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
        }
        return;
    }
    // ---- experts ----
    for (int e = tid; e < n; e += NT) {
        int c = 0;
        for (int w = 0; w < W; ++w) c += __popc(sm.emask[e * W + w]);
        sm.cnt[e] = c;
        sm.act[e] = c > 0 ? 1 : 0;
        ws.exp_count[e] = c;
    }
    __syncthreads();
    const int total = block_exclusive_scan<NT>(sm.cnt, n, sm.warp_tmp);
    const int A_e = block_exclusive_scan<NT>(sm.act, n, sm.warp_tmp);
    for (int e = tid; e < n; e += NT) {
        ws.exp_off[e] = sm.cnt[e];
        const bool active = (e + 1 < n ? sm.act[e + 1] : A_e) != sm.act[e];
        if (active) ws.act_exp[sm.act[e]] = e;
    }
    if (tid == 0) {
        ws.exp_off[n] = total;
        ws.counts[0] = A_e;
    }
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
        if (tid == 0) ws.counts[1] = 0;
        return;
    }
    // ---- departments: X^j = tokens that chose any expert of department j ----
    const int m = n / g;
    for (int i = tid; i < m * W; i += NT) {
        const int j = i / W, w = i - (i / W) * W;
        uint32_t v = 0u;
        for (int e = j * g; e < (j + 1) * g; ++e) v |= sm.emask[e * W + w];
        sm.dmask[i] = v;
    }
    __syncthreads();
    for (int j = tid; j < m; j += NT) {
        int c = 0;
        for (int w = 0; w < W; ++w) c += __popc(sm.dmask[j * W + w]);
        sm.cnt[j] = c;
        sm.act[j] = c > 0 ? 1 : 0;
        ws.dept_count[j] = c;
    }
    __syncthreads();
    const int dtotal = block_exclusive_scan<NT>(sm.cnt, m, sm.warp_tmp);
    const int A_d = block_exclusive_scan<NT>(sm.act, m, sm.warp_tmp);
    for (int j = tid; j < m; j += NT) {
        ws.dept_off[j] = sm.cnt[j];
        const bool active = (j + 1 < m ? sm.act[j + 1] : A_d) != sm.act[j];
        if (active) ws.act_dept[sm.act[j]] = j;
    }
    if (tid == 0) {
        ws.dept_off[m] = dtotal;
        ws.counts[1] = A_d;
    }
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

// Top-k of one token's keys (logit + bias) by one warp; lane holds experts
// lane + 32*j.  Descending key, equal keys -> lower expert index first.  The
// weights are scale * softmax over the selected unbiased logits.
template <int J>
__device__ void topk_warp(const float* logits_row, const float* bias, int n, int k, float scale,
                          int32_t* idx_out, float* w_out, int32_t* status) {
    const int lane = threadIdx.x & 31;
    float key[J], lg[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        if (e < n) {
            const float l = __ldcg(logits_row + e);
            lg[j] = l;
            key[j] = bias ? l + __ldg(bias + e) : l;
        } else {
            lg[j] = 0.0f;
            key[j] = -INFINITY;
        }
    }
    uint32_t taken = 0u;
    int my_idx = 0;
    float my_lg = 0.0f;
    bool bad = false;
    for (int r = 0; r < k; ++r) {
        float bk = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            if (e < n && !((taken >> j) & 1u)) {
                if (key[j] > bk || (key[j] == bk && e < bi)) {
                    bk = key[j];
                    bi = e;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ok > bk || (ok == bk && oi < bi)) {
                bk = ok;
                bi = oi;
            }
        }
        if (bi == INT_MAX) {  // only non-finite keys left
            bad = true;
            bi = 0;
        }
        const int owner = bi & 31, jb = bi >> 5;
        float v = 0.0f;
#pragma unroll
        for (int j = 0; j < J; ++j)
            if (j == jb) v = lg[j];
        if (lane == owner) taken |= 1u << jb;
        v = __shfl_sync(0xffffffffu, v, owner);
        if (lane == r) {
            my_idx = bi;
            my_lg = v;
        }
    }
    float mx = lane < k ? my_lg : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float ex = lane < k ? expf(my_lg - mx) : 0.0f;
    const float s = warp_sum(ex);
    if (lane < k) {
        idx_out[lane] = my_idx;
        w_out[lane] = scale * (ex / s);
    }
    if (bad && lane == 0) set_status(status, kDevErrRouting);
}

// Router logits: warp w of block b computes expert b*4+w for every token.
// The last block to finish picks the top-k of every token and, on the
// whole-layer path, builds the dispatch lists.
template <int J>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteArgs a) {
    __shared__ DispatchSmem sm;
    __shared__ int s_last;
    // Let the FFN grid (launched as a programmatic dependent) start its prologue.
    pdl_allow_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (a.y_zero) {
        float4* y4 = reinterpret_cast<float4*>(a.y_zero);
        const long long n4 = a.y_elems >> 2;
        for (long long i = blockIdx.x * (long long)kRouteThreads + tid; i < n4;
             i += (long long)gridDim.x * kRouteThreads)
            y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    const int e = blockIdx.x * kRouteWarps + warp;
    if (e < a.n) {
        const float4* wr = reinterpret_cast<const float4*>(a.w_router + (size_t)e * a.d);
        const int d4 = a.d >> 2;
        for (int t0 = 0; t0 < a.T; t0 += 8) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
            for (int c = lane; c < d4; c += 32) {
                const float4 wv = __ldg(wr + c);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (t0 + i < a.T) {
                        const float4 xv =
                            __ldg(reinterpret_cast<const float4*>(a.x + (size_t)(t0 + i) * a.d) + c);
                        acc[i] = fmaf(wv.x, xv.x, acc[i]);
                        acc[i] = fmaf(wv.y, xv.y, acc[i]);
                        acc[i] = fmaf(wv.z, xv.z, acc[i]);
                        acc[i] = fmaf(wv.w, xv.w, acc[i]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float v = warp_sum(acc[i]);
                if (lane == 0 && t0 + i < a.T) a.ws.logits[(size_t)(t0 + i) * a.n + e] = v;
            }
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&a.ws.sync[0], 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int t = warp; t < a.T; t += kRouteWarps)
        topk_warp<J>(a.ws.logits + (size_t)t * a.n, a.bias, a.n, a.k, a.scale,
                     a.topk_idx + (size_t)t * a.k, a.topk_w + (size_t)t * a.k, a.ws.status);
    if (tid == 0) a.ws.sync[0] = 0u;  // ready for the next call
    if (a.fuse_dispatch) {
        __syncthreads();
        dispatch_block<kRouteThreads>(a.topk_idx, a.topk_w, a.T, a.n, a.k, a.g, a.ws, sm);
    }
}

__global__ void __launch_bounds__(kDispatchThreads) dispatch_kernel(DispatchArgs a) {
    __shared__ DispatchSmem sm;
    dispatch_block<kDispatchThreads>(a.topk_idx, a.topk_w, a.T, a.n, a.k, a.g, a.ws, sm);
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
    const int blocks = (a.n + kRouteWarps - 1) / kRouteWarps;
    const int J = (a.n + 31) / 32;
    if (J <= 1) route_kernel<1><<<blocks, kRouteThreads, 0, s>>>(a);
    else if (J <= 2) route_kernel<2><<<blocks, kRouteThreads, 0, s>>>(a);
    else if (J <= 4) route_kernel<4><<<blocks, kRouteThreads, 0, s>>>(a);
    else if (J <= 8) route_kernel<8><<<blocks, kRouteThreads, 0, s>>>(a);
    else if (J <= 16) route_kernel<16><<<blocks, kRouteThreads, 0, s>>>(a);
    else route_kernel<32><<<blocks, kRouteThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s) {
    dispatch_kernel<<<1, kDispatchThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
