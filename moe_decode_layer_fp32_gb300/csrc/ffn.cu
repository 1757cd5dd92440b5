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
// split evenly over one CTA per SM.  A producer warp streams each CTA's rows
// (gate, up, then down; every row is contiguous) from HBM into a 12-stage
// shared-memory ring with bulk copies (cp.async.bulk + mbarrier transaction
// counts).  Consumer warps own fixed 8-column chunks of the hidden dimension:
// the gate/up dot products are reduced across the warp and then across warps
// with shared atomics, the SwiGLU is applied in shared memory, and the down
// projection accumulates each thread's columns in registers.  The partial
// output of the CTA's rows is added into the output with vector atomics.
#include <cuda_bf16.h>

#include "../../include/moe_decode.h"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kStageBytes = 16384;   // one ring slot
constexpr int kStages = 12;          // 192 KB of weights in flight per SM
constexpr int kMT = 4;               // tokens per group (register tile)
constexpr int kSegMax = 256;         // rows per segment (gate/up/h buffers)
constexpr int kMaxUnits = 1 + 2 * kMaxN;  // shared + two per-expert classes

template <typename WT>
struct WLoad;
template <>
struct WLoad<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    __device__ static __forceinline__ void load8(const char* p, float (&f)[8]) {
        unpack_bf16x8(*reinterpret_cast<const uint4*>(p), f);
    }
};
template <>
struct WLoad<float> {
    static constexpr int kBytes = 4;
    __device__ static __forceinline__ void load8(const char* p, float (&f)[8]) {
        const float4 a = reinterpret_cast<const float4*>(p)[0];
        const float4 b = reinterpret_cast<const float4*>(p)[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
};

// Shared-memory carve-up (after the ring).
struct FfnSmem {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    float gu[2][kSegMax * kMT];       // gate / up pre-activations of the segment
    float h[kSegMax * kMT];           // SwiGLU output (times the token weight)
    int gpre[kMaxUnits];              // per class: inclusive prefix of groups
    int cls_units[3];
    int cls_groups[3];
    int cls_off[3];                   // offset of the class's entries in gpre
    int warp_tmp[32];
};

// A segment: rows [row0, row0+nrows) of one token group of one unit.
struct Seg {
    int cls, q, grp, row0, nrows;
};

__device__ __forceinline__ int unit_tokens(const FfnArgs& a, int cls, int q) {
    const UnitClass& c = a.cls[cls];
    if (c.kind == kUnitShared) return a.T;
    if (c.kind == kUnitDept) return a.ws.dept_count[a.ws.act_dept[q]];
    return a.ws.exp_count[a.ws.act_exp[q]];
}

// Next segment of [r, r_end) in the class / unit / group / row order.
__device__ __forceinline__ bool next_seg(const FfnArgs& a, const FfnSmem& sm, long long& r,
                                         long long r_end, Seg& s) {
    if (r >= r_end) return false;
    long long base = 0;
    int c = 0;
    while (c < a.ncls - 1 && r >= base + (long long)a.cls[c].rows * sm.cls_groups[c]) {
        base += (long long)a.cls[c].rows * sm.cls_groups[c];
        ++c;
    }
    const int rows = a.cls[c].rows;
    const long long rel = r - base;
    const int vg = (int)(rel / rows);
    const int rin = (int)(rel - (long long)vg * rows);
    const int* gp = sm.gpre + sm.cls_off[c];
    int lo = 0, hi = sm.cls_units[c] - 1;  // first q with gp[q] > vg
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (gp[mid] > vg) hi = mid; else lo = mid + 1;
    }
    s.cls = c;
    s.q = lo;
    s.grp = vg - (lo > 0 ? gp[lo - 1] : 0);
    s.row0 = rin;
    long long n = rows - rin;
    if (n > r_end - r) n = r_end - r;
    if (n > kSegMax) n = kSegMax;
    s.nrows = (int)n;
    r += n;
    return true;
}

__device__ __forceinline__ int unit_weight_index(const FfnArgs& a, int cls, int q) {
    const int kind = a.cls[cls].kind;
    if (kind == kUnitShared) return 0;
    if (kind == kUnitDept) return a.ws.act_dept[q];
    return a.ws.act_exp[q];
}

// Tokens of a group: token id, weight and output row (ROWS or ACCUM mode).
__device__ __forceinline__ int group_tokens(const FfnArgs& a, const Seg& s, int (&tok)[kMT],
                                            float (&wt)[kMT], int (&orow)[kMT]) {
    const int kind = a.cls[s.cls].kind;
    int base, count;
    if (kind == kUnitShared) {
        base = 0;
        count = a.T;
    } else if (kind == kUnitDept) {
        const int j = a.ws.act_dept[s.q];
        base = a.ws.dept_off[j];
        count = a.ws.dept_count[j];
    } else {
        const int e = a.ws.act_exp[s.q];
        base = a.ws.exp_off[e];
        count = a.ws.exp_count[e];
    }
    const int first = s.grp * kMT;
    const int mg = min(kMT, count - first);
#pragma unroll
    for (int i = 0; i < kMT; ++i) {
        tok[i] = 0;
        wt[i] = 0.0f;
        orow[i] = 0;
        if (i < mg) {
            const int p = base + first + i;
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
            tok[i] = t;
            wt[i] = w;
            orow[i] = a.out_mode == MOE_OUT_ACCUM ? t : row;
        }
    }
    return mg;
}

// Reduce V values across the warp; afterwards the lanes whose low
// (5 - log2 V) bits are zero hold the full sum of value index `vi`.
template <int V>
__device__ __forceinline__ float warp_reduce_spread(float (&v)[V], int lane, int& vi) {
    int cnt = V;
    vi = 0;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (cnt > 1) {
            const int half = cnt >> 1;
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < half) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            if (upper) vi += half;
            cnt = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        }
    }
    return v[0];
}

template <typename WT, int NCW, int CH, int RMAX>
struct Ffn {
    static constexpr int kNT = (NCW + 1) * 32;
    static constexpr int kNC = NCW * 32;      // consumer threads
    static constexpr int kBw = WLoad<WT>::kBytes;

    // One gate or up stage: nr rows of one matrix against MTC tokens.
    template <int MTC>
    __device__ static __forceinline__ void gu_stage(const char* stage, int nr, int row_bytes,
                                                    int ctid, int nchunks,
                                                    const float (&xr)[CH][kMT][8],
                                                    float* gu_rows, int mg, int lane) {
        float acc[RMAX][MTC];
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
#pragma unroll
            for (int m = 0; m < MTC; ++m) acc[r][m] = 0.0f;
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            if (r < nr) {
#pragma unroll
                for (int j = 0; j < CH; ++j) {
                    const int c = ctid + j * kNC;
                    if (c < nchunks) {
                        float w8[8];
                        WLoad<WT>::load8(stage + (size_t)r * row_bytes + (size_t)c * 8 * kBw, w8);
#pragma unroll
                        for (int m = 0; m < MTC; ++m)
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[r][m] = fmaf(w8[e], xr[j][m][e], acc[r][m]);
                    }
                }
            }
        }
        constexpr int V = RMAX * MTC;
        float v[V];
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
#pragma unroll
            for (int m = 0; m < MTC; ++m) v[r * MTC + m] = acc[r][m];
        int vi;
        const float sum = warp_reduce_spread<V>(v, lane, vi);
        if ((lane & (32 / V - 1)) == 0) {
            const int r = vi / MTC, m = vi - (vi / MTC) * MTC;
            if (r < nr && m < mg) atomicAdd(&gu_rows[r * kMT + m], sum);
        }
    }

    // One down stage: y[col] += W_down[row, col] * h[row, token].
    template <int MTC>
    __device__ static __forceinline__ void down_stage(const char* stage, int nr, int row_bytes,
                                                      int ctid, int nchunks, const float* h_rows,
                                                      float (&yacc)[CH][kMT][8]) {
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            if (r < nr) {
                const float4 hv4 = *reinterpret_cast<const float4*>(h_rows + r * kMT);
                const float hv[4] = {hv4.x, hv4.y, hv4.z, hv4.w};
#pragma unroll
                for (int j = 0; j < CH; ++j) {
                    const int c = ctid + j * kNC;
                    if (c < nchunks) {
                        float w8[8];
                        WLoad<WT>::load8(stage + (size_t)r * row_bytes + (size_t)c * 8 * kBw, w8);
#pragma unroll
                        for (int m = 0; m < MTC; ++m)
#pragma unroll
                            for (int e = 0; e < 8; ++e) yacc[j][m][e] = fmaf(w8[e], hv[m], yacc[j][m][e]);
                    }
                }
            }
        }
    }
};

template <typename WT, int NCW, int CH, int RMAX>
__global__ void __launch_bounds__((NCW + 1) * 32, 1) ffn_stream_kernel(FfnArgs a) {
    using K = Ffn<WT, NCW, CH, RMAX>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char* ring = smem_raw;
    FfnSmem& sm = *reinterpret_cast<FfnSmem*>(smem_raw + (size_t)kStages * kStageBytes);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], NCW);
        }
        mbar_init_fence();
    }
    for (int i = tid; i < 2 * kSegMax * kMT; i += K::kNT) (&sm.gu[0][0])[i] = 0.0f;

    // Everything below reads what the routing / dispatch kernel wrote.
    pdl_wait_primary();

    // ---- unit tables: groups per unit, prefix-summed per class ----
    int off = 0;
    for (int c = 0; c < a.ncls; ++c) {
        const UnitClass& uc = a.cls[c];
        const int units = uc.kind == kUnitShared ? 1
                          : uc.kind == kUnitDept ? a.ws.counts[1]
                                                 : a.ws.counts[0];
        for (int q = tid; q < units; q += K::kNT)
            sm.gpre[off + q] = (unit_tokens(a, c, q) + kMT - 1) / kMT;
        __syncthreads();
        const int total = block_exclusive_scan<K::kNT>(sm.gpre + off, units, sm.warp_tmp);
        // exclusive -> inclusive prefix
        for (int q = tid; q < units; q += K::kNT)
            sm.gpre[off + q] += (unit_tokens(a, c, q) + kMT - 1) / kMT;
        if (tid == 0) {
            sm.cls_units[c] = units;
            sm.cls_groups[c] = total;
            sm.cls_off[c] = off;
        }
        off += units;
        __syncthreads();
    }
    long long R = 0;
    for (int c = 0; c < a.ncls; ++c) R += (long long)a.cls[c].rows * sm.cls_groups[c];
    const long long r_begin = R * blockIdx.x / gridDim.x;
    const long long r_end = R * (blockIdx.x + 1) / gridDim.x;

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
                const int slot = it % kStages;
                const uint32_t par = ((it / kStages) & 1u) ^ 1u;
                if (!mbar_wait_bounded(&sm.empty[slot], par)) return false;
                const uint32_t bytes = (uint32_t)nr * row_bytes;
                mbar_arrive_expect_tx(&sm.full[slot], bytes);
                bulk_load(ring + (size_t)slot * kStageBytes, src, bytes, &sm.full[slot], pol);
                ++it;
                return true;
            };
            while (ok && next_seg(a, sm, r, r_end, s)) {
                const UnitClass& uc = a.cls[s.cls];
                const size_t ubase = ((size_t)unit_weight_index(a, s.cls, s.q) * uc.rows + s.row0) *
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
            const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0u;
            for (uint32_t i = first; i < it; ++i)
                mbar_wait_bounded(&sm.full[i % kStages], (i / kStages) & 1u);
        }
        return;
    }

    // ===================== consumers =====================
    const int ctid = tid;  // 0 .. kNC-1
    uint32_t it = 0;
    long long r = r_begin;
    Seg s;
    bool ok = true;
    auto wait_full = [&](int slot, uint32_t i) -> bool {
        if (!ok) return false;
        if (!mbar_wait_bounded(&sm.full[slot], (i / kStages) & 1u)) {
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
        const int mg = group_tokens(a, s, tok, wt, orow);

        // ---- phase A: gate / up dot products ----
        {
            float xr[CH][kMT][8];
#pragma unroll
            for (int j = 0; j < CH; ++j) {
                const int c = ctid + j * K::kNC;
#pragma unroll
                for (int m = 0; m < kMT; ++m) {
                    if (c < nchunks && m < mg) {
                        const float4* xp =
                            reinterpret_cast<const float4*>(a.x + (size_t)tok[m] * a.d + c * 8);
                        const float4 lo = __ldg(xp), hi = __ldg(xp + 1);
                        xr[j][m][0] = lo.x; xr[j][m][1] = lo.y; xr[j][m][2] = lo.z; xr[j][m][3] = lo.w;
                        xr[j][m][4] = hi.x; xr[j][m][5] = hi.y; xr[j][m][6] = hi.z; xr[j][m][7] = hi.w;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) xr[j][m][e] = 0.0f;
                    }
                }
            }
            for (int rb = 0; rb < s.nrows; rb += rps) {
                const int nr = min(rps, s.nrows - rb);
#pragma unroll 1
                for (int mat = 0; mat < 2; ++mat) {
                    const int slot = it % kStages;
                    if (wait_full(slot, it)) {
                        const char* st = reinterpret_cast<const char*>(ring + (size_t)slot * kStageBytes);
                        float* gr = &sm.gu[mat][rb * kMT];
                        if (mg == 1)
                            K::template gu_stage<1>(st, nr, row_bytes, ctid, nchunks, xr, gr, mg, lane);
                        else if (mg == 2)
                            K::template gu_stage<2>(st, nr, row_bytes, ctid, nchunks, xr, gr, mg, lane);
                        else
                            K::template gu_stage<4>(st, nr, row_bytes, ctid, nchunks, xr, gr, mg, lane);
                        release(slot);
                    }
                    ++it;
                }
            }
        }
        // every consumer leaves the barrier with the same abort decision
        if (named_bar_or(1, K::kNC, !ok)) break;

        // ---- SwiGLU: h = SiLU(g) * u (times the token's weight when accumulating) ----
        for (int i = ctid; i < s.nrows * kMT; i += K::kNC) {
            const int m = i & (kMT - 1);
            float hv = 0.0f;
            if (m < mg) {
                hv = silu_f(sm.gu[0][i]) * sm.gu[1][i];
                if (a.out_mode == MOE_OUT_ACCUM)
                    hv *= m == 0 ? wt[0] : m == 1 ? wt[1] : m == 2 ? wt[2] : wt[3];
            }
            sm.h[i] = hv;
            sm.gu[0][i] = 0.0f;
            sm.gu[1][i] = 0.0f;
        }
        named_bar_sync(1, K::kNC);

        // ---- phase B: down projection into per-thread column accumulators ----
        float yacc[CH][kMT][8];
#pragma unroll
        for (int j = 0; j < CH; ++j)
#pragma unroll
            for (int m = 0; m < kMT; ++m)
#pragma unroll
                for (int e = 0; e < 8; ++e) yacc[j][m][e] = 0.0f;
        for (int rb = 0; rb < s.nrows; rb += rps) {
            const int nr = min(rps, s.nrows - rb);
            const int slot = it % kStages;
            if (wait_full(slot, it)) {
                const char* st = reinterpret_cast<const char*>(ring + (size_t)slot * kStageBytes);
                const float* hr = &sm.h[rb * kMT];
                if (mg == 1)
                    K::template down_stage<1>(st, nr, row_bytes, ctid, nchunks, hr, yacc);
                else if (mg == 2)
                    K::template down_stage<2>(st, nr, row_bytes, ctid, nchunks, hr, yacc);
                else
                    K::template down_stage<4>(st, nr, row_bytes, ctid, nchunks, hr, yacc);
                release(slot);
            }
            ++it;
        }
        if (named_bar_or(1, K::kNC, !ok)) break;
        // ---- add this CTA's partial rows into the output ----
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const int c = ctid + j * K::kNC;
            if (c < nchunks) {
#pragma unroll
                for (int m = 0; m < kMT; ++m) {
                    if (m < mg) {
                        float4* dst = reinterpret_cast<float4*>(a.out + (size_t)orow[m] * a.d + c * 8);
                        atomicAdd(dst, make_float4(yacc[j][m][0], yacc[j][m][1], yacc[j][m][2], yacc[j][m][3]));
                        atomicAdd(dst + 1, make_float4(yacc[j][m][4], yacc[j][m][5], yacc[j][m][6], yacc[j][m][7]));
                    }
                }
            }
        }
    }
}

template <typename WT, int NCW, int CH, int RMAX>
cudaError_t launch_ffn_t(const FfnArgs& a, cudaStream_t s) {
    auto kern = ffn_stream_kernel<WT, NCW, CH, RMAX>;
    const size_t smem = (size_t)kStages * kStageBytes + sizeof(FfnSmem);
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(device_sm_count(), 1, 1);
    cfg.blockDim = dim3((NCW + 1) * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
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

__global__ void zero_kernel(uint4* p, size_t n16) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16;
         i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

cudaError_t launch_ffn(const FfnArgs& a, cudaStream_t s) {
    // Consumer warps x chunks per thread must cover d/8 chunks; RMAX is the
    // most rows one 16 KB stage holds at that width.
    // (15 consumer warps + 1 producer = 512 threads keeps a 128-register cap.)
    if (a.dtype == MOE_DTYPE_BF16) {
        if (a.d <= 2048) return launch_ffn_t<__nv_bfloat16, 8, 1, 4>(a, s);
        return launch_ffn_t<__nv_bfloat16, 15, 2, 1>(a, s);
    }
    if (a.d <= 1024) return launch_ffn_t<float, 4, 1, 8>(a, s);
    return launch_ffn_t<float, 15, 2, 1>(a, s);
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
