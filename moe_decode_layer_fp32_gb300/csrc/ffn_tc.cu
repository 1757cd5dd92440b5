// Expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM), for units
// whose gathered token count makes the contraction dense enough.
//
// Same computation as the CUDA-core stream (ffn.cu): for each unit u (shared
// expert, department backbone, expert rows) and its tokens X_u,
//     Y_u = W_down^T ( SiLU(W_gate X_u) * (W_up X_u) ),
// the SwiGLU expert of "DeaMoE: Efficient MoE Structure for Fast Small-Batch
// Decoding" §2.1 eq. (1); a department backbone runs once over its token set
// X^j (two-stage routing, §3.2).
//
// Mapping onto the MMA (D[M x N] = A[M x K] * B[N x K]^T, fp32 accumulate):
//  * gate/up: A = a tile of <= 64 weight rows (K-major, 128 B swizzle, loaded
//    by TMA in 16-row boxes), B = the tokens' activations, N = tokens;
//  * down:    A = W_down rows of the same tile read as an MN-major operand
//    (M = 128 hidden columns, K = the tile's rows), B = H = SiLU(g) * u.
// Activations and H are split into bf16 hi + lo parts (x = hi + lo up to
// 2^-17 relative), so the products keep close to fp32 accuracy: each token
// occupies two B rows and the epilogue adds the two result columns.
//
// Warp roles (one CTA per SM): warp 0 issues TMA loads of weight tiles into an
// 8-stage ring; warp 1 issues the MMAs (one thread) and owns the TMEM
// allocation; warps 2-5 are the epilogue (TMEM -> registers, SwiGLU, H tile,
// output atomics); warps 6-9 convert activations into swizzled bf16 B tiles.
// Every wait is bounded; on a timeout the kernel records an error status,
// drains its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include "../../include/moe_decode.h"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kTcStages = 8;
constexpr int kTcRows = 64;                 // weight rows per tile
constexpr int kTcTokens = 32;               // tokens per group (hi + lo rows: N <= 64)
constexpr int kTcMaxN = 2 * kTcTokens;
constexpr int kAStage = 16384;              // gate+up tiles, or one down tile (2 halves)
constexpr int kBStage = kTcMaxN * 128;      // activation tile: N rows x 64 bf16
constexpr int kHTile = kTcMaxN * 128;       // H tile: N rows x (K <= 64) bf16
constexpr int kTmemCols = 256;
constexpr uint32_t kColG = 0, kColU = 64, kColY0 = 128, kColY1 = 192;
constexpr int kTcWarps = 10;
constexpr int kTcThreads = kTcWarps * 32;

struct TcSmem {
    uint64_t full[kTcStages];     // producer TMA bytes landed (weight ring)
    uint64_t empty[kTcStages];    // MMAs reading the weight stage are done
    uint64_t bx_full[kTcStages];  // converter wrote the activation tile (own ring)
    uint64_t bx_empty[kTcStages]; // MMAs reading the activation tile are done
    uint64_t acc_full, acc_empty, h_full, mma_done;
    uint64_t y_full[2], y_empty[2];
    uint32_t tmem_base;
    int cls_units[3];
    int cls_groups[3];
    int cls_off[3];
    int4 units[1];                // per class: {unit, first entry, tokens, group prefix}
};

struct TSeg {
    int cls, q, grp, row0, nrows;
};

// Next tile of the CTA's row range [r, r_end) (rows; tiles <= kTcRows).
__device__ __forceinline__ bool next_tile(const TcArgs& a, const TcSmem& sm, int& r, int r_end,
                                          TSeg& s) {
    if (r >= r_end) return false;
    int base = 0, c = 0;
    while (c < a.f.ncls - 1 && r >= base + a.f.cls[c].rows * sm.cls_groups[c]) {
        base += a.f.cls[c].rows * sm.cls_groups[c];
        ++c;
    }
    const int rows = a.f.cls[c].rows;
    const int rel = r - base;
    const int vg = rel / rows;
    const int rin = rel - vg * rows;
    const int4* u = sm.units + sm.cls_off[c];
    int lo = 0, hi = sm.cls_units[c] - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (u[mid].w > vg) hi = mid; else lo = mid + 1;
    }
    s.cls = c;
    s.q = lo;
    s.grp = vg - (lo > 0 ? u[lo - 1].w : 0);
    s.row0 = rin;
    s.nrows = min(min(rows - rin, r_end - r), kTcRows);
    r += s.nrows;
    return true;
}

// Token t, routing weight and output row of entry j of a unit's token list.
__device__ __forceinline__ void tile_token(const TcArgs& a, int kind, int entry, int& t,
                                           float& w, int& row) {
    if (kind == kUnitShared) {
        t = entry;
        w = 1.0f;
        row = a.f.rows_shared_base + entry;
    } else if (kind == kUnitDept) {
        t = a.f.ws.dept_tok[entry];
        w = a.f.ws.dept_w[entry];
        row = a.f.rows_dept_base + entry;
    } else {
        t = a.f.ws.asg_tok[entry];
        w = a.f.ws.asg_w[entry];
        row = entry;
    }
    if (a.f.out_mode == MOE_OUT_ACCUM) row = t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

__global__ void __launch_bounds__(kTcThreads, 1) ffn_tc_kernel(const __grid_constant__ TcArgs a) {
    extern __shared__ unsigned char smem_dyn[];
    // 1024-byte aligned tile regions (128 B swizzle atoms)
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    unsigned char* aring = base;
    unsigned char* bring = aring + kTcStages * kAStage;
    unsigned char* htile = bring + kTcStages * kBStage;
    TcSmem& sm = *reinterpret_cast<TcSmem*>(htile + kHTile);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.f.d;
    const int KB = d / 64, DT = d / 128;

    if (tid == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
            mbar_init(&sm.bx_full[i], 4);
            mbar_init(&sm.bx_empty[i], 1);
        }
        mbar_init(&sm.acc_full, 1);
        mbar_init(&sm.acc_empty, 4);
        mbar_init(&sm.h_full, 4);
        mbar_init(&sm.mma_done, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.y_full[b], 1);
            mbar_init(&sm.y_empty[b], 4);
        }
        mbar_init_fence();
    }
    if (warp == 0 && lane == 0) {
        for (int c = 0; c < a.f.ncls; ++c)
            for (int m = 0; m < 3; ++m) tma_prefetch_map(&a.maps[c][m]);
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;

    // Everything below reads what the routing / dispatch kernel wrote.
    pdl_wait_primary();

    // ---- unit table: this kernel's units (>= min_tokens tokens), groups of kTcTokens ----
    if (warp == 0) {
        int off = 0;
        for (int c = 0; c < a.f.ncls; ++c) {
            const UnitClass& uc = a.f.cls[c];
            int kept, groups;
            if (uc.kind == kUnitShared) {
                const bool keep = a.f.T >= a.min_tokens;
                kept = keep ? 1 : 0;
                groups = keep ? (a.f.T + kTcTokens - 1) / kTcTokens : 0;
                if (lane == 0 && keep) sm.units[off] = make_int4(0, 0, a.f.T, groups);
            } else {
                const int4* src = uc.kind == kUnitDept ? a.f.ws.dept_units : a.f.ws.exp_units;
                const int A = uc.kind == kUnitDept ? a.f.ws.counts[1] : a.f.ws.counts[0];
                kept = filter_units_warp(src, A, a.min_tokens, 1 << 30, kTcTokens, sm.units + off,
                                         &groups);
            }
            if (lane == 0) {
                sm.cls_units[c] = kept;
                sm.cls_groups[c] = groups;
                sm.cls_off[c] = off;
            }
            off += class_capacity(uc, a.f.n, a.f.g);
        }
    }
    __syncthreads();

    // CTA's share of the row space, in 16-row quanta
    int Q = 0;
    for (int c = 0; c < a.f.ncls; ++c) Q += a.f.cls[c].rows / 16 * sm.cls_groups[c];
    const int r_begin = (int)((long long)Q * blockIdx.x / gridDim.x) * 16;
    const int r_end = (int)((long long)Q * (blockIdx.x + 1) / gridDim.x) * 16;

    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (!ok) return false;
        if (!mbar_wait_bounded(bar, parity)) {
            ok = false;
            set_status(a.f.ws.status, kDevErrTimeout);
        }
        return ok;
    };

    if (warp == 0) {
        // ===================== TMA producer =====================
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            uint32_t it = 0;
            int r = r_begin;
            TSeg s;
            while (ok && next_tile(a, sm, r, r_end, s)) {
                const int4 rec = sm.units[sm.cls_off[s.cls] + s.q];
                const int ybase = rec.x * a.f.cls[s.cls].rows + s.row0;
                const int nq = s.nrows / 16;
                const uint32_t bytes = (uint32_t)s.nrows * 128u * 2u;
                const CUtensorMap* mg = &a.maps[s.cls][0];
                const CUtensorMap* mu = &a.maps[s.cls][1];
                const CUtensorMap* md = &a.maps[s.cls][2];
                for (int kb = 0; ok && kb < KB; ++kb, ++it) {
                    const int slot = it % kTcStages;
                    if (!wait(&sm.empty[slot], ((it / kTcStages) & 1u) ^ 1u)) break;
                    mbar_arrive_expect_tx(&sm.full[slot], bytes);
                    unsigned char* A = aring + slot * kAStage;
                    for (int q = 0; q < nq; ++q) {
                        tma_load_2d(A + q * 2048, mg, kb * 64, ybase + q * 16, &sm.full[slot], pol);
                        tma_load_2d(A + 8192 + q * 2048, mu, kb * 64, ybase + q * 16, &sm.full[slot], pol);
                    }
                }
                for (int dt = 0; ok && dt < DT; ++dt, ++it) {
                    const int slot = it % kTcStages;
                    if (!wait(&sm.empty[slot], ((it / kTcStages) & 1u) ^ 1u)) break;
                    mbar_arrive_expect_tx(&sm.full[slot], bytes);
                    unsigned char* A = aring + slot * kAStage;
                    for (int h = 0; h < 2; ++h)
                        for (int q = 0; q < nq; ++q)
                            tma_load_2d(A + h * s.nrows * 128 + q * 2048, md, dt * 128 + h * 64,
                                        ybase + q * 16, &sm.full[slot], pol);
                }
            }
            // every issued copy must land before the CTA may exit
            const uint32_t first = it > (uint32_t)kTcStages ? it - kTcStages : 0u;
            for (uint32_t i = first; i < it; ++i)
                mbar_wait_bounded(&sm.full[i % kTcStages], (i / kTcStages) & 1u);
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (lane == 0) {
            uint32_t it = 0, bit = 0, ti = 0, dtc = 0;
            int r = r_begin;
            TSeg s;
            const uint32_t a_base = smem_u32(aring), b_base = smem_u32(bring), h_base = smem_u32(htile);
            while (ok && next_tile(a, sm, r, r_end, s)) {
                const int4 rec = sm.units[sm.cls_off[s.cls] + s.q];
                const int mg = min(kTcTokens, rec.z - s.grp * kTcTokens);
                const int Mp = (mg + 7) & ~7;
                const int N = 2 * Mp;
                const uint32_t id_gu = idesc_bf16_f32(128, N, false, false);
                const uint32_t id_dn = idesc_bf16_f32(128, N, true, false);
                if (!wait(&sm.acc_empty, (ti & 1u) ^ 1u)) break;
                tc_fence_after_sync();
                for (int kb = 0; ok && kb < KB; ++kb, ++it, ++bit) {
                    const int slot = it % kTcStages, bslot = bit % kTcStages;
                    if (!wait(&sm.full[slot], (it / kTcStages) & 1u) ||
                        !wait(&sm.bx_full[bslot], (bit / kTcStages) & 1u))
                        break;
                    tc_fence_after_sync();
                    const uint32_t A = a_base + slot * kAStage, Bx = b_base + bslot * kBStage;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t bd = smem_desc_sw128(Bx + ks * 32, 16, 1024);
                        const uint32_t acc = (kb | ks) ? 1u : 0u;
                        umma_bf16(tmem + kColG, smem_desc_sw128(A + ks * 32, 16, 1024), bd, id_gu, acc);
                        umma_bf16(tmem + kColU, smem_desc_sw128(A + 8192 + ks * 32, 16, 1024), bd, id_gu, acc);
                    }
                    umma_commit(&sm.empty[slot]);
                    umma_commit(&sm.bx_empty[bslot]);
                }
                if (!ok) break;
                umma_commit(&sm.acc_full);
                if (!wait(&sm.h_full, ti & 1u)) break;
                tc_fence_after_sync();
                const int ksteps = s.nrows / 16;
                for (int dt = 0; ok && dt < DT; ++dt, ++it, ++dtc) {
                    const uint32_t b = dtc & 1u, use = dtc >> 1;
                    const int slot = it % kTcStages;
                    if (!wait(&sm.y_empty[b], (use & 1u) ^ 1u)) break;
                    if (!wait(&sm.full[slot], (it / kTcStages) & 1u)) break;
                    tc_fence_after_sync();
                    const uint32_t A = a_base + slot * kAStage;
                    for (int ks = 0; ks < ksteps; ++ks)
                        umma_bf16(tmem + (b ? kColY1 : kColY0),
                                  smem_desc_sw128(A + ks * 2048, s.nrows * 128, 1024),
                                  smem_desc_sw128(h_base + ks * 32, 16, 1024), id_dn, ks ? 1u : 0u);
                    umma_commit(&sm.empty[slot]);
                    umma_commit(&sm.y_full[b]);
                }
                ++ti;
            }
            umma_commit(&sm.mma_done);
            mbar_wait_bounded(&sm.mma_done, 0);  // all MMAs finished before TMEM is freed
        }
    } else if (warp < 6) {
        // ===================== epilogue =====================
        const int quarter = warp & 3;                   // TMEM lanes this warp may access
        const int m = quarter * 32 + lane;              // tile row (gate/up) / hidden column (down)
        const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
        uint32_t ti = 0, dtc = 0;
        int r = r_begin;
        TSeg s;
        while (ok && next_tile(a, sm, r, r_end, s)) {
            const int4 rec = sm.units[sm.cls_off[s.cls] + s.q];
            const int kind = a.f.cls[s.cls].kind;
            const int first = rec.y + s.grp * kTcTokens;
            const int mg = min(kTcTokens, rec.z - s.grp * kTcTokens);
            const int Mp = (mg + 7) & ~7;
            if (!wait(&sm.acc_full, ti & 1u)) break;
            tc_fence_after_sync();
            for (int c0 = 0; c0 < Mp; c0 += 16) {
                float ghi[16], glo[16], uhi[16], ulo[16];
                tmem_ld16(tmem + lanes + kColG + c0, ghi);
                tmem_ld16(tmem + lanes + kColG + Mp + c0, glo);
                tmem_ld16(tmem + lanes + kColU + c0, uhi);
                tmem_ld16(tmem + lanes + kColU + Mp + c0, ulo);
                if (m < s.nrows) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = c0 + jj;
                        if (j < mg) {
                            int t, row;
                            float w;
                            tile_token(a, kind, first + j, t, w, row);
                            float h = silu_f(ghi[jj] + glo[jj]) * (uhi[jj] + ulo[jj]);
                            if (a.f.out_mode == MOE_OUT_ACCUM) h *= w;
                            const __nv_bfloat16 hh = __float2bfloat16_rn(h);
                            const __nv_bfloat16 hl = __float2bfloat16_rn(h - __bfloat162float(hh));
                            // H is K-major: token row j (hi) / Mp + j (lo), K index m
                            const int chunk = m >> 3, within = m & 7;
                            *reinterpret_cast<__nv_bfloat16*>(
                                htile + j * 128 + (((chunk ^ (j & 7)) << 4) + within * 2)) = hh;
                            const int jl = Mp + j;
                            *reinterpret_cast<__nv_bfloat16*>(
                                htile + jl * 128 + (((chunk ^ (jl & 7)) << 4) + within * 2)) = hl;
                        }
                    }
                }
            }
            tc_fence_before_sync();
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.acc_empty);
                mbar_arrive(&sm.h_full);
            }
            for (int dt = 0; ok && dt < DT; ++dt, ++dtc) {
                const uint32_t b = dtc & 1u, use = dtc >> 1;
                if (!wait(&sm.y_full[b], use & 1u)) break;
                tc_fence_after_sync();
                const uint32_t ycol = b ? kColY1 : kColY0;
                for (int c0 = 0; c0 < Mp; c0 += 16) {
                    float yhi[16], ylo[16];
                    tmem_ld16(tmem + lanes + ycol + c0, yhi);
                    tmem_ld16(tmem + lanes + ycol + Mp + c0, ylo);
                    if (c0 + 16 >= Mp) {
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sm.y_empty[b]);
                    }
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = c0 + jj;
                        if (j < mg) {
                            int t, row;
                            float w;
                            tile_token(a, kind, first + j, t, w, row);
                            atomicAdd(a.f.out + (size_t)row * d + dt * 128 + m, yhi[jj] + ylo[jj]);
                        }
                    }
                }
            }
            ++ti;
        }
    } else {
        // ===================== activation converter =====================
        const int ct = tid - 6 * 32;                    // 0..127
        uint32_t bit = 0;
        int r = r_begin;
        TSeg s;
        while (ok && next_tile(a, sm, r, r_end, s)) {
            const int4 rec = sm.units[sm.cls_off[s.cls] + s.q];
            const int kind = a.f.cls[s.cls].kind;
            const int first = rec.y + s.grp * kTcTokens;
            const int mg = min(kTcTokens, rec.z - s.grp * kTcTokens);
            const int Mp = (mg + 7) & ~7;
            const int items = 2 * Mp * 8;               // (B row, 16-byte chunk) pairs
            // this thread's items are fixed for the tile: resolve their token rows once
            const float* src[4];
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const int item = ct + k4 * 128;
                const int n = item >> 3;
                const int j = n < Mp ? n : n - Mp;
                src[k4] = nullptr;
                if (item < items && j < mg) {
                    int t, row;
                    float w;
                    tile_token(a, kind, first + j, t, w, row);
                    src[k4] = a.f.x + (size_t)t * d + (item & 7) * 8;
                }
            }
            for (int kb = 0; ok && kb < KB; ++kb, ++bit) {
                const int slot = bit % kTcStages;
                if (!wait(&sm.bx_empty[slot], ((bit / kTcStages) & 1u) ^ 1u)) break;
                unsigned char* Bt = bring + slot * kBStage;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const int item = ct + k4 * 128;
                    if (item < items) {
                        const int n = item >> 3, c = item & 7;
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (src[k4]) {
                            const float4* p = reinterpret_cast<const float4*>(src[k4] + kb * 64);
                            const float4 x0 = __ldg(p), x1 = __ldg(p + 1);
                            const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                            float o[8];
                            if (n < Mp) {
#pragma unroll
                                for (int e = 0; e < 8; ++e) o[e] = xv[e];
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    o[e] = xv[e] - __bfloat162float(__float2bfloat16_rn(xv[e]));
                            }
                            v = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                                           pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
                        }
                        *reinterpret_cast<uint4*>(Bt + n * 128 + ((c ^ (n & 7)) << 4)) = v;
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.bx_full[slot]);
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t ffn_tc_smem_bytes(int units) {
    return 1024 + (size_t)kTcStages * (kAStage + kBStage) + kHTile + sizeof(TcSmem) +
           (size_t)units * sizeof(int4);
}

cudaError_t launch_ffn_tc(const TcArgs& a, cudaStream_t s) {
    int units = 0;
    for (int c = 0; c < a.f.ncls; ++c) units += class_capacity(a.f.cls[c], a.f.n, a.f.g);
    const size_t smem = ffn_tc_smem_bytes(units);
    cudaError_t e = cudaFuncSetAttribute(ffn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(device_sm_count(), 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ffn_tc_kernel, a);
}

}  // namespace moe
