// Weight-row streaming core shared by the CUDA-core FFN kernels: weight
// decoding to fp32 pairs and the two per-stage routines of a row stream.
// Consumer threads own fixed 8-column chunks of a row (a thread's chunks
// are `coff`, valid where `cval`); a stage holds up to RMAX rows.
//  - gu_stage: dot products of every row with up to kMT token vectors held
//    in registers, reduced across the warp and then across warps with shared
//    atomics (what a gate or up projection needs);
//  - down_stage: every row, scaled by a per-(row, token) coefficient from
//    shared memory, accumulated into per-thread column accumulators (what a
//    down projection W^T h needs).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"

namespace moe {

namespace {

constexpr int kMT = kGroupTokens;    // tokens per group (register tile)

template <typename WT>
struct WLoad;
template <>
struct WLoad<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    __device__ static __forceinline__ void load8(const char* p, float2 (&f)[4]) {
        unpack_bf16x8_f2(*reinterpret_cast<const uint4*>(p), f);
    }
};
// FP8 E4M3 codes: 8 per 8 bytes, decoded pairwise (exactly) through half2 by
// the conversion unit; the row scale is applied by the caller.  (Decoding
// with integer bit operations instead measured 1.5x slower on the stream.)
template <>
struct WLoad<__nv_fp8_e4m3> {
    static constexpr int kBytes = 1;
    __device__ static __forceinline__ void load8(const char* p, float2 (&f)[4]) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        const uint32_t w[2] = {v.x, v.y};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xffffu), __NV_E4M3);
            const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
            f[2 * i] = __half22float2(*reinterpret_cast<const __half2*>(&lo));
            f[2 * i + 1] = __half22float2(*reinterpret_cast<const __half2*>(&hi));
        }
    }
};
template <>
struct WLoad<float> {
    static constexpr int kBytes = 4;
    __device__ static __forceinline__ void load8(const char* p, float2 (&f)[4]) {
        const float4 a = reinterpret_cast<const float4*>(p)[0];
        const float4 b = reinterpret_cast<const float4*>(p)[1];
        f[0] = make_float2(a.x, a.y);
        f[1] = make_float2(a.z, a.w);
        f[2] = make_float2(b.x, b.y);
        f[3] = make_float2(b.z, b.w);
    }
};

template <typename WT, int NCW, int CH, int RMAX>
struct Ffn {
    static constexpr int kNC = NCW * 32;      // consumer threads
    static constexpr int kBw = WLoad<WT>::kBytes;

    // One gate or up stage: nr rows of one matrix against MTC tokens.  FULL:
    // the stage holds RMAX rows (no row checks).
    template <int MTC, bool FULL>
    __device__ static __forceinline__ void gu_stage(const char* stage, int nr, int row_bytes,
                                                    const int (&coff)[CH], const bool (&cval)[CH],
                                                    const float2 (&xr)[CH][kMT][4],
                                                    float* gu_rows, int mg, int lane) {
        float2 acc[RMAX][MTC];
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
#pragma unroll
            for (int m = 0; m < MTC; ++m) acc[r][m] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            if (FULL || r < nr) {
#pragma unroll
                for (int j = 0; j < CH; ++j) {
                    if (cval[j]) {
                        float2 w2[4];
                        WLoad<WT>::load8(stage + (size_t)r * row_bytes + coff[j], w2);
#pragma unroll
                        for (int m = 0; m < MTC; ++m)
#pragma unroll
                            for (int e = 0; e < 4; ++e) acc[r][m] = ffma2(w2[e], xr[j][m][e], acc[r][m]);
                    }
                }
            }
        }
        constexpr int V = RMAX * MTC;
        float v[V];
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
#pragma unroll
            for (int m = 0; m < MTC; ++m) v[r * MTC + m] = acc[r][m].x + acc[r][m].y;
        int vi;
        const float sum = warp_reduce_spread<V>(v, lane, vi);
        if ((lane & (32 / V - 1)) == 0) {
            const int r = vi / MTC, m = vi - (vi / MTC) * MTC;
            if ((FULL || r < nr) && m < mg) atomicAdd(&gu_rows[r * kMT + m], sum);
        }
    }

    // One down stage: y[col] += W_down[row, col] * h[row, token].
    template <int MTC, bool FULL>
    __device__ static __forceinline__ void down_stage(const char* stage, int nr, int row_bytes,
                                                      const int (&coff)[CH], const bool (&cval)[CH],
                                                      const float* h_rows,
                                                      float2 (&yacc)[CH][kMT][4]) {
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            if (FULL || r < nr) {
                const float4 hv4 = *reinterpret_cast<const float4*>(h_rows + r * kMT);
                const float hv[4] = {hv4.x, hv4.y, hv4.z, hv4.w};
#pragma unroll
                for (int j = 0; j < CH; ++j) {
                    if (cval[j]) {
                        float2 w2[4];
                        WLoad<WT>::load8(stage + (size_t)r * row_bytes + coff[j], w2);
#pragma unroll
                        for (int m = 0; m < MTC; ++m) {
                            const float2 hh = make_float2(hv[m], hv[m]);
#pragma unroll
                            for (int e = 0; e < 4; ++e) yacc[j][m][e] = ffma2(w2[e], hh, yacc[j][m][e]);
                        }
                    }
                }
            }
        }
    }

    template <int MTC>
    __device__ static __forceinline__ void gu_any(const char* st, int nr, int row_bytes,
                                                  const int (&coff)[CH], const bool (&cval)[CH],
                                                  const float2 (&xr)[CH][kMT][4], float* gr,
                                                  int mg, int lane) {
        if (nr == RMAX) gu_stage<MTC, true>(st, nr, row_bytes, coff, cval, xr, gr, mg, lane);
        else gu_stage<MTC, false>(st, nr, row_bytes, coff, cval, xr, gr, mg, lane);
    }
    template <int MTC>
    __device__ static __forceinline__ void down_any(const char* st, int nr, int row_bytes,
                                                    const int (&coff)[CH], const bool (&cval)[CH],
                                                    const float* hr, float2 (&yacc)[CH][kMT][4]) {
        if (nr == RMAX) down_stage<MTC, true>(st, nr, row_bytes, coff, cval, hr, yacc);
        else down_stage<MTC, false>(st, nr, row_bytes, coff, cval, hr, yacc);
    }
};

}  // namespace

}  // namespace moe
