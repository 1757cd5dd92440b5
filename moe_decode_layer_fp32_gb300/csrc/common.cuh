// Device helpers shared by the decode-layer kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

// Device status codes written into the workspace status word.
constexpr int kDevErrTimeout = -5;
constexpr int kDevErrRouting = -6;

// Every bounded wait gives up after this long and reports kDevErrTimeout.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Device view of the workspace (pointers resolved on the host from the
// documented byte offsets).
struct WsPtrs {
    int32_t* status;
    int32_t* counts;
    float* logits;
    int32_t* exp_count;
    int32_t* exp_off;
    int32_t* asg_tok;
    int32_t* asg_slot;
    float* asg_w;
    int32_t* tok_asg;
    int32_t* act_exp;
    int32_t* dept_count;
    int32_t* dept_off;
    int32_t* dept_tok;
    float* dept_w;
    int32_t* tok_dpos;
    int32_t* act_dept;
    int4* exp_units;    // per active expert: {expert, token offset, token count, group prefix}
    int4* dept_units;   // per active department: same
    uint32_t* sync;
    __nv_bfloat16* xb;  // [2][T][d] activations as bf16 hi, lo (x = hi + lo)
};

// Widest hidden size the activation split buffer holds.
constexpr int kMaxXbHidden = 8192;

// x -> (hi, lo) bf16 with hi = bf16(x), lo = bf16(x - hi): 8 elements.
__device__ __forceinline__ void split_bf16x8(const float4 a, const float4 b, uint4& hi, uint4& lo) {
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * i]), h1 = __float2bfloat16_rn(v[2 * i + 1]);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * i] - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * i + 1] - __bfloat162float(h1));
        h[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        l[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Grid-stride split of x[T*d] into ws.xb (hi rows, then lo rows).
__device__ __forceinline__ void split_activations(const float* x, long long elems, __nv_bfloat16* xb,
                                                  long long tid0, long long stride) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    uint4* hi = reinterpret_cast<uint4*>(xb);
    uint4* lo = reinterpret_cast<uint4*>(xb + elems);
    for (long long i = tid0; i < elems / 8; i += stride) {
        uint4 h, l;
        split_bf16x8(x4[2 * i], x4[2 * i + 1], h, l);
        hi[i] = h;
        lo[i] = l;
    }
}

// E4M3 activation terms (the tensor-core path for E4M3 weights, whose MMAs
// take 8-bit operands on both sides).  Row t of x is scaled by 2^e0(t), e0
// chosen so that max |x_t| 2^e0 lies in [128, 256), and written as kXTerms
// E4M3 terms: q_0 = e4m3(v), v_1 = 16 (v - q_0), q_1 = e4m3(v_1), ... so that
//     x_t = 2^-e0 (q_0 + q_1 / 16 + q_2 / 256 + q_3 / 4096) + residual,
// each residual step exact in fp32 (|v - q_p| is at most half an E4M3 step,
// at most v / 16, and representable), and the residual at most 2^-16 of
// |x| per element (plus 2^-30 of max |x_t| from E4M3's subnormal floor).
// Layout in the xb region: terms [kXTerms][T][d] bytes, then e0 as int32[T]
// at byte offset xq_exp_offset(T).
constexpr int kXTerms = 4;
__host__ __device__ __forceinline__ size_t xq_exp_offset(int T) { return (size_t)4 * T * kMaxXbHidden; }

// One token's row: lanes of one warp.  d % 8 == 0.
__device__ __forceinline__ void split_e4m3_terms_warp(const float* x, int T, int d, int t, uint8_t* xq, int lane) {
    const float4* xr = reinterpret_cast<const float4*>(x + (size_t)t * d);
    float mx = 0.0f;
    for (int i = lane; i < d / 4; i += 32) {
        const float4 v = xr[i];
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    __syncwarp();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    // mx = f 2^E with f in [0.5, 1): mx 2^(8 - E) in [128, 256); kept within
    // the range where 2^e0 and 2^(e0 + 4 (kXTerms - 1)) are normal floats
    int e0 = 0;
    if (mx > 0.0f) {
        int E;
        frexpf(mx, &E);
        e0 = min(max(8 - E, -120), 126 - 4 * (kXTerms - 1));
    }
    if (lane == 0) reinterpret_cast<int32_t*>(xq + xq_exp_offset(T))[t] = e0;
    const float sc = __int_as_float((e0 + 127) << 23);
    for (int i = lane; i < d / 8; i += 32) {
        float v[8];
        const float4 a = xr[2 * i], b = xr[2 * i + 1];
        v[0] = a.x * sc; v[1] = a.y * sc; v[2] = a.z * sc; v[3] = a.w * sc;
        v[4] = b.x * sc; v[5] = b.y * sc; v[6] = b.z * sc; v[7] = b.w * sc;
#pragma unroll
        for (int p = 0; p < kXTerms; ++p) {
            uint32_t w[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t word = 0u;
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int j = 4 * h + e;
                    const __nv_fp8x2_storage_t q =
                        __nv_cvt_float2_to_fp8x2(make_float2(v[j], v[j + 1]), __NV_SATFINITE, __NV_E4M3);
                    const float2 back = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(q, __NV_E4M3)));
                    v[j] = 16.0f * (v[j] - back.x);
                    v[j + 1] = 16.0f * (v[j + 1] - back.y);
                    word |= (uint32_t)q << (8 * e);
                }
                w[h] = word;
            }
            *reinterpret_cast<uint2*>(xq + ((size_t)p * T + t) * d + 8 * (size_t)i) = make_uint2(w[0], w[1]);
        }
    }
}

// Tokens per register group of the FFN kernels; a unit with M tokens is
// processed as ceil(M / kGroupTokens) groups.
constexpr int kGroupTokens = 4;

__device__ __forceinline__ void set_status(int32_t* status, int code) {
    atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- programmatic dependent launch -----------------------------------------
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Atomic add with GPU-scope acquire-release semantics; returns the old value.
__device__ __forceinline__ uint32_t atomic_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Wait for the phase with the given parity to complete; false after the
// limit (kWaitLimitNs unless the caller passes a shorter one).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// ---- bulk copies (TMA, untiled) ----------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// Global -> shared copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned); completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy (bulk
// copies, tensor core).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Shared -> global element-wise fp32 add of `bytes` (multiple of 16, both
// addresses 16-byte aligned), performed by the bulk-copy unit at L2 as one
// operation; the shared source must be made visible to the async proxy
// first (fence_async_smem).  bulk_wait_all() returns once every reduction
// this thread committed has completed.
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst_global, const void* src_smem, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst_global),
                 "r"(smem_u32(src_smem)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Returns once every committed reduction has finished reading its shared source.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// ---- cp.async (16-byte global -> shared, L2 only) ---------------------------------
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- named barrier among a subset of warps -----------------------------------
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Named barrier that also ORs a predicate over the participating threads, so
// every thread leaves with the same answer.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ---- numerics -----------------------------------------------------------------
__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }
// The same with the hardware exponential and division (a few ulp, about 1e-6
// relative): for epilogues where one warp per SM sub-partition applies it to
// a whole tile column and the precise forms are its critical path.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// 8 bf16 (one 16-byte word) -> 8 fp32, exact.
__device__ __forceinline__ void unpack_bf16x8(const uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Two-wide fp32 fused multiply-add (sm_100+): returns a * b + c per lane pair.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%1, %2};\n\t"
        "mov.b64 rb, {%3, %4};\n\t"
        "mov.b64 rc, {%5, %6};\n\t"
        "fma.rn.f32x2 %0, ra, rb, rc;\n\t}"
        : "=l"(d)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
    return r;
}

// 8 bf16 (one 16-byte word) -> 4 fp32 pairs (elements 2i, 2i+1), exact.
__device__ __forceinline__ void unpack_bf16x8_f2(const uint4 v, float2 (&f)[4]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

// Warp collectives start from a converged warp (__syncwarp): after a
// lane-dependent branch the lanes may still run as separate groups, and then
// every full-mask shuffle waits for the groups to meet.  Measured in the
// one-token table build: about 720 cycles per round of three shuffles on a
// split warp, about 33 once converged.
__device__ __forceinline__ int warp_sum_int(int v) {
    __syncwarp();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    __syncwarp();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---- routing: top-k of one token by one warp --------------------------------
// Router of "DeaMoE: Efficient MoE Structure for Fast Small-Batch Decoding"
// §2.1 eqs. (2)-(3): the k largest keys (logit + selection bias of "DeepSeekMoE
// Guide", routing-bias formulation), descending, equal keys -> lower expert
// index first; weights = scale * softmax over the selected unbiased logits.
//
// Keys are mapped to unsigned integers that order like the floats (-0 folded
// into +0 so that it ties with +0, as a float comparison does).  Each round
// takes the warp maximum of the lanes' best remaining keys and then the
// smallest expert index holding it, both with single-instruction warp
// reductions.  0 marks a taken (or absent) entry; NaN and -inf keys map below
// every finite key, and picking one flags the routing as bad.
__device__ __forceinline__ uint32_t ordered_key(float v) {
    if (v == 0.0f) v = 0.0f;
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Lane holds experts lane + 32*j of logits_row[0..n) (J*32 >= n, k <= n).
// On return lane r < k holds the r-th selected expert and its weight; the
// result (same on every lane) says whether a non-finite key was selected.
// SMEM: logits_row points to shared memory (plain loads) instead of global
// memory (L2 loads).
template <int J, bool SMEM = false>
__device__ __forceinline__ bool topk_select_warp(const float* logits_row, const float* bias, int n,
                                                 int k, float scale, int& out_idx, float& out_w) {
    const int lane = threadIdx.x & 31;
    constexpr uint32_t kLowest = 0x007fffffu;   // ordered_key(-inf)
    uint32_t key[J];
    float lg[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        lg[j] = 0.0f;
        key[j] = 0u;
        if (e < n) {
            const float l = SMEM ? logits_row[e] : __ldcg(logits_row + e);
            const float kv = bias ? l + __ldg(bias + e) : l;
            lg[j] = l;
            // finite keys rank above kLowest; -inf and NaN take kLowest (still
            // selectable, after every finite key, lowest index first)
            key[j] = (kv == kv && kv != -INFINITY) ? ordered_key(kv) : kLowest;
        }
    }
    // A round is two warp reductions and selects: the picked index is
    // warp-uniform, its owner clears the entry, and lane r keeps the r-th
    // index; the picked logits are fetched once after the rounds.
    int my_idx = 0;
    bool bad = false;
    __syncwarp();
    for (int r = 0; r < k; ++r) {
        uint32_t bk = 0u;
        int bj = 0;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const bool gt = key[j] > bk;
            bk = gt ? key[j] : bk;
            bj = gt ? j : bj;
        }
        const uint32_t top = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t cand = (bk == top && top != 0u) ? (uint32_t)(lane + 32 * bj) : 0xffffffffu;
        const uint32_t bi = __reduce_min_sync(0xffffffffu, cand);
        bad = bad || top <= kLowest;   // a non-finite key (or none) was selected
        const int e = bi == 0xffffffffu ? 0 : (int)bi;
        const bool mine = (e & 31) == lane;
#pragma unroll
        for (int j = 0; j < J; ++j) key[j] = (mine && j == (e >> 5)) ? 0u : key[j];
        my_idx = lane == r ? e : my_idx;
    }
    // lane r < k: the logit of its pick, from the owning lane (one shuffle per slot)
    float my_lg = 0.0f;
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const float v = __shfl_sync(0xffffffffu, lg[j], my_idx & 31);
        my_lg = (my_idx >> 5) == j ? v : my_lg;
    }
    float mx = lane < k ? my_lg : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float ex = lane < k ? expf(my_lg - mx) : 0.0f;
    float s = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    out_idx = my_idx;
    out_w = lane < k ? scale * (ex / s) : 0.0f;
    return bad;
}

// Group-limited top-k of "DeaMoE: Efficient MoE Structure for Fast Small-Batch
// Decoding" §3.3 (at most k_dept departments per token), with the strict
// department-coverage variant of its appendix ablation (Table 4).  Expert e
// belongs to department e / g; a department's score is its best key.
//
// Round r of the department stage takes the best key among the experts of the
// departments not kept yet (ties -> lower expert index, hence lower
// department): that expert leads its department, which is kept.  The soft
// selection is then the top-k over the kept departments' experts.  The strict
// selection is every kept department's leader plus the best k - k_dept other
// experts of the kept departments; this is what replacing, one at a time, the
// lowest-ranked expert whose department keeps another selected expert by the
// leader of the best uncovered kept department ends with, because such an
// expert is never a leader and a new leader is never replaced.  Either way the
// selected experts come out by descending key.  Same lane layout and result as
// topk_select_warp (k <= k_dept * g; strict needs k >= k_dept).
template <int J, bool SMEM = false>
__device__ __forceinline__ bool topk_select_warp_grouped(const float* logits_row, const float* bias, int n,
                                                         int k, int g, int k_dept, bool strict, float scale,
                                                         int& out_idx, float& out_w) {
    const int lane = threadIdx.x & 31;
    constexpr uint32_t kLowest = 0x007fffffu;   // ordered_key(-inf)
    uint32_t key[J];
    float lg[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        lg[j] = 0.0f;
        key[j] = 0u;
        if (e < n) {
            const float l = SMEM ? logits_row[e] : __ldcg(logits_row + e);
            const float kv = bias ? l + __ldg(bias + e) : l;
            lg[j] = l;
            key[j] = (kv == kv && kv != -INFINITY) ? ordered_key(kv) : kLowest;
        }
    }
    // Warp-wide best (key, then lowest index) among the entries whose bit is
    // set in the lane's mask; -1 when there is none.
    auto best = [&](uint32_t mask, uint32_t& top) -> int {
        __syncwarp();
        uint32_t bk = 0u;
        int bj = 0;
#pragma unroll
        for (int j = 0; j < J; ++j)
            if (((mask >> j) & 1u) && key[j] > bk) {
                bk = key[j];
                bj = j;
            }
        top = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t cand = (bk == top && top != 0u) ? (uint32_t)(lane + 32 * bj) : 0xffffffffu;
        const uint32_t bi = __reduce_min_sync(0xffffffffu, cand);
        return bi == 0xffffffffu ? -1 : (int)bi;
    };
    uint32_t all = 0u;
#pragma unroll
    for (int j = 0; j < J; ++j)
        if (lane + 32 * j < n) all |= 1u << j;
    uint32_t kept = 0u, lead = 0u;
    bool bad = false;
    for (int r = 0; r < k_dept; ++r) {
        uint32_t top;
        const int e = best(all & ~kept, top);
        if (e < 0) {
            bad = true;
            break;
        }
        const int first = e - e % g;   // the department's first expert (warp-uniform)
#pragma unroll
        for (int j = 0; j < J; ++j)
            if ((uint32_t)(lane + 32 * j - first) < (uint32_t)g) kept |= 1u << j;
        kept &= all;
        if (lane == (e & 31)) lead |= 1u << (e >> 5);
    }
    // the experts to output: soft, the whole kept pool (top-k taken below);
    // strict, the leaders plus the best k - k_dept non-leaders
    uint32_t pool = kept;
    if (strict) {
        pool = lead;
        for (int r = k_dept; r < k; ++r) {
            uint32_t top;
            const int e = best(kept & ~pool, top);
            if (e < 0) {
                bad = true;
                break;
            }
            if (lane == (e & 31)) pool |= 1u << (e >> 5);
        }
    }
    int my_idx = 0;
    float my_lg = 0.0f;
    for (int r = 0; r < k; ++r) {
        uint32_t top;
        const int e = best(pool, top);
        if (e < 0 || top <= kLowest) bad = true;
        const int ee = e < 0 ? 0 : e;
        const int owner = ee & 31, jb = ee >> 5;
        float v = 0.0f;
#pragma unroll
        for (int j = 0; j < J; ++j)
            if (j == jb) v = lg[j];
        if (lane == owner && e >= 0) pool &= ~(1u << jb);
        v = __shfl_sync(0xffffffffu, v, owner);
        if (lane == r) {
            my_idx = ee;
            my_lg = v;
        }
    }
    __syncwarp();
    float mx = lane < k ? my_lg : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float ex = lane < k ? expf(my_lg - mx) : 0.0f;
    float s = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    out_idx = my_idx;
    out_w = lane < k ? scale * (ex / s) : 0.0f;
    return bad;
}

// Exclusive prefix sum of data[0..len) in place; returns the total.  All NT
// threads of the block must call it.
template <int NT>
__device__ int block_exclusive_scan(int* data, int len, int* warp_tmp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (len + NT - 1) / NT;
    const int b = min(len, tid * per), e = min(len, b + per);
    int s = 0;
    for (int i = b; i < e; ++i) s += data[i];
    int v = s;
    __syncwarp();
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_tmp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int x = lane < NT / 32 ? warp_tmp[lane] : 0;
        __syncwarp();
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += t;
        }
        if (lane < NT / 32) warp_tmp[lane] = x;
    }
    __syncthreads();
    int run = v - s + (warp > 0 ? warp_tmp[warp - 1] : 0);
    const int total = warp_tmp[NT / 32 - 1];
    for (int i = b; i < e; ++i) {
        const int c = data[i];
        data[i] = run;
        run += c;
    }
    __syncthreads();
    return total;
}

// Reduce V values across the warp; afterwards the lanes whose low
// (5 - log2 V) bits are zero hold the full sum of value index `vi`.
template <int V>
__device__ __forceinline__ float warp_reduce_spread(float (&v)[V], int lane, int& vi) {
    __syncwarp();
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


// Exclusive prefix sums of three arrays at once (one pass, two barriers);
// returns the three totals.  All NT threads of the block must call it.
template <int NT>
__device__ int3 block_exclusive_scan3(int* a0, int* a1, int* a2, int len, int3* warp_tmp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (len + NT - 1) / NT;
    const int b = min(len, tid * per), e = min(len, b + per);
    int3 s = make_int3(0, 0, 0);
    for (int i = b; i < e; ++i) {
        s.x += a0[i];
        s.y += a1[i];
        s.z += a2[i];
    }
    int3 v = s;
    __syncwarp();
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int tx = __shfl_up_sync(0xffffffffu, v.x, o);
        const int ty = __shfl_up_sync(0xffffffffu, v.y, o);
        const int tz = __shfl_up_sync(0xffffffffu, v.z, o);
        if (lane >= o) {
            v.x += tx;
            v.y += ty;
            v.z += tz;
        }
    }
    if (lane == 31) warp_tmp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int3 x = lane < NT / 32 ? warp_tmp[lane] : make_int3(0, 0, 0);
        __syncwarp();
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int tx = __shfl_up_sync(0xffffffffu, x.x, o);
            const int ty = __shfl_up_sync(0xffffffffu, x.y, o);
            const int tz = __shfl_up_sync(0xffffffffu, x.z, o);
            if (lane >= o) {
                x.x += tx;
                x.y += ty;
                x.z += tz;
            }
        }
        if (lane < NT / 32) warp_tmp[lane] = x;
    }
    __syncthreads();
    int3 run = make_int3(v.x - s.x, v.y - s.y, v.z - s.z);
    if (warp > 0) {
        run.x += warp_tmp[warp - 1].x;
        run.y += warp_tmp[warp - 1].y;
        run.z += warp_tmp[warp - 1].z;
    }
    const int3 total = warp_tmp[NT / 32 - 1];
    for (int i = b; i < e; ++i) {
        const int c0 = a0[i], c1 = a1[i], c2 = a2[i];
        a0[i] = run.x;
        a1[i] = run.y;
        a2[i] = run.z;
        run.x += c0;
        run.y += c1;
        run.z += c2;
    }
    __syncthreads();
    return total;
}


// One warp: keep the unit records {unit, first entry, entries, .} of src[0..A)
// whose entry count lies in [lo, hi]; write them compacted to dst with .w =
// inclusive prefix over the kept records of ceil(entries / gsize).  Returns
// the number kept and the group total (same on every lane).
__device__ __forceinline__ int filter_units_warp(const int4* src, int A, int lo, int hi, int gsize,
                                                 int4* dst, int* total_groups) {
    const int lane = threadIdx.x & 31;
    int kept = 0, gsum = 0;
    for (int b = 0; b < A; b += 32) {
        const int q = b + lane;
        __syncwarp();
        const int4 r = q < A ? src[q] : make_int4(0, 0, 0, 0);
        const bool keep = q < A && r.z >= lo && r.z <= hi;
        int gi = keep ? (r.z + gsize - 1) / gsize : 0;
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, gi, o);
            if (lane >= o) gi += t;
        }
        if (keep) dst[kept + __popc(bal & ((1u << lane) - 1u))] = make_int4(r.x, r.y, r.z, gsum + gi);
        kept += __popc(bal);
        gsum += __shfl_sync(0xffffffffu, gi, 31);
    }
    *total_groups = gsum;
    return kept;
}
}  // namespace moe
