// DeaMoE layer in the paper's own parameterisation ("form P"), "DeaMoE:
// Efficient MoE Structure for Fast Small-Batch Decoding" §3.1 eq. (4) with
// sigma = SiLU (§3.4): department j holds W_g^j, W_u^j, W_d^j ([r, h] row
// blocks), expert i of department j holds A_g^i, A_u^i, A_d^i ([r, r]), and
//     g^ = SiLU(A_g SiLU(W_g x)),  u^ = A_u SiLU(W_u x),
//     DeaMoE_i(x) = W_d^T SiLU(A_d^T (g^ * u^)),
// combined with the routing weights of eq. (3).  By linearity of W_d^T the
// layer output of token t is sum_j W_d^jT H_{t,j} with
// H_{t,j} = sum over the token's experts i in department j of p_i Z_{t,i},
// Z_{t,i} = SiLU(A_d^iT Y_{t,i}).
//
// Three weight-streaming passes, each a persistent grid chained to the one
// before by a programmatic dependent launch:
//   up:   per active department and its tokens X^j: G = SiLU(W_g x) and
//         U = SiLU(W_u x) into [department entry, r] buffers;
//   priv: per active expert and its assignments: Y = SiLU(A_g G) * (A_u U),
//         then A_d^T Y added into an [assignment, r] buffer (rows of A_d
//         are split over CTAs, so the SiLU is applied by the next pass);
//   down: per active department: H from the assignment buffer (SiLU, routing
//         weights), then W_d^T H added into y.
// Every pass splits the row space of its units evenly over the CTAs; a
// producer warp streams whole rows with bulk copies into a shared-memory
// ring and the consumer warps run the row-stream core (stream_core.cuh).
#include <cuda_bf16.h>

#include "../../include/moe_decode.h"
#include "kernels.h"
#include "stream_core.cuh"

namespace moe {

namespace {

constexpr int kPStageBytes = 16384;              // one ring slot
constexpr int kPRingBytesPerSM = 10 * kPStageBytes;
constexpr int kPSegMax = 256;                    // rows per segment

template <int NS>
struct PSmem {
    uint64_t full[NS];
    uint64_t empty[NS];
    float gu[2][kPSegMax * kMT];      // dot products of the segment (gate / up)
    float h[kPSegMax * kMT];          // down-projection coefficients
    int dn_cnt[kMT];                  // down pass: the group's tokens' assignments
    int dn_pos[kMT][kMaxK];           //   in the department: position and
    float dn_w[kMT][kMaxK];           //   routing weight
    int4 units[1];                    // active unit records (from the dispatch), sized at launch
};

struct PSeg {
    int q, grp, row0, nrows;
};

// Next segment of [rho, r_end): unit q (records ascending by inclusive group
// prefix .w), token group grp, rows [row0, row0 + nrows) of r.
template <int NS>
__device__ __forceinline__ bool p_next_seg(const PSmem<NS>& sm, int A, int r, long long& rho, long long r_end,
                                           PSeg& s) {
    if (rho >= r_end) return false;
    const long long gam = rho / r;
    int lo = 0, hi = A - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((long long)sm.units[mid].w > gam) hi = mid;
        else lo = mid + 1;
    }
    s.q = lo;
    s.grp = (int)(gam - (lo > 0 ? sm.units[lo - 1].w : 0));
    s.row0 = (int)(rho - gam * r);
    long long nr = r - s.row0;
    if (nr > r_end - rho) nr = r_end - rho;
    if (nr > kPSegMax) nr = kPSegMax;
    s.nrows = (int)nr;
    rho += nr;
    return true;
}

template <int STAGE, int NCW, int CH, int RMAX, int CPS>
__global__ void __launch_bounds__((NCW + 1) * 32, CPS) formp_kernel(FormPArgs a) {
    using K = Ffn<__nv_bfloat16, NCW, CH, RMAX>;
    constexpr int NS = kPRingBytesPerSM / kPStageBytes / CPS;
    constexpr int kNT = (NCW + 1) * 32;
    constexpr bool DOT = STAGE != kFormPDown;     // gate / up rows
    constexpr bool DOWN = STAGE != kFormPUp;      // down rows
    // Narrow rows (the 4-warp layout): a stage carries as many whole rows as
    // fit and the consumers take them RMAX at a time, so that each copy still
    // moves 16 KB.  Wider rows fill a stage with RMAX rows or fewer (measured
    // faster there: the sub-block loop costs more than it saves).
    constexpr bool SUB = NCW <= 4;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char* ring = smem_raw;
    PSmem<NS>& sm = *reinterpret_cast<PSmem<NS>*>(smem_raw + (size_t)NS * kPStageBytes);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], NCW);
        }
        mbar_init_fence();
    }
    for (int i = tid; i < 2 * kPSegMax * kMT; i += kNT) (&sm.gu[0][0])[i] = 0.0f;
    pdl_allow_dependents();
    // Everything below reads what the pass before (and the routing) wrote.
    pdl_wait_primary();

    if (STAGE == kFormPUp) {
        // the private pass adds into the assignment buffer, the down pass
        // into y (when no routing kernel cleared it): clear them here
        float4* z4 = reinterpret_cast<float4*>(a.zbuf);
        const long long n4 = (long long)a.T * a.k * a.r / 4;
        for (long long i = blockIdx.x * (long long)kNT + tid; i < n4; i += (long long)gridDim.x * kNT)
            z4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.zero_y) {
            float4* y4 = reinterpret_cast<float4*>(a.y);
            const long long m4 = (long long)a.T * a.d / 4;
            for (long long i = blockIdx.x * (long long)kNT + tid; i < m4; i += (long long)gridDim.x * kNT)
                y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    const bool dept_units = STAGE != kFormPPriv;
    const int A = dept_units ? a.ws.counts[1] : a.ws.counts[0];
    const int4* rec = dept_units ? a.ws.dept_units : a.ws.exp_units;
    for (int q = tid; q < A; q += kNT) sm.units[q] = rec[q];
    __syncthreads();
    const long long G = A > 0 ? sm.units[A - 1].w : 0;
    const long long R = G * a.r;
    const long long r_begin = R * blockIdx.x / gridDim.x;
    const long long r_end = R * (blockIdx.x + 1) / gridDim.x;

    const int width = STAGE == kFormPPriv ? a.r : a.d;   // row length (elements)
    const int row_bytes = width * 2;
    const int rps = min(SUB ? kPSegMax : RMAX, kPStageBytes / row_bytes);   // rows per stage
    const int nchunks = width / 8;

    if (warp == NCW) {
        // ===================== producer =====================
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            uint32_t it = 0;
            long long rho = r_begin;
            PSeg s;
            bool ok = true;
            auto issue = [&](const char* src, int nr) -> bool {
                const int slot = it % NS;
                const uint32_t par = ((it / NS) & 1u) ^ 1u;
                if (!mbar_wait_bounded(&sm.empty[slot], par)) return false;
                const uint32_t bytes = (uint32_t)nr * row_bytes;
                mbar_arrive_expect_tx(&sm.full[slot], bytes);
                bulk_load(ring + (size_t)slot * kPStageBytes, src, bytes, &sm.full[slot], pol);
                ++it;
                return true;
            };
            while (ok && p_next_seg(sm, A, a.r, rho, r_end, s)) {
                const size_t ubase = ((size_t)sm.units[s.q].x * a.r + s.row0) * (size_t)row_bytes;
                if (DOT) {
                    const char* g = static_cast<const char*>(STAGE == kFormPUp ? a.dgate : a.agate) + ubase;
                    const char* u = static_cast<const char*>(STAGE == kFormPUp ? a.dup : a.aup) + ubase;
                    for (int rb = 0; ok && rb < s.nrows; rb += rps) {
                        const int nr = min(rps, s.nrows - rb);
                        ok = issue(g + (size_t)rb * row_bytes, nr) && issue(u + (size_t)rb * row_bytes, nr);
                    }
                }
                if (DOWN) {
                    const char* dn = static_cast<const char*>(STAGE == kFormPPriv ? a.adown : a.ddown) + ubase;
                    for (int rb = 0; ok && rb < s.nrows; rb += rps)
                        ok = issue(dn + (size_t)rb * row_bytes, min(rps, s.nrows - rb));
                }
            }
            if (!ok) set_status(a.ws.status, kDevErrTimeout);
            // every issued copy lands before the CTA may exit
            const uint32_t first = it > (uint32_t)NS ? it - NS : 0u;
            for (uint32_t i = first; i < it; ++i) mbar_wait_bounded(&sm.full[i % NS], (i / NS) & 1u);
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
        coff[j] = c * 16;
    }
    uint32_t it = 0;
    long long rho = r_begin;
    PSeg s;
    bool ok = true;
    auto wait_full = [&](int slot, uint32_t i) -> bool {
        if (!ok) return false;
        if (!mbar_wait_bounded(&sm.full[slot], (i / NS) & 1u)) {
            ok = false;
            set_status(a.ws.status, kDevErrTimeout);
        }
        return ok;
    };
    auto release = [&](int slot) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
    };
    // token t of entry `pos`, checked (a bad list entry is reported, never
    // used as an address)
    auto checked_token = [&](int t) -> int {
        if ((unsigned)t >= (unsigned)a.T) {
            set_status(a.ws.status, kDevErrRouting);
            return -1;
        }
        return t;
    };

    while (p_next_seg(sm, A, a.r, rho, r_end, s)) {
        const int4 rc = sm.units[s.q];
        const int first = s.grp * kMT;
        const int mg = min(kMT, rc.z - first);
        int pos[kMT], tok[kMT];
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
            pos[m] = rc.y + first + m;
            tok[m] = -1;
            if (m < mg) tok[m] = checked_token(STAGE == kFormPPriv ? a.ws.asg_tok[pos[m]] : a.ws.dept_tok[pos[m]]);
        }

        if (DOT) {
            // inputs: the token rows (up pass, one set for gate and up) or the
            // token's department entries of the G and U buffers (private pass)
            constexpr int NX = STAGE == kFormPPriv ? 2 : 1;
            float2 xin[NX][CH][kMT][4];
#pragma unroll
            for (int m = 0; m < kMT; ++m) {
                const float* src[NX];
#pragma unroll
                for (int v = 0; v < NX; ++v) src[v] = nullptr;
                if (m < mg && tok[m] >= 0) {
                    if (STAGE == kFormPUp) {
                        src[0] = a.x + (size_t)tok[m] * a.d;
                    } else {
                        const int dpos = a.ws.tok_dpos[tok[m] * a.m + rc.x / a.g];
                        if ((unsigned)dpos < (unsigned)(a.T * a.mk)) {
                            src[0] = a.gbuf + (size_t)dpos * a.r;
                            src[NX - 1] = a.ubuf + (size_t)dpos * a.r;
                        } else {
                            set_status(a.ws.status, kDevErrRouting);
                        }
                    }
                }
#pragma unroll
                for (int v = 0; v < NX; ++v)
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const int c = (tid + j * K::kNC) * 8;
                        if (cval[j] && src[v]) {
                            const float4 p0 = __ldcg(reinterpret_cast<const float4*>(src[v] + c));
                            const float4 p1 = __ldcg(reinterpret_cast<const float4*>(src[v] + c) + 1);
                            xin[v][j][m][0] = make_float2(p0.x, p0.y);
                            xin[v][j][m][1] = make_float2(p0.z, p0.w);
                            xin[v][j][m][2] = make_float2(p1.x, p1.y);
                            xin[v][j][m][3] = make_float2(p1.z, p1.w);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) xin[v][j][m][e] = make_float2(0.f, 0.f);
                        }
                    }
            }
            for (int rb = 0; rb < s.nrows; rb += rps) {
                const int nr = min(rps, s.nrows - rb);
#pragma unroll 1
                for (int mat = 0; mat < 2; ++mat) {
                    const int slot = it % NS;
                    if (wait_full(slot, it)) {
                        const char* st0 = reinterpret_cast<const char*>(ring + (size_t)slot * kPStageBytes);
                        // the stage's rows RMAX at a time against one input set
                        auto dots = [&](const float2 (&xv)[CH][kMT][4]) {
                            for (int sb = 0; sb < (SUB ? nr : 1); sb += RMAX) {
                                const int ns = SUB ? min(RMAX, nr - sb) : nr;
                                const char* st = st0 + (size_t)sb * row_bytes;
                                float* gr = &sm.gu[mat][(rb + sb) * kMT];
                                if (mg == 1) K::template gu_any<1>(st, ns, row_bytes, coff, cval, xv, gr, mg, lane);
                                else if (mg == 2) K::template gu_any<2>(st, ns, row_bytes, coff, cval, xv, gr, mg, lane);
                                else K::template gu_any<4>(st, ns, row_bytes, coff, cval, xv, gr, mg, lane);
                            }
                        };
                        if (mat == 0) dots(xin[0]);
                        else dots(xin[NX - 1]);
                        release(slot);
                    }
                    ++it;
                }
            }
            if (named_bar_or(1, K::kNC, !ok)) break;
        }

        if (STAGE == kFormPUp) {
            // G = SiLU(W_g x), U = SiLU(W_u x), stored per department entry
            for (int i = tid; i < s.nrows * kMT; i += K::kNC) {
                const int m = i & (kMT - 1), row = i / kMT;
                if (m < mg && tok[m] >= 0) {
                    const size_t o = (size_t)pos[m] * a.r + s.row0 + row;
                    a.gbuf[o] = silu_f(sm.gu[0][i]);
                    a.ubuf[o] = silu_f(sm.gu[1][i]);
                }
                sm.gu[0][i] = 0.0f;
                sm.gu[1][i] = 0.0f;
            }
            named_bar_sync(1, K::kNC);
            continue;
        }

        if (STAGE == kFormPPriv) {
            // Y = SiLU(A_g G) * (A_u U)
            for (int i = tid; i < s.nrows * kMT; i += K::kNC) {
                const int m = i & (kMT - 1);
                sm.h[i] = m < mg ? silu_f(sm.gu[0][i]) * sm.gu[1][i] : 0.0f;
                sm.gu[0][i] = 0.0f;
                sm.gu[1][i] = 0.0f;
            }
        } else {
            // H_{t,j}[row] = sum over the token's experts in department j of
            // p_i SiLU(Z_{t,i}[row]); first the (position, weight) lists
            if (tid < mg) {
                const int t = tok[tid];
                const int j = rc.x;
                int c = 0;
                if (t >= 0) {
                    for (int sl = 0; sl < a.k; ++sl) {
                        const int e = a.topk_idx[t * a.k + sl];
                        if (e / a.g == j) {
                            const int p = a.ws.tok_asg[t * a.k + sl];
                            sm.dn_pos[tid][c] = p;
                            sm.dn_w[tid][c] = a.ws.asg_w[p];
                            ++c;
                        }
                    }
                }
                sm.dn_cnt[tid] = c;
            }
            named_bar_sync(1, K::kNC);
            for (int i = tid; i < s.nrows * kMT; i += K::kNC) {
                const int m = i & (kMT - 1), row = i / kMT;
                float hv = 0.0f;
                if (m < mg)
                    for (int c = 0; c < sm.dn_cnt[m]; ++c)
                        hv += sm.dn_w[m][c] * silu_f(__ldcg(a.zbuf + (size_t)sm.dn_pos[m][c] * a.r + s.row0 + row));
                sm.h[i] = hv;
            }
        }
        named_bar_sync(1, K::kNC);

        // ---- down rows: A_d^T Y (private pass) or W_d^T H (down pass) ----
        float2 yacc[CH][kMT][4];
#pragma unroll
        for (int j = 0; j < CH; ++j)
#pragma unroll
            for (int m = 0; m < kMT; ++m)
#pragma unroll
                for (int e = 0; e < 4; ++e) yacc[j][m][e] = make_float2(0.0f, 0.0f);
        for (int rb = 0; rb < s.nrows; rb += rps) {
            const int nr = min(rps, s.nrows - rb);
            const int slot = it % NS;
            if (wait_full(slot, it)) {
                const char* st0 = reinterpret_cast<const char*>(ring + (size_t)slot * kPStageBytes);
                for (int sb = 0; sb < (SUB ? nr : 1); sb += RMAX) {
                    const int ns = SUB ? min(RMAX, nr - sb) : nr;
                    const char* st = st0 + (size_t)sb * row_bytes;
                    const float* hr = &sm.h[(rb + sb) * kMT];
                    if (mg == 1) K::template down_any<1>(st, ns, row_bytes, coff, cval, hr, yacc);
                    else if (mg == 2) K::template down_any<2>(st, ns, row_bytes, coff, cval, hr, yacc);
                    else K::template down_any<4>(st, ns, row_bytes, coff, cval, hr, yacc);
                }
                release(slot);
            }
            ++it;
        }
        if (named_bar_or(1, K::kNC, !ok)) break;
        // private pass: into the assignment's row of the Z buffer (r wide);
        // down pass: into the token's output row (d wide)
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            if (cval[j]) {
                const int col = (tid + j * K::kNC) * 8;
#pragma unroll
                for (int m = 0; m < kMT; ++m) {
                    if (m < mg && tok[m] >= 0) {
                        float* orow = STAGE == kFormPPriv ? a.zbuf + (size_t)pos[m] * a.r : a.y + (size_t)tok[m] * a.d;
                        float4* dst = reinterpret_cast<float4*>(orow + col);
                        atomicAdd(dst, make_float4(yacc[j][m][0].x, yacc[j][m][0].y, yacc[j][m][1].x, yacc[j][m][1].y));
                        atomicAdd(dst + 1, make_float4(yacc[j][m][2].x, yacc[j][m][2].y, yacc[j][m][3].x, yacc[j][m][3].y));
                    }
                }
            }
        }
    }
}

template <int STAGE, int NCW, int CH, int RMAX, int CPS>
cudaError_t launch_formp_cfg(const FormPArgs& a, int sms, cudaStream_t s) {
    constexpr int NS = kPRingBytesPerSM / kPStageBytes / CPS;
    const int cap = STAGE == kFormPPriv ? a.n : a.m;   // unit records the dispatch may hold
    const size_t smem = (size_t)NS * kPStageBytes + sizeof(PSmem<NS>) + (size_t)cap * sizeof(int4);
    auto kern = formp_kernel<STAGE, NCW, CH, RMAX, CPS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sms * CPS));
    cfg.blockDim = dim3((NCW + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Consumer layout by row length: up to 1024 elements 4 warps of one 8-column
// chunk per thread (two CTAs per SM), up to 2048 8 warps, up to 7680 15 warps
// of two chunks (one CTA per SM, so that the register tiles fit).  The
// private pass takes rows of at most 2048.
template <int STAGE>
cudaError_t launch_formp_stage(const FormPArgs& a, int width, int sms, cudaStream_t s) {
#ifndef MOE_FP_NARROW_PRIV
#define MOE_FP_NARROW_PRIV 1
#endif
    // rows of at most 512 (64 chunks): two consumer warps, four CTAs per SM
    if (MOE_FP_NARROW_PRIV && width <= 512) return launch_formp_cfg<STAGE, 2, 1, 4, 4>(a, sms, s);
    if (width <= 1024) return launch_formp_cfg<STAGE, 4, 1, 4, 2>(a, sms, s);
    if (width <= 2048) return launch_formp_cfg<STAGE, 8, 1, 4, 1>(a, sms, s);
    if constexpr (STAGE != kFormPPriv) return launch_formp_cfg<STAGE, 15, 2, 1, 1>(a, sms, s);
    return cudaErrorInvalidValue;
}

}  // namespace

int formp_max_hidden() { return 15 * 32 * 2 * 8; }
int formp_max_width() { return 2048; }

cudaError_t launch_formp(const FormPArgs& a, int sms, cudaStream_t s) {
    cudaError_t e = launch_formp_stage<kFormPUp>(a, a.d, sms, s);
    if (e == cudaSuccess) e = launch_formp_stage<kFormPPriv>(a, a.r, sms, s);
    if (e == cudaSuccess) e = launch_formp_stage<kFormPDown>(a, a.d, sms, s);
    return e;
}

cudaError_t launch_formp_pass(const FormPArgs& a, int stage, int sms, cudaStream_t s) {
    if (stage == kFormPUp) return launch_formp_stage<kFormPUp>(a, a.d, sms, s);
    if (stage == kFormPPriv) return launch_formp_stage<kFormPPriv>(a, a.r, sms, s);
    return launch_formp_stage<kFormPDown>(a, a.d, sms, s);
}

}  // namespace moe
