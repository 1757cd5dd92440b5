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
// Mapping onto the MMA (D[M x N] = A[M x K] * B[N x K]^T, fp32 accumulate,
// M = 128):
//  * gate/up: A = a tile of 128 weight rows (K-major, 128 B swizzle), B = the
//    tokens' activations, N = tokens;
//  * down:    A = W_down rows of the same tile read as an MN-major operand
//    (M = 128 hidden columns, K = the tile's 128 rows), B = H = SiLU(g) * u.
// An MMA costs the tensor pipe a fixed ~45 cycles whatever N <= 64 is, so
// each one must carry a full 128-row (4 KB) slice of weights to outrun HBM.
// Weight tiles arrive as 3-D TMA boxes of 128 rows x 128 columns (256
// contiguous bytes per row; 32 KB), which stream at full HBM rate.
// Activations and H are split into bf16 hi + lo parts (x = hi + lo up to
// 2^-17 relative), so the products keep close to fp32 accuracy: each token
// occupies two B rows and the epilogue adds the two result columns.
//
// Warp roles (one CTA per SM): warp 0 issues TMA loads of weight boxes into a
// 4-stage ring; warp 1 issues the MMAs (one thread) and owns the TMEM
// allocation; warps 2-5 are the epilogue (TMEM -> registers, SwiGLU, H tile,
// output atomics); warps 6-9 gather the bf16 hi/lo activations (split once per
// layer) into swizzled B tiles with cp.async; the CTA has 16 warps so that the
// in-CTA top-k (a warp per token) takes up to 16 tokens in one round, and the
// warps past the roles only take part in that prologue.
//
// FP8 (E4M3 codes, one fp32 scale per weight row): TMA lands 16 KB boxes of
// codes (128 rows x 128 columns, 128 B swizzle) in a 6-stage ring.  Gate / up
// boxes are the A operand of kind::f8f6f4 MMAs as they are (K = 32 per
// instruction: half the instructions of the bf16 path per weight column, and
// an MMA instruction, not HBM, is what bounds a tile of few tokens); B holds
// the activations as four E4M3 terms per token (x = 2^-e0 sum_p 16^-p q_p,
// split once per layer), so N = 4 Mp and the epilogue sums the four result
// columns of each token.  Down boxes are expanded to bf16 by four more warps
// (10-13) into a 2-stage ring that the down MMAs read MN-major as on the bf16
// path (W_down is read transposed).  E4M3 values are exact in bf16 and the
// products of two E4M3 values exact in the MMA, so the rounding is that of the
// fp32 accumulation and of the activation terms (2^-16 of each element); the
// epilogue multiplies the gate and up results by their row scales and folds the
// down row scale into H (a down row is a K index of the down MMA).  Groups
// hold 16 tokens here, which frees the shared memory for the code ring.
// Every wait is bounded; on a timeout the kernel records an error status,
// drains its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <climits>

#include "../../include/moe_decode.h"
#include "kernels.h"
#ifndef MOE_ROUTE_PDL
#define MOE_ROUTE_PDL 1
#endif
#include "local_route.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

// Geometry.  A weight stage is one TMA box: kTcRows rows x 2 column chunks of
// 64 (K-blocks for gate/up, 128 hidden columns for down), landing as
// [chunk][row][128 B] with 128 B swizzle.  Gate/up run in K-pairs: the gate
// stage, then the up stage, of the same two K-blocks.
constexpr int kTcRows = kTcBoxRows;               // 128
constexpr int kChunkBytes = kTcRows * 128;        // 16 KB: one 64-column chunk
constexpr int kF8Box = kTcRows * 128;             // 16 KB: 128 rows x 128 E4M3 codes
#ifndef MOE_TC_STAGES
#define MOE_TC_STAGES 4
#endif
#ifndef MOE_TC_BPAIRS
#define MOE_TC_BPAIRS 3
#endif
#ifndef MOE_TC_F8_STAGES
#define MOE_TC_F8_STAGES 6
#endif
#ifndef MOE_TC_F8_CSTAGES
#define MOE_TC_F8_CSTAGES 2
#endif
#ifndef MOE_TC_F8_CROWS
#define MOE_TC_F8_CROWS 128
#endif
constexpr int kTmemCols = 512;

// Per weight type: bf16 (F8 = false) or E4M3 codes with row scales.
template <bool F8>
struct TcGeo {
    static constexpr int kTok = F8 ? 16 : kTcGroupTokens;   // tokens per group
    static constexpr int kMaxN = 2 * kTok;                   // down MMA N: H hi + lo rows
    // gate / up B operand: rows per token (bf16 hi + lo, or the E4M3 terms)
    static constexpr int kBTerms = F8 ? kXTerms : 2;
    static constexpr int kMaxNgu = kBTerms * kTok;           // 64
    static constexpr int kAStages = F8 ? MOE_TC_F8_CSTAGES : MOE_TC_STAGES;   // bf16 slots the MMAs read
    // rows (down: K) of a bf16 slot: whole boxes (half boxes, which let the
    // down MMAs of one half run while the converters fill the next, measured
    // slower: twice the hand-offs)
    static constexpr int kCRows = F8 ? MOE_TC_F8_CROWS : kTcRows;
    static constexpr int kAChunk = kCRows * 128;             // one 64-column chunk of a slot
    static constexpr int kASlot = 2 * kAChunk;
    static constexpr int kF8Stages = F8 ? MOE_TC_F8_STAGES : 0;                // code boxes
    static constexpr int kBPairs = MOE_TC_BPAIRS;            // activation ring (128-column K steps)
    static constexpr int kBBlock = kMaxNgu * 128;            // one 128-byte K-block of every B row: 8 KB
    static constexpr int kBBlocks = F8 ? 1 : 2;              // K-blocks per 128-column step
    static constexpr int kBPair = kBBlocks * kBBlock;
    static constexpr int kHChunk = kMaxN * 128;              // H: [K chunk][N rows][128 B]
    static constexpr int kHTile = 2 * kHChunk;               // K = 128 tile rows
    static constexpr int kYStage = kTok * 128 * 4;           // down output of one M-tile: [token][128 fp32]
    static constexpr int kCvtWarps = F8 ? 4 : 0;
    // 16 warps: the in-CTA top-k takes one token per warp, so up to 16 tokens
    // are selected in one round; warps past the roles idle after the prologue
    static constexpr int kWarps = 16;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kPdTok = F8 ? 1 : kTok;             // form-P down lists (bf16 only)
    // Tensor memory (512 columns): the G and U accumulators (N = kBTerms Mp
    // columns each), then the down accumulators (kYBufs of kYCols columns).
    static constexpr uint32_t kColG = 0;
    static constexpr uint32_t kColU = kMaxNgu;
    static constexpr uint32_t kColY = 2 * kMaxNgu;
    static constexpr uint32_t kYCols = kMaxN;
    static constexpr int kYBufs = (int)((kTmemCols - kColY) / kYCols);
};

template <class G>
struct TcSmem {
    uint64_t full[G::kAStages];   // weight stage ready: TMA bytes landed (bf16) / converted (FP8)
    uint64_t empty[G::kAStages];  // MMAs reading the weight stage are done
    uint64_t full8[G::kF8Stages > 0 ? G::kF8Stages : 1];   // gate / up code box landed (MMA waits)
    uint64_t full8d[G::kF8Stages > 0 ? G::kF8Stages : 1];  // down code box landed (converters wait)
    uint64_t empty8[G::kF8Stages > 0 ? G::kF8Stages : 1];  // code box slot free again
    uint64_t bx_full[G::kBPairs];  // activation K-pair gathered
    uint64_t bx_empty[G::kBPairs]; // MMAs reading the activation K-pair are done
    uint64_t acc_full, acc_empty, h_full, mma_done;
    uint64_t y_full[G::kYBufs], y_empty[G::kYBufs];
    uint32_t tmem_base;
    int cls_units[3];
    int cls_groups[3];
    int cls_off[3];
    int ep_row[4][G::kTok];       // epilogue warps: output row of each tile token
    float ep_w[4][G::kTok];       // ... and its routing weight
    float ep_xs[4][G::kTok];      // ... and (E4M3 terms) 2^-e0 of its activation row
    // form-P down pass: each tile token's assignments in the department
    // (zbuf row and routing weight)
    int pd_cnt[G::kPdTok];
    int pd_pos[G::kPdTok][kMaxK];
    float pd_w[G::kPdTok][kMaxK];
    int4 units[1];                // per class: {unit, first entry, tokens, group prefix}
};

// E4M3 -> bf16 on the integer and FMA pipes (the conversion instructions
// issue at a quarter of their rate).  A code
// s eeee mmm and the bf16 pattern s 0000eeee mmm0000 have the same sign and
// significand, and the pattern's value is the code's times 2^-120 (exponent
// bias 127 against 7); codes with eeee = 0 (E4M3 subnormals) land on bf16
// subnormals with the same scaling.  So each code of a pair goes to its own
// 16-bit half, the magnitude bits move up by 4, the sign from bit 11 to bit 15
// (t + 15 (t & m) moves a set bit 11 to bit 15, bits 12-15 being clear), and
// one bf16 multiply by 2^120 restores the value; it is exact, every code
// value being a bf16 normal.  sel picks the pair: 0x4140 codes 0 and 1 of the
// word, 0x4342 codes 2 and 3; code 2i+0 lands in the low half.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t w, uint32_t sel) {
    const uint32_t t = __byte_perm(w, 0u, sel) << 4;
    const uint32_t r = t + 15u * (t & 0x08000800u);
    const __nv_bfloat162 v = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&r),
                                     __halves2bfloat162(__ushort_as_bfloat16((unsigned short)0x7B80u),
                                                        __ushort_as_bfloat16((unsigned short)0x7B80u)));
    return *reinterpret_cast<const uint32_t*>(&v);
}

// 16 E4M3 codes (one 16-byte load, code 0 in the low byte) -> 16 bf16 values
// in two 16-byte units, in order.
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 w, uint4& o0, uint4& o1) {
    o0 = make_uint4(e4m3x2_to_bf16x2(w.x, 0x4140u), e4m3x2_to_bf16x2(w.x, 0x4342u),
                    e4m3x2_to_bf16x2(w.y, 0x4140u), e4m3x2_to_bf16x2(w.y, 0x4342u));
    o1 = make_uint4(e4m3x2_to_bf16x2(w.z, 0x4140u), e4m3x2_to_bf16x2(w.z, 0x4342u),
                    e4m3x2_to_bf16x2(w.w, 0x4140u), e4m3x2_to_bf16x2(w.w, 0x4342u));
}

struct TSeg {
    int cls, q, grp, row0;
};

// Next tile (kTcRows rows) of the CTA's row range [r, r_end).
template <class S>
__device__ __forceinline__ bool next_tile(const TcArgs& a, const S& sm, int& r, int r_end, TSeg& s) {
    if (r >= r_end) return false;
    int base = 0, c = 0;
    while (c < a.f.ncls - 1 && r >= base + a.f.cls[c].rows * sm.cls_groups[c]) {
        base += a.f.cls[c].rows * sm.cls_groups[c];
        ++c;
    }
    const int rows = a.f.cls[c].rows;
    const int rel = r - base;
    const int vg = rel / rows;
    const int4* u = sm.units + sm.cls_off[c];
    int lo = 0, hi = sm.cls_units[c] - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (u[mid].w > vg) hi = mid; else lo = mid + 1;
    }
    s.cls = c;
    s.q = lo;
    s.grp = vg - (lo > 0 ? u[lo - 1].w : 0);
    s.row0 = rel - vg * rows;
    r += kTcRows;
    return true;
}

// Token t, routing weight and output row of entry j of a unit's token list
// (from the CTA's own lists on the in-CTA routing path, LOCAL).
template <bool LOCAL>
__device__ __forceinline__ void tile_token(const TcArgs& a, const LocalRoute& lr, int kind, int entry,
                                           int& t, float& w, int& row) {
    if (LOCAL) {
        local_entry(lr, kind, entry, t, w);
        row = t;
        return;
    }
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
    // a token id from the workspace outside [0, T) (a workspace the dispatch
    // did not write for this step) is reported, never used as an address
    if ((unsigned)t >= (unsigned)a.f.T) {
        set_status(a.f.ws.status, kDevErrRouting);
        t = 0;
        w = 0.0f;
    }
    if (a.f.out_mode == MOE_OUT_ACCUM) row = t;
}

// LOCAL: the in-CTA routing path (a.f.local_route); a separate instantiation
// so that the path reading the dispatch from global memory keeps its code.
// F8: E4M3 weights with row scales (converter warps, TcGeo<true>).
template <bool LOCAL, bool F8>
__global__ void __launch_bounds__(TcGeo<F8>::kThreads, 1) ffn_tc_kernel(const __grid_constant__ TcArgs a) {
    using G = TcGeo<F8>;
    constexpr int kTcTokens = G::kTok;
    constexpr int kTcStages = G::kAStages;
    constexpr int kF8Stages = G::kF8Stages;
    constexpr int kTcBPairs = G::kBPairs;
    constexpr int kBBlock = G::kBBlock, kBPair = G::kBPair, kHChunk = G::kHChunk, kHTile = G::kHTile;
    constexpr int kYStage = G::kYStage;
    constexpr int kTcWarps = G::kWarps, kTcThreads = G::kThreads;
    constexpr uint32_t kColG = G::kColG, kColU = G::kColU, kColY = G::kColY, kYCols = G::kYCols;
    constexpr int kYBufs = G::kYBufs;
    extern __shared__ unsigned char smem_dyn[];
    // 1024-byte aligned tile regions (128 B swizzle atoms)
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    unsigned char* f8ring = base;                    // FP8: code boxes (empty for bf16)
    unsigned char* aring = f8ring + kF8Stages * kF8Box;
    unsigned char* bring = aring + kTcStages * G::kASlot;
    unsigned char* htile = bring + kTcBPairs * kBPair;
    float* ystage = reinterpret_cast<float*>(htile + kHTile);
    TcSmem<G>& sm = *reinterpret_cast<TcSmem<G>*>(htile + kHTile + kYStage);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.f.d;
    const int KP = d / 128, DT = d / 128;          // K-pairs (gate/up), M-tiles (down)
    // The CTAs take the down M-tiles (128 output columns each) in orders
    // rotated by the block index, so that their output reductions spread
    // over the whole row of y instead of all landing on the same columns.
    const int mt_rot = (int)(blockIdx.x % (unsigned)DT);

    if (tid == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(&sm.full[i], F8 ? G::kCvtWarps : 1);
            mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < kF8Stages; ++i) {
            mbar_init(&sm.full8[i], 1);
            mbar_init(&sm.full8d[i], 1);
            mbar_init(&sm.empty8[i], 1);
        }
        for (int i = 0; i < kTcBPairs; ++i) {
            mbar_init(&sm.bx_full[i], 4);
            mbar_init(&sm.bx_empty[i], 1);
        }
        mbar_init(&sm.acc_full, 1);
        mbar_init(&sm.acc_empty, 4);
        mbar_init(&sm.h_full, 4);
        mbar_init(&sm.mma_done, 1);
        for (int b = 0; b < kYBufs; ++b) {
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
    // in-CTA routing: its state follows the unit table
    LocalRoute lr = {};
    if (LOCAL) {
        int cap = 0;
        for (int c = 0; c < a.f.ncls; ++c) cap += class_capacity(a.f.cls[c], a.f.n, a.f.g);
        lr = local_route_at(reinterpret_cast<unsigned char*>(sm.units + cap), a.f.T, a.f.n, a.f.k, a.f.g,
                            kTcWarps);
        for (int i = tid; i < a.f.n * lr.W; i += kTcThreads) lr.emask[i] = 0u;
        if (tid == 0) {
            int off = 0;
            for (int c = 0; c < a.f.ncls; ++c) {
                sm.cls_off[c] = off;
                off += class_capacity(a.f.cls[c], a.f.n, a.f.g);
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;

    // The next layer's routing grid (a programmatic dependent) may take SMs
    // as this grid's CTAs finish; it waits for this grid's completion.
    if (MOE_ROUTE_PDL) pdl_allow_dependents();
    // Everything below reads what the routing / dispatch kernel wrote.
    pdl_wait_primary();
    if (a.pmode == kTcFormPUp) {
        // the private pass adds into the assignment rows, the down pass into
        // y (when no routing kernel cleared it): clear them here
        const long long z4 = (long long)a.f.T * a.f.k * a.f.cls[0].rows / 4;
        for (long long i = blockIdx.x * (long long)kTcThreads + tid; i < z4; i += (long long)gridDim.x * kTcThreads)
            reinterpret_cast<float4*>(a.zbuf)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.zero_y) {
            const long long y4 = (long long)a.f.T * a.f.d / 4;
            for (long long i = blockIdx.x * (long long)kTcThreads + tid; i < y4; i += (long long)gridDim.x * kTcThreads)
                reinterpret_cast<float4*>(a.f.out)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    const bool has_gu = a.pmode != kTcFormPDown;    // gate / up rows of each tile
    const bool has_dn = a.pmode != kTcFormPUp;      // down rows of each tile

    // ---- unit table: on the in-CTA routing path every unit, built here from
    // the router logits (CTA 0 also stores the routing and the dispatch).
    // Otherwise this kernel's units (>= min_tokens tokens), groups of kTcTokens;
    // warp c filters class c.  With auto_tc the kernel takes every unit when
    // prefer_tc() holds and none otherwise (the CUDA-core kernel decides alike). ----
    if (LOCAL) {
        const bool writer = blockIdx.x == 0;
        local_topk<kTcThreads>(a.f, lr, writer);
        const UnitTableView view = {sm.units, sm.cls_off, sm.cls_units, sm.cls_groups, nullptr, nullptr};
        local_tables<kTcThreads, kTcTokens, false>(a.f, view, lr, writer);
        if (writer && tid == 0) a.f.ws.sync[1] = 2u;
    } else {
    __shared__ int s_min_tok;
    if (tid == 0) {
        const bool take = a.f.auto_tc && prefer_tc(a.f);
        s_min_tok = a.f.auto_tc ? (take ? 1 : INT_MAX) : a.min_tokens;
        // launched first: record the choice for the CUDA-core kernel that follows
        if (a.f.tc_first && blockIdx.x == 0) a.f.ws.sync[1] = take ? 2u : 1u;
    }
    __syncthreads();
    const int min_tok = s_min_tok;
    if (warp < a.f.ncls) {
        int off = 0;
        for (int c = 0; c < warp; ++c) off += class_capacity(a.f.cls[c], a.f.n, a.f.g);
        {
            const int c = warp;
            const UnitClass& uc = a.f.cls[c];
            int kept, groups;
            if (uc.kind == kUnitShared) {
                const bool keep = a.f.T >= min_tok;
                kept = keep ? 1 : 0;
                groups = keep ? (a.f.T + kTcTokens - 1) / kTcTokens : 0;
                if (lane == 0 && keep) sm.units[off] = make_int4(0, 0, a.f.T, groups);
            } else {
                const int4* src = uc.kind == kUnitDept ? a.f.ws.dept_units : a.f.ws.exp_units;
                const int A = uc.kind == kUnitDept ? a.f.ws.counts[1] : a.f.ws.counts[0];
                kept = filter_units_warp(src, A, min_tok, 1 << 30, kTcTokens, sm.units + off,
                                         &groups);
            }
            if (lane == 0) {
                sm.cls_units[c] = kept;
                sm.cls_groups[c] = groups;
                sm.cls_off[c] = off;
            }
        }
    }
    __syncthreads();
    }

    // CTA's share of the row space, in whole tiles
    int Q = 0;
    for (int c = 0; c < a.f.ncls; ++c) Q += a.f.cls[c].rows / kTcRows * sm.cls_groups[c];
    const int r_begin = (int)grid_share(Q, blockIdx.x, gridDim.x, a.f.grid_magic) * kTcRows;
    const int r_end = (int)grid_share(Q, blockIdx.x + 1, gridDim.x, a.f.grid_magic) * kTcRows;

    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (!ok) return false;
        if (!mbar_wait_bounded(bar, parity, ffn_wait_limit(a.f))) {
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
            // the ring TMA writes: the MMAs' (bf16) or the code boxes (FP8),
            // whose gate / up boxes complete on full8 (the MMA reads them)
            // and down boxes on full8d (the converters read them): each
            // barrier has one waiter, which takes its phases in order
            constexpr int NS = F8 ? kF8Stages : kTcStages;
            constexpr int SB = F8 ? kF8Box : G::kASlot;
            unsigned char* ring = F8 ? f8ring : aring;
            uint64_t* emptyb = F8 ? sm.empty8 : sm.empty;
            uint32_t par_g = 0u, par_d = 0u, last_d = 0u;   // per slot: next phase parity, last box kind
            // columns [128 cb, 128 cb + 128) of weight rows [y, y + 128)
            auto load = [&](const CUtensorMap* m, int y, int cb, bool down) -> bool {
                const int slot = it % NS;
                if (!wait(&emptyb[slot], ((it / NS) & 1u) ^ 1u)) return false;
                uint64_t* fb = F8 ? (down ? &sm.full8d[slot] : &sm.full8[slot]) : &sm.full[slot];
                mbar_arrive_expect_tx(fb, SB);
                if (F8) tma_load_2d(ring + slot * SB, m, 128 * cb, y, fb, pol);
                else tma_load_3d(ring + slot * SB, m, 0, y, 2 * cb, fb, pol);
                const uint32_t bit = 1u << slot;
                if (down) {
                    par_d ^= bit;
                    last_d |= bit;
                } else {
                    par_g ^= bit;
                    last_d &= ~bit;
                }
                ++it;
                return true;
            };
            while (ok && !a.f.stall_copies && next_tile(a, sm, r, r_end, s)) {
                const int4 rec = sm.units[sm.cls_off[s.cls] + s.q];
                const int y = rec.x * a.f.cls[s.cls].rows + s.row0;
                const CUtensorMap* maps = a.maps[s.cls];
                for (int p = 0; ok && has_gu && p < KP; ++p) {
                    if (!load(&maps[0], y, p, false)) break;
                    if (!load(&maps[1], y, p, false)) break;
                }
                for (int mt = 0; ok && has_dn && mt < DT; ++mt) {
                    const int mc = mt + mt_rot < DT ? mt + mt_rot : mt + mt_rot - DT;
                    if (!load(&maps[2], y, mc, F8)) break;
                }
            }
            // every issued copy must land before the CTA may exit: the last
            // copy into each slot (the earlier ones were waited for before
            // the slot was refilled), on the barrier it completes
            for (int slot = 0; slot < NS && slot < (int)it; ++slot) {
                const bool dn = (last_d >> slot) & 1u;
                uint64_t* fb = F8 ? (dn ? &sm.full8d[slot] : &sm.full8[slot]) : &sm.full[slot];
                mbar_wait_bounded(fb, (((dn ? par_d : par_g) >> slot) & 1u) ^ 1u);
            }
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (lane == 0) {
            uint32_t it = 0, bp = 0, ti = 0, dtc = 0;
            uint32_t it8 = 0, par_g = 0u;   // FP8: code boxes taken; per slot, next full8 phase parity
            int r = r_begin;
            TSeg s;
            // descriptors: address field += byte offset >> 4 (all of smem < 256 KB)
            const uint64_t a_k = smem_desc_sw128(smem_u32(aring), 16, 1024);          // K-major
            const uint64_t a_mn = smem_desc_sw128(smem_u32(aring), G::kAChunk, 1024);  // MN-major
            const uint64_t b_k = smem_desc_sw128(smem_u32(bring), 16, 1024);
            const uint64_t h_k = smem_desc_sw128(smem_u32(htile), 16, 1024);
            const uint64_t a8 = smem_desc_sw128(smem_u32(f8ring), 16, 1024);         // code boxes, K-major
            while (ok && next_tile(a, sm, r, r_end, s)) {
                const int4 rec = sm.units[sm.cls_off[s.cls] + s.q];
                const int mg = min(kTcTokens, rec.z - s.grp * kTcTokens);
                const int N = 2 * ((mg + 7) & ~7);
                const uint32_t id_gu = F8 ? idesc_e4m3_f32(128, G::kBTerms * (N / 2))
                                          : idesc_bf16_f32(128, N, false, false);
                const uint32_t id_dn = idesc_bf16_f32(128, N, true, false);
                if (has_gu) {
                if (!wait(&sm.acc_empty, (ti & 1u) ^ 1u)) break;
                tc_fence_after_sync();
                for (int p = 0; ok && p < KP; ++p, ++bp) {
                    const uint32_t bslot = bp % kTcBPairs;
                    if (!wait(&sm.bx_full[bslot], (bp / kTcBPairs) & 1u)) break;
                    const uint64_t bd = b_k + ((bslot * kBPair) >> 4);
                    if constexpr (F8) {
                        // A: the code box itself (128 rows x 128 codes, K-major,
                        // 128 B swizzle); B: the activation terms; K = 32 a MMA
#pragma unroll
                        for (int gu = 0; gu < 2; ++gu, ++it8) {
                            const uint32_t slot = it8 % kF8Stages;
                            const uint32_t par = (par_g >> slot) & 1u;
                            par_g ^= 1u << slot;
                            if (!wait(&sm.full8[slot], par)) break;
                            tc_fence_after_sync();
                            const uint32_t acc_col = tmem + (gu ? kColU : kColG);
                            const uint64_t ad = a8 + ((slot * kF8Box) >> 4);
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                umma_e4m3(acc_col, ad + ((ks * 32) >> 4), bd + ((ks * 32) >> 4), id_gu,
                                          (p | ks) ? 1u : 0u);
                            umma_commit(&sm.empty8[slot]);
                        }
                    } else {
#pragma unroll
                    for (int gu = 0; gu < 2; ++gu, ++it) {
                        const uint32_t slot = it % kTcStages;
                        if (!wait(&sm.full[slot], (it / kTcStages) & 1u)) break;
                        tc_fence_after_sync();
                        const uint32_t acc_col = tmem + (gu ? kColU : kColG);
                        const uint64_t ad = a_k + ((slot * G::kASlot) >> 4);
#pragma unroll
                        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                umma_bf16(acc_col, ad + ((kb * kChunkBytes + ks * 32) >> 4),
                                          bd + ((kb * kBBlock + ks * 32) >> 4), id_gu,
                                          (p | kb | ks) ? 1u : 0u);
                        umma_commit(&sm.empty[slot]);
                    }
                    }
                    umma_commit(&sm.bx_empty[bslot]);
                }
                if (!ok) break;
                umma_commit(&sm.acc_full);
                }
                if (!has_dn) {
                    ++ti;
                    continue;
                }
                if (!wait(&sm.h_full, ti & 1u)) break;
                tc_fence_after_sync();
                // down: M-tile mt = 128 hidden columns; A is W_down read MN-major
                // (chunk slabs kAChunk apart), K = the tile's 128 rows, in
                // slots of kCRows rows
                constexpr int kSlotsPerTile = kTcRows / G::kCRows;
                for (int mt = 0; ok && mt < DT; ++mt, ++dtc) {
                    const uint32_t yb = dtc % kYBufs;
                    if (!wait(&sm.y_empty[yb], ((dtc / kYBufs) & 1u) ^ 1u)) break;
                    const uint32_t ycol = tmem + kColY + yb * kYCols;
                    for (int h = 0; h < kSlotsPerTile; ++h, ++it) {
                        const uint32_t slot = it % kTcStages;
                        if (!wait(&sm.full[slot], (it / kTcStages) & 1u)) break;
                        if (F8 && h == kSlotsPerTile - 1) {
                            // the converters are done with the code box: its
                            // slot may be refilled
                            mbar_arrive(&sm.empty8[it8 % kF8Stages]);
                            ++it8;
                        }
                        tc_fence_after_sync();
                        const uint64_t ad = a_mn + ((slot * G::kASlot) >> 4);
#pragma unroll
                        for (int ks = 0; ks < G::kCRows / 16; ++ks) {
                            const int kg = h * (G::kCRows / 16) + ks;   // K step in the tile
                            umma_bf16(ycol, ad + ((ks * 2048) >> 4),
                                      h_k + (((kg >> 2) * kHChunk + (kg & 3) * 32) >> 4), id_dn,
                                      kg ? 1u : 0u);
                        }
                        umma_commit(&sm.empty[slot]);
                    }
                    if (!ok) break;
                    umma_commit(&sm.y_full[yb]);
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
        // H is K-major [K chunk][token row][128 B]: this thread's K index is m
        unsigned char* hcol = htile + (m >> 6) * kHChunk + (m & 7) * 2;
        const int hchunk = (m & 63) >> 3;
        uint32_t ti = 0, dtc = 0;
        int r = r_begin;
        TSeg s;
        while (ok && next_tile(a, sm, r, r_end, s)) {
            const int4 rec = sm.units[sm.cls_off[s.cls] + s.q];
            const int kind = a.f.cls[s.cls].kind;
            const int first = rec.y + s.grp * kTcTokens;
            const int mg = min(kTcTokens, rec.z - s.grp * kTcTokens);
            const int Mp = (mg + 7) & ~7;
            if (lane < mg) {
                int t, row;
                float w;
                tile_token<LOCAL>(a, lr, kind, first + lane, t, w, row);
                sm.ep_row[quarter][lane] = row;
                sm.ep_w[quarter][lane] = w;
                if constexpr (F8) {
                    // 2^-e0 of the token's activation terms (e0 in [-120, 114])
                    const int e0 = reinterpret_cast<const int32_t*>(
                        reinterpret_cast<const unsigned char*>(a.f.ws.xb) + xq_exp_offset(a.f.T))[t];
                    sm.ep_xs[quarter][lane] = __int_as_float((127 - e0) << 23);
                }
            }
            // FP8: this thread's weight row's scales (gate, up, down)
            float sg = 1.0f, su = 1.0f, sdn = 1.0f;
            if constexpr (F8) {
                const UnitClass& uc = a.f.cls[s.cls];
                const size_t ur = (size_t)rec.x * uc.rows + s.row0 + m;
                sg = __ldg(uc.sc_gate + ur);
                su = __ldg(uc.sc_up + ur);
                sdn = __ldg(uc.sc_down + ur);
            }
            __syncwarp();
            if (a.pmode == kTcFormPDown) {
                // H[row, token] = sum over the token's experts i in the
                // department of p_i SiLU(Z_i[row]).  Warp 2 collects each tile
                // token's assignments (zbuf row, routing weight) and the four
                // epilogue warps meet at named barrier 1 after that; they also
                // meet at the end of every tile (below), where they agree on
                // their waits' outcomes, so that all of them reach this barrier
                // or none does.
                if (warp == 2 && lane < mg) {
                    const int t = sm.ep_row[2][lane];
                    int c = 0;
                    for (int sl = 0; sl < a.f.k; ++sl) {
                        const int e = a.topk_idx[t * a.f.k + sl];
                        if (e / a.f.g == rec.x && c < kMaxK) {
                            const int p = a.f.ws.tok_asg[t * a.f.k + sl];
                            sm.pd_pos[lane][c] = p;
                            sm.pd_w[lane][c] = a.f.ws.asg_w[p];
                            ++c;
                        }
                    }
                    sm.pd_cnt[lane] = c;
                }
                named_bar_sync(1, 128);
                const int rws = a.f.cls[0].rows;
                for (int c0 = 0; c0 < Mp; c0 += 16) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = c0 + jj;
                        if (j < mg) {
                            float h = 0.0f;
                            for (int c = 0; c < sm.pd_cnt[j]; ++c)
                                h += sm.pd_w[j][c] *
                                     silu_f(__ldcg(a.zbuf + (size_t)sm.pd_pos[j][c] * rws + s.row0 + m));
                            const __nv_bfloat16 hh = __float2bfloat16_rn(h);
                            const __nv_bfloat16 hl = __float2bfloat16_rn(h - __bfloat162float(hh));
                            const int jl = Mp + j;
                            *reinterpret_cast<__nv_bfloat16*>(hcol + j * 128 + ((hchunk ^ (j & 7)) << 4)) = hh;
                            *reinterpret_cast<__nv_bfloat16*>(hcol + jl * 128 + ((hchunk ^ (jl & 7)) << 4)) = hl;
                        }
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.h_full);
            } else {
            if (!wait(&sm.acc_full, ti & 1u)) break;
            tc_fence_after_sync();
            if (a.pmode == kTcFormPUp) {
                // G = SiLU(W_g x), U = SiLU(W_u x) of each department entry
                const int rws = a.f.cls[0].rows;
                for (int c0 = 0; c0 < Mp; c0 += 16) {
                    uint32_t ghi[16], glo[16], uhi[16], ulo[16];
                    tmem_ld16_async(tmem + lanes + kColG + c0, ghi);
                    tmem_ld16_async(tmem + lanes + kColG + Mp + c0, glo);
                    tmem_ld16_async(tmem + lanes + kColU + c0, uhi);
                    tmem_ld16_async(tmem + lanes + kColU + Mp + c0, ulo);
                    tmem_wait_ld();
                    tmem_regs_ready(ghi);
                    tmem_regs_ready(glo);
                    tmem_regs_ready(uhi);
                    tmem_regs_ready(ulo);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = c0 + jj;
                        if (j < mg) {
                            const size_t o = (size_t)(first + j) * rws + s.row0 + m;
                            a.gbuf[o] = silu_f(__uint_as_float(ghi[jj]) + __uint_as_float(glo[jj]));
                            a.ubuf[o] = silu_f(__uint_as_float(uhi[jj]) + __uint_as_float(ulo[jj]));
                        }
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.acc_empty);
                ++ti;
                continue;
            }
            for (int c0 = 0; c0 < Mp; c0 += 16) {
                // every column of the block is computed (the unused ones from
                // whatever TMEM holds) and only the stores are guarded, so the
                // sixteen chains interleave
                float hv[16];
                if constexpr (F8) {
                    // g = 2^-e0 sum_p 16^-p G_p, the same for u; then the rows' scales
                    float gs[16], us[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) gs[jj] = us[jj] = 0.0f;
                    // two terms per TMEM round trip
#pragma unroll
                    for (int p = 0; p < kXTerms; p += 2) {
                        uint32_t g0[16], u0[16], g1[16], u1[16];
                        tmem_ld16_async(tmem + lanes + kColG + p * Mp + c0, g0);
                        tmem_ld16_async(tmem + lanes + kColU + p * Mp + c0, u0);
                        tmem_ld16_async(tmem + lanes + kColG + (p + 1) * Mp + c0, g1);
                        tmem_ld16_async(tmem + lanes + kColU + (p + 1) * Mp + c0, u1);
                        tmem_wait_ld();
                        tmem_regs_ready(g0);
                        tmem_regs_ready(u0);
                        tmem_regs_ready(g1);
                        tmem_regs_ready(u1);
                        const float f0 = 1.0f / (float)(1 << (4 * p)), f1 = f0 * (1.0f / 16.0f);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            gs[jj] += __uint_as_float(g0[jj]) * f0 + __uint_as_float(g1[jj]) * f1;
                            us[jj] += __uint_as_float(u0[jj]) * f0 + __uint_as_float(u1[jj]) * f1;
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const float xs = sm.ep_xs[quarter][(c0 + jj) & (kTcTokens - 1)];
                        hv[jj] = silu_fast(gs[jj] * xs * sg) * (us[jj] * xs * su) * sdn;
                        if (a.f.out_mode == MOE_OUT_ACCUM) hv[jj] *= sm.ep_w[quarter][(c0 + jj) & (kTcTokens - 1)];
                    }
                } else {
                    // the four loads of a column block share one completion wait
                    uint32_t ghi[16], glo[16], uhi[16], ulo[16];
                    tmem_ld16_async(tmem + lanes + kColG + c0, ghi);
                    tmem_ld16_async(tmem + lanes + kColG + Mp + c0, glo);
                    tmem_ld16_async(tmem + lanes + kColU + c0, uhi);
                    tmem_ld16_async(tmem + lanes + kColU + Mp + c0, ulo);
                    tmem_wait_ld();
                    tmem_regs_ready(ghi);
                    tmem_regs_ready(glo);
                    tmem_regs_ready(uhi);
                    tmem_regs_ready(ulo);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        hv[jj] = silu_fast(__uint_as_float(ghi[jj]) + __uint_as_float(glo[jj])) *
                                 (__uint_as_float(uhi[jj]) + __uint_as_float(ulo[jj]));
                        if (a.f.out_mode == MOE_OUT_ACCUM) hv[jj] *= sm.ep_w[quarter][c0 + jj];
                    }
                }
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int j = c0 + jj;
                    if (j < mg) {
                        const float h = hv[jj];
                        const __nv_bfloat16 hh = __float2bfloat16_rn(h);
                        const __nv_bfloat16 hl = __float2bfloat16_rn(h - __bfloat162float(hh));
                        const int jl = Mp + j;
                        *reinterpret_cast<__nv_bfloat16*>(hcol + j * 128 + ((hchunk ^ (j & 7)) << 4)) = hh;
                        *reinterpret_cast<__nv_bfloat16*>(hcol + jl * 128 + ((hchunk ^ (jl & 7)) << 4)) = hl;
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
            }
            // Down outputs: each warp transposes its 32 columns of the M-tile
            // through its own shared-memory block, so that a lane adds four
            // consecutive columns of one token per vector atomic (a quarter
            // of the atomic instructions of one per element and token).
            float* wst = ystage + quarter * (kTcTokens * 32);
            for (int dt = 0; ok && dt < DT; ++dt, ++dtc) {
                const uint32_t yb = dtc % kYBufs;
                if (!wait(&sm.y_full[yb], (dtc / kYBufs) & 1u)) break;
                tc_fence_after_sync();
                const uint32_t ycol = kColY + yb * kYCols;
                for (int c0 = 0; c0 < Mp; c0 += 16) {
                    uint32_t yhi[16], ylo[16];
                    tmem_ld16_async(tmem + lanes + ycol + c0, yhi);
                    tmem_ld16_async(tmem + lanes + ycol + Mp + c0, ylo);
                    tmem_wait_ld();
                    tmem_regs_ready(yhi);
                    tmem_regs_ready(ylo);
                    if (c0 + 16 >= Mp) {
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sm.y_empty[yb]);
                    }
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        wst[(c0 + jj) * 32 + lane] = __uint_as_float(yhi[jj]) + __uint_as_float(ylo[jj]);
                }
                __syncwarp();
                const int dc = dt + mt_rot < DT ? dt + mt_rot : dt + mt_rot - DT;   // the producer's order
                float* ybase = a.f.out + dc * 128 + quarter * 32;
                for (int q = lane; q < mg * 8; q += 32) {
                    const int j = q >> 3, c4 = (q & 7) * 4;
                    const float4 v = *reinterpret_cast<const float4*>(wst + j * 32 + c4);
                    atomicAdd(reinterpret_cast<float4*>(ybase + (size_t)sm.ep_row[quarter][j] * d + c4), v);
                }
                __syncwarp();
            }
            __syncwarp();
            ++ti;
            if (a.pmode == kTcFormPDown && named_bar_or(1, 128, !ok)) ok = false;
        }
    } else if (warp < 10) {
        // ===================== activation gather =====================
        // B tiles (one 128-column K step per slot) are copied with cp.async
        // from the split activations (once per layer), kPre steps ahead of
        // the MMA: B row n = term * Mp + j holds term n / Mp (bf16 hi, lo; or
        // E4M3 term 0..3) of the tile's token j, 128 bytes per K-block.
        constexpr int kPre = kTcBPairs - 1;
        const int ct = tid - 6 * 32;                    // 0..127
        const unsigned char* xs = reinterpret_cast<const unsigned char*>(a.f.ws.xb);
        // bytes of one term's [T, d] rows, and of one row
        const size_t term_bytes = (size_t)a.f.T * d * (F8 ? 1 : 2), row_bytes = (size_t)d * (F8 ? 1 : 2);
        uint32_t bp = 0;
        int r = r_begin;
        TSeg s;
        while (ok && has_gu && next_tile(a, sm, r, r_end, s)) {
            const int4 rec = sm.units[sm.cls_off[s.cls] + s.q];
            const int kind = a.f.cls[s.cls].kind;
            const int first = rec.y + s.grp * kTcTokens;
            const int mg = min(kTcTokens, rec.z - s.grp * kTcTokens);
            const int Mp = (mg + 7) & ~7;
            const int items = G::kBTerms * Mp * 8;      // (B row, 16-byte chunk) pairs per K-block
            // this thread's items are fixed for the tile: resolve them once
            const unsigned char* src[4];
            int dst[4];
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const int item = ct + k4 * 128;
                const int n = item >> 3, c = item & 7;
                const int term = n / Mp, j = n - term * Mp;
                src[k4] = nullptr;
                dst[k4] = item < items ? n * 128 + ((c ^ (n & 7)) << 4) : -1;
                if (item < items && j < mg) {
                    int t, row;
                    float w;
                    tile_token<LOCAL>(a, lr, kind, first + j, t, w, row);
                    src[k4] = xs + term * term_bytes + (size_t)t * row_bytes + c * 16;
                }
            }
            auto issue = [&](int p) -> bool {
                const uint32_t b = bp + p;
                const int slot = b % kTcBPairs;
                if (!wait(&sm.bx_empty[slot], ((b / kTcBPairs) & 1u) ^ 1u)) return false;
                unsigned char* Bt = bring + slot * kBPair;
#pragma unroll
                for (int kb = 0; kb < G::kBBlocks; ++kb)
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        if (dst[k4] >= 0) {
                            unsigned char* dp = Bt + kb * kBBlock + dst[k4];
                            if (src[k4]) cp_async16(dp, src[k4] + (size_t)(G::kBBlocks * p + kb) * 128);
                            else *reinterpret_cast<uint4*>(dp) = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                cp_async_commit();
                return true;
            };
            // exactly kPre groups in flight before the first wait (empty ones
            // when the tile has fewer pairs), one more per pair after.  Pair
            // p is handed to the MMA as soon as it lands, before the copies of
            // pair p + kPre wait for the MMA to release a slot, so that the
            // MMAs of pair p never wait on those of pair p - 1.
            for (int p = 0; ok && p < kPre; ++p) {
                if (p < KP) {
                    if (!issue(p)) break;
                } else {
                    cp_async_commit();
                }
            }
            for (int p = 0; ok && p < KP; ++p) {
                cp_async_wait<kPre - 1>();              // pair p has landed
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.bx_full[(bp + p) % kTcBPairs]);
                if (p + kPre < KP) {
                    if (!issue(p + kPre)) break;
                } else {
                    cp_async_commit();                  // keep one group per pair
                }
            }
            bp += KP;
        }
        cp_async_wait<0>();
    } else if constexpr (F8) {
        // ===================== FP8 converters =====================
        // Down code boxes (128 rows of W_down x 128 hidden columns, landed
        // with the 128 B swizzle: unit u of row r at u ^ (r & 7)) -> the bf16
        // shared-memory ring the down MMAs read MN-major.  Warp cw expands
        // rows [32 cw, 32 cw + 32), four rows a step; within a step the eight
        // lanes of each shared-memory phase read half a row each of two
        // adjacent rows and write their bf16 units to one chunk's even and
        // the other chunk's odd swizzled positions, so neither the loads nor
        // the stores conflict.  Gate / up boxes go to the MMA as they are.
        constexpr int kRowsPerCvt = G::kCRows / G::kCvtWarps;   // rows of each slot per warp
        const int cw = warp - 10;
        const int pr = lane >> 4, ph = (lane >> 3) & 1, sub = (lane >> 2) & 1;
        const int q = ((sub ^ ph) << 2) | (lane & 3);   // 16-code unit of the row
        const int rsub = 2 * pr + sub;                   // row within the step
        const int u0 = 2 * (q & 3);                      // first bf16 unit in the chunk
        uint32_t it8 = 0, itc = 0, par_d = 0u;           // boxes, bf16 slots, per-slot full8d parity
        int r = r_begin;
        TSeg s;
        while (cw < G::kCvtWarps && ok && next_tile(a, sm, r, r_end, s)) {
            it8 += 2 * KP;                               // the tile's gate / up boxes
            for (int mt = 0; ok && mt < DT; ++mt, ++it8) {
                const uint32_t s8 = it8 % kF8Stages;
                const uint32_t par = (par_d >> s8) & 1u;
                par_d ^= 1u << s8;
                if (!wait(&sm.full8d[s8], par)) break;
                const unsigned char* box = f8ring + s8 * kF8Box;
                for (int h = 0; h < kTcRows / G::kCRows; ++h, ++itc) {
                    const uint32_t sc = itc % kTcStages;
                    if (!wait(&sm.empty[sc], ((itc / kTcStages) & 1u) ^ 1u)) break;
                    unsigned char* dst = aring + sc * G::kASlot + (q >> 2) * G::kAChunk;
                    // all loads first: the compiler cannot tell the two rings
                    // apart and would otherwise keep each load behind the
                    // previous step's stores
                    uint4 w[kRowsPerCvt / 4];
#pragma unroll
                    for (int i = 0; i < kRowsPerCvt / 4; ++i) {
                        const int row = h * G::kCRows + cw * kRowsPerCvt + i * 4 + rsub;   // row of the box
                        w[i] = *reinterpret_cast<const uint4*>(box + row * 128 + ((q ^ (row & 7)) << 4));
                    }
#pragma unroll
                    for (int i = 0; i < kRowsPerCvt / 4; ++i) {
                        const int row = cw * kRowsPerCvt + i * 4 + rsub;                    // row of the slot
                        uint4 o0, o1;
                        e4m3x16_to_bf16(w[i], o0, o1);
                        unsigned char* drow = dst + row * 128;
                        *reinterpret_cast<uint4*>(drow + ((u0 ^ (row & 7)) << 4)) = o0;
                        *reinterpret_cast<uint4*>(drow + (((u0 + 1) ^ (row & 7)) << 4)) = o1;
                    }
                    fence_async_smem();      // the stores are read by the MMA (async proxy)
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.full[sc]);
                }
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

template <bool F8>
static size_t tc_smem_bytes(int units, const FfnArgs* local) {
    using G = TcGeo<F8>;
    return 1024 + (size_t)G::kF8Stages * kF8Box + (size_t)G::kAStages * G::kASlot + (size_t)G::kBPairs * G::kBPair +
           G::kHTile + G::kYStage + sizeof(TcSmem<G>) + (size_t)units * sizeof(int4) +
           (local ? local_route_bytes(local->T, local->n, local->k, local->g, G::kWarps) : 0);
}

size_t ffn_tc_smem_bytes(int units, const FfnArgs* local, bool f8) {
    return f8 ? tc_smem_bytes<true>(units, local) : tc_smem_bytes<false>(units, local);
}

int ffn_tc_threads(bool f8) { return f8 ? TcGeo<true>::kThreads : TcGeo<false>::kThreads; }

bool ffn_tc_local_route_fits(const FfnArgs& a) {
    const bool f8 = a.dtype == MOE_DTYPE_FP8_E4M3;
    int units = 0;
    for (int c = 0; c < a.ncls; ++c) units += class_capacity(a.cls[c], a.n, a.g);
    const int m = a.g > 1 ? a.n / a.g : 0;
    // one thread per unit: the experts, then the departments from the next
    // warp on; the top-k's lane-held candidates: n <= 256
    return a.n <= 256 && ((a.n + 31) / 32) * 32 + m <= ffn_tc_threads(f8) &&
           ffn_tc_smem_bytes(units, &a, f8) <= 227 * 1024;
}

cudaError_t launch_ffn_tc(const TcArgs& a, cudaStream_t s) {
    // a matrix-form pass needs its buffers; anything else is the FFN step
    if (a.pmode != 0 && (a.pmode != kTcFormPUp && a.pmode != kTcFormPDown)) return cudaErrorInvalidValue;
    if (a.pmode != 0 && (!a.gbuf || !a.ubuf || !a.zbuf || !a.topk_idx || a.f.ncls != 1)) return cudaErrorInvalidValue;
    // FP8 weights: E4M3 codes with row scales, the FFN step only
    const bool f8 = a.f.dtype == MOE_DTYPE_FP8_E4M3;
    if (f8 && a.pmode != 0) return cudaErrorInvalidValue;
    if (f8) {
        for (int c = 0; c < a.f.ncls; ++c)
            if (!a.f.cls[c].sc_gate || !a.f.cls[c].sc_up || !a.f.cls[c].sc_down) return cudaErrorInvalidValue;
    } else if (a.f.dtype != MOE_DTYPE_BF16) {
        return cudaErrorInvalidValue;
    }
    int units = 0;
    for (int c = 0; c < a.f.ncls; ++c) units += class_capacity(a.f.cls[c], a.f.n, a.f.g);
    const size_t smem = ffn_tc_smem_bytes(units, a.f.local_route ? &a.f : nullptr, f8);
    auto kern = a.f.local_route ? (f8 ? ffn_tc_kernel<true, true> : ffn_tc_kernel<true, false>)
                                : (f8 ? ffn_tc_kernel<false, true> : ffn_tc_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)device_sm_count();
    TcArgs args = a;
    args.f.grid_magic = grid_magic_of(grid);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3((unsigned)ffn_tc_threads(f8), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

}  // namespace moe
