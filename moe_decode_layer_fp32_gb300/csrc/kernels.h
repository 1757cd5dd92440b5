// Host-side launchers of the decode-layer kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

constexpr int kMaxT = 128;       // tokens per step
constexpr int kMaxN = 1024;      // routed experts
constexpr int kMaxK = 32;        // experts per token

struct RouteArgs {
    const float* x;
    const float* w_router;
    const float* bias;       // may be null
    int T, d, n, k;
    float scale;
    int32_t* topk_idx;
    float* topk_w;
    WsPtrs ws;
    // Fused dispatch (whole-layer path): build the lists in the last block.
    int fuse_dispatch;
    int g;                   // experts per department
    float* y_zero;           // zeroed by the route grid when non-null
    long long y_elems;
    int split_x;             // also write the activations into ws.xb: 1 bf16 hi/lo,
                             // 2 E4M3 terms (split_e4m3_terms_warp)
    // Whole-layer path with routing in the FFN kernel: write the logits only
    // (no top-k, no dispatch); the FFN CTAs take it from there.
    int logits_only;
    // Group-limited top-k: k_dept > 0 keeps at most k_dept departments of
    // route_g experts per token (strict != 0: exactly k_dept); 0 = plain top-k.
    int route_g, k_dept, strict;
};

struct DispatchArgs {
    const int32_t* topk_idx;
    const float* topk_w;
    int T, n, k, g;
    WsPtrs ws;
};

// One class of FFN units: the shared expert, the department backbones or the
// per-expert blocks (vanilla experts / DeaMoE private columns).
enum UnitKind { kUnitShared = 0, kUnitDept = 1, kUnitExpert = 2 };
struct UnitClass {
    const void* w_gate;
    const void* w_up;
    const void* w_down;
    int rows;       // intermediate rows of one unit
    int kind;       // UnitKind
    // FP8 weights: one fp32 scale per row, [units * rows] per matrix (null
    // for bf16 / fp32 weights)
    const float* sc_gate;
    const float* sc_up;
    const float* sc_down;
};

struct FfnArgs {
    const float* x;
    int T, d, n, k, g;
    int dtype;            // MOE_DTYPE_*
    UnitClass cls[3];
    int ncls;
    WsPtrs ws;
    float* out;
    int out_mode;         // MOE_OUT_ROWS / MOE_OUT_ACCUM
    int rows_dept_base;   // ROWS mode: first department row
    int rows_shared_base; // ROWS mode: first shared-expert row
    int pdl;              // launch as a programmatic dependent
    int max_tokens;       // CUDA-core kernel: units with more tokens are skipped
    int auto_tc;          // both kernels launched; they pick one by prefer_tc()
    // auto_tc with the tensor-core kernel launched first: it records its
    // choice in ws.sync[1] (1 CUDA cores, 2 tensor cores) and the CUDA-core
    // kernel, its programmatic dependent, follows it.
    int tc_first;
    int sms;              // SMs of the device (grid of the tensor-core kernel)
    unsigned long long grid_magic;   // set by the launcher: ceil(2^64 / grid)
    // Routing inside the CUDA-core kernel (whole-layer path, ACCUM mode, no
    // tensor-core kernel): every CTA takes the top-k of ws.logits and builds
    // its own unit records in shared memory; CTA 0 also stores the routing
    // and the dispatch lists in the workspace.
    int local_route;
    const float* bias;    // selection bias or null
    float scale;
    int32_t* topk_idx;    // [T, k] routing outputs (written by CTA 0)
    float* topk_w;
    // Timeout test (moe_test_stall_weight_copies): the weight producers issue
    // no copy, and the consumers' waits give up after wait_ns (the drains
    // keep the normal limit).  0 in every other call.
    int stall_copies;
    unsigned long long wait_ns;
};

// Limit of a consumer wait in an FFN kernel.
__host__ __device__ __forceinline__ unsigned long long ffn_wait_limit(const FfnArgs& a) {
    return a.wait_ns ? a.wait_ns : kWaitLimitNs;
}

// ceil(2^64 / g) for g >= 2 (2^64 / g when g divides it); grid_share() divides
// by g with it.
inline unsigned long long grid_magic_of(unsigned g) {
    return g <= 1 ? 0ull : ~0ull / g + 1ull;
}
// floor(x * b / g) for x * b < 2^40 and g = gridDim.x, without a 64-bit
// division (a long software routine on the GPU).  Exact: the product with
// the rounded-up reciprocal errs by less than x * b / 2^64, below the 1/g
// gap between a non-integer quotient and the next integer.
__device__ __forceinline__ long long grid_share(long long x, unsigned b, unsigned g,
                                                unsigned long long magic) {
    if (g <= 1) return b ? x : 0;
    return (long long)__umul64hi((unsigned long long)x * b, magic);
}

// Capacity of a class's unit table (records the dispatch may have written).
__host__ __device__ __forceinline__ int class_capacity(const UnitClass& c, int n, int g) {
    return c.kind == kUnitShared ? 1 : c.kind == kUnitDept ? n / g : n;
}

// Tensor-core FFN: the FFN arguments plus one TMA descriptor per class and
// matrix (gate, up, down) over the [units * rows, d] weight tensor (bf16, or
// E4M3 codes whose row scales the FfnArgs classes carry).
struct TcArgs {
    FfnArgs f;
    CUtensorMap maps[3][3];
    int min_tokens;       // units with at least this many tokens
    // Matrix-form department passes of "DeaMoE" §3.1 eq. (4) on one class of
    // department units (rows = r): 0 = the SwiGLU FFN step; kTcFormPUp =
    // G = SiLU(W_g x) and U = SiLU(W_u x) of each department entry into gbuf
    // / ubuf (no down rows; also clears zbuf, and y with zero_y);
    // kTcFormPDown = H = sum_i p_i SiLU(Z_i) of each department entry from
    // the assignment rows of zbuf, then W_d^T H into y (no gate / up rows).
    int pmode;
    float* gbuf;          // [T * min(k, m), r] per department entry
    float* ubuf;
    float* zbuf;          // [T * k, r] per assignment: A_d^T Y (before SiLU)
    const int32_t* topk_idx;
    int zero_y;
};
constexpr int kTcFormPUp = 1;
constexpr int kTcFormPDown = 2;

// Rows of one tensor-core weight tile / TMA box (unit rows must be a multiple),
// the hidden-size granularity of its stages, and its tokens per group.
constexpr int kTcBoxRows = 128;
constexpr int kTcHiddenQuantum = 128;
constexpr int kTcGroupTokens = 32;

// Per-call choice between the two FFN kernels, made on the device from the
// dispatch's unit records so that no host round trip is needed.  Both kernels
// evaluate it on the same data and so agree.  Cost in weight rows streamed by
// the busiest SM: the CUDA-core stream re-reads a unit's rows once per group
// of kGroupTokens tokens and spreads rows evenly over the SMs; the tensor-core
// kernel reads them once per kTcGroupTokens tokens but in whole 128-row tiles,
// one SM per tile.  At d <= kTcWideHidden both stream at about the same rate
// per SM, so the busiest SM's row count decides; on wider rows the CUDA-core
// stream is measured about 4/3 slower per row and is weighted so.
constexpr int kTcWideHidden = 4096;
__device__ __forceinline__ bool prefer_tc(const FfnArgs& a) {
    long long rows_cc = 0, tiles = 0;
    for (int c = 0; c < a.ncls; ++c) {
        const UnitClass& uc = a.cls[c];
        int g_cc, g_tc;
        if (uc.kind == kUnitShared) {
            g_cc = (a.T + kGroupTokens - 1) / kGroupTokens;
            g_tc = (a.T + kTcGroupTokens - 1) / kTcGroupTokens;
        } else {
            const bool dept = uc.kind == kUnitDept;
            const int A = a.ws.counts[dept ? 1 : 0];
            g_cc = A > 0 ? (dept ? a.ws.dept_units : a.ws.exp_units)[A - 1].w : 0;
            g_tc = a.ws.counts[dept ? 3 : 2];
        }
        rows_cc += (long long)uc.rows * g_cc;
        tiles += (long long)(uc.rows / kTcBoxRows) * g_tc;
    }
    const long long S = a.sms;
    const long long tc_rows = (long long)((unsigned)(tiles + S - 1) / (unsigned)S) * kTcBoxRows;
    const long long cc_weight = a.d > kTcWideHidden ? 4 : 3;
    return tiles > 0 && tc_rows * S * 3 < rows_cc * cc_weight;
}

// DeaMoE form P ([DeaMoE] §3.1 eq. (4)): three passes over one layer.
enum FormPStage { kFormPUp = 0, kFormPPriv = 1, kFormPDown = 2 };
struct FormPArgs {
    const float* x;          // [T, d]
    int T, d, n, k, g, m;    // m = n / g departments
    int mk;                  // min(k, m): department entries per token at most
    int r;                   // department / expert width (hffn)
    const void* dgate;       // [m, r, d] bf16
    const void* dup;
    const void* ddown;
    const void* agate;       // [n, r, r] bf16
    const void* aup;
    const void* adown;
    const int32_t* topk_idx; // [T, k] routing of the step
    float* gbuf;             // [T*mk, r] SiLU(W_g x) per department entry
    float* ubuf;             // [T*mk, r] SiLU(W_u x)
    float* zbuf;             // [T*k, r] A_d^T Y per assignment (before SiLU)
    float* y;                // [T, d], zeroed by the routing kernel or, with
    int zero_y;              //   zero_y, by the up pass
    WsPtrs ws;
};
cudaError_t launch_formp(const FormPArgs& a, int sms, cudaStream_t s);
// One of the three passes (FormPStage) on the CUDA cores.
cudaError_t launch_formp_pass(const FormPArgs& a, int stage, int sms, cudaStream_t s);
int formp_max_hidden();   // widest h the up / down passes take
int formp_max_width();    // widest r the private pass takes

struct CombineArgs {
    const float* rows;
    int T, d, k, m;        // m = departments (0 for vanilla)
    int has_shared;
    int rows_dept_base, rows_shared_base;
    WsPtrs ws;
    float* y;
};

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);
cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s);
// Router-bias update and imbalance ratio over n <= 1024 expert counts.
cudaError_t launch_bias_update(const int32_t* counts, int n, float gamma, int rule, float* bias,
                               float* imbalance, cudaStream_t s);
cudaError_t launch_ffn(const FfnArgs& a, cudaStream_t s);
// Whether the CUDA-core kernel's shared memory still holds the routing state
// of the local path (a.local_route) at its usual CTAs per SM.
bool ffn_local_route_fits(const FfnArgs& a);
cudaError_t launch_ffn_tc(const TcArgs& a, cudaStream_t s);
// Dynamic shared memory of the tensor-core kernel (f8: the E4M3 variant) and
// its block size.
size_t ffn_tc_smem_bytes(int units, const FfnArgs* local, bool f8);
int ffn_tc_threads(bool f8);
// Whether the tensor-core kernel can route inside its CTAs (a.local_route).
bool ffn_tc_local_route_fits(const FfnArgs& a);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);
cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t s);
cudaError_t launch_split_x(const float* x, long long elems, __nv_bfloat16* xb, cudaStream_t s);
// x [T, d] -> the E4M3 activation terms and exponents in the xb region.
cudaError_t launch_split_terms(const float* x, int T, int d, __nv_bfloat16* xb, cudaStream_t s);

int device_sm_count();

}  // namespace moe
