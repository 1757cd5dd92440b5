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
    int split_x;             // also write the bf16 hi/lo activations (ws.xb)
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
};

// Capacity of a class's unit table (records the dispatch may have written).
__host__ __device__ __forceinline__ int class_capacity(const UnitClass& c, int n, int g) {
    return c.kind == kUnitShared ? 1 : c.kind == kUnitDept ? n / g : n;
}

// Tensor-core FFN: the FFN arguments plus one TMA descriptor per class and
// matrix (gate, up, down) over the [units * rows, d] bf16 weight tensor.
struct TcArgs {
    FfnArgs f;
    CUtensorMap maps[3][3];
    int min_tokens;       // units with at least this many tokens
};

// Units with at least this many tokens run on the tensor cores (library
// default: none; the caller opts in with moe_set_tc_min_tokens).
constexpr int kTcMinTokens = 1 << 30;
// Rows of one tensor-core weight tile / TMA box (unit rows must be a multiple),
// and the hidden-size granularity of its down-projection stages.
constexpr int kTcBoxRows = 128;
constexpr int kTcHiddenQuantum = 128;

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
cudaError_t launch_ffn(const FfnArgs& a, cudaStream_t s);
cudaError_t launch_ffn_tc(const TcArgs& a, cudaStream_t s);
size_t ffn_tc_smem_bytes(int units);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);
cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t s);
cudaError_t launch_split_x(const float* x, long long elems, __nv_bfloat16* xb, cudaStream_t s);

int device_sm_count();

}  // namespace moe
