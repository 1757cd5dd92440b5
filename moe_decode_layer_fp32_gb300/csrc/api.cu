// C ABI of the decode layer: host-side argument checks, workspace layout and
// kernel launches.  See include/moe_decode.h for the contract of each call.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/moe_decode.h"
#include "kernels.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* where) {
    return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

// Widest hidden size the streaming FFN covers: 15 consumer warps x 2 chunks x 8 columns.
constexpr int kMaxHidden = 15 * 32 * 2 * 8;
// Widest hidden size the router kernel covers: 128 threads x 16 float4 chunks.
constexpr int kMaxRouterHidden = 128 * 16 * 4;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
// Workspace counters of the routing kernel and the FFN kernels: [0] token
// blocks done (split top-k), [1] FFN path choice, [2 + b] blocks done on
// token block b (every block counts on [2] when the top-k is not split).
constexpr int kSyncWords = 2 + moe::kMaxT / 8;
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool layout_of(int T, int n, int k, int g, moe_ws_layout* L) {
    if (T < 1 || T > moe::kMaxT || n < 1 || n > moe::kMaxN || k < 1 || k > n ||
        k > moe::kMaxK || g < 1 || n % g != 0)
        return false;
    const int m = g > 1 ? n / g : 0;
    const int dk = g > 1 ? T * (k < m ? k : m) : 0;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    // The words that persist between calls (status, counts, the counters) sit
    // at fixed offsets, whatever the step's sizes, so that one workspace serves
    // steps of any T up to the one it was sized for, and a routing call (laid
    // out for g = 1) on a department workspace finds the same counters.  The
    // arrays every layout has come next; the department arrays come last.
    L->status = take(4 * sizeof(int32_t));                 // offset 0
    L->counts = take(4 * sizeof(int32_t));                 // offset 256
    L->sync = take(kSyncWords * sizeof(uint32_t));         // offset 512
    L->logits = take((size_t)T * n * sizeof(float));
    L->exp_count = take((size_t)n * sizeof(int32_t));
    L->exp_off = take((size_t)(n + 1) * sizeof(int32_t));
    L->asg_tok = take((size_t)T * k * sizeof(int32_t));
    L->asg_slot = take((size_t)T * k * sizeof(int32_t));
    L->asg_w = take((size_t)T * k * sizeof(float));
    L->tok_asg = take((size_t)T * k * sizeof(int32_t));
    L->act_exp = take((size_t)n * sizeof(int32_t));
    L->exp_units = take((size_t)n * 4 * sizeof(int32_t));
    // bf16 hi / lo rows, or the E4M3 activation terms and their exponents
    L->xb = take(moe::xq_exp_offset(T) + (size_t)T * sizeof(int32_t));
    L->dept_count = take((size_t)m * sizeof(int32_t));
    L->dept_off = take((size_t)(m + 1) * sizeof(int32_t));
    L->dept_tok = take((size_t)dk * sizeof(int32_t));
    L->dept_w = take((size_t)dk * sizeof(float));
    L->tok_dpos = take((size_t)T * m * sizeof(int32_t));
    L->act_dept = take((size_t)m * sizeof(int32_t));
    L->dept_units = take((size_t)m * 4 * sizeof(int32_t));
    L->total = off;
    return true;
}

moe::WsPtrs resolve(const void* ws, const moe_ws_layout& L) {
    char* b = static_cast<char*>(const_cast<void*>(ws));
    moe::WsPtrs p;
    p.status = reinterpret_cast<int32_t*>(b + L.status);
    p.counts = reinterpret_cast<int32_t*>(b + L.counts);
    p.logits = reinterpret_cast<float*>(b + L.logits);
    p.exp_count = reinterpret_cast<int32_t*>(b + L.exp_count);
    p.exp_off = reinterpret_cast<int32_t*>(b + L.exp_off);
    p.asg_tok = reinterpret_cast<int32_t*>(b + L.asg_tok);
    p.asg_slot = reinterpret_cast<int32_t*>(b + L.asg_slot);
    p.asg_w = reinterpret_cast<float*>(b + L.asg_w);
    p.tok_asg = reinterpret_cast<int32_t*>(b + L.tok_asg);
    p.act_exp = reinterpret_cast<int32_t*>(b + L.act_exp);
    p.dept_count = reinterpret_cast<int32_t*>(b + L.dept_count);
    p.dept_off = reinterpret_cast<int32_t*>(b + L.dept_off);
    p.dept_tok = reinterpret_cast<int32_t*>(b + L.dept_tok);
    p.dept_w = reinterpret_cast<float*>(b + L.dept_w);
    p.tok_dpos = reinterpret_cast<int32_t*>(b + L.tok_dpos);
    p.act_dept = reinterpret_cast<int32_t*>(b + L.act_dept);
    p.exp_units = reinterpret_cast<int4*>(b + L.exp_units);
    p.dept_units = reinterpret_cast<int4*>(b + L.dept_units);
    p.sync = reinterpret_cast<uint32_t*>(b + L.sync);
    p.xb = reinterpret_cast<__nv_bfloat16*>(b + L.xb);
    return p;
}

// Workspace check shared by every step.
int check_ws(const void* ws, size_t ws_bytes, int T, int n, int k, int g, moe_ws_layout* L,
             const char* who) {
    if (!layout_of(T, n, k, g, L))
        return fail(MOE_ERR_INVALID_ARG,
                    "%s: need 1<=T<=%d, 1<=n<=%d, 1<=k<=min(n,%d), g>=1, n%%g==0 "
                    "(T=%d n=%d k=%d g=%d)",
                    who, moe::kMaxT, moe::kMaxN, moe::kMaxK, T, n, k, g);
    if (!ws || !aligned16(ws)) return fail(MOE_ERR_INVALID_ARG, "%s: workspace null or unaligned", who);
    if (ws_bytes < L->total)
        return fail(MOE_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu required", who, ws_bytes,
                    L->total);
    return MOE_OK;
}

int weight_bytes(int dtype) {
    return dtype == MOE_DTYPE_BF16 ? 2 : dtype == MOE_DTYPE_F32 ? 4 : dtype == MOE_DTYPE_FP8_E4M3 ? 1 : 0;
}
// Bytes of one intermediate row of a unit (gate, up and down rows), FP8 row
// scales included.
long long unit_row_bytes(int d, int dtype) {
    return 3LL * d * weight_bytes(dtype) + (dtype == MOE_DTYPE_FP8_E4M3 ? 3 * 4 : 0);
}

int check_hidden(const float* x, int d, const char* who) {
    if (!x || !aligned16(x)) return fail(MOE_ERR_INVALID_ARG, "%s: x null or unaligned", who);
    if (d < 8 || d % 8 != 0) return fail(MOE_ERR_INVALID_ARG, "%s: d=%d must be a positive multiple of 8", who, d);
    return MOE_OK;
}

int check_unit(const void* g, const void* u, const void* dn, int rows, int d, int dtype,
               const char* what, const char* who) {
    if (rows <= 0 || rows % 16 != 0)
        return fail(MOE_ERR_INVALID_ARG, "%s: %s rows=%d must be a positive multiple of 16", who, what, rows);
    if (!g || !u || !dn || !aligned16(g) || !aligned16(u) || !aligned16(dn))
        return fail(MOE_ERR_INVALID_ARG, "%s: %s weights null or unaligned", who, what);
    if ((long long)d * weight_bytes(dtype) > 16384 || d > kMaxHidden)
        return fail(MOE_ERR_UNSUPPORTED, "%s: d=%d exceeds the streaming kernel's %d (one row <= 16 KB)",
                    who, d, kMaxHidden);
    return MOE_OK;
}

int check_ffn_common(const float* x, int d, int dtype, int out_mode, const float* out,
                     const char* who) {
    int rc = check_hidden(x, d, who);
    if (rc) return rc;
    if (weight_bytes(dtype) == 0) return fail(MOE_ERR_UNSUPPORTED, "%s: dtype %d", who, dtype);
    if (out_mode != MOE_OUT_ROWS && out_mode != MOE_OUT_ACCUM)
        return fail(MOE_ERR_INVALID_ARG, "%s: out_mode %d", who, out_mode);
    if (!out || !aligned16(out)) return fail(MOE_ERR_INVALID_ARG, "%s: out null or unaligned", who);
    return MOE_OK;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

long long rows_count(int T, int n, int k, int g, int has_shared) {
    const int m = g > 1 ? n / g : 0;
    const long long dk = g > 1 ? (long long)T * (k < m ? k : m) : 0;
    return (long long)T * k + dk + (has_shared ? T : 0);
}

// Minimum gathered tokens for a unit to run on the tensor cores (0 = default).
std::atomic<int> g_tc_min_tokens{0};
// Timeout test (moe_test_stall_weight_copies): 0 = off, else the consumer
// wait limit in ns of the FFN steps launched while it is set.
std::atomic<long long> g_stall_wait_ns{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// TMA descriptor of one [units * rows, d] bf16 weight tensor viewed as 3-D
// {64 columns, rows, d / 64 column chunks}; boxes of 64 x kTcBoxRows x 2
// (256 contiguous bytes of each row per op), 128 B swizzle.
bool encode_weight_map(CUtensorMap* map, const void* base, int units, int rows, int d) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {64, (cuuint64_t)units * rows, (cuuint64_t)(d / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)moe::kTcBoxRows, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// TMA descriptor of one [units * rows, d] E4M3 weight tensor (one byte per
// code): boxes of 128 columns x kTcBoxRows rows (16 KB) with the 128 B
// swizzle; the kernel's converter warps lay the values out for the MMA.
bool encode_weight_map_f8(CUtensorMap* map, const void* base, int units, int rows, int d) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)units * rows};
    const cuuint64_t strides[1] = {(cuuint64_t)d};
    const cuuint32_t box[2] = {128, (cuuint32_t)moe::kTcBoxRows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 0 (default): automatic per-call choice on the device; > 0: fixed threshold.
int tc_min_tokens() { return g_tc_min_tokens.load(); }

// Whether the tensor-core kernel takes part in this FFN step, and its TMA
// descriptors: bf16 or E4M3 weights, d a multiple of 128, and a batch large enough for
// some unit to reach the token threshold.
// Expected tokens per active unit of the busiest class under uniform routing:
// T*k/n per expert, T*P(department chosen) per department, T for the shared
// expert.  P(department of g experts chosen) = 1 - C(n-g, k) / C(n, k).
double expected_unit_tokens(const moe::FfnArgs& a, int T) {
    double best = 0.0;
    for (int c = 0; c < a.ncls; ++c) {
        const moe::UnitClass& uc = a.cls[c];
        double e = T;
        if (uc.kind == moe::kUnitExpert) {
            e = (double)T * a.k / a.n;
        } else if (uc.kind == moe::kUnitDept) {
            double miss = 1.0;
            for (int i = 0; i < a.k; ++i)
                miss *= a.n - a.g - i > 0 ? (double)(a.n - a.g - i) / (a.n - i) : 0.0;
            e = T * (1.0 - miss);
        }
        best = e > best ? e : best;
    }
    return best;
}

bool prepare_tc(const moe::FfnArgs& a, int T, moe::TcArgs* t) {
    const int thr = tc_min_tokens();
    // Automatic mode launches the tensor-core kernel for wide rows always
    // (both kernels run and choose on the device), and otherwise only when
    // some class expects more than one CUDA-core group of tokens per unit:
    // then the CUDA-core stream would read those rows once per group, and the
    // tensor-core kernel runs alone with the routing inside its CTAs
    // (DeaMoE-7B layer at T = 8: 43.5 vs 50.1 µs on the CUDA cores).
    if (thr == 0 && a.d <= moe::kTcWideHidden &&
        (T <= moe::kGroupTokens || expected_unit_tokens(a, T) <= moe::kGroupTokens))
        return false;
    const int mt = thr > 0 ? thr : 1;
    int units = 0;
    for (int c = 0; c < a.ncls; ++c) units += moe::class_capacity(a.cls[c], a.n, a.g);
    const bool f8 = a.dtype == MOE_DTYPE_FP8_E4M3;
    if ((a.dtype != MOE_DTYPE_BF16 && !f8) || a.d % moe::kTcHiddenQuantum != 0 || a.d > moe::kMaxXbHidden ||
        T < mt || moe::ffn_tc_smem_bytes(units, nullptr, f8) > 227 * 1024)
        return false;
    for (int c = 0; c < a.ncls; ++c)
        if (a.cls[c].rows % moe::kTcBoxRows != 0) return false;
    *t = moe::TcArgs{};   // the form-C FFN step: no matrix-form pass mode or buffers
    t->f = a;
    t->min_tokens = thr > 0 ? thr : 1;
    for (int c = 0; c < a.ncls; ++c) {
        const moe::UnitClass& uc = a.cls[c];
        const int nu = moe::class_capacity(uc, a.n, a.g);
        auto enc = f8 ? encode_weight_map_f8 : encode_weight_map;
        if (!enc(&t->maps[c][0], uc.w_gate, nu, uc.rows, a.d) || !enc(&t->maps[c][1], uc.w_up, nu, uc.rows, a.d) ||
            !enc(&t->maps[c][2], uc.w_down, nu, uc.rows, a.d))
            return false;
    }
    return true;
}

// FFN step: the CUDA-core stream for units with few tokens and, when `tc`, the
// tensor-core kernel for the others.  x_split: ws.xb already holds the split
// activations (the whole-layer path writes it in the routing kernel).
int run_ffn(moe::FfnArgs& a, int T, int n, int k, int g, int has_shared, bool tc,
            moe::TcArgs& t, bool x_split, void* stream, const char* who) {
    a.rows_dept_base = T * k;
    a.rows_shared_base = (int)rows_count(T, n, k, g, 0);
    cudaError_t e;
    if (a.out_mode == MOE_OUT_ROWS) {
        const size_t bytes = (size_t)rows_count(T, n, k, g, has_shared) * a.d * sizeof(float);
        e = moe::launch_zero(a.out, bytes, as_stream(stream));
        if (e != cudaSuccess) return cuda_fail(e, who);
    }
    if (tc && !x_split) {
        e = a.dtype == MOE_DTYPE_FP8_E4M3 ? moe::launch_split_terms(a.x, T, a.d, a.ws.xb, as_stream(stream))
                                           : moe::launch_split_x(a.x, (long long)T * a.d, a.ws.xb, as_stream(stream));
        if (e != cudaSuccess) return cuda_fail(e, who);
    }
    a.auto_tc = tc && tc_min_tokens() == 0;
    a.sms = moe::device_sm_count();
    a.max_tokens = tc && !a.auto_tc ? t.min_tokens - 1 : INT_MAX;
    // Automatic choice: the tensor-core kernel goes first (the host launches
    // it only when it is expected to win) and records the choice; the
    // CUDA-core kernel follows it and returns at once when it lost.
    a.tc_first = a.auto_tc ? 1 : 0;
    if (a.tc_first) {
        t.f = a;
        e = moe::launch_ffn_tc(t, as_stream(stream));
        if (e != cudaSuccess) return cuda_fail(e, who);
    }
    e = moe::launch_ffn(a, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, who);
    if (tc && !a.tc_first) {
        t.f = a;
        e = moe::launch_ffn_tc(t, as_stream(stream));
        if (e != cudaSuccess) return cuda_fail(e, who);
    }
    return MOE_OK;
}

}  // namespace

namespace moe {
int device_sm_count() {
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int sms = 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (dev >= 0 && dev < 64) cache[dev] = sms;
    return sms;
}
}  // namespace moe

// ---- fixed router scratch for moe_route_topk_noalloc ----------------------
// Some callers cannot hand the library a workspace or let it allocate one:
// an engine whose device memory is carved up once at start-up, or a caller
// that must not stall the device (cudaFree synchronises) or fail for lack of
// memory in the middle of a decode step.  For them the router step can run on
// this array, which the loader reserves with the module.  Its size bounds the
// step to T * n <= kNoAllocMaxLogits.
constexpr int kNoAllocMaxLogits = 64 * 1024;          // T * n router logits (256 KB)
constexpr size_t kNoAllocHeader = 256;                // [0] status word, [128] block counters
static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocHeader +
                                                               (size_t)kNoAllocMaxLogits * sizeof(float)];

namespace {
constexpr int kScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kScratchDevices] = {};

// This device's address of g_route_scratch, looked up on the first call made
// on the device and remembered after that.
int route_scratch(void** out, const char* who) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, who);
    if (dev < 0 || dev >= kScratchDevices)
        return fail(MOE_ERR_UNSUPPORTED, "%s: device %d is beyond the %d the scratch table tracks", who,
                    dev, kScratchDevices);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return cuda_fail(e, who);
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}
}  // namespace

extern "C" {

int moe_version(void) { return 100; }

int64_t moe_test_stall_weight_copies(int64_t wait_ns) {
    if (wait_ns < 0) return fail(MOE_ERR_INVALID_ARG, "moe_test_stall_weight_copies: negative limit");
    return g_stall_wait_ns.exchange(wait_ns);
}

int moe_set_tc_min_tokens(int min_tokens) {
    if (min_tokens < 0) return fail(MOE_ERR_INVALID_ARG, "moe_set_tc_min_tokens: negative");
    return g_tc_min_tokens.exchange(min_tokens);
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

size_t moe_workspace_bytes(int T, int n, int k, int experts_per_dept) {
    moe_ws_layout L;
    return layout_of(T, n, k, experts_per_dept, &L) ? L.total : 0;
}

int moe_workspace_layout(int T, int n, int k, int experts_per_dept, moe_ws_layout* out) {
    if (!out) return fail(MOE_ERR_INVALID_ARG, "moe_workspace_layout: out is null");
    if (!layout_of(T, n, k, experts_per_dept, out))
        return fail(MOE_ERR_INVALID_ARG, "moe_workspace_layout: invalid sizes");
    return MOE_OK;
}

int moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!ws || !aligned16(ws)) return fail(MOE_ERR_INVALID_ARG, "moe_workspace_init: ws null or unaligned");
    cudaError_t e = moe::launch_zero(ws, ws_bytes & ~size_t(15), as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "moe_workspace_init");
    return MOE_OK;
}

int moe_read_status(const void* ws, size_t ws_bytes, int32_t* host_status, int32_t* host_counts,
                    void* stream) {
    if (!ws || ws_bytes < 512) return fail(MOE_ERR_INVALID_ARG, "moe_read_status: bad workspace");
    int32_t buf[8];
    // status at offset 0, counts at offset 256 (see layout_of)
    cudaError_t e = cudaMemcpyAsync(buf, ws, 4 * sizeof(int32_t), cudaMemcpyDeviceToHost, as_stream(stream));
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(buf + 4, static_cast<const char*>(ws) + 256, 4 * sizeof(int32_t),
                            cudaMemcpyDeviceToHost, as_stream(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "moe_read_status");
    if (host_status) host_status[0] = buf[0];
    if (host_counts) {
        host_counts[0] = buf[4];
        host_counts[1] = buf[5];
    }
    return MOE_OK;
}

// Host <-> device activation copies of a step: one cudaMemcpyAsync each, on
// the step's stream, so that a caller holding host buffers goes through the
// library from input to output.
static int host_copy_checks(const void* dev, const void* host, int T, int d, const char* who) {
    if (!dev || !host) return fail(MOE_ERR_INVALID_ARG, "%s: null pointer", who);
    if (T < 1 || d < 1) return fail(MOE_ERR_INVALID_ARG, "%s: T=%d, d=%d must be >= 1", who, T, d);
    return MOE_OK;
}

int moe_input_from_host(float* x, const float* x_host, int T, int d, void* stream) {
    const char* who = "moe_input_from_host";
    int rc = host_copy_checks(x, x_host, T, d, who);
    if (rc) return rc;
    cudaError_t e = cudaMemcpyAsync(x, x_host, (size_t)T * d * sizeof(float), cudaMemcpyHostToDevice,
                                    as_stream(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, who);
}

int moe_output_to_host(float* y_host, const float* y, int T, int d, void* stream) {
    const char* who = "moe_output_to_host";
    int rc = host_copy_checks(y, y_host, T, d, who);
    if (rc) return rc;
    cudaError_t e = cudaMemcpyAsync(y_host, y, (size_t)T * d * sizeof(float), cudaMemcpyDeviceToHost,
                                    as_stream(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, who);
}

int moe_route_topk(const float* x, const float* w_router, const float* bias, int T, int d, int n,
                   int k, float scale, int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                   void* stream) {
    const char* who = "moe_route_topk";
    moe_ws_layout L;
    int rc = check_ws(ws, ws_bytes, T, n, k, 1, &L, who);
    if (rc) return rc;
    if ((rc = check_hidden(x, d, who))) return rc;
    if (d > kMaxRouterHidden)
        return fail(MOE_ERR_UNSUPPORTED, "%s: d=%d exceeds the router kernel's %d", who, d, kMaxRouterHidden);
    if (!w_router || !aligned16(w_router)) return fail(MOE_ERR_INVALID_ARG, "%s: w_router null or unaligned", who);
    if (!topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "%s: outputs are null", who);
    moe::RouteArgs a = {};
    a.x = x;
    a.w_router = w_router;
    a.bias = bias;
    a.T = T; a.d = d; a.n = n; a.k = k;
    a.scale = scale;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.ws = resolve(ws, L);
    a.fuse_dispatch = 0;
    a.g = 1;
    cudaError_t e = moe::launch_route(a, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, who);
    return MOE_OK;
}

int moe_route_topk_grouped(const float* x, const float* w_router, const float* bias, int T, int d, int n,
                           int k, int experts_per_dept, int k_dept, int strict, float scale,
                           int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, void* stream) {
    const char* who = "moe_route_topk_grouped";
    if (experts_per_dept < 1 || n < 1 || n % experts_per_dept)
        return fail(MOE_ERR_INVALID_ARG, "%s: experts_per_dept=%d must divide n=%d", who, experts_per_dept, n);
    const int m = n / experts_per_dept;
    if (k_dept < 1 || k_dept > m)
        return fail(MOE_ERR_INVALID_ARG, "%s: k_dept=%d outside [1, %d]", who, k_dept, m);
    if ((long long)k > (long long)k_dept * experts_per_dept)
        return fail(MOE_ERR_INVALID_ARG, "%s: k=%d exceeds the %d experts of k_dept=%d departments", who, k,
                    k_dept * experts_per_dept, k_dept);
    if (strict && k < k_dept)
        return fail(MOE_ERR_INVALID_ARG, "%s: strict coverage needs k >= k_dept (k=%d, k_dept=%d)", who, k,
                    k_dept);
    moe_ws_layout L;
    int rc = check_ws(ws, ws_bytes, T, n, k, 1, &L, who);
    if (rc) return rc;
    if ((rc = check_hidden(x, d, who))) return rc;
    if (d > kMaxRouterHidden)
        return fail(MOE_ERR_UNSUPPORTED, "%s: d=%d exceeds the router kernel's %d", who, d, kMaxRouterHidden);
    if (!w_router || !aligned16(w_router)) return fail(MOE_ERR_INVALID_ARG, "%s: w_router null or unaligned", who);
    if (!topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "%s: outputs are null", who);
    moe::RouteArgs a = {};
    a.x = x;
    a.w_router = w_router;
    a.bias = bias;
    a.T = T; a.d = d; a.n = n; a.k = k;
    a.scale = scale;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.ws = resolve(ws, L);
    a.fuse_dispatch = 0;
    a.g = 1;
    a.route_g = experts_per_dept;
    a.k_dept = k_dept;
    a.strict = strict ? 1 : 0;
    cudaError_t e = moe::launch_route(a, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, who);
    return MOE_OK;
}

int moe_bias_update(const int32_t* counts, int n, float gamma, int rule, float* bias, float* imbalance,
                    void* stream) {
    const char* who = "moe_bias_update";
    if (n < 1 || n > moe::kMaxN) return fail(MOE_ERR_INVALID_ARG, "%s: n=%d outside [1, %d]", who, n, moe::kMaxN);
    if (!counts) return fail(MOE_ERR_INVALID_ARG, "%s: counts is null", who);
    if (!bias && !imbalance) return fail(MOE_ERR_INVALID_ARG, "%s: bias and imbalance are both null", who);
    if (rule != MOE_BIAS_SIGN && rule != MOE_BIAS_PROPORTIONAL)
        return fail(MOE_ERR_INVALID_ARG, "%s: unknown rule %d", who, rule);
    if (!(gamma >= 0.0f) || gamma == INFINITY)
        return fail(MOE_ERR_INVALID_ARG, "%s: gamma must be finite and >= 0", who);
    cudaError_t e = moe::launch_bias_update(counts, n, gamma, rule, bias, imbalance, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, who);
    return MOE_OK;
}

int moe_route_topk_noalloc(const float* x, const float* w_router, const float* bias, int T, int d,
                           int n, int k, float scale, int32_t* topk_idx, float* topk_w,
                           int32_t* status, void* stream) {
    const char* who = "moe_route_topk_noalloc";
    if (T < 1 || T > moe::kMaxT || n < 1 || n > moe::kMaxN || k < 1 || k > n || k > moe::kMaxK)
        return fail(MOE_ERR_INVALID_ARG, "%s: invalid sizes T=%d n=%d k=%d", who, T, n, k);
    if ((long long)T * n > kNoAllocMaxLogits)
        return fail(MOE_ERR_UNSUPPORTED,
                    "%s: T*n = %lld router logits exceed the fixed scratch (%d); use moe_route_topk "
                    "with a workspace", who, (long long)T * n, kNoAllocMaxLogits);
    int rc = check_hidden(x, d, who);
    if (rc) return rc;
    if (d > kMaxRouterHidden)
        return fail(MOE_ERR_UNSUPPORTED, "%s: d=%d exceeds the router kernel's %d", who, d, kMaxRouterHidden);
    if (!w_router || !aligned16(w_router)) return fail(MOE_ERR_INVALID_ARG, "%s: w_router null or unaligned", who);
    if (!topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "%s: outputs are null", who);
    void* scratch = nullptr;
    if ((rc = route_scratch(&scratch, who))) return rc;
    char* b = static_cast<char*>(scratch);
    cudaStream_t s = as_stream(stream);
    // the status word and the last-block counter start every call at zero
    cudaError_t e = cudaMemsetAsync(b, 0, kNoAllocHeader, s);
    if (e != cudaSuccess) return cuda_fail(e, who);
    moe::RouteArgs a = {};
    a.x = x;
    a.w_router = w_router;
    a.bias = bias;
    a.T = T; a.d = d; a.n = n; a.k = k;
    a.scale = scale;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.ws.status = reinterpret_cast<int32_t*>(b);
    a.ws.sync = reinterpret_cast<uint32_t*>(b + 128);
    a.ws.logits = reinterpret_cast<float*>(b + kNoAllocHeader);
    a.fuse_dispatch = 0;
    a.g = 1;
    e = moe::launch_route(a, s);
    if (e != cudaSuccess) return cuda_fail(e, who);
    if (status) {
        e = cudaMemcpyAsync(status, b, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, who);
    }
    return MOE_OK;
}

int moe_dispatch(const int32_t* topk_idx, const float* topk_w, int T, int n, int k,
                 int experts_per_dept, void* ws, size_t ws_bytes, void* stream) {
    const char* who = "moe_dispatch";
    moe_ws_layout L;
    int rc = check_ws(ws, ws_bytes, T, n, k, experts_per_dept, &L, who);
    if (rc) return rc;
    if (!topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "%s: inputs are null", who);
    moe::DispatchArgs a = {topk_idx, topk_w, T, n, k, experts_per_dept, resolve(ws, L)};
    cudaError_t e = moe::launch_dispatch(a, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, who);
    return MOE_OK;
}

int64_t moe_rows_count(int T, int n, int k, int experts_per_dept, int has_shared) {
    moe_ws_layout L;
    if (!layout_of(T, n, k, experts_per_dept, &L)) return -1;
    return rows_count(T, n, k, experts_per_dept, has_shared);
}

// FP8 weights: the row scales of every class, in the order the *_fp8 calls
// take them (the main class -- experts or departments --, the private rows,
// then the shared expert); nsets is the number of triples.  Other dtypes
// take none.
static int attach_row_scales(moe::FfnArgs& a, const float* const* sc, int nsets, const char* who) {
    if (a.dtype != MOE_DTYPE_FP8_E4M3) {
        if (sc) return fail(MOE_ERR_INVALID_ARG, "%s: row scales are for FP8 weights only", who);
        return MOE_OK;
    }
    if (!sc) return fail(MOE_ERR_INVALID_ARG, "%s: FP8 weights need the *_fp8 call and its row scales", who);
    int next = 0;
    for (int c = 0; c < a.ncls; ++c) {
        moe::UnitClass& uc = a.cls[c];
        const int set = uc.kind == moe::kUnitShared ? nsets - 1 : next++;
        const float* g = sc[3 * set];
        const float* u = sc[3 * set + 1];
        const float* dn = sc[3 * set + 2];
        if (!g || !u || !dn || (reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(u) |
                                reinterpret_cast<uintptr_t>(dn)) & 3u)
            return fail(MOE_ERR_INVALID_ARG, "%s: row scales of set %d null or unaligned", who, set);
        uc.sc_gate = g;
        uc.sc_up = u;
        uc.sc_down = dn;
    }
    return MOE_OK;
}

static int setup_vanilla(moe::FfnArgs& a, const float* x, int T, int d, int n, int k, int I,
                         int dtype, const void* w_gate, const void* w_up, const void* w_down,
                         int I_s, const void* s_gate, const void* s_up, const void* s_down,
                         const void* ws, size_t ws_bytes, int out_mode, float* out,
                         const char* who) {
    moe_ws_layout L;
    int rc = check_ws(ws, ws_bytes, T, n, k, 1, &L, who);
    if (rc) return rc;
    if ((rc = check_ffn_common(x, d, dtype, out_mode, out, who))) return rc;
    if ((rc = check_unit(w_gate, w_up, w_down, I, d, dtype, "expert", who))) return rc;
    if (I_s < 0) return fail(MOE_ERR_INVALID_ARG, "%s: I_s < 0", who);
    if (I_s > 0 && (rc = check_unit(s_gate, s_up, s_down, I_s, d, dtype, "shared expert", who))) return rc;
    a = moe::FfnArgs{};
    a.x = x;
    a.T = T; a.d = d; a.n = n; a.k = k; a.g = 1;
    a.dtype = dtype;
    a.ncls = 0;
    if (I_s > 0) a.cls[a.ncls++] = moe::UnitClass{s_gate, s_up, s_down, I_s, moe::kUnitShared};
    a.cls[a.ncls++] = moe::UnitClass{w_gate, w_up, w_down, I, moe::kUnitExpert};
    a.ws = resolve(ws, L);
    a.out = out;
    a.out_mode = out_mode;
    a.pdl = 1;
    const long long stall = g_stall_wait_ns.load();
    a.stall_copies = stall > 0 ? 1 : 0;
    a.wait_ns = stall > 0 ? (unsigned long long)stall : 0ull;
    return MOE_OK;
}

static int ffn_vanilla_impl(const float* const* sc, const char* who, const float* x, int T, int d, int n, int k, int I, int dtype,
                    const void* w_gate, const void* w_up, const void* w_down, int I_s,
                    const void* s_gate, const void* s_up, const void* s_down, const void* ws,
                    size_t ws_bytes, int out_mode, float* out, void* stream) {
    moe::FfnArgs a;
    int rc = setup_vanilla(a, x, T, d, n, k, I, dtype, w_gate, w_up, w_down, I_s, s_gate, s_up,
                           s_down, ws, ws_bytes, out_mode, out, who);
    if (rc) return rc;
    if ((rc = attach_row_scales(a, sc, 2, who))) return rc;
    moe::TcArgs t = {};
    const bool tc = prepare_tc(a, T, &t);
    return run_ffn(a, T, n, k, 1, I_s > 0, tc, t, false, stream, who);
}

static int setup_deamoe(moe::FfnArgs& a, const float* x, int T, int d, int n, int k, int g,
                        int I_sh, int I_pr, int dtype, const void* dept_gate, const void* dept_up,
                        const void* dept_down, const void* priv_gate, const void* priv_up,
                        const void* priv_down, int I_s, const void* s_gate, const void* s_up,
                        const void* s_down, const void* ws, size_t ws_bytes, int out_mode,
                        float* out, const char* who) {
    moe_ws_layout L;
    int rc = check_ws(ws, ws_bytes, T, n, k, g, &L, who);
    if (rc) return rc;
    if ((rc = check_ffn_common(x, d, dtype, out_mode, out, who))) return rc;
    if ((rc = check_unit(dept_gate, dept_up, dept_down, I_sh, d, dtype, "department", who))) return rc;
    if (I_pr < 0 || I_s < 0) return fail(MOE_ERR_INVALID_ARG, "%s: negative size", who);
    if (I_pr > 0 && (rc = check_unit(priv_gate, priv_up, priv_down, I_pr, d, dtype, "private", who))) return rc;
    if (I_s > 0 && (rc = check_unit(s_gate, s_up, s_down, I_s, d, dtype, "shared expert", who))) return rc;
    a = moe::FfnArgs{};
    a.x = x;
    a.T = T; a.d = d; a.n = n; a.k = k; a.g = g;
    a.dtype = dtype;
    a.ncls = 0;
    if (I_s > 0) a.cls[a.ncls++] = moe::UnitClass{s_gate, s_up, s_down, I_s, moe::kUnitShared};
    // With one expert per department the department rows are the expert's own rows.
    a.cls[a.ncls++] = moe::UnitClass{dept_gate, dept_up, dept_down, I_sh,
                                     g > 1 ? moe::kUnitDept : moe::kUnitExpert};
    if (I_pr > 0) a.cls[a.ncls++] = moe::UnitClass{priv_gate, priv_up, priv_down, I_pr, moe::kUnitExpert};
    a.ws = resolve(ws, L);
    a.out = out;
    a.out_mode = out_mode;
    a.pdl = 1;
    const long long stall = g_stall_wait_ns.load();
    a.stall_copies = stall > 0 ? 1 : 0;
    a.wait_ns = stall > 0 ? (unsigned long long)stall : 0ull;
    return MOE_OK;
}

static int deamoe_ffn_impl(const float* const* sc, const char* who, const float* x, int T, int d, int n, int k, int experts_per_dept, int I_sh,
               int I_pr, int dtype, const void* dept_gate, const void* dept_up,
               const void* dept_down, const void* priv_gate, const void* priv_up,
               const void* priv_down, int I_s, const void* s_gate, const void* s_up,
               const void* s_down, const void* ws, size_t ws_bytes, int out_mode, float* out,
               void* stream) {
    moe::FfnArgs a;
    int rc = setup_deamoe(a, x, T, d, n, k, experts_per_dept, I_sh, I_pr, dtype, dept_gate, dept_up,
                          dept_down, priv_gate, priv_up, priv_down, I_s, s_gate, s_up, s_down, ws,
                          ws_bytes, out_mode, out, who);
    if (rc) return rc;
    if ((rc = attach_row_scales(a, sc, 3, who))) return rc;
    moe::TcArgs t = {};
    const bool tc = prepare_tc(a, T, &t);
    return run_ffn(a, T, n, k, experts_per_dept, I_s > 0, tc, t, false, stream, who);
}

int moe_combine(const float* rows, int T, int d, int n, int k, int experts_per_dept,
                int has_shared, const void* ws, size_t ws_bytes, float* y, void* stream) {
    const char* who = "moe_combine";
    moe_ws_layout L;
    int rc = check_ws(ws, ws_bytes, T, n, k, experts_per_dept, &L, who);
    if (rc) return rc;
    if (!rows || !aligned16(rows) || !y || !aligned16(y))
        return fail(MOE_ERR_INVALID_ARG, "%s: rows / y null or unaligned", who);
    if (d < 8 || d % 8) return fail(MOE_ERR_INVALID_ARG, "%s: d=%d must be a positive multiple of 8", who, d);
    moe::CombineArgs a = {};
    a.rows = rows;
    a.T = T; a.d = d; a.k = k;
    a.m = experts_per_dept > 1 ? n / experts_per_dept : 0;
    a.has_shared = has_shared ? 1 : 0;
    a.rows_dept_base = T * k;
    a.rows_shared_base = (int)(rows_count(T, n, k, experts_per_dept, 0));
    a.ws = resolve(ws, L);
    a.y = y;
    cudaError_t e = moe::launch_combine(a, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, who);
    return MOE_OK;
}

// How the whole-layer step runs its FFN:
//  - kLayerCudaLocal: the CUDA-core kernel alone, routing inside its CTAs;
//  - kLayerTcLocal: the tensor-core kernel alone, routing inside its CTAs
//    (automatic mode, rows up to kTcWideHidden wide, T <= 32, when the host
//    rule expects the tensor cores to win: at least two CUDA-core groups per
//    unit);
//  - kLayerGlobal: the routing kernel builds the dispatch, and the FFN kernels
//    read it (automatic choice on the device for wide rows, or a fixed
//    tensor-core threshold).
enum { kLayerCudaLocal = 0, kLayerTcLocal = 1, kLayerGlobal = 2 };

static int layer_path(const moe::FfnArgs& a, bool tc, const moe::TcArgs& t) {
    (void)t;
    if (!tc) return moe::ffn_local_route_fits(a) ? kLayerCudaLocal : kLayerGlobal;
    // beyond 32 tokens one CTA's top-k (a warp per token) takes more rounds
    // than the routing kernel's split top-k saves
    if (tc_min_tokens() == 0 && a.d <= moe::kTcWideHidden && a.T <= 32) {
        moe::FfnArgs b = a;
        b.local_route = 1;
        if (moe::ffn_tc_local_route_fits(b)) return kLayerTcLocal;
    }
    return kLayerGlobal;
}

// FFN step of the whole-layer path (after layer_route).
static int layer_ffn(moe::FfnArgs& a, int T, int n, int k, int g, int has_shared, bool tc, moe::TcArgs& t,
                     int path, void* stream, const char* who) {
    if (path != kLayerTcLocal) return run_ffn(a, T, n, k, g, has_shared, tc, t, true, stream, who);
    a.rows_dept_base = T * k;
    a.rows_shared_base = (int)rows_count(T, n, k, g, 0);
    a.auto_tc = 0;
    a.tc_first = 0;
    a.max_tokens = INT_MAX;
    a.sms = moe::device_sm_count();
    t.f = a;
    t.min_tokens = 1;
    cudaError_t e = moe::launch_ffn_tc(t, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, who);
    return MOE_OK;
}

// Routing step of the whole-layer path.  With `local` the routing kernel
// writes the logits only and the CUDA-core FFN kernel (a.local_route) takes
// the top-k and builds the dispatch in every CTA; otherwise the routing
// kernel's last block does both for the FFN kernels to read.
static int layer_route(const float* x, int T, int d, int n, int k, float scale, const float* w_router,
                       const float* bias, int g, const moe_ws_layout& L, void* ws, int32_t* topk_idx,
                       float* topk_w, float* y, bool split_x, bool local, moe::FfnArgs& a,
                       void* stream, const char* who) {
    if (!w_router || !aligned16(w_router)) return fail(MOE_ERR_INVALID_ARG, "%s: w_router null or unaligned", who);
    if (!topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "%s: routing outputs are null", who);
    moe::RouteArgs r = {};
    r.x = x;
    r.w_router = w_router;
    r.bias = bias;
    r.T = T; r.d = d; r.n = n; r.k = k;
    r.scale = scale;
    r.topk_idx = topk_idx;
    r.topk_w = topk_w;
    r.ws = resolve(ws, L);
    r.g = g;
    r.y_zero = y;
    r.y_elems = (long long)T * d;
    r.split_x = split_x ? (a.dtype == MOE_DTYPE_FP8_E4M3 ? 2 : 1) : 0;
    r.fuse_dispatch = local ? 0 : 1;
    r.logits_only = local ? 1 : 0;
    if (local) {
        a.local_route = 1;
        a.bias = bias;
        a.scale = scale;
        a.topk_idx = topk_idx;
        a.topk_w = topk_w;
    }
    cudaError_t e = moe::launch_route(r, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, who);
    return MOE_OK;
}

static int layer_forward_impl(const float* const* sc, const char* who, const float* x, int T, int d, int n, int k, float scale,
                      const float* w_router, const float* bias, int I, int dtype,
                      const void* w_gate, const void* w_up, const void* w_down, int I_s,
                      const void* s_gate, const void* s_up, const void* s_down, void* ws,
                      size_t ws_bytes, int32_t* topk_idx, float* topk_w, float* y, void* stream) {
    moe::FfnArgs a;
    int rc = setup_vanilla(a, x, T, d, n, k, I, dtype, w_gate, w_up, w_down, I_s, s_gate, s_up,
                           s_down, ws, ws_bytes, MOE_OUT_ACCUM, y, who);
    if (rc) return rc;
    if ((rc = attach_row_scales(a, sc, 2, who))) return rc;
    moe_ws_layout L;
    layout_of(T, n, k, 1, &L);
    moe::TcArgs t = {};
    const bool tc = prepare_tc(a, T, &t);
    const int path = layer_path(a, tc, t);
    if ((rc = layer_route(x, T, d, n, k, scale, w_router, bias, 1, L, ws, topk_idx, topk_w, y, tc,
                          path != kLayerGlobal, a, stream, who)))
        return rc;
    return layer_ffn(a, T, n, k, 1, I_s > 0, tc, t, path, stream, who);
}

static int deamoe_layer_forward_impl(const float* const* sc, const char* who, const float* x, int T, int d, int n, int k, float scale,
                         const float* w_router, const float* bias, int experts_per_dept, int I_sh,
                         int I_pr, int dtype, const void* dept_gate, const void* dept_up,
                         const void* dept_down, const void* priv_gate, const void* priv_up,
                         const void* priv_down, int I_s, const void* s_gate, const void* s_up,
                         const void* s_down, void* ws, size_t ws_bytes, int32_t* topk_idx,
                         float* topk_w, float* y, void* stream) {
    moe::FfnArgs a;
    int rc = setup_deamoe(a, x, T, d, n, k, experts_per_dept, I_sh, I_pr, dtype, dept_gate, dept_up,
                          dept_down, priv_gate, priv_up, priv_down, I_s, s_gate, s_up, s_down, ws,
                          ws_bytes, MOE_OUT_ACCUM, y, who);
    if (rc) return rc;
    if ((rc = attach_row_scales(a, sc, 3, who))) return rc;
    moe_ws_layout L;
    layout_of(T, n, k, experts_per_dept, &L);
    moe::TcArgs t = {};
    const bool tc = prepare_tc(a, T, &t);
    const int path = layer_path(a, tc, t);
    if ((rc = layer_route(x, T, d, n, k, scale, w_router, bias, experts_per_dept, L, ws, topk_idx,
                          topk_w, y, tc, path != kLayerGlobal, a, stream, who)))
        return rc;
    return layer_ffn(a, T, n, k, experts_per_dept, I_s > 0, tc, t, path, stream, who);
}

int moe_ffn_vanilla(const float* x, int T, int d, int n, int k, int I, int dtype,
                    const void* w_gate, const void* w_up, const void* w_down, int I_s,
                    const void* s_gate, const void* s_up, const void* s_down, const void* ws,
                    size_t ws_bytes, int out_mode, float* out, void* stream) {
    return ffn_vanilla_impl(nullptr, "moe_ffn_vanilla", x, T, d, n, k, I, dtype, w_gate, w_up, w_down, I_s,
                            s_gate, s_up, s_down, ws, ws_bytes, out_mode, out, stream);
}

int moe_ffn_vanilla_fp8(const float* x, int T, int d, int n, int k, int I, const void* w_gate,
                        const void* w_up, const void* w_down, int I_s, const void* s_gate,
                        const void* s_up, const void* s_down, const float* const row_scales[6],
                        const void* ws, size_t ws_bytes, int out_mode, float* out, void* stream) {
    const char* who = "moe_ffn_vanilla_fp8";
    if (!row_scales) return fail(MOE_ERR_INVALID_ARG, "%s: row_scales is null", who);
    return ffn_vanilla_impl(row_scales, who, x, T, d, n, k, I, MOE_DTYPE_FP8_E4M3, w_gate, w_up, w_down, I_s,
                            s_gate, s_up, s_down, ws, ws_bytes, out_mode, out, stream);
}

int deamoe_ffn(const float* x, int T, int d, int n, int k, int experts_per_dept, int I_sh,
               int I_pr, int dtype, const void* dept_gate, const void* dept_up,
               const void* dept_down, const void* priv_gate, const void* priv_up,
               const void* priv_down, int I_s, const void* s_gate, const void* s_up,
               const void* s_down, const void* ws, size_t ws_bytes, int out_mode, float* out,
               void* stream) {
    return deamoe_ffn_impl(nullptr, "deamoe_ffn", x, T, d, n, k, experts_per_dept, I_sh, I_pr, dtype, dept_gate,
                           dept_up, dept_down, priv_gate, priv_up, priv_down, I_s, s_gate, s_up, s_down, ws,
                           ws_bytes, out_mode, out, stream);
}

int deamoe_ffn_fp8(const float* x, int T, int d, int n, int k, int experts_per_dept, int I_sh,
                   int I_pr, const void* dept_gate, const void* dept_up, const void* dept_down,
                   const void* priv_gate, const void* priv_up, const void* priv_down, int I_s,
                   const void* s_gate, const void* s_up, const void* s_down,
                   const float* const row_scales[9], const void* ws, size_t ws_bytes, int out_mode,
                   float* out, void* stream) {
    const char* who = "deamoe_ffn_fp8";
    if (!row_scales) return fail(MOE_ERR_INVALID_ARG, "%s: row_scales is null", who);
    return deamoe_ffn_impl(row_scales, who, x, T, d, n, k, experts_per_dept, I_sh, I_pr, MOE_DTYPE_FP8_E4M3,
                           dept_gate, dept_up, dept_down, priv_gate, priv_up, priv_down, I_s, s_gate, s_up,
                           s_down, ws, ws_bytes, out_mode, out, stream);
}

int moe_layer_forward(const float* x, int T, int d, int n, int k, float scale,
                      const float* w_router, const float* bias, int I, int dtype,
                      const void* w_gate, const void* w_up, const void* w_down, int I_s,
                      const void* s_gate, const void* s_up, const void* s_down, void* ws,
                      size_t ws_bytes, int32_t* topk_idx, float* topk_w, float* y, void* stream) {
    return layer_forward_impl(nullptr, "moe_layer_forward", x, T, d, n, k, scale, w_router, bias, I, dtype,
                              w_gate, w_up, w_down, I_s, s_gate, s_up, s_down, ws, ws_bytes, topk_idx, topk_w,
                              y, stream);
}

int moe_layer_forward_fp8(const float* x, int T, int d, int n, int k, float scale,
                          const float* w_router, const float* bias, int I, const void* w_gate,
                          const void* w_up, const void* w_down, int I_s, const void* s_gate,
                          const void* s_up, const void* s_down, const float* const row_scales[6],
                          void* ws, size_t ws_bytes, int32_t* topk_idx, float* topk_w, float* y,
                          void* stream) {
    const char* who = "moe_layer_forward_fp8";
    if (!row_scales) return fail(MOE_ERR_INVALID_ARG, "%s: row_scales is null", who);
    return layer_forward_impl(row_scales, who, x, T, d, n, k, scale, w_router, bias, I, MOE_DTYPE_FP8_E4M3,
                              w_gate, w_up, w_down, I_s, s_gate, s_up, s_down, ws, ws_bytes, topk_idx, topk_w,
                              y, stream);
}

int deamoe_layer_forward(const float* x, int T, int d, int n, int k, float scale,
                         const float* w_router, const float* bias, int experts_per_dept, int I_sh,
                         int I_pr, int dtype, const void* dept_gate, const void* dept_up,
                         const void* dept_down, const void* priv_gate, const void* priv_up,
                         const void* priv_down, int I_s, const void* s_gate, const void* s_up,
                         const void* s_down, void* ws, size_t ws_bytes, int32_t* topk_idx,
                         float* topk_w, float* y, void* stream) {
    return deamoe_layer_forward_impl(nullptr, "deamoe_layer_forward", x, T, d, n, k, scale, w_router, bias,
                                     experts_per_dept, I_sh, I_pr, dtype, dept_gate, dept_up, dept_down,
                                     priv_gate, priv_up, priv_down, I_s, s_gate, s_up, s_down, ws, ws_bytes,
                                     topk_idx, topk_w, y, stream);
}

int deamoe_layer_forward_fp8(const float* x, int T, int d, int n, int k, float scale,
                             const float* w_router, const float* bias, int experts_per_dept, int I_sh,
                             int I_pr, const void* dept_gate, const void* dept_up, const void* dept_down,
                             const void* priv_gate, const void* priv_up, const void* priv_down, int I_s,
                             const void* s_gate, const void* s_up, const void* s_down,
                             const float* const row_scales[9], void* ws, size_t ws_bytes,
                             int32_t* topk_idx, float* topk_w, float* y, void* stream) {
    const char* who = "deamoe_layer_forward_fp8";
    if (!row_scales) return fail(MOE_ERR_INVALID_ARG, "%s: row_scales is null", who);
    return deamoe_layer_forward_impl(row_scales, who, x, T, d, n, k, scale, w_router, bias, experts_per_dept,
                                     I_sh, I_pr, MOE_DTYPE_FP8_E4M3, dept_gate, dept_up, dept_down, priv_gate,
                                     priv_up, priv_down, I_s, s_gate, s_up, s_down, ws, ws_bytes, topk_idx,
                                     topk_w, y, stream);
}

// Form-P scratch after the standard layout: G and U [T*min(k,m), r], then
// Z [T*k, r], all fp32.
static bool formp_layout(int T, int n, int k, int g, int r, moe_ws_layout* L, size_t* og, size_t* ou,
                         size_t* oz, size_t* total) {
    if (g < 2 || r < 16 || r % 16 != 0 || !layout_of(T, n, k, g, L)) return false;
    const int m = n / g;
    const size_t mk = (size_t)T * (k < m ? k : m);
    *og = align_up(L->total, 256);
    *ou = align_up(*og + mk * r * sizeof(float), 256);
    *oz = align_up(*ou + mk * r * sizeof(float), 256);
    *total = align_up(*oz + (size_t)T * k * r * sizeof(float), 256);
    return true;
}

size_t moe_formp_workspace_bytes(int T, int n, int k, int experts_per_dept, int r) {
    moe_ws_layout L;
    size_t og, ou, oz, total;
    return formp_layout(T, n, k, experts_per_dept, r, &L, &og, &ou, &oz, &total) ? total : 0;
}

// Checks shared by the form-P layer and its FFN step; fills the layout and
// the scratch offsets.
static int formp_checks(const float* x, int T, int d, int n, int k, int g, int r, int dtype,
                        const void* const (&wts)[6], const void* ws, size_t ws_bytes, const float* y,
                        moe_ws_layout* L, size_t* og, size_t* ou, size_t* oz, const char* who) {
    size_t total;
    if (!formp_layout(T, n, k, g, r, L, og, ou, oz, &total))
        return fail(MOE_ERR_INVALID_ARG,
                    "%s: need 1<=T<=%d, 1<=n<=%d, 1<=k<=min(n,%d), experts_per_dept>=2 dividing n, "
                    "r a positive multiple of 16 (T=%d n=%d k=%d g=%d r=%d)",
                    who, moe::kMaxT, moe::kMaxN, moe::kMaxK, T, n, k, g, r);
    if (!ws || !aligned16(ws)) return fail(MOE_ERR_INVALID_ARG, "%s: workspace null or unaligned", who);
    if (ws_bytes < total)
        return fail(MOE_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu required (moe_formp_workspace_bytes)",
                    who, ws_bytes, total);
    int rc = check_hidden(x, d, who);
    if (rc) return rc;
    if (dtype != MOE_DTYPE_BF16) return fail(MOE_ERR_UNSUPPORTED, "%s: form P takes bf16 weights only", who);
    if (d > moe::formp_max_hidden() || d > kMaxRouterHidden)
        return fail(MOE_ERR_UNSUPPORTED, "%s: d=%d exceeds %d", who, d, moe::formp_max_hidden());
    if (r > moe::formp_max_width()) return fail(MOE_ERR_UNSUPPORTED, "%s: r=%d exceeds %d", who, r, moe::formp_max_width());
    for (const void* p : wts)
        if (!p || !aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s: weights null or unaligned", who);
    if (!y || !aligned16(y)) return fail(MOE_ERR_INVALID_ARG, "%s: y null or unaligned", who);
    return MOE_OK;
}

// Whether the matrix form's department passes (up, down) run on the tensor
// cores: bf16 rows of d and r both multiples of 128 and d within the
// activation split; with a fixed threshold (moe_set_tc_min_tokens) when T
// reaches it; otherwise when the department rows streamed by the busiest SM
// are fewer, estimated from the expected occupancy of the departments (a
// token reaches a department with probability k_dept / m under group-limited
// routing, else 1 - C(n - g, k) / C(n, k)): the CUDA-core passes read a
// department's rows once per group of 4 tokens spread over every SM, the
// tensor-core passes once per 32 tokens in 128-row tiles, one SM per tile.
// As for the form-C FFN, the CUDA-core rows are weighted 4/3 on rows wider
// than 4096; on narrower rows the tensor cores must win by half again (their
// tiles are few there and the kernel's fixed costs weigh more: measured on
// the 7B match, h = 1024, r = 384).  The private pass (A matrices, about one
// token per expert) stays on the CUDA cores.
static bool formp_tc(int T, int d, int n, int k, int g, int k_dept, int r) {
    if (d % moe::kTcHiddenQuantum != 0 || r % moe::kTcBoxRows != 0 || d > moe::kMaxXbHidden) return false;
    const int thr = tc_min_tokens();
    if (thr > 0) return T >= thr;
    const int m = n / g;
    double p = 1.0;
    if (k_dept > 0) {
        p = (double)k_dept / m;
    } else {
        double miss = 1.0;
        for (int i = 0; i < k; ++i) miss *= n - g - i > 0 ? (double)(n - g - i) / (n - i) : 0.0;
        p = 1.0 - miss;
    }
    p = p < 1.0 ? p : 1.0;
    const double hit = 1.0 - std::pow(1.0 - p, T);        // a department is active
    const double active = m * hit;
    const double tokens = hit > 0.0 ? T * p / hit : 0.0;   // tokens of an active department
    const double sms = moe::device_sm_count();
    const double cc = active * r * std::ceil(tokens / moe::kGroupTokens) / sms * (d > moe::kTcWideHidden ? 4.0 : 3.0);
    const double tiles = active * (r / moe::kTcBoxRows) * std::ceil(tokens / moe::kTcGroupTokens);
    const double tc = std::ceil(tiles / sms) * moe::kTcBoxRows * 3.0 * (d > moe::kTcWideHidden ? 1.0 : 1.5);
    return tc < cc;
}

static int formp_launch(const float* x, int T, int d, int n, int k, int g, int r, const void* const (&wts)[6],
                        const int32_t* topk_idx, void* ws, const moe_ws_layout& L, size_t og, size_t ou,
                        size_t oz, float* y, bool zero_y, bool tc, cudaStream_t s, const char* who) {
    char* b = static_cast<char*>(ws);
    const int m = n / g;
    moe::FormPArgs a = {};
    a.x = x;
    a.T = T; a.d = d; a.n = n; a.k = k; a.g = g; a.m = m;
    a.mk = k < m ? k : m;
    a.r = r;
    a.dgate = wts[0]; a.dup = wts[1]; a.ddown = wts[2];
    a.agate = wts[3]; a.aup = wts[4]; a.adown = wts[5];
    a.topk_idx = topk_idx;
    a.gbuf = reinterpret_cast<float*>(b + og);
    a.ubuf = reinterpret_cast<float*>(b + ou);
    a.zbuf = reinterpret_cast<float*>(b + oz);
    a.y = y;
    a.zero_y = zero_y ? 1 : 0;
    a.ws = resolve(ws, L);
    const int sms = moe::device_sm_count();
    if (!tc) {
        cudaError_t e = moe::launch_formp(a, sms, s);
        if (e != cudaSuccess) return cuda_fail(e, who);
        return MOE_OK;
    }
    // department passes on the tensor cores, the private pass between them on
    // the CUDA cores; each a programmatic dependent of the one before
    moe::TcArgs t = {};
    moe::FfnArgs& f = t.f;
    f.x = x;
    f.T = T; f.d = d; f.n = n; f.k = k; f.g = g;
    f.dtype = MOE_DTYPE_BF16;
    f.cls[0].w_gate = wts[0];
    f.cls[0].w_up = wts[1];
    f.cls[0].w_down = wts[2];
    f.cls[0].rows = r;
    f.cls[0].kind = moe::kUnitDept;
    f.ncls = 1;
    f.ws = a.ws;
    f.out = y;
    f.out_mode = MOE_OUT_ACCUM;
    f.pdl = 1;
    f.sms = sms;
    f.max_tokens = INT_MAX;
    t.min_tokens = 1;
    for (int mat = 0; mat < 3; ++mat)
        if (!encode_weight_map(&t.maps[0][mat], wts[mat], n / g, r, d))
            return fail(MOE_ERR_CUDA, "%s: tensor map encoding failed", who);
    t.gbuf = a.gbuf;
    t.ubuf = a.ubuf;
    t.zbuf = a.zbuf;
    t.topk_idx = topk_idx;
    t.zero_y = zero_y ? 1 : 0;
    t.pmode = moe::kTcFormPUp;
    cudaError_t e = moe::launch_ffn_tc(t, s);
    if (e == cudaSuccess) e = moe::launch_formp_pass(a, moe::kFormPPriv, sms, s);
    if (e == cudaSuccess) {
        t.pmode = moe::kTcFormPDown;
        e = moe::launch_ffn_tc(t, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, who);
    return MOE_OK;
}

int deamoe_p_layer_forward(const float* x, int T, int d, int n, int k, float scale, const float* w_router,
                           const float* bias, int experts_per_dept, int k_dept, int r, int dtype,
                           const void* dept_gate, const void* dept_up, const void* dept_down,
                           const void* a_gate, const void* a_up, const void* a_down, void* ws,
                           size_t ws_bytes, int32_t* topk_idx, float* topk_w, float* y, void* stream) {
    const char* who = "deamoe_p_layer_forward";
    const int g = experts_per_dept;
    const void* const wts[6] = {dept_gate, dept_up, dept_down, a_gate, a_up, a_down};
    moe_ws_layout L;
    size_t og, ou, oz;
    int rc = formp_checks(x, T, d, n, k, g, r, dtype, wts, ws, ws_bytes, y, &L, &og, &ou, &oz, who);
    if (rc) return rc;
    const int m = n / g;
    if (k_dept < 0 || k_dept > m || (k_dept > 0 && (long long)k > (long long)k_dept * g))
        return fail(MOE_ERR_INVALID_ARG, "%s: k_dept=%d must be 0 (plain top-k) or in [1, %d] with k <= k_dept*g",
                    who, k_dept, m);
    if (!w_router || !aligned16(w_router)) return fail(MOE_ERR_INVALID_ARG, "%s: w_router null or unaligned", who);
    if (!topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "%s: routing outputs are null", who);
    moe::RouteArgs ra = {};
    ra.x = x;
    ra.w_router = w_router;
    ra.bias = bias;
    ra.T = T; ra.d = d; ra.n = n; ra.k = k;
    ra.scale = scale;
    ra.topk_idx = topk_idx;
    ra.topk_w = topk_w;
    ra.ws = resolve(ws, L);
    ra.g = g;
    ra.y_zero = y;
    ra.y_elems = (long long)T * d;
    ra.fuse_dispatch = 1;
    ra.route_g = g;
    ra.k_dept = k_dept;
    const bool tc = formp_tc(T, d, n, k, g, k_dept, r);
    ra.split_x = tc ? 1 : 0;
    cudaStream_t s = as_stream(stream);
    cudaError_t e = moe::launch_route(ra, s);
    if (e != cudaSuccess) return cuda_fail(e, who);
    return formp_launch(x, T, d, n, k, g, r, wts, topk_idx, ws, L, og, ou, oz, y, false, tc, s, who);
}

int deamoe_p_ffn(const float* x, int T, int d, int n, int k, int experts_per_dept, int r, int dtype,
                 const void* dept_gate, const void* dept_up, const void* dept_down, const void* a_gate,
                 const void* a_up, const void* a_down, const int32_t* topk_idx, void* ws, size_t ws_bytes,
                 float* y, void* stream) {
    const char* who = "deamoe_p_ffn";
    const int g = experts_per_dept;
    const void* const wts[6] = {dept_gate, dept_up, dept_down, a_gate, a_up, a_down};
    moe_ws_layout L;
    size_t og, ou, oz;
    int rc = formp_checks(x, T, d, n, k, g, r, dtype, wts, ws, ws_bytes, y, &L, &og, &ou, &oz, who);
    if (rc) return rc;
    if (!topk_idx) return fail(MOE_ERR_INVALID_ARG, "%s: topk_idx is null", who);
    // the standalone step takes no k_dept: the plain top-k's occupancy
    const bool tc = formp_tc(T, d, n, k, g, 0, r);
    cudaStream_t s = as_stream(stream);
    if (tc) {
        cudaError_t e = moe::launch_split_x(x, (long long)T * d, resolve(ws, L).xb, s);
        if (e != cudaSuccess) return cuda_fail(e, who);
    }
    return formp_launch(x, T, d, n, k, g, r, wts, topk_idx, ws, L, og, ou, oz, y, true, tc, s, who);
}

int64_t moe_unique_weight_bytes_formp(int d, int n, int r, int A_d, int A_e) {
    if (d <= 0 || n <= 0 || r <= 0 || A_d < 0 || A_e < 0 || A_e > n) return -1;
    return 4LL * d * n + 2LL * ((int64_t)A_d * 3 * d * r + (int64_t)A_e * 3 * r * r);
}

int64_t moe_unique_weight_bytes_vanilla(int d, int n, int I, int I_s, int dtype, int A_e) {
    const int bw = weight_bytes(dtype);
    if (d <= 0 || n <= 0 || I < 0 || I_s < 0 || bw == 0 || A_e < 0 || A_e > n) return -1;
    return 4LL * d * n + unit_row_bytes(d, dtype) * ((int64_t)A_e * I + I_s);
}

int64_t moe_unique_weight_bytes_deamoe(int d, int n, int I_sh, int I_pr, int I_s, int dtype,
                                       int A_d, int A_e) {
    const int bw = weight_bytes(dtype);
    if (d <= 0 || n <= 0 || I_sh < 0 || I_pr < 0 || I_s < 0 || bw == 0 || A_d < 0 || A_e < 0 ||
        A_e > n)
        return -1;
    return 4LL * d * n + unit_row_bytes(d, dtype) * ((int64_t)A_d * I_sh + (int64_t)A_e * I_pr + I_s);
}

}  // extern "C"
