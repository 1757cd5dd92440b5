/*
 * moe_decode.h -- C ABI of the GB300 (sm_103a) MoE / DeaMoE small-batch decode layer.
 *
 * The layer (vanilla top-k SwiGLU MoE with an optional always-on shared expert,
 * and the DeaMoE department variant) is split into the steps the pages describe:
 * routing, dispatch, expert FFN, combine.  Each step is one entry point; the
 * *_layer_forward calls chain them with fewer launches.
 *
 * Sources:
 *   [DeaMoE]  "DeaMoE: Efficient MoE Structure for Fast Small-Batch Decoding":
 *             §2.1 eqs. (1)-(3), §3.1-3.2 (departments, two-stage routing).
 *   [DSMoE]   "DeepSeekMoE Guide: Fine-Grained Experts & Dynamic Routing":
 *             "Mathematical Formulation of the DeepSeekMoE Forward Pass".
 *   [MoE-inf] "MoE inference engineering, clearly explained": "How a batch
 *             becomes expert-specific matrices", "Local MoE execution pipeline".
 *
 * Conventions (all entry points):
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless a
 *     parameter says "host".  The library never allocates, frees or
 *     synchronises inside a step; all scratch lives in the caller's workspace
 *     (moe_route_topk_noalloc, which has none, uses the library's own fixed
 *     array instead; its declaration states its own terms).
 *   - Every step is asynchronous on the given stream (a cudaStream_t passed as
 *     void*; NULL = legacy default stream).  The workspace steps may be
 *     captured in a CUDA graph.
 *   - Activations, router weights, routing weights and outputs are fp32.
 *     Expert weights are fp32 or bf16 (MOE_DTYPE_*), row-major.
 *   - Weight layout (per unit: an expert, a department backbone, a private
 *     block or the shared expert): gate, up and down are each [rows, d]
 *     row-major.  Gate/up rows are the rows of W_gate / W_up; the down tensor
 *     holds W_down in the paper's [hffn, h] shape and is applied transposed
 *     ([DeaMoE] §2.1).  Stacked tensors are [units, rows, d].
 *   - Pointers must be 16-byte aligned; d must be a multiple of 8 and every
 *     intermediate size a multiple of 16.
 *   - Routing kernels launch as programmatic dependents of the kernel before
 *     them on the stream and may read the router weights before waiting for
 *     that kernel to complete (everything else they read waits).  A kernel of
 *     the caller's that writes router weights must therefore not trigger its
 *     dependents early (griddepcontrol.launch_dependents) before those writes;
 *     copies, memsets and kernels without that trigger need nothing.
 *   - Return value: MOE_OK or a negative MOE_ERR_* code; nothing is launched
 *     when the host-side checks fail.  moe_last_error() gives a message
 *     (thread-local).  Device-side checks (an expert index out of range, a
 *     token choosing an expert twice, a wait that timed out) write a code into
 *     the workspace status word, read with moe_read_status().
 */
#ifndef MOE_DECODE_H
#define MOE_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK               0
#define MOE_ERR_INVALID_ARG (-1)  /* null pointer, bad size, misalignment    */
#define MOE_ERR_UNSUPPORTED (-2)  /* valid but outside what the kernels take */
#define MOE_ERR_WORKSPACE   (-3)  /* workspace smaller than required         */
#define MOE_ERR_CUDA        (-4)  /* a CUDA runtime call failed              */
#define MOE_ERR_TIMEOUT     (-5)  /* device status: a bounded wait expired   */
#define MOE_ERR_DEVICE      (-6)  /* device status: bad routing input        */

#define MOE_DTYPE_F32  0
#define MOE_DTYPE_BF16 1
#define MOE_DTYPE_FP8_E4M3 2  /* E4M3 codes + one fp32 scale per row: the *_fp8 calls */

/* Output modes of the FFN steps. */
#define MOE_OUT_ROWS  0  /* one unweighted row per (unit, token); moe_combine sums them */
#define MOE_OUT_ACCUM 1  /* routing weights applied in the epilogue, added into y[T,d]   */

/* Library version (major*10000 + minor*100 + patch). */
int moe_version(void);

/* Message for the last failed call on this thread ("" if none). */
const char* moe_last_error(void);

/*
 * Tensor-core threshold of the FFN steps.  0 (the library default) chooses per
 * call, on the device, between the tcgen05 kernel and the CUDA-core weight
 * stream from the dispatched token counts (whichever streams fewer weight rows
 * on the busiest SM, CUDA-core rows weighted 4/3 when d > 4096).  For
 * d <= 4096 the tensor-core kernel is launched for that choice only when
 * T > 4 and some unit class expects more than 4 tokens per unit under uniform
 * routing (always, with a shared expert).  min_tokens > 0 fixes the split instead: units (experts,
 * departments, the shared expert) with at least min_tokens gathered tokens
 * run on the tcgen05 kernel, the others on the CUDA cores; a value above every
 * batch size keeps everything on the CUDA cores.  Process-wide; returns the
 * previous setting, or MOE_ERR_INVALID_ARG for a negative value.  The
 * tensor-core kernel applies to bf16 and E4M3 weights with d % 128 == 0 and unit row
 * counts that are multiples of 128.
 */
int moe_set_tc_min_tokens(int min_tokens);

/*
 * Test hook for the FFN kernels' bounded waits (failure detection without a
 * GPU fault; the paper has no counterpart).  wait_ns > 0: every FFN step
 * launched while it is set (moe_ffn_vanilla, deamoe_ffn, the *_layer_forward
 * calls and their FP8 variants) runs with its weight producers issuing no
 * copy, and each consumer wait on a weight stage gives up after wait_ns
 * nanoseconds instead of the normal two seconds.  The kernels then write
 * MOE_ERR_TIMEOUT into the workspace status word (moe_read_status), drain
 * what they started (no copy or MMA is left in flight), free their tensor
 * memory and return; the routing of the step still runs and the output is
 * left incomplete.  wait_ns = 0 turns it off (the default).  Process-wide,
 * read when a step is launched; returns the previous setting, or
 * MOE_ERR_INVALID_ARG for a negative value.
 */
int64_t moe_test_stall_weight_copies(int64_t wait_ns);

/* ------------------------------------------------------------------------- */
/* Workspace                                                                 */
/* ------------------------------------------------------------------------- */

/*
 * Byte offsets of the workspace arrays for a (T, n, k, experts_per_dept) step,
 * in the order they are laid out.
 * The dispatch lists follow [MoE-inf] "How a batch becomes expert-specific
 * matrices" (group the T*k assignments by expert, keep each token id and an
 * inverse map for the combine) and the department token sets X^j of [DeaMoE]
 * §3.2.  Canonical order everywhere: ascending expert (department) id, then
 * ascending token id.
 *
 *   status    int32[4]   offset 0: [0] first device error code (0 = none)
 *   counts    int32[4]   offset 256: [0] active experts A_e, [1] active
 *                        departments A_d, [2], [3] their totals of
 *                        ceil(tokens / 32)
 *   sync      uint32[18] offset 512: [0], [2..17] internal counters (kept at
 *                        zero between calls); [1] FFN kernel choice of the
 *                        last FFN step: 0 none made (fixed threshold, or the
 *                        step is not eligible for the tensor-core kernel),
 *                        1 CUDA cores, 2 tensor cores
 *   logits    float[T*n] router logits (scratch of moe_route_topk)
 *   exp_count int32[n]   assignments per expert
 *   exp_off   int32[n+1] exclusive prefix sum of exp_count
 *   asg_tok   int32[T*k] token of each assignment (expert-sorted)
 *   asg_slot  int32[T*k] top-k slot of each assignment
 *   asg_w     float[T*k] routing weight of each assignment
 *   tok_asg   int32[T*k] inverse map: (token, slot) -> assignment position
 *   act_exp   int32[n]   active experts, ascending (first A_e valid)
 *   exp_units int32[n][4] per active expert q < A_e: {expert, first assignment,
 *                        assignments, inclusive prefix over active experts of
 *                        ceil(assignments / 4)} -- the FFN's work table
 *   xb        4*T*8192 + 4*T bytes of tensor-core FFN scratch: bf16[2][T][d]
 *                        activations split as x = hi + lo (bf16 weights), or
 *                        for E4M3 weights four E4M3 terms u8[4][T][d] of the
 *                        scaled activations and, at byte 4*T*8192, the scale
 *                        exponent int32[T] of each token (rows packed at the
 *                        call's d)
 *   dept_count int32[m]  tokens per department (m = n / experts_per_dept)
 *   dept_off  int32[m+1] exclusive prefix sum of dept_count
 *   dept_tok  int32[T*min(k,m)] tokens of each department (X^j), each once
 *   dept_w    float[T*min(k,m)] sum of the token's routing weights inside X^j
 *   tok_dpos  int32[T*m] (token, department) -> position in dept_tok, or -1
 *   act_dept  int32[m]   active departments, ascending (first A_d valid)
 *   dept_units int32[m][4] the same as exp_units per active department over X^j
 * The department arrays are present only when experts_per_dept > 1.  status,
 * counts and sync do not move with the sizes, and the offsets of the arrays
 * before the department arrays depend on T, n and k only.  So a workspace
 * sized for (T_max, n, k, g) serves every call with T <= T_max, and a call
 * that takes no experts_per_dept (routing) may use a department workspace.
 * A step's calls (route, dispatch, FFN, combine) use the same T.
 */
typedef struct moe_ws_layout {
    size_t total;
    size_t status, counts, logits;
    size_t exp_count, exp_off, asg_tok, asg_slot, asg_w, tok_asg, act_exp;
    size_t dept_count, dept_off, dept_tok, dept_w, tok_dpos, act_dept;
    size_t exp_units, dept_units;
    size_t sync;
    size_t xb;
} moe_ws_layout;

/* Required workspace bytes; 0 on invalid arguments.  T, n, k as for routing;
 * experts_per_dept = g (1 for a vanilla layer; n % g == 0). */
size_t moe_workspace_bytes(int T, int n, int k, int experts_per_dept);

/* Fill *out (host) with the layout above.  MOE_ERR_INVALID_ARG on bad sizes. */
int moe_workspace_layout(int T, int n, int k, int experts_per_dept, moe_ws_layout* out);

/* Zero a workspace once before its first use (enqueued on stream). The library
 * leaves its internal counters at zero after every call, so one init serves
 * any number of steps on that workspace. */
int moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Copy the status word and the active counts to the host (synchronises the
 * stream).  host_status: int32[1], host_counts: int32[2] (A_e, A_d); either may
 * be NULL.  Off the timed path. */
int moe_read_status(const void* ws, size_t ws_bytes, int32_t* host_status,
                    int32_t* host_counts, void* stream);

/* ------------------------------------------------------------------------- */
/* Step 1: router GEMV + top-k + routing weights                             */
/* ------------------------------------------------------------------------- */

/*
 * [DeaMoE] §2.1 eq. (2) S(x) = TopK(W_r x, k) and the weights of eq. (3);
 * [DSMoE] routing-bias form: the bias takes part in the selection only.
 *   x        float[T, d]   hidden states
 *   w_router float[n, d]   router rows (row e = expert e)
 *   bias     float[n] or NULL  selection-only bias b_e
 *   scale    routing-weight scale (1.0 = plain softmax)
 *   topk_idx int32[T, k]   out: experts by descending (logit + bias); equal
 *                          keys -> lower expert index first
 *   topk_w   float[T, k]   out: scale * softmax over the k selected UNBIASED
 *                          logits
 *   ws       workspace (logits scratch + a counter)
 * Limits: 1 <= T <= 128, 1 <= k <= min(n, 32), n <= 1024, d % 8 == 0.
 */
int moe_route_topk(const float* x, const float* w_router, const float* bias,
                   int T, int d, int n, int k, float scale,
                   int32_t* topk_idx, float* topk_w,
                   void* ws, size_t ws_bytes, void* stream);

/*
 * Group-limited top-k: [DeaMoE] §3.3 caps the departments a token activates
 * at k_dept; the strict variant (its appendix ablation, Table 4) makes the
 * selection cover exactly k_dept departments.  Expert e belongs to department
 * e / experts_per_dept.  Per token:
 *   1. a department's score is the best key (logit + bias) of its experts;
 *      the k_dept best-scored departments are kept (equal scores -> lower
 *      department first);
 *   2. soft (strict == 0): the top-k of the kept departments' experts, by key
 *      as in moe_route_topk;
 *      strict (strict != 0): each kept department's best expert, plus the best
 *      k - k_dept other experts of the kept departments (the end point of
 *      replacing the lowest-ranked expert whose department holds another
 *      selected expert by the best expert of an uncovered kept department);
 *   3. topk_idx by descending key (equal keys -> lower index), topk_w =
 *      scale * softmax over the selected unbiased logits.
 * Other arguments, the workspace and the device status as moe_route_topk.
 * Limits: those of moe_route_topk; experts_per_dept divides n;
 * 1 <= k_dept <= n / experts_per_dept; k <= k_dept * experts_per_dept;
 * strict needs k >= k_dept.  Violations return MOE_ERR_INVALID_ARG and
 * launch nothing.
 */
int moe_route_topk_grouped(const float* x, const float* w_router, const float* bias,
                           int T, int d, int n, int k, int experts_per_dept, int k_dept,
                           int strict, float scale, int32_t* topk_idx, float* topk_w,
                           void* ws, size_t ws_bytes, void* stream);

/*
 * moe_route_topk without a workspace and without allocating.  The paper has no
 * counterpart: this is a library convenience.
 *
 * It is for callers that can neither pass a workspace nor let the library
 * allocate: an engine that carves up all device memory once at start-up, or
 * a decode loop that must not stall the device (cudaFree synchronises) or
 * fail for lack of memory mid-step.  The logits scratch and the last-block
 * counter live in one fixed device array that the library reserves when it
 * is loaded; the call makes no cudaMalloc/cudaFree and calls no allocating
 * routine.
 *   Same arguments and results as moe_route_topk, except:
 *   status   int32[1] device memory or NULL: receives the call's device status
 *            word (0, or MOE_ERR_DEVICE for a non-finite logit), stream-ordered
 *            after the kernel.
 * Limits: those of moe_route_topk, and T * n <= 65536 (the fixed scratch
 * holds 65536 fp32 logits, 256 KB); larger steps return MOE_ERR_UNSUPPORTED
 * and launch nothing.
 * Set-up: the first call on each device looks up the scratch's device address
 * (cudaGetSymbolAddress) and remembers it for the life of the process; make
 * that first call before any stream capture.  The address remembered is the
 * one in the device's primary context (the runtime's context): calls from
 * another context on the same device, or after cudaDeviceReset, are not
 * supported.
 * Each call clears the scratch's status word and counter (stream-ordered)
 * before its kernel runs.  There is one scratch per device and process:
 * calls that overlap on the device (other streams, other host threads) race
 * on it and give wrong results, so issue them one after another.
 */
int moe_route_topk_noalloc(const float* x, const float* w_router, const float* bias,
                           int T, int d, int n, int k, float scale,
                           int32_t* topk_idx, float* topk_w,
                           int32_t* status, void* stream);

/* ------------------------------------------------------------------------- */
/* Step 2: dispatch (two-level index lists, built on the device)             */
/* ------------------------------------------------------------------------- */

/*
 * Build the expert and department lists of the workspace from (topk_idx,
 * topk_w), with no host round trip.  Expert e belongs to department
 * e / experts_per_dept; a department's token weight is the sum of the token's
 * routing weights over the department's selected experts, in slot order.
 * experts_per_dept = 1 builds only the expert lists (vanilla layer).
 * Device errors (index outside [0,n), a token repeating an expert) set the
 * status word to MOE_ERR_DEVICE.
 */
int moe_dispatch(const int32_t* topk_idx, const float* topk_w, int T, int n, int k,
                 int experts_per_dept, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------- */
/* Step 3: expert FFN                                                        */
/* ------------------------------------------------------------------------- */

/* Rows needed by MOE_OUT_ROWS: T*k assignment rows, then T*min(k,m) department
 * rows (DeaMoE only), then T shared-expert rows (if has_shared).  Each row is
 * float[d].  Returns -1 on invalid arguments. */
int64_t moe_rows_count(int T, int n, int k, int experts_per_dept, int has_shared);

/*
 * Vanilla expert FFN of [DeaMoE] eq. (1) for every active expert over its
 * gathered tokens, plus the shared expert of [DSMoE] (weight 1, all tokens)
 * when I_s > 0.  Reads the dispatch lists from ws.
 *   w_gate, w_up, w_down  [n, I, d] (dtype)
 *   s_gate, s_up, s_down  [I_s, d] or NULL when I_s == 0
 *   out_mode MOE_OUT_ROWS:  out = rows[moe_rows_count, d], overwritten; row
 *            p (< T*k) is expert asg's unweighted output for assignment p;
 *            shared rows start at T*k.
 *   out_mode MOE_OUT_ACCUM: out = y[T, d]; y[t] += sum_s w[t,s] FFN_e(x_t)
 *            (+ FFN_shared(x_t)).  The caller zeroes y beforehand.
 */
int moe_ffn_vanilla(const float* x, int T, int d, int n, int k, int I, int dtype,
                    const void* w_gate, const void* w_up, const void* w_down,
                    int I_s, const void* s_gate, const void* s_up, const void* s_down,
                    const void* ws, size_t ws_bytes, int out_mode, float* out,
                    void* stream);

/*
 * DeaMoE FFN, form C: expert i of department j = i / g has the intermediate
 * [department j's I_sh shared rows ; expert i's I_pr private rows].  Following
 * the two-stage routing of [DeaMoE] §3.2, each active department's backbone
 * runs once over its token set X^j (rows weighted by the department token
 * weight), and each active expert's private rows run over its own tokens.
 *   dept_gate, dept_up, dept_down  [m, I_sh, d]
 *   priv_gate, priv_up, priv_down  [n, I_pr, d] (NULL allowed when I_pr == 0)
 *   s_gate, s_up, s_down           [I_s, d] or NULL when I_s == 0
 *   out_mode as for moe_ffn_vanilla: ROWS puts private rows at assignment
 *   positions, department rows at T*k + dept position, shared rows after.
 * experts_per_dept = 1 is allowed: each department is then one expert whose
 * intermediate is [I_sh rows ; I_pr rows], i.e. a vanilla layer with
 * I = I_sh + I_pr, and there are no department rows.
 */
int deamoe_ffn(const float* x, int T, int d, int n, int k, int experts_per_dept,
               int I_sh, int I_pr, int dtype,
               const void* dept_gate, const void* dept_up, const void* dept_down,
               const void* priv_gate, const void* priv_up, const void* priv_down,
               int I_s, const void* s_gate, const void* s_up, const void* s_down,
               const void* ws, size_t ws_bytes, int out_mode, float* out,
               void* stream);

/* ------------------------------------------------------------------------- */
/* Step 4: combine                                                           */
/* ------------------------------------------------------------------------- */

/*
 * [MoE-inf] combine: return every row to its token through the inverse map and
 * add it with its routing weight ([DeaMoE] eq. (3)).  For token t, in this
 * fixed order: slots s = 0..k-1 (weight topk_w[t,s]), then its departments in
 * ascending id (department weight), then its shared-expert row (weight 1).
 *   rows float[moe_rows_count(...), d] from an FFN step in MOE_OUT_ROWS mode
 *   y    float[T, d], overwritten
 */
int moe_combine(const float* rows, int T, int d, int n, int k, int experts_per_dept,
                int has_shared, const void* ws, size_t ws_bytes, float* y,
                void* stream);

/* ------------------------------------------------------------------------- */
/* Host activations                                                          */
/* ------------------------------------------------------------------------- */

/*
 * A step whose activations live on the host: moe_input_from_host copies
 * x_host (host, float[T, d]) into x (device, float[T, d]) before the layer
 * call, and moe_output_to_host copies its output y (device, float[T, d]) into
 * y_host (host) after it.  Each is one asynchronous copy on `stream`, ordered
 * with the layer's launches.  Page-locked host memory keeps the copy
 * asynchronous; pageable memory works, but the copy blocks the host.  Either
 * buffer stays owned by the caller, and y_host is complete once the stream
 * reaches the copy (synchronise before reading it).  MOE_ERR_INVALID_ARG for a
 * null pointer or T, d < 1; MOE_ERR_CUDA if the copy cannot be enqueued.
 */
int moe_input_from_host(float* x, const float* x_host, int T, int d, void* stream);
int moe_output_to_host(float* y_host, const float* y, int T, int d, void* stream);

/* ------------------------------------------------------------------------- */
/* Whole layer                                                               */
/* ------------------------------------------------------------------------- */

/*
 * route -> dispatch -> FFN (MOE_OUT_ACCUM) in two or three launches.  The
 * router kernel also zeroes y; the FFN launches as its programmatic dependent.
 * When the step runs on one FFN kernel alone (n <= 256) the router kernel
 * writes the logits only and every CTA of that FFN kernel takes the top-k
 * and builds the dispatch itself in shared memory: the CUDA-core kernel
 * when the tensor-core kernel is not launched, the tensor-core kernel when
 * rows are at most 4096 wide, T <= 32 and the automatic choice launches it.
 * Otherwise the router kernel builds the dispatch for the FFN kernels to read
 * (and both run, one of them choosing on the device).  Either way topk_idx /
 * topk_w receive the routing like moe_route_topk, and the workspace
 * afterwards holds the dispatch lists of moe_dispatch (so an FFN step in
 * MOE_OUT_ROWS mode and moe_combine can follow on the same workspace).
 */
int moe_layer_forward(const float* x, int T, int d, int n, int k, float scale,
                      const float* w_router, const float* bias,
                      int I, int dtype, const void* w_gate, const void* w_up,
                      const void* w_down, int I_s, const void* s_gate,
                      const void* s_up, const void* s_down,
                      void* ws, size_t ws_bytes, int32_t* topk_idx, float* topk_w,
                      float* y, void* stream);

int deamoe_layer_forward(const float* x, int T, int d, int n, int k, float scale,
                         const float* w_router, const float* bias,
                         int experts_per_dept, int I_sh, int I_pr, int dtype,
                         const void* dept_gate, const void* dept_up, const void* dept_down,
                         const void* priv_gate, const void* priv_up, const void* priv_down,
                         int I_s, const void* s_gate, const void* s_up, const void* s_down,
                         void* ws, size_t ws_bytes, int32_t* topk_idx, float* topk_w,
                         float* y, void* stream);

/* ------------------------------------------------------------------------- */
/* FP8 (E4M3) expert weights                                                 */
/* ------------------------------------------------------------------------- */

/*
 * The FFN steps and layer calls above with FP8 E4M3 weights and one fp32
 * scale per weight row.  The pages count expert weights in FP8 ([DeaMoE] §1:
 * a DeepSeek-V3 expert is about 44 MB of FP8 weights) and note that
 * quantised weights change the model's numbers ([MoE-inf], quantisation);
 * the scale granularity (one per row of each gate / up / down matrix, i.e.
 * per intermediate index of a unit) is this library's choice.
 *   Weight tensors: E4M3 codes (1 byte) in the layouts of the bf16 calls.
 *   row_scales: a host array of device pointers to float scales, three per
 *     class -- gate, up, down -- each [units * rows] (row r of unit u at
 *     u * rows + r): the value of a weight is scale[row] * e4m3(code).
 *     moe_*_vanilla_fp8 / moe_layer_forward_fp8: [0..2] the experts,
 *     [3..5] the shared expert (ignored when I_s == 0);
 *     deamoe_*_fp8: [0..2] the departments, [3..5] the private rows
 *     (ignored when I_pr == 0), [6..8] the shared expert (ignored when
 *     I_s == 0).
 * Other arguments, limits, kernel choice and results as for the bf16 calls.
 * On the tensor cores the gate and up products take the codes as they are
 * (8-bit MMAs) against the activations written as four E4M3 terms per token
 * with a power-of-two scale (x = 2^-e0 (q0 + q1/16 + q2/256 + q3/4096), within
 * 2^-16 of each element; the workspace's xb region holds them); the down
 * product expands the codes to bf16 exactly.  Either kernel's output is
 * within 1e-4 of the layer on the exactly decoded weights.  The bf16 / fp32
 * calls reject dtype MOE_DTYPE_FP8_E4M3.
 */
int moe_ffn_vanilla_fp8(const float* x, int T, int d, int n, int k, int I,
                        const void* w_gate, const void* w_up, const void* w_down, int I_s,
                        const void* s_gate, const void* s_up, const void* s_down,
                        const float* const row_scales[6], const void* ws, size_t ws_bytes,
                        int out_mode, float* out, void* stream);

int deamoe_ffn_fp8(const float* x, int T, int d, int n, int k, int experts_per_dept, int I_sh,
                   int I_pr, const void* dept_gate, const void* dept_up, const void* dept_down,
                   const void* priv_gate, const void* priv_up, const void* priv_down, int I_s,
                   const void* s_gate, const void* s_up, const void* s_down,
                   const float* const row_scales[9], const void* ws, size_t ws_bytes,
                   int out_mode, float* out, void* stream);

int moe_layer_forward_fp8(const float* x, int T, int d, int n, int k, float scale,
                          const float* w_router, const float* bias, int I,
                          const void* w_gate, const void* w_up, const void* w_down, int I_s,
                          const void* s_gate, const void* s_up, const void* s_down,
                          const float* const row_scales[6], void* ws, size_t ws_bytes,
                          int32_t* topk_idx, float* topk_w, float* y, void* stream);

int deamoe_layer_forward_fp8(const float* x, int T, int d, int n, int k, float scale,
                             const float* w_router, const float* bias, int experts_per_dept,
                             int I_sh, int I_pr, const void* dept_gate, const void* dept_up,
                             const void* dept_down, const void* priv_gate, const void* priv_up,
                             const void* priv_down, int I_s, const void* s_gate, const void* s_up,
                             const void* s_down, const float* const row_scales[9], void* ws,
                             size_t ws_bytes, int32_t* topk_idx, float* topk_w, float* y,
                             void* stream);

/* ------------------------------------------------------------------------- */
/* DeaMoE layer in the paper's parameterisation ("form P")                   */
/* ------------------------------------------------------------------------- */

/*
 * [DeaMoE] §3.1 eq. (4) with sigma = SiLU at all three interfaces (§3.4):
 * department j holds W_g^j, W_u^j, W_d^j, expert i (of department i / g)
 * holds A_g^i, A_u^i, A_d^i, and
 *     g^ = SiLU(A_g SiLU(W_g x)),   u^ = A_u SiLU(W_u x),
 *     DeaMoE_i(x) = W_d^T SiLU(A_d^T (g^ * u^)),
 *     y_t = sum over the token's selected experts of p_i DeaMoE_i(x_t)
 * (eq. (3)), with the routing of moe_route_topk, or of
 * moe_route_topk_grouped (soft) when k_dept > 0 (the paper's configurations
 * cap the departments per token, §3.3 and Table 1).
 *   x, T, d (= h), n, k, scale, w_router, bias, topk_idx, topk_w: as for
 *            deamoe_layer_forward
 *   experts_per_dept  g >= 2 dividing n (m = n / g departments)
 *   k_dept   0 for plain top-k, else 1 <= k_dept <= m with k <= k_dept * g
 *   r        department / expert width (hffn): a multiple of 16, <= 2048
 *   dtype    MOE_DTYPE_BF16 only (others: MOE_ERR_UNSUPPORTED)
 *   dept_gate, dept_up, dept_down  bf16[m][r][d]: the rows of W_g^j, W_u^j
 *            and of W_d^j in the paper's [hffn, h] shape (applied
 *            transposed)
 *   a_gate, a_up, a_down  bf16[n][r][r]: A_g^i, A_u^i and A_d^i, row-major
 *            (A_d^i is applied transposed)
 *   ws       moe_formp_workspace_bytes(T, n, k, g, r) bytes: the layout of
 *            moe_workspace_layout(T, n, k, g) followed by fp32 scratch for
 *            SiLU(W_g x) and SiLU(W_u x) per department entry and for
 *            A_d^T Y per assignment
 *   y        float[T, d] out (overwritten)
 * d <= 7680; every pointer 16-byte aligned.  Four launches: routing with the
 * fused dispatch, then three weight passes chained by programmatic dependent
 * launches (department up-projection, expert A matrices, department
 * down-projection).  The workspace holds the dispatch lists afterwards.
 */
size_t moe_formp_workspace_bytes(int T, int n, int k, int experts_per_dept, int r);

int deamoe_p_layer_forward(const float* x, int T, int d, int n, int k, float scale,
                           const float* w_router, const float* bias,
                           int experts_per_dept, int k_dept, int r, int dtype,
                           const void* dept_gate, const void* dept_up, const void* dept_down,
                           const void* a_gate, const void* a_up, const void* a_down,
                           void* ws, size_t ws_bytes, int32_t* topk_idx, float* topk_w,
                           float* y, void* stream);

/*
 * The three weight passes of deamoe_p_layer_forward alone, on a routing the
 * caller already made: topk_idx [T, k] and the workspace's dispatch lists
 * (moe_dispatch with experts_per_dept, or an earlier layer call on the same
 * inputs).  y is overwritten.  Arguments and limits as above.
 */
int deamoe_p_ffn(const float* x, int T, int d, int n, int k, int experts_per_dept, int r,
                 int dtype, const void* dept_gate, const void* dept_up, const void* dept_down,
                 const void* a_gate, const void* a_up, const void* a_down,
                 const int32_t* topk_idx, void* ws, size_t ws_bytes, float* y, void* stream);

/* ------------------------------------------------------------------------- */
/* Router-bias load balancing                                                */
/* ------------------------------------------------------------------------- */

#define MOE_BIAS_SIGN         0  /* b_i - gamma over the target, + gamma under it */
#define MOE_BIAS_PROPORTIONAL 1  /* b_i + gamma * (target - counts_i)             */

/*
 * One gradient-free update of the selection-only router bias from a batch's
 * expert loads: [DSMoE] "Algorithmic Mechanics: Auxiliary-Loss-Free Dynamic
 * Load Balancing", step 4 of its routing loop (sign rule) and its part 2
 * (proportional rule), with the imbalance ratio of its part 3.
 *   counts    int32[n] device: tokens routed to each expert in the batch (the
 *             workspace's exp_count after a dispatch or a layer forward)
 *   n         1 <= n <= 1024
 *   gamma     step size, finite and >= 0
 *   rule      MOE_BIAS_SIGN or MOE_BIAS_PROPORTIONAL
 *   bias      float[n] device, updated in place; NULL to only measure
 *   imbalance float[1] device or NULL: max_i counts_i / mean_i counts_i
 *             (0 when no token was routed)
 * The target load is the mean, sum(counts) / n; an expert exactly on it keeps
 * its bias under the sign rule.  The arithmetic is fp64 (IEEE, one rounding
 * to fp32 at the end), so results are the same on every run.  One kernel of
 * one block, stream-ordered; bias and imbalance may not both be NULL.
 */
int moe_bias_update(const int32_t* counts, int n, float gamma, int rule,
                    float* bias, float* imbalance, void* stream);

/* ------------------------------------------------------------------------- */
/* Byte accounting (host only)                                               */
/* ------------------------------------------------------------------------- */

/*
 * Weight bytes one step must read at least once ("unique weight bytes"): the
 * fp32 router, the shared expert, and each active unit's three matrices once.
 *   vanilla: 4*d*n + R*(A_e*I + I_s)
 *   DeaMoE:  4*d*n + R*(A_d*I_sh + A_e*I_pr + I_s)
 * where R, the bytes of one intermediate row of a unit, is 3*d*bw with
 * bw = 2 (bf16) or 4 (fp32), and 3*(d + 4) for FP8 (codes and the three
 * fp32 row scales).  Returns -1 on invalid arguments.
 */
int64_t moe_unique_weight_bytes_vanilla(int d, int n, int I, int I_s, int dtype, int A_e);
int64_t moe_unique_weight_bytes_deamoe(int d, int n, int I_sh, int I_pr, int I_s,
                                       int dtype, int A_d, int A_e);
/* Form P (bf16 weights): 4*d*n + 2*(A_d*3*d*r + A_e*3*r*r). */
int64_t moe_unique_weight_bytes_formp(int d, int n, int r, int A_d, int A_e);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_H */
