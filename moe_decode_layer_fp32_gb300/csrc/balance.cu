// Router-bias load balancing of "DeepSeekMoE Guide: Fine-Grained Experts &
// Dynamic Routing", section "Algorithmic Mechanics: Auxiliary-Loss-Free Dynamic
// Load Balancing": after a batch, each expert's selection-only bias moves
// against its load (step 4 of the routing loop: -gamma when over the target,
// +gamma when under; part 2: gamma times the distance to the target), and the
// batch's load balance is reported as max load / mean load (part 3).
//
// The target is the mean load, sum(counts) / n.  The whole update is one
// block: n <= 1024 experts, one thread each, two block reductions.  The
// arithmetic is fp64 with explicit IEEE round-to-nearest operations (no
// contraction) and one rounding to the fp32 bias at the end, so the result
// does not depend on the reduction order.
#include <climits>

#include "kernels.h"
#include "moe_decode.h"

namespace moe {

namespace {

constexpr int kBalanceThreads = 1024;

__global__ void __launch_bounds__(kBalanceThreads)
    bias_update_kernel(const int32_t* counts, int n, float gamma, int rule, float* bias, float* imbalance) {
    __shared__ long long s_sum[kBalanceThreads / 32];
    __shared__ int s_max[kBalanceThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = tid < n ? __ldg(counts + tid) : 0;
    long long sum = c;
    int mx = tid < n ? c : INT_MIN;
    __syncwarp();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
        s_sum[warp] = sum;
        s_max[warp] = mx;
    }
    __syncthreads();
    long long total = 0;
    int cmax = INT_MIN;
#pragma unroll 4
    for (int w = 0; w < kBalanceThreads / 32; ++w) {
        total += s_sum[w];
        cmax = max(cmax, s_max[w]);
    }
    if (bias && tid < n) {
        double b = (double)bias[tid];
        const double gd = (double)gamma;
        if (rule == MOE_BIAS_SIGN) {
            // c vs total / n, compared exactly as c * n vs total
            const long long lhs = (long long)c * n;
            if (lhs > total) b = __dsub_rn(b, gd);
            else if (lhs < total) b = __dadd_rn(b, gd);
        } else {
            const double target = __ddiv_rn((double)total, (double)n);
            b = __dadd_rn(b, __dmul_rn(gd, __dsub_rn(target, (double)c)));
        }
        bias[tid] = __double2float_rn(b);
    }
    if (imbalance && tid == 0)
        *imbalance = total == 0 ? 0.0f
                                : __double2float_rn(__ddiv_rn((double)cmax, __ddiv_rn((double)total, (double)n)));
}

}  // namespace

cudaError_t launch_bias_update(const int32_t* counts, int n, float gamma, int rule, float* bias,
                               float* imbalance, cudaStream_t s) {
    bias_update_kernel<<<1, kBalanceThreads, 0, s>>>(counts, n, gamma, rule, bias, imbalance);
    return cudaGetLastError();
}

}  // namespace moe
