// Auxiliary-loss-free load balancing, applied after a layer step.
//
// The V3 architecture page (section 1.2) keeps a per-expert bias that only
// steers expert selection; after each step the load of every expert is
// checked and the bias is lowered by gamma (the bias update speed) for an
// overloaded expert and raised by gamma for an underloaded one.  Here an
// expert is overloaded when it took more than the mean number of assignments
// T*k/E (counts[e] * E > sum of counts, decided exactly in integers),
// underloaded when it took fewer, and unchanged at exactly the mean.
//
// The kernel also reports the load statistics of the balance-loss listing on
// the Tencent Cloud page: the load fractions counts/sum, their unbiased
// standard deviation, and the largest and smallest load relative to the mean.
#include "internal.h"

namespace moe {
namespace {

constexpr int BAL_THREADS = 256;   // one thread per expert (E <= 256)

__device__ __forceinline__ double block_sum_f64(double v, double* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double s = 0.0;
  for (int w = 0; w < BAL_THREADS / 32; ++w) s += red[w];   // fixed order: deterministic
  __syncthreads();
  return s;
}

__global__ void __launch_bounds__(BAL_THREADS) balance_update_kernel(const int32_t* __restrict__ counts, int E,
                                                                     float* __restrict__ bias, float gamma,
                                                                     float* __restrict__ stats, int* status) {
  // the only kernel of its call: dependents start after it has begun, and it
  // reads the counts only once the kernels before it have completed
  pdl_wait();
  pdl_launch_dependents();
  __shared__ double red[BAL_THREADS / 32];
  __shared__ int imax[BAL_THREADS / 32], imin[BAL_THREADS / 32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  int c = e < E ? counts[e] : 0;
  if (c < 0) {
    flag_status(status, DEV_BAD_ROW);
    c = 0;
  }
  const double total = block_sum_f64(double(c), red);
  if (e < E) {
    const double lhs = double(c) * E;   // exact: counts and E are small integers
    float b = bias[e];
    if (lhs > total) b = b - gamma;
    else if (lhs < total) b = b + gamma;
    bias[e] = b;
  }
  if (stats == nullptr) return;
  // load fractions and their unbiased standard deviation (mean fraction = 1/E)
  const double load = (e < E && total > 0.0) ? double(c) / total : 0.0;
  const double dev = e < E ? load - (total > 0.0 ? 1.0 / E : 0.0) : 0.0;
  const double ss = block_sum_f64(dev * dev, red);
  int mx = e < E ? c : INT_MIN, mn = e < E ? c : INT_MAX;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  if (lane == 0) {
    imax[warp] = mx;
    imin[warp] = mn;
  }
  __syncthreads();
  if (e == 0) {
    for (int w = 1; w < BAL_THREADS / 32; ++w) {
      mx = max(mx, imax[w]);
      mn = min(mn, imin[w]);
    }
    mx = max(mx, imax[0]);
    mn = min(mn, imin[0]);
    stats[0] = E > 1 ? float(sqrt(ss / (E - 1))) : 0.0f;
    stats[1] = total > 0.0 ? float(double(mx) * E / total) : 0.0f;
    stats[2] = total > 0.0 ? float(double(mn) * E / total) : 0.0f;
  }
}

}  // namespace

cudaError_t launch_balance_update(const moe_config& c, const int32_t* counts, float* bias, float gamma, float* stats,
                                  int* status, cudaStream_t s, int* launches) {
  cudaError_t e = launch_pdl(balance_update_kernel, dim3(1), dim3(BAL_THREADS), 0, s, counts, c.E, bias, gamma, stats,
                             status);
  if (launches) ++*launches;
  return e;
}

}  // namespace moe
