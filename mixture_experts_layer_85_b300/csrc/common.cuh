// Shared device/host helpers of the MoE library (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Bits of the device status word (first int32 of the workspace).
enum DevStatusBits : int {
  DEV_TIMEOUT = 1,       // a bounded mbarrier wait gave up
  DEV_BAD_EXPERT = 2,    // an expert index outside [0,E)
  DEV_BAD_ROW = 4,       // a row index outside its buffer
  DEV_RANGE = 8,         // FP8 layer: an activation beyond the f16 range of its operands
};

// Wait limit of every device-side spin (ns of %globaltimer).  A legitimate
// wait in these kernels lasts microseconds; two seconds means a broken pipeline.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch.  Every kernel of the layer lets the next
// kernel of the stream begin launching as soon as all of its own CTAs are
// running, and waits for its predecessor grid to complete (with its memory
// visible) before it reads that grid's outputs or writes anything the
// predecessor might still read.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void flag_status(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// (value, index) arg-max over the warp; equal values go to the lower index.
__device__ __forceinline__ void warp_argmax(float& v, int& id) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oid = __shfl_xor_sync(0xffffffffu, id, o);
    if (ov > v || (ov == v && oid < id)) { v = ov; id = oid; }
  }
}

template <typename T> struct ElemTraits;
template <> struct ElemTraits<float> {
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct ElemTraits<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// Host-side launch accounting (moe_launch_count).
void count_launches(int n);

}  // namespace moe
