// Backward of the MoE layer: gradients of <dout, out> with respect to x, W_g
// and every expert weight, with the forward's expert choice held fixed.
//
// The chain rule through the layer (DeepSeek-V2 walkthrough, MoE listing; the
// SwiGLU of intelliparadigm.com section 3.3.1; the gate of the V3 page section
// 1.2):
//   dg[t,j]  = <dout_t, y_{idx[t,j]}(x_t)>           (gate-weighted sum)
//   dy rows  = g[t,j] * dout_t                       (per routed row)
//   dH = dY W2,  dW2 = dY^T H,  H = silu(G) * U, G = X W1^T, U = X W3^T
//   dG = dH * U * silu'(G),  dU = dH * silu(G)
//   dX = dG W1 + dU W3,  dW1 = dG^T X,  dW3 = dU^T X
//   gates -> affinities (renormalisation, scale) -> logits (sigmoid, or
//   softmax over all experts) -> dW_g = dl^T x, dx += dl W_g
// The expert and gate GEMMs are plain per-expert matrix products and run in
// cuBLAS (bf16 operands, fp32 accumulation and outputs); every other step is a
// kernel here.  Group sizes are read back to the host, so a backward call
// synchronises its stream once.
#include <cublas_v2.h>
#include <cuda_bf16.h>

#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// out32 = float(src), out16 = bf16(src) (either output may be null)
template <typename T>
__global__ void convert_kernel(const T* __restrict__ src, long long n, float* __restrict__ out32,
                               __nv_bfloat16* __restrict__ out16) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float v = to_f(src[i]);
    if (out32) out32[i] = v;
    if (out16) out16[i] = __float2bfloat16_rn(v);
  }
}

// H = bf16(silu(G) * U) (the forward's GEMM1 epilogue, from fp32 accumulators)
__global__ void silu_mul_kernel(const float* __restrict__ G, const float* __restrict__ U, long long n,
                                __nv_bfloat16* __restrict__ H) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float g = G[i];
    H[i] = __float2bfloat16_rn(g * sigmoid_f(g) * U[i]);
  }
}

// dG = dH * U * silu'(G), dU = dH * silu(G); silu'(g) = s (1 + g (1 - s)), s = sigmoid(g)
__global__ void swiglu_bwd_kernel(const float* __restrict__ G, const float* __restrict__ U,
                                  const float* __restrict__ dH, long long n, __nv_bfloat16* __restrict__ dG,
                                  __nv_bfloat16* __restrict__ dU) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float g = G[i], sg = sigmoid_f(g), dh = dH[i];
    dG[i] = __float2bfloat16_rn(dh * U[i] * sg * (1.0f + g * (1.0f - sg)));
    dU[i] = __float2bfloat16_rn(dh * g * sg);
  }
}

// One warp per routed row r (token t, slot j): dY[r] = bf16(g[t,j] * dout[t])
// and dg[t,j] = <dout[t], Y[r]> (fp32, lane-strided then a fixed butterfly).
__global__ void gate_rows_kernel(const float* __restrict__ dout, const float* __restrict__ Y,
                                 const int32_t* __restrict__ row2tok, const int32_t* __restrict__ tok2row,
                                 const float* __restrict__ gates, int R, int k, int d,
                                 __nv_bfloat16* __restrict__ dY, float* __restrict__ dg) {
  const int lane = threadIdx.x & 31;
  const long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long r = warp; r < R; r += nwarps) {
    const int t = row2tok[r];
    int j = 0;
    for (int q = 0; q < k; ++q)
      if (tok2row[(long long)t * k + q] == r) j = q;
    const float gv = gates[(long long)t * k + j];
    const float* dr = dout + (long long)t * d;
    const float* yr = Y + r * (long long)d;
    __nv_bfloat16* o = dY + r * (long long)d;
    float acc = 0.0f;
    for (int c = lane; c < d; c += 32) {
      const float v = dr[c];
      o[c] = __float2bfloat16_rn(gv * v);
      acc = fmaf(v, yr[c], acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) dg[(long long)t * k + j] = acc;
  }
}

// dx[t] = sum over slots j (in order) of dXr[tok2row[t,j]] + dXs[t] (dXs may be null)
__global__ void scatter_rows_kernel(const float* __restrict__ dXr, const float* __restrict__ dXs,
                                    const int32_t* __restrict__ tok2row, int T, int k, int d, float* __restrict__ dx) {
  const long long n = (long long)T * d;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long t = i / d, c = i - t * d;
    float v = 0.0f;
    for (int j = 0; j < k; ++j) v += dXr[(long long)tok2row[t * k + j] * d + c];
    if (dXs) v += dXs[i];
    dx[i] = v;
  }
}

struct GateBwdArgs {
  int T, E, k, score_fn, norm;
  float scale;
};

// One warp per token: d logits [E] from dg [k] through the gate values
// (c * raw / sum(raw), or c * raw; raw = the chosen experts' affinities) and
// the affinities (sigmoid, or softmax over all experts).
__global__ void gate_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                                const float* __restrict__ dg, GateBwdArgs a, float* __restrict__ dl) {
  const int lane = threadIdx.x & 31;
  const long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long t = warp; t < a.T; t += nwarps) {
    const float* lr = logits + t * a.E;
    float* out = dl + t * a.E;
    // softmax normaliser (max-shifted)
    float m = -INFINITY;
    if (a.score_fn == MOE_SCORE_SOFTMAX) {
      for (int e = lane; e < a.E; e += 32) m = fmaxf(m, lr[e]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    }
    float z = 0.0f;
    if (a.score_fn == MOE_SCORE_SOFTMAX) {
      for (int e = lane; e < a.E; e += 32) z += expf(lr[e] - m);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    }
    auto score = [&](int e) {
      return a.score_fn == MOE_SCORE_SOFTMAX ? expf(lr[e] - m) / z : sigmoid_f(lr[e]);
    };
    // raw affinities of the choice, their sum and the sum of dg * raw
    float rsum = 0.0f, dgr = 0.0f;
    for (int j = 0; j < a.k; ++j) {
      const float rj = score(idx[t * a.k + j]);
      rsum += rj;
      dgr += dg[t * a.k + j] * rj;
    }
    // ds at the chosen experts; <ds, s> for the softmax Jacobian
    float dss = 0.0f;
    for (int j = 0; j < a.k; ++j) {
      const int e = idx[t * a.k + j];
      const float g = dg[t * a.k + j];
      const float dr = a.norm ? a.scale * (g / rsum - dgr / (rsum * rsum)) : a.scale * g;
      dss += dr * score(e);
    }
    for (int e = lane; e < a.E; e += 32) {
      float ds = 0.0f;
      for (int j = 0; j < a.k; ++j) {
        if (idx[t * a.k + j] == e) {
          const float g = dg[t * a.k + j];
          ds = a.norm ? a.scale * (g / rsum - dgr / (rsum * rsum)) : a.scale * g;
        }
      }
      const float s = score(e);
      out[e] = a.score_fn == MOE_SCORE_SOFTMAX ? s * (ds - dss) : ds * s * (1.0f - s);
    }
  }
}

int grid_for(long long n) {
  const long long b = (n + 255) / 256;
  return int(b < 8LL * num_sms() ? (b > 0 ? b : 1) : 8LL * num_sms());
}

cublasHandle_t blas() {
  static cublasHandle_t h = nullptr;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (h == nullptr && cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) h = nullptr;
  return h;
}

// Row-major C[m,n] (fp32) = op(A) op(B) + beta C, A and B of type `ty` stored
// row-major (op = transpose when ta / tb), fp32 accumulation.  cuBLAS works
// column-major, so it computes C^T = op(B)^T op(A)^T on the same memory.
bool gemm_rm(cublasHandle_t h, bool ta, bool tb, int m, int n, int k, const void* A, int lda, const void* B,
             int ldb, float* C, int ldc, float beta, cudaDataType ty) {
  if (m == 0 || n == 0) return true;
  const float alpha = 1.0f;
  return cublasGemmEx(h, tb ? CUBLAS_OP_T : CUBLAS_OP_N, ta ? CUBLAS_OP_T : CUBLAS_OP_N, n, m, k, &alpha, B, ty, ldb,
                      A, ty, lda, &beta, C, CUDA_R_32F, ldc, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) ==
         CUBLAS_STATUS_SUCCESS;
}

}  // namespace

size_t backward_extra_bytes(const moe_config& c) {
  const BwdLayout L = backward_layout(c, 0);
  return L.total;
}

BwdLayout backward_layout(const moe_config& c, size_t base) {
  BwdLayout L;
  const size_t R = size_t(c.T) * c.k, T = size_t(c.T), d = size_t(c.d), I = size_t(c.I),
               Is = size_t(c.n_shared) * c.I, E = size_t(c.E);
  size_t off = base;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.G = take(R * I * 4);
  L.U = take(R * I * 4);
  L.Hb = take(R * I * 2);
  L.dYb = take(R * d * 2);
  L.dH = take(R * I * 4);
  L.dGb = take(R * I * 2);
  L.dUb = take(R * I * 2);
  L.dXr = take(R * d * 4);
  L.Gs = take(T * Is * 4);
  L.Us = take(T * Is * 4);
  L.Hsb = take(T * Is * 2);
  L.dHs = take(T * Is * 4);
  L.dGsb = take(T * Is * 2);
  L.dUsb = take(T * Is * 2);
  L.dXs = take(T * d * 4);
  L.dout32 = take(T * d * 4);
  L.doutb = take(T * d * 2);
  L.x32 = take(T * d * 4);
  L.wg32 = take(E * d * 4);
  L.logits = take(T * E * 4);
  L.dl = take(T * E * 4);
  L.dg = take(R * 4);
  L.total = off - base;
  return L;
}

cudaError_t run_backward_core(const moe_config& c, const BwdPtrs& p, cudaStream_t s) {
  cublasHandle_t h = blas();
  if (h == nullptr || cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  const int T = c.T, d = c.d, I = c.I, E = c.E, k = c.k;
  const int Is = c.n_shared * c.I;
  const long long R = (long long)T * k;
  const cudaDataType BF = CUDA_R_16BF;
  cudaError_t e;
  auto ok = [&]() { return (e = cudaGetLastError()) == cudaSuccess; };

  // group sizes on the host (offsets come from the dispatch on this stream)
  std::vector<int32_t> off(E + 1);
  if ((e = cudaMemcpyAsync(off.data(), p.offsets, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToHost, s)) !=
      cudaSuccess)
    return e;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
  for (int g = 0; g < E; ++g)
    if (off[g] < 0 || off[g + 1] < off[g] || off[g + 1] > R) return cudaErrorInvalidValue;

  // upstream gradient as fp32 and bf16
  if (c.out_dtype == MOE_BF16)
    convert_kernel<<<grid_for((long long)T * d), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(p.dout),
                                                               (long long)T * d, p.dout32, p.doutb);
  else
    convert_kernel<<<grid_for((long long)T * d), 256, 0, s>>>(static_cast<const float*>(p.dout), (long long)T * d,
                                                               p.dout32, p.doutb);
  if (!ok()) return e;

  // forward recomputation of the routed experts: G, U, H, Y
  const auto* W1 = static_cast<const __nv_bfloat16*>(p.W1);
  const auto* W3 = static_cast<const __nv_bfloat16*>(p.W3);
  const auto* W2 = static_cast<const __nv_bfloat16*>(p.W2);
  const auto* X = static_cast<const __nv_bfloat16*>(p.x_perm);
  for (int g = 0; g < E; ++g) {
    const int o = off[g], n = off[g + 1] - off[g];
    if (n == 0) continue;
    const auto* w1 = W1 + (size_t)g * I * d;
    const auto* w3 = W3 + (size_t)g * I * d;
    if (!gemm_rm(h, false, true, n, I, d, X + (size_t)o * d, d, w1, d, p.G + (size_t)o * I, I, 0.0f, BF) ||
        !gemm_rm(h, false, true, n, I, d, X + (size_t)o * d, d, w3, d, p.U + (size_t)o * I, I, 0.0f, BF))
      return cudaErrorUnknown;
  }
  silu_mul_kernel<<<grid_for(R * I), 256, 0, s>>>(p.G, p.U, R * I, p.Hb);
  if (!ok()) return e;
  for (int g = 0; g < E; ++g) {
    const int o = off[g], n = off[g + 1] - off[g];
    if (n == 0) continue;
    if (!gemm_rm(h, false, true, n, d, I, p.Hb + (size_t)o * I, I, W2 + (size_t)g * d * I, I, p.Y + (size_t)o * d, d,
                 0.0f, BF))
      return cudaErrorUnknown;
  }
  // dY rows and dg
  gate_rows_kernel<<<grid_for(R * 32), 256, 0, s>>>(p.dout32, p.Y, p.row2tok, p.tok2row, p.gates, int(R), k, d, p.dYb,
                                                    p.dg);
  if (!ok()) return e;
  // GEMM2 backward, SwiGLU backward, GEMM1 backward
  for (int g = 0; g < E; ++g) {
    const int o = off[g], n = off[g + 1] - off[g];
    float* dw2 = p.dW2 + (size_t)g * d * I;
    if (n == 0) {
      if ((e = cudaMemsetAsync(dw2, 0, sizeof(float) * d * I, s)) != cudaSuccess) return e;
      continue;
    }
    const auto* w2 = W2 + (size_t)g * d * I;
    if (!gemm_rm(h, false, false, n, I, d, p.dYb + (size_t)o * d, d, w2, I, p.dH + (size_t)o * I, I, 0.0f, BF) ||
        !gemm_rm(h, true, false, d, I, n, p.dYb + (size_t)o * d, d, p.Hb + (size_t)o * I, I, dw2, I, 0.0f, BF))
      return cudaErrorUnknown;
  }
  swiglu_bwd_kernel<<<grid_for(R * I), 256, 0, s>>>(p.G, p.U, p.dH, R * I, p.dGb, p.dUb);
  if (!ok()) return e;
  for (int g = 0; g < E; ++g) {
    const int o = off[g], n = off[g + 1] - off[g];
    float* dw1 = p.dW1 + (size_t)g * I * d;
    float* dw3 = p.dW3 + (size_t)g * I * d;
    if (n == 0) {
      if ((e = cudaMemsetAsync(dw1, 0, sizeof(float) * I * d, s)) != cudaSuccess) return e;
      if ((e = cudaMemsetAsync(dw3, 0, sizeof(float) * I * d, s)) != cudaSuccess) return e;
      continue;
    }
    const auto* w1 = W1 + (size_t)g * I * d;
    const auto* w3 = W3 + (size_t)g * I * d;
    float* dx = p.dXr + (size_t)o * d;
    if (!gemm_rm(h, false, false, n, d, I, p.dGb + (size_t)o * I, I, w1, d, dx, d, 0.0f, BF) ||
        !gemm_rm(h, false, false, n, d, I, p.dUb + (size_t)o * I, I, w3, d, dx, d, 1.0f, BF) ||
        !gemm_rm(h, true, false, I, d, n, p.dGb + (size_t)o * I, I, X + (size_t)o * d, d, dw1, d, 0.0f, BF) ||
        !gemm_rm(h, true, false, I, d, n, p.dUb + (size_t)o * I, I, X + (size_t)o * d, d, dw3, d, 0.0f, BF))
      return cudaErrorUnknown;
  }

  // shared expert (every token, gate 1)
  if (Is > 0) {
    const auto* x16 = static_cast<const __nv_bfloat16*>(p.x);
    const auto* ws1 = static_cast<const __nv_bfloat16*>(p.Ws1);
    const auto* ws3 = static_cast<const __nv_bfloat16*>(p.Ws3);
    const auto* ws2 = static_cast<const __nv_bfloat16*>(p.Ws2);
    if (!gemm_rm(h, false, true, T, Is, d, x16, d, ws1, d, p.Gs, Is, 0.0f, BF) ||
        !gemm_rm(h, false, true, T, Is, d, x16, d, ws3, d, p.Us, Is, 0.0f, BF))
      return cudaErrorUnknown;
    silu_mul_kernel<<<grid_for((long long)T * Is), 256, 0, s>>>(p.Gs, p.Us, (long long)T * Is, p.Hsb);
    if (!ok()) return e;
    if (!gemm_rm(h, false, false, T, Is, d, p.doutb, d, ws2, Is, p.dHs, Is, 0.0f, BF) ||
        !gemm_rm(h, true, false, d, Is, T, p.doutb, d, p.Hsb, Is, p.dWs2, Is, 0.0f, BF))
      return cudaErrorUnknown;
    swiglu_bwd_kernel<<<grid_for((long long)T * Is), 256, 0, s>>>(p.Gs, p.Us, p.dHs, (long long)T * Is, p.dGsb,
                                                                   p.dUsb);
    if (!ok()) return e;
    if (!gemm_rm(h, false, false, T, d, Is, p.dGsb, Is, ws1, d, p.dXs, d, 0.0f, BF) ||
        !gemm_rm(h, false, false, T, d, Is, p.dUsb, Is, ws3, d, p.dXs, d, 1.0f, BF) ||
        !gemm_rm(h, true, false, Is, d, T, p.dGsb, Is, x16, d, p.dWs1, d, 0.0f, BF) ||
        !gemm_rm(h, true, false, Is, d, T, p.dUsb, Is, x16, d, p.dWs3, d, 0.0f, BF))
      return cudaErrorUnknown;
  }
  scatter_rows_kernel<<<grid_for((long long)T * d), 256, 0, s>>>(p.dXr, Is > 0 ? p.dXs : nullptr, p.tok2row, T, k,
                                                                  d, p.dx);
  if (!ok()) return e;

  // router: fp32 logits, d logits, dW_g, and dx += dl W_g
  convert_kernel<<<grid_for((long long)T * d), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(p.x), (long long)T * d,
                                                             p.x32, nullptr);
  if (!ok()) return e;
  if (c.gate_w_dtype == MOE_BF16)
    convert_kernel<<<grid_for((long long)E * d), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(p.Wg),
                                                               (long long)E * d, p.wg32, nullptr);
  else
    convert_kernel<<<grid_for((long long)E * d), 256, 0, s>>>(static_cast<const float*>(p.Wg), (long long)E * d,
                                                               p.wg32, nullptr);
  if (!ok()) return e;
  const cudaDataType F = CUDA_R_32F;
  if (!gemm_rm(h, false, true, T, E, d, p.x32, d, p.wg32, d, p.logits, E, 0.0f, F)) return cudaErrorUnknown;
  GateBwdArgs a;
  a.T = T;
  a.E = E;
  a.k = k;
  a.score_fn = c.score_fn;
  a.norm = c.norm_topk;
  a.scale = c.routed_scaling_factor;
  gate_bwd_kernel<<<grid_for((long long)T * 32), 256, 0, s>>>(p.logits, p.idx, p.dg, a, p.dl);
  if (!ok()) return e;
  if (!gemm_rm(h, true, false, E, d, T, p.dl, E, p.x32, d, p.dWg, d, 0.0f, F) ||
      !gemm_rm(h, false, false, T, d, E, p.dl, E, p.wg32, d, p.dx, d, 1.0f, F))
    return cudaErrorUnknown;
  return cudaGetLastError();
}

}  // namespace moe
