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
// Every matrix product runs on this library's CTA-pair tensor-core kernel
// (bf16 operands, fp32 accumulation and outputs), the weights read in place
// through transposed (MN-major) views where a product needs W^T.  The routed
// rows use a padded layout: expert g's rows start at koff[g], a multiple of
// 128, and its pad rows are zero, so a weight gradient reduces over whole
// 128-row stages of its own rows.  Group sizes stay on the device: no host
// synchronisation.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int KPAD = 128;   // rows of one reduction stage of the expert kernel

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

// One block: koff[g] = sum over g' < g of n_g' rounded up to KPAD (the padded
// layout), then tok2row_pad[t][j] = koff[g] + (tok2row[t][j] - offsets[g]) with
// g = idx[t][j] (-1 for a skipped slot).
__global__ void __launch_bounds__(1024) pad_rows_kernel(const int32_t* __restrict__ offsets,
                                                        const int32_t* __restrict__ idx,
                                                        const int32_t* __restrict__ tok2row, int E, long long R,
                                                        int32_t* __restrict__ koff, int32_t* __restrict__ tok2row_pad,
                                                        int* status) {
  __shared__ int32_t base[257];
  if (threadIdx.x == 0) {
    int run = 0;
    for (int g = 0; g < E; ++g) {
      base[g] = run;
      const int n = offsets[g + 1] - offsets[g];
      run += (n + KPAD - 1) / KPAD * KPAD;
    }
    base[E] = run;
  }
  __syncthreads();
  for (int g = threadIdx.x; g <= E; g += blockDim.x) koff[g] = base[g];
  for (long long i = threadIdx.x; i < R; i += blockDim.x) {
    const int g = idx[i];
    const int r = tok2row[i];
    if (g < 0 || g >= E || r < 0) {
      tok2row_pad[i] = -1;
      if (r >= 0) flag_status(status, DEV_BAD_EXPERT);
      continue;
    }
    tok2row_pad[i] = base[g] + (r - offsets[g]);
  }
}

// Zeroes the pad rows koff[g] + n_g .. koff[g+1] of every group g (one block
// per group) of a [rows, row_vec * 16 B] buffer.
__global__ void zero_pad_rows_kernel(uint4* __restrict__ buf, int row_vec, const int32_t* __restrict__ koff,
                                     const int32_t* __restrict__ offsets) {
  const int g = blockIdx.x;
  const long long r0 = (long long)koff[g] + (offsets[g + 1] - offsets[g]);
  const long long n = ((long long)koff[g + 1] - r0) * row_vec;
  uint4* p = buf + r0 * row_vec;
  for (long long i = threadIdx.x; i < n; i += blockDim.x) p[i] = make_uint4(0u, 0u, 0u, 0u);
}

// H = bf16(silu(G) * U) (the forward's GEMM1 epilogue, from fp32 accumulators)
__global__ void silu_mul_kernel(const float* __restrict__ G, const float* __restrict__ U, long long n,
                                __nv_bfloat16* __restrict__ H) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float g = G[i];
    H[i] = __float2bfloat16_rn(g * sigmoid_f(g) * U[i]);
  }
}

// dG = dH * U * silu'(G), dU = dH * silu(G) (silu'(g) = s (1 + g (1 - s)),
// s = sigmoid(g)), stored side by side: dGU[r][i] = dG, dGU[r][h + i] = dU.
__global__ void swiglu_bwd_kernel(const float* __restrict__ G, const float* __restrict__ U,
                                  const float* __restrict__ dH, long long rows, int h, __nv_bfloat16* __restrict__ dGU) {
  const long long n = rows * h;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / h, c = i - r * h;
    const float g = G[i], sg = sigmoid_f(g), dh = dH[i];
    dGU[r * 2 * h + c] = __float2bfloat16_rn(dh * U[i] * sg * (1.0f + g * (1.0f - sg)));
    dGU[r * 2 * h + h + c] = __float2bfloat16_rn(dh * g * sg);
  }
}

// One warp per (token t, slot j), row r = tok2row_pad[t][j]: dY[r] =
// bf16(g[t,j] * dout[t]) and dg[t,j] = <dout[t], Y[r]> (fp32, lane-strided
// then a fixed butterfly).
__global__ void gate_rows_kernel(const float* __restrict__ dout, const float* __restrict__ Y,
                                 const int32_t* __restrict__ tok2row_pad, const float* __restrict__ gates, long long R,
                                 int k, int d, __nv_bfloat16* __restrict__ dY, float* __restrict__ dg) {
  const int lane = threadIdx.x & 31;
  const long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long i = warp; i < R; i += nwarps) {
    const long long r = tok2row_pad[i];
    if (r < 0) {
      if (lane == 0) dg[i] = 0.0f;
      continue;
    }
    const long long t = i / k;
    const float gv = gates[i];
    const float* dr = dout + t * d;
    const float* yr = Y + r * d;
    __nv_bfloat16* o = dY + r * d;
    float acc = 0.0f;
    for (int c = lane; c < d; c += 32) {
      const float v = dr[c];
      o[c] = __float2bfloat16_rn(gv * v);
      acc = fmaf(v, yr[c], acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) dg[i] = acc;
  }
}

// dx[t] = sum over slots j (in order) of dXr[tok2row_pad[t,j]] + dXs[t] + dXg[t]
// (dXs may be null).
__global__ void scatter_rows_kernel(const float* __restrict__ dXr, const float* __restrict__ dXs,
                                    const float* __restrict__ dXg, const int32_t* __restrict__ tok2row_pad, int T,
                                    int k, int d, float* __restrict__ dx) {
  const long long n = (long long)T * d;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long t = i / d, c = i - t * d;
    float v = 0.0f;
    for (int j = 0; j < k; ++j) {
      const long long r = tok2row_pad[t * k + j];
      if (r >= 0) v += dXr[r * d + c];
    }
    if (dXs) v += dXs[i];
    dx[i] = v + dXg[i];
  }
}

struct GateBwdArgs {
  int T, E, k, score_fn, norm, nsplit, e_pad;
  long long plane;
  float scale;
};

// One warp per token: d logits [E] from dg [k] through the gate values
// (c * raw / sum(raw), or c * raw; raw = the chosen experts' affinities) and
// the affinities (sigmoid, or softmax over all experts).  The logits are the
// forward router's: `nsplit` fp32 planes added in order.  Output: bf16 rows of
// e_pad columns, zero past E.
__global__ void gate_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                                const float* __restrict__ dg, GateBwdArgs a, __nv_bfloat16* __restrict__ dl) {
  const int lane = threadIdx.x & 31;
  const long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long t = warp; t < a.T; t += nwarps) {
    auto logit = [&](int e) {
      float v = 0.0f;
      for (int q = 0; q < a.nsplit; ++q) v += logits[q * a.plane + t * a.E + e];
      return v;
    };
    __nv_bfloat16* out = dl + t * a.e_pad;
    float m = -INFINITY;
    if (a.score_fn == MOE_SCORE_SOFTMAX) {
      for (int e = lane; e < a.E; e += 32) m = fmaxf(m, logit(e));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    }
    float z = 0.0f;
    if (a.score_fn == MOE_SCORE_SOFTMAX) {
      for (int e = lane; e < a.E; e += 32) z += expf(logit(e) - m);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    }
    auto score = [&](int e) {
      return a.score_fn == MOE_SCORE_SOFTMAX ? expf(logit(e) - m) / z : sigmoid_f(logit(e));
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
    for (int e = lane; e < a.e_pad; e += 32) {
      if (e >= a.E) {
        out[e] = __float2bfloat16_rn(0.0f);
        continue;
      }
      float ds = 0.0f;
      for (int j = 0; j < a.k; ++j) {
        if (idx[t * a.k + j] == e) {
          const float g = dg[t * a.k + j];
          ds = a.norm ? a.scale * (g / rsum - dgr / (rsum * rsum)) : a.scale * g;
        }
      }
      const float s = score(e);
      out[e] = __float2bfloat16_rn(a.score_fn == MOE_SCORE_SOFTMAX ? s * (ds - dss) : ds * s * (1.0f - s));
    }
  }
}

int grid_for(long long n) {
  const long long b = (n + 255) / 256;
  return int(b < 8LL * num_sms() ? (b > 0 ? b : 1) : 8LL * num_sms());
}

// Upper bound of the expert kernel's tiles (only sizes its grid).
constexpr long long kManyTiles = 1LL << 30;

}  // namespace

BwdLayout backward_layout(const moe_config& c, size_t base) {
  BwdLayout L;
  const size_t T = size_t(c.T), d = size_t(c.d), I = size_t(c.I), Is = size_t(c.n_shared) * c.I, E = size_t(c.E);
  L.R_max = (long long)c.T * c.k + (long long)(KPAD - 1) * c.E;
  L.E_pad = (c.E + KPAD - 1) / KPAD * KPAD;
  const size_t R = size_t(L.R_max);
  size_t off = base;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.koff = take((E + 1) * 4);
  L.tok2row_pad = take(T * c.k * 4);
  L.Xp = take(R * d * 2);
  L.G = take(R * I * 4);
  L.U = take(R * I * 4);
  L.H = take(R * I * 2);
  L.Y = take(R * d * 4);   // expert output rows; later the rows of dx
  L.dY = take(R * d * 2);
  L.dH = take(R * I * 4);
  L.dGU = take(R * 2 * I * 2);
  L.Gs = take(T * Is * 4);
  L.Us = take(T * Is * 4);
  L.Hs = take(T * Is * 2);
  L.dHs = take(T * Is * 4);
  L.dGUs = take(T * 2 * Is * 2);
  L.dXs = take(T * d * 4);
  L.doutb = take(T * d * 2);
  L.dout32 = take(T * d * 4);
  L.dlb = take(T * size_t(L.E_pad) * 2);
  L.dg = take(T * c.k * 4);
  L.dXg = take(T * d * 4);
  L.wgb = take(E * d * 2);
  L.total = off - base;
  return L;
}

size_t backward_extra_bytes(const moe_config& c) { return backward_layout(c, 0).total; }

cudaError_t run_backward_core(const moe_config& c, const BwdPtrs& p, const BwdLayout& L, cudaStream_t s) {
  const int T = c.T, d = c.d, I = c.I, E = c.E, k = c.k;
  const int Is = c.n_shared * c.I;
  const long long R = (long long)T * k, Rm = L.R_max;
  const int T_pad = (T + KPAD - 1) / KPAD * KPAD;
  char* b = p.base;
  auto at = [&](size_t o) { return static_cast<void*>(b + o); };
  int32_t* koff = static_cast<int32_t*>(at(L.koff));
  int32_t* t2r = static_cast<int32_t*>(at(L.tok2row_pad));
  auto* Xp = static_cast<__nv_bfloat16*>(at(L.Xp));
  float* G = static_cast<float*>(at(L.G));
  float* U = static_cast<float*>(at(L.U));
  auto* H = static_cast<__nv_bfloat16*>(at(L.H));
  float* Y = static_cast<float*>(at(L.Y));
  float* dXr = Y;   // Y is dead once dY and dg are formed
  auto* dY = static_cast<__nv_bfloat16*>(at(L.dY));
  float* dH = static_cast<float*>(at(L.dH));
  auto* dGU = static_cast<__nv_bfloat16*>(at(L.dGU));
  float* Gs = static_cast<float*>(at(L.Gs));
  float* Us = static_cast<float*>(at(L.Us));
  auto* Hs = static_cast<__nv_bfloat16*>(at(L.Hs));
  float* dHs = static_cast<float*>(at(L.dHs));
  auto* dGUs = static_cast<__nv_bfloat16*>(at(L.dGUs));
  float* dXs = static_cast<float*>(at(L.dXs));
  auto* doutb = static_cast<__nv_bfloat16*>(at(L.doutb));
  float* dout32 = static_cast<float*>(at(L.dout32));
  auto* dlb = static_cast<__nv_bfloat16*>(at(L.dlb));
  float* dg = static_cast<float*>(at(L.dg));
  float* dXg = static_cast<float*>(at(L.dXg));
  auto* wgb = static_cast<__nv_bfloat16*>(at(L.wgb));
  const bool shared = Is > 0;
  cudaError_t e;
  int n = 0;
  struct CountOnExit {
    int* n;
    ~CountOnExit() { count_launches(*n); }
  } count_on_exit{&n};
  int* ticket = p.tickets;
  auto next_ticket = [&]() { return ticket++; };
  // after each plain launch: count it and check it was accepted
  auto ok = [&]() {
    ++n;
    return (e = cudaGetLastError()) == cudaSuccess;
  };
  auto zero_pads = [&](void* buf, size_t row_bytes) {
    zero_pad_rows_kernel<<<E, 256, 0, s>>>(static_cast<uint4*>(buf), int(row_bytes / 16), koff, p.offsets);
    return ok();
  };

  // padded layout of the routed rows, and the tokens gathered into it
  pad_rows_kernel<<<1, 1024, 0, s>>>(p.offsets, p.idx, p.tok2row, E, R, koff, t2r, p.status);
  if (!ok()) return e;
  if ((e = launch_gather_rows(p.x, t2r, T, k, Rm, size_t(d) * 2, Xp, p.status, s, &n)) != cudaSuccess) return e;
  if (!zero_pads(Xp, size_t(d) * 2)) return e;
  // upstream gradient as fp32 and bf16; the gate weight as bf16
  if (c.out_dtype == MOE_BF16)
    convert_kernel<<<grid_for((long long)T * d), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(p.dout),
                                                               (long long)T * d, dout32, doutb);
  else
    convert_kernel<<<grid_for((long long)T * d), 256, 0, s>>>(static_cast<const float*>(p.dout), (long long)T * d,
                                                               dout32, doutb);
  if (!ok()) return e;
  if (c.gate_w_dtype == MOE_BF16)
    convert_kernel<<<grid_for((long long)E * d), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(p.Wg),
                                                               (long long)E * d, nullptr, wgb);
  else
    convert_kernel<<<grid_for((long long)E * d), 256, 0, s>>>(static_cast<const float*>(p.Wg), (long long)E * d,
                                                               nullptr, wgb);
  if (!ok()) return e;

  // ---- forward recomputation: G = X W1^T, U = X W3^T (routed rows and shared), H, Y = H W2^T
  PairOperands r, sh;
  for (int which = 0; which < 2; ++which) {
    r = PairOperands();
    r.A = which == 0 ? p.W1 : p.W3; r.a_rows = (long long)E * I; r.a_cols = d; r.w_step = I;
    r.B = Xp; r.b_rows = Rm; r.b_cols = d;
    r.M = I; r.K = d; r.out = which == 0 ? G : U; r.ld_out = I; r.out_rows = Rm;
    sh = PairOperands();
    sh.A = which == 0 ? p.Ws1 : p.Ws3; sh.a_rows = Is; sh.a_cols = d;
    sh.B = p.x; sh.b_rows = T; sh.b_cols = d;
    sh.M = Is; sh.K = d; sh.out = which == 0 ? Gs : Us; sh.ld_out = Is; sh.out_rows = T;
    if ((e = launch_pair_gemm(&r, shared ? &sh : nullptr, p.offsets, koff, Rm, E, shared ? T : 0, 0, next_ticket(),
                              p.status, kManyTiles, s, &n)) != cudaSuccess)
      return e;
  }
  silu_mul_kernel<<<grid_for(Rm * I), 256, 0, s>>>(G, U, Rm * I, H);
  if (!ok() || !zero_pads(H, size_t(I) * 2)) return e;   // (counts both launches)
  if (shared) {
    silu_mul_kernel<<<grid_for((long long)T * Is), 256, 0, s>>>(Gs, Us, (long long)T * Is, Hs);
    if (!ok()) return e;
  }
  r = PairOperands();
  r.A = p.W2; r.a_rows = (long long)E * d; r.a_cols = I; r.w_step = d;
  r.B = H; r.b_rows = Rm; r.b_cols = I;
  r.M = d; r.K = I; r.out = Y; r.ld_out = d; r.out_rows = Rm;
  if ((e = launch_pair_gemm(&r, nullptr, p.offsets, koff, Rm, E, 0, 0, next_ticket(), p.status, kManyTiles, s, &n)) !=
      cudaSuccess)
    return e;

  // ---- dY rows and dg, then dH = dY W2 (W2^T read transposed), SwiGLU backward
  gate_rows_kernel<<<grid_for(R * 32), 256, 0, s>>>(dout32, Y, t2r, p.gates, R, k, d, dY, dg);
  if (!ok() || !zero_pads(dY, size_t(d) * 2)) return e;
  r = PairOperands();
  r.A = p.W2; r.a_mn = true; r.a_rows = (long long)E * d; r.a_cols = I; r.a_kstep = d;
  r.B = dY; r.b_rows = Rm; r.b_cols = d;
  r.M = I; r.K = d; r.out = dH; r.ld_out = I; r.out_rows = Rm;
  sh = PairOperands();
  sh.A = p.Ws2; sh.a_mn = true; sh.a_rows = d; sh.a_cols = Is;
  sh.B = doutb; sh.b_rows = T; sh.b_cols = d;
  sh.M = Is; sh.K = d; sh.out = dHs; sh.ld_out = Is; sh.out_rows = T;
  if ((e = launch_pair_gemm(&r, shared ? &sh : nullptr, p.offsets, koff, Rm, E, shared ? T : 0, 0, next_ticket(),
                            p.status, kManyTiles, s, &n)) != cudaSuccess)
    return e;
  swiglu_bwd_kernel<<<grid_for(Rm * I), 256, 0, s>>>(G, U, dH, Rm, I, dGU);
  if (!ok() || !zero_pads(dGU, size_t(2) * I * 2)) return e;
  if (shared) {
    swiglu_bwd_kernel<<<grid_for((long long)T * Is), 256, 0, s>>>(Gs, Us, dHs, T, Is, dGUs);
    if (!ok()) return e;
  }

  // ---- dX rows = dG W1 + dU W3 (W1^T, W3^T read transposed, K concatenated)
  r = PairOperands();
  r.A = p.W1; r.a_mn = true; r.a_rows = (long long)E * I; r.a_cols = d; r.a_kstep = I;
  r.A2 = p.W3; r.a2_rows = (long long)E * I; r.K1 = I;
  r.B = dGU; r.b_rows = Rm; r.b_cols = 2 * I;
  r.M = d; r.K = 2 * I; r.out = dXr; r.ld_out = d; r.out_rows = Rm;
  sh = PairOperands();
  sh.A = p.Ws1; sh.a_mn = true; sh.a_rows = Is; sh.a_cols = d;
  sh.A2 = p.Ws3; sh.a2_rows = Is; sh.K1 = Is;
  sh.B = dGUs; sh.b_rows = T; sh.b_cols = 2 * Is;
  sh.M = d; sh.K = 2 * Is; sh.out = dXs; sh.ld_out = d; sh.out_rows = T;
  if ((e = launch_pair_gemm(&r, shared ? &sh : nullptr, p.offsets, koff, Rm, E, shared ? T : 0, 0, next_ticket(),
                            p.status, kManyTiles, s, &n)) != cudaSuccess)
    return e;

  // ---- router: d logits (bf16, E_pad columns), dx part dl W_g (W_g^T read transposed)
  GateBwdArgs a;
  a.T = T;
  a.E = E;
  a.k = k;
  a.score_fn = c.score_fn;
  a.norm = c.norm_topk;
  a.nsplit = p.ksplit;
  a.plane = p.plane;
  a.e_pad = L.E_pad;
  a.scale = c.routed_scaling_factor;
  gate_bwd_kernel<<<grid_for((long long)T * 32), 256, 0, s>>>(p.logits, p.idx, dg, a, dlb);
  if (!ok()) return e;
  sh = PairOperands();
  sh.A = wgb; sh.a_mn = true; sh.a_rows = E; sh.a_cols = d;
  sh.B = dlb; sh.b_rows = T; sh.b_cols = L.E_pad;
  sh.M = d; sh.K = L.E_pad; sh.out = dXg; sh.ld_out = d; sh.out_rows = T;
  if ((e = launch_pair_gemm(nullptr, &sh, nullptr, nullptr, Rm, 0, T, 0, next_ticket(), p.status, kManyTiles, s,
                            &n)) != cudaSuccess)
    return e;
  scatter_rows_kernel<<<grid_for((long long)T * d), 256, 0, s>>>(dXr, shared ? dXs : nullptr, dXg, t2r, T, k, d, p.dx);
  if (!ok()) return e;

  // ---- weight gradients: each a reduction over the group's token rows (kmode)
  // dW2[g][c][i] = sum_t dY[t][c] H[t][i]
  r = PairOperands();
  r.A = H; r.a_mn = true; r.a_rows = Rm; r.a_cols = I;
  r.B = dY; r.b_mn = true; r.b_rows = Rm; r.b_cols = d;
  r.M = I; r.N = d; r.K = KPAD; r.out = p.dW2; r.ld_out = I; r.out_gstride = (long long)d * I;
  sh = PairOperands();
  sh.A = Hs; sh.a_mn = true; sh.a_rows = T; sh.a_cols = Is;
  sh.B = doutb; sh.b_mn = true; sh.b_rows = T; sh.b_cols = d;
  sh.M = Is; sh.N = d; sh.K = KPAD; sh.out = p.dWs2; sh.ld_out = Is;
  if ((e = launch_pair_gemm(&r, shared ? &sh : nullptr, koff, nullptr, Rm, E, shared ? T_pad : 0, 1, next_ticket(),
                            p.status, kManyTiles, s, &n)) != cudaSuccess)
    return e;
  // dW1[g][i][c] = sum_t dG[t][i] X[t][c], dW3 likewise with dU (the second half of dGU)
  for (int which = 0; which < 2; ++which) {
    r = PairOperands();
    r.A = Xp; r.a_mn = true; r.a_rows = Rm; r.a_cols = d;
    r.B = dGU; r.b_mn = true; r.b_rows = Rm; r.b_cols = 2 * I; r.b_col0 = which * I;
    r.M = d; r.N = I; r.K = KPAD; r.out = which == 0 ? p.dW1 : p.dW3; r.ld_out = d; r.out_gstride = (long long)I * d;
    sh = PairOperands();
    sh.A = p.x; sh.a_mn = true; sh.a_rows = T; sh.a_cols = d;
    sh.B = dGUs; sh.b_mn = true; sh.b_rows = T; sh.b_cols = 2 * Is; sh.b_col0 = which * Is;
    sh.M = d; sh.N = Is; sh.K = KPAD; sh.out = which == 0 ? p.dWs1 : p.dWs3; sh.ld_out = d;
    if ((e = launch_pair_gemm(&r, shared ? &sh : nullptr, koff, nullptr, Rm, E, shared ? T_pad : 0, 1, next_ticket(),
                              p.status, kManyTiles, s, &n)) != cudaSuccess)
      return e;
  }
  // dW_g[e][c] = sum_t dl[t][e] x[t][c]
  sh = PairOperands();
  sh.A = p.x; sh.a_mn = true; sh.a_rows = T; sh.a_cols = d;
  sh.B = dlb; sh.b_mn = true; sh.b_rows = T; sh.b_cols = L.E_pad;
  sh.M = d; sh.N = E; sh.K = KPAD; sh.out = p.dWg; sh.ld_out = d;
  if ((e = launch_pair_gemm(nullptr, &sh, nullptr, nullptr, Rm, 0, T_pad, 1, next_ticket(), p.status, kManyTiles, s,
                            &n)) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

}  // namespace moe
