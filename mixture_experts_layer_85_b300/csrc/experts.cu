// Expert weight packing, the SIMT fp32 expert path, and the combine.
//
// SwiGLU expert: FFN(u) = W2 (silu(W1 u) * (W3 u)) with nn.Linear layouts
// (intelliparadigm.com page, section 3.3.1).  The MoE listing of the
// DeepSeek-V2 walkthrough sums the k routed expert outputs weighted by their
// gates and adds the shared experts, fused as one SwiGLU of hidden
// n_shared * I, evaluated on every token; no residual is added.
#include <cuda_fp8.h>

#include "internal.h"

namespace moe {
namespace {

// W1/W3 [G,H,d] -> W13 [G,2H,d]: for each block of `bi` hidden units, the W1
// rows followed by the matching W3 rows.
__global__ void interleave_w13_kernel(const uint4* __restrict__ w1, const uint4* __restrict__ w3,
                                      uint4* __restrict__ dst, long long G, int H, int bi, int vec_per_row) {
  const long long rows = G * 2LL * H;
  const long long n = rows * vec_per_row;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / vec_per_row;
    const int v = int(i % vec_per_row);
    const long long g = row / (2LL * H);
    const int p = int(row % (2LL * H));
    const int blk = p / (2 * bi), r = p % (2 * bi);
    const uint4* src = (r < bi ? w1 : w3) + ((g * H + (long long)blk * bi + (r % bi)) * vec_per_row);
    dst[i] = src[v];
  }
}

// Block quantisation to FP8 e4m3 (intelliparadigm.com page, section 4): one
// thread per run of 64 consecutive weights of an output row.  The scale is the
// smallest power of two with max|w| <= 448 * scale (amax = f * 2^x with f in
// [0.5, 1): 2^(x-9) when f <= 0.875, else 2^(x-8); 1 for an all-zero run), so
// w / scale is exact and the e4m3 value times the scale is a bf16 number.
// Output row p of a [G, R_out, cols] matrix comes from src_a (or, for the
// interleaved W1/W3 layout, from W1 or W3 by the same rule as
// interleave_w13_kernel).
//
// Output layout (the shared-memory image the expert GEMM consumes, so one bulk
// copy moves a stage): rows in tiles of 128, each tile a run of cols / 128
// stage blocks of FP8_STAGE_BYTES:
//   bytes [0, 16384): row r's 128 e4m3 values at r * 128, its 16-byte chunk c
//     (values 16c .. 16c + 15 of the stage) at chunk position c ^ (r % 8)
//     (the 128-byte swizzle);
//   bytes [16384, 17408): int32 scale exponents [2][128], [h][r] for the
//     stage's 64-value block h of row r (its scale is 2^e).
__global__ void quantize_fp8_kernel(const __nv_bfloat16* __restrict__ src_a, const __nv_bfloat16* __restrict__ src_b,
                                    long long G, int H, int bi, int cols, uint8_t* __restrict__ dst) {
  const int nb = cols / 64, n_st = cols / 128;
  const long long rows_out = src_b != nullptr ? G * 2LL * H : G * (long long)H;
  const long long n = rows_out * nb;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long row = i % rows_out;
    const int b = int(i / rows_out);
    const __nv_bfloat16* src;
    if (src_b != nullptr) {
      const long long g = row / (2LL * H);
      const int p = int(row % (2LL * H));
      const int blk = p / (2 * bi), r = p % (2 * bi);
      src = (r < bi ? src_a : src_b) + (g * H + (long long)blk * bi + (r % bi)) * cols;
    } else {
      src = src_a + row * cols;
    }
    const uint4* s4 = reinterpret_cast<const uint4*>(src + b * 64);
    uint4 v[8];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = s4[j];
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v[j]);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 f = __bfloat1622float2(h2[t]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
    int x = 0;
    const float f = frexpf(amax, &x);
    const int e = amax == 0.0f ? 0 : (f <= 0.875f ? x - 9 : x - 8);
    const float inv = ldexpf(1.0f, -e);   // exact power of two
    uint32_t out[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v[j]);
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 w = __bfloat1622float2(h2[t]);
        const uint32_t q0 = __nv_cvt_float_to_fp8(w.x * inv, __NV_SATFINITE, __NV_E4M3);
        const uint32_t q1 = __nv_cvt_float_to_fp8(w.y * inv, __NV_SATFINITE, __NV_E4M3);
        const uint32_t pair = q0 | (q1 << 8);
        if (t < 2) lo |= pair << (16 * t);
        else hi |= pair << (16 * (t - 2));
      }
      out[2 * j] = lo;
      out[2 * j + 1] = hi;
    }
    const int r = int(row % 128), st = b / 2, h = b % 2;
    uint8_t* blk = dst + ((row / 128) * n_st + st) * (long long)FP8_STAGE_BYTES;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = 4 * h + q;
      *reinterpret_cast<uint4*>(blk + r * 128 + ((c ^ (r & 7)) << 4)) =
          make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
    }
    reinterpret_cast<int32_t*>(blk + FP8_IMAGE_BYTES)[h * 128 + r] = e;
  }
}

// Largest |w| of each of G matrices of vec_per_matrix 16-byte vectors of bf16
// (the matrix of blockIdx.y), into amax[(g0 + g) * 3 + slot] as float bits: one
// atomicMax per block (non-negative floats order like their bit patterns).
__global__ void __launch_bounds__(256) matrix_amax_kernel(const uint4* __restrict__ src, long long vec_per_matrix,
                                                          int g0, int slot, uint32_t* __restrict__ amax) {
  __shared__ float part[8];
  const uint4* m = src + (long long)blockIdx.y * vec_per_matrix;
  float a = 0.0f;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < vec_per_matrix;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 v = m[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int t = 0; t < 4; ++t)
      a = fmaxf(a, fmaxf(fabsf(__uint_as_float(w[t] << 16)), fabsf(__uint_as_float(w[t] & 0xffff0000u))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int wi = 1; wi < 8; ++wi) a = fmaxf(a, part[wi]);
    atomicMax(&amax[(g0 + (long long)blockIdx.y) * 3 + slot], __float_as_uint(a));
  }
}

// A matrix's reference exponent: the scale exponent its largest |w| gets by
// the block rule above (the largest block exponent of the matrix; 0 when the
// matrix is zero).  In place over the amax bits.
__global__ void eref_from_amax_kernel(int32_t* eref, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float amax = __uint_as_float(uint32_t(eref[i]));
  int x = 0;
  const float f = frexpf(amax, &x);
  eref[i] = amax == 0.0f ? 0 : (f <= 0.875f ? x - 9 : x - 8);
}

// bf16 weights -> stage blocks (layout in internal.h), one thread per 16-byte
// chunk of the output: output row p of group g comes from src_a (or, with
// src_b, from W1 / W3 interleaved in blocks of `bi` rows as in
// interleave_w13_kernel); columns and rows past the matrix are zeros.
__global__ void pack_bf16_stages_kernel(const uint4* __restrict__ src_a, const uint4* __restrict__ src_b, long long G,
                                        int H, int bi, int M, int cols, int tpg, int nst, uint4* __restrict__ dst) {
  const long long n = G * tpg * nst * (IMG_BLOCK_BYTES / 16);
  const int vrow = cols / 8;   // 16-byte chunks of a source row
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int c8 = int(i & 7);                 // chunk of the 64-column k-block row
    const int r = int((i >> 3) & 127);         // row within the tile
    const int kb = int((i >> 10) & 1);         // k-block within the stage
    const long long blk = i >> 11;
    const int st = int(blk % nst);
    const long long t = blk / nst;
    const int tr = int(t % tpg);
    const long long g = t / tpg;
    const int prow = tr * IMG_ROWS + r;
    const int k = st * IMG_COLS + kb * 64 + c8 * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (prow < M && k < cols) {
      const uint4* row;
      if (src_b != nullptr) {
        const int blk2 = prow / (2 * bi), rr = prow % (2 * bi);
        row = (rr < bi ? src_a : src_b) + (g * H + (long long)blk2 * bi + (rr % bi)) * vrow;
      } else {
        row = src_a + (g * M + prow) * vrow;
      }
      v = row[k / 8];
    }
    dst[i] = v;
  }
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Expert of routed row r: the last e with offsets[e] <= r.
__device__ __forceinline__ int expert_of_row(const int32_t* __restrict__ offsets, int E, long long r) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (offsets[mid] <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

struct SimtArgs {
  long long R;
  int T, d, E, I, Is, bi, bis;
};

// fp32 GEMM1 + SwiGLU, one thread per (row, hidden unit).  Rows [0,R) are the
// routed rows, rows [R, R+T) are the tokens for the shared expert.
__global__ void swiglu_simt_h_kernel(const float* __restrict__ x_perm, const int32_t* __restrict__ offsets,
                                     const float* __restrict__ x, const float* __restrict__ w13,
                                     const float* __restrict__ w13s, SimtArgs a, float* __restrict__ h,
                                     float* __restrict__ hs, int* status) {
  const long long n_routed = a.R * a.I;
  const long long n = n_routed + (long long)a.T * a.Is;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float* xr;
    const float* wa;
    const float* wb;
    float* dst;
    if (i < n_routed) {
      const long long r = i / a.I;
      const int u = int(i % a.I);
      const int e = expert_of_row(offsets, a.E, r);
      if (r >= offsets[a.E]) {
        flag_status(status, DEV_BAD_ROW);
        continue;
      }
      xr = x_perm + r * a.d;
      const long long base = (long long)e * 2 * a.I + (u / a.bi) * 2LL * a.bi + (u % a.bi);
      wa = w13 + base * a.d;
      wb = w13 + (base + a.bi) * a.d;
      dst = h + r * a.I + u;
    } else {
      const long long j = i - n_routed;
      const long long t = j / a.Is;
      const int u = int(j % a.Is);
      xr = x + t * a.d;
      const long long base = (u / a.bis) * 2LL * a.bis + (u % a.bis);
      wa = w13s + base * a.d;
      wb = w13s + (base + a.bis) * a.d;
      dst = hs + t * a.Is + u;
    }
    float s1 = 0.0f, s3 = 0.0f;
    for (int c = 0; c < a.d; ++c) {
      const float xv = xr[c];
      s1 = fmaf(xv, wa[c], s1);
      s3 = fmaf(xv, wb[c], s3);
    }
    *dst = silu(s1) * s3;
  }
}

// fp32 GEMM2, one thread per (row, output feature).
__global__ void swiglu_simt_y_kernel(const float* __restrict__ h, const float* __restrict__ hs,
                                     const int32_t* __restrict__ offsets, const float* __restrict__ w2,
                                     const float* __restrict__ w2s, SimtArgs a, float* __restrict__ y,
                                     float* __restrict__ ys) {
  const long long n_routed = a.R * a.d;
  const long long n = n_routed + (long long)a.T * a.d;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float* hr;
    const float* wr;
    float* dst;
    int H;
    if (i < n_routed) {
      const long long r = i / a.d;
      const int c = int(i % a.d);
      if (r >= offsets[a.E]) continue;
      const int e = expert_of_row(offsets, a.E, r);
      hr = h + r * a.I;
      wr = w2 + ((long long)e * a.d + c) * a.I;
      dst = y + r * a.d + c;
      H = a.I;
    } else {
      const long long j = i - n_routed;
      const long long t = j / a.d;
      const int c = int(j % a.d);
      hr = hs + t * a.Is;
      wr = w2s + (long long)c * a.Is;
      dst = ys + t * a.d + c;
      H = a.Is;
    }
    float acc = 0.0f;
    for (int u = 0; u < H; ++u) acc = fmaf(hr[u], wr[u], acc);
    *dst = acc;
  }
}

template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void load(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ uint4 store(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void load(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ uint4 store(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <typename O, int N> struct StoreN;
template <> struct StoreN<float, 8> {
  static __device__ __forceinline__ void st(float* p, const float* f) {
    reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
};
template <> struct StoreN<float, 4> {
  static __device__ __forceinline__ void st(float* p, const float* f) {
    reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  }
};
template <> struct StoreN<__nv_bfloat16, 8> {
  static __device__ __forceinline__ void st(__nv_bfloat16* p, const float* f) {
    *reinterpret_cast<uint4*>(p) = Vec16<__nv_bfloat16>::store(f);
  }
};
template <> struct StoreN<__nv_bfloat16, 4> {
  static __device__ __forceinline__ void st(__nv_bfloat16* p, const float* f) {
    __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]), b = __floats2bfloat162_rn(f[2], f[3]);
    *reinterpret_cast<uint2*>(p) = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  }
};

// out[t] = sum_j w[t,j] * y_perm[tok2row[t,j]] + y_shared[t], fp32 accumulation
// in slot order.  Blocks stride over tokens; blockIdx.y splits each row into
// gridDim.y slices so that small batches still spread over the GPU.  16-byte
// vector loads.
template <typename T, typename O, int MAXK>
__global__ void __launch_bounds__(128) combine_kernel(const uint4* __restrict__ y_perm, const uint4* __restrict__ y_shared,
                                                      const int32_t* __restrict__ tok2row, const float* __restrict__ w,
                                                      int Tn, int k, long long R, int vec_per_row,
                                                      O* __restrict__ out, int* status) {
  constexpr int N = Vec16<T>::N;
  pdl_launch_dependents();
  pdl_wait();
  for (int t = blockIdx.x; t < Tn; t += gridDim.x) {
    long long rows[MAXK];
    float g[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      rows[j] = -1;
      g[j] = 0.0f;
      if (j < k) {
        const long long r = tok2row[(long long)t * k + j];
        if (r >= 0 && r < R) {
          rows[j] = r;
          g[j] = w[(long long)t * k + j];
        } else if (threadIdx.x == 0) {
          flag_status(status, DEV_BAD_ROW);
        }
      }
    }
    const int per = (vec_per_row + gridDim.y - 1) / gridDim.y;
    const int v_end = min(vec_per_row, int(blockIdx.y + 1) * per);
    for (int v = blockIdx.y * per + threadIdx.x; v < v_end; v += blockDim.x) {
      float acc[N];
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int j = 0; j < MAXK; ++j) {
        if (rows[j] >= 0) {
          float f[N];
          Vec16<T>::load(y_perm[rows[j] * vec_per_row + v], f);
#pragma unroll
          for (int i = 0; i < N; ++i) acc[i] = fmaf(g[j], f[i], acc[i]);
        }
      }
      if (y_shared != nullptr) {
        float f[N];
        Vec16<T>::load(y_shared[(long long)t * vec_per_row + v], f);
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] += f[i];
      }
      StoreN<O, N>::st(out + ((long long)t * vec_per_row + v) * N, acc);
    }
  }
}

template <typename T, typename O>
cudaError_t combine_typed(const moe_config& c, const uint4* yp, const uint4* ys, const int32_t* tok2row, const float* w,
                          void* out, int* status, cudaStream_t s) {
  const int vec = int(size_t(c.d) * sizeof(T) / 16);
  const int gx = c.T < 65535 ? c.T : 65535;
  // row slices of at least 128 vectors until the grid covers the SMs twice
  int gy = 1;
  while ((long long)gx * gy < 2LL * num_sms() && (vec + 2 * gy - 1) / (2 * gy) >= 128) gy *= 2;
  const dim3 grid(gx, gy);
  const long long R = (long long)c.T * c.k;
  O* o = static_cast<O*>(out);
  if (c.k <= 8) return launch_pdl(combine_kernel<T, O, 8>, grid, dim3(128), 0, s, yp, ys, tok2row, w, c.T, c.k, R, vec, o, status);
  return launch_pdl(combine_kernel<T, O, 16>, grid, dim3(128), 0, s, yp, ys, tok2row, w, c.T, c.k, R, vec, o, status);
}

}  // namespace

PackedLayout packed_layout(const moe_config& c) {
  PackedLayout L;
  L.fp8 = c.expert_w_dtype == MOE_FP8_E4M3;
  const size_t eb = dtype_bytes(c.act_dtype);
  const long long Is = (long long)c.n_shared * c.I;
  // blocks of 16 hidden units: W1 rows, then the W3 rows of the same units
  L.bi = (c.I % 16 == 0) ? 16 : c.I;
  L.bis = (Is % 16 == 0) ? 16 : int(Is > 0 ? Is : 1);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  if (L.fp8) {
    L.w13 = take(fp8_tiled_bytes(2LL * c.E * c.I, c.d));
    L.w2 = take(fp8_tiled_bytes((long long)c.E * c.d, c.I));
    L.w13s = take(Is > 0 ? fp8_tiled_bytes(2 * Is, c.d) : 0);
    L.w2s = take(Is > 0 ? fp8_tiled_bytes(c.d, Is) : 0);
    L.eref = take(size_t(c.E + 1) * 3 * sizeof(int32_t));
  } else if (c.act_dtype == MOE_BF16) {
    L.img = true;
    L.w13 = take(img_bytes(c.E, 2LL * c.I, c.d));
    L.w2 = take(img_bytes(c.E, c.d, c.I));
    L.w13s = take(Is > 0 ? img_bytes(1, 2 * Is, c.d) : 0);
    L.w2s = take(Is > 0 ? img_bytes(1, c.d, Is) : 0);
  } else {
    L.w13 = take(size_t(c.E) * 2 * c.I * c.d * eb);
    L.w2 = take(size_t(c.E) * c.d * c.I * eb);
    L.w13s = take(size_t(2 * Is) * c.d * eb);
    L.w2s = take(size_t(c.d) * Is * eb);
  }
  L.total = off;
  return L;
}

cudaError_t launch_prepack(const moe_config& c, const void* W1, const void* W3, const void* W2,
                           const void* Ws1, const void* Ws3, const void* Ws2, void* packed, cudaStream_t s,
                           int* launches) {
  const PackedLayout L = packed_layout(c);
  const size_t eb = dtype_bytes(c.act_dtype);
  const int vec = int(size_t(c.d) * eb / 16);
  char* base = static_cast<char*>(packed);
  const long long Is = (long long)c.n_shared * c.I;
  auto grid_for = [](long long n) { long long g = (n + 255) / 256; return int(g < 8192 ? g : 8192); };
  if (L.fp8) {
    using bf = __nv_bfloat16;
    auto q = [&](const void* a, const void* b, long long G, int H, int bi, int cols, size_t off) {
      const long long rows = b != nullptr ? G * 2LL * H : G * (long long)H;
      uint8_t* dst = reinterpret_cast<uint8_t*>(base + off);
      // the tile past the last row (read by the odd CTA of a pair at the end) is zero
      const size_t tile = size_t(cols / 128) * FP8_STAGE_BYTES;
      cudaError_t e = cudaMemsetAsync(dst + size_t(rows / 128) * tile, 0, tile, s);
      if (e != cudaSuccess) return e;
      quantize_fp8_kernel<<<grid_for(rows * (cols / 64)), 256, 0, s>>>(
          static_cast<const bf*>(a), static_cast<const bf*>(b), G, H, bi, cols, dst);
      if (launches) ++*launches;
      return cudaGetLastError();
    };
    // reference exponents: the largest |w| of every matrix, then its exponent
    int32_t* eref = reinterpret_cast<int32_t*>(base + L.eref);
    const int n_ref = (c.E + 1) * 3;
    cudaError_t e = cudaMemsetAsync(eref, 0, size_t(n_ref) * sizeof(int32_t), s);
    auto amax = [&](const void* w, long long G, long long rows, long long cols, int g0, int slot) {
      const long long vec = rows * cols / 8;
      long long bx = (vec + 255) / 256;
      if (bx > 64) bx = 64;
      matrix_amax_kernel<<<dim3(unsigned(bx), unsigned(G)), 256, 0, s>>>(static_cast<const uint4*>(w), vec, g0, slot,
                                                                      reinterpret_cast<uint32_t*>(eref));
      if (launches) ++*launches;
      return cudaGetLastError();
    };
    if (e == cudaSuccess) e = amax(W1, c.E, c.I, c.d, 0, 0);
    if (e == cudaSuccess) e = amax(W3, c.E, c.I, c.d, 0, 1);
    if (e == cudaSuccess) e = amax(W2, c.E, c.d, c.I, 0, 2);
    if (e == cudaSuccess && Is > 0) e = amax(Ws1, 1, Is, c.d, c.E, 0);
    if (e == cudaSuccess && Is > 0) e = amax(Ws3, 1, Is, c.d, c.E, 1);
    if (e == cudaSuccess && Is > 0) e = amax(Ws2, 1, c.d, Is, c.E, 2);
    if (e == cudaSuccess) {
      eref_from_amax_kernel<<<(n_ref + 255) / 256, 256, 0, s>>>(eref, n_ref);
      if (launches) ++*launches;
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = q(W1, W3, c.E, c.I, L.bi, c.d, L.w13);
    if (e == cudaSuccess) e = q(W2, nullptr, 1, c.E * c.d, 1, c.I, L.w2);
    if (e == cudaSuccess && Is > 0) e = q(Ws1, Ws3, 1, int(Is), L.bis, c.d, L.w13s);
    if (e == cudaSuccess && Is > 0) e = q(Ws2, nullptr, 1, c.d, 1, int(Is), L.w2s);
    return e;
  }
  if (L.img) {
    auto pk = [&](const void* a, const void* b, long long G, int H, int bi, int M, int cols, size_t off) {
      const long long n = G * img_tiles(M) * img_stages(cols) * (IMG_BLOCK_BYTES / 16);
      pack_bf16_stages_kernel<<<grid_for(n), 256, 0, s>>>(static_cast<const uint4*>(a), static_cast<const uint4*>(b),
                                                          G, H, bi, M, cols, img_tiles(M), img_stages(cols),
                                                          reinterpret_cast<uint4*>(base + off));
      if (launches) ++*launches;
      return cudaGetLastError();
    };
    cudaError_t e = pk(W1, W3, c.E, c.I, L.bi, 2 * c.I, c.d, L.w13);
    if (e == cudaSuccess) e = pk(W2, nullptr, c.E, c.d, 1, c.d, c.I, L.w2);
    if (e == cudaSuccess && Is > 0) e = pk(Ws1, Ws3, 1, int(Is), L.bis, int(2 * Is), c.d, L.w13s);
    if (e == cudaSuccess && Is > 0) e = pk(Ws2, nullptr, 1, c.d, 1, c.d, int(Is), L.w2s);
    return e;
  }
  interleave_w13_kernel<<<grid_for((long long)c.E * 2 * c.I * vec), 256, 0, s>>>(
      static_cast<const uint4*>(W1), static_cast<const uint4*>(W3), reinterpret_cast<uint4*>(base + L.w13), c.E, c.I,
      L.bi, vec);
  if (launches) ++*launches;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyAsync(base + L.w2, W2, size_t(c.E) * c.d * c.I * eb, cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return e;
  if (Is > 0) {
    interleave_w13_kernel<<<grid_for(2 * Is * vec), 256, 0, s>>>(
        static_cast<const uint4*>(Ws1), static_cast<const uint4*>(Ws3), reinterpret_cast<uint4*>(base + L.w13s), 1,
        int(Is), L.bis, vec);
    if (launches) ++*launches;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyAsync(base + L.w2s, Ws2, size_t(c.d) * Is * eb, cudaMemcpyDeviceToDevice, s);
  }
  return e;
}

cudaError_t launch_swiglu_simt_f32(const moe_config& c, const float* x_perm, const int32_t* offsets,
                                   const float* x, const void* packed, float* h, float* hs, float* y, float* ys,
                                   int* status, cudaStream_t s, int* launches) {
  const PackedLayout L = packed_layout(c);
  const char* base = static_cast<const char*>(packed);
  SimtArgs a;
  a.R = (long long)c.T * c.k;
  a.T = c.T;
  a.d = c.d;
  a.E = c.E;
  a.I = c.I;
  a.Is = c.n_shared * c.I;
  a.bi = L.bi;
  a.bis = L.bis;
  const long long n1 = a.R * a.I + (long long)a.T * a.Is;
  const long long n2 = (a.R + a.T) * a.d;
  auto grid_for = [](long long n) { long long g = (n + 255) / 256; return int(g < 65535 ? g : 65535); };
  swiglu_simt_h_kernel<<<grid_for(n1), 256, 0, s>>>(x_perm, offsets, x, reinterpret_cast<const float*>(base + L.w13),
                                                    reinterpret_cast<const float*>(base + L.w13s), a, h, hs, status);
  swiglu_simt_y_kernel<<<grid_for(n2), 256, 0, s>>>(h, hs, offsets, reinterpret_cast<const float*>(base + L.w2),
                                                    reinterpret_cast<const float*>(base + L.w2s), a, y, ys);
  if (launches) *launches += 2;
  return cudaGetLastError();
}

cudaError_t launch_combine(const moe_config& c, const void* y_perm, const void* y_shared, const int32_t* tok2row,
                           const float* w, void* out, int* status, cudaStream_t s, int* launches) {
  auto yp = static_cast<const uint4*>(y_perm);
  // without shared experts there is no shared term to add
  auto ys = c.n_shared > 0 ? static_cast<const uint4*>(y_shared) : nullptr;
  // expert outputs are fp32 for every activation dtype
  cudaError_t e = c.out_dtype == MOE_F32 ? combine_typed<float, float>(c, yp, ys, tok2row, w, out, status, s)
                                         : combine_typed<float, __nv_bfloat16>(c, yp, ys, tok2row, w, out, status, s);
  if (launches) ++*launches;
  return e;
}

}  // namespace moe
