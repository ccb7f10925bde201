// Router: gate logits, affinities and (group-limited) top-k selection.
//
// Follows the MoEGate listing of the DeepSeek-V2 walkthrough: logits of a
// bias-free linear layer computed in fp32, softmax over all experts, greedy
// top-k, or group-limited greedy (group score = max, keep topk_group groups,
// pick top-k inside them).  The V3 architecture page (section 1.2) adds the
// sigmoid affinity, a per-expert bias used only to choose the experts, gates
// renormalised over the chosen experts, and node-limited routing whose group
// score sums the group's highest affinities.
//
// Decisions are taken on fp32 selection scores s + b; equal scores go to the
// lower expert (or group) index.  Experts of dropped groups are excluded, not
// zero-filled.
#include "internal.h"

namespace moe {
namespace {

// fp32 W_g -> [hi | mid | lo] bf16 along K, so that x . w = x . hi + x . mid + x . lo
// exactly in fp32 products (bf16 x times bf16 parts) for the tensor-core gate.
__global__ void gate_split_kernel(const float* __restrict__ wg, int E, int d, __nv_bfloat16* __restrict__ out) {
  // first kernel of a call: its dependents may start only once everything
  // earlier in the stream has completed
  pdl_wait();
  pdl_launch_dependents();
  const long long n = (long long)E * d;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long e = i / d, c = i % d;
    const float w = wg[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    __nv_bfloat16* row = out + e * 3LL * d;
    row[c] = hi;
    row[d + c] = mid;
    row[2LL * d + c] = lo;
  }
}

// SIMT fp32 logits: block = 8 warps over TB tokens (staged in shared memory)
// and a slice of experts; each warp owns one expert at a time and reduces the
// TB dot products with warp shuffles.
template <typename TX, typename TW, int TB>
__global__ void __launch_bounds__(256) gate_logits_simt_kernel(const TX* __restrict__ x, const TW* __restrict__ wg,
                                                               int T, int d, int E, int experts_per_block,
                                                               float* __restrict__ logits) {
  extern __shared__ float xs[];  // [TB][d] fp32
  const int t0 = blockIdx.x * TB;
  const int nt = min(TB, T - t0);
  for (int i = threadIdx.x; i < TB * d; i += blockDim.x) {
    const int tt = i / d, c = i % d;
    xs[i] = tt < nt ? ElemTraits<TX>::to_f(x[(long long)(t0 + tt) * d + c]) : 0.0f;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e_begin = blockIdx.y * experts_per_block;
  const int e_end = min(E, e_begin + experts_per_block);
  for (int e = e_begin + warp; e < e_end; e += 8) {
    const TW* w = wg + (long long)e * d;
    float acc[TB];
#pragma unroll
    for (int tt = 0; tt < TB; ++tt) acc[tt] = 0.0f;
    for (int c = lane; c < d; c += 32) {
      const float wv = ElemTraits<TW>::to_f(w[c]);
#pragma unroll
      for (int tt = 0; tt < TB; ++tt) acc[tt] = fmaf(xs[tt * d + c], wv, acc[tt]);
    }
#pragma unroll
    for (int tt = 0; tt < TB; ++tt) {
      const float v = warp_sum(acc[tt]);
      if (lane == 0 && tt < nt) logits[(long long)(t0 + tt) * E + e] = v;
    }
  }
}

constexpr int MAXV = 8;        // experts per lane (E <= 256)

struct TopkArgs {
  int T, E, k, score_fn, method, n_group, topk_group, group_score, group_top, norm;
  float scale;
  int nsplit;          // partial logit planes to add, in order
  long long plane;     // elements between planes
};

constexpr int TOPK_WARPS = 8;   // tokens per block

// Block of TOPK_WARPS warps, one token per warp.  First the whole block forms
// the logits of its tokens in shared memory (partial planes added in plane
// order, loads batched so they are in flight together); then lane l of a
// token's warp holds experts l, l+32, l+64, ...
__global__ void __launch_bounds__(TOPK_WARPS * 32) topk_kernel(const float* __restrict__ logits,
                                                               const float* __restrict__ bias, TopkArgs a,
                                                               int32_t* __restrict__ idx_out,
                                                               float* __restrict__ w_out) {
  __shared__ float lg_s[TOPK_WARPS][MAXV * 32];
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * TOPK_WARPS;
  for (int i = threadIdx.x; i < TOPK_WARPS * a.E; i += blockDim.x) {
    const int tt = i / a.E, e = i - tt * a.E;
    float v = 0.0f;
    if (t0 + tt < a.T) {
      const float* p = logits + (long long)(t0 + tt) * a.E + e;
      v = p[0];
      int sp = 1;
      for (; sp + 8 <= a.nsplit; sp += 8) {
        float u[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) u[j] = p[(sp + j) * a.plane];
#pragma unroll
        for (int j = 0; j < 8; ++j) v = __fadd_rn(v, u[j]);
      }
      for (; sp < a.nsplit; ++sp) v = __fadd_rn(v, p[sp * a.plane]);
    }
    lg_s[tt][e] = v;
  }
  __syncthreads();
  const int t = t0 + warp;
  if (t >= a.T) return;
  const float NEG = -INFINITY;
  float s[MAXV], sel[MAXV];

  float lg[MAXV];
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int e = lane + 32 * i;
    lg[i] = e < a.E ? lg_s[warp][e] : NEG;
  }
  if (a.score_fn == MOE_SCORE_SOFTMAX) {
    float m = NEG;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) m = fmaxf(m, lg[i]);
    m = warp_max(m);
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      s[i] = (lane + 32 * i) < a.E ? expf(lg[i] - m) : 0.0f;
      sum += s[i];
    }
    sum = warp_sum(sum);
#pragma unroll
    for (int i = 0; i < MAXV; ++i) s[i] = s[i] / sum;
  } else {
#pragma unroll
    for (int i = 0; i < MAXV; ++i) s[i] = (lane + 32 * i) < a.E ? 1.0f / (1.0f + expf(-lg[i])) : 0.0f;
  }
  // selection score sigma = s + b; NEG marks "not selectable"
  uint32_t elig = 0;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int e = lane + 32 * i;
    if (e < a.E) {
      sel[i] = bias != nullptr ? __fadd_rn(s[i], bias[e]) : s[i];
      elig |= 1u << i;
    } else {
      sel[i] = NEG;
    }
  }

  if (a.method == MOE_TOPK_GROUP_LIMITED && a.topk_group < a.n_group) {
    const int gsz = a.E / a.n_group;
    int gid[MAXV];   // group of each slot (contiguous blocks of gsz experts)
#pragma unroll
    for (int i = 0; i < MAXV; ++i) gid[i] = (lane + 32 * i) / gsz;
    uint32_t kept = 0;   // bit g: group g stays eligible (same in every lane)
    float my_gscore = NEG;   // lane g holds the score of group g
    for (int g = 0; g < a.n_group; ++g) {
      float gscore;
      if (a.group_score == MOE_GROUP_MAX) {
        float m = NEG;
#pragma unroll
        for (int i = 0; i < MAXV; ++i)
          if ((elig >> i & 1u) && gid[i] == g) m = fmaxf(m, sel[i]);
        gscore = warp_max(m);
      } else if (a.group_top == 2) {
        // the group's two largest scores: each lane's pair, then a butterfly
        // merge of sorted pairs; their fp32 sum
        float v1 = NEG, v2 = NEG;
#pragma unroll
        for (int i = 0; i < MAXV; ++i) {
          if ((elig >> i & 1u) && gid[i] == g) {
            const float x = sel[i];
            if (x > v1) {
              v2 = v1;
              v1 = x;
            } else if (x > v2) {
              v2 = x;
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float b1 = __shfl_xor_sync(0xffffffffu, v1, o);
          const float b2 = __shfl_xor_sync(0xffffffffu, v2, o);
          const float hi = fmaxf(v1, b1);
          v2 = fmaxf(fminf(v1, b1), fmaxf(v2, b2));
          v1 = hi;
        }
        gscore = __fadd_rn(v1, v2);
      } else {
        // sum of the group's top-m scores, in descending order, in fp32
        uint32_t used = 0;
        float acc = 0.0f;
        for (int r = 0; r < a.group_top; ++r) {
          float v = NEG;
          int id = 0x7fffffff;
#pragma unroll
          for (int i = 0; i < MAXV; ++i) {
            const int e = lane + 32 * i;
            if ((elig >> i & 1u) && !(used >> i & 1u) && gid[i] == g && (sel[i] > v || (sel[i] == v && e < id))) {
              v = sel[i];
              id = e;
            }
          }
          warp_argmax(v, id);
          if (id != 0x7fffffff && (id & 31) == lane) used |= 1u << (id >> 5);
          acc = (r == 0) ? v : __fadd_rn(acc, v);
        }
        gscore = acc;
      }
      if (lane == g) my_gscore = gscore;
    }
    // the topk_group best groups; equal scores go to the lower group index
    for (int r = 0; r < a.topk_group; ++r) {
      float v = (lane < a.n_group && !(kept >> lane & 1u)) ? my_gscore : NEG;
      int id = lane < a.n_group && !(kept >> lane & 1u) ? lane : 0x7fffffff;
      warp_argmax(v, id);
      kept |= 1u << id;
    }
#pragma unroll
    for (int i = 0; i < MAXV; ++i)
      if ((elig >> i & 1u) && !(kept >> gid[i] & 1u)) elig &= ~(1u << i);
  }

  // k rounds of warp arg-max over the eligible, not yet chosen experts
  int my_idx = 0;
  float my_s = 0.0f;
  float ssum = 0.0f;
  for (int j = 0; j < a.k; ++j) {
    float v = NEG;
    int id = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int e = lane + 32 * i;
      if ((elig >> i & 1u) && (sel[i] > v || (sel[i] == v && e < id))) {
        v = sel[i];
        id = e;
      }
    }
    warp_argmax(v, id);
    // fetch the unbiased affinity of the winner from its owner lane
    float sv = 0.0f;
    const int owner = id & 31, slot = id >> 5;
#pragma unroll
    for (int i = 0; i < MAXV; ++i)
      if (i == slot) sv = s[i];
    sv = __shfl_sync(0xffffffffu, sv, owner);
    if (lane == owner) elig &= ~(1u << slot);
    ssum = (j == 0) ? sv : __fadd_rn(ssum, sv);
    if (lane == j) {
      my_idx = id;
      my_s = sv;
    }
  }
  if (lane < a.k) {
    float g = my_s;
    if (a.norm) g = g / ssum;
    g = g * a.scale;
    idx_out[(long long)t * a.k + lane] = my_idx;
    w_out[(long long)t * a.k + lane] = g;
  }
}

}  // namespace

cudaError_t launch_gate_split(const float* wg, int E, int d, void* wsplit, cudaStream_t s, int* launches) {
  const long long n = (long long)E * d;
  const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  cudaError_t e = launch_pdl(gate_split_kernel, dim3(grid), dim3(256), 0, s, wg, E, d, static_cast<__nv_bfloat16*>(wsplit));
  if (launches) ++*launches;
  return e;
}

template <typename TX, typename TW, int TB>
static cudaError_t gate_simt_typed(const moe_config& c, const void* x, const void* wg, float* logits,
                                   cudaStream_t s) {
  const size_t smem = size_t(TB) * c.d * sizeof(float);
  static PerDevice<int> attr;
  int unused = 0;
  cudaError_t e = attr.get(&unused, [](int*) {
    return cudaFuncSetAttribute(gate_logits_simt_kernel<TX, TW, TB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                200 * 1024);
  });
  if (e != cudaSuccess) return e;
  const int tblocks = (c.T + TB - 1) / TB;
  // split the experts across blocks until the grid covers the GPU
  int epb = c.E;
  while (epb > 8 && (long long)tblocks * ((c.E + epb - 1) / epb) < 2LL * num_sms()) epb = (epb + 1) / 2;
  dim3 grid(tblocks, (c.E + epb - 1) / epb);
  gate_logits_simt_kernel<TX, TW, TB><<<grid, 256, smem, s>>>(static_cast<const TX*>(x), static_cast<const TW*>(wg),
                                                               c.T, c.d, c.E, epb, logits);
  return cudaGetLastError();
}

cudaError_t launch_gate_logits_simt(const moe_config& c, const void* x, const void* wg, float* logits,
                                    cudaStream_t s, int* launches) {
  cudaError_t e;
  // TB tokens of fp32 x per block must fit in 200 KB of shared memory
  const bool wide = size_t(8) * c.d * sizeof(float) > 200 * 1024;
  if (c.act_dtype == MOE_F32) {
    if (c.gate_w_dtype == MOE_F32)
      e = wide ? gate_simt_typed<float, float, 4>(c, x, wg, logits, s) : gate_simt_typed<float, float, 8>(c, x, wg, logits, s);
    else
      e = wide ? gate_simt_typed<float, __nv_bfloat16, 4>(c, x, wg, logits, s)
               : gate_simt_typed<float, __nv_bfloat16, 8>(c, x, wg, logits, s);
  } else {
    if (c.gate_w_dtype == MOE_F32)
      e = wide ? gate_simt_typed<__nv_bfloat16, float, 4>(c, x, wg, logits, s)
               : gate_simt_typed<__nv_bfloat16, float, 8>(c, x, wg, logits, s);
    else
      e = wide ? gate_simt_typed<__nv_bfloat16, __nv_bfloat16, 4>(c, x, wg, logits, s)
               : gate_simt_typed<__nv_bfloat16, __nv_bfloat16, 8>(c, x, wg, logits, s);
  }
  if (e == cudaSuccess && launches) ++*launches;
  return e;
}

cudaError_t launch_topk(const moe_config& c, const float* logits, int nsplit, long long plane, const float* bias,
                        int32_t* idx, float* w, cudaStream_t s, int* launches) {
  TopkArgs a;
  a.nsplit = nsplit;
  a.plane = plane;
  a.T = c.T;
  a.E = c.E;
  a.k = c.k;
  a.score_fn = c.score_fn;
  a.method = c.topk_method;
  a.n_group = c.n_group;
  a.topk_group = c.topk_group;
  a.group_score = c.group_score;
  a.group_top = c.group_top;
  a.norm = c.norm_topk;
  a.scale = c.routed_scaling_factor;
  cudaError_t e = launch_pdl(topk_kernel, dim3((c.T + TOPK_WARPS - 1) / TOPK_WARPS), dim3(TOPK_WARPS * 32), 0, s,
                             logits, bias, a, idx, w);
  if (launches) ++*launches;
  return e;
}

}  // namespace moe
