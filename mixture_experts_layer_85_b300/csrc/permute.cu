// Dispatch of the (token, slot) assignments into expert-contiguous rows.
//
// The MoE listing of the DeepSeek-V2 walkthrough repeats every token k times
// and, for each expert, gathers the rows routed to it.  Here that gather is a
// deterministic counting sort: rows of expert e are its tokens in increasing
// order, experts in increasing id, so counts, offsets and the row order are
// exactly reproducible.
//
//   1. count    per 128-token chunk: a 128-bit token mask per expert in shared
//               memory (atomicOr), popcounts -> chunk_counts[chunk][e]
//   2. scan     one block per expert: chunk_base[chunk][e] (rank of the
//               chunk's first token within expert e) and counts[e]; then one
//               block: offsets[e] = exclusive prefix sum of counts
//   3. scatter  per chunk: rank of a token inside its expert = popcount of the
//               mask bits of earlier tokens -> row2tok / tok2row
//   4. gather   x rows -> x_perm rows: each token's row is read once and
//               written to its k destination rows (16-byte vectors)
//
// Decode-sized batches (T <= SMALL_T) run steps 1-3 in one block instead
// (permute_small_kernel: the same masks and ranks over 1024-token chunks taken
// in order), so the dispatch costs two launches, not five.  Its results are
// identical to the multi-block path.
#include <cuda_fp16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int CHUNK = 128;   // tokens per chunk = 4 mask words per expert
constexpr int WORDS = CHUNK / 32;
constexpr int MAX_E = 256;

__device__ __forceinline__ void build_masks(uint32_t (*mask)[WORDS], const int32_t* __restrict__ idx, int T, int E,
                                            int k, int chunk, int* status) {
  for (int i = threadIdx.x; i < E * WORDS; i += blockDim.x) mask[i / WORDS][i % WORDS] = 0u;
  __syncthreads();
  const int t = chunk * CHUNK + threadIdx.x;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int e = idx[(long long)t * k + j];
      if (e < 0 || e >= E) {
        flag_status(status, DEV_BAD_EXPERT);
        continue;
      }
      atomicOr(&mask[e][threadIdx.x >> 5], 1u << (threadIdx.x & 31));
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(CHUNK) permute_count_kernel(const int32_t* __restrict__ idx, int T, int E, int k,
                                                              int32_t* __restrict__ chunk_counts, int* status) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ uint32_t mask[MAX_E][WORDS];
  build_masks(mask, idx, T, E, k, blockIdx.x, status);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int n = 0;
#pragma unroll
    for (int w = 0; w < WORDS; ++w) n += __popc(mask[e][w]);
    chunk_counts[(long long)blockIdx.x * E + e] = n;
  }
}

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* total_out) {
  __shared__ int warp_tot[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
  const int nw = (blockDim.x + 31) >> 5;
  for (int w = 0; w < nw; ++w) {
    if (w < warp) before += warp_tot[w];
    all += warp_tot[w];
  }
  __syncthreads();
  *total_out = all;
  return before + incl - v;
}

// One block per expert: exclusive scan over chunks -> chunk_base[chunk][e]
// (row of the chunk's first token within expert e), counts[e].
__global__ void __launch_bounds__(CHUNK) permute_chunk_scan_kernel(const int32_t* __restrict__ chunk_counts,
                                                                   int nchunks, int E,
                                                                   int32_t* __restrict__ chunk_base,
                                                                   int32_t* __restrict__ counts) {
  pdl_launch_dependents();
  pdl_wait();
  const int e = blockIdx.x;
  int carry = 0;
  for (int c0 = 0; c0 < nchunks; c0 += blockDim.x) {
    const int c = c0 + threadIdx.x;
    const int v = c < nchunks ? chunk_counts[(long long)c * E + e] : 0;
    int tot;
    const int ex = block_exclusive_scan(v, &tot);
    if (c < nchunks) chunk_base[(long long)c * E + e] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) counts[e] = carry;
}

// One block: offsets = exclusive prefix sum of counts over experts (E <= 256).
__global__ void __launch_bounds__(256) permute_offsets_kernel(const int32_t* __restrict__ counts, int E,
                                                              int32_t* __restrict__ offsets) {
  pdl_launch_dependents();
  pdl_wait();
  const int e = threadIdx.x;
  int tot;
  const int ex = block_exclusive_scan(e < E ? counts[e] : 0, &tot);
  if (e < E) offsets[e] = ex;
  if (e == 0) offsets[E] = tot;
}

__global__ void __launch_bounds__(CHUNK) permute_scatter_kernel(const int32_t* __restrict__ idx, int T, int E, int k,
                                                                const int32_t* __restrict__ chunk_base,
                                                                const int32_t* __restrict__ offsets,
                                                                int32_t* __restrict__ row2tok,
                                                                int32_t* __restrict__ tok2row, int* status) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ uint32_t mask[MAX_E][WORDS];
  build_masks(mask, idx, T, E, k, blockIdx.x, nullptr);
  const int t = blockIdx.x * CHUNK + threadIdx.x;
  if (t >= T) return;
  const int w = threadIdx.x >> 5;
  const uint32_t below = (1u << (threadIdx.x & 31)) - 1u;
  const long long R = (long long)T * k;
  for (int j = 0; j < k; ++j) {
    const int e = idx[(long long)t * k + j];
    if (e < 0 || e >= E) {
      tok2row[(long long)t * k + j] = -1;
      continue;
    }
    int rank = __popc(mask[e][w] & below);
    for (int ww = 0; ww < w; ++ww) rank += __popc(mask[e][ww]);
    const long long row = (long long)offsets[e] + chunk_base[(long long)blockIdx.x * E + e] + rank;
    if (row < 0 || row >= R) {
      flag_status(status, DEV_BAD_ROW);
      tok2row[(long long)t * k + j] = -1;
      continue;
    }
    row2tok[row] = t;
    tok2row[(long long)t * k + j] = (int32_t)row;
  }
}

constexpr int SMALL_BLOCK = 1024;           // tokens per chunk of the one-block path
constexpr int SMALL_WORDS = SMALL_BLOCK / 32;
constexpr int SMALL_T = 4 * SMALL_BLOCK;

// Steps 1-3 in one block of SMALL_BLOCK threads (thread = token of the chunk).
__global__ void __launch_bounds__(SMALL_BLOCK) permute_small_kernel(const int32_t* __restrict__ idx, int T, int E,
                                                                    int k, int32_t* __restrict__ counts,
                                                                    int32_t* __restrict__ offsets,
                                                                    int32_t* __restrict__ row2tok,
                                                                    int32_t* __restrict__ tok2row, int* status) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ uint32_t mask[MAX_E][SMALL_WORDS];
  __shared__ int base[MAX_E];
  const int tid = threadIdx.x;
  const int w = tid >> 5;
  const uint32_t below = (1u << (tid & 31)) - 1u;
  const int nch = (T + SMALL_BLOCK - 1) / SMALL_BLOCK;
  const long long R = (long long)T * k;
  if (tid < MAX_E) base[tid] = 0;
  // pass 0 counts, pass 1 ranks; each pass walks the chunks in token order
  for (int pass = 0; pass < 2; ++pass) {
    for (int ch = 0; ch < nch; ++ch) {
      for (int i = tid; i < E * SMALL_WORDS; i += SMALL_BLOCK) mask[i / SMALL_WORDS][i % SMALL_WORDS] = 0u;
      __syncthreads();
      const int t = ch * SMALL_BLOCK + tid;
      if (t < T) {
        for (int j = 0; j < k; ++j) {
          const int e = idx[(long long)t * k + j];
          if (e < 0 || e >= E) {
            if (pass == 0) flag_status(status, DEV_BAD_EXPERT);
            continue;
          }
          atomicOr(&mask[e][w], 1u << (tid & 31));
        }
      }
      __syncthreads();
      if (pass == 1 && t < T) {
        for (int j = 0; j < k; ++j) {
          const int e = idx[(long long)t * k + j];
          if (e < 0 || e >= E) {
            tok2row[(long long)t * k + j] = -1;
            continue;
          }
          int rank = __popc(mask[e][w] & below);
          for (int ww = 0; ww < w; ++ww) rank += __popc(mask[e][ww]);
          const long long row = (long long)base[e] + rank;
          if (row < 0 || row >= R) {
            flag_status(status, DEV_BAD_ROW);
            tok2row[(long long)t * k + j] = -1;
            continue;
          }
          row2tok[row] = t;
          tok2row[(long long)t * k + j] = (int32_t)row;
        }
      }
      __syncthreads();
      if (tid < E) {
        int n = 0;
        for (int ww = 0; ww < SMALL_WORDS; ++ww) n += __popc(mask[tid][ww]);
        base[tid] += n;
      }
      __syncthreads();
    }
    if (pass == 0) {
      // base holds the counts: turn them into offsets
      int tot;
      const int cnt = tid < E ? base[tid] : 0;
      const int ex = block_exclusive_scan(cnt, &tot);
      if (tid < E) {
        counts[tid] = cnt;
        offsets[tid] = ex;
      }
      if (tid == 0) offsets[E] = tot;
      __syncthreads();
      if (tid < E) base[tid] = ex;
      __syncthreads();
    }
  }
}

// The same tables for batches of at most TINY_T tokens, by one warp: counts
// with shared-memory atomics, a warp scan for the offsets, then the ranks in
// token order (a running row per expert; equal experts within one token, which
// valid input does not have, are ordered by slot).  A one-token step pays a few
// warp instructions instead of the one-block kernel's passes over 1024 threads.
constexpr int TINY_T = 32;
__global__ void __launch_bounds__(32) permute_tiny_kernel(const int32_t* __restrict__ idx, int T, int E, int k,
                                                          int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ row2tok,
                                                          int32_t* __restrict__ tok2row, int* status) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int cnt[MAX_E];
  __shared__ int run[MAX_E];
  const int lane = threadIdx.x;
  const long long R = (long long)T * k;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  for (int a = lane; a < T * k; a += 32) {
    const int e = idx[a];
    if (e < 0 || e >= E) flag_status(status, DEV_BAD_EXPERT);
    else atomicAdd(&cnt[e], 1);
  }
  __syncwarp();
  // exclusive scan over the experts: each lane sums a contiguous run of them
  const int per = (E + 31) / 32;
  const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
  int mine = 0;
  for (int e = e0; e < e1; ++e) mine += cnt[e];
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int ex = incl - mine;
  for (int e = e0; e < e1; ++e) {
    counts[e] = cnt[e];
    offsets[e] = ex;
    run[e] = ex;
    ex += cnt[e];
  }
  if (lane == 31) offsets[E] = incl;
  __syncwarp();
  // rows in token order; slot order among equal experts of one token
  for (int t = 0; t < T; ++t) {
    for (int j0 = 0; j0 < k; j0 += 32) {
      const int j = j0 + lane;
      const bool act = j < k;
      const int e = act ? idx[(long long)t * k + j] : -1;
      const bool ok = act && e >= 0 && e < E;
      const unsigned m = __match_any_sync(0xffffffffu, ok ? e : -1);
      if (ok) {
        const long long row = (long long)run[e] + __popc(m & ((1u << lane) - 1u));
        if (row < 0 || row >= R) {
          flag_status(status, DEV_BAD_ROW);
          tok2row[(long long)t * k + j] = -1;
        } else {
          row2tok[row] = t;
          tok2row[(long long)t * k + j] = (int32_t)row;
        }
      } else if (act) {
        tok2row[(long long)t * k + j] = -1;
      }
      __syncwarp();
      // the lowest lane of each group of equal experts advances its run
      if (ok && (m & ((1u << lane) - 1u)) == 0u) run[e] += __popc(m);
      __syncwarp();
    }
  }
}


// x_perm[tok2row[t][j]] = x[t] for every slot j: one warp per token reads the
// row once (chunks of 8 vectors per lane) and stores it k times, so x streams
// from memory once and the k copies are plain writes.
constexpr int GATHER_CHUNK = 8;   // 16-byte vectors per lane per chunk

// Eight bf16 values to f16 (round to nearest even); `over` is set when one
// lands beyond the f16 range (|v| >= 65520 rounds to infinity).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, bool& over) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
    over |= fabsf(lo) >= 65520.0f || fabsf(hi) >= 65520.0f;
    const __half2 h = __floats2half2_rn(lo, hi);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// seg warps share a token's row (seg > 1 for small batches, so that more
// than one warp's loads are in flight per row).
__global__ void __launch_bounds__(256) gather_tokens_kernel(const uint4* __restrict__ x,
                                                            const int32_t* __restrict__ tok2row, int T, int k,
                                                            long long R, int vec_per_row, uint4* __restrict__ x_perm,
                                                            int to_f16, int seg, int* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  bool over = false;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const int per = (vec_per_row + seg - 1) / seg;
  for (long long item = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < (long long)T * seg;
       item += warps) {
    const long long t = item / seg;
    const int sg = int(item % seg);
    const int v_begin = sg * per, v_end = min(vec_per_row, v_begin + per);
    const int32_t* rows = tok2row + t * k;
    const uint4* src = x + t * vec_per_row;
    for (int v0 = v_begin; v0 < v_end; v0 += 32 * GATHER_CHUNK) {
      uint4 buf[GATHER_CHUNK];
#pragma unroll
      for (int i = 0; i < GATHER_CHUNK; ++i) {
        const int v = v0 + i * 32 + lane;
        if (v < v_end) buf[i] = src[v];
      }
      if (to_f16) {
        // after all the chunk's loads are in flight
#pragma unroll
        for (int i = 0; i < GATHER_CHUNK; ++i)
          if (v0 + i * 32 + lane < v_end) buf[i] = bf16x8_to_f16x8(buf[i], over);
      }
      for (int j = 0; j < k; ++j) {
        const long long r = rows[j];   // warp-uniform, cached after the first chunk
        if (r < 0) continue;           // an expert index the dispatch already flagged
        if (r >= R) {
          if (lane == 0 && v0 == v_begin && sg == 0) flag_status(status, DEV_BAD_ROW);
          continue;
        }
        uint4* dst = x_perm + r * vec_per_row;
#pragma unroll
        for (int i = 0; i < GATHER_CHUNK; ++i) {
          const int v = v0 + i * 32 + lane;
          if (v < v_end) dst[v] = buf[i];
        }
      }
    }
  }
  if (over) flag_status(status, DEV_RANGE);
}

__global__ void __launch_bounds__(256) bf16_to_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                          long long n_vec, int* status) {
  // heads its call's chain: predecessors complete before dependents start
  pdl_wait();
  pdl_launch_dependents();
  bool over = false;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_vec; i += (long long)gridDim.x * blockDim.x)
    dst[i] = bf16x8_to_f16x8(src[i], over);
  if (over) flag_status(status, DEV_RANGE);
}

}  // namespace

cudaError_t launch_gather_rows(const void* x, const int32_t* tok2row, int T, int k, long long rows, size_t row_bytes,
                               void* x_perm, int* status, cudaStream_t s, int* launches) {
  if (T <= 0) return cudaSuccess;
  long long blocks = (T + 7) / 8;
  const long long cap = 8LL * num_sms();
  if (blocks > cap) blocks = cap;
  cudaError_t e = launch_pdl(gather_tokens_kernel, dim3((int)blocks), dim3(256), 0, s, static_cast<const uint4*>(x),
                             tok2row, T, k, rows, int(row_bytes / 16), static_cast<uint4*>(x_perm), 0, 1, status);
  if (launches) ++*launches;
  return e;
}

cudaError_t launch_bf16_to_f16(const void* src, void* dst, long long n, int* status, cudaStream_t s, int* launches) {
  if (n <= 0) return cudaSuccess;
  const long long n_vec = n / 8;
  long long blocks = (n_vec + 255) / 256;
  const long long cap = 8LL * num_sms();
  if (blocks > cap) blocks = cap;
  cudaError_t e = launch_pdl(bf16_to_f16_kernel, dim3((int)blocks), dim3(256), 0, s, static_cast<const uint4*>(src),
                             static_cast<uint4*>(dst), n_vec, status);
  if (launches) ++*launches;
  return e;
}

int permute_chunks(int T) { return (T + CHUNK - 1) / CHUNK; }
int permute_launches(int T) { return T <= SMALL_T ? 1 : 4; }

cudaError_t launch_permute(const moe_config& c, const void* x, const int32_t* idx, int32_t* counts,
                           int32_t* offsets, int32_t* row2tok, int32_t* tok2row, void* x_perm,
                           int32_t* chunk_counts, int32_t* chunk_base, int* status, cudaStream_t s,
                           int* launches, bool x_perm_f16) {
  const int nch = permute_chunks(c.T);
  if (c.T <= TINY_T && c.E <= MAX_E) {
    cudaError_t e = launch_pdl(permute_tiny_kernel, dim3(1), dim3(32), 0, s, idx, c.T, c.E, c.k, counts, offsets,
                               row2tok, tok2row, status);
    if (launches) *launches += 1;
    if (e != cudaSuccess) return e;
  } else if (c.T <= SMALL_T) {
    cudaError_t e = launch_pdl(permute_small_kernel, dim3(1), dim3(SMALL_BLOCK), 0, s, idx, c.T, c.E, c.k, counts,
                               offsets, row2tok, tok2row, status);
    if (launches) *launches += 1;
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = launch_pdl(permute_count_kernel, dim3(nch), dim3(CHUNK), 0, s, idx, c.T, c.E, c.k, chunk_counts,
                               status);
    if (e == cudaSuccess)
      e = launch_pdl(permute_chunk_scan_kernel, dim3(c.E), dim3(CHUNK), 0, s, chunk_counts, nch, c.E, chunk_base,
                     counts);
    if (e == cudaSuccess) e = launch_pdl(permute_offsets_kernel, dim3(1), dim3(256), 0, s, counts, c.E, offsets);
    if (e == cudaSuccess)
      e = launch_pdl(permute_scatter_kernel, dim3(nch), dim3(CHUNK), 0, s, idx, c.T, c.E, c.k, chunk_base, offsets,
                     row2tok, tok2row, status);
    if (launches) *launches += 4;
    if (e != cudaSuccess) return e;
  }
  if (x == nullptr || x_perm == nullptr) return cudaSuccess;
  const long long R = (long long)c.T * c.k;
  const int vec = int((size_t)c.d * dtype_bytes(c.act_dtype) / 16);
  // small batches: the 8 warps of a block share each token's row
  const int seg = c.T <= 64 ? 8 : 1;
  long long blocks = ((long long)c.T * seg + 7) / 8;
  const long long cap = 8LL * num_sms();
  if (blocks > cap) blocks = cap;
  cudaError_t e = launch_pdl(gather_tokens_kernel, dim3((int)blocks), dim3(256), 0, s, static_cast<const uint4*>(x),
                             tok2row, c.T, c.k, R, vec, static_cast<uint4*>(x_perm), x_perm_f16 ? 1 : 0, seg, status);
  if (launches) ++*launches;
  return e;
}

}  // namespace moe
