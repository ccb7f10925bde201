// Expert FFNs with FP8 weights for decode batches (every group at most
// GEMV_MAX_T token rows): a GEMV over the packed FP8 stage images whose dot
// products run as warp-level MMAs, GEMV_MAX_ROWS token rows at a time.
//
// At a handful of tokens per expert the op is a matrix-vector product bound
// by the weight stream.  The tcgen05 FP8 path pays a per-stage hand-off
// (converter warps of two CTAs -> one MMA issuer -> freed buffer) that caps it
// well below the HBM rate, and FMAs on the CUDA cores cost one instruction per
// weight and token.  Here each CTA streams whole stage images (128 weight rows
// x 128 columns of e4m3 plus their block exponents, one 2-D TMA box) and the
// token rows' 128 matching values (bulk copies) through a ring of shared-memory
// stages; every warp turns its 16 x 64 piece of a stage into f16 (e4m3 -> f16
// is exact) and multiplies it by the token values (f16; the shared expert's
// bf16 x rounded to f16) with four m16n8k16 MMAs, the item's up to 8 token
// rows being the 8 columns of B.  Products of f16 values are exact and the MMA sums them
// in fp32; each 64-column partial times its block's 2^e (exact) is added to
// the fp32 accumulator.  One MMA serves 1 to 8 tokens at the same cost, so the
// instruction count per weight no longer grows with the batch.  The expert
// FFN is w2(silu(w1 x) * w3 x) (intelliparadigm.com page, section 3.3.1) with
// the FP8 block quantisation of its section 4; two launches: GEMM1 with the
// SwiGLU epilogue (f16 hidden rows), then GEMM2 (fp32 rows).
//
// Work items are (group, 128-row weight tile, chunk of up to 8 token rows),
// the shared expert's first: their token rows do not depend on the dispatch,
// so in the GEMM1 launch they stream while the preceding kernels still run;
// the routed groups' items wait for the dispatch (griddepcontrol.wait), after
// which the producer warp lists the groups that received rows and their item
// counts.  A tile's chunks are consecutive items, so the CTAs that take them
// stream the same weights at about the same time and all but one read them
// from L2.  CTA b takes items b, b + G, b + 2G, ...
// (one CTA per SM, a ring of 11 stages: 215 KB of weights and token values in
// flight per SM).  Every wait is bounded; a CTA that gives up flags the status
// word and its roles leave without waiting on each other.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int GV_WARPS = 16;                         // compute warps: 8 row tiles x 2 k-blocks of a stage
constexpr int GV_THREADS = 32 * (GV_WARPS + 1);      // plus the producer warp
constexpr int GV_STAGES = 11;
constexpr int GV_XBYTES = 128 * 2;                   // one token row's 128 values of a stage (2-byte types)
constexpr int GV_XSTRIDE = GV_XBYTES + 16;           // token rows 16 bytes apart in the banks
constexpr int GV_STAGE_BYTES = FP8_STAGE_BYTES + GEMV_MAX_ROWS * GV_XSTRIDE;
constexpr int GV_MAX_GROUPS = 272;
static_assert(GV_STAGE_BYTES % 128 == 0 && GEMV_MAX_ROWS == 8, "stage alignment; one MMA column per token row");

struct GemvClass {
  const uint8_t* w;    // stage images: tiles of 128 rows, nst stages each; group g's first tile is g * tpg
  const uint8_t* x;    // token rows, K 2-byte values each
  int x_f16;           // 1: f16 values, 0: bf16
  void* out;           // GEMM1: f16 [rows, M / 2]; GEMM2: fp32 [rows, M]
  long long out_ld;    // elements per output row
  int tpg;             // 128-row weight tiles per group (M / 128)
  int nst;             // stages per tile (K / 128)
  int K;
};

constexpr int GV_IMG_ROWS = FP8_STAGE_BYTES / 128;   // a stage image as rows of 128 bytes
static_assert(FP8_STAGE_BYTES % 128 == 0 && GV_IMG_ROWS <= 256, "image box");

struct GemvParams {
  CUtensorMap tm[2];   // the classes' stage images as [images * GV_IMG_ROWS][128] bytes, box = one image
  GemvClass cls[2];    // 0: routed, 1: shared
  const int32_t* offsets;   // [num_routed + 1] routed rows of each group
  int num_routed;
  int shared_rows;          // 0: no shared expert
  int max_rows;             // bound of every group's token rows (GEMV_MAX_T or less)
  long long routed_rows;    // bound of every routed row index
  int gemm1;                // 1: SwiGLU epilogue, 0: fp32 rows
  int x_from_prev;          // 1: every item's token rows come from the preceding grid
  int* status;
};

struct GemvCtrl {
  uint64_t full[GV_STAGES];    // a stage's image and token values landed
  uint64_t empty[GV_STAGES];   // every compute warp finished with a stage
  uint64_t list_ready;         // the active-group list is built
  uint64_t sums_full;          // every compute warp wrote its rows' sums
  uint64_t sums_free;          // every compute warp read the sums
  int abort;
  int n_active;
  int active[GV_MAX_GROUPS];     // groups with rows, in index order
  int item_end[GV_MAX_GROUPS];   // routed items of active groups 0 .. i (running sum)
  float sums[2][128][GEMV_MAX_ROWS];   // the tile's row sums of each k-block half, [half][row][token]
};

// Bounded wait with a short sleep between polls, the give-up rule of mbar_wait:
// the compute warps all wait on the same stage barriers, and sleeping leaves
// the issue slots to the producer warp and to the warps still working (the
// T=1 expert stage measured 0.122 against 0.127 ms with back-to-back polls).
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, int* abort_flag, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  volatile int* ab = abort_flag;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    __nanosleep(64);
    if (mbar_try_wait(bar, parity)) return true;
    if (*ab) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *ab = 1;
      flag_status(status, DEV_TIMEOUT);
      return false;
    }
  }
}

struct GemvItem {
  int cls, rows, tile_w;        // class, token rows (<= GEMV_MAX_ROWS), weight tile (of the class's whole matrix)
  int tile;                     // tile within the group
  long long row0;               // first token row (x) and output row
};

// Items of a group with `rows` token rows, per weight tile.
__device__ __forceinline__ int gv_chunks(int rows) { return (rows + GEMV_MAX_ROWS - 1) / GEMV_MAX_ROWS; }

// The shared expert's items (they come first).
__device__ __forceinline__ int gv_shared_items(const GemvParams& p) {
  return p.shared_rows > 0 ? p.cls[1].tpg * gv_chunks(p.shared_rows) : 0;
}

// Item -> operands, or false past the last item.  nsh: the shared expert's
// items.  Within a group, item = tile * chunks + chunk.
__device__ __forceinline__ bool gemv_item(const GemvParams& p, const GemvCtrl* c, int nsh, int item, GemvItem& it) {
  if (item < nsh) {
    const int nch = gv_chunks(p.shared_rows);
    const int tile = item / nch, ch = item - tile * nch;
    it.cls = 1;
    it.tile = tile;
    it.tile_w = tile;
    it.row0 = (long long)ch * GEMV_MAX_ROWS;
    it.rows = min(GEMV_MAX_ROWS, p.shared_rows - ch * GEMV_MAX_ROWS);
    return true;
  }
  const int j = item - nsh;
  const int n = c->n_active;
  if (n == 0 || j >= c->item_end[n - 1]) return false;
  int lo = 0, hi = n - 1;   // the first active group whose items end past j
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (c->item_end[mid] > j) hi = mid;
    else lo = mid + 1;
  }
  const int g = c->active[lo];
  const long long r0 = p.offsets[g];
  const int rows = int(p.offsets[g + 1] - r0);
  const int nch = gv_chunks(rows);
  const int local = j - (lo > 0 ? c->item_end[lo - 1] : 0);
  const int tile = local / nch, ch = local - tile * nch;
  it.cls = 0;
  it.tile = tile;
  it.tile_w = g * p.cls[0].tpg + tile;
  it.row0 = r0 + (long long)ch * GEMV_MAX_ROWS;
  it.rows = min(GEMV_MAX_ROWS, rows - ch * GEMV_MAX_ROWS);
  return true;
}

// Producer warp: lists the routed groups with rows (after the dispatch), then
// lane 0 streams every item's stages.  Returns with all its copies landed.
__device__ void gemv_producer(const GemvParams& p, GemvCtrl* c, uint8_t* ring, int lane) {
  const int nsh = gv_shared_items(p);
  const int G = gridDim.x;
  bool waited = false, listed = false;
  int s = 0;
  uint32_t ph = 0;
  uint32_t used = 0, used_par = 0;
  for (int item = blockIdx.x;; item += G) {
    if ((item >= nsh || p.x_from_prev) && !waited) {
      pdl_wait();   // the dispatch (and, for GEMM2, the hidden rows) come from the preceding grids
      waited = true;
    }
    if (item >= nsh && !listed) {
      // warp-wide scan of the groups: the ones with rows, in index order, and
      // the running count of their items
      int base = 0, items = 0;
      for (int g0 = 0; g0 < p.num_routed; g0 += 32) {
        const int g = g0 + lane;
        int rows = 0;
        if (g < p.num_routed) {
          const long long lo = p.offsets[g], hi = p.offsets[g + 1];
          rows = int(hi - lo);
          if (lo < 0 || hi > p.routed_rows || rows < 0 || rows > p.max_rows) {
            flag_status(p.status, DEV_BAD_ROW);
            rows = 0;
          }
        }
        const uint32_t m = __ballot_sync(0xffffffffu, rows > 0);
        int incl = rows > 0 ? p.cls[0].tpg * gv_chunks(rows) : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        if (rows > 0) {
          const int pos = base + __popc(m & ((1u << lane) - 1u));
          c->active[pos] = g;
          c->item_end[pos] = items + incl;
        }
        base += __popc(m);
        items += __shfl_sync(0xffffffffu, incl, 31);
      }
      __syncwarp();   // every lane's entries are ordered before lane 0's release
      if (lane == 0) {
        c->n_active = base;
        mbar_arrive(&c->list_ready);   // release (CTA): orders the list above
      }
      __syncwarp();
      listed = true;
    }
    GemvItem it;
    if (!gemv_item(p, c, nsh, item, it)) break;
    if (lane == 0) {
      const GemvClass& k = p.cls[it.cls];
      const uint32_t bytes = uint32_t(FP8_STAGE_BYTES + it.rows * GV_XBYTES);
      for (int ks = 0; ks < k.nst; ++ks) {
        if (!mbar_wait(&c->empty[s], ph ^ 1u, &c->abort, p.status)) break;
        uint8_t* st = ring + size_t(s) * GV_STAGE_BYTES;
        mbar_arrive_expect_tx(&c->full[s], bytes);
        tma_load_2d(st, &p.tm[it.cls], &c->full[s], 0, (it.tile_w * k.nst + ks) * GV_IMG_ROWS);
        for (int t = 0; t < it.rows; ++t)
          bulk_load(st + FP8_STAGE_BYTES + t * GV_XSTRIDE,
                    k.x + ((it.row0 + t) * (long long)k.K + (long long)ks * 128) * 2, GV_XBYTES, &c->full[s]);
        used |= 1u << s;
        used_par = (used_par & ~(1u << s)) | (ph << s);
        if (++s == GV_STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&c->abort), 0)) break;
  }
  if (!listed && lane == 0) {
    c->n_active = 0;
    mbar_arrive(&c->list_ready);
  }
  if (lane == 0) {
    // every copy issued here lands before the CTA may leave (bounded)
    const unsigned long long t0 = globaltimer_ns();
    for (int i = 0; i < GV_STAGES; ++i) {
      if (!(used & (1u << i))) continue;
      while (!mbar_try_wait(&c->full[i], (used_par >> i) & 1u))
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
  }
}

// 16 e4m3 values -> 8 f16 pairs (exact: every e4m3 value is an f16 number).
__device__ __forceinline__ void e4m3x16_to_f16x2(const uint4 q, uint32_t* w) {
  const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw a = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(qw[i] & 0xffffu), __NV_E4M3);
    const __half2_raw b = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(qw[i] >> 16), __NV_E4M3);
    w[2 * i] = uint32_t(a.x) | (uint32_t(a.y) << 16);
    w[2 * i + 1] = uint32_t(b.x) | (uint32_t(b.y) << 16);
  }
}

// 16 two-byte token values -> 8 f16 pairs: f16 values as they are; bf16 ones
// rounded to f16 (exact between 2^-14 and 65504; the gather reports values
// beyond the f16 range for FP8 layers).
__device__ __forceinline__ void x16_to_f16x2(const uint8_t* src, bool f16, uint32_t* x) {
  const uint4 a = *reinterpret_cast<const uint4*>(src);
  const uint4 b = *reinterpret_cast<const uint4*>(src + 16);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (f16) {
      x[i] = w[i];
    } else {
      const __half2 h = __floats2half2_rn(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
      x[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
  }
}

// D += A B for one m16n8k16 tile: f16 operands (A row-major 16 x 16, B
// column-major 16 x 8), fp32 accumulators.  Lane (g, t) = (lane / 4, lane % 4)
// holds A rows g and g + 8 at columns 2t, 2t + 1 (a0, a1) and 2t + 8, 2t + 9
// (a2, a3), B column g at rows 2t, 2t + 1 (b0) and 2t + 8, 2t + 9 (b1), and D
// rows g (d0, d1) and g + 8 (d2, d3) at columns 2t, 2t + 1.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^e as a float (exact; normal range directly).
__device__ __forceinline__ float pow2f(int e) {
  return (e >= -126 && e <= 127) ? __int_as_float((e + 127) << 23) : ldexpf(1.0f, e);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

// Weight row of MMA row g (0..7) within a 16-row tile; MMA row g + 8 takes the
// row 8 below.  Lanes 8q .. 8q + 7 of a warp (MMA rows 2q, 2q + 1) then read
// rows whose 128-byte swizzle phases differ by 4, so their 16-byte chunks of a
// k-block land in different banks.
__device__ __forceinline__ int gv_tile_row(int g) { return (g >> 1) + 4 * (g & 1); }

// One stage of a warp's products: weight rows r0 = 16 rt + gv_tile_row(g) and
// r0 + 8 (MMA rows g and g + 8), the 64 columns of k-block kh, and the group's
// token rows as the 8 columns of B (zero beyond `rows`).  Lane (g, t) reads
// 16-byte chunk 4 kh + t of both weight rows and the same 16 columns of token
// row g.  The MMAs take the 64 columns in a permuted order, the same for A and
// B (step s, MMA column slot j of thread t <- column 16 t + 4 s + j), so each
// thread's operands are contiguous in shared memory.  Each row's 64-column sum
// times 2^e of its block is added into acc (d0, d1: row r0; d2, d3: row r0 + 8;
// tokens 2t and 2t + 1).
__device__ __forceinline__ void gemv_stage(const uint8_t* st, int r0, int kh, int g, int t, int rows, bool f16,
                                           float (&acc)[4]) {
  const int r1 = r0 + 8;
  const int c = kh * 4 + t;
  const uint4 q0 = *reinterpret_cast<const uint4*>(st + r0 * 128 + ((c ^ (r0 & 7)) << 4));
  const uint4 q1 = *reinterpret_cast<const uint4*>(st + r1 * 128 + ((c ^ (r1 & 7)) << 4));
  const int32_t* ex = reinterpret_cast<const int32_t*>(st + FP8_IMAGE_BYTES) + kh * 128;
  const float s0 = pow2f(ex[r0]), s1 = pow2f(ex[r1]);
  uint32_t xv[8];
  if (g < rows) {
    x16_to_f16x2(st + FP8_STAGE_BYTES + g * GV_XSTRIDE + c * 32, f16, xv);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) xv[i] = 0u;
  }
  uint32_t w0[8], w1[8];
  e4m3x16_to_f16x2(q0, w0);
  e4m3x16_to_f16x2(q1, w1);
  float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int st4 = 0; st4 < 4; ++st4)
    mma_16816(d, w0[2 * st4], w1[2 * st4], w0[2 * st4 + 1], w1[2 * st4 + 1], xv[2 * st4], xv[2 * st4 + 1]);
  acc[0] = fmaf(d[0], s0, acc[0]);
  acc[1] = fmaf(d[1], s0, acc[1]);
  acc[2] = fmaf(d[2], s1, acc[2]);
  acc[3] = fmaf(d[3], s1, acc[3]);
}

// Compute warps: warp w multiplies row tile rt = w % 8 (16 weight rows of the
// item's 128) by k-block kh = w / 8 of every stage, GV_PER stages per wait (more
// independent MMA chains between synchronisations).  At the item's end the two
// k-block halves of each row meet in shared memory and every compute thread
// takes part in the epilogue.  Every lane waits on each barrier itself
// (bounded) and the warp leaves together when any lane gave up.
constexpr int GV_PER = 4;
__device__ void gemv_compute(const GemvParams& p, GemvCtrl* c, uint8_t* ring, int warp, int lane) {
  const int nsh = gv_shared_items(p);
  const int G = gridDim.x;
  const int rt = warp & 7, kh = warp >> 3;
  const int g = lane >> 2, t = lane & 3;
  const int r0 = rt * 16 + gv_tile_row(g);
  const int tid = warp * 32 + lane;
  bool listed = false;
  int s = 0;
  uint32_t ph = 0;
  uint32_t n1 = 0;   // items done (parity of the sums barriers)
  for (int item = blockIdx.x;; item += G) {
    if (item >= nsh && !listed) {
      if (!__all_sync(0xffffffffu, mbar_wait(&c->list_ready, 0u, &c->abort, p.status))) return;
      listed = true;
    }
    GemvItem it;
    if (!gemv_item(p, c, nsh, item, it)) return;
    const GemvClass& k = p.cls[it.cls];
    const bool f16 = k.x_f16 != 0;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int ks = 0; ks < k.nst; ks += GV_PER) {
      const int n = min(GV_PER, k.nst - ks);
      int si[GV_PER];
      uint32_t pi[GV_PER];
      si[0] = s;
      pi[0] = ph;
#pragma unroll
      for (int j = 1; j < GV_PER; ++j) {
        si[j] = si[j - 1] + 1 == GV_STAGES ? 0 : si[j - 1] + 1;
        pi[j] = si[j - 1] + 1 == GV_STAGES ? pi[j - 1] ^ 1u : pi[j - 1];
      }
      bool got = true;
#pragma unroll
      for (int j = 0; j < GV_PER; ++j)
        if (j < n) got = got && mbar_wait_sleep(&c->full[si[j]], pi[j], &c->abort, p.status);
      if (!__all_sync(0xffffffffu, got)) return;
      if (n == GV_PER) {
#pragma unroll
        for (int j = 0; j < GV_PER; ++j)
          gemv_stage(ring + size_t(si[j]) * GV_STAGE_BYTES, r0, kh, g, t, it.rows, f16, acc);
      } else {
        for (int j = 0; j < n; ++j)
          gemv_stage(ring + size_t(si[j]) * GV_STAGE_BYTES, r0, kh, g, t, it.rows, f16, acc);
      }
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < GV_PER; ++j)
          if (j < n) mbar_arrive(&c->empty[si[j]]);
      }
      // advance past the n stages
      for (int j = 0; j < n; ++j) {
        if (++s == GV_STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    // the two k-block halves of every row meet in shared memory (bounded barrier waits)
    if (!__all_sync(0xffffffffu, mbar_wait(&c->sums_free, (n1 & 1u) ^ 1u, &c->abort, p.status))) return;
    *reinterpret_cast<float2*>(&c->sums[kh][r0][2 * t]) = make_float2(acc[0], acc[1]);
    *reinterpret_cast<float2*>(&c->sums[kh][r0 + 8][2 * t]) = make_float2(acc[2], acc[3]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&c->sums_full);
    if (!__all_sync(0xffffffffu, mbar_wait(&c->sums_full, n1 & 1u, &c->abort, p.status))) return;
    if (!p.gemm1) {
      float* out = static_cast<float*>(k.out);
      for (int i = tid; i < 128 * it.rows; i += 32 * GV_WARPS) {
        const int r = i & 127, tk = i >> 7;
        out[(it.row0 + tk) * k.out_ld + it.tile * 128 + r] = c->sums[0][r][tk] + c->sums[1][r][tk];
      }
    } else {
      // GEMM1: rows come in blocks of 32 (16 W1 rows of 16 features, then their W3 rows)
      bool over = false;
      __half* out = static_cast<__half*>(k.out);
      for (int i = tid; i < 64 * it.rows; i += 32 * GV_WARPS) {
        const int f = i & 63, tk = i >> 6;
        const int r1 = (f >> 4) * 32 + (f & 15);
        const float gv = c->sums[0][r1][tk] + c->sums[1][r1][tk];
        const float uv = c->sums[0][r1 + 16][tk] + c->sums[1][r1 + 16][tk];
        const float hv = silu_f(gv) * uv;
        over |= fabsf(hv) >= 65520.0f;
        out[(it.row0 + tk) * k.out_ld + it.tile * 64 + f] = __float2half_rn(hv);
      }
      if (over) flag_status(p.status, DEV_RANGE);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&c->sums_free);
    ++n1;
  }
}

__global__ void __launch_bounds__(GV_THREADS, 1) gemv_fp8_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  GemvCtrl* c = reinterpret_cast<GemvCtrl*>(ring + size_t(GV_STAGES) * GV_STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < GV_STAGES; ++i) {
      mbar_init(&c->full[i], 1);
      mbar_init(&c->empty[i], GV_WARPS);
    }
    mbar_init(&c->list_ready, 1);
    mbar_init(&c->sums_full, GV_WARPS);
    mbar_init(&c->sums_free, GV_WARPS);
    c->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  if (warp == GV_WARPS) gemv_producer(p, c, ring, lane);
  else gemv_compute(p, c, ring, warp, lane);
}

constexpr size_t kGemvSmem = 128 + size_t(GV_STAGES) * GV_STAGE_BYTES + sizeof(GemvCtrl);
static_assert(kGemvSmem <= 232448, "shared memory of one CTA");

}  // namespace

cudaError_t launch_fp8_gemv(const GemvOperands& routed, const GemvOperands* shared, const int32_t* offsets,
                            int num_routed, int shared_rows, int max_rows, long long routed_rows, bool gemm1,
                            bool x_from_prev, int* status, cudaStream_t stream, int* launches) {
  if (num_routed < 1 || num_routed > GV_MAX_GROUPS || offsets == nullptr) return cudaErrorInvalidValue;
  if (max_rows < 1 || max_rows > GEMV_MAX_T || shared_rows > max_rows) return cudaErrorInvalidValue;
  if ((shared == nullptr) != (shared_rows <= 0)) return cudaErrorInvalidValue;
  GemvParams p;
  memset(&p, 0, sizeof(p));
  const GemvOperands* ops[2] = {&routed, shared};
  for (int i = 0; i < 2; ++i) {
    const GemvOperands* o = ops[i] != nullptr ? ops[i] : ops[0];
    if (o->M % 128 != 0 || o->K % 128 != 0 || o->M <= 0 || o->K <= 0) return cudaErrorInvalidValue;
    if (reinterpret_cast<uintptr_t>(o->w) % 16 != 0 || reinterpret_cast<uintptr_t>(o->x) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(o->out) % 16 != 0 || (!gemm1 && o->out_ld % 4 != 0))
      return cudaErrorInvalidValue;
    GemvClass& k = p.cls[i];
    k.w = static_cast<const uint8_t*>(o->w);
    k.x = static_cast<const uint8_t*>(o->x);
    k.x_f16 = o->x_f16 ? 1 : 0;
    k.out = o->out;
    k.out_ld = o->out_ld;
    k.tpg = o->M / 128;
    k.nst = o->K / 128;
    k.K = o->K;
  }
  // each class's images as a 2-D byte tensor, one box per image (no swizzle:
  // the images are stored in their shared-memory layout)
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorInvalidValue;
  for (int i = 0; i < 2; ++i) {
    const GemvOperands* o = ops[i] != nullptr ? ops[i] : ops[0];
    const long long groups = (i == 0 || ops[i] == nullptr) ? num_routed : 1;
    const long long rows = groups * (o->M / 128) * (o->K / 128) * GV_IMG_ROWS;
    if (rows >= (1LL << 31)) return cudaErrorInvalidValue;
    cuuint64_t dims[2] = {128u, cuuint64_t(rows)};
    cuuint64_t strides[1] = {128u};
    cuuint32_t box[2] = {128u, cuuint32_t(GV_IMG_ROWS)};
    cuuint32_t es[2] = {1u, 1u};
    if (enc(&p.tm[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(o->w), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  p.offsets = offsets;
  p.num_routed = num_routed;
  p.shared_rows = shared != nullptr ? shared_rows : 0;
  p.max_rows = max_rows;
  p.routed_rows = routed_rows;
  p.gemm1 = gemm1 ? 1 : 0;
  p.x_from_prev = x_from_prev ? 1 : 0;
  p.status = status;
  static PerDevice<int> attr;
  int ok = 0;
  cudaError_t e = attr.get(&ok, [](int* v) {
    *v = 1;
    return cudaFuncSetAttribute(gemv_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kGemvSmem));
  });
  if (e != cudaSuccess) return e;
  e = launch_pdl(gemv_fp8_kernel, dim3(num_sms()), dim3(GV_THREADS), kGemvSmem, stream, p);
  if (e == cudaSuccess && launches) ++*launches;
  return e;
}

}  // namespace moe
