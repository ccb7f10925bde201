// Expert GEMMs of the routed and shared SwiGLU experts on CTA pairs
// (tcgen05.mma.cta_group::2 + TMEM + TMA): both GEMMs of the expert FFN in one
// persistent launch, the SwiGLU fused into the first one's epilogue.
//
// The expert FFN is w2(silu(w1 x) * w3 x) (intelliparadigm.com page, section
// 3.3.1); the MoE listing of the DeepSeek-V2 walkthrough runs it per expert on
// the rows routed to that expert, plus the shared experts on every token.
//
// Operand roles are swapped with respect to the layer's "tokens x weights^T":
//
//   D[f][j] = sum_k W[f][k] * X[j][k]
//     W: 256 weight rows of one group (M, split 128/128 over the CTA pair)
//     X: up to 256 token rows of the same group (N, split N/2 per CTA)
//
// so the ragged dimension (tokens per expert) is the MMA's N, which comes in
// steps of 16: a group of n tokens costs ceil(n/16)*16 columns of tensor work.
// The pair shares each token tile between its two SMs.
//
//   phase 1 (GEMM1): W = packed W1/W3 rows interleaved in blocks of 16 (rows
//     32q..32q+15 of a CTA's 128 hold W1 features, 32q+16..32q+31 the W3 rows
//     of the same features), X = token rows; the epilogue pairs lane l with
//     lane l+16 by a warp shuffle and stores H[token][f] = silu(g)*u in bf16.
//   phase 2 (GEMM2): W = W2 rows, X = H rows; Y[token][f] in fp32.
//
// Tiles are numbered [GEMM1 shared][GEMM2 shared][GEMM1 routed][GEMM2 routed]
// and handed out in that order at run time: a dispatcher warp of each cluster
// draws the next tile number from a global ticket counter whenever a slot of
// its cluster's tile ring frees up, and every role of both CTAs takes the
// cluster's tiles from that ring in order.  An idle cluster so takes the next
// tile wherever it is, and only running clusters hold tiles.  A GEMM2 tile of
// a group waits on a per-group counter that every CTA bumps (release) after
// storing its part of a GEMM1 tile of that group, so GEMM2 work starts expert
// by expert while other clusters still run GEMM1 tiles.  A group's GEMM1
// tickets are all drawn before its GEMM2 tickets, by clusters that are running
// and that finish those tiles without waiting on anything drawn later, so the
// waits resolve whether or not every cluster of the grid is resident at once.
// The shared expert's tiles read only x and their own hidden rows, so the
// whole shared FFN may run before the preceding kernels of the same layer call
// (router, dispatch) complete (programmatic dependent launch): those kernels
// touch neither, and the completion counters were cleared with the call's
// status word before any of its kernels started.  Early starts never reach further back: every call of the
// library begins with an ordinary stream operation (clearing its status word),
// which starts only after all earlier work in the stream has completed, so a
// previous call that still reads the hidden rows, or a previous layer that
// writes x, has finished.  Routed tiles wait for the routed tile table, which
// a scheduler warp builds from the dispatch offsets once the dispatch has
// completed.
//
// Each TMA copy moves two k-blocks (3-D tensor maps: 64 columns x rows x 2
// k-blocks): a copy instruction has a fixed cost in the copy engine, so fewer,
// larger copies raise the rate at which an SM's shared memory fills.
//
// CTA layout (256 threads, one CTA per SM, clusters of two CTAs):
//   warp 0      TMA producer of this CTA's halves (3-stage ring of 2 k-blocks,
//               128-byte swizzle); completion bytes count on rank 0's barrier
//   warp 1      tensor-memory allocation (both CTAs); on rank 0 one thread
//               issues the M=256 MMAs and commits to both CTAs' barriers
//   warps 2..5  epilogue: tcgen05.ld of this CTA's 128 accumulator rows
//   warp 6      routed tile tables (from the dispatch offsets)
//   warp 7      rank 0: tile dispatcher (ticket counter -> tile ring)
//   warps 8..23 FP8 weights only (768 threads): converter warps that turn
//               each stage's e4m3 weight image into the bf16 A operand (in
//               shared memory, or in tensor memory for decode-sized launches)
// Two accumulators per CTA (256 columns each; 64 for FP8 decode-sized
// launches) let the epilogue overlap the next tile's main loop.  Every wait
// is bounded; a CTA that gives up flags the status word and tells its peer to
// stop too.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int PM = 128;               // weight rows per CTA
constexpr int PAIR_M = 2 * PM;        // weight rows per pair tile
constexpr int PN = 256;               // token columns per pair tile at most
constexpr int XB = PN / 2;            // token rows loaded by each CTA
constexpr int BK = 64;                // K of one k-block (one 128-byte swizzle row)
constexpr int KB_STAGE = 2;           // k-blocks per stage and per TMA copy
// Ring geometry.  Regular launches: 3 stages of 64 KB (weights 32 KB + tokens
// 32 KB per CTA).  Decode-sized launches (every group at most 64 tokens, so
// every tile uses the 32-row token box): 5 stages of 40 KB, a deeper queue of
// weight copies for streaming-bound work; at most 16 tokens (the 8-row box):
// 6 stages of 34 KB.  A cluster streams about (weights in flight) / (DRAM
// latency under load), so the depth of the queue sets its rate.
constexpr int MAX_STAGES = 6;
constexpr int THREADS = 256;
constexpr int TABLE_WARP = 6;
constexpr int DISPATCH_WARP = 7;
constexpr int TILE_RING = 4;         // tile numbers a cluster holds ahead of its slowest role
constexpr int A_KB_BYTES = PM * BK * 2;          // one k-block of this CTA's weight rows
constexpr int B_KB_BYTES = XB * BK * 2;          // one k-block of this CTA's token rows
constexpr int A_BYTES = KB_STAGE * A_KB_BYTES;
constexpr int B_BYTES = KB_STAGE * B_KB_BYTES;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int RING_BYTES = 216 * 1024;
constexpr int XSMALL = 32;                       // token rows of the small box (decode-sized tiles)
constexpr int XS_KB_BYTES = XSMALL * BK * 2;
constexpr int XTINY = 8;                         // token rows of the tiny box (tiles of at most 16 tokens)
constexpr int XT_KB_BYTES = XTINY * BK * 2;
constexpr int SMALL_STAGE_BYTES = A_BYTES + KB_STAGE * XS_KB_BYTES;
constexpr int TINY_STAGE_BYTES = A_BYTES + KB_STAGE * XT_KB_BYTES;
static_assert(3 * STAGE_BYTES <= RING_BYTES && 5 * SMALL_STAGE_BYTES <= RING_BYTES &&
                  MAX_STAGES * TINY_STAGE_BYTES <= RING_BYTES && TINY_STAGE_BYTES % 1024 == 0 &&
                  SMALL_STAGE_BYTES % 1024 == 0,
              "ring");
constexpr int MAX_GROUPS = 272;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_STRIDE = 256;  // columns between the two accumulators
// FP8 decode-sized launches keep the converted A operand in tensor memory:
// accumulators of at most 64 columns (tiles of at most 64 tokens), then
// A_TMEM_STAGES buffers of 64 columns (128 rows x 128 bf16 each).
constexpr uint32_t ACC_STRIDE_SMALL = 64;
constexpr uint32_t A_TMEM_COL0 = 2 * ACC_STRIDE_SMALL;
constexpr int A_TMEM_STAGES = 4;
static_assert(A_TMEM_COL0 + 64 * A_TMEM_STAGES <= TMEM_COLS, "tensor memory budget");
constexpr int EPI_WARPS = 4;
// FP8 weights: converter warps dequantize each stage's e4m3 weight image into
// the bf16 A buffer, four threads per weight row (32 weights each).  A slot of
// the FP8 ring holds up to two consecutive stages of one tile: their weight
// images (one bulk copy; FP8_STAGE_BYTES each, a multiple of 1024 as the
// swizzled operand reads need) and then their token tiles.
constexpr int CONV_WARPS = 16;
constexpr int THREADS_FP8 = THREADS + 32 * CONV_WARPS;
constexpr int CONV_TPR = CONV_WARPS * 32 / PM;   // converter threads per weight row
constexpr int CONV_CPT = 8 / CONV_TPR;           // 16-weight chunks of a stage row per thread
static_assert(FP8_IMAGE_BYTES == PM * 128 && FP8_STAGE_BYTES % 1024 == 0 && CONV_TPR * CONV_CPT == 8 &&
                  CONV_CPT <= 4,
              "converter geometry");
constexpr int MAX_F8 = 6;           // slots
constexpr int MAX_SPS = 2;          // stages per slot
constexpr int MAX_FULL = MAX_F8 * MAX_SPS > MAX_STAGES ? MAX_F8 * MAX_SPS : MAX_STAGES;

// Operand classes: GEMM1 routed, GEMM1 shared, GEMM2 routed, GEMM2 shared.
constexpr int C1R = 0, C1S = 1, C2R = 2, C2S = 3, NCLS = 4;

struct PairParams {
  CUtensorMap tmW[NCLS];     // weights: 64 x 128 rows x 2 k-blocks
  CUtensorMap tmX[NCLS];     // tokens: 64 x 128 rows x 2 k-blocks
  CUtensorMap tmXs[NCLS];    // tokens: 64 x 32 rows x 2 k-blocks
  CUtensorMap tmXt[NCLS];    // tokens: 64 x 8 rows x 2 k-blocks
  void* out[NCLS];
  long long ld_out[NCLS];
  long long out_rows[NCLS];
  int M[NCLS];          // weight rows of one group (GEMM1: 2 x hidden, GEMM2: d)
  int K[NCLS];          // reduction length (multiple of 64)
  int w_step[NCLS];     // weight rows between consecutive groups of the class
  const int32_t* offsets;
  int num_routed;
  int shared_rows;      // tokens of the shared expert (0: none)
  int phases;           // bit 0: GEMM1 tiles, bit 1: GEMM2 tiles in this launch
  int* done;            // [num_routed + 1] GEMM1 completion counters, zero at launch (both phases only)
  int* ticket;          // tile ticket counter of this launch, zero at launch
  int* status;
  int stages;           // ring depth (3, or MAX_STAGES for decode-sized launches; FP8: bf16 A buffers)
  int stage_bytes;      // bytes of one stage in this CTA's shared memory (FP8: of one A buffer)
  // FP8 weights
  const void* wimg[NCLS];   // FP8 stage images of the class's weights
  int nf;                   // FP8 slots
  int sps;                  // FP8 stages per slot (1 or 2)
  int f8_off;               // byte offset of the slot ring
  int slot_bytes;           // bytes of one slot
  int x_kb_bytes;           // bytes of one k-block of the largest token box of the launch
  int a_tmem;               // FP8: the converted A operand lives in tensor memory (A_TMEM_STAGES buffers)
  // FP8: per group the reference exponents of its W1, W3 and W2 ([num_routed
  // + 1][3], the shared expert last), and per class whether its operands are
  // f16 (weights dequantized relative to the reference exponent, token rows
  // f16, accumulator scaled by 2^e_ref) or bf16 (full block scales; the
  // shared expert's GEMM1, which reads the bf16 x).
  const int32_t* eref;
  int f16op[NCLS];
  uint32_t acc_stride;      // tensor-memory columns between the two accumulators
  // Limit of every bounded wait (ns of %globaltimer), and completions a GEMM2
  // tile waits for beyond its group's GEMM1 tiles (0; a positive value makes
  // those waits run out: host-side fault injection for tests).
  unsigned long long wait_ns;
  int need_extra;
  // Operand layouts beyond the forward's (all zero there).  a_mn / b_mn: the
  // weight (A) / token (B) operand is MN-major, read through a 2-D map over
  // [K rows][M or N columns] in boxes of 64 x 128 (a transposed view of a
  // row-major buffer).  MN-major A: group g's K rows start at g * a_kstep, and
  // K indices from K1 on come from tmW2 (a second matrix: K concatenated).
  int a_mn[NCLS];
  int b_mn[NCLS];
  int K1[NCLS];
  int a_kstep[NCLS];
  CUtensorMap tmW2[NCLS];
  // kmode = 1: the reduction runs over each group's token rows (K of group g
  // = offsets[g+1] - offsets[g] rows from offsets[g], a multiple of 128, zero
  // rows allowed), every group has N[cls] columns, and the routed class's
  // output moves out_gstride elements per group (weight gradients).
  int kmode;
  int N[NCLS];
  int b_col0[NCLS];          // MN-major B: first column of the class's N range in its buffer
  long long out_gstride[NCLS];
  // Token rows of group g start at row_base[g] when given (a padded layout),
  // else at offsets[g]; row_bound bounds every group's rows.
  const int32_t* row_base;
  long long row_bound;
  // bf16 stage blocks (w_img): the weight map is 4-D {64, 128 rows, 2 k-blocks,
  // blocks}; group g's row tile tr and stage s is block (g * w_tpg + tr) * w_nst + s.
  int w_img[NCLS];
  int w_tpg[NCLS];
  int w_nst[NCLS];
};

struct PairCtrl {
  uint64_t full[MAX_FULL];     // rank 0: both CTAs' operands of a stage are ready
  uint64_t empty[MAX_STAGES];  // each CTA: the MMAs that read a stage (FP8: an A buffer) completed
  uint64_t tfull[2];         // each CTA: an accumulator buffer is complete
  uint64_t tempty[2];        // rank 0: both CTAs' epilogues drained a buffer
  uint64_t drain;            // rank 0: every issued MMA completed
  uint64_t f8_full[MAX_F8];  // FP8: a slot's weight images landed (this CTA)
  uint64_t f8_empty[MAX_F8]; // FP8: the MMAs that read a slot completed (this CTA)
  uint64_t tile_full[TILE_RING];    // each CTA: the dispatcher wrote a tile number into the slot
  uint64_t tile_empty[TILE_RING];   // rank 0: every role of both CTAs read the slot
  int tile_ring[TILE_RING];         // tile number, or -1: no more tiles
  uint32_t tmem_base;
  int abort;
  unsigned long long wait_ns;   // copy of PairParams::wait_ns
  int seg[5];                // tile numbers where the four segments start, and the total
  int routed_ready;          // the routed tile tables (and seg[3..4]) are built
  int tile_start[2][MAX_GROUPS + 1];   // per phase: exclusive prefix of routed tiles
  int row_start[MAX_GROUPS];
  int rows[MAX_GROUPS];
};

constexpr size_t kPairSmem = 1024 + size_t(RING_BYTES) + sizeof(PairCtrl);
static_assert(kPairSmem <= 227 * 1024, "shared memory budget");
// More than half of an SM's shared memory: one CTA per SM, so the full
// tensor-memory allocation never waits on another resident CTA.
static_assert(kPairSmem > 114 * 1024, "one CTA per SM");

struct PairTile {
  int cls;       // operand class (C1R, C1S, C2R, C2S)
  int g;         // group: routed expert, or num_routed for the shared expert
  int fb, tb, row_start, rows;
  int n_valid;   // token rows of this tile
  int n_mma;     // MMA N = n_valid rounded up to 16
  int n0;        // first N index of the tile (token row, or column in kmode)
  int k0;        // first K index (kmode: the group's first token row)
  int nks;       // stages of 128 K
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Token box of a tile: this CTA's n_mma / 2 rows fit the tiny (8), small (32)
// or full (128) box; one k-block of it in shared memory takes the returned bytes.
__device__ __forceinline__ int x_kb_bytes(int n_mma) {
  return n_mma / 2 <= XTINY ? XT_KB_BYTES : (n_mma / 2 <= XSMALL ? XS_KB_BYTES : B_KB_BYTES);
}
__device__ __forceinline__ const CUtensorMap* x_map(const PairParams& p, int cls, int n_mma) {
  return n_mma / 2 <= XTINY ? &p.tmXt[cls] : (n_mma / 2 <= XSMALL ? &p.tmXs[cls] : &p.tmX[cls]);
}

// Tiles of a group with `rows` token rows: token blocks x weight blocks (in
// kmode the N extent is fixed and the rows are the reduction).
__device__ __forceinline__ int pair_group_tiles(const PairParams& p, int cls, int rows) {
  return cdiv(p.kmode ? p.N[cls] : rows, PN) * cdiv(p.M[cls], PAIR_M);
}

// GEMM1 counter value at which a group's hidden rows are complete: every
// epilogue warp of both CTAs bumps it once per GEMM1 tile of the group.
__device__ __forceinline__ int gemm1_need(const PairParams& p, int cls1, int rows) {
  return 2 * EPI_WARPS * pair_group_tiles(p, cls1, rows) + p.need_extra;
}

// Warp-cooperative: row ranges of the routed groups (from the dispatch
// offsets), the exclusive prefix of their tiles in both phases, and the
// segment boundaries that depend on them.
__device__ void pair_schedule(PairCtrl* c, const PairParams& p, int lane) {
  const int ng = p.num_routed;
  const int per = cdiv(ng, 32);
  const int lo = min(ng, lane * per), hi = min(ng, lo + per);
  int local1 = 0, local2 = 0;
  for (int g = lo; g < hi; ++g) {
    int rows = p.offsets[g + 1] - p.offsets[g];
    int rs = p.row_base != nullptr ? p.row_base[g] : p.offsets[g];
    if (rows < 0 || rs < 0 || (long long)rs + rows > p.row_bound || (p.kmode && (rows & 127))) {
      flag_status(p.status, DEV_BAD_ROW);
      rs = 0;
      rows = 0;
    }
    c->row_start[g] = rs;
    c->rows[g] = rows;
    local1 += pair_group_tiles(p, C1R, rows);
    local2 += pair_group_tiles(p, C2R, rows);
  }
  int incl1 = local1, incl2 = local2;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v1 = __shfl_up_sync(0xffffffffu, incl1, o);
    const int v2 = __shfl_up_sync(0xffffffffu, incl2, o);
    if (lane >= o) {
      incl1 += v1;
      incl2 += v2;
    }
  }
  int run1 = incl1 - local1, run2 = incl2 - local2;
  for (int g = lo; g < hi; ++g) {
    c->tile_start[0][g] = run1;
    c->tile_start[1][g] = run2;
    run1 += pair_group_tiles(p, C1R, c->rows[g]);
    run2 += pair_group_tiles(p, C2R, c->rows[g]);
  }
  if (lane == 31) {
    c->tile_start[0][ng] = incl1;
    c->tile_start[1][ng] = incl2;
    // seg[0..2] (the shared expert's segments) were set at start-up
    const bool g1 = p.phases & 1, g2 = p.phases & 2;
    c->seg[3] = c->seg[2] + (g1 ? incl1 : 0);
    c->seg[4] = c->seg[3] + (g2 ? incl2 : 0);
  }
}

// Tile number -> class, group, weight block and token block.  Within a group
// the block order keeps the operand that is re-read the most resident in L2:
// with more token blocks than weight blocks the token block is the outer loop
// (its rows are re-used by every weight block), otherwise the weight block is.
__device__ __forceinline__ PairTile pair_tile(const PairCtrl* c, const PairParams& p, int tile) {
  PairTile t;
  int local;
  int seg = 0;
  if (tile >= c->seg[1]) seg = tile < c->seg[2] ? 1 : (tile < c->seg[3] ? 2 : 3);
  local = tile - c->seg[seg];
  if (seg < 2) {
    t.cls = seg == 0 ? C1S : C2S;
    t.g = p.num_routed;
    t.row_start = 0;
    t.rows = p.shared_rows;
  } else {
    const int ph = seg == 2 ? 0 : 1;
    const int* ts = c->tile_start[ph];
    int lo = 0, hi = p.num_routed - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ts[mid] <= local) lo = mid;
      else hi = mid - 1;
    }
    t.cls = ph == 0 ? C1R : C2R;
    t.g = lo;
    t.row_start = c->row_start[lo];
    t.rows = c->rows[lo];
    local -= ts[lo];
  }
  const int ncols = p.kmode ? p.N[t.cls] : t.rows;   // N extent of the group
  const int tbn = cdiv(ncols, PN), fbn = cdiv(p.M[t.cls], PAIR_M);
  if (tbn > fbn) {
    t.tb = local / fbn;
    t.fb = local % fbn;
  } else {
    t.fb = local / tbn;
    t.tb = local % tbn;
  }
  t.n_valid = min(PN, ncols - t.tb * PN);
  t.n_mma = (t.n_valid + 15) & ~15;
  t.n0 = (p.kmode ? 0 : t.row_start) + t.tb * PN;
  t.k0 = p.kmode ? t.row_start : 0;
  t.nks = p.kmode ? t.rows / 128 : (p.K[t.cls] / BK + KB_STAGE - 1) / KB_STAGE;
  return t;
}

// Bounded wait on the routed tile tables (built by the scheduler warp once
// the dispatch has completed).  Returns false when it gave up.
__device__ __forceinline__ bool wait_routed_ready(PairCtrl* c, int* status) {
  volatile int* ready = &c->routed_ready;
  if (!*ready) {
    const unsigned long long t0 = globaltimer_ns();
    while (!*ready) {
      if (*reinterpret_cast<volatile int*>(&c->abort)) return false;
      if (globaltimer_ns() - t0 > c->wait_ns) {
        c->abort = 1;
        flag_status(status, DEV_TIMEOUT);
        return false;
      }
      __nanosleep(64);
    }
  }
  __threadfence_block();
  return true;
}

// Position in a ring of n barriers/buffers and the parity of its current use,
// advanced one step at a time (no division on the per-stage path).
struct RingPos {
  int i = 0;
  uint32_t par = 0;
  __device__ __forceinline__ void next(int n) {
    if (++i == n) {
      i = 0;
      par ^= 1u;
    }
  }
};

// Bounded wait; on giving up it flags the status word and stops both CTAs.
// It also gives up as soon as this CTA has been told to stop, unless
// honor_abort is false (the final waits for this CTA's own copies and MMAs,
// which complete whatever else happened).
__device__ __forceinline__ bool pair_wait(uint64_t* bar, uint32_t parity, PairCtrl* c, uint32_t peer_abort,
                                          int* status, bool cluster_scope = false, bool honor_abort = true) {
  if (cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  volatile int* ab = &c->abort;
  const unsigned long long t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if ((++n & 63u) == 0u) {
      if (honor_abort && *ab) return false;
      if (globaltimer_ns() - t0 > c->wait_ns) {
        *ab = 1;
        st_remote_u32(peer_abort, 1u);
        flag_status(status, DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// Roles that take tiles from the ring: per CTA the producer thread, the
// epilogue warps and the FP8 converter warps, plus the MMA issuer on rank 0.
__host__ __device__ constexpr int tile_readers(bool fp8) { return 2 * (1 + EPI_WARPS + (fp8 ? CONV_WARPS : 0)) + 1; }

// Rank 0's dispatcher thread: whenever a ring slot is free (every reader of
// both CTAs took its last tile number), draw the next ticket from the
// launch's counter and publish it to both CTAs (-1 once the tiles run out).
__device__ void pair_dispatch(PairCtrl* c, const PairParams& p, uint32_t peer_abort) {
  RingPos slot;
  const uint32_t peer_ring = map_to_rank(smem_u32(&c->tile_ring[0]), 1);
  const uint32_t peer_full = map_to_rank(smem_u32(&c->tile_full[0]), 1);
  while (true) {
    if (!pair_wait(&c->tile_empty[slot.i], slot.par ^ 1u, c, peer_abort, p.status, true)) return;
    int t = atomicAdd(p.ticket, 1);
    // tiles past the shared expert's are counted by the routed tables
    if (t >= c->seg[2] && (!wait_routed_ready(c, p.status) || t >= c->seg[4])) t = -1;
    c->tile_ring[slot.i] = t;
    st_remote_u32(peer_ring + 4u * uint32_t(slot.i), uint32_t(t));
    mbar_arrive_remote(peer_full + 8u * uint32_t(slot.i));   // release (cluster): orders the store above
    mbar_arrive(&c->tile_full[slot.i]);
    if (t < 0) return;
    slot.next(TILE_RING);
  }
}

// The cluster's next tile number from the ring (position r), or -1 when the
// tiles ran out or this CTA stopped.  Frees the slot on rank 0.
__device__ int next_tile(PairCtrl* c, const PairParams& p, RingPos& r, uint32_t peer_abort) {
  if (!pair_wait(&c->tile_full[r.i], r.par, c, peer_abort, p.status, true)) return -1;
  const int t = *reinterpret_cast<volatile int*>(&c->tile_ring[r.i]);
  mbar_arrive_remote(map_to_rank(smem_u32(&c->tile_empty[r.i]), 0));
  r.next(TILE_RING);
  if (t >= c->seg[2] && !wait_routed_ready(c, p.status)) return -1;
  return t;
}

// A GEMM2 tile of group t.g needs the group's hidden rows: wait (acquire, GPU
// scope) until every epilogue warp of every GEMM1 tile of the group has
// published its part.  Returns false when the wait gave up or the CTA stopped.
__device__ bool wait_gemm1_done(PairCtrl* c, const PairParams& p, const PairTile& t, uint32_t peer_abort) {
  const int need = gemm1_need(p, t.cls == C2R ? C1R : C1S, t.rows);
  const unsigned long long t0 = globaltimer_ns();
  while (ld_acquire_gpu(p.done + t.g) < need) {
    if (*reinterpret_cast<volatile int*>(&c->abort)) return false;
    if (globaltimer_ns() - t0 > c->wait_ns) {
      c->abort = 1;
      st_remote_u32(peer_abort, 1u);
      flag_status(p.status, DEV_TIMEOUT);
      return false;
    }
    __nanosleep(128);
  }
  fence_proxy_async_global();   // the copy engine reads what the acquire made visible
  return true;
}

// Before a producer leaves, every copy it issued into its ring must have
// landed.  The last use of each ring position (bit s of `used`, parity bit s
// of `par`) completes once the MMAs consumed it, which on the normal path has
// happened or soon will.  After a stop some positions are never consumed;
// the wait then ends after min(limit, kDrainAfterStopNs), far longer than a
// copy takes to land, so no copy still lands once the CTA has left.
constexpr unsigned long long kDrainAfterStopNs = 1000000ull;
__device__ void pair_drain(uint64_t* bars, int n, uint32_t used, uint32_t par, PairCtrl* c) {
  const unsigned long long t0 = globaltimer_ns();
  for (int s = 0; s < n; ++s) {
    if (!(used & (1u << s))) continue;
    while (!mbar_try_wait(&bars[s], (par >> s) & 1u)) {
      const unsigned long long dt = globaltimer_ns() - t0;
      const bool stopped = *reinterpret_cast<volatile int*>(&c->abort) != 0;
      if (dt > c->wait_ns || (stopped && dt > kDrainAfterStopNs)) return;
    }
  }
}

__device__ void pair_producer(PairCtrl* c, const PairParams& p, uint8_t* stages, uint32_t rank,
                              uint32_t peer_abort) {
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0, issued_par = 0;
  bool ok = true;
  bool waited = false;
  int ready_group = -1;   // GEMM2 group whose hidden rows are known complete
  RingPos tr;
  while (ok) {
    const int tile = next_tile(c, p, tr, peer_abort);
    if (tile < 0) break;
    const PairTile t = pair_tile(c, p, tile);
    if (t.cls == C1R && !waited) {
      pdl_wait();   // the permuted token rows come from the preceding grid
      waited = true;
    }
    if ((t.cls == C2R || t.cls == C2S) && p.phases == 3 && t.g != ready_group) {
      // the group's GEMM1 tiles (any cluster) have stored its hidden rows
      if (!wait_gemm1_done(c, p, t, peer_abort)) {
        ok = false;
        break;
      }
      ready_group = t.g;
    }
    const bool routed = t.cls == C1R || t.cls == C2R;
    const int cls = t.cls;
    const int w_row = (routed ? t.g * p.w_step[cls] : 0) + t.fb * PAIR_M + int(rank) * PM;
    const int x_row = t.n0 + int(rank) * (t.n_mma / 2);
    const CUtensorMap* xmap = x_map(p, cls, t.n_mma);
    // MN-major B: this CTA's n_mma / 2 columns in boxes of 64
    const int nbx = (t.n_mma / 2 + 63) / 64;
    // both CTAs' full boxes (a box past the tensor's end reads as zeros and still counts)
    const uint32_t bytes =
        2u * uint32_t(A_BYTES + (p.b_mn[cls] ? nbx * B_KB_BYTES : KB_STAGE * x_kb_bytes(t.n_mma)));
    for (int ks = 0; ks < t.nks; ++ks) {
      if (!pair_wait(&c->empty[stage], phase ^ 1u, c, peer_abort, p.status)) {
        ok = false;
        break;
      }
      uint8_t* sa = stages + stage * p.stage_bytes;
      if (rank == 0) mbar_arrive_expect_tx(&c->full[stage], bytes);
      const uint32_t fb = map_to_rank(smem_u32(&c->full[stage]), 0);   // rank 0's barrier
      const int kk = t.k0 + ks * (KB_STAGE * BK);                     // first K index of the stage
      if (p.w_img[cls]) {
        // one contiguous 32 KB stage block: this CTA's 128 rows x 128 columns
        const int tr = (routed ? t.g * p.w_tpg[cls] : 0) + t.fb * 2 + int(rank);
        tma_load_4d_pair(sa, &p.tmW[cls], fb, 0, 0, 0, tr * p.w_nst[cls] + kk / (KB_STAGE * BK));
      } else if (!p.a_mn[cls]) {
        tma_load_3d_pair(sa, &p.tmW[cls], fb, w_row, kk / BK);
      } else {
        const bool second = kk >= p.K1[cls];
        const CUtensorMap* wm = second ? &p.tmW2[cls] : &p.tmW[cls];
        const int krow = (routed ? t.g * p.a_kstep[cls] : 0) + (second ? kk - p.K1[cls] : kk);
        const int mn = t.fb * PAIR_M + int(rank) * PM;
        tma_load_2d_pair(sa, wm, fb, mn, krow);
        tma_load_2d_pair(sa + A_KB_BYTES, wm, fb, mn + BK, krow);
      }
      if (!p.b_mn[cls]) {
        tma_load_3d_pair(sa + A_BYTES, xmap, fb, x_row, kk / BK);
      } else {
        for (int h = 0; h < nbx; ++h)
          tma_load_2d_pair(sa + A_BYTES + h * B_KB_BYTES, &p.tmX[cls], fb, p.b_col0[cls] + x_row + h * BK, kk);
      }
      issued |= 1u << stage;
      issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  pair_drain(c->empty, p.stages, issued, issued_par, c);
}

__device__ __forceinline__ int weight_row(const PairParams& p, const PairTile& t, uint32_t rank) {
  const bool routed = t.cls == C1R || t.cls == C2R;
  return (routed ? t.g * p.w_step[t.cls] : 0) + t.fb * PAIR_M + int(rank) * PM;
}

// FP8 producer.  Each slot of the ring takes up to sps consecutive stages of
// one tile: their weight images in one bulk copy (this CTA's barrier) and
// their token tiles (completion counted on the even CTA's per-stage barriers,
// like the bf16 path), issued together so that a token tile never queues
// behind weight copies of later stages.  The converters turn each image into
// a bf16 A buffer; the MMAs of the slot's last stage free the slot.
__device__ void pair_producer_fp8(PairCtrl* c, const PairParams& p, uint8_t* stages, uint32_t rank,
                                  uint32_t peer_abort) {
  uint8_t* ring = stages + p.f8_off;
  RingPos slot, fpos;                 // slot ring; per-stage barriers full[0 .. nf * sps)
  const int nfull = p.nf * p.sps;
  uint32_t used = 0, used_par = 0;    // slots written, and the parity of their last use
  bool ok = true;
  bool waited = false;
  int ready_group = -1;
  RingPos tr;
  while (ok) {
    const int tile = next_tile(c, p, tr, peer_abort);
    if (tile < 0) break;
    const PairTile t = pair_tile(c, p, tile);
    if (t.cls == C1R && !waited) {
      pdl_wait();   // the permuted token rows come from the preceding grid
      waited = true;
    }
    if ((t.cls == C2R || t.cls == C2S) && p.phases == 3 && t.g != ready_group) {
      // the group's GEMM1 tiles (any cluster) have stored its hidden rows
      if (!wait_gemm1_done(c, p, t, peer_abort)) {
        ok = false;
        break;
      }
      ready_group = t.g;
    }
    const int nks = p.K[t.cls] / 128;   // stages of this tile (K is a multiple of 128)
    const uint8_t* wsrc = static_cast<const uint8_t*>(p.wimg[t.cls]) +
                          size_t(weight_row(p, t, rank) / PM) * size_t(nks) * FP8_STAGE_BYTES;
    const int x_row = t.row_start + t.tb * PN + int(rank) * (t.n_mma / 2);
    const CUtensorMap* xmap = x_map(p, t.cls, t.n_mma);
    const uint32_t xbytes = 2u * uint32_t(KB_STAGE * x_kb_bytes(t.n_mma));
    for (int ks = 0; ks < nks; ks += p.sps) {
      const int n_in = min(p.sps, nks - ks);
      if (!pair_wait(&c->f8_empty[slot.i], slot.par ^ 1u, c, peer_abort, p.status)) {
        ok = false;
        break;
      }
      uint8_t* dst = ring + size_t(slot.i) * p.slot_bytes;
      const uint32_t wbytes = uint32_t(n_in) * FP8_STAGE_BYTES;
      mbar_arrive_expect_tx(&c->f8_full[slot.i], wbytes);
      bulk_load(dst, wsrc + size_t(ks) * FP8_STAGE_BYTES, wbytes, &c->f8_full[slot.i]);
      uint8_t* xdst = dst + p.sps * FP8_STAGE_BYTES;
      for (int j = 0; j < n_in; ++j) {
        uint64_t* fb = &c->full[fpos.i];
        if (rank == 0) mbar_arrive_expect_tx(fb, xbytes);
        tma_load_3d_pair(xdst + j * KB_STAGE * p.x_kb_bytes, xmap, map_to_rank(smem_u32(fb), 0), x_row,
                         (ks + j) * KB_STAGE);
        fpos.next(nfull);
      }
      used |= 1u << slot.i;
      used_par = (used_par & ~(1u << slot.i)) | (slot.par << slot.i);
      slot.next(p.nf);
    }
  }
  pair_drain(c->f8_empty, p.nf, used, used_par, c);
}

// 16 e4m3 values (k order) times a power-of-two scale -> 8 words of bf16 pairs
// (exact: e4m3 -> f16 -> f32 conversions are exact and so is the product).
__device__ __forceinline__ void convert_e4m3x16(const uint4 q, float scale, uint32_t* o) {
  const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(qw[i] & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(qw[i] >> 16), __NV_E4M3);
    const float2 a = __half22float2(__half2(lo)), b = __half22float2(__half2(hi));
    const __nv_bfloat162 x = __floats2bfloat162_rn(a.x * scale, a.y * scale);
    const __nv_bfloat162 y = __floats2bfloat162_rn(b.x * scale, b.y * scale);
    o[2 * i] = *reinterpret_cast<const uint32_t*>(&x);
    o[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&y);
  }
}

// 16 e4m3 values (k order) times 2^rel, rel in [-24, 0] -> 8 words of f16
// pairs: the e4m3 -> f16 conversion is exact, and so is the product whenever
// it is a multiple of 2^-24 (always for rel >= -15).  `fac` holds 2^rel twice.
__device__ __forceinline__ void convert_e4m3x16_f16(const uint4 q, __half2 fac, uint32_t* o) {
  const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 lo = __hmul2(__half2(__nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(qw[i] & 0xffffu), __NV_E4M3)),
                               fac);
    const __half2 hi = __hmul2(__half2(__nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(qw[i] >> 16), __NV_E4M3)), fac);
    o[2 * i] = *reinterpret_cast<const uint32_t*>(&lo);
    o[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hi);
  }
}

// 2^rel as an f16 pair (rel <= 0 clamped to 0 above; below -24 it is zero).
__device__ __forceinline__ __half2 f16_pow2_pair(int rel) {
  rel = min(rel, 0);
  const unsigned short b = rel >= -14 ? (unsigned short)((rel + 15) << 10)
                                      : (rel >= -24 ? (unsigned short)(1u << (rel + 24)) : (unsigned short)0);
  __half_raw h;
  h.x = b;
  return __half2(__half(h), __half(h));
}

// Reference-exponent slot of weight row r of a CTA's 128 rows: GEMM1 rows
// alternate 16 W1 and 16 W3 rows (tiles start on multiples of 32 rows), GEMM2
// rows are W2's.
__device__ __forceinline__ int eref_slot(int cls, int r) { return (cls == C1R || cls == C1S) ? ((r >> 4) & 1) : 2; }

// One converter thread's part of a stage image `img`: chunks c0 .. c0 +
// CONV_CPT - 1 (16 weights each, 64-weight block h) of weight row r, as f16
// relative to the matrix's reference exponent or as bf16 with the full block
// scale, into o [8 * CONV_CPT] words.
__device__ __forceinline__ void convert_stage_part(const uint8_t* img, int h, int r, int c0, bool f16, int e_ref,
                                                   uint32_t* o) {
  const int e_blk = reinterpret_cast<const int32_t*>(img + FP8_IMAGE_BYTES)[h * PM + r];
  const uint8_t* src = img + r * 128;
  const int sw = r & 7;   // 128-byte swizzle phase of the row
  if (f16) {
    const __half2 fac = f16_pow2_pair(e_blk - e_ref);
#pragma unroll
    for (int qc = 0; qc < CONV_CPT; ++qc)
      convert_e4m3x16_f16(*reinterpret_cast<const uint4*>(src + (((c0 + qc) ^ sw) << 4)), fac, o + 8 * qc);
  } else {
    const float scale = ldexpf(1.0f, e_blk);
#pragma unroll
    for (int qc = 0; qc < CONV_CPT; ++qc)
      convert_e4m3x16(*reinterpret_cast<const uint4*>(src + (((c0 + qc) ^ sw) << 4)), scale, o + 8 * qc);
  }
}

// FP8 converter warps: thread i owns 16-weight chunks (i / 128) * CONV_CPT ..
// of weight row i % 128 of this CTA's 128 (all in one 64-weight k-block).
// Per stage it reads those e4m3 bytes (128-byte swizzle) and the block's scale
// (a power of two, so the products are exact), writes the bf16 values into a
// free A buffer in the MMA's swizzled K-major layout, then tells the MMA
// issuer on the even CTA (on the stage's barrier, which also counts the token
// tile's bytes).  The arrival orders the writes at CTA scope only: each CTA's
// tensor core reads its own A rows, so the data never crosses CTAs.
// With A in tensor memory the warp's lane quarter fixes its rows (warp % 4),
// and the four warps of a quarter take 32 weights of the stage row each; a
// thread writes its 16 columns with one tcgen05.st.
__device__ void pair_converter(PairCtrl* c, const PairParams& p, uint8_t* stages, uint32_t tmem, int warp, int lane,
                               uint32_t peer_abort) {
  uint8_t* ring = stages + p.f8_off;
  const int cw = warp - THREADS / 32;
  const int ct = cw * 32 + lane;
  const int r = p.a_tmem ? (warp & 3) * 32 + lane : ct % PM;   // weight row within this CTA's 128
  const int c0 = p.a_tmem ? (cw / 4) * CONV_CPT : (ct / PM) * CONV_CPT;   // first 16-weight chunk
  const int h = c0 / 4;                   // its k-block
  const int sw = r & 7;                   // 128-byte swizzle phase of that row
  const uint32_t a_lane = uint32_t((warp & 3) * 32) << 16;
  RingPos slot, stage, fpos;      // slot ring, A buffers, per-stage barriers
  const int nfull = p.nf * p.sps;
  bool ok = true;
  RingPos tr;
  while (ok) {
    int tile = 0;
    if (lane == 0) tile = next_tile(c, p, tr, peer_abort);
    tile = __shfl_sync(0xffffffffu, tile, 0);
    if (tile < 0) break;
    const PairTile t = pair_tile(c, p, tile);
    const int nks = p.K[t.cls] / 128;
    const bool f16 = p.f16op[t.cls] != 0;
    const int e_ref = p.eref[t.g * 3 + eref_slot(t.cls, r)];
    for (int ks = 0; ks < nks; ++ks) {
      const int half = ks & (p.sps - 1);   // sps is 1 or 2
      int good = 1;
      if (lane == 0) {
        good = (half != 0 || pair_wait(&c->f8_full[slot.i], slot.par, c, peer_abort, p.status)) &&
               pair_wait(&c->empty[stage.i], stage.par ^ 1u, c, peer_abort, p.status);
      }
      if (!__shfl_sync(0xffffffffu, good, 0)) {
        ok = false;
        break;
      }
      const uint8_t* img = ring + size_t(slot.i) * p.slot_bytes + size_t(half) * FP8_STAGE_BYTES;
      if (p.a_tmem) {
        // the MMAs that read this A buffer completed (empty wait above)
        tc_fence_after();
        uint32_t o[16];
        convert_stage_part(img, h, r, c0, f16, e_ref, o);
        // 32 values = 16 columns at k offset 16 * c0 of the stage
        tmem_st16(tmem + a_lane + A_TMEM_COL0 + uint32_t(stage.i) * 64u + uint32_t(c0) * 8u, o);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_cta(map_to_rank(smem_u32(&c->full[fpos.i]), 0));
        stage.next(p.stages);
        fpos.next(nfull);
        if (half == p.sps - 1 || ks == nks - 1) slot.next(p.nf);
        continue;
      }
      uint8_t* kb = stages + size_t(stage.i) * p.stage_bytes + h * A_KB_BYTES + r * 128;
      uint32_t o[8 * CONV_CPT];
      convert_stage_part(img, h, r, c0, f16, e_ref, o);
#pragma unroll
      for (int qc = 0; qc < CONV_CPT; ++qc) {
        // chunk c0 + qc of the stage row (weights 16 q4 .. 16 q4 + 15 of k-block h)
        // -> 16-byte chunks 2 q4 and 2 q4 + 1 of row r of the A buffer's k-block h
        const int j = 2 * ((c0 + qc) & 3);
        *reinterpret_cast<uint4*>(kb + ((j ^ sw) << 4)) =
            make_uint4(o[8 * qc], o[8 * qc + 1], o[8 * qc + 2], o[8 * qc + 3]);
        *reinterpret_cast<uint4*>(kb + (((j + 1) ^ sw) << 4)) =
            make_uint4(o[8 * qc + 4], o[8 * qc + 5], o[8 * qc + 6], o[8 * qc + 7]);
      }
      // the tensor cores read the A buffer through the async proxy
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote_cta(map_to_rank(smem_u32(&c->full[fpos.i]), 0));
      stage.next(p.stages);
      fpos.next(nfull);
      if (half == p.sps - 1 || ks == nks - 1) slot.next(p.nf);
    }
  }
}

// FP8: the A operand comes from the A buffers in turn, the token tile from the
// stage's part of its slot; the MMAs' completion frees the A buffer, and after
// the slot's last stage the slot.
template <bool FP8>
__device__ void pair_mma(PairCtrl* c, const PairParams& p, uint8_t* stages, uint32_t tmem, uint32_t peer_abort) {
  int stage = 0;
  uint32_t phase = 0;
  int slot = 0;
  RingPos fpos;   // FP8: per-stage barriers full[0 .. nf * sps)
  int ctr = 0;
  bool ok = true;
  RingPos tr;
  for (; ok; ++ctr) {
    const int tile = next_tile(c, p, tr, peer_abort);
    if (tile < 0) break;
    const PairTile t = pair_tile(c, p, tile);
    const uint32_t a_mn = FP8 ? 0u : uint32_t(p.a_mn[t.cls]), b_mn = FP8 ? 0u : uint32_t(p.b_mn[t.cls]);
    const uint32_t idesc = (FP8 && p.f16op[t.cls] ? idesc_f16_f32(PAIR_M, t.n_mma) : idesc_bf16_f32(PAIR_M, t.n_mma)) |
                           (a_mn << 15) | (b_mn << 16);
    const int acc = ctr & 1;
    if (!pair_wait(&c->tempty[acc], (uint32_t(ctr >> 1) & 1u) ^ 1u, c, peer_abort, p.status, true)) break;
    tc_fence_after();
    const uint32_t d_tmem = tmem + uint32_t(acc) * p.acc_stride;
    const int nks = t.nks;
    const uint32_t b_kb = uint32_t(x_kb_bytes(t.n_mma));
    for (int ks = 0; ks < nks; ++ks) {
      const int half = FP8 ? (ks & (p.sps - 1)) : 0;
      if (!pair_wait(&c->full[FP8 ? fpos.i : stage], FP8 ? fpos.par : phase, c, peer_abort, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a0 = smem_u32(stages + stage * p.stage_bytes);
      const uint32_t b0 = FP8 ? smem_u32(stages + p.f8_off + size_t(slot) * p.slot_bytes +
                                         size_t(p.sps) * FP8_STAGE_BYTES + size_t(half) * KB_STAGE * p.x_kb_bytes)
                              : a0 + A_BYTES;
      if (FP8 && p.a_tmem) {
        // A buffer `stage` in tensor memory: 8 columns per 16 k
        const uint32_t a_t = tmem + A_TMEM_COL0 + uint32_t(stage) * 64u;
#pragma unroll
        for (int j = 0; j < KB_STAGE; ++j)
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16_pair_ta(d_tmem, a_t + uint32_t(j * 32 + kk * 8), sw128_kmajor_desc(b0 + j * b_kb + kk * 32),
                             idesc, (ks | j | kk) != 0 ? 1u : 0u);
      } else if (!FP8 && (a_mn | b_mn)) {
        // MN-major operands: a stage is 128 K rows of 128-byte MN rows, 16 K per MMA
#pragma unroll
        for (int j = 0; j < KB_STAGE; ++j)
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const int s16 = j * (BK / 16) + kk;
            const uint64_t ad = a_mn ? sw128_mnmajor_desc(a0 + s16 * 2048, KB_STAGE * BK)
                                     : sw128_kmajor_desc(a0 + j * A_KB_BYTES + kk * 32);
            const uint64_t bd = b_mn ? sw128_mnmajor_desc(b0 + s16 * 2048, KB_STAGE * BK)
                                     : sw128_kmajor_desc(b0 + j * b_kb + kk * 32);
            mma_bf16_pair(d_tmem, ad, bd, idesc, (ks | j | kk) != 0 ? 1u : 0u);
          }
      } else {
#pragma unroll
        for (int j = 0; j < KB_STAGE; ++j)
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16_pair(d_tmem, sw128_kmajor_desc(a0 + j * A_KB_BYTES + kk * 32),
                          sw128_kmajor_desc(b0 + j * b_kb + kk * 32), idesc, (ks | j | kk) != 0 ? 1u : 0u);
      }
      mma_commit_pair(&c->empty[stage], 0x3);
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
      if (FP8) {
        fpos.next(p.nf * p.sps);
        if (half == p.sps - 1 || ks == nks - 1) {
          mma_commit_pair(&c->f8_empty[slot], 0x3);
          if (++slot == p.nf) slot = 0;
        }
      }
    }
    if (ok) mma_commit_pair(&c->tfull[acc], 0x3);
  }
  // Every MMA issued here completes before tensor memory is released (this
  // wait holds after a stop too: issued MMAs always complete).
  mma_commit_pair(&c->drain, 0x1);
  pair_wait(&c->drain, 0u, c, peer_abort, p.status, false, false);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

// One lane waits and the result is broadcast, so the warp-collective tensor
// memory loads that follow run on the whole warp.
__device__ __forceinline__ bool pair_warp_wait(uint64_t* bar, uint32_t parity, PairCtrl* c, uint32_t peer_abort,
                                               int* status, int lane) {
  int ok = 1;
  if (lane == 0) ok = pair_wait(bar, parity, c, peer_abort, status) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <bool FP8>
__device__ void pair_epilogue(PairCtrl* c, const PairParams& p, uint32_t tmem, int warp, int lane, uint32_t rank,
                              uint32_t peer_abort) {
  const int q = warp & 3;   // the tensor-memory lane quarter this warp may read
  int ctr = 0;
  RingPos tr;
  for (;; ++ctr) {
    int tile = 0;
    if (lane == 0) tile = next_tile(c, p, tr, peer_abort);
    tile = __shfl_sync(0xffffffffu, tile, 0);
    if (tile < 0) break;
    const PairTile t = pair_tile(c, p, tile);
    const int acc = ctr & 1;
    if (!pair_warp_wait(&c->tfull[acc], uint32_t(ctr >> 1) & 1u, c, peer_abort, p.status, lane)) break;
    tc_fence_after();
    const uint32_t tbase = tmem + uint32_t(acc) * p.acc_stride + (uint32_t(q * 32) << 16);
    const long long row0 = t.n0;
    const int ncols = (t.n_valid + 15) & ~15;
    const bool gemm1 = t.cls == C1R || t.cls == C1S;
    // FP8 weights with f16 operands: the accumulator carries 2^-e_ref of the
    // product (this lane's weight row's matrix)
    const bool fp8 = FP8 && p.eref != nullptr;
    const float acc_scale = fp8 && p.f16op[t.cls] ? ldexpf(1.0f, p.eref[t.g * 3 + eref_slot(t.cls, q * 32 + lane)])
                                                   : 1.0f;
    if (gemm1) {
      // lane l < 16: W1 row of feature f; lane l + 16: the W3 row of the same f
      const int f = t.fb * (PAIR_M / 2) + int(rank) * (PM / 2) + q * 16 + (lane & 15);
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out[t.cls]) + f;
      __half* out16 = static_cast<__half*>(p.out[t.cls]) + f;   // FP8 layers: f16 hidden rows
      const long long ld = p.ld_out[t.cls];
      const bool lo_half = lane < 16;
      bool over = false;
#pragma unroll 1
      for (int cc = 0; cc < ncols; cc += 16) {
        float v[16];
        tmem_ld16(tbase + cc, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= acc_scale;
        // lanes < 16 keep tokens cc..cc+7, lanes >= 16 tokens cc+8..cc+15
        float mine[8], other[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float send = lo_half ? v[8 + i] : v[i];
          other[i] = __shfl_xor_sync(0xffffffffu, send, 16);
          mine[i] = lo_half ? v[i] : v[8 + i];
        }
        const int j0 = cc + (lo_half ? 0 : 8);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float g = lo_half ? mine[i] : other[i];
          const float u = lo_half ? other[i] : mine[i];
          const float h = silu_f(g) * u;
          if (j0 + i < t.n_valid) {
            if (fp8) {
              over |= fabsf(h) >= 65520.0f;
              out16[(row0 + j0 + i) * ld] = __float2half_rn(h);
            } else {
              out[(row0 + j0 + i) * ld] = __float2bfloat16_rn(h);
            }
          }
        }
      }
      if (over) flag_status(p.status, DEV_RANGE);
    } else {
      const int f = t.fb * PAIR_M + int(rank) * PM + q * 32 + lane;
      const bool fvalid = f < p.M[t.cls];
      float* out = static_cast<float*>(p.out[t.cls]) + f +
                   (p.kmode && t.cls == C2R ? (long long)t.g * p.out_gstride[C2R] : 0LL);
      const long long ld = p.ld_out[t.cls];
#pragma unroll 1
      for (int cc = 0; cc < ncols; cc += 16) {
        float v[16];
        if (t.nks > 0) {
          tmem_ld16(tbase + cc, v);
        } else {
          // a group without rows to reduce over (kmode): its block of D is zero
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.0f;
        }
        if (fvalid) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (cc + i < t.n_valid) out[(row0 + cc + i) * ld] = v[i] * acc_scale;
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_remote(map_to_rank(smem_u32(&c->tempty[acc]), 0));
    if (gemm1 && p.phases == 3) {
      // publish this warp's part of the tile: the lanes' stores, then one
      // release increment of the group's counter (zero since the call began)
      __threadfence();
      __syncwarp();
      if (lane == 0) red_release_gpu_add(p.done + t.g, 1);
    }
  }
}

template <bool FP8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(FP8 ? THREADS_FP8 : THREADS, 1)
    pair_gemm_kernel(const __grid_constant__ PairParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;
  PairCtrl* c = reinterpret_cast<PairCtrl*>(base + size_t(RING_BYTES));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer_abort = map_to_rank(smem_u32(&c->abort), rank ^ 1u);

  if (threadIdx.x == 0) {
    // FP8: the even CTA's producer (token bytes) and the converter warps of both CTAs
    for (int s = 0; s < MAX_FULL; ++s) mbar_init(&c->full[s], FP8 ? 1 + 2 * CONV_WARPS : 1);
    for (int s = 0; s < MAX_STAGES; ++s) mbar_init(&c->empty[s], 1);
    if (FP8) {
      for (int s = 0; s < MAX_F8; ++s) {
        mbar_init(&c->f8_full[s], 1);
        mbar_init(&c->f8_empty[s], 1);
      }
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&c->tfull[a], 1);
      mbar_init(&c->tempty[a], 2 * EPI_WARPS);
    }
    mbar_init(&c->drain, 1);
    for (int i = 0; i < TILE_RING; ++i) {
      mbar_init(&c->tile_full[i], 1);
      mbar_init(&c->tile_empty[i], tile_readers(FP8));
    }
    c->abort = 0;
    c->wait_ns = p.wait_ns;
    c->routed_ready = 0;
    c->seg[0] = 0;
    c->seg[1] = (p.phases & 1) && p.shared_rows > 0 ? pair_group_tiles(p, C1S, p.shared_rows) : 0;
    c->seg[2] = c->seg[1] + ((p.phases & 2) && p.shared_rows > 0 ? pair_group_tiles(p, C2S, p.shared_rows) : 0);
    fence_mbar_init();
    pdl_launch_dependents();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < NCLS; ++i) {
      tma_prefetch_desc(&p.tmW[i]);
      tma_prefetch_desc(&p.tmX[i]);
      tma_prefetch_desc(&p.tmXs[i]);
      tma_prefetch_desc(&p.tmXt[i]);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(&c->tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // both CTAs' barriers and tensor memory are ready
  cluster_sync_all();
  tc_fence_after();
  // A GEMM2-only launch reads the hidden rows of the preceding GEMM1 launch.
  if (p.phases == 2) pdl_wait();

  const uint32_t tmem = c->tmem_base;
  if (warp == 0) {
    if (lane == 0) {
      if (FP8) pair_producer_fp8(c, p, stages, rank, peer_abort);
      else pair_producer(c, p, stages, rank, peer_abort);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) pair_mma<FP8>(c, p, stages, tmem, peer_abort);
  } else if (warp < 2 + EPI_WARPS) {
    pair_epilogue<FP8>(c, p, tmem, warp, lane, rank, peer_abort);
  } else if (warp >= THREADS / 32) {
    pair_converter(c, p, stages, tmem, warp, lane, peer_abort);
  } else if (warp == TABLE_WARP) {
    // the routed tables need the dispatch offsets
    pdl_wait();
    pair_schedule(c, p, lane);
    __syncwarp();
    __threadfence_block();
    if (lane == 0) *reinterpret_cast<volatile int*>(&c->routed_ready) = 1;
  } else if (warp == DISPATCH_WARP) {
    if (lane == 0 && rank == 0) pair_dispatch(c, p, peer_abort);
  }
  tc_fence_before();
  // neither CTA leaves while the other may still signal its barriers
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

template <bool FP8>
cudaError_t launch_pair(const PairParams& p, long long max_tiles, cudaStream_t stream) {
  constexpr int kThreads = FP8 ? THREADS_FP8 : THREADS;
  static PerDevice<int> clusters;
  int max_clusters = 0;
  cudaError_t e = clusters.get(&max_clusters, [](int* n) {
    cudaError_t err = cudaFuncSetAttribute(pair_gemm_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           int(kPairSmem));
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kPairSmem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    *n = 0;
    if (cudaOccupancyMaxActiveClusters(n, pair_gemm_kernel<FP8>, &cfg) != cudaSuccess || *n <= 0) {
      cudaGetLastError();
      *n = num_sms() / 2;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  // one cluster per pair of SMs that can hold one (more would only queue)
  const long long pairs = max_tiles < max_clusters ? max_tiles : max_clusters;
  return launch_pdl(pair_gemm_kernel<FP8>, dim3(int(2 * pairs)), dim3(kThreads), kPairSmem, stream, p);
}

std::atomic<unsigned long long> g_wait_ns{0};   // 0: kWaitLimitNs
std::atomic<int> g_need_extra{0};

}  // namespace

void set_expert_fault(unsigned long long wait_ns, int need_extra) {
  g_wait_ns.store(wait_ns);
  g_need_extra.store(need_extra);
}

void get_expert_fault(unsigned long long* wait_ns, int* need_extra) {
  *wait_ns = g_wait_ns.load();
  *need_extra = g_need_extra.load();
}

cudaError_t launch_pair_experts(const PairClass cls[4], const int32_t* offsets, int num_routed, int shared_rows,
                                int max_group_rows, int phases, int* done, int* ticket, int* status,
                                long long max_tiles, cudaStream_t stream, int* launches, const int32_t* fp8_eref) {
  if (max_tiles <= 0) return cudaSuccess;
  const bool fp8 = fp8_eref != nullptr;
  if (num_routed < 1 || num_routed + 1 > MAX_GROUPS || phases < 1 || phases > 3) return cudaErrorInvalidValue;
  if (ticket == nullptr) return cudaErrorInvalidValue;
  if (phases == 3 && done == nullptr) return cudaErrorInvalidValue;
  PairParams p;
  memset(&p, 0, sizeof(p));
  for (int i = 0; i < NCLS; ++i) {
    // without a shared expert its classes repeat the routed ones (never used)
    const PairClass& g = (shared_rows > 0 || i == C1R || i == C2R) ? cls[i] : cls[i - 1];
    if (g.K % BK != 0) return cudaErrorInvalidValue;
    if (fp8) {
      // stage images of 128-row tiles (a zero tile follows the last row)
      if (g.K % 128 != 0 || g.w_rows % PM != 0 || reinterpret_cast<uintptr_t>(g.W) % 16 != 0)
        return cudaErrorInvalidValue;
      p.wimg[i] = g.W;
      p.f16op[i] = i != C1S ? 1 : 0;   // the shared expert's GEMM1 reads the bf16 x
    } else if (g.img) {
      // stage blocks: groups of M rows (w_rows / M groups), K columns
      if (g.M <= 0 || g.w_rows % g.M != 0) return cudaErrorInvalidValue;
      p.w_img[i] = 1;
      p.w_tpg[i] = img_tiles(g.M);
      p.w_nst[i] = img_stages(g.K);
      if (g.w_step != 0 && g.w_step != g.M) return cudaErrorInvalidValue;
      const long long blocks = (g.w_rows / g.M) * (long long)p.w_tpg[i] * p.w_nst[i];
      if (!encode_stage_block_map(&p.tmW[i], g.W, blocks)) return cudaErrorInvalidValue;
    } else if (!encode_bf16_map(&p.tmW[i], g.W, g.w_rows, g.K, PM, KB_STAGE)) {
      return cudaErrorInvalidValue;
    }
    if (!encode_bf16_map(&p.tmX[i], g.X, g.x_rows, g.K, XB, KB_STAGE)) return cudaErrorInvalidValue;
    if (!encode_bf16_map(&p.tmXs[i], g.X, g.x_rows, g.K, XSMALL, KB_STAGE)) return cudaErrorInvalidValue;
    if (!encode_bf16_map(&p.tmXt[i], g.X, g.x_rows, g.K, XTINY, KB_STAGE)) return cudaErrorInvalidValue;
    p.out[i] = g.out;
    p.ld_out[i] = g.ld_out;
    p.out_rows[i] = g.out_rows;
    p.M[i] = g.M;
    p.K[i] = g.K;
    p.K1[i] = INT_MAX;
    p.w_step[i] = g.w_step;
  }
  p.offsets = offsets;
  p.eref = fp8_eref;
  p.row_bound = cls[C1R].out_rows;
  p.num_routed = num_routed;
  p.shared_rows = shared_rows;
  p.done = done;
  p.ticket = ticket;
  p.phases = phases;
  p.status = status;
  const unsigned long long wns = g_wait_ns.load();
  p.wait_ns = wns > 0 ? wns : kWaitLimitNs;
  p.need_extra = phases == 3 ? g_need_extra.load() : 0;
  // A group never holds more tokens than the batch, so with at most 64 tokens
  // every tile takes the 32-row token box (at most 16: the 8-row box): use the
  // deeper rings of smaller stages.
  const bool small = max_group_rows <= 2 * XSMALL;
  const bool tiny_box = max_group_rows <= 2 * XTINY;
  p.stage_bytes = tiny_box ? TINY_STAGE_BYTES : (small ? SMALL_STAGE_BYTES : STAGE_BYTES);
  cudaError_t e;
  if (fp8) {
    // two bf16 A buffers (written by the converters) and a ring of slots,
    // each holding the weight images and token tiles of sps stages: decode-
    // sized launches take two stages per slot (groups of at most 16 tokens:
    // 4 slots of 38 KB; at most 64: 3 of 50 KB), others one (3 slots of 49 KB)
    // Decode-sized launches put the A buffers in tensor memory (the
    // accumulators need at most 64 columns there), which leaves all of the
    // ring to the slots: 5 of 38 KB (groups of at most 16 tokens) or 4 of 50 KB.
    const bool tiny = max_group_rows <= 2 * XTINY;
    p.a_tmem = small ? 1 : 0;
    p.acc_stride = small ? ACC_STRIDE_SMALL : ACC_STRIDE;
    p.stages = small ? A_TMEM_STAGES : 2;
    p.stage_bytes = small ? 0 : A_BYTES;
    p.f8_off = small ? 0 : 2 * A_BYTES;
    p.sps = small ? 2 : 1;
    p.x_kb_bytes = tiny ? XT_KB_BYTES : (small ? XS_KB_BYTES : B_KB_BYTES);
    p.slot_bytes = p.sps * (FP8_STAGE_BYTES + KB_STAGE * p.x_kb_bytes);
    p.nf = (RING_BYTES - p.f8_off) / p.slot_bytes;
    if (p.nf > MAX_F8) p.nf = MAX_F8;
    e = launch_pair<true>(p, max_tiles, stream);
  } else {
    p.stages = tiny_box ? MAX_STAGES : (small ? 5 : 3);
    p.acc_stride = ACC_STRIDE;
    e = launch_pair<false>(p, max_tiles, stream);
  }
  if (e == cudaSuccess && launches) ++*launches;
  return e;
}

cudaError_t launch_pair_gemm(const PairOperands* routed, const PairOperands* shared, const int32_t* offsets,
                             const int32_t* row_base, long long row_bound, int num_routed, int shared_rows,
                             int kmode, int* ticket, int* status, long long max_tiles, cudaStream_t stream,
                             int* launches) {
  if (max_tiles <= 0) return cudaSuccess;
  if (num_routed < 0 || num_routed + 1 > MAX_GROUPS || ticket == nullptr) return cudaErrorInvalidValue;
  if ((routed == nullptr) != (num_routed == 0) || (shared == nullptr) != (shared_rows <= 0))
    return cudaErrorInvalidValue;
  PairParams p;
  memset(&p, 0, sizeof(p));
  bool any_b_mn = false;
  const PairOperands* ops[2] = {routed, shared};
  for (int r = 0; r < 2; ++r) {
    const int i = r == 0 ? C2R : C2S;
    const PairOperands* o = ops[r] != nullptr ? ops[r] : ops[1 - r];   // an absent class repeats the other (unused)
    if (o == nullptr) return cudaErrorInvalidValue;
    if (o->K % (KB_STAGE * BK) != 0 || o->M <= 0) return cudaErrorInvalidValue;
    if (o->a_mn) {
      if (!encode_bf16_map(&p.tmW[i], o->A, o->a_rows, o->a_cols, KB_STAGE * BK, 1)) return cudaErrorInvalidValue;
      const void* a2 = o->A2 != nullptr ? o->A2 : o->A;
      const int64_t a2_rows = o->A2 != nullptr ? o->a2_rows : o->a_rows;
      if (!encode_bf16_map(&p.tmW2[i], a2, a2_rows, o->a_cols, KB_STAGE * BK, 1)) return cudaErrorInvalidValue;
      if (o->K1 % (KB_STAGE * BK) != 0) return cudaErrorInvalidValue;
    } else if (!encode_bf16_map(&p.tmW[i], o->A, o->a_rows, o->a_cols, PM, KB_STAGE)) {
      return cudaErrorInvalidValue;
    }
    if (o->b_mn) {
      if (!encode_bf16_map(&p.tmX[i], o->B, o->b_rows, o->b_cols, KB_STAGE * BK, 1)) return cudaErrorInvalidValue;
      any_b_mn = true;
    } else {
      if (!encode_bf16_map(&p.tmX[i], o->B, o->b_rows, o->b_cols, XB, KB_STAGE)) return cudaErrorInvalidValue;
      if (!encode_bf16_map(&p.tmXs[i], o->B, o->b_rows, o->b_cols, XSMALL, KB_STAGE)) return cudaErrorInvalidValue;
      if (!encode_bf16_map(&p.tmXt[i], o->B, o->b_rows, o->b_cols, XTINY, KB_STAGE)) return cudaErrorInvalidValue;
    }
    p.a_mn[i] = o->a_mn ? 1 : 0;
    p.b_mn[i] = o->b_mn ? 1 : 0;
    p.K1[i] = o->a_mn && o->A2 != nullptr ? o->K1 : INT_MAX;   // no second source: never switch
    p.a_kstep[i] = o->a_kstep;
    p.out[i] = o->out;
    p.ld_out[i] = o->ld_out;
    p.out_rows[i] = o->out_rows;
    p.out_gstride[i] = o->out_gstride;
    p.M[i] = o->M;
    p.K[i] = o->K;
    p.N[i] = o->N;
    p.b_col0[i] = o->b_col0;
    p.w_step[i] = o->w_step;
  }
  // the GEMM1 classes are not used (GEMM2 tiles only); keep them well-formed
  p.tmW[C1R] = p.tmW[C2R];
  p.tmW[C1S] = p.tmW[C2S];
  p.M[C1R] = p.M[C2R];
  p.M[C1S] = p.M[C2S];
  p.K[C1R] = p.K[C2R];
  p.K[C1S] = p.K[C2S];
  p.offsets = offsets;
  p.row_base = row_base;
  p.row_bound = row_bound;
  p.num_routed = num_routed;
  p.shared_rows = shared != nullptr ? shared_rows : 0;
  p.kmode = kmode;
  p.phases = 2;
  p.ticket = ticket;
  p.status = status;
  const unsigned long long wns = g_wait_ns.load();
  p.wait_ns = wns > 0 ? wns : kWaitLimitNs;
  p.stages = 3;
  p.stage_bytes = STAGE_BYTES;
  p.acc_stride = ACC_STRIDE;
  (void)any_b_mn;
  cudaError_t e = launch_pair<false>(p, max_tiles, stream);
  if (e == cudaSuccess && launches) ++*launches;
  return e;
}

}  // namespace moe
