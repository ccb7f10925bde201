// Router gate GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA):
//
//   logits[t][e] = sum_c x[t][c] * W_g[e][c]
//
// The MoEGate listing of the DeepSeek-V2 walkthrough computes the logits in
// fp32.  bf16 x times bf16 W_g (or times each bf16 part of an fp32 W_g split
// three ways along K) gives exact products, and the tensor cores accumulate
// them in fp32; every 256-long partial sum is then added into registers with
// fp32 round-to-nearest, so the logits carry the rounding of 256-long sums
// only.  For small batches K is split into ranges whose fp32 partial planes
// the top-k kernel adds in order.
//
// Persistent CTAs, one per SM (192 threads):
//   warp 0      TMA producer: A tile 128x64 (tokens), B tile 128x64 (W_g rows)
//               per stage into a 4-deep shared-memory ring (128-byte swizzle)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//               (M=128, N=128, K=16 per instruction)
//   warps 2..5  epilogue: tcgen05.ld of the partial sums, fp32 accumulation
//               in registers, stores of the logits
// Two accumulators in TMEM let the epilogue of one chunk overlap the MMAs of
// the next.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;        // widest tile; TMEM accumulator stride
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int THREADS = 192;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int MAX_GROUPS = 272;
constexpr uint32_t TMEM_COLS = 512;

struct Params {
  CUtensorMap tmA[2];
  CUtensorMap tmB[2];
  void* out[2];
  long long ld_out[2];
  long long out_rows[2];
  int N[2], K[2], a_k_mod[2], b_step[2], mma_n[2];
  int ksplit;                 // EPI_GATE_F32: K ranges per output tile (partial planes)
  long long split_stride;     // elements between consecutive partial planes
  const int32_t* offsets;
  int num_routed;
  int rows_single0;
  int shared_rows;
  int* status;
};

struct Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int ngroups;
  int g0;
  int tile_start[MAX_GROUPS + 1];
  int row_start[MAX_GROUPS];
  int rows[MAX_GROUPS];
};

constexpr size_t kSmemBytes = 1024 + size_t(STAGES) * STAGE_BYTES + sizeof(Ctrl);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
// More than half of an SM's shared memory: at most one CTA per SM, so the
// full-TMEM allocation below can never wait on another resident CTA.
static_assert(kSmemBytes > 114 * 1024, "one CTA per SM");

struct TileInfo {
  int cls, g, m_blk, n_blk, row_start, rows;
  int kb_lo, kb_hi;   // k-block range of this tile
  int ks;             // partial plane (split index) of the output
};

// Tile width and accumulation chunk of each epilogue mode.  EPI_GATE_F32 keeps
// 128-column tiles so that an epilogue thread can hold a whole accumulator row
// in registers, and restarts the tensor-core accumulation every PROMOTE_KB
// k-blocks: each 256-long partial sum is added into the registers with fp32
// round-to-nearest, so the result carries the error of 256-long tensor-core
// sums only, not of a d-long one.
constexpr int PROMOTE_KB = 4;
template <int EPI> struct Mode {
  static constexpr int kBN = EPI == EPI_GATE_F32 ? 128 : BN;
  static constexpr int kChunk = EPI == EPI_GATE_F32 ? PROMOTE_KB : (1 << 30);
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

template <int EPI>
__device__ __forceinline__ int splits(const Params& p) {
  return EPI == EPI_GATE_F32 ? p.ksplit : 1;
}

template <int EPI>
__device__ __forceinline__ int group_tiles(const Params& p, int cls, int rows) {
  return cdiv(rows, BM) * cdiv(p.N[cls], Mode<EPI>::kBN) * splits<EPI>(p);
}

// Warp-cooperative: per-group row ranges and the exclusive prefix of tiles.
template <int EPI>
__device__ void build_schedule(Ctrl* c, const Params& p, int lane) {
  const int g0 = p.num_routed > 0 ? p.num_routed : (p.rows_single0 > 0 ? 1 : 0);
  const int ng = g0 + (p.shared_rows > 0 ? 1 : 0);
  const int per = cdiv(ng, 32);
  const int lo = min(ng, lane * per), hi = min(ng, lo + per);
  int local = 0;
  for (int g = lo; g < hi; ++g) {
    const int cls = g < g0 ? 0 : 1;
    int rs = 0, rows = 0;
    if (cls == 0) {
      if (p.num_routed > 0) {
        rs = p.offsets[g];
        rows = p.offsets[g + 1] - rs;
      } else {
        rows = p.rows_single0;
      }
    } else {
      rows = p.shared_rows;
    }
    if (rows < 0 || rs < 0 || (long long)rs + rows > p.out_rows[cls]) {
      flag_status(p.status, DEV_BAD_ROW);
      rs = 0;
      rows = 0;
    }
    c->row_start[g] = rs;
    c->rows[g] = rows;
    local += group_tiles<EPI>(p, cls, rows);
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - local;
  for (int g = lo; g < hi; ++g) {
    c->tile_start[g] = run;
    run += group_tiles<EPI>(p, g < g0 ? 0 : 1, c->rows[g]);
  }
  if (lane == 31) {
    c->tile_start[ng] = incl;
    c->ngroups = ng;
    c->g0 = g0;
  }
}

// Tile -> (group, m block, n block).  Within a group, the block order keeps
// the operand that is re-read the most resident in L2: groups with more row
// blocks than column blocks walk columns fastest (the A rows are re-used),
// others walk rows fastest (the weight tile is re-used).
template <int EPI>
__device__ __forceinline__ TileInfo tile_info(const Ctrl* c, const Params& p, int tile) {
  int lo = 0, hi = c->ngroups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c->tile_start[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  TileInfo t;
  t.g = lo;
  t.cls = lo < c->g0 ? 0 : 1;
  t.row_start = c->row_start[lo];
  t.rows = c->rows[lo];
  int local = tile - c->tile_start[lo];
  const int mb = cdiv(t.rows, BM), nb = cdiv(p.N[t.cls], Mode<EPI>::kBN);
  // K split (gate mode): the split index is the slowest, and each split owns
  // a contiguous run of whole promotion chunks
  const int nk = p.K[t.cls] / BK;
  const int ns = splits<EPI>(p);
  t.ks = local / (mb * nb);
  local -= t.ks * mb * nb;
  if (ns > 1) {
    const int nch = cdiv(nk, Mode<EPI>::kChunk);
    const int c_lo = t.ks * nch / ns, c_hi = (t.ks + 1) * nch / ns;
    t.kb_lo = c_lo * Mode<EPI>::kChunk;
    t.kb_hi = min(nk, c_hi * Mode<EPI>::kChunk);
  } else {
    t.kb_lo = 0;
    t.kb_hi = nk;
  }
  if (mb > nb) {
    t.m_blk = local / nb;
    t.n_blk = local % nb;
  } else {
    t.n_blk = local / mb;
    t.m_blk = local % mb;
  }
  return t;
}

template <int EPI>
__device__ void producer(Ctrl* c, const Params& p, uint8_t* stages, int total) {
  volatile int* ab = &c->abort;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0, issued_par = 0;
  bool ok = true;
  for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
    const TileInfo t = tile_info<EPI>(c, p, tile);
    const int a_row = t.row_start + t.m_blk * BM;
    const int b_row = (t.cls == 0 ? t.g * p.b_step[0] : 0) + t.n_blk * Mode<EPI>::kBN;
    const uint32_t bytes = A_BYTES + uint32_t(p.mma_n[t.cls]) * BK * 2;
    for (int kb = t.kb_lo; kb < t.kb_hi; ++kb) {
      if (!mbar_wait(&c->empty[stage], phase ^ 1u, ab, p.status)) {
        ok = false;
        break;
      }
      uint8_t* sa = stages + stage * STAGE_BYTES;
      mbar_arrive_expect_tx(&c->full[stage], bytes);
      const int kc = kb * BK;
      tma_load_2d(sa, &p.tmA[t.cls], &c->full[stage], kc % p.a_k_mod[t.cls], a_row);
      tma_load_2d(sa + A_BYTES, &p.tmB[t.cls], &c->full[stage], kc, b_row);
      issued |= 1u << stage;
      issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  // Every issued copy must land before the CTA exits (normally all of them
  // were already consumed by the MMA thread and these waits return at once).
  for (int s = 0; s < STAGES; ++s)
    if (issued & (1u << s)) mbar_wait(&c->full[s], (issued_par >> s) & 1u, nullptr, p.status);
}

// Each tile's k-blocks are issued in chunks of Mode<EPI>::kChunk (one chunk
// per tile unless the mode promotes partial sums); every chunk accumulates
// into one of the two TMEM buffers and is handed to the epilogue on tfull.
template <int EPI>
__device__ void mma_issuer(Ctrl* c, const Params& p, uint8_t* stages, uint32_t tmem, int total) {
  volatile int* ab = &c->abort;
  int stage = 0;
  uint32_t phase = 0;
  int chunk_ctr = 0;
  bool ok = true;
  for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
    const TileInfo t = tile_info<EPI>(c, p, tile);
    const uint32_t idesc = idesc_bf16_f32(BM, p.mma_n[t.cls]);
    const int nk = t.kb_hi;
    const int ck = Mode<EPI>::kChunk < nk - t.kb_lo ? Mode<EPI>::kChunk : nk - t.kb_lo;
    for (int kb0 = t.kb_lo; ok && kb0 < nk; kb0 += ck, ++chunk_ctr) {
      const int acc = chunk_ctr & 1;
      const uint32_t acc_par = uint32_t(chunk_ctr >> 1) & 1u;
      if (!mbar_wait(&c->tempty[acc], acc_par ^ 1u, ab, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + uint32_t(acc * BN);
      const int kend = kb0 + ck < nk ? kb0 + ck : nk;
      for (int kb = kb0; kb < kend; ++kb) {
        if (!mbar_wait(&c->full[stage], phase, ab, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(stages + stage * STAGE_BYTES);
        const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_bf16_ss(d_tmem, sw128_kmajor_desc(a0 + kk * 32), sw128_kmajor_desc(b0 + kk * 32), idesc,
                      (kb != kb0 || kk != 0) ? 1u : 0u);
        mma_commit(&c->empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) mma_commit(&c->tfull[acc]);
    }
  }
  // All MMAs this thread issued complete before TMEM is released.
  mma_commit(&c->drain);
  mbar_wait(&c->drain, 0u, nullptr, p.status);
}

// One lane waits and the result is broadcast, so the warp-collective TMEM
// loads that follow are always executed by the whole warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* ab, int* status, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(bar, parity, ab, status) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int EPI>
__device__ void epilogue(Ctrl* c, const Params& p, uint32_t tmem, int total, int warp, int lane) {
  volatile int* ab = &c->abort;
  const int q = warp & 3;  // the TMEM lane quarter this warp may read
  const int r_in_tile = q * 32 + lane;
  int chunk_ctr = 0;
  bool ok = true;
  for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
    const TileInfo t = tile_info<EPI>(c, p, tile);
    const int row_local = t.m_blk * BM + r_in_tile;
    const bool valid = row_local < t.rows;
    const long long grow = (long long)t.row_start + row_local;
    {
      // sum of the tile's 256-long partial products, fp32 round-to-nearest
      const int nchunks = cdiv(t.kb_hi - t.kb_lo, PROMOTE_KB);
      float racc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) racc[i] = 0.0f;
      for (int ch = 0; ch < nchunks; ++ch, ++chunk_ctr) {
        const int acc = chunk_ctr & 1;
        if (!warp_wait(&c->tfull[acc], uint32_t(chunk_ctr >> 1) & 1u, ab, p.status, lane)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem + uint32_t(acc * BN) + (uint32_t(q * 32) << 16);
#pragma unroll
        for (int cc = 0; cc < 128; cc += 16) {
          float v[16];
          tmem_ld16(tbase + cc, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) racc[cc + i] = __fadd_rn(racc[cc + i], v[i]);
        }
        tc_fence_before();
        mbar_arrive(&c->tempty[acc]);
      }
      if (ok && valid) {
        const int col0 = t.n_blk * 128;
        const int ncol = min(128, p.N[t.cls] - col0);
        float* orow = static_cast<float*>(p.out[t.cls]) + t.ks * p.split_stride + grow * p.ld_out[t.cls] + col0;
        if (ncol == 128) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            reinterpret_cast<float4*>(orow)[i] =
                make_float4(racc[4 * i], racc[4 * i + 1], racc[4 * i + 2], racc[4 * i + 3]);
        } else {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i < ncol) orow[i] = racc[i];
        }
      }
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;
  Ctrl* c = reinterpret_cast<Ctrl*>(base + size_t(STAGES) * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c->full[s], 1);
      mbar_init(&c->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&c->tfull[a], 1);
      mbar_init(&c->tempty[a], 128);
    }
    mbar_init(&c->drain, 1);
    c->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA[0]);
    tma_prefetch_desc(&p.tmB[0]);
    tma_prefetch_desc(&p.tmA[1]);
    tma_prefetch_desc(&p.tmB[1]);
  }
  if (warp == 1) {
    tmem_alloc(&c->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) build_schedule<EPI>(c, p, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the inputs (tokens) come from earlier work in the stream.  The gate is the
  // first kernel of a call (or follows the W_g split), so its dependents are
  // released only after that earlier work has completed.
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();

  const uint32_t tmem = c->tmem_base;
  const int total = c->tile_start[c->ngroups];
  if (warp == 0) {
    if (lane == 0) producer<EPI>(c, p, stages, total);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<EPI>(c, p, stages, tmem, total);
  } else {
    epilogue<EPI>(c, p, tmem, total, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------- host side
}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// bf16 [rows, cols] row-major, 128-byte swizzle.  box_kblocks = 1: a 2-D map
// with 64-column x box_rows boxes.  box_kblocks > 1: a 3-D view
// (64 columns, rows, cols / 64 k-blocks) whose box covers box_kblocks
// consecutive k-blocks of box_rows rows, stored k-block after k-block.
// Encoded maps are kept in a small table keyed by their arguments, so repeated
// layer calls on the same buffers skip the driver call (a host-side cost that
// dominates decode-sized steps).
bool encode_bf16_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, uint32_t box_rows,
                     uint32_t box_kblocks) {
  return encode_tiled_map(m, ptr, rows, cols, 2, box_rows, box_kblocks);
}

// bf16 (elem_bytes 2) or byte-sized (elem_bytes 1) elements; the box's inner
// extent is always one 128-byte swizzle row (64 bf16 or 128 bytes).
bool encode_tiled_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int elem_bytes,
                      uint32_t box_rows, uint32_t box_kblocks) {
  struct Entry {
    const void* ptr;
    int64_t rows, cols;
    uint32_t box, kbs;
    int eb;
    CUtensorMap map;
  };
  constexpr int kEntries = 64;
  static Entry table[kEntries];
  static int filled = 0, next = 0;
  static std::mutex mu;
  if (rows <= 0 || cols <= 0) return false;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < filled; ++i) {
      const Entry& e = table[i];
      if (e.ptr == ptr && e.rows == rows && e.cols == cols && e.box == box_rows && e.kbs == box_kblocks &&
          e.eb == elem_bytes) {
        *m = e.map;
        return true;
      }
    }
  }
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  if (elem_bytes != 1 && elem_bytes != 2) return false;
  const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const cuuint32_t inner = 128u / cuuint32_t(elem_bytes);
  CUresult r;
  if (box_kblocks <= 1) {
    cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(cols) * elem_bytes};
    cuuint32_t box[2] = {inner, box_rows};
    cuuint32_t es[2] = {1u, 1u};
    r = enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    if (cols % inner != 0) return false;
    cuuint64_t dims[3] = {inner, cuuint64_t(rows), cuuint64_t(cols / inner)};
    cuuint64_t strides[2] = {cuuint64_t(cols) * elem_bytes, 128u};
    cuuint32_t box[3] = {inner, box_rows, box_kblocks};
    cuuint32_t es[3] = {1u, 1u, 1u};
    r = enc(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(mu);
  Entry& e = table[next];
  e.ptr = ptr;
  e.rows = rows;
  e.cols = cols;
  e.box = box_rows;
  e.kbs = box_kblocks;
  e.eb = elem_bytes;
  e.map = *m;
  next = (next + 1) % kEntries;
  if (filled < kEntries) ++filled;
  return true;
}

bool encode_stage_block_map(CUtensorMap* m, const void* ptr, long long blocks) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr || blocks <= 0) return false;
  // {64 columns, 128 rows, 2 k-blocks, blocks}: one box is one contiguous block
  cuuint64_t dims[4] = {64u, cuuint64_t(IMG_ROWS), 2u, cuuint64_t(blocks)};
  cuuint64_t strides[3] = {128u, cuuint64_t(IMG_ROWS) * 128u, cuuint64_t(IMG_BLOCK_BYTES)};
  cuuint32_t box[4] = {64u, cuuint32_t(IMG_ROWS), 2u, 1u};
  cuuint32_t es[4] = {1u, 1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {


template <int EPI>
cudaError_t launch_epi(const Params& p, int grid, cudaStream_t stream) {
  static PerDevice<int> attr;
  int unused = 0;
  cudaError_t e = attr.get(&unused, [](int*) {
    return cudaFuncSetAttribute(grouped_gemm_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(kSmemBytes));
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(grouped_gemm_kernel<EPI>, dim3(grid), dim3(THREADS), kSmemBytes, stream, p);
}

}  // namespace

int num_sms() {
  static PerDevice<int> sms;
  int n = 1;
  if (sms.get(&n, [](int* v) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess && *v <= 0) *v = 1;
        return e;
      }) != cudaSuccess)
    return 1;
  return n;
}

cudaError_t launch_grouped_gemm(int epi, const GemmClass& c0, const GemmClass* c1, const int32_t* offsets,
                                int num_routed, int rows_single0, int shared_rows, int* status,
                                long long max_tiles, cudaStream_t stream, int* launches) {
  if (max_tiles <= 0) return cudaSuccess;
  Params p;
  memset(&p, 0, sizeof(p));
  const GemmClass* cls[2] = {&c0, c1 != nullptr ? c1 : &c0};
  for (int i = 0; i < 2; ++i) {
    const GemmClass& g = *cls[i];
    if (!encode_bf16_map(&p.tmA[i], g.A, g.a_rows, g.a_cols, BM, 1)) return cudaErrorInvalidValue;
    if (!encode_bf16_map(&p.tmB[i], g.B, g.b_rows, g.b_cols, uint32_t(g.mma_n), 1)) return cudaErrorInvalidValue;
    p.out[i] = g.out;
    p.ld_out[i] = g.ld_out;
    p.out_rows[i] = g.out_rows;
    p.N[i] = g.N;
    p.K[i] = g.K;
    p.a_k_mod[i] = g.a_k_mod > 0 ? g.a_k_mod : g.K;
    p.b_step[i] = g.b_rows_per_group;
    p.mma_n[i] = g.mma_n;
  }
  p.ksplit = c0.ksplit > 0 ? c0.ksplit : 1;
  p.split_stride = c0.split_stride;
  p.offsets = offsets;
  p.num_routed = num_routed;
  p.rows_single0 = rows_single0;
  p.shared_rows = c1 != nullptr ? shared_rows : 0;
  p.status = status;
  const int grid = int(max_tiles < num_sms() ? max_tiles : num_sms());
  cudaError_t e;
  if (epi != EPI_GATE_F32) return cudaErrorInvalidValue;
  e = launch_epi<EPI_GATE_F32>(p, grid, stream);
  if (e == cudaSuccess && launches) ++*launches;
  return e;
}

}  // namespace moe
