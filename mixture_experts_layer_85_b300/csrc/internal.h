// Host-side launchers shared between the kernel files and the C ABI (api.cu).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"

namespace moe {

// Launch with programmatic stream serialization: the kernel may start while
// its predecessor in the stream is still running (it calls pdl_wait() before
// depending on it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// One-time set-up per device (a kernel's shared-memory attribute, an
// occupancy figure, a symbol address): get() runs `init` the first time it
// is called with a given current device and returns the stored value on
// later calls on that device.  Thread-safe.  A context reset
// (cudaDeviceReset) does not clear it.
constexpr int kMaxDevices = 64;
template <typename T>
class PerDevice {
 public:
  template <typename F>
  cudaError_t get(T* out, F&& init) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu_);
    if (!ready_[dev]) {
      T v{};
      e = init(&v);
      if (e != cudaSuccess) return e;
      value_[dev] = v;
      ready_[dev] = true;
    }
    *out = value_[dev];
    return cudaSuccess;
  }

 private:
  std::mutex mu_;
  bool ready_[kMaxDevices] = {};
  T value_[kMaxDevices] = {};
};

// ---------------------------------------------------------------- grouped GEMM
// One operand class of the grouped GEMM: A [a_rows, K'] and B [b_rows, K] bf16,
// both K-major (row-major with K contiguous).  Class 0 holds either the routed
// groups (rows of group g start at offsets[g]) or a single group of
// `rows_single0` rows; class 1 holds one group (the shared expert, T rows).
struct GemmClass {
  const void* A = nullptr;
  int64_t a_rows = 0, a_cols = 0;
  const void* B = nullptr;
  int64_t b_rows = 0, b_cols = 0;
  void* out = nullptr;
  int64_t ld_out = 0;       // output row stride in elements
  int64_t out_rows = 0;     // rows of the output buffer (store bound)
  int N = 0;                // columns of D before the epilogue
  int K = 0;                // reduction length (multiple of 64)
  int a_k_mod = 0;          // A column = k % a_k_mod (K-split gate); = K otherwise
  int b_rows_per_group = 0; // B row step between consecutive groups of the class
  int mma_n = 256;          // MMA N (<= 256, multiple of 16); B box rows
  int ksplit = 1;           // EPI_GATE_F32 only: K ranges, one fp32 partial plane each
  int64_t split_stride = 0; // elements between partial planes
};

enum EpiMode : int { EPI_GATE_F32 = 3 };

int num_sms();

// cuTensorMapEncodeTiled from the driver (nullptr when unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// bf16 tensor map of a row-major [rows, cols] buffer, 128-byte swizzle, boxes
// of 64 columns x box_rows rows x box_kblocks consecutive 64-column k-blocks
// (box_kblocks = 1: a plain 2-D map).  Cached by argument.
bool encode_bf16_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, uint32_t box_rows,
                     uint32_t box_kblocks);
// 4-D bf16 map over `blocks` stage blocks (the layout of IMG_BLOCK_BYTES
// blocks above), one block per box, 128-byte swizzle.
bool encode_stage_block_map(CUtensorMap* m, const void* ptr, long long blocks);
// The same for elem_bytes 1 (bytes: FP8 weights) or 2 (bf16); the inner box
// extent is one 128-byte row.
bool encode_tiled_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int elem_bytes,
                      uint32_t box_rows, uint32_t box_kblocks);


// Records the next armed profiling event on `s` (no-op when disarmed).
void profile_mark(cudaStream_t s);

cudaError_t launch_grouped_gemm(int epi, const GemmClass& c0, const GemmClass* c1, const int32_t* offsets,
                                int num_routed, int rows_single0, int shared_rows, int* status,
                                long long max_tiles, cudaStream_t stream, int* launches);

// ------------------------------------------------------- expert GEMMs (pairs)
// One operand class of the CTA-pair expert GEMM, D = W * X^T per group: W
// [w_rows, K] weight rows (group g of class 0 starts at row g * w_step; M rows
// per group), X [x_rows, K] token rows (class 0: rows offsets[g] ..
// offsets[g+1]; class 1: one group of shared_rows rows), both bf16 K-major.
struct PairClass {
  const void* W = nullptr;   // bf16 rows, bf16 stage blocks (img), or FP8 stage images (fp8_tiled_bytes layout)
  int64_t w_rows = 0;
  bool img = false;          // W holds bf16 stage blocks of groups of M rows and K columns
  const void* X = nullptr;
  int64_t x_rows = 0;
  int K = 0;               // multiple of 64
  int M = 0;               // weight rows (output features before SwiGLU) per group
  int w_step = 0;
  void* out = nullptr;     // [rows, M/2] bf16 (SwiGLU) or [rows, M] fp32
  int64_t ld_out = 0;
  int64_t out_rows = 0;
};

// The expert GEMMs.  cls = {GEMM1 routed, GEMM1 shared, GEMM2 routed, GEMM2
// shared}; GEMM1 outputs bf16 silu(W1 x) * (W3 x) (W = packed W1/W3 rows,
// 16-row interleave), GEMM2 fp32.  phases: 1 = GEMM1 tiles, 2 = GEMM2 tiles,
// 3 = both in one launch, GEMM2 tiles of a group waiting on per-group GEMM1
// completion counters done [num_routed + 1], which must then be zero before
// anything of the call that launches it starts (the kernel may start early).  ticket: the launch's tile ticket counter, zero when the
// launch starts (and not touched by anything that may still run then).
// max_group_rows: an upper bound of any group's rows (the batch size T).  The
// shared expert's GEMM1 tiles may run before the preceding grid completes.
// fp8_eref (non-null: FP8 weights): the weights are FP8 stage images (one
// bulk copy per stage), dequantized by converter warps before each MMA, and
// fp8_eref [num_routed + 1][3] holds each group's reference exponents of its
// W1, W3 and W2.  The shared expert's GEMM1 (bf16 x) then dequantizes to bf16
// with the full block scales; every other tile takes f16 token rows (x_perm as
// f16, and the hidden rows GEMM1 writes as f16), dequantizes to f16 relative
// to the reference exponent and scales its fp32 accumulator by 2^e_ref.
cudaError_t launch_pair_experts(const PairClass cls[4], const int32_t* offsets, int num_routed, int shared_rows,
                                int max_group_rows, int phases, int* done, int* ticket, int* status,
                                long long max_tiles, cudaStream_t stream, int* launches,
                                const int32_t* fp8_eref = nullptr);

// FP8 expert FFNs for decode batches as a GEMV with warp-level MMAs
// (csrc/gemv_fp8.cu): every group holds at most GEMV_MAX_T token rows, taken
// GEMV_MAX_ROWS at a time (the MMA's N).  One launch per GEMM: gemm1 = GEMM1
// with the SwiGLU epilogue (f16 hidden rows [rows, M/2]), else GEMM2 (fp32
// rows [rows, M]).  w: FP8 stage images of groups of M rows and K
// columns; x: token rows, K 2-byte values each (x_f16: f16, else bf16).  The
// routed class's groups take rows offsets[g] .. offsets[g+1] (all below
// routed_rows); the shared class, rows 0 .. shared_rows; no group holds more
// than max_rows (<= GEMV_MAX_T; a group that does is flagged and skipped).
// x_from_prev: every item's token rows come from the preceding grid (else
// only the routed ones).
constexpr int GEMV_MAX_ROWS = 8;
constexpr int GEMV_MAX_T = 64;
struct GemvOperands {
  const void* w = nullptr;
  const void* x = nullptr;
  bool x_f16 = false;
  void* out = nullptr;
  long long out_ld = 0;
  int M = 0, K = 0;
};
cudaError_t launch_fp8_gemv(const GemvOperands& routed, const GemvOperands* shared, const int32_t* offsets,
                            int num_routed, int shared_rows, int max_rows, long long routed_rows, bool gemm1,
                            bool x_from_prev, int* status, cudaStream_t stream, int* launches);

// Fault injection for tests of the device-side time-out path
// (moe_debug_inject): the expert kernel's wait limit for later launches
// (0 = kWaitLimitNs) and the extra GEMM1 completions each GEMM2 tile of a
// one-launch expert kernel waits for (> 0 makes those waits run out).
void set_expert_fault(unsigned long long wait_ns, int need_extra);
void get_expert_fault(unsigned long long* wait_ns, int* need_extra);

// One operand class of a launch of the expert kernel with fp32 output rows
// (GEMM2 tiles only), for products beyond the forward's: D[f][j] = sum_k
// A[f][k] * B[j][k], out[j][f] (row j, column f, ld_out).
//   A: K-major rows [a_rows, a_cols = K] (group g from row g * w_step), or
//      MN-major (a_mn): a row-major [a_rows = K rows][a_cols = M] buffer read
//      transposed, group g's K rows from g * a_kstep; with A2 the K indices
//      from K1 on come from A2 (same layout, a2_rows rows).
//   B: K-major token rows [b_rows, b_cols = K], or MN-major (b_mn): a
//      row-major [b_rows = K rows][b_cols = N] buffer read transposed.
//   kmode launches (weight gradients): the token rows are K, N is fixed, and
//   the routed output moves out_gstride elements per group.
struct PairOperands {
  const void* A = nullptr;
  int64_t a_rows = 0, a_cols = 0;
  bool a_mn = false;
  const void* A2 = nullptr;
  int64_t a2_rows = 0;
  int K1 = 0;
  int a_kstep = 0;
  int w_step = 0;
  const void* B = nullptr;
  int64_t b_rows = 0, b_cols = 0;
  bool b_mn = false;
  int b_col0 = 0;           // MN-major B: first column of N within the buffer's b_cols
  int M = 0, K = 0, N = 0;
  float* out = nullptr;
  int64_t ld_out = 0, out_rows = 0, out_gstride = 0;
};
// routed (nullable when num_routed = 0) over groups g with rows offsets[g] ..
// offsets[g+1] (starting at row_base[g] when given), shared (nullable) over
// shared_rows token rows (kmode: the K extent, a multiple of 128).
cudaError_t launch_pair_gemm(const PairOperands* routed, const PairOperands* shared, const int32_t* offsets,
                             const int32_t* row_base, long long row_bound, int num_routed, int shared_rows,
                             int kmode, int* ticket, int* status, long long max_tiles, cudaStream_t stream,
                             int* launches);

// ---------------------------------------------------------------------- router
cudaError_t launch_gate_split(const float* wg, int E, int d, void* wsplit, cudaStream_t s, int* launches);
cudaError_t launch_gate_logits_simt(const moe_config& c, const void* x, const void* wg, float* logits,
                                    cudaStream_t s, int* launches);
// logits: `nsplit` fp32 partial planes of [T,E], `plane` elements apart, summed
// in plane order before scoring (nsplit = 1: plain logits).
cudaError_t launch_topk(const moe_config& c, const float* logits, int nsplit, long long plane, const float* bias,
                        int32_t* idx, float* w, cudaStream_t s, int* launches);

// ---------------------------------------------------------------- permutation
int permute_chunks(int T);
int permute_launches(int T);   // kernels of steps 1-3 (the gather is one more)
// x or x_perm null: the dispatch tables only (no gather).  x_perm_f16: bf16
// rows of x are written to x_perm as f16 (the FP8 expert GEMM's token
// operand); a value that rounds beyond the f16 range sets DEV_RANGE.
cudaError_t launch_permute(const moe_config& c, const void* x, const int32_t* idx, int32_t* counts,
                           int32_t* offsets, int32_t* row2tok, int32_t* tok2row, void* x_perm,
                           int32_t* chunk_counts, int32_t* chunk_base, int* status, cudaStream_t s,
                           int* launches, bool x_perm_f16 = false);
// n bf16 values (n a multiple of 8, 16-byte aligned) to f16, DEV_RANGE as above.
cudaError_t launch_bf16_to_f16(const void* src, void* dst, long long n, int* status, cudaStream_t s, int* launches);

// x rows [T, row_bytes] -> x_perm rows tok2row[t][j] (rows < `rows`; -1 skipped).
cudaError_t launch_gather_rows(const void* x, const int32_t* tok2row, int T, int k, long long rows, size_t row_bytes,
                               void* x_perm, int* status, cudaStream_t s, int* launches);

// -------------------------------------------------------------------- experts
cudaError_t launch_prepack(const moe_config& c, const void* W1, const void* W3, const void* W2,
                           const void* Ws1, const void* Ws3, const void* Ws2, void* packed, cudaStream_t s,
                           int* launches);
cudaError_t launch_swiglu_simt_f32(const moe_config& c, const float* x_perm, const int32_t* offsets,
                                   const float* x, const void* packed, float* h, float* hs, float* y,
                                    float* ys, int* status, cudaStream_t s, int* launches);

// -------------------------------------------------------------------- combine
cudaError_t launch_combine(const moe_config& c, const void* y_perm, const void* y_shared,
                           const int32_t* tok2row, const float* w, void* out, int* status, cudaStream_t s,
                           int* launches);

// ----------------------------------------------------------- load balancing
cudaError_t launch_balance_update(const moe_config& c, const int32_t* counts, float* bias, float gamma, float* stats,
                                  int* status, cudaStream_t s, int* launches);

// FP8 expert weights are stored as the expert GEMM's shared-memory images:
// tiles of 128 rows, each a run of cols / 128 stage blocks of FP8_STAGE_BYTES
// (128 x 128 e4m3 values with the 128-byte swizzle, then their int32 scale
// exponents [2][128]), plus one zero tile after the last row.  The layout's
// eref area holds int32 [E+1][3]: for each group's W1, W3 and W2 (the shared
// expert at E) the exponent its largest |w| gets by the block rule (the
// largest exponent among its nonzero blocks; 0 for a zero matrix).
constexpr int FP8_IMAGE_BYTES = 128 * 128;
constexpr int FP8_STAGE_BYTES = FP8_IMAGE_BYTES + 2 * 128 * 4;
inline size_t fp8_tiled_bytes(long long rows, long long cols) {
  return size_t(rows / 128 + 1) * size_t(cols / 128) * FP8_STAGE_BYTES;
}

// Packed expert blob layout (byte offsets, each 256-byte aligned).
// bf16 expert weights are stored as stage blocks: per group, per tile of 128
// output rows and per stage of 128 reduction columns, the two 64-column
// k-blocks of the tile, each 128 rows x 64 bf16 (16 KB, rows of 128 B), so one
// stage is 32 KB contiguous (zero-padded past the matrix's rows or columns).
constexpr int IMG_ROWS = 128, IMG_COLS = 128;
constexpr int IMG_BLOCK_BYTES = IMG_ROWS * IMG_COLS * 2;
inline int img_tiles(long long rows_per_group) { return int((rows_per_group + IMG_ROWS - 1) / IMG_ROWS); }
inline int img_stages(long long cols) { return int((cols + IMG_COLS - 1) / IMG_COLS); }
inline size_t img_bytes(long long groups, long long rows_per_group, long long cols) {
  return size_t(groups) * img_tiles(rows_per_group) * img_stages(cols) * IMG_BLOCK_BYTES;
}

struct PackedLayout {
  size_t w13 = 0, w2 = 0, w13s = 0, w2s = 0, eref = 0, total = 0;
  bool fp8 = false;
  bool img = false;      // bf16 stage blocks (otherwise row-major, the fp32 path)
  int bi = 0, bis = 0;   // interleave block of W1/W3 rows (routed, shared)
};
PackedLayout packed_layout(const moe_config& c);

// --------------------------------------------------------------- backward
// Backward-only workspace (byte offsets from the forward workspace's start,
// 256-byte aligned).  Routed rows use a padded layout of R_max rows: expert g's
// rows start at koff[g], a multiple of 128, pad rows zero.
struct BwdLayout {
  size_t koff, tok2row_pad, Xp, G, U, H, Y, dY, dH, dGU, Gs, Us, Hs, dHs, dGUs, dXs, doutb, dout32, dlb, dg, dXg, wgb,
      total;
  long long R_max;
  int E_pad;
};
BwdLayout backward_layout(const moe_config& c, size_t base);
size_t backward_extra_bytes(const moe_config& c);

// One backward call: the caller's tensors and the forward router's results
// in the workspace (routing, dispatch, the logits planes).
struct BwdPtrs {
  const void *x, *Wg, *W1, *W3, *W2, *Ws1, *Ws3, *Ws2, *dout;
  float *dx, *dWg, *dW1, *dW3, *dW2, *dWs1, *dWs3, *dWs2;
  const int32_t *idx, *offsets, *tok2row;
  const float* gates;
  const float* logits;   // `ksplit` fp32 partial planes of [T, E], `plane` elements apart
  int ksplit;
  long long plane;
  int* status;
  int* tickets;          // zeroed tile ticket counters, one per expert-kernel launch (10)
  char* base;            // workspace base
};
constexpr int kBackwardTickets = 10;
// Everything after the routing and dispatch, stream-ordered, no host synchronisation.
cudaError_t run_backward_core(const moe_config& c, const BwdPtrs& p, const BwdLayout& L, cudaStream_t s);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline size_t dtype_bytes(int dt) { return dt == MOE_BF16 ? 2 : 4; }

}  // namespace moe
