// C ABI of the MoE layer library: argument checks, workspace layout and the
// launch sequence of each call.  See include/moe.h for the contract.
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace moe {

static std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n); }

static void* const* g_prof_events = nullptr;
static int g_prof_n = 0;
static int g_prof_cursor = 0;

void profile_mark(cudaStream_t s) {
  if (g_prof_events != nullptr && g_prof_cursor < g_prof_n)
    cudaEventRecord(static_cast<cudaEvent_t>(g_prof_events[g_prof_cursor++]), s);
}

namespace {

constexpr int kMaxE = 256;
constexpr int kMaxK = 16;
// The tensor-core gate splits K until its output tiles cover the GPU about
// twice (a fixed figure, so workspace sizes do not depend on the device).
constexpr int kGateTargetTiles = 296;
constexpr int kGatePromoteK = 256;   // K per fp32-promoted tensor-core partial sum

constexpr int kTicketFirst = 1, kTicketSecond = 2, kTicketBackward = 3;
constexpr int kStatusInts = 16;
static_assert(kTicketBackward + kBackwardTickets <= kStatusInts, "status block");

struct WsLayout {
  size_t status, logits, wsplit, chunk_counts, chunk_base, counts, offsets, row2tok, tok2row, idx, w, x_perm, h, hs,
      y, ys, done, total;
};

bool is_bf16(const moe_config& c) { return c.act_dtype == MOE_BF16; }
long long I_s(const moe_config& c) { return (long long)c.n_shared * c.I; }

// Both expert GEMMs in one launch pays off when GEMM1 has few tile rounds, so
// its last partial round would leave SMs idle (decode-sized batches); large
// batches run the GEMMs as two launches (measured faster on B300 there).
constexpr long long kFuseMaxRows = 8192;   // T * k
bool fuse_expert_gemms(const moe_config& c) { return (long long)c.T * c.k <= kFuseMaxRows; }

bool use_tc_gate(const moe_config& c) {
  return is_bf16(c) && c.E <= 256;
}

// K ranges of the tensor-core gate: each writes one fp32 partial plane of the
// logits, which the top-k kernel adds in order.  Decode-sized batches have only
// a few output tiles, so they split K the most.
int gate_ksplit(const moe_config& c) {
  if (!use_tc_gate(c) || c.T == 0) return 1;
  const long long tiles = (long long)((c.T + 127) / 128) * ((c.E + 127) / 128);
  const int K = c.gate_w_dtype == MOE_F32 ? 3 * c.d : c.d;
  const int nchunks = (K + kGatePromoteK - 1) / kGatePromoteK;
  long long want = (kGateTargetTiles + tiles - 1) / tiles;
  if (want > nchunks) want = nchunks;
  return want < 1 ? 1 : int(want);
}

WsLayout ws_layout(const moe_config& c) {
  WsLayout L;
  const size_t eb = dtype_bytes(c.act_dtype);
  const size_t R = size_t(c.T) * c.k;
  const size_t nch = size_t(permute_chunks(c.T));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  // the status word, the expert kernel's tile tickets and its GEMM1
  // completion counters: one block that the call's first memset clears
  L.status = take(size_t(kStatusInts) * 4 + size_t(c.E + 1) * 4);
  L.done = L.status + size_t(kStatusInts) * 4;
  L.logits = take(size_t(gate_ksplit(c)) * c.T * c.E * 4);
  L.wsplit = take(use_tc_gate(c) && c.gate_w_dtype == MOE_F32 ? size_t(c.E) * 3 * c.d * 2 : 0);
  L.chunk_counts = take(nch * c.E * 4);
  L.chunk_base = take(nch * c.E * 4);
  L.counts = take(size_t(c.E) * 4);
  L.offsets = take(size_t(c.E + 1) * 4);
  L.row2tok = take(R * 4);
  L.tok2row = take(R * 4);
  L.idx = take(R * 4);
  L.w = take(R * 4);
  L.x_perm = take(R * c.d * eb);
  L.h = take(R * c.I * eb);
  L.hs = take(size_t(c.T) * I_s(c) * eb);
  L.y = take(R * c.d * 4);
  L.ys = take(size_t(c.T) * c.d * 4);
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_config(const moe_config* cp) {
  if (cp == nullptr) return MOE_ERR_INVALID_ARG;
  const moe_config& c = *cp;
  if (c.T < 0 || c.d <= 0 || c.E <= 0 || c.I <= 0 || c.k <= 0 || c.n_shared < 0) return MOE_ERR_INVALID_ARG;
  if (c.act_dtype != MOE_F32 && c.act_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c.gate_w_dtype != MOE_F32 && c.gate_w_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c.out_dtype != MOE_F32 && c.out_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c.expert_w_dtype != c.act_dtype && c.expert_w_dtype != MOE_FP8_E4M3) return MOE_ERR_INVALID_ARG;
  if (c.expert_w_dtype == MOE_FP8_E4M3 && (c.act_dtype != MOE_BF16 || c.d % 128 != 0 || c.I % 128 != 0))
    return MOE_ERR_UNSUPPORTED;
  if (c.score_fn != MOE_SCORE_SOFTMAX && c.score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (c.topk_method != MOE_TOPK_GREEDY && c.topk_method != MOE_TOPK_GROUP_LIMITED) return MOE_ERR_INVALID_ARG;
  if (c.k > c.E) return MOE_ERR_INVALID_ARG;
  if ((long long)c.T * c.k > (1LL << 30)) return MOE_ERR_INVALID_ARG;
  if (c.topk_method == MOE_TOPK_GROUP_LIMITED) {
    if (c.n_group <= 0 || c.E % c.n_group != 0 || c.topk_group <= 0 || c.topk_group > c.n_group)
      return MOE_ERR_INVALID_ARG;
    if (c.group_score != MOE_GROUP_MAX && c.group_score != MOE_GROUP_SUM_TOP) return MOE_ERR_INVALID_ARG;
    const int gsz = c.E / c.n_group;
    if (c.group_score == MOE_GROUP_SUM_TOP && (c.group_top <= 0 || c.group_top > gsz)) return MOE_ERR_INVALID_ARG;
    if ((long long)c.topk_group * gsz < c.k) return MOE_ERR_INVALID_ARG;
    if (c.n_group > 32) return MOE_ERR_UNSUPPORTED;
  }
  if (c.E > kMaxE || c.k > kMaxK) return MOE_ERR_UNSUPPORTED;
  if (is_bf16(c)) {
    // tensor-core tiles: K in steps of 64 (d, I and I_s); whole 256-row weight
    // tiles of interleaved W1/W3 rows per expert (I and I_s multiples of 128)
    if (c.d % 64 != 0 || c.I % 128 != 0 || I_s(c) % 128 != 0) return MOE_ERR_UNSUPPORTED;
  } else {
    if (c.d % 4 != 0) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

struct Ws {
  char* base;
  WsLayout L;
  template <typename T>
  T* at(size_t off) const { return reinterpret_cast<T*>(base + off); }
  int* status() const { return at<int>(L.status); }
};

moe_status check_ws(const moe_config& c, void* ws, size_t ws_bytes, Ws* out) {
  if (ws == nullptr || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  out->base = static_cast<char*>(ws);
  out->L = ws_layout(c);
  if (ws_bytes < out->L.total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// The status word's block also holds the expert kernel's tile ticket counters
// ([1] for a one-launch or GEMM1 launch, [2] for a GEMM2 launch, [3 .. 3 +
// kBackwardTickets) for the backward's launches) and, after kStatusInts ints,
// its E + 1 GEMM1 completion counters.  Every call clears the block with this
// one memset, an ordinary stream operation, before any of its kernels can start.
moe_status reset_status(const Ws& w, cudaStream_t s, int E) {
  return cuda_status(cudaMemsetAsync(w.status(), 0, (kStatusInts + size_t(E) + 1) * sizeof(int), s));
}

moe_status run_gate(const moe_config& c, const void* x, const void* wg, const float* bias, int32_t* idx, float* w,
                    const Ws& ws, cudaStream_t s, int* launches) {
  float* logits = ws.at<float>(ws.L.logits);
  cudaError_t e;
  if (use_tc_gate(c)) {
    GemmClass g;
    g.A = x;
    g.a_rows = c.T;
    g.a_cols = c.d;
    if (c.gate_w_dtype == MOE_F32) {
      void* split = ws.at<void>(ws.L.wsplit);
      e = launch_gate_split(static_cast<const float*>(wg), c.E, c.d, split, s, launches);
      if (e != cudaSuccess) return MOE_ERR_CUDA;
      g.B = split;
      g.b_cols = 3LL * c.d;
      g.K = 3 * c.d;
    } else {
      g.B = wg;
      g.b_cols = c.d;
      g.K = c.d;
    }
    g.b_rows = c.E;
    g.out = logits;
    g.ld_out = c.E;
    g.out_rows = c.T;
    g.N = c.E;
    g.a_k_mod = c.d;
    g.b_rows_per_group = 0;
    g.mma_n = 128;   // 128-column tiles with fp32 promotion of the partial sums
    g.ksplit = gate_ksplit(c);
    g.split_stride = (long long)c.T * c.E;
    e = launch_grouped_gemm(EPI_GATE_F32, g, nullptr, nullptr, 0, c.T, 0, ws.status(),
                            (long long)((c.T + 127) / 128) * ((c.E + 127) / 128) * g.ksplit, s, launches);
  } else {
    e = launch_gate_logits_simt(c, x, wg, logits, s, launches);
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_topk(c, logits, gate_ksplit(c), (long long)c.T * c.E, bias, idx, w, s, launches));
}

moe_status run_experts(const moe_config& c, const void* x_perm, const int32_t* offsets, const void* x,
                       const void* packed, void* y_perm, void* y_shared, const Ws& ws, cudaStream_t s,
                       int* launches) {
  const PackedLayout P = packed_layout(c);
  const char* pb = static_cast<const char*>(packed);
  const long long R = (long long)c.T * c.k;
  const long long Is = I_s(c);
  if (!is_bf16(c)) {
    return cuda_status(launch_swiglu_simt_f32(c, static_cast<const float*>(x_perm), offsets,
                                              static_cast<const float*>(x), packed, ws.at<float>(ws.L.h),
                                              ws.at<float>(ws.L.hs), static_cast<float*>(y_perm),
                                              static_cast<float*>(y_shared), ws.status(), s, launches));
  }
  void* h = ws.at<void>(ws.L.h);
  void* hs = ws.at<void>(ws.L.hs);
  int* done = ws.at<int>(ws.L.done);   // cleared with the status word
  PairClass cls[4];
  // GEMM1 + SwiGLU: H[rows, I] = silu(X W1^T) * (X W3^T), packed W1/W3 rows [2I, d] per expert.
  // FP8 weights: x_perm and H hold f16 rows (see launch_pair_experts).
  const int32_t* eref = P.fp8 ? reinterpret_cast<const int32_t*>(pb + P.eref) : nullptr;
  PairClass& r1 = cls[0];
  r1.W = pb + P.w13; r1.w_rows = 2LL * c.E * c.I; r1.X = x_perm; r1.x_rows = R; r1.K = c.d;
  r1.M = 2 * c.I; r1.w_step = 2 * c.I; r1.out = h; r1.ld_out = c.I; r1.out_rows = R;
  PairClass& s1 = cls[1];
  s1.W = pb + P.w13s; s1.w_rows = 2 * Is; s1.X = x; s1.x_rows = c.T; s1.K = c.d;
  s1.M = int(2 * Is); s1.w_step = 0; s1.out = hs; s1.ld_out = Is; s1.out_rows = c.T;
  // GEMM2: Y[rows, d] = H W2^T (fp32), W2 [d, I] per expert
  PairClass& r2 = cls[2];
  r2.W = pb + P.w2; r2.w_rows = (long long)c.E * c.d; r2.X = h; r2.x_rows = R; r2.K = c.I;
  r2.M = c.d; r2.w_step = c.d; r2.out = y_perm; r2.ld_out = c.d; r2.out_rows = R;
  PairClass& s2 = cls[3];
  s2.W = pb + P.w2s; s2.w_rows = c.d; s2.X = hs; s2.x_rows = c.T; s2.K = int(Is);
  s2.M = c.d; s2.w_step = 0; s2.out = y_shared; s2.ld_out = c.d; s2.out_rows = c.T;
  for (PairClass& q : cls) q.img = P.img;   // bf16 weights: contiguous stage blocks
  // upper bound of the pair tiles (256 tokens x 256 weight rows), for sizing the grid
  const long long tb_routed = R / 256 + c.E;
  const long long tb_shared = Is > 0 ? (c.T + 255) / 256 : 0;
  const long long tiles1 = tb_routed * ((2LL * c.I + 255) / 256) + tb_shared * ((2 * Is + 255) / 256);
  const long long tiles2 = (tb_routed + tb_shared) * ((c.d + 255) / 256);
  const int shared_rows = Is > 0 ? c.T : 0;
  if (P.fp8 && c.T <= GEMV_MAX_T) {
    // decode batches of FP8 experts: GEMV with warp-level MMAs (a group holds at most T rows)
    GemvOperands g1, g1s, g2, g2s;
    g1.w = pb + P.w13; g1.x = x_perm; g1.x_f16 = true; g1.out = h; g1.out_ld = c.I; g1.M = 2 * c.I; g1.K = c.d;
    g1s.w = pb + P.w13s; g1s.x = x; g1s.x_f16 = false; g1s.out = hs; g1s.out_ld = Is; g1s.M = int(2 * Is);
    g1s.K = c.d;
    g2.w = pb + P.w2; g2.x = h; g2.x_f16 = true; g2.out = y_perm; g2.out_ld = c.d; g2.M = c.d; g2.K = c.I;
    g2s.w = pb + P.w2s; g2s.x = hs; g2s.x_f16 = true; g2s.out = y_shared; g2s.out_ld = c.d; g2s.M = c.d;
    g2s.K = int(Is);
    cudaError_t e = launch_fp8_gemv(g1, Is > 0 ? &g1s : nullptr, offsets, c.E, shared_rows, c.T, R, true, false,
                                    ws.status(), s, launches);
    if (e == cudaSuccess)
      e = launch_fp8_gemv(g2, Is > 0 ? &g2s : nullptr, offsets, c.E, shared_rows, c.T, R, false, true,
                          ws.status(), s, launches);
    return cuda_status(e);
  }
  int* tickets = ws.status();
  if (fuse_expert_gemms(c)) {
    // one launch: GEMM2 tiles start expert by expert while GEMM1 finishes
    return cuda_status(launch_pair_experts(cls, offsets, c.E, shared_rows, c.T, 3, done, tickets + kTicketFirst,
                                           ws.status(), tiles1 + tiles2, s, launches, eref));
  }
  cudaError_t e = launch_pair_experts(cls, offsets, c.E, shared_rows, c.T, 1, nullptr, tickets + kTicketFirst,
                                      ws.status(), tiles1, s, launches, eref);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_pair_experts(cls, offsets, c.E, shared_rows, c.T, 2, nullptr, tickets + kTicketSecond,
                                         ws.status(), tiles2, s, launches, eref));
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(*cfg).total;
  return MOE_OK;
}

moe_status moe_packed_size(const moe_config* cfg, size_t* bytes) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = packed_layout(*cfg).total;
  return MOE_OK;
}

moe_status moe_prepack_experts(const moe_config* cfg, const void* W1, const void* W3, const void* W2,
                               const void* Ws1, const void* Ws3, const void* Ws2, void* packed, size_t packed_bytes,
                               void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  const bool shared = I_s(c) > 0;
  if (!W1 || !W3 || !W2 || !packed || (shared && (!Ws1 || !Ws3 || !Ws2))) return MOE_ERR_INVALID_ARG;
  if (!aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(packed)) return MOE_ERR_INVALID_ARG;
  if (shared && (!aligned16(Ws1) || !aligned16(Ws3) || !aligned16(Ws2))) return MOE_ERR_INVALID_ARG;
  if (packed_bytes < packed_layout(c).total) return MOE_ERR_WORKSPACE;
  int n = 0;
  cudaError_t e = launch_prepack(c, W1, W3, W2, Ws1, Ws3, Ws2, packed, static_cast<cudaStream_t>(stream), &n);
  count_launches(n);
  return cuda_status(e);
}

moe_status moe_gate_topk(const moe_config* cfg, const void* x, const void* Wg, const float* bias, int32_t* idx,
                         float* w, void* ws, size_t ws_bytes, void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  if (!x || !Wg || !idx || !w || !aligned16(x) || !aligned16(Wg) || !aligned16(idx) || !aligned16(w))
    return MOE_ERR_INVALID_ARG;
  if (bias != nullptr && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
  Ws W;
  if ((st = check_ws(c, ws, ws_bytes, &W)) != MOE_OK) return st;
  if (c.T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = reset_status(W, s, c.E)) != MOE_OK) return st;
  int n = 0;
  st = run_gate(c, x, Wg, bias, idx, w, W, s, &n);
  count_launches(n);
  return st;
}

moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* idx, int32_t* counts, int32_t* offsets,
                       int32_t* row2tok, int32_t* tok2row, void* x_perm, void* ws, size_t ws_bytes, void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  if (!x || !idx || !counts || !offsets || !row2tok || !tok2row || !x_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(idx) || !aligned16(counts) || !aligned16(offsets) || !aligned16(row2tok) ||
      !aligned16(tok2row) || !aligned16(x_perm))
    return MOE_ERR_INVALID_ARG;
  Ws W;
  if ((st = check_ws(c, ws, ws_bytes, &W)) != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c.T == 0) {
    // no tokens: every expert is empty
    if (cudaMemsetAsync(offsets, 0, size_t(c.E + 1) * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(cudaMemsetAsync(counts, 0, size_t(c.E) * 4, s));
  }
  if ((st = reset_status(W, s, c.E)) != MOE_OK) return st;
  int n = 0;
  cudaError_t e = launch_permute(c, x, idx, counts, offsets, row2tok, tok2row, x_perm, W.at<int32_t>(W.L.chunk_counts),
                                 W.at<int32_t>(W.L.chunk_base), W.status(), s, &n);
  count_launches(n);
  return cuda_status(e);
}

moe_status moe_grouped_swiglu(const moe_config* cfg, const void* x_perm, const int32_t* offsets, const void* x,
                              const void* packed, void* y_perm, void* y_shared, void* ws, size_t ws_bytes,
                              void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  if (!x_perm || !offsets || !x || !packed || !y_perm || !y_shared) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(offsets) || !aligned16(x) || !aligned16(packed) || !aligned16(y_perm) ||
      !aligned16(y_shared))
    return MOE_ERR_INVALID_ARG;
  Ws W;
  if ((st = check_ws(c, ws, ws_bytes, &W)) != MOE_OK) return st;
  if (c.T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = reset_status(W, s, c.E)) != MOE_OK) return st;
  int n = 0;
  if (c.expert_w_dtype == MOE_FP8_E4M3) {
    // the FP8 expert GEMM takes f16 token rows: convert into the workspace's x_perm
    void* x16 = W.at<void>(W.L.x_perm);
    if (launch_bf16_to_f16(x_perm, x16, (long long)c.T * c.k * c.d, W.status(), s, &n) != cudaSuccess) {
      count_launches(n);
      return MOE_ERR_CUDA;
    }
    x_perm = x16;
  }
  st = run_experts(c, x_perm, offsets, x, packed, y_perm, y_shared, W, s, &n);
  count_launches(n);
  return st;
}

moe_status moe_combine(const moe_config* cfg, const void* y_perm, const void* y_shared, const int32_t* tok2row,
                       const float* w, void* out, void* ws, size_t ws_bytes, void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  if (!y_perm || !y_shared || !tok2row || !w || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(y_shared) || !aligned16(tok2row) || !aligned16(w) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  Ws W;
  if ((st = check_ws(c, ws, ws_bytes, &W)) != MOE_OK) return st;
  if (c.T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = reset_status(W, s, c.E)) != MOE_OK) return st;
  int n = 0;
  cudaError_t e = launch_combine(c, y_perm, y_shared, tok2row, w, out, W.status(), s, &n);
  count_launches(n);
  return cuda_status(e);
}

moe_status moe_forward(const moe_config* cfg, const void* x, const void* Wg, const float* bias, const void* packed,
                       void* out, int32_t* idx_out, float* w_out, int32_t* counts_out, void* ws, size_t ws_bytes,
                       void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  if (!x || !Wg || !packed || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(packed) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if ((bias && !aligned16(bias)) || (idx_out && !aligned16(idx_out)) || (w_out && !aligned16(w_out)) ||
      (counts_out && !aligned16(counts_out)))
    return MOE_ERR_INVALID_ARG;
  Ws W;
  if ((st = check_ws(c, ws, ws_bytes, &W)) != MOE_OK) return st;
  if (c.T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = reset_status(W, s, c.E)) != MOE_OK) return st;
  int n = 0;
  int32_t* idx = idx_out ? idx_out : W.at<int32_t>(W.L.idx);
  float* w = w_out ? w_out : W.at<float>(W.L.w);
  int32_t* counts = counts_out ? counts_out : W.at<int32_t>(W.L.counts);
  int32_t* offsets = W.at<int32_t>(W.L.offsets);
  int32_t* tok2row = W.at<int32_t>(W.L.tok2row);
  void* x_perm = W.at<void>(W.L.x_perm);
  void* y = W.at<void>(W.L.y);
  void* ys = W.at<void>(W.L.ys);
  profile_mark(s);
  st = run_gate(c, x, Wg, bias, idx, w, W, s, &n);
  if (st == MOE_OK) {
    profile_mark(s);
    cudaError_t e = launch_permute(c, x, idx, counts, offsets, W.at<int32_t>(W.L.row2tok), tok2row, x_perm,
                                   W.at<int32_t>(W.L.chunk_counts), W.at<int32_t>(W.L.chunk_base), W.status(), s, &n,
                                   c.expert_w_dtype == MOE_FP8_E4M3);
    st = cuda_status(e);
  }
  if (st == MOE_OK) {
    profile_mark(s);
    st = run_experts(c, x_perm, offsets, x, packed, y, ys, W, s, &n);
  }
  if (st == MOE_OK) {
    profile_mark(s);
    st = cuda_status(launch_combine(c, y, ys, tok2row, w, out, W.status(), s, &n));
  }
  if (st == MOE_OK) profile_mark(s);
  count_launches(n);
  return st;
}

moe_status moe_backward_workspace_size(const moe_config* cfg, size_t* bytes) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  const moe_config& c = *cfg;
  // bf16 only; d a multiple of 128 (the products read each expert's weights in
  // whole 128-row stages through transposed views)
  if (!is_bf16(c) || c.expert_w_dtype != MOE_BF16 || c.d % 128 != 0) return MOE_ERR_UNSUPPORTED;
  *bytes = ws_layout(c).total + backward_extra_bytes(c);
  return MOE_OK;
}

moe_status moe_backward(const moe_config* cfg, const void* x, const void* Wg, const float* bias, const void* W1,
                        const void* W3, const void* W2, const void* Ws1, const void* Ws3, const void* Ws2,
                        const void* dout, float* dx, float* dWg, float* dW1, float* dW3, float* dW2, float* dWs1,
                        float* dWs3, float* dWs2, void* ws, size_t ws_bytes, void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  // bf16 only; d a multiple of 128 (the products read each expert's weights in
  // whole 128-row stages through transposed views)
  if (!is_bf16(c) || c.expert_w_dtype != MOE_BF16 || c.d % 128 != 0) return MOE_ERR_UNSUPPORTED;
  const bool shared = c.n_shared > 0;
  const void* need[] = {x, Wg, W1, W3, W2, dout, dx, dWg, dW1, dW3, dW2};
  for (const void* q : need)
    if (q == nullptr || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (shared) {
    const void* need_s[] = {Ws1, Ws3, Ws2, dWs1, dWs3, dWs2};
    for (const void* q : need_s)
      if (q == nullptr || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  }
  if (bias && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  Ws W;
  W.base = static_cast<char*>(ws);
  W.L = ws_layout(c);
  const BwdLayout B = backward_layout(c, W.L.total);
  if (ws_bytes < W.L.total + B.total) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c.T == 0) {
    // no token: every gradient is zero
    const long long Is = I_s(c);
    const struct {
      void* p;
      size_t n;
    } z[] = {{dWg, size_t(c.E) * c.d}, {dW1, size_t(c.E) * c.I * c.d}, {dW3, size_t(c.E) * c.I * c.d},
             {dW2, size_t(c.E) * c.d * c.I}, {dWs1, size_t(Is) * c.d}, {dWs3, size_t(Is) * c.d},
             {dWs2, size_t(c.d) * Is}};
    for (const auto& q : z)
      if (q.p && q.n && cudaMemsetAsync(q.p, 0, q.n * sizeof(float), s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  if ((st = reset_status(W, s, c.E)) != MOE_OK) return st;
  int n = 0;
  int32_t* idx = W.at<int32_t>(W.L.idx);
  float* w = W.at<float>(W.L.w);
  st = run_gate(c, x, Wg, bias, idx, w, W, s, &n);
  // the dispatch tables only: the backward gathers the tokens into its own padded layout
  if (st == MOE_OK)
    st = cuda_status(launch_permute(c, nullptr, idx, W.at<int32_t>(W.L.counts), W.at<int32_t>(W.L.offsets),
                                    W.at<int32_t>(W.L.row2tok), W.at<int32_t>(W.L.tok2row), nullptr,
                                    W.at<int32_t>(W.L.chunk_counts), W.at<int32_t>(W.L.chunk_base), W.status(), s, &n));
  count_launches(n);
  if (st != MOE_OK) return st;
  BwdPtrs p;
  p.x = x;
  p.Wg = Wg;
  p.W1 = W1;
  p.W3 = W3;
  p.W2 = W2;
  p.Ws1 = Ws1;
  p.Ws3 = Ws3;
  p.Ws2 = Ws2;
  p.dout = dout;
  p.dx = dx;
  p.dWg = dWg;
  p.dW1 = dW1;
  p.dW3 = dW3;
  p.dW2 = dW2;
  p.dWs1 = dWs1;
  p.dWs3 = dWs3;
  p.dWs2 = dWs2;
  p.idx = idx;
  p.gates = w;
  p.offsets = W.at<int32_t>(W.L.offsets);
  p.tok2row = W.at<int32_t>(W.L.tok2row);
  p.logits = W.at<float>(W.L.logits);
  p.ksplit = gate_ksplit(c);
  p.plane = (long long)c.T * c.E;
  p.status = W.status();
  p.tickets = W.status() + kTicketBackward;
  p.base = W.base;
  return cuda_status(run_backward_core(c, p, B, s));
}

moe_status moe_balance_update(const moe_config* cfg, const int32_t* counts, float* bias, float gamma, float* stats,
                              int32_t* device_status, void* stream) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (!counts || !bias || !aligned16(counts) || !aligned16(bias)) return MOE_ERR_INVALID_ARG;
  if (stats != nullptr && !aligned16(stats)) return MOE_ERR_INVALID_ARG;
  if (!(gamma == gamma) || gamma > 3.0e38f || gamma < -3.0e38f) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (device_status != nullptr && cudaMemsetAsync(device_status, 0, sizeof(int32_t), s) != cudaSuccess)
    return MOE_ERR_CUDA;
  int n = 0;
  cudaError_t e = launch_balance_update(*cfg, counts, bias, gamma, stats, device_status, s, &n);
  count_launches(n);
  return cuda_status(e);
}

moe_status moe_get_device_status(const void* ws, void* stream, int32_t* detail) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t word = 0;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (detail) *detail = word;
  if (word & DEV_TIMEOUT) return MOE_ERR_DEVICE_TIMEOUT;
  if (word & (DEV_BAD_EXPERT | DEV_BAD_ROW)) return MOE_ERR_DEVICE_BOUNDS;
  if (word & DEV_RANGE) return MOE_ERR_DEVICE_RANGE;
  return MOE_OK;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS";
    case MOE_ERR_DEVICE_RANGE: return "MOE_ERR_DEVICE_RANGE";
  }
  return "MOE_ERR_UNKNOWN";
}

uint64_t moe_launch_count(void) { return g_launches.load(); }

moe_status moe_debug_inject(int32_t what, int64_t value) {
  unsigned long long wait_ns = 0;
  int extra = 0;
  get_expert_fault(&wait_ns, &extra);
  switch (what) {
    case MOE_DEBUG_WAIT_LIMIT_NS:
      if (value < 0 || value > 10000000000LL) return MOE_ERR_INVALID_ARG;
      if (value != 0 && value < 100000) return MOE_ERR_INVALID_ARG;   // at least 0.1 ms
      set_expert_fault((unsigned long long)value, extra);
      return MOE_OK;
    case MOE_DEBUG_STALL_GEMM2:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      set_expert_fault(wait_ns, int(value));
      return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status moe_profile_arm(void* const* events, int32_t n_events) {
  if (events != nullptr && n_events < 0) return MOE_ERR_INVALID_ARG;
  g_prof_events = n_events > 0 ? events : nullptr;
  g_prof_n = events != nullptr ? n_events : 0;
  g_prof_cursor = 0;
  return MOE_OK;
}

const char* moe_forward_stage_name(int32_t i) {
  static const char* names[MOE_FORWARD_STAGES] = {"router", "permute", "experts", "combine"};
  return (i >= 0 && i < MOE_FORWARD_STAGES) ? names[i] : nullptr;
}

int32_t moe_forward_kernel_count(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return -1;
  const moe_config& c = *cfg;
  if (c.T == 0) return 0;
  int n = 2;                                                        // logits + top-k
  if (use_tc_gate(c) && c.gate_w_dtype == MOE_F32) n += 1;          // W_g split
  n += permute_launches(c.T) + 1;                                   // permute + gather
  const bool gemv = c.expert_w_dtype == MOE_FP8_E4M3 && c.T <= GEMV_MAX_T;
  n += is_bf16(c) && !gemv && fuse_expert_gemms(c) ? 1 : 2;         // expert GEMMs
  n += 1;                                                           // combine
  return n;
}

}  // extern "C"
