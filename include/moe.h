/*
 * moe.h - C ABI of the DeepSeekMoE layer forward on one B300 GPU (sm_103a).
 *
 * The layer (DeepSeek-V2 walkthrough, "DeepSeekMoE" output definition and the
 * MoEGate / MoE listings; V3 architecture page, section 1.2):
 *
 *   h'_t = sum_{j<k} g_{t,j} * FFN_{idx_{t,j}}(u_t) + FFN_shared(u_t)
 *   FFN(u) = W2 (silu(W1 u) * (W3 u))                      (SwiGLU, no bias)
 *
 * with idx/g from the router: logits = u W_g^T, s = softmax (over all E) or
 * sigmoid, selection score s + b (b steers selection only), greedy or
 * group-limited top-k, g = s_idx (optionally renormalised) * scale.
 * No residual term is added.
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers, owned by the caller, 16-byte
 *    aligned, dense row-major.  Weights use the nn.Linear layout (out x in).
 *    The library never allocates or frees device memory.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  Arguments are validated on the host first; on any error the call
 *    returns a non-zero moe_status and launches nothing.
 *  - Every call's kernels start only after all earlier work in `stream` has
 *    completed (the call begins with an ordinary stream operation, clearing
 *    its status word, or with a kernel that waits for its predecessor before
 *    letting its successors start).  Inside one call, a kernel may begin while
 *    its predecessor finishes, but only where it touches nothing that
 *    predecessor writes.  So a layer's output may be the next call's input on
 *    the same stream.
 *  - `ws` is the caller's workspace of at least moe_workspace_size() bytes.
 *    Each compute call clears and then uses a device status word at its start;
 *    moe_get_device_status() reads it (bounds violations, device-side wait
 *    time-outs).  Kernels never trap or assert.
 *  - Two calls sharing one `ws` must not run concurrently.
 *  - Activation dtype (x, permuted rows, expert outputs) is cfg->act_dtype:
 *    MOE_F32 runs SIMT fp32 kernels; MOE_BF16 runs the tcgen05 tensor-core
 *    kernels with fp32 accumulation.  The SwiGLU hidden state is stored in
 *    act_dtype; expert outputs (y_perm, y_shared) are stored in fp32; the
 *    gate-weighted sum is formed in fp32 and stored as cfg->out_dtype (MOE_F32
 *    is the MoE listing's fp32 result of multiplying by the fp32 gates).
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,     /* null / misaligned pointer, bad size or enum   */
  MOE_ERR_UNSUPPORTED = 2,     /* valid layer the kernels do not handle          */
  MOE_ERR_WORKSPACE = 3,       /* ws or packed buffer smaller than required      */
  MOE_ERR_CUDA = 4,            /* a CUDA runtime call or kernel launch failed    */
  MOE_ERR_DEVICE_TIMEOUT = 5,  /* a device-side wait gave up (status word)       */
  MOE_ERR_DEVICE_BOUNDS = 6,   /* a device-side index was out of range           */
  MOE_ERR_DEVICE_RANGE = 7     /* FP8 layer: an activation beyond f16 range      */
} moe_status;

typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1, MOE_FP8_E4M3 = 2 } moe_dtype;
typedef enum moe_score_fn { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_fn;
typedef enum moe_topk_method { MOE_TOPK_GREEDY = 0, MOE_TOPK_GROUP_LIMITED = 1 } moe_topk_method;
typedef enum moe_group_score { MOE_GROUP_MAX = 0, MOE_GROUP_SUM_TOP = 1 } moe_group_score;

/* Layer hyper-parameters (names of the MoEGate / MoE listings).
 *   T tokens, d model dim, E routed experts (n_routed_experts), I routed
 *   expert hidden size, k = num_experts_per_tok, n_shared shared experts fused
 *   as one SwiGLU of hidden I_s = n_shared * I.
 *   Group-limited routing: E/n_group contiguous experts per group; the group
 *   score is the max selection score (MOE_GROUP_MAX, DeepSeek-V2) or the sum of
 *   the group_top largest ones (MOE_GROUP_SUM_TOP, the V3 node-limited rule);
 *   the topk_group best groups stay eligible.  norm_topk = 1 divides the k
 *   gates by their sum; routed_scaling_factor multiplies them. */
typedef struct moe_config {
  int32_t T, d, E, I, k, n_shared;
  int32_t score_fn;        /* moe_score_fn    */
  int32_t topk_method;     /* moe_topk_method */
  int32_t n_group, topk_group;
  int32_t group_score;     /* moe_group_score */
  int32_t group_top;
  int32_t norm_topk;
  float routed_scaling_factor;
  int32_t act_dtype;       /* moe_dtype of x, expert weights and rows */
  int32_t gate_w_dtype;    /* moe_dtype of W_g                        */
  int32_t out_dtype;       /* moe_dtype of the layer output h'        */
  int32_t expert_w_dtype;  /* storage of the packed expert weights: act_dtype, or
                              MOE_FP8_E4M3 (with MOE_BF16 activations): FP8
                              e4m3 values with one power-of-two scale per 64
                              consecutive weights of a row (intelliparadigm.com
                              page section 4, block quantisation; d and I
                              multiples of 128).  The GEMMs dequantize on the
                              fly and multiply on the f16 tensor cores, as the
                              page's fp8 matmul does: each weight enters as
                              e4m3 x 2^(e - e_ref), exact in f16 whenever its
                              block's exponent e is within 15 of the largest
                              one of its matrix (e_ref), and the product is
                              scaled by 2^e_ref in fp32.  Token rows and the
                              SwiGLU hidden rows enter as f16 (the bf16 x is
                              exact in f16 between 2^-14 and 65504; smaller
                              values round to multiples of 2^-24, larger ones
                              set MOE_ERR_DEVICE_RANGE); the shared expert's
                              first GEMM reads x as bf16 and dequantizes its
                              weights to bf16 (exact).  Batches of at most 64
                              tokens run as a GEMV with warp-level MMAs
                              instead: e4m3 -> f16 weights times f16 token
                              values (the shared expert's too), exact
                              products summed in fp32 per 64-weight block,
                              then 2^e per block. */
} moe_config;

/* Bytes of workspace every compute call needs for `cfg`. */
MOE_API moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Bytes of the packed expert blob moe_prepack_experts() writes for `cfg`. */
MOE_API moe_status moe_packed_size(const moe_config* cfg, size_t* bytes);

/* Re-lays the expert weights for the grouped GEMMs (MoE listing: E routed
 * SwiGLU experts + one shared SwiGLU of hidden I_s).
 *   W1, W3 [E,I,d], W2 [E,d,I]; Ws1, Ws3 [I_s,d], Ws2 [d,I_s]; act_dtype.
 *   `packed` (>= moe_packed_size bytes) receives W1/W3 rows interleaved in
 *   blocks of 16 so that one GEMM tile holds matching gate and up rows, and
 *   W2 / Ws2.  bf16: every matrix (per expert, and the shared one) is stored as
 *   stage blocks, one per tile of 128 rows and stage of 128 columns, in
 *   row-tile-major then stage order: each 32 KB block holds the two 64-column
 *   halves of the stage one after the other, each 128 rows x 64 bf16 row-major,
 *   zero past the matrix's rows or columns (so the expert kernel streams each
 *   stage as one contiguous read).  fp32: row-major.
 *   With expert_w_dtype = MOE_FP8_E4M3 every matrix is quantised
 *   block by block on the way and stored as the expert GEMM's shared-memory
 *   images: per tile of 128 rows (same row order), cols/128 stage blocks of
 *   17408 bytes, each the tile's 128 x 128 e4m3 values (row r at byte r*128,
 *   its 16-byte chunk c at chunk position c ^ (r % 8)) followed by their
 *   int32 scale exponents [2][128] (64-value block h of row r at [h][r]; the
 *   block's scale is 2^e); a zero tile follows each matrix's last row.  After
 *   the four matrices, int32 e_ref [E+1][3]: for each expert (the shared one
 *   last) the exponent its W1's, W3's and W2's largest |w| gets by the block
 *   rule (the largest exponent among the matrix's nonzero blocks; 0 for a
 *   zero matrix).  FP8 needs d and I
 *   multiples of 128.
 *   Inputs may be freed once the stream reaches this call. */
MOE_API moe_status moe_prepack_experts(const moe_config* cfg, const void* W1, const void* W3, const void* W2,
                               const void* Ws1, const void* Ws3, const void* Ws2,
                               void* packed, size_t packed_bytes, void* stream);

/* Router (MoEGate.forward; V3 page section 1.2 for the sigmoid score and the
 * selection-only bias).
 *   x [T,d] act_dtype, Wg [E,d] gate_w_dtype, bias [E] fp32 or NULL.
 *   idx [T,k] int32 out: chosen experts ordered by selection score desc, ties
 *   to the lower index; w [T,k] fp32 out: gate values.  Logits are fp32-exact:
 *   bf16 x times a bf16 (or 3-way bf16-split fp32) W_g on the tensor cores
 *   with fp32 accumulation, or SIMT fp32. */
MOE_API moe_status moe_gate_topk(const moe_config* cfg, const void* x, const void* Wg, const float* bias,
                         int32_t* idx, float* w, void* ws, size_t ws_bytes, void* stream);

/* Dispatch (MoE listing: repeat each token k times, group rows by expert).
 *   idx [T,k] in.  counts [E] out; offsets [E+1] out (exclusive prefix sum);
 *   row2tok [T*k] out: token of each expert-contiguous row; tok2row [T,k] out:
 *   row of each (token, slot); x_perm [T*k,d] act_dtype out: gathered rows.
 *   Rows of one expert are in increasing token order (deterministic).
 *   idx entries outside [0,E) are skipped and flagged in the status word. */
MOE_API moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* idx, int32_t* counts,
                       int32_t* offsets, int32_t* row2tok, int32_t* tok2row, void* x_perm,
                       void* ws, size_t ws_bytes, void* stream);

/* Experts (intelliparadigm.com page section 3.3.1 SwiGLU; MoE listing).
 *   x_perm [T*k,d] rows grouped by expert per `offsets` [E+1] (device);
 *   x [T,d] for the shared expert; packed = moe_prepack_experts output.
 *   y_perm [T*k,d] fp32 out: FFN_e of each row; y_shared [T,d] fp32 out:
 *   FFN_shared(x).
 *   bf16: GEMM1 with the fused silu(W1 u)*(W3 u) epilogue (hidden rounded to
 *   bf16), then GEMM2; both on tcgen05 with fp32 accumulation in TMEM. */
MOE_API moe_status moe_grouped_swiglu(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                              const void* x, const void* packed, void* y_perm, void* y_shared,
                              void* ws, size_t ws_bytes, void* stream);

/* Combine (MoE listing: gate-weighted sum over the k slots plus the shared
 * expert; the dense einsum form of the intelliparadigm.com page 3.3.3).
 *   y_perm [T*k,d], y_shared [T,d] fp32 (moe_grouped_swiglu's outputs).
 *   out[t] = sum_j w[t,j] * y_perm[tok2row[t,j]] + y_shared[t], accumulated in
 *   fp32 in slot order j = 0..k-1 (deterministic), stored as out_dtype. */
MOE_API moe_status moe_combine(const moe_config* cfg, const void* y_perm, const void* y_shared,
                       const int32_t* tok2row, const float* w, void* out,
                       void* ws, size_t ws_bytes, void* stream);

/* The whole layer: gate_topk -> permute -> grouped_swiglu -> combine, on one
 * stream with no host synchronisation.  idx_out [T,k], w_out [T,k] and
 * counts_out [E] are optional copies of the routing (NULL to skip). */
MOE_API moe_status moe_forward(const moe_config* cfg, const void* x, const void* Wg, const float* bias,
                       const void* packed, void* out, int32_t* idx_out, float* w_out,
                       int32_t* counts_out, void* ws, size_t ws_bytes, void* stream);

/* Dispatch without any device allocation (the pages have no counterpart: it
 * exists for callers, not for the method).  Same inputs, outputs and results
 * as moe_permute, but the per-chunk scratch lives in a fixed array inside the
 * library's device image instead of a caller workspace.  Meant for callers
 * that cannot call cudaMalloc or hand out workspace: plug-ins whose device
 * memory belongs to a host framework's arena, processes held to a hard memory
 * budget, and latency-critical loops that must not risk cudaMalloc's
 * device-wide blocking or its failure under fragmentation.
 *   Limit: permute_chunks(T) * E <= 32768, with 128 tokens per chunk (e.g.
 *   T <= 16384 with E = 256); larger sizes return MOE_ERR_WORKSPACE without
 *   launching.  The array (~256 KB) is held on every device that loads the
 *   library until the process exits.
 *   device_status [1] int32 (device, nullable) receives this call's status
 *   word (as read by moe_get_device_status for the workspace calls).
 *   The first call on each device looks up the array's device address with
 *   cudaGetSymbolAddress; make that first call before any stream capture.
 *   The address is kept for the life of the process: after a context reset
 *   (cudaDeviceReset) do not call this entry point on that device again.
 *   With T = 0 it writes empty counts/offsets and a zero device_status.
 *   All calls share the one array, so calls whose kernels overlap on the GPU
 *   (other streams, other host threads) race: serialise them.  No cudaMalloc,
 *   cudaFree or allocating library routine is called. */
MOE_API moe_status moe_permute_noalloc(const moe_config* cfg, const void* x, const int32_t* idx,
                                       int32_t* counts, int32_t* offsets, int32_t* row2tok,
                                       int32_t* tok2row, void* x_perm, int32_t* device_status,
                                       void* stream);

/* Bytes of workspace moe_backward needs for `cfg` (the forward's workspace
 * plus the backward's buffers).  bf16 activations and bf16 expert weights,
 * d a multiple of 128 (MOE_ERR_UNSUPPORTED otherwise). */
MOE_API moe_status moe_backward_workspace_size(const moe_config* cfg, size_t* bytes);

/* Backward of the layer: the gradient of L = <dout, out> with respect to x,
 * W_g and every expert weight, by the chain rule through the gate-weighted sum
 * and the shared expert (MoE listing), the SwiGLU experts (intelliparadigm.com
 * page section 3.3.1), the gate values (renormalised and scaled, V3 page
 * section 1.2) and the affinities (softmax over all experts or sigmoid), with
 * the expert choice of the forward held fixed (the selection bias carries no
 * gradient).
 *   x [T,d] bf16, Wg [E,d] gate_w_dtype, bias [E] fp32 or NULL (as for
 *   moe_gate_topk: the routing is recomputed with the forward's kernels).
 *   W1, W3 [E,I,d], W2 [E,d,I], Ws1, Ws3 [I_s,d], Ws2 [d,I_s]: the unpacked
 *   bf16 weights (as given to moe_prepack_experts; Ws* unused when
 *   n_shared = 0).  dout [T,d] out_dtype: the upstream gradient.
 *   Outputs (device, fp32, written, not accumulated): dx [T,d], dWg [E,d],
 *   dW1, dW3 [E,I,d], dW2 [E,d,I], dWs1, dWs3 [I_s,d], dWs2 [d,I_s].
 *   ws: >= moe_backward_workspace_size bytes, 16-byte aligned.
 * Every matrix product runs on the library's CTA-pair tensor-core kernel
 * (bf16 operands, fp32 accumulation and outputs): the expert weights are read
 * in place through transposed views where a product needs W^T, and the
 * routed rows use a padded per-expert layout so each weight gradient reduces
 * over its own rows.  The routed rows' intermediate gradients are rounded to
 * bf16 before their products, as the forward rounds H; the router's d logits
 * are rounded to bf16 for dW_g and for their part of dx.  Group sizes stay on
 * the device: the call neither synchronises `stream` nor allocates.
 * d must be a multiple of 128 (MOE_ERR_UNSUPPORTED otherwise).
 * All pointers 16-byte aligned. */
MOE_API moe_status moe_backward(const moe_config* cfg, const void* x, const void* Wg, const float* bias,
                                const void* W1, const void* W3, const void* W2, const void* Ws1,
                                const void* Ws3, const void* Ws2, const void* dout, float* dx, float* dWg,
                                float* dW1, float* dW3, float* dW2, float* dWs1, float* dWs3, float* dWs2,
                                void* ws, size_t ws_bytes, void* stream);

/* Auxiliary-loss-free load balancing after a layer step (V3 architecture
 * page, section 1.2), with the load statistics of the balance-loss listing
 * (Tencent Cloud DeepSeek page).
 *   counts [E] int32 (device): assignments per expert of the step, e.g.
 *   moe_forward's counts_out.  bias [E] fp32 (device), updated in place with
 *   one fp32 addition: b_e - gamma when counts_e * E > sum(counts) (the expert
 *   took more than the mean), b_e + gamma when it took fewer, unchanged at the
 *   mean.  stats [3] fp32 (device, nullable): the unbiased standard deviation
 *   of the load fractions counts / sum(counts), and the largest and smallest
 *   count divided by the mean count.  device_status [1] int32 (device,
 *   nullable): set to a non-zero DEV bit if a count is negative (treated as
 *   zero).  One single-block kernel; no workspace; gamma must be finite. */
MOE_API moe_status moe_balance_update(const moe_config* cfg, const int32_t* counts, float* bias, float gamma,
                                      float* stats, int32_t* device_status, void* stream);

/* Synchronises `stream`, reads the device status word of `ws` and returns
 * MOE_OK, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_DEVICE_BOUNDS or
 * MOE_ERR_DEVICE_RANGE (in that order of precedence).  `detail` (nullable)
 * receives the raw word. */
MOE_API moe_status moe_get_device_status(const void* ws, void* stream, int32_t* detail);

/* Human-readable name of a status code (static storage). */
MOE_API const char* moe_status_string(moe_status s);

/* Fault injection for tests of the device-side time-out path (the pages have
 * no counterpart: it exists to show that a stalled pipeline reports an error
 * instead of hanging, and that the next call runs normally).
 *   what = MOE_DEBUG_WAIT_LIMIT_NS: the limit of every bounded wait in the
 *     expert GEMM kernel for later calls, in ns (0 restores the default of
 *     2 s; otherwise 1e5 .. 1e10).
 *   what = MOE_DEBUG_STALL_GEMM2 (value 0 or 1): when 1, every GEMM2 tile of
 *     a one-launch expert GEMM (T*k <= 8192) waits for one more GEMM1
 *     completion than its group produces, so that wait runs out: the call
 *     sets DEV_TIMEOUT in its status word (moe_get_device_status returns
 *     MOE_ERR_DEVICE_TIMEOUT), its kernels end, and its outputs are undefined.
 * Process-wide settings read when a call launches its kernels; not
 * thread-safe.  Returns MOE_ERR_INVALID_ARG for an unknown knob or value. */
typedef enum moe_debug_knob { MOE_DEBUG_WAIT_LIMIT_NS = 0, MOE_DEBUG_STALL_GEMM2 = 1 } moe_debug_knob;
MOE_API moe_status moe_debug_inject(int32_t what, int64_t value);

/* Number of kernels this library has launched in the process so far. */
MOE_API uint64_t moe_launch_count(void);

/* Stage timing for benchmarks.  While armed, every moe_forward records the
 * caller's CUDA events (cudaEvent_t, created by the caller) on its stream at
 * the boundaries of its MOE_FORWARD_STAGES stages and once at the end, i.e.
 * MOE_FORWARD_STAGES + 1 events per call, taken from `events` in order until
 * `n_events` are used.  Stages: 0 router (gate GEMM + top-k), 1 permutation,
 * 2 experts (GEMM1 with the SwiGLU epilogue and GEMM2, one launch on the
 * tensor-core path), 3 combine.  NULL disarms.  The events split the
 * kernels' launch overlap, so armed calls run slightly slower.
 * Not thread-safe; arm, run, disarm from one host thread. */
#define MOE_FORWARD_STAGES 4
MOE_API moe_status moe_profile_arm(void* const* events, int32_t n_events);

/* Name of stage i of moe_forward ("router", "permute", ...), or NULL. */
MOE_API const char* moe_forward_stage_name(int32_t i);

/* Number of kernels one moe_forward launches for `cfg` (host-side plan). */
MOE_API int32_t moe_forward_kernel_count(const moe_config* cfg);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
