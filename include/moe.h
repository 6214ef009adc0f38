/*
 * moe.h -- C ABI of libmoe.so, the fused mixture-of-experts expert layer for one
 * NVIDIA GB300 (sm_103a).
 *
 * The layer (sources are named by page title and section):
 *   out[t] = sum_{j<k} w[t,j] * FFN_{idx[t,j]}(x[t]) + FFN_shared(x[t])
 * with
 *   - fp32 router logits and softmax top-k with renormalised weights
 *     ("Optimising Ling-2.6-1T on TPU with SGLang-JAX", s.1: 256 routed experts,
 *     top-8 plus one shared expert; "Kimi K3 ... feasibility analysis", s.2.4:
 *     moe_renormalize, routed_scaling_factor 1.0);
 *   - dynamic per-token fp8 e4m3 activation quantisation before the scatter
 *     (Ling write-up, s.5 "activation quantisation");
 *   - scatter of token rows into expert-contiguous order, which on one GPU is a
 *     local permutation (Ling write-up, s.1: scatter -> local expert FFN -> gather);
 *   - SwiGLU experts h = silu(W1 x) * (W3 x), y = W2 h on fp8 per-output-channel
 *     weights with the scale applied after the full-K sum (Ling write-up, s.5
 *     "per-channel direct_scaled_dot": out[m,n] = (sum_k A W) * scale[n]);
 *     MXFP4 (e2m1 + e8m0 per 32) for the LatentMoE case (Kimi K3 report, s.2.5);
 *   - weighted top-k gather back to token order plus the shared expert (Ling
 *     write-up, s.5 "in-kernel shared expert").
 *
 * Conventions for every entry point
 *   - Pointers named *_host are host pointers; every other tensor pointer is a
 *     DEVICE pointer owned by the caller, C-contiguous (row-major), on the
 *     current CUDA device.  bf16 tensors are passed as void* (IEEE bfloat16
 *     bits), fp8 tensors as void* (OCP E4M3FN bytes).
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *     stream.  Every call is asynchronous on `stream` and returns once its
 *     kernels are queued; no call synchronises except moe_get_last_error and
 *     moe_profile_read.
 *   - The library allocates no device memory on the call path: scratch comes
 *     from the caller's workspace `ws` of `ws_bytes` bytes (moe_workspace_bytes),
 *     256-byte aligned.  Outputs must not alias inputs.
 *   - Return value: a moe_status.  Argument checks happen on the host before any
 *     launch and return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *     MOE_ERR_WORKSPACE with nothing queued; a failed launch returns
 *     MOE_ERR_CUDA.  Faults detected on the device (a pipeline wait that ran out
 *     of time) set a per-device error word that moe_get_last_error returns.
 *     Nothing aborts, throws or falls back to another implementation.
 *   - Shapes: H, I, I_shared (and latent) must be multiples of 128; T >= 0
 *     (T = 0 is a no-op); 1 <= top_k <= min(E, 32); E <= 1024.
 *   - Per-device state: the library looks up, once per device and then keeps,
 *     the device addresses of its own global variables (the error word, the
 *     scratch array of moe_permute_static) and raises kernel attributes.  All
 *     of it belongs to the device's primary context, which cudaDeviceReset
 *     destroys: do not reset a device that this library has run on while the
 *     process goes on calling the library.
 */
#ifndef MOE_GB300_MOE_H_
#define MOE_GB300_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, bad size, top_k > E, misaligned pointer */
  MOE_ERR_UNSUPPORTED = 2, /* valid problem this library does not implement      */
  MOE_ERR_WORKSPACE = 3,   /* ws NULL or ws_bytes < moe_workspace_bytes           */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed         */
  MOE_ERR_TIMEOUT = 5      /* a device-side pipeline wait exceeded its limit      */
} moe_status;

typedef enum {
  MOE_W_FP8_E4M3_PER_CHANNEL = 0, /* e4m3 bytes + fp32 scale per output channel   */
  MOE_W_MXFP4_E2M1_E8M0_B32 = 1,  /* packed e2m1 (low nibble = even k) + e8m0/32  */
  MOE_W_FP8_E4M3_BLOCK128 = 2     /* e4m3 bytes + fp32 scale per 128 x 128 block  */
} moe_wfmt;

#define MOE_F_ROUTER_BIAS 0x1u /* add router_bias[e] to every logit before top-k    */
#define MOE_F_SHARED_BF16 0x2u /* shared expert weights are bf16 (no quantisation)   */
#define MOE_F_PACKED_WEIGHTS 0x4u /* routed (and fp8 shared) expert weights are in
                                     moe_pack_weights' tile order                  */
#define MOE_F_SIGMOID_ROUTING 0x8u /* noaux_tc routing: scores sigmoid(logit), the
                                      router bias steers selection only, weights =
                                      chosen scores renormalised (K3 report s.2.4) */
#define MOE_F_SITU 0x10u /* SiTU experts: h = 4 tanh(g/4) sigmoid(g) u instead of
                            SwiGLU's silu(g) u (K3 report s.2.6)                 */
#define MOE_F_FUSED_COMBINE 0x20u /* S7 in the FFN2 epilogue: see moe_forward     */

typedef struct {
  int32_t T;        /* tokens                                                      */
  int32_t H;        /* hidden width                                                */
  int32_t I;        /* routed expert intermediate width                            */
  int32_t E;        /* routed experts                                              */
  int32_t top_k;    /* experts per token                                           */
  int32_t I_shared; /* shared expert intermediate width; 0 = no shared expert      */
  int32_t latent;   /* LatentMoE width L (experts run on L instead of H); 0 = none */
  int32_t wfmt;     /* moe_wfmt of the routed expert weights                       */
  uint32_t flags;   /* MOE_F_*                                                     */
} moe_problem;

/* Stage indices for the profiling counters. */
enum {
  MOE_STAGE_ROUTER = 0,  /* S1 router logits                     */
  MOE_STAGE_TOPK = 1,    /* S2 top-k + renormalise               */
  MOE_STAGE_INDEX = 2,   /* S3 histogram, scan, ranks, tile list */
  MOE_STAGE_SCATTER = 3, /* S4 per-token fp8 quant + row scatter */
  MOE_STAGE_FFN1 = 4,    /* S5 grouped W1|W3 GEMM + SiLU*gate    */
  MOE_STAGE_REQUANT = 5, /* S6a per-row fp8 requant of h         */
  MOE_STAGE_FFN2 = 6,    /* S6 grouped W2 GEMM + routing weight  */
  MOE_STAGE_COMBINE = 7, /* S7/S8 weighted gather + shared add   */
                         /*   (LatentMoE: gather + RMSNorm)     */
  MOE_STAGE_LATENT_DOWN = 8, /* S9 z = x Wd^T                   */
  MOE_STAGE_SHARED = 9,      /* S8 bf16 shared expert gate/up   */
  MOE_STAGE_LATENT_UP = 10,  /* S9 yn Wu^T + shared down        */
  MOE_STAGE_COUNT = 11
};

/* Human-readable name of a moe_status (static storage). */
const char* moe_status_string(int status);

/* Host-only: a one-line description of how moe_forward runs problem `p` (the
 * grouped-GEMM kernels, token-tile rows, weight format, router, workspace
 * bytes),
 * written NUL-terminated into buf[len].  MOE_ERR_INVALID_ARG if `p` is invalid
 * or buf too short, MOE_ERR_UNSUPPORTED for a combination this library does not
 * run.  For logs and benchmarks; the text format may change. */
int moe_describe(const moe_problem* p, char* buf, size_t len);

/* Bytes of device workspace that moe_forward, moe_permute, moe_expert_ffn,
 * moe_router_topk and moe_latent_down need for problem `p` (0 if `p` is
 * invalid).  Host computation; it reads the current device's SM count (small
 * batches split the router GEMM into more K ranges on more SMs), so size the
 * workspace on the device that will run the calls. */
size_t moe_workspace_bytes(const moe_problem* p);

/* S1 -- router logits.  logits[t,e] = sum_h float(x[t,h]) * router_w[e,h]
 * (+ bias[e] when MOE_F_ROUTER_BIAS without MOE_F_SIGMOID_ROUTING; with sigmoid
 * routing the bias belongs to moe_route), fp32, summed in one fixed order: 32
 * partial sums (partial l takes h = l, l+32, ... ascending, fused multiply-add
 * from +0), then p_l += p_{l+o} for o = 16, 8, 4, 2, 1, bias added last.  The
 * order is fixed so that routing is reproducible bit for bit.
 * (Ling write-up, s.6: routing metadata.)
 *   x        [T, H] bf16           router_w [E, H] fp32
 *   bias     [E] fp32, required iff MOE_F_ROUTER_BIAS, else ignored
 *   logits   [T, E] fp32 (output) */
int moe_router_logits(const moe_problem* p, const void* x, const float* router_w,
                      const float* bias, float* logits, void* stream);

/* S2 -- top-k.  For each token the top_k largest logits in descending order,
 * equal logits ordered by lower expert index; weights are the softmax over the
 * chosen logits, w_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0), fp32.
 * (Ling write-up, s.1 top-8 routing; Kimi K3 report, s.2.4 moe_renormalize.)
 * With MOE_F_SIGMOID_ROUTING (K3 report s.2.4, noaux_tc + sigmoid, ungrouped,
 * scaling factor 1): scores s_e = sigmoid(l_e), the top_k largest keys s_e +
 * bias[e] are chosen (ties to the lower index; bias only with
 * MOE_F_ROUTER_BIAS), and w_j = s_j / sum_j' s_j'.  For the selection sigmoid
 * is one fixed fp32 sequence (Cody-Waite reduction, Taylor series to degree 7
 * through fma, IEEE add and divide) so that it is reproducible bit for bit.
 *   logits [T, E] fp32; bias [E] fp32 (sigmoid routing with MOE_F_ROUTER_BIAS,
 *   else ignored) -> topk_idx [T, top_k] int32, topk_w [T, top_k] fp32 */
int moe_route(const moe_problem* p, const float* logits, const float* bias, int32_t* topk_idx,
              float* topk_w, void* stream);

/* S1 + S2 in one call, as moe_forward runs them: the routing that
 * moe_router_logits followed by moe_route gives (Ling write-up, s.1 top-8
 * routing; "Kimi K3 ... feasibility analysis", s.2.4), bit for bit in
 * topk_idx wherever the margins below hold.  The logits are computed on the
 * tensor cores: every fp32 router weight is split exactly into three bf16
 * pieces and x . w is a tensor-core accumulation of exact products (for
 * small batches over several K ranges whose sums are added), taken to lie
 * within m = 8 2^-23 |x_t| |w_e| (plus the additions' rounding) of the
 * canonical logit.  A token's order is kept wherever those margins separate
 * the keys (every lower bound up to a position above every upper bound after
 * it); the experts between undecided positions get their canonical logits,
 * computed in moe_router_logits' order, and are ordered by them.  The margin
 * is a calibrated bound (measured errors ~40 times smaller on normally
 * distributed inputs), not a worst-case one: inputs built so that large
 * partial sums cancel could exceed it.  moe_router_logits + moe_route, or
 * moe_tuning's router_tile 1..4, give the canonical routing for any input.
 * topk_w is the softmax (or sigmoid share) of the logits the selection used,
 * within 2 (m_i + max_j m_j) relative of moe_route's.
 *   x [T, H] bf16, router_w [E, H] fp32, bias as for moe_router_logits (softmax
 *   routing) or moe_route (MOE_F_SIGMOID_ROUTING)
 *   topk_idx [T, top_k] int32, topk_w [T, top_k] fp32 (outputs)
 *   ws / ws_bytes: workspace of at least moe_workspace_bytes(p) */
int moe_router_topk(const moe_problem* p, const void* x, const float* router_w,
                    const float* bias, int32_t* topk_idx, float* topk_w, void* ws,
                    size_t ws_bytes, void* stream);

/* S9 (LatentMoE) -- down projection onto the latent on which the routed experts
 * run ("Kimi K3 ... feasibility analysis", s.2.4 routed_expert_down_proj):
 * z[t,l] = bf16(sum_h x[t,h] * latent_down[l,h]), rounded to nearest-even from
 * the exact dot product, so that the per-token fp8 quantisation of z that
 * follows is reproducible bit for bit.  A tensor-core GEMM with short fp32
 * accumulations computes every element; the elements lying so near a bf16
 * rounding boundary that its remaining error could matter are recomputed
 * exactly (two-fp32 sums of the exact bf16 products).  moe_forward runs this
 * as its first latent step.
 *   x [T, H] bf16, latent_down [latent, H] bf16 -> z [T, latent] bf16 (output)
 *   ws / ws_bytes: workspace of at least moe_workspace_bytes(p) (per-element
 *   recompute flags live there)
 * Needs latent > 0; H and latent multiples of 256 and 2 H + 2 latent <=
 * 163840 (else MOE_ERR_UNSUPPORTED); pointers 16-byte aligned. */
int moe_latent_down(const moe_problem* p, const void* x, const void* latent_down, void* z,
                    void* ws, size_t ws_bytes, void* stream);

/* S3 + S4 -- expert-contiguous permutation and per-token fp8 quantisation.
 * counts[e] = #{(t,j): idx[t,j] = e}; offsets[e] = sum_{e'<e} counts[e'],
 * offsets[E] = T*top_k; the row of (t,j) is offsets[e] + #{t' < t : e in
 * idx[t']} (stable in token order), perm[t,j] = that row, src_row[row] = t.
 * Each token is quantised once, s[t] = max_h |x[t,h]| / 448 in fp32 (1 if the
 * row is all zero), q = e4m3(x / s) rounded to nearest even and saturated to
 * +-448, and copied to each of its rows: xq_perm[row] = q[t], xscale_perm[row]
 * = s[t].  (Ling write-up, s.5 activation quantisation before the scatter;
 * s.6 per-expert offsets and scatter indices.)  With a latent problem, x is
 * the latent input [T, latent].
 *   topk_idx [T, top_k] int32 in [0, E)   x [T, H] bf16
 *   counts [E], offsets [E+1], perm [T, top_k], src_row [T*top_k] int32 (out)
 *   xq_perm [T*top_k, H] e4m3 (out), xscale_perm [T*top_k] fp32 (out)
 *   ws / ws_bytes: workspace, at least moe_workspace_bytes(p)
 * Indices outside [0, E) are reported as MOE_ERR_INVALID_ARG by
 * moe_get_last_error and their rows are left unwritten. */
int moe_permute(const moe_problem* p, const int32_t* topk_idx, const void* x, int32_t* counts,
                int32_t* offsets, int32_t* perm, int32_t* src_row, void* xq_perm,
                float* xscale_perm, void* ws, size_t ws_bytes, void* stream);

/* moe_permute without a workspace.  The pages have no counterpart for this
 * entry point: it exists for callers that cannot allocate device memory --
 * hosts that plan every byte up front and hand a plugin only its input and
 * output buffers, or latency-critical loops where cudaMalloc is not allowed
 * because it may synchronise the device.  Same arguments, results and errors
 * as moe_permute minus `ws`/`ws_bytes`: its scratch (two int32 tables of
 * E * ceil(T/32) entries) lives in a fixed 4 MiB array inside libmoe.so
 * (2^19 entries per table), which every GPU that loads the library holds
 * until the process exits.  Problems with E * ceil(T/32) > 2^19 return
 * MOE_ERR_WORKSPACE.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  Nothing is allocated: no cudaMalloc,
 * cudaFree or allocating library routine.  All calls on a device share the
 * array and it keeps the last call's contents; every entry a call reads is
 * written earlier in the same call, but calls whose kernels overlap on the
 * GPU (other streams or threads) race on it and must be serialised.  The
 * cached address does not survive a cudaDeviceReset of the device (see
 * "Per-device state" above). */
int moe_permute_static(const moe_problem* p, const int32_t* topk_idx, const void* x,
                       int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* src_row,
                       void* xq_perm, float* xscale_perm, void* stream);

/* One-time weight preparation (the "process weights after loading" step of a
 * serving stack, Kimi K3 report s.12.2): copies routed expert weights (and
 * MXFP4 scales) into the order the grouped GEMMs stream them.  Bytes are only
 * permuted.  Pass the results with MOE_F_PACKED_WEIGHTS.
 *   fp8: tile-major [E][rows/128][K/128][128 rows][128 bytes], so every 128 x
 *     128 tile a stage reads is one contiguous 16 KB block instead of 128
 *     strided rows; per-channel scales are unchanged (scale arguments unused).
 *     An fp8 shared expert is packed by calling this with E = 1 and I =
 *     I_shared on its two matrices.
 *   MXFP4 (K = H or latent a multiple of 256): a stage reads two 128-row
 *     blocks, W1 and W3 block p (rows p*128 and I + p*128) of w13, or W2 blocks
 *     2p and 2p+1 of w2.  Weights become [E][P][K/128][2][128 rows][64 bytes]
 *     and scales [E][P][K/128][4][2][8][4] 32-bit words, word (j, b, i, c)
 *     holding the four e8m0 bytes of k-stage kb of row 32c + 8j + i of block
 *     b (the tensor-memory image of the block-scaled MMAs, lane 8j + i,
 *     column c): one 256-row copy and one 1 KB copy per stage.
 *   w13 [E, 2I, K] / w2 [E, K, I]: fp8 bytes, or MXFP4 bytes of two e2m1 each
 *     ([E, 2I, K/2] / [E, K, I/2]), 16-byte aligned (K = H, or latent)
 *   w13_scale [E, 2I, K/32], w2_scale [E, K, I/32] e8m0 and their packed
 *     outputs of the same sizes: MXFP4 only (16-byte aligned), else ignored
 *   outputs: device buffers of the same sizes, not aliasing the inputs
 * Asynchronous on `stream`; MOE_ERR_INVALID_ARG for bad shapes or pointers. */
int moe_pack_weights(const moe_problem* p, const void* w13, const void* w2, const void* w13_scale,
                     const void* w2_scale, void* w13_packed, void* w2_packed,
                     void* w13_scale_packed, void* w2_scale_packed, void* stream);

/* S5 + S6 -- grouped SwiGLU experts over expert-contiguous rows.  For rows r
 * in [offsets[e], offsets[e+1]):
 *   g[n] = (sum_k xq[r,k] W1_e[n,k]) * xscale[r] * s13_e[n]      (W1 = rows 0..I-1)
 *   u[n] = (sum_k xq[r,k] W3_e[n,k]) * xscale[r] * s13_e[I+n]    (W3 = rows I..2I-1)
 *   h[n] = bf16(silu(g[n]) * u[n]);  s_h = max_n |h[n]| / 448;  hq = e4m3(h / s_h)
 *   y[r,m] = bf16(row_w[r] * (sum_n hq[n] W2_e[m,n]) * s_h * s2_e[m])
 * (Ling write-up, s.5 per-channel direct_scaled_dot; FFN1/FFN2 of s.1.)
 *   offsets   [E+1] int32 (device), offsets[E] = R rows
 *   xq_perm   [R, K] e4m3, xscale_perm [R] fp32, row_w [R] fp32 or NULL (= 1)
 *   fp8:   w13 [E, 2I, K] e4m3, w13_scale [E, 2I] fp32,
 *          w2  [E, K, I] e4m3,  w2_scale  [E, K] fp32
 *   MXFP4 (Kimi K3 report, s.2.5): w13 [E, 2I, K/2] and w2 [E, K, I/2] bytes
 *          holding two e2m1 values each (low nibble = even k), w13_scale
 *          [E, 2I, K/32] and w2_scale [E, K, I/32] e8m0 bytes (one per 32
 *          consecutive k, 4-byte aligned); the block scale multiplies inside the
 *          K-sum, so the per-channel factors s13/s2 above are 1; K must be a
 *          multiple of 256.
 *   block-wise fp8 (K3 report s.3.7, weight_block_size [128, 128]): w13, w2 as
 *          fp8, w13_scale [E, 2I/128, K/128] and w2_scale [E, K/128, I/128]
 *          fp32, one per 128 x 128 weight block; the block scale multiplies
 *          each 128-wide slice of the K-sum (g = xs * sum_kb s13[n/128, kb] *
 *          sum_{k in kb} xq W1, likewise u and y), so s13/s2 above become these
 *          block scales; K, I <= 16384.  An fp8 shared expert uses the same
 *          format ([2*I_shared/128, H/128] and [H/128, I_shared/128] scales).
 *   y         [R, K] bf16 (out); K = H (or latent)
 * R is read from p as T*top_k. */
int moe_expert_ffn(const moe_problem* p, const int32_t* offsets, const void* xq_perm,
                   const float* xscale_perm, const float* row_w, const void* w13,
                   const void* w13_scale, const void* w2, const void* w2_scale, void* y,
                   void* ws, size_t ws_bytes, void* stream);

/* S7 (+ S8 add) -- weighted gather back to token order.
 *   out[t,:] = bf16( sum_{j ascending} float(y_rows[perm[t,j],:]) + float(shared[t,:]) )
 * in fp32.  The routing weight is already folded into y_rows (moe_expert_ffn).
 * (Ling write-up, s.1 gather results; s.5 shared expert on every token.)
 *   y_rows [T*top_k, H] bf16, perm [T, top_k] int32,
 *   shared [T, H] bf16 or NULL, out [T, H] bf16 (out) */
int moe_unpermute(const moe_problem* p, const void* y_rows, const int32_t* perm,
                  const void* shared, void* out, void* stream);

/* The whole layer, S1..S8, queued on `stream` with no host round trip.
 * S1 + S2 run as moe_router_topk does (tensor-core logits, selection made
 * exact against the canonical order within its calibrated margins; the
 * CUDA-core router when moe_tuning's router_tile picks one of its tiles).
 *   x [T, H] bf16; router_w [E, H] fp32; router_bias [E] fp32 (MOE_F_ROUTER_BIAS:
 *   added to the logits, or with MOE_F_SIGMOID_ROUTING to the scores for
 *   selection only); MOE_F_SITU switches every expert (routed and shared) to
 *   SiTU
 *   routed experts: see moe_expert_ffn (K = H, or latent for a LatentMoE problem)
 *   shared expert (I_shared > 0): fp8 shared_w13 [2*I_shared, H] e4m3 +
 *     shared_w13_scale [2*I_shared] fp32, shared_w2 [H, I_shared] e4m3 +
 *     shared_w2_scale [H] fp32; with MOE_F_SHARED_BF16 the two weights are bf16
 *     and the scales are ignored.  The shared expert takes weight 1 and the
 *     same per-token fp8 activations as the routed experts.
 *   latent (L > 0): latent_down [L, H] bf16, latent_up [H, L] bf16,
 *     latent_gamma [L] bf16 (RMSNorm weight, eps 1e-6), Kimi K3 report s.2.4.
 *   out [T, H] bf16 (output); ws / ws_bytes as for moe_permute.
 * MOE_F_FUSED_COMBINE (the Ling write-up's gather of results done inside the
 * expert kernel, s.4; the SparseCore gather-reduce of the sglang-jax gap list,
 * s.8): the FFN2 epilogue adds each routed row, already scaled by its routing
 * weight, and each shared-expert row straight into an fp32 [T, H] sum in the
 * workspace (zeroed by S4) with fp32 reductions, and a last pass rounds that
 * sum to bf16 out.  No y rows are written or read back.  The order of the
 * top_k + 1 additions per element is not fixed, so two calls can differ in the
 * last bit of out; without the flag the gather combine sums in a fixed order
 * and repeats bit for bit.  The flag is a request: it is honoured for fp8
 * per-channel experts on the single-SM grouped GEMMs without latent (moe_describe
 * names the combine that runs) and ignored elsewhere.
 * Combinations this library runs (others return MOE_ERR_UNSUPPORTED): without
 * latent, an fp8 shared expert with I_shared = I or none; with latent, a bf16
 * shared expert or none and H, L multiples of 256; MXFP4 experts with K (H or
 * L) a multiple of 256 and no fp8 shared expert. */
int moe_forward(const moe_problem* p, const void* x, const float* router_w,
                const float* router_bias, const void* w13, const void* w13_scale,
                const void* w2, const void* w2_scale, const void* shared_w13,
                const void* shared_w13_scale, const void* shared_w2,
                const void* shared_w2_scale, const void* latent_down, const void* latent_up,
                const void* latent_gamma, void* out, void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream`, then returns and clears the current device's error
 * word (MOE_OK if no device-side fault was recorded; MOE_ERR_CUDA if the
 * synchronisation itself failed). */
int moe_get_last_error(void* stream);

/* Self-test of the device watchdog (no counterpart in the pages: it checks this
 * library's failure handling).  Launches one CTA shaped like the grouped GEMMs
 * (one warp holding 32 tensor-memory columns, four warps in pipeline waits)
 * whose mbarriers nothing arrives on.  Each wait gives up after the kernels'
 * wait limit (2 s), the first to expire records MOE_ERR_TIMEOUT in the error
 * word and raises the CTA's abort flag, the others stop on the flag, tensor
 * memory is freed and the kernel returns; the context stays usable.
 *   role_status [4] int32 device (out, nullable): 1 if warp w's wait completed,
 *     0 if it gave up (always 0 here)
 * Asynchronous on `stream`: read the result with moe_get_last_error, which then
 * returns MOE_ERR_TIMEOUT.  Returns MOE_OK, or MOE_ERR_CUDA if the launch
 * failed. */
int moe_watchdog_selftest(int32_t* role_status, void* stream);

/* Number of kernels this library has launched in this process (all devices).
 * Host-side counter, for accounting; never reset. */
int64_t moe_launch_count(void);

/* Launch choices that change no result, only which kernels run and how
 * (process-wide, every device).  At its first use the library reads them once
 * from the environment -- MOE_TILE_N=<rows>, MOE_GATHER=1, MOE_INDEX=3pass,
 * MOE_GEMM=1cta, MOE_PAIR_SMALL=0, MOE_MX=1cta,
 * MOE_ROUTER_TILE=8x8|8x16|8x16s4|12w8x16|tc, MOE_PDL=0 -- and moe_set_tuning
 * replaces them for every later call.  For benchmarks and tests; the defaults
 * are the measured best. */
typedef struct {
  int32_t tile_n;      /* 0 automatic; else token rows per grouped-GEMM tile where the
                          weight format has kernels for it (fp8 per-channel 32, 64,
                          128, 256; block-wise 32, 64; MXFP4 32, 64, 96), ignored
                          otherwise                                                  */
  int32_t ffn1_gather; /* 1: the single-SM fp8 per-channel FFN1 gathers its rows by
                          token and S4 writes one row per token                      */
  int32_t index_3pass; /* 1: count / scan / rank kernels even where one block would do */
  int32_t gemm_1cta;   /* 1: single-SM fp8 grouped GEMMs for 256-row tiles as well    */
  int32_t pair_small;  /* 1 (default): SM-pair items of <= 128 rows as M = 128 tiles  */
  int32_t mx_1cta;     /* 1: single-SM MXFP4 grouped GEMMs; 0 (default): SM pairs where
                          the weights are packed (moe_pack_weights) and the
                          128-row weight blocks pair up                              */
  int32_t router_tile; /* 0 (default) or 6: tensor-core logits with the selection
                          made exact (moe_router_topk); the CUDA-core router in
                          the canonical order: 1: 8 warps of 8 tokens x 8 experts,
                          2: 8 x 16, 3: 8 x 16 with four chunks a stage, 4: 12
                          warps of 8 x 16                                        */
  int32_t pdl;         /* 1 (default): programmatic dependent launch between kernels */
} moe_tuning;

/* Current launch choices.  MOE_ERR_INVALID_ARG if t is NULL. */
int moe_get_tuning(moe_tuning* t);

/* Replace the launch choices (host only; takes effect for calls made after it
 * returns).  MOE_ERR_INVALID_ARG, changing nothing, if t is NULL or a field is
 * out of range (tile_n not 0/32/64/96/128/256, flags not 0/1, router_tile
 * not 0..4 or 6). */
int moe_set_tuning(const moe_tuning* t);

/* Per-stage device timing.  mask selects the stages to time (bit s = stage
 * MOE_STAGE_s; -1 = all, 0 = off); each launch of a selected stage is
 * bracketed by CUDA events recorded on the launching stream.  moe_profile_read
 * waits for the recorded events, writes the summed milliseconds and launch
 * counts per stage (MOE_STAGE_*, arrays of MOE_STAGE_COUNT) and clears the
 * record.  Returns MOE_OK, or MOE_ERR_CUDA. */
int moe_profile_enable(int mask);
int moe_profile_read(double* stage_ms, int64_t* stage_launches);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_MOE_H_ */
