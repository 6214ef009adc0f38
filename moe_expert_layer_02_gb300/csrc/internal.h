// internal.h -- host-side launchers shared between the translation units of
// libmoe.so.  Not part of the public C ABI (include/moe.h).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <atomic>

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Tokens per warp chunk in the index kernels (one token per lane).
// Raise kernel K's dynamic shared-memory limit to `bytes`, once per device
// (the attribute belongs to the device's context; setting it on every launch
// costs host time and is not needed inside a stream capture).  `bytes` must be
// the same on every call for a given K.
template <auto K>
inline cudaError_t ensure_max_smem(int bytes) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// The driver's cuTensorMapEncodeTiled, looked up once per process (thread-safe);
// nullptr if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// The launch choices of moe_tuning (include/moe.h): read once from the MOE_*
// environment variables, replaced by moe_set_tuning; a snapshot per call.
moe_tuning tuning();

// Launch `kernel` on `s` with programmatic stream serialization (unless
// tuning().pdl is 0) and, when cluster_x > 1, clusters of cluster_x CTAs.  The
// kernel must call pdl_wait() before touching global memory.
bool pdl_enabled();
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kChunk = 32;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;

inline int num_chunks(int T) { return (T + kChunk - 1) / kChunk; }

// ---------------------------------------------------------------- route.cu
cudaError_t launch_router_logits(const void* x, const float* wr, const float* bias, float* logits,
                                 int T, int H, int E, int* err, cudaStream_t s);
// sigmoid = 0: softmax over the top-k logits; 1: noaux_tc, keys sigmoid(l) +
// sel_bias (nullable), weights the chosen sigmoid scores renormalised
cudaError_t launch_topk(const float* logits, const float* sel_bias, int sigmoid, int32_t* idx,
                        float* w, int T, int E, int k, cudaStream_t s);
// S1 + S2 with tensor-core logits (route.cu): launch_router_tc writes the
// approximate logits approx [T, E] (without bias) from the router weights split
// into three bf16 pieces wp [E][3H], with the norms xnorm [T] and wnorm [E];
// launch_topk_tc then makes the same selection as the canonical router logits
// followed by launch_topk (recomputing canonical logits where the approximate
// ones leave the order in doubt).  logit_bias: softmax routing's bias (added to
// the logits); sel_bias: sigmoid routing's selection bias.
// approx: `splits` blocks [T, E] fp32 (splits = dense_split_k(T, E, 3 H));
// with splits > 1 launch_router_tc leaves their sum in the first block and a
// bound on the running sums' magnitudes in the second, which launch_topk_tc
// reads
cudaError_t launch_router_tc(const void* x, const float* wr, int T, int H, int E, uint16_t* wp,
                             float* xnorm, float* wnorm, float* approx, int splits, int* err,
                             cudaStream_t s);
cudaError_t launch_topk_tc(const float* approx, int splits, const float* logit_bias,
                           const float* sel_bias, int sigmoid, const void* x, const float* wr,
                           const float* xnorm, const float* wnorm, int32_t* idx, float* w, int T,
                           int H, int E, int k, cudaStream_t s);

// ---------------------------------------------------------------- permute.cu
// cc[e * nch + c] = #tokens of chunk c that picked expert e.
// ticket: one int the count kernel zeroes and the scan kernel's blocks count on
cudaError_t launch_count(const int32_t* idx, int32_t* cc, int32_t* ticket, int T, int E, int k,
                         int* err, cudaStream_t s);
// cbase[e * nch + c] = rows of expert e in chunks < c; cnt, off (E+1); then the
// tile work list: groups 0..E-1 are the routed experts (rows off[g]..off[g+1]),
// group E (if shared_rows > 0) covers rows shared_row0 .. shared_row0+shared_rows.
cudaError_t launch_scan(const int32_t* cc, int32_t* cbase, int32_t* cnt, int32_t* off,
                        int32_t* ticket, int T, int E, int k, int4* items, int32_t* n_items,
                        int max_items, int BN, int shared_row0, int shared_rows, cudaStream_t s);
cudaError_t launch_items_from_offsets(const int32_t* off, int E, int4* items, int32_t* n_items,
                                      int max_items, int BN, cudaStream_t s);
// count + scan + rank in one single-block launch, for T <= 1024 when the
// per-chunk masks and bases ([nch][E] words each) fit kIndexSmallSmem bytes of
// shared memory.
constexpr size_t kIndexSmallSmem = 96 * 1024;
bool index_small_fits(int T, int E);
cudaError_t launch_index_small(const int32_t* idx, const float* topk_w, int32_t* cnt, int32_t* off,
                               int32_t* perm, int32_t* src, float* row_w, int T, int E, int k,
                               int4* items, int32_t* n_items, int max_items, int BN,
                               int shared_row0, int shared_rows, int* err, cudaStream_t s);
cudaError_t launch_rank(const int32_t* idx, const float* topk_w, const int32_t* off,
                        const int32_t* cbase, int32_t* perm, int32_t* src, float* row_w, int T,
                        int E, int k, cudaStream_t s);
// Per-token fp8 quantisation of x, copied to each routed row perm[t, :] and
// (when shared_row0 >= 0) to row shared_row0 + t.  acc_zero [T, H] fp32, when
// given, is zeroed (the fused combine's sum).
cudaError_t launch_quant_scatter(const void* x, const int32_t* perm, void* xq, float* xscale,
                                 int T, int H, int k, int shared_row0, int* err, cudaStream_t s,
                                 float* acc_zero = nullptr);
// Per-row fp8 requantisation of h [rows, I] bf16.
cudaError_t launch_requant(const void* h, void* hq, float* hs, int rows, int I, cudaStream_t s);
// out[t] = bf16(sum_j y[perm[t,j]] + shared[t]); shared may be NULL.
cudaError_t launch_combine(const void* y, const int32_t* perm, const void* shared, void* out,
                           int T, int H, int k, int* err, cudaStream_t s);
// out = bf16(acc) element-wise, n elements (n % 8 == 0): the fused combine's
// last pass.
cudaError_t launch_acc_to_bf16(const float* acc, void* out, size_t n, cudaStream_t s);
// yn[t] = bf16(RMSNorm(sum_j y[perm[t,j]]) * gamma), width L, eps given.
cudaError_t launch_combine_rmsnorm(const void* y, const int32_t* perm, const void* gamma, void* yn,
                                   int T, int L, int k, float eps, int* err, cudaStream_t s);

// ---------------------------------------------------------------- ffn_gemm.cu
struct GroupedFfnArgs {
  // work list
  const int4* items;      // {group, row0, rows, 0}
  const int32_t* n_items;
  int max_items;
  int E;                  // group index E is the shared expert
  int K;                  // expert input/output width (H or latent)
  int I;                  // expert intermediate width (shared must match)
  int rows_total;         // rows in the activation buffers
  // operands
  const void* xq;         // [rows_total, K] e4m3
  const float* xscale;    // [rows_total]
  const float* row_w;     // [rows_total] or NULL (=1)
  const void* w13;        // [E, 2I, K] e4m3
  const float* w13_scale; // [E, 2I]
  const void* w2;         // [E, K, I] e4m3
  const float* w2_scale;  // [E, K]
  const void* sw13;       // [2I, K] e4m3 or NULL
  const float* sw13_scale;
  const void* sw2;        // [K, I] e4m3 or NULL
  const float* sw2_scale;
  // intermediates / outputs
  void* h;                // [rows_total, I] bf16
  void* hq;               // [rows_total, I] e4m3
  float* hs;              // [rows_total]
  void* y;                // [rows_total, K] bf16
  float* out_acc;         // [T, K] fp32 or NULL: FFN2 adds rows into out_acc[token]
                          // with fp32 reductions instead of storing y
  const int32_t* src;     // [R] token of each routed row (out_acc only)
  int R;                  // routed rows; rows R.. are the shared expert's (token = row - R)
  int T;                  // tokens (rows of out_acc)
  int BN;                 // token rows per tile (32, 64, 128, 256)
  int packed;             // fp8 weights in tile-major order (pack.cu)
  int act;                // FFN1 activation: 0 SwiGLU, 1 SiTU (gated_act)
  int gather;             // FFN1 (single-SM, per-channel): xq / xscale hold one row per
                          // token; the producer gathers row r of a tile from token
                          // src[r] (routed) or r - R (shared expert)
  int blockwise;          // fp8 weights with fp32 scales per 128 x 128 block:
                          // w13_scale [E][2I/128][K/128], w2_scale [E][K/128][I/128]
  int* err;
};

cudaError_t launch_ffn1(const GroupedFfnArgs& a, cudaStream_t s);
cudaError_t launch_ffn2(const GroupedFfnArgs& a, cudaStream_t s);

// ---------------------------------------------------------------- ffn_gemm_2cta.cu
// Same contract on pairs of SMs (256-row tiles); needs BN == 256, K % 256 == 0.
cudaError_t launch_ffn1_pair(const GroupedFfnArgs& a, cudaStream_t s);
cudaError_t launch_ffn2_pair(const GroupedFfnArgs& a, cudaStream_t s);

// Dense bf16 GEMM on SM pairs: out[rows, N] = bf16(x w^T (+ x2 w2^T)), or with
// swiglu: w holds 2N rows (gate rows then up rows) and out = bf16(silu(g) u).
// K1, K2 multiples of 64; N a multiple of 256 (128 with swiglu).
struct DenseGemmArgs {
  const void* x;   // [rows, K1] bf16
  const void* w;   // [N or 2N, K1] bf16
  int K1;
  const void* x2;  // [rows, K2] bf16 (K2 = 0: none)
  const void* w2;  // [N, K2] bf16
  int K2;
  int rows, N;
  bool swiglu;
  int act;                // with swiglu: 0 SwiGLU, 1 SiTU (gated_act)
  void* out;       // [rows, N] bf16
  int* err;
};
cudaError_t launch_dense_bf16(const DenseGemmArgs& d, cudaStream_t s);
// out[rows, N] fp32 = sum_{k < Kw} x[:, k mod Kx] * w[:, k] (x [rows, Kx], w [N, Kw]
// bf16, Kx % 64 == 0, Kw a multiple of Kx): one accumulation in tensor memory.
// K ranges for the dense fp32-output GEMM (1 = none): enough for every SM pair
// when its output has few 256 x 256 tiles, each range non-empty.
int dense_split_k(int rows, int N, int Kw);
cudaError_t launch_dense_bf16_f32(const void* x, int Kx, const void* w, int Kw, int rows, int N,
                                  float* out, int ksplit, int* err, cudaStream_t s);

// ---------------------------------------------------------------- latent_down.cu
// z [T, L] = nearest-even bf16 of the exact x Wd^T (x [T, H], Wd [L, H] bf16):
// a chunked SM-pair GEMM, then an exact recomputation of the elements whose
// rounding the GEMM's remaining error could change.  flags: workspace of
// latent_down_flag_bytes(T, L).  H % 128 == 0, L % 128 == 0, 4 H + 2 L <= 160 KiB.
size_t latent_down_flag_bytes(int T, int L);
cudaError_t launch_latent_down(const void* x, const void* wd, void* z, uint32_t* flags, int T,
                               int H, int L, int* err, cudaStream_t s);

// ---------------------------------------------------------------- ffn_gemm_mx.cu
// MXFP4 routed experts (w13/w2 packed e2m1, w13_scale/w2_scale e8m0 bytes);
// BN in {32, 64, 96}; no shared-expert group.
// True when the MXFP4 GEMM of FFN1 (ffn1) or FFN2 runs on SM pairs.
bool mx_pair_eligible(const GroupedFfnArgs& a, bool ffn1);
cudaError_t launch_ffn1_mx(const GroupedFfnArgs& a, cudaStream_t s);
cudaError_t launch_ffn2_mx(const GroupedFfnArgs& a, cudaStream_t s);

// Shared helpers (moe_api.cu)
// Host-side validation of a problem (moe_status): the checks every entry point
// that takes a moe_problem applies before it launches anything.
int check_problem(const moe_problem* p);
int device_sm_count();
void count_launch();
int* device_error_word();  // device address of the current device's error word

}  // namespace moe
