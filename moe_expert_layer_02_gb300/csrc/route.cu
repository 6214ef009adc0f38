// route.cu -- S1 router logits and S2 top-k routing.
//
// S1: logits[t,e] = sum_h float(x[t,h]) * Wr[e,h] (+ bias[e]) in fp32, in one
// fixed order: lane l of a warp owns h = l, l+32, l+64, ... and chains fused
// multiply-adds over them in ascending h; the 32 partials are combined by a
// shuffle-down tree (p_l += p_{l+16}, then 8, 4, 2, 1), and the bias is added
// last.  Any implementation that follows the same order gets the same bits, so
// the top-k selection can be checked exactly.  (Routing metadata, "Optimising
// Ling-2.6-1T on TPU with SGLang-JAX", s.6; fp32 logits on the router.)
//
// S2: one warp per token picks the top-k logits by repeated warp arg-max over
// 64-bit keys (order-preserving logit bits, then the complement of the expert
// index, so equal logits go to the lower index), then w_j = exp(l_j - l_0) /
// sum exp(l_j' - l_0): the softmax over the chosen k (Ling write-up, s.1 top-8;
// "Kimi K3 ... feasibility analysis", s.2.4, moe_renormalize, scaling 1.0).
#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int RT_TOK = 32;  // tokens per block
constexpr int RT_EXP = 16;  // experts per block
constexpr int RT_HK = 128;  // h per staged chunk
constexpr int RT_TW = 8;    // tokens per warp
constexpr int RT_EW = 8;    // experts per warp

__global__ void __launch_bounds__(256)
    router_logits_kernel(const uint16_t* __restrict__ x, const float* __restrict__ wr,
                         const float* __restrict__ bias, float* __restrict__ logits, int T, int H,
                         int E) {
  __shared__ float xs[RT_TOK][RT_HK];
  __shared__ float ws[RT_EXP][RT_HK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tg = warp & 3, eg = warp >> 2;
  const int t0 = blockIdx.x * RT_TOK, e0 = blockIdx.y * RT_EXP;
  float acc[RT_TW][RT_EW];
#pragma unroll
  for (int i = 0; i < RT_TW; ++i)
#pragma unroll
    for (int j = 0; j < RT_EW; ++j) acc[i][j] = 0.0f;

  for (int h0 = 0; h0 < H; h0 += RT_HK) {
    // x tile: 32 tokens x 128 h, 8 bf16 per thread-iteration
    for (int i = threadIdx.x; i < RT_TOK * (RT_HK / 8); i += blockDim.x) {
      const int r = i / (RT_HK / 8), c = (i % (RT_HK / 8)) * 8;
      const int t = t0 + r;
      uint4 u = make_uint4(0, 0, 0, 0);
      if (t < T) u = *reinterpret_cast<const uint4*>(x + (size_t)t * H + h0 + c);
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xs[r][c + 2 * q] = bf16_bits_to_f32(w4[q] & 0xFFFFu);
        xs[r][c + 2 * q + 1] = bf16_bits_to_f32(w4[q] >> 16);
      }
    }
    for (int i = threadIdx.x; i < RT_EXP * (RT_HK / 4); i += blockDim.x) {
      const int r = i / (RT_HK / 4), c = (i % (RT_HK / 4)) * 4;
      const int e = e0 + r;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < E) v = *reinterpret_cast<const float4*>(wr + (size_t)e * H + h0 + c);
      ws[r][c] = v.x;
      ws[r][c + 1] = v.y;
      ws[r][c + 2] = v.z;
      ws[r][c + 3] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int s = 0; s < RT_HK / 32; ++s) {
      float xv[RT_TW], wv[RT_EW];
#pragma unroll
      for (int i = 0; i < RT_TW; ++i) xv[i] = xs[tg * RT_TW + i][s * 32 + lane];
#pragma unroll
      for (int j = 0; j < RT_EW; ++j) wv[j] = ws[eg * RT_EW + j][s * 32 + lane];
#pragma unroll
      for (int i = 0; i < RT_TW; ++i)
#pragma unroll
        for (int j = 0; j < RT_EW; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < RT_TW; ++i) {
#pragma unroll
    for (int j = 0; j < RT_EW; ++j) {
      float v = acc[i][j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = v + __shfl_down_sync(0xffffffffu, v, o);
      const int t = t0 + tg * RT_TW + i, e = e0 + eg * RT_EW + j;
      if (lane == 0 && t < T && e < E) logits[(size_t)t * E + e] = bias ? v + bias[e] : v;
    }
  }
}

template <int VPL>
__global__ void __launch_bounds__(256)
    topk_kernel(const float* __restrict__ logits, int32_t* __restrict__ idx, float* __restrict__ w,
                int T, int E, int k) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* row = logits + (size_t)warp * E;
  uint64_t key[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = i * 32 + lane;
    key[i] = (e < E) ? ((uint64_t)float_order_key(row[e]) << 32) | (uint64_t)(0xFFFFFFFFu - e) : 0;
  }
  float my_logit = 0.0f;  // lane j keeps the j-th chosen logit
  int my_idx = 0;
  float l0 = 0.0f;
  for (int j = 0; j < k; ++j) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    const int e = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFu));
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (key[i] == best) key[i] = 0;  // owner drops the winner
    const float le = row[e];
    if (j == 0) l0 = le;
    if (lane == j) {
      my_logit = le;
      my_idx = e;
    }
  }
  const float ex = lane < k ? expf(my_logit - l0) : 0.0f;
  float sum = 0.0f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);  // j ascending
  if (lane < k) {
    idx[(size_t)warp * k + lane] = my_idx;
    w[(size_t)warp * k + lane] = ex / sum;
  }
}

}  // namespace

cudaError_t launch_router_logits(const void* x, const float* wr, const float* bias, float* logits,
                                 int T, int H, int E, cudaStream_t s) {
  dim3 grid((T + RT_TOK - 1) / RT_TOK, (E + RT_EXP - 1) / RT_EXP);
  count_launch();
  router_logits_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(x), wr, bias, logits, T,
                                            H, E);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, int32_t* idx, float* w, int T, int E, int k,
                        cudaStream_t s) {
  const int blocks = (T * 32 + 255) / 256;
  count_launch();
  const int vpl = (E + 31) / 32;
  if (vpl <= 1)
    topk_kernel<1><<<blocks, 256, 0, s>>>(logits, idx, w, T, E, k);
  else if (vpl <= 2)
    topk_kernel<2><<<blocks, 256, 0, s>>>(logits, idx, w, T, E, k);
  else if (vpl <= 4)
    topk_kernel<4><<<blocks, 256, 0, s>>>(logits, idx, w, T, E, k);
  else if (vpl <= 8)
    topk_kernel<8><<<blocks, 256, 0, s>>>(logits, idx, w, T, E, k);
  else if (vpl <= 16)
    topk_kernel<16><<<blocks, 256, 0, s>>>(logits, idx, w, T, E, k);
  else
    topk_kernel<32><<<blocks, 256, 0, s>>>(logits, idx, w, T, E, k);
  return cudaGetLastError();
}

}  // namespace moe
