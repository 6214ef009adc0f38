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
// Sigmoid routing (K3 s.2.4, noaux_tc + sigmoid, ungrouped): the keys are
// s_e + bias_e with s_e = sigmoid(logit_e) in a canonical fp32 sequence, the
// bias steering selection only; w_j = s_j / sum_j' s_j'.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>

#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

// ---------------------------------------------------------------- S1 router
// Block = WT x 2 warps (token groups x expert groups); thread 0 also issues
// the loads.  Warp tile TW tokens x EW experts; lane l owns h = l (mod 32) of
// every 128-wide chunk, so each logit is one fma chain over h ascending, as
// the canonical order requires.  Stages of NSUB chunks stream through a
// shared-memory ring filled by 2-D TMA loads (one [rows][128] box per chunk:
// x bf16, router fp32; out-of-range rows read as zero).  Pairs of experts share
// one packed fma.rn.f32x2 (two independent fp32 fused multiply-adds, same
// rounding as fmaf).
// No separate producer warp: the register file is handed to a block in groups
// of four warps, so a ninth warp would cost the eight compute warps a quarter
// of their registers.  Per packed FMA the loop also issues ~0.4 shared loads,
// and the load pipe and shared-memory bandwidth run at about half their peak
// beside the FMA pipe's ~60%, so more warps per scheduler (twelve) pay off
// when the grid is large.
constexpr int RT_CH = 128;  // h per chunk (one TMA box)

template <int TW, int EW, int NSUB_ = 0, int WT_ = 4>
struct RouterCfg {
  static constexpr int WT = WT_, WE = 2;  // warp grid: token groups x expert groups
  static constexpr int WARPS = WT * WE;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int BT = WT * TW;  // tokens per block
  static constexpr int BE = WE * EW;  // experts per block
  // small warp tiles fit two blocks per SM (128 registers a thread), large
  // ones one (up to 255 with 8 warps)
  static constexpr int MIN_BLOCKS = (TW * EW <= 64 && WARPS <= 8) ? 2 : 1;
  static constexpr int BUDGET = 216 * 1024 / MIN_BLOCKS;  // ring bytes per block
  static constexpr int XBOX = BT * RT_CH * 2;            // bf16 [BT][128]
  static constexpr int WBOX = BE * RT_CH * 4;            // fp32 [BE][128]
  // every stage costs a barrier round trip and a load-latency bubble, so a
  // stage carries four chunks when three such stages fit, else two
  static constexpr int NSUB = NSUB_ ? NSUB_ : (3 * 4 * (XBOX + WBOX) <= BUDGET) ? 4 : 2;
  static constexpr int HK = NSUB * RT_CH;  // h per stage
  static constexpr int X_BYTES = NSUB * XBOX;
  static constexpr int W_BYTES = NSUB * WBOX;
  static constexpr int STAGE = X_BYTES + W_BYTES;  // NSUB x boxes, then NSUB router boxes
  static constexpr int STAGES = BUDGET / STAGE;
  static constexpr int SMEM = 128 + STAGES * STAGE + 2 * STAGES * 8 + 16;
};

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ void fma2(uint64_t& acc, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

template <int TW, int EW, int NS, int WT>
__global__ void __launch_bounds__(RouterCfg<TW, EW, NS, WT>::THREADS,
                                  RouterCfg<TW, EW, NS, WT>::MIN_BLOCKS)
    router_logits_kernel(const __grid_constant__ CUtensorMap tm_x,
                         const __grid_constant__ CUtensorMap tm_w, const float* __restrict__ bias,
                         float* __restrict__ logits, int T, int H, int E, int* err) {
  using C = RouterCfg<TW, EW, NS, WT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
  uint64_t* empty = full + C::STAGES;
  volatile int* s_abort = reinterpret_cast<volatile int*>(empty + C::STAGES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // token tiles are the fast grid dimension: the concurrent blocks share each
  // router-weight tile in L2 (T=16384, H=8192, E=256: expert tiles first was
  // slower; within a single wave the order makes no difference)
  const int t0 = blockIdx.x * C::BT, e0 = blockIdx.y * C::BE;
  // H % 128 == 0; the chunks of a partly filled last stage beyond H read
  // zeros, and a zero product leaves a chain unchanged
  const int nstage = (H + C::HK - 1) / C::HK;
  const bool producer = threadIdx.x == 0;

  if (producer) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), C::WARPS);
    }
    *s_abort = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  pdl_wait();  // the previous kernel's outputs are complete and visible
  pdl_release();

  auto issue = [&](int c) {  // stage c into slot c % STAGES
    const uint32_t st = smem_u32(smem + (c % C::STAGES) * C::STAGE);
    const uint32_t fb = smem_u32(&full[c % C::STAGES]);
    mbar_arrive_expect_tx(fb, C::STAGE);
#pragma unroll
    for (int u = 0; u < C::NSUB; ++u) {
      tma_load_2d(st + u * C::XBOX, &tm_x, c * C::HK + u * RT_CH, t0, fb);
      tma_load_2d(st + C::X_BYTES + u * C::WBOX, &tm_w, c * C::HK + u * RT_CH, e0, fb);
    }
  };
  int issued = 0;  // stages whose loads thread 0 has issued
  if (producer) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
    for (; issued < C::STAGES && issued < nstage; ++issued) issue(issued);
  }

  const int tg = warp % C::WT, eg = warp / C::WT;
  uint64_t acc[TW][EW / 2];  // {chain of expert 2j, chain of expert 2j+1} for token i
#pragma unroll
  for (int i = 0; i < TW; ++i)
#pragma unroll
    for (int j = 0; j < EW / 2; ++j) acc[i][j] = 0;  // +0.0f, +0.0f
  bool ok = true;
  for (int c = 0; c < nstage; ++c) {
    // refill stage c-1's slot with the next stage once every warp let go of it
    if (producer && issued < nstage && c >= 1) {
      const int p = c - 1;
      if (mbar_wait(smem_u32(&empty[p % C::STAGES]), (uint32_t)(p / C::STAGES) & 1u, err,
                    s_abort))
        issue(issued++);
    }
    const int s = c % C::STAGES;
    const uint32_t ph = (uint32_t)(c / C::STAGES) & 1u;
    int got = 1;
    if (lane == 0) got = mbar_wait(smem_u32(&full[s]), ph, err, s_abort) ? 1 : 0;
    got = __shfl_sync(0xffffffffu, got, 0);
    if (!got) {
      ok = false;
      break;
    }
#pragma unroll
    for (int u = 0; u < C::NSUB; ++u) {  // the chunks of the stage, h ascending
      const uint16_t* xs = reinterpret_cast<const uint16_t*>(smem + s * C::STAGE + u * C::XBOX) +
                           tg * TW * RT_CH;
      const float* ws = reinterpret_cast<const float*>(smem + s * C::STAGE + C::X_BYTES +
                                                       u * C::WBOX) +
                        eg * EW * RT_CH;
#pragma unroll
      for (int q = 0; q < RT_CH / 32; ++q) {
        const int h = q * 32 + lane;
        uint64_t wv[EW / 2];
#pragma unroll
        for (int j = 0; j < EW / 2; ++j)
          wv[j] = pack2(ws[(2 * j) * RT_CH + h], ws[(2 * j + 1) * RT_CH + h]);
#pragma unroll
        for (int i = 0; i < TW; ++i) {
          const float xv = bf16_bits_to_f32(xs[i * RT_CH + h]);
          const uint64_t xx = pack2(xv, xv);
#pragma unroll
          for (int j = 0; j < EW / 2; ++j) fma2(acc[i][j], xx, wv[j]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
  }
  if (!ok) {
    // a wait gave up: the last STAGES issued stages may still be in flight
    // (every earlier one was consumed by all warps); let them land before exit
    if (producer)
      for (int c = max(0, issued - C::STAGES); c < issued; ++c)
        mbar_wait_drain(smem_u32(&full[c % C::STAGES]), (uint32_t)(c / C::STAGES) & 1u);
    return;
  }

#pragma unroll
  for (int i = 0; i < TW; ++i) {
#pragma unroll
    for (int j = 0; j < EW / 2; ++j) {
      float v[2];
      unpack2(acc[i][j], v[0], v[1]);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        float r = v[u];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) r = r + __shfl_down_sync(0xffffffffu, r, o);
        const int t = t0 + tg * TW + i, e = e0 + eg * EW + 2 * j + u;
        if (lane == 0 && t < T && e < E) logits[(size_t)t * E + e] = bias ? r + bias[e] : r;
      }
    }
  }
}

// exp(a) for a <= 0 in one fixed fp32 sequence: Cody-Waite reduction a = n ln2
// + r with n = rint(a log2 e) and ln2 split into a head exact in 15 bits plus a
// tail, e^r by its Taylor series through r^7/7! in Horner form (|r| <= 0.35,
// truncation < 2^-26), then an exact multiply by 2^n (n >= -125).  a <= -86
// gives 0.  Every step is an IEEE-rounded fp32 operation, so the result is the
// same on any machine that follows the sequence.
__device__ __forceinline__ float exp_fixed(float a) {
  if (!(a > -86.0f)) return 0.0f;
  if (a > 0.0f) a = 0.0f;
  const float n = rintf(__fmul_rn(a, 1.44269504f));
  float r = fmaf(-n, 0.693145751953125f, a);
  r = fmaf(-n, 1.42860677e-6f, r);
  float q = 1.0f / 5040.0f;
  q = fmaf(q, r, 1.0f / 720.0f);
  q = fmaf(q, r, 1.0f / 120.0f);
  q = fmaf(q, r, 1.0f / 24.0f);
  q = fmaf(q, r, 1.0f / 6.0f);
  q = fmaf(q, r, 0.5f);
  q = fmaf(q, r, 1.0f);
  q = fmaf(q, r, 1.0f);
  return __fmul_rn(q, __int_as_float(((int)n + 127) << 23));
}

// sigmoid(l): 1 / (1 + e^-l) for l >= 0, e^l / (1 + e^l) below, IEEE add/divide.
__device__ __forceinline__ float sigmoid_fixed(float l) {
  const float u = exp_fixed(l >= 0.0f ? -l : l);
  const float d = __fadd_rn(1.0f, u);
  return l >= 0.0f ? __fdiv_rn(1.0f, d) : __fdiv_rn(u, d);
}

template <int VPL>
__global__ void __launch_bounds__(256)
    topk_kernel(const float* __restrict__ logits, const float* __restrict__ sel_bias,
                int32_t* __restrict__ idx, float* __restrict__ w, int T, int E, int k,
                int sigmoid) {
  pdl_wait();  // the previous kernel's outputs are complete and visible
  pdl_release();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* row = logits + (size_t)warp * E;
  uint64_t key[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = i * 32 + lane;
    float v = 0.0f;
    if (e < E) {
      v = row[e];
      if (sigmoid) {
        v = sigmoid_fixed(v);
        if (sel_bias) v = __fadd_rn(v, sel_bias[e]);
      }
    }
    key[i] = (e < E) ? ((uint64_t)float_order_key(v) << 32) | (uint64_t)(0xFFFFFFFFu - e) : 0;
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
  const float ex =
      lane >= k ? 0.0f : sigmoid ? sigmoid_fixed(my_logit) : expf(my_logit - l0);
  float sum = 0.0f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);  // j ascending
  if (lane < k) {
    idx[(size_t)warp * k + lane] = my_idx;
    w[(size_t)warp * k + lane] = ex / sum;
  }
}

// ---------------------------------------------------------------- S1 + S2 on tensor cores
// The router GEMM has T x E x H multiply-adds (69 G at T=16384, H=8192,
// E=256), which the CUDA cores take 1.4 ms over in the canonical order.  Here
// the tensor cores compute the logits: x is bf16, and every fp32 router weight
// splits exactly into three bf16 pieces, w = w_lo + w_mid + w_hi (8 + 8 + 8
// significant bits), so x . w = x . w_lo + x . w_mid + x . w_hi with products
// exact in fp32; one tcgen05 accumulation over K = 3H, small pieces first,
// gives an approximate logit a[t,e] within a few units of 2^-23 |x_t| |w_e|
// of the canonical one.  The selection is then made exact: per token, the top
// k + 1 approximate keys are compared with per-element margins
// m[t,e] = MOE_RFLAG_ULPS * 2^-23 * |x_t| * |w_e| (|.| the Euclidean norm);
// when every adjacent gap exceeds the two margins, the approximate order is the
// canonical order.  Otherwise every expert that could still take a place
// (key + margin >= the k-th key - its margin) gets its canonical logit (32
// fused multiply-add chains over h = l (mod 32), the halving tree, the bias
// last: bit for bit the router kernel's value), and the top k among those are
// chosen exactly.  The routing weights come from the logits the selection used.
//
// Margin calibration (GB300; x N(0,1), router N(0, 1/H); tokens whose
// selection or order came out different from the canonical routing, by margin
// in units of 2^-23 |x_t| |w_e|): 0 -> 3 of 16384 at T=16384, H=8192, E=256,
// k=8 and 1 of 8192 on the Zipf-biased T=8192 batch; 1, 4, 16 and 64 -> none
// on those and on T=4096, H=7168, E=896, k=16.  Eight leaves a factor of
// eight over the smallest clean margin; the recompute then runs on a few per
// cent of tokens (S1 + S2: 0.38 ms at T=16384 against 1.49 ms canonical).
#ifndef MOE_RFLAG_ULPS
#define MOE_RFLAG_ULPS 8.0f
#endif

// Blocks [0, E): router row e -> pieces (lo, mid, hi) at wp[e][0..3H) and its
// norm.  Blocks past E: eight tokens each, one warp per token: |x_t|.
__global__ void __launch_bounds__(256)
    router_prep_kernel(const uint16_t* __restrict__ x, const float* __restrict__ wr,
                       uint16_t* __restrict__ wp, float* __restrict__ xnorm,
                       float* __restrict__ wnorm, int T, int H, int E) {
  pdl_wait();
  pdl_release();
  __shared__ float s_part[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int)blockIdx.x < E) {
    const int e = blockIdx.x;
    const float* row = wr + (size_t)e * H;
    uint16_t* lo = wp + (size_t)e * 3 * H;
    float ss = 0.0f;
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
      const float v = row[h];
      const __nv_bfloat16 bh = __float2bfloat16_rn(v);
      const float r1 = __fsub_rn(v, __bfloat162float(bh));  // exact
      const __nv_bfloat16 bm = __float2bfloat16_rn(r1);
      const float r2 = __fsub_rn(r1, __bfloat162float(bm));  // exact, <= 8 significant bits
      const __nv_bfloat16 bl = __float2bfloat16_rn(r2);      // exact
      lo[h] = *reinterpret_cast<const uint16_t*>(&bl);
      lo[H + h] = *reinterpret_cast<const uint16_t*>(&bm);
      lo[2 * H + h] = *reinterpret_cast<const uint16_t*>(&bh);
      ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s_part[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.0f;
      for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += s_part[i];
      wnorm[e] = sqrtf(t);
    }
  } else {
    const int t = ((int)blockIdx.x - E) * 8 + warp;
    if (t >= T) return;
    const uint16_t* row = x + (size_t)t * H;
    float ss = 0.0f;
    for (int h = lane; h < H; h += 32) {
      const float v = bf16_bits_to_f32(row[h]);
      ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) xnorm[t] = sqrtf(ss);
  }
}

// The canonical logit of (token row xr, router row wrow), as the router kernel
// computes it, in every lane of the warp.
__device__ __forceinline__ float canonical_logit(const uint16_t* __restrict__ xr,
                                                 const float* __restrict__ wrow, int H, int lane) {
  float p = 0.0f;
  for (int h = lane; h < H; h += 32) p = fmaf(bf16_bits_to_f32(xr[h]), wrow[h], p);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) p = p + __shfl_down_sync(0xffffffffu, p, o);
  return __shfl_sync(0xffffffffu, p, 0);
}

template <int VPL>
__global__ void __launch_bounds__(256)
    topk_tc_kernel(const float* __restrict__ approx, const float* __restrict__ logit_bias,
                   const float* __restrict__ sel_bias, int sigmoid,
                   const uint16_t* __restrict__ x, const float* __restrict__ wr,
                   const float* __restrict__ xnorm, const float* __restrict__ wnorm,
                   int32_t* __restrict__ idx, float* __restrict__ w, int T, int H, int E, int k) {
  pdl_wait();
  pdl_release();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* row = approx + (size_t)t * E;
  const float xm = MOE_RFLAG_ULPS * 0x1p-23f * xnorm[t];
  // keys (as the canonical top-k forms them) and their margins
  float kv[VPL], km[VPL], lv[VPL];
  uint64_t key[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = i * 32 + lane;
    float l = 0.0f, v = 0.0f, m = 0.0f;
    if (e < E) {
      l = row[e];
      if (logit_bias) l = __fadd_rn(l, logit_bias[e]);
      const float ml = xm * wnorm[e];
      if (sigmoid) {
        v = sigmoid_fixed(l);
        if (sel_bias) v = __fadd_rn(v, sel_bias[e]);
        m = 0.25f * ml + 0x1p-20f;  // sigmoid' <= 1/4, plus its own last-bit error
      } else {
        v = l;
        m = ml + 0x1p-22f * fabsf(l);  // plus the bias addition's rounding
      }
    }
    lv[i] = l;
    kv[i] = v;
    km[i] = m;
    key[i] = (e < E) ? ((uint64_t)float_order_key(v) << 32) | (uint64_t)(0xFFFFFFFFu - e) : 0;
  }
  // the k + 1 best keys by the approximate values: lane j keeps the j-th
  const int nsel = k < E ? k + 1 : k;
  float my_v = 0.0f, my_m = 0.0f, my_l = 0.0f;
  int my_e = 0;
  for (int j = 0; j < nsel; ++j) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    const int e = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFu));
    float bv = 0.0f, bm = 0.0f, bl = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (key[i] == best) {  // the owner drops the winner and shares its values
        key[i] = 0;
        bv = kv[i];
        bm = km[i];
        bl = lv[i];
      }
    const int owner = e & 31;
    bv = __shfl_sync(0xffffffffu, bv, owner);
    bm = __shfl_sync(0xffffffffu, bm, owner);
    bl = __shfl_sync(0xffffffffu, bl, owner);
    if (lane == j) {
      my_v = bv;
      my_m = bm;
      my_l = bl;
      my_e = e;
    }
  }
  // the approximate order is the canonical one when every adjacent gap of the
  // k + 1 best keys exceeds both margins
  const float nx_v = __shfl_down_sync(0xffffffffu, my_v, 1);
  const float nx_m = __shfl_down_sync(0xffffffffu, my_m, 1);
  const bool close = lane < k && lane + 1 < nsel && !(my_v - nx_v > my_m + nx_m);
  if (__any_sync(0xffffffffu, close)) {
    // exact: the canonical keys of every expert that could still place
    const float kth_v = __shfl_sync(0xffffffffu, my_v, k - 1);
    const float kth_m = __shfl_sync(0xffffffffu, my_m, k - 1);
    const float floor_v = kth_v - kth_m;
    uint64_t top = 0;  // lane j < k: the j-th best canonical key so far
    float top_l = 0.0f;
    const uint16_t* xr = x + (size_t)t * H;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e0 = i * 32 + lane;
      unsigned cand = __ballot_sync(0xffffffffu, e0 < E && kv[i] + km[i] >= floor_v);
      while (cand) {
        const int b = __ffs(cand) - 1;
        cand &= cand - 1u;
        const int e = i * 32 + b;
        float l = canonical_logit(xr, wr + (size_t)e * H, H, lane);
        if (logit_bias) l = __fadd_rn(l, logit_bias[e]);
        float v = l;
        if (sigmoid) {
          v = sigmoid_fixed(l);
          if (sel_bias) v = __fadd_rn(v, sel_bias[e]);
        }
        const uint64_t ck = ((uint64_t)float_order_key(v) << 32) | (uint64_t)(0xFFFFFFFFu - e);
        // insert into the sorted top-k list held by lanes 0..k-1
        const int pos = __popc(__ballot_sync(0xffffffffu, lane < k && top > ck));
        const uint64_t up = __shfl_up_sync(0xffffffffu, top, 1);
        const float up_l = __shfl_up_sync(0xffffffffu, top_l, 1);
        if (lane < k && pos < k) {
          if (lane == pos) {
            top = ck;
            top_l = l;
          } else if (lane > pos) {
            top = up;
            top_l = up_l;
          }
        }
      }
    }
    my_e = (int)(0xFFFFFFFFu - (uint32_t)(top & 0xFFFFFFFFu));
    my_l = top_l;
  }
  const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
  const float ex = lane >= k ? 0.0f : sigmoid ? sigmoid_fixed(my_l) : expf(my_l - l0);
  float sum = 0.0f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);  // j ascending
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_e;
    w[(size_t)t * k + lane] = ex / sum;
  }
}

}  // namespace

namespace {

bool router_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, int H,
                int rows, int box_rows) {  // [box_rows][128] boxes
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (!enc) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)H * esize};
  cuuint32_t box[2] = {(cuuint32_t)RT_CH, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int TW, int EW, int NS = 0, int WT = 4>
cudaError_t launch_router_impl(const void* x, const float* wr, const float* bias, float* logits,
                               int T, int H, int E, int* err, cudaStream_t s) {
  using C = RouterCfg<TW, EW, NS, WT>;
  CUtensorMap tx, tw;
  if (!router_map(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, H, T, C::BT) ||
      !router_map(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, wr, H, E, C::BE))
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_max_smem<router_logits_kernel<TW, EW, NS, WT>>(C::SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid((T + C::BT - 1) / C::BT, (E + C::BE - 1) / C::BE);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  count_launch();
  e = launch_kernel(router_logits_kernel<TW, EW, NS, WT>, grid, dim3(C::THREADS), C::SMEM, s, 1, tx,
                    tw, bias, logits, T, H, E, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_logits(const void* x, const float* wr, const float* bias, float* logits,
                                 int T, int H, int E, int* err, cudaStream_t s) {
  // tuning().router_tile overrides the choice: 1 = 8 warps of 8 tokens x 8
  // experts (two blocks per SM), 2 = 8 warps of 8 x 16, 3 = the same with four
  // chunks per stage, 4 = 12 warps of 8 x 16 (48 tokens x 32 experts)
  switch (tuning().router_tile) {
    case 1: return launch_router_impl<8, 8>(x, wr, bias, logits, T, H, E, err, s);
    case 2: return launch_router_impl<8, 16>(x, wr, bias, logits, T, H, E, err, s);
    case 3: return launch_router_impl<8, 16, 4>(x, wr, bias, logits, T, H, E, err, s);
    case 4: return launch_router_impl<8, 16, 0, 6>(x, wr, bias, logits, T, H, E, err, s);
    default: break;
  }
  const long sms = device_sm_count();
  const long e32 = (E + 31) / 32;
  // Twelve warps (three per scheduler, 168 registers) hide more latency and
  // share each stage over 48 x 32 (token, expert) pairs; they need at least
  // two blocks per SM (T=16384, H=8192, E=256: 1.36 vs 1.44 ms with eight
  // warps; T=4096, H=7168, E=896: 1.08 ms)
  if ((long)((T + 47) / 48) * e32 >= 2L * sms)
    return launch_router_impl<8, 16, 0, 6>(x, wr, bias, logits, T, H, E, err, s);
  // eight warps of 8 x 16 when they still give every SM two blocks; in a
  // single wave of at least half the SMs, with four chunks per stage (T=512,
  // E=256: 56 us vs 59 us with two and 69 us with 8 x 8 tiles at two per SM)
  const long big_blocks = (long)((T + 31) / 32) * e32;
  if (big_blocks >= 2L * sms)
    return launch_router_impl<8, 16>(x, wr, bias, logits, T, H, E, err, s);
  if (2L * big_blocks >= sms && big_blocks <= sms)
    return launch_router_impl<8, 16, 4>(x, wr, bias, logits, T, H, E, err, s);
  return launch_router_impl<8, 8>(x, wr, bias, logits, T, H, E, err, s);
}

cudaError_t launch_router_tc(const void* x, const float* wr, int T, int H, int E, uint16_t* wp,
                             float* xnorm, float* wnorm, float* approx, int* err, cudaStream_t s) {
  if (T <= 0 || H % 64 || E <= 0 || E > 1024) return cudaErrorInvalidValue;
  count_launch();
  cudaError_t e = launch_kernel(router_prep_kernel, dim3(E + (T + 7) / 8), dim3(256), 0, s, 1,
                                static_cast<const uint16_t*>(x), wr, wp, xnorm, wnorm, T, H, E);
  if (e != cudaSuccess) return e;
  count_launch();
  e = launch_dense_bf16_f32(x, H, wp, 3 * H, T, E, approx, err, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_topk_tc(const float* approx, const float* logit_bias, const float* sel_bias,
                           int sigmoid, const void* x, const float* wr, const float* xnorm,
                           const float* wnorm, int32_t* idx, float* w, int T, int H, int E, int k,
                           cudaStream_t s) {
  if (T <= 0 || E <= 0 || E > 1024 || k > 32 || k > E) return cudaErrorInvalidValue;
  const int blocks = (T * 32 + 255) / 256;
  const int vpl = (E + 31) / 32;
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  count_launch();
  cudaError_t e;
#define MOE_TOPK_TC(V)                                                                      \
  launch_kernel(topk_tc_kernel<V>, dim3(blocks), dim3(256), 0, s, 1, approx, logit_bias,   \
                sel_bias, sigmoid, xb, wr, xnorm, wnorm, idx, w, T, H, E, k)
  if (vpl <= 1) e = MOE_TOPK_TC(1);
  else if (vpl <= 2) e = MOE_TOPK_TC(2);
  else if (vpl <= 4) e = MOE_TOPK_TC(4);
  else if (vpl <= 8) e = MOE_TOPK_TC(8);
  else if (vpl <= 16) e = MOE_TOPK_TC(16);
  else e = MOE_TOPK_TC(32);
#undef MOE_TOPK_TC
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, const float* sel_bias, int sigmoid, int32_t* idx,
                        float* w, int T, int E, int k, cudaStream_t s) {
  const int blocks = (T * 32 + 255) / 256;
  count_launch();
  const int vpl = (E + 31) / 32;
  if (vpl <= 1)
    return launch_kernel(topk_kernel<1>, dim3(blocks), dim3(256), 0, s, 1, logits, sel_bias, idx, w,
                         T, E, k, sigmoid);
  else if (vpl <= 2)
    return launch_kernel(topk_kernel<2>, dim3(blocks), dim3(256), 0, s, 1, logits, sel_bias, idx, w,
                         T, E, k, sigmoid);
  else if (vpl <= 4)
    return launch_kernel(topk_kernel<4>, dim3(blocks), dim3(256), 0, s, 1, logits, sel_bias, idx, w,
                         T, E, k, sigmoid);
  else if (vpl <= 8)
    return launch_kernel(topk_kernel<8>, dim3(blocks), dim3(256), 0, s, 1, logits, sel_bias, idx, w,
                         T, E, k, sigmoid);
  else if (vpl <= 16)
    return launch_kernel(topk_kernel<16>, dim3(blocks), dim3(256), 0, s, 1, logits, sel_bias, idx, w,
                         T, E, k, sigmoid);
  else
    return launch_kernel(topk_kernel<32>, dim3(blocks), dim3(256), 0, s, 1, logits, sel_bias, idx, w,
                         T, E, k, sigmoid);
}

}  // namespace moe
