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
// of the canonical one.  The selection is then made exact.  Each expert's
// canonical key lies within m[t,e] = MOE_RFLAG_ULPS * 2^-23 * |x_t| * |w_e|
// (|.| the Euclidean norm) of its approximate key.  Per token, the experts
// come out in approximate order, and a cut after position j is proven where
// every lower bound (key - margin) up to j lies above every upper bound after
// it, those of the experts not yet taken out included: the true order then
// keeps positions 0..j, as a set, above all the rest.  Once a cut at or past
// position k - 1 is proven, only the runs of two or more positions between
// cuts are uncertain; their experts get canonical logits (32 fused
// multiply-add chains over h = l (mod 32), the halving tree, the bias last:
// bit for bit the router kernel's value) and each run is sorted by the
// canonical keys.  If 32 positions prove no such cut, every expert whose
// upper bound reaches the least lower bound of the first k is recomputed.
// The routing weights come from the logits the selection used.
//
// Margin calibration (GB300; x N(0,1), router N(0, 1/H); tokens whose
// selection or order came out different from the canonical routing, by margin
// in units of 2^-23 |x_t| |w_e|): 0 -> 3 of 16384 at T=16384, H=8192, E=256,
// k=8 and 1 of 8192 on the Zipf-biased T=8192 batch; 1, 4, 16 and 64 -> none
// on those and on T=4096, H=7168, E=896, k=16.  Eight leaves a factor of
// eight over the smallest clean margin; the recompute then runs on a few per
// cent of tokens (S1 + S2: 0.25 ms at T=16384, E=256 alone, 0.31 ms inside
// the layer, against 1.49 ms canonical).
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
    const float4* row = reinterpret_cast<const float4*>(wr + (size_t)e * H);
    uint16_t* lo = wp + (size_t)e * 3 * H;
    float ss = 0.0f;
    for (int c = threadIdx.x; c < H / 4; c += blockDim.x) {
      const float4 v4 = row[c];
      const float v[4] = {v4.x, v4.y, v4.z, v4.w};
      uint16_t pl[4], pm[4], ph[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __nv_bfloat16 bh = __float2bfloat16_rn(v[j]);
        const float r1 = __fsub_rn(v[j], __bfloat162float(bh));  // exact
        const __nv_bfloat16 bm = __float2bfloat16_rn(r1);
        const float r2 = __fsub_rn(r1, __bfloat162float(bm));  // exact, <= 8 significant bits
        const __nv_bfloat16 bl = __float2bfloat16_rn(r2);      // exact
        pl[j] = *reinterpret_cast<const uint16_t*>(&bl);
        pm[j] = *reinterpret_cast<const uint16_t*>(&bm);
        ph[j] = *reinterpret_cast<const uint16_t*>(&bh);
        ss = fmaf(v[j], v[j], ss);
      }
      auto pack = [](const uint16_t (&q)[4]) {
        return make_uint2((uint32_t)q[0] | ((uint32_t)q[1] << 16),
                          (uint32_t)q[2] | ((uint32_t)q[3] << 16));
      };
      reinterpret_cast<uint2*>(lo)[c] = pack(pl);
      reinterpret_cast<uint2*>(lo + H)[c] = pack(pm);
      reinterpret_cast<uint2*>(lo + 2 * H)[c] = pack(ph);
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
    const long t = ((long)blockIdx.x - E) * 8 + warp;
    if (t >= T) return;
    // eight bf16 per 16-byte load (rows start 16-byte aligned: H % 64 == 0)
    const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    float ss = 0.0f;
    for (int c = lane; c < H / 8; c += 32) {
      const uint4 q = row[c];
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a0 = __uint_as_float(w[j] << 16), a1 = __uint_as_float(w[j] & 0xFFFF0000u);
        ss = fmaf(a0, a0, ss);
        ss = fmaf(a1, a1, ss);
      }
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

// Four canonical logits of one token row against four router rows at once
// (the x loads shared); each is computed exactly as canonical_logit does.
__device__ __forceinline__ void canonical_logits4(const uint16_t* __restrict__ xr,
                                                  const float* __restrict__ w0,
                                                  const float* __restrict__ w1,
                                                  const float* __restrict__ w2,
                                                  const float* __restrict__ w3, int H, int lane,
                                                  float (&out)[4]) {
  float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
#pragma unroll 8
  for (int h = lane; h < H; h += 32) {
    const float xv = bf16_bits_to_f32(xr[h]);
    p0 = fmaf(xv, w0[h], p0);
    p1 = fmaf(xv, w1[h], p1);
    p2 = fmaf(xv, w2[h], p2);
    p3 = fmaf(xv, w3[h], p3);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    p0 = p0 + __shfl_down_sync(0xffffffffu, p0, o);
    p1 = p1 + __shfl_down_sync(0xffffffffu, p1, o);
    p2 = p2 + __shfl_down_sync(0xffffffffu, p2, o);
    p3 = p3 + __shfl_down_sync(0xffffffffu, p3, o);
  }
  out[0] = __shfl_sync(0xffffffffu, p0, 0);
  out[1] = __shfl_sync(0xffffffffu, p1, 0);
  out[2] = __shfl_sync(0xffffffffu, p2, 0);
  out[3] = __shfl_sync(0xffffffffu, p3, 0);
}

// Split-K router GEMM: blocks 0..splits-1 of n logits each -> block 0 = their
// sum (block order), block 1 = the sum of their magnitudes (rounded up), one
// thread per logit.
__global__ void __launch_bounds__(256)
    router_sum_splits_kernel(float* __restrict__ p, size_t n, int splits) {
  pdl_wait();
  pdl_release();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float l = p[i], a = fabsf(l);
  for (int sp = 1; sp < splits; ++sp) {
    const float v = p[(size_t)sp * n + i];
    l = __fadd_rn(l, v);
    a = __fadd_ru(a, fabsf(v));
  }
  p[i] = l;
  p[n + i] = a;
}

// Blocks of four warps, one token per warp: a warp that recomputes canonical
// logits holds back only three others.
constexpr int TOPK_TC_THREADS = 128;

// The warp's 32 values sorted in descending order (lane 0 the largest) by a
// bitonic network: blocks of 2, 4, .. 16 lanes are sorted in alternating
// directions and merged, the last merge descending.
template <typename K>
__device__ __forceinline__ K warp_sort_desc(K v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const K o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
    }
  }
  return v;
}

// The float a key's upper half was made from (float_order_key inverted).
__device__ __forceinline__ float key_value(uint64_t key) {
  const uint32_t k = (uint32_t)(key >> 32);
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

template <int VPL>
__global__ void __launch_bounds__(TOPK_TC_THREADS, 1)
    topk_tc_kernel(const float* __restrict__ approx, int splits, size_t split_stride,
                   const float* __restrict__ logit_bias,
                   const float* __restrict__ sel_bias, int sigmoid,
                   const uint16_t* __restrict__ x, const float* __restrict__ wr,
                   const float* __restrict__ xnorm, const float* __restrict__ wnorm,
                   int32_t* __restrict__ idx, float* __restrict__ w, int T, int H, int E, int k) {
  pdl_wait();
  pdl_release();
  __shared__ uint64_t s_cand[TOPK_TC_THREADS / 32][32];  // per warp: candidate keys
  const long t = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* row = approx + (size_t)t * E;
  // split-K logits (router_sum_splits_kernel): block 0 holds the sum of the
  // blocks, block 1 the sum of their magnitudes, which bounds every running
  // sum, so the splits - 1 additions add at most (splits - 1) 2^-24 of it to
  // a logit's error
  const float* row_a = row + split_stride;
  const float xm = MOE_RFLAG_ULPS * 0x1p-23f * xnorm[t];
  const float am = (float)(splits - 1) * 0x1p-24f;
  // key of expert e (as the canonical top-k forms it) from its approximate
  // logit l; its margin follows from the key's value and |w_e|
  auto logit_of = [&](int e) {
    float l = row[e];
    if (logit_bias) l = __fadd_rn(l, logit_bias[e]);
    return l;
  };
  auto value_of = [&](int e, float l) {
    float v = l;
    if (sigmoid) {
      v = sigmoid_fixed(l);
      if (sel_bias) v = __fadd_rn(v, sel_bias[e]);
    }
    return v;
  };
  auto margin_of = [&](int e, float v) {
    const float ml = xm * wnorm[e] + (splits > 1 ? am * row_a[e] : 0.0f);
    // sigmoid' <= 1/4, plus its own last-bit error; either way the bias
    // addition's rounding (two units of the key's last place)
    return (sigmoid ? 0.25f * ml + 0x1p-20f : ml) + 0x1p-22f * fabsf(v);
  };
  uint64_t key[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = i * 32 + lane;
    key[i] = (e < E) ? ((uint64_t)float_order_key(value_of(e, logit_of(e))) << 32) |
                           (uint64_t)(0xFFFFFFFFu - e)
                     : 0;
  }
  // Experts in approximate order: lane j holds the j-th (value, margin, logit,
  // index).  Every expert whose value key reaches the (k + 1)-th largest of
  // the 32 lanes' best -- at least k + 1 experts, seldom more than 32 -- comes
  // out at once, compacted one per lane and sorted by a bitonic network.
  // More follow, one at a time, only while no cut at or past position k - 1
  // is proven (below); past 32 candidates all of them come out that way.
  float my_v = 0.0f, my_m = 0.0f, my_l = 0.0f;
  int my_e = 0;
  const int n_max = E < 32 ? E : 32;
  const int nsel = k < n_max ? k + 1 : n_max;
  int n = 0;
  {
    uint32_t lm = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) lm = max(lm, (uint32_t)(key[i] >> 32));
    const uint32_t theta = __shfl_sync(0xffffffffu, warp_sort_desc(lm, lane), nsel - 1);
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) cnt += (key[i] != 0 && (uint32_t)(key[i] >> 32) >= theta);
    const int total = __reduce_add_sync(0xffffffffu, cnt);
    if (total <= 32) {
      int off = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, off, o);
        if (lane >= o) off += u;
      }
      off -= cnt;
      uint64_t* slot = s_cand[threadIdx.x >> 5];
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (key[i] != 0 && (uint32_t)(key[i] >> 32) >= theta) {
          slot[off++] = key[i];
          key[i] = 0;
        }
      __syncwarp();
      const uint64_t c = warp_sort_desc(lane < total ? slot[lane] : (uint64_t)0, lane);
      n = total;
      if (lane < n) {
        my_e = (int)(0xFFFFFFFFu - (uint32_t)(c & 0xFFFFFFFFu));
        my_l = logit_of(my_e);
        my_v = value_of(my_e, my_l);
        my_m = margin_of(my_e, my_v);
      }
    }
  }
  int target = n > nsel ? n : nsel;
  int b = -1;         // the first proven cut at or past position k - 1
  unsigned cuts = 0;  // bit j: positions 0..j are, in truth, the j + 1 best
  float pl = 0.0f;    // min of the lower bounds v - m over positions 0..lane
  for (;;) {
    for (; n < target; ++n) {
      uint64_t best = 0;
#pragma unroll
      for (int i = 0; i < VPL; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
      }
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (key[i] == best) key[i] = 0;  // the owner drops the winner
      if (lane == n) {
        my_e = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFu));
        my_l = logit_of(my_e);
        my_v = value_of(my_e, my_l);
        my_m = margin_of(my_e, my_v);
      }
    }
    // the largest upper bound v + m among the experts not taken out
    float tail_u = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (key[i] != 0) {
        const float v = key_value(key[i]);
        tail_u = fmaxf(tail_u, v + margin_of(i * 32 + lane, v));
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tail_u = fmaxf(tail_u, __shfl_xor_sync(0xffffffffu, tail_u, o));
    // A cut after position j is proven when every lower bound up to j lies
    // above every upper bound after it (those of the experts not taken out
    // included): true values then keep positions 0..j above all others.
    pl = lane < n ? my_v - my_m : INFINITY;
    float su = lane < n ? my_v + my_m : -INFINITY;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float lo = __shfl_up_sync(0xffffffffu, pl, o);
      const float hi = __shfl_down_sync(0xffffffffu, su, o);
      if (lane >= o) pl = fminf(pl, lo);
      if (lane + o < 32) su = fmaxf(su, hi);
    }
    float su_next = __shfl_down_sync(0xffffffffu, su, 1);
    if (lane == 31) su_next = -INFINITY;
    su_next = fmaxf(su_next, tail_u);
    cuts = __ballot_sync(0xffffffffu, lane < n && pl > su_next);
    const unsigned late = cuts >> (k - 1);
    if (late) {
      b = k - 2 + __ffs(late);
      break;
    }
    if (n >= n_max) break;
    target = n + 1;
  }
  const uint16_t* xr = x + (size_t)t * H;
  if (b >= 0) {
    // Between two cuts the approximate order proves nothing: every run of two
    // or more positions up to b gets canonical keys and is sorted by them.
    const unsigned below = cuts & ((1u << lane) - 1u);
    const int start = below ? 32 - __clz(below) : 0;
    const unsigned from = lane == 0 ? cuts : cuts & ~((1u << lane) - 1u);
    const int end = from ? __ffs(from) - 1 : 31;
    const unsigned redo = __ballot_sync(0xffffffffu, lane <= b && end > start);
    if (redo) {
      // the rows the recompute streams, into L2 first: x[t] (mostly evicted
      // since the GEMM read it) and the undecided experts' router rows
      if (lane == 0) prefetch_l2(xr, (uint32_t)H * 2);
      if ((redo >> lane) & 1u) prefetch_l2(wr + (size_t)my_e * H, (uint32_t)H * 4);
      uint64_t ck = 0;
      unsigned todo = redo;
      while (todo) {  // up to four canonical logits per pass over x
        int pos[4], ex[4], c = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          pos[q] = todo ? __ffs(todo) - 1 : -1;
          if (todo) {
            todo &= todo - 1u;
            ++c;
          }
          ex[q] = __shfl_sync(0xffffffffu, my_e, pos[q] < 0 ? pos[0] : pos[q]);
        }
        float cl[4];
        canonical_logits4(xr, wr + (size_t)ex[0] * H, wr + (size_t)ex[1] * H,
                          wr + (size_t)ex[2] * H, wr + (size_t)ex[3] * H, H, lane, cl);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q < c && lane == pos[q]) {
            float l = cl[q];
            if (logit_bias) l = __fadd_rn(l, logit_bias[ex[q]]);
            float v = l;
            if (sigmoid) {
              v = sigmoid_fixed(l);
              if (sel_bias) v = __fadd_rn(v, sel_bias[ex[q]]);
            }
            my_l = l;
            ck = ((uint64_t)float_order_key(v) << 32) | (uint64_t)(0xFFFFFFFFu - ex[q]);
          }
        }
      }
      // rank within the run, then move every lane to its place
      int rank = 0;
      for (int i = 0; i <= b; ++i) {
        const uint64_t ki = __shfl_sync(0xffffffffu, ck, i);
        const int si = __shfl_sync(0xffffffffu, start, i);
        if (si == start && ki > ck) ++rank;
      }
      const int dest = lane <= b ? start + rank : lane;
      int src = lane;
      for (int i = 0; i <= b; ++i)
        if (__shfl_sync(0xffffffffu, dest, i) == lane) src = i;
      my_e = __shfl_sync(0xffffffffu, my_e, src);
      my_l = __shfl_sync(0xffffffffu, my_l, src);
    }
  } else {
    // No cut within 32 positions: the canonical keys of every expert whose
    // upper bound reaches the least lower bound of the first k, sorted by
    // insertion into lanes 0..k-1.
    const float floor_v = __shfl_sync(0xffffffffu, pl, k - 1);
    uint64_t top = 0;  // lane j < k: the j-th best canonical key so far
    float top_l = 0.0f;
    // the 32 taken out (lane j: position j), then the rest in index order
#pragma unroll
    for (int i = -1; i < VPL; ++i) {
      bool c;
      if (i < 0) {
        c = lane < n && !(my_v + my_m < floor_v);  // a NaN bound keeps the expert
      } else {
        const int e0 = i * 32 + lane;
        const float v = key_value(key[i]);
        c = key[i] != 0 && !(v + margin_of(e0, v) < floor_v);
      }
      unsigned cand = __ballot_sync(0xffffffffu, c);
      while (cand) {
        const int bb = __ffs(cand) - 1;
        cand &= cand - 1u;
        const int e = i < 0 ? __shfl_sync(0xffffffffu, my_e, bb) : i * 32 + bb;
        float l = canonical_logit(xr, wr + (size_t)e * H, H, lane);
        if (logit_bias) l = __fadd_rn(l, logit_bias[e]);
        float v = l;
        if (sigmoid) {
          v = sigmoid_fixed(l);
          if (sel_bias) v = __fadd_rn(v, sel_bias[e]);
        }
        const uint64_t ck = ((uint64_t)float_order_key(v) << 32) | (uint64_t)(0xFFFFFFFFu - e);
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
  const auto enc = tensor_map_encoder();
  if (!enc) return false;
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
                             float* xnorm, float* wnorm, float* approx, int splits, int* err,
                             cudaStream_t s) {
  if (T <= 0 || H % 64 || E <= 0 || E > 1024) return cudaErrorInvalidValue;
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(wr) % 16 ||
      reinterpret_cast<uintptr_t>(wp) % 16)
    return cudaErrorInvalidValue;  // the prep kernel's vector loads and stores
  count_launch();
  cudaError_t e = launch_kernel(router_prep_kernel, dim3(E + (T + 7) / 8), dim3(256), 0, s, 1,
                                static_cast<const uint16_t*>(x), wr, wp, xnorm, wnorm, T, H, E);
  if (e != cudaSuccess) return e;
  e = launch_dense_bf16_f32(x, H, wp, 3 * H, T, E, approx, splits, err, s);  // counts itself
  if (e != cudaSuccess) return e;
  if (splits > 1) {
    const size_t n = (size_t)T * E;
    count_launch();
    e = launch_kernel(router_sum_splits_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s,
                      1, approx, n, splits);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_topk_tc(const float* approx, int splits, const float* logit_bias,
                           const float* sel_bias, int sigmoid, const void* x, const float* wr,
                           const float* xnorm, const float* wnorm, int32_t* idx, float* w, int T,
                           int H, int E, int k, cudaStream_t s) {
  if (T <= 0 || E <= 0 || E > 1024 || k > 32 || k > E || splits < 1) return cudaErrorInvalidValue;
  const size_t stride = (size_t)T * E;
  const long blocks = ((long)T * 32 + TOPK_TC_THREADS - 1) / TOPK_TC_THREADS;
  if (blocks > 0x7FFFFFFFL) return cudaErrorInvalidValue;
  const int vpl = (E + 31) / 32;
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  count_launch();
  cudaError_t e;
#define MOE_TOPK_TC(V)                                                                      \
  launch_kernel(topk_tc_kernel<V>, dim3((unsigned)blocks), dim3(TOPK_TC_THREADS), 0, s, 1, \
                approx, splits, stride, logit_bias, sel_bias, sigmoid, xb, wr, xnorm, wnorm, idx,  \
                w, T, H, E, k)
  if (vpl <= 1) e = MOE_TOPK_TC(1);
  else if (vpl <= 2) e = MOE_TOPK_TC(2);
  else if (vpl <= 4) e = MOE_TOPK_TC(4);
  else if (vpl <= 8) e = MOE_TOPK_TC(8);
  else if (vpl <= 16) e = MOE_TOPK_TC(16);
  else if (vpl <= 28) e = MOE_TOPK_TC(28);  // E <= 896
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
