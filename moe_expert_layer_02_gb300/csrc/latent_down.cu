// latent_down.cu -- the LatentMoE down projection z = bf16(x Wd^T), rounded
// exactly ("Kimi K3 ... feasibility analysis", s.2.4: routed_expert_down_proj
// maps the hidden x [T, H] to the latent [T, L] on which the routed experts
// run).  x [T, H] and Wd [L, H] are bf16; z [T, L] is the nearest-even bf16 of
// the exact dot product.
//
// Why exactly.  z is quantised per token to fp8 before the experts.  A z that
// is one bf16 ulp off moves an e4m3 code now and then, and one moved code
// perturbs h of every routed row of the token by ~0.1%, which shifts the bf16
// rounding of some rows' amax and so their whole per-row fp8 requantisation.
// A single tensor-core accumulation over K = 7168 misses the exactly rounded
// bf16 in 0.4% of the elements (measured on a GB300; the share grows linearly
// with K, 0.06% at K = 1024, so the accumulation error is systematic, not a
// random walk), and through that cascade 7.6% of LatentMoE tokens ended more
// than 5% of the output RMS away from the exact layer.
//
// How.
//  1. latent_down_kernel: a GEMM on SM pairs (tcgen05.mma cta_group::2,
//     kind::f16, bf16 operands, fp32 accumulation in tensor memory).  A tile is
//     256 token rows (128 per CTA) x 256 latent features (128 weight rows
//     staged per CTA).  The accumulation restarts every kChunkStages K stages
//     (128 K, eight MMAs) in the other of two tensor-memory buffers, and eight
//     epilogue warps (two per lane quarter, 128 columns each) add every chunk's
//     partial sums into registers: S in fp32 (the dot product) and Q in bf16
//     (the sum of the partials' squares, which scales the remaining error:
//     the chunks' rounding errors add like independent terms of their size).
//     Short accumulations keep the tensor core's own error ~30x smaller than
//     one long one (0.014% of roundings off instead of 0.40%).  At the tile's
//     end each element is rounded to bf16 from S and flagged when a bf16
//     rounding boundary lies within MOE_ZFLAG_ULPS * 2^-23 * sqrt(Q) of S:
//     only there can the remaining error change the rounding.
//  2. latent_fix_kernel: one block per token recomputes every flagged element
//     on the CUDA cores in two-fp32 arithmetic -- a product of two bf16 values
//     is exact in fp32, and TwoSum keeps every addition's rounding error -- and
//     rounds the unevaluated sum hi + lo to nearest-even bf16.
//
// Pipeline and waits follow ffn_gemm_2cta.cu: warp 0 TMA producer, warp 1 MMA
// issuer (even CTA), warps 4-11 epilogue; both CTAs' loads complete on the even
// CTA's `full` barriers; commits multicast to both CTAs; the epilogues hand a
// buffer back on the even CTA's `tempty` barrier.  Every wait is bounded.
#include <cudaTypedefs.h>

#include <algorithm>

#include "device.cuh"
#include "internal.h"

// Margin of the flag test in units of 2^-23 * sqrt(Q), Q = the sum of the
// squared chunk partials.  Calibrated on a GB300 at the LatentMoE shape (x
// [4096, 7168] N(0,1), Wd N(0, 1/7168), 14.7 M elements; margin -> share
// flagged, elements whose bf16 rounding still differed from the exact one):
// 0 -> 0.003%, 2013; 4 -> 0.14%, 2; 6 -> 0.20%, 1; 8 -> 0.26%, 0; 12 -> 0.37%,
// 0; 16 -> 0.48%, 0.  Twelve leaves a factor 1.5 over the first margin without
// a miss and 2 over the last with one; a larger margin only sends more
// elements to the exact recomputation.  (A margin from the sum of the
// partials' magnitudes needed 0.41% flagged for its first zero.)
#ifndef MOE_ZFLAG_ULPS
#define MOE_ZFLAG_ULPS 12.0f
#endif

namespace moe {

namespace {

constexpr int LD_ROWS = 128;            // token rows per CTA (M = 256 per pair)
constexpr int LD_BK = 128;              // K bytes per stage (64 bf16)
constexpr int LD_EL = LD_BK / 2;        // K elements per stage
constexpr int LD_UMMA_B = 32;           // K bytes per tcgen05.mma (16 bf16)
constexpr int LD_A_BYTES = LD_ROWS * LD_BK;  // 16 KB
constexpr int kChunkStages = 2;         // K stages per tensor-core accumulation
constexpr int LD_EPI_WARPS = 8;         // two per tensor-memory lane quarter

// Tiles of N = 256 latent features (128 weight rows staged per CTA), two
// partial-sum buffers filling the 512 tensor-memory columns, twelve warps:
// warp 0 loads, warp 1 issues the MMAs, warps 2-3 idle, warps 4-11 add the
// partials, 128 columns each.  The first warp group gives its registers up
// (setmaxnreg) so that the epilogue threads can hold 128 fp32 sums and 64 bf16
// pairs of squares.  x is read from L2 L/256 times, and a K stage moves 32 KB into each
// SM's shared memory per 2.1 M multiply-adds.  (A first version with 128-wide
// tiles and ten warps, within the 168 registers a thread gets when three warps
// share a scheduler, read x twice as often and moved 24 KB per 1.05 M
// multiply-adds: 0.30 ms at the LatentMoE shape, tensor pipe 31% busy.)
template <int N>
struct LdCfg {
  static_assert(N == 256, "the register split below is laid out for 256-wide tiles");
  static constexpr int WIDE = 1;
  static constexpr int WARPS = 12;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int EPI0 = 4;             // first epilogue warp
  static constexpr int COLS = N / 2;         // columns per epilogue thread
  static constexpr int BUFS = 512 / N;
  static constexpr int B_BYTES = (N / 2) * LD_BK;
  static constexpr int STAGE = LD_A_BYTES + B_BYTES;
  static constexpr int STAGES = 6;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * BUFS + 1;
  static constexpr int SMEM = 1024 + STAGES * STAGE + NUM_BARS * 8 + 16 + STAGES * 4;
  // the wide kernel's register split: launched at 168 a thread (384 x 168 =
  // 64512), the first warp group drops to 40 and the two epilogue groups rise
  // to 232 (4 x 32 x 40 + 8 x 32 x 232 = 64512)
  static constexpr int LAUNCH_REGS = 168, LOW_REGS = 40, HIGH_REGS = 232;
};

struct LatentDown {
  int T, H, L;
  void* z;           // [T, L] bf16
  uint32_t* flags;   // [T, L / 32]: bit j of word w = element (t, 32 w + j) needs recomputing
  int* err;
};

// f32 accumulate (bits 4-5 = 1), bf16 A and B (kind::f16 format 1 at bits 7-9
// and 10-12), both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
template <int N>
__device__ __forceinline__ uint32_t ld_idesc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)((2 * LD_ROWS) >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// Two fp32 additions in one instruction (round to nearest, as two adds).
__device__ __forceinline__ void add_f32x2(uint64_t& acc, uint32_t lo, uint32_t hi) {
  asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%1, %2};\n\tadd.rn.f32x2 %0, %0, t;\n\t}"
      : "+l"(acc)
      : "r"(lo), "r"(hi));
}

// acc (two bf16) += (lo^2, hi^2), with lo and hi rounded to bf16 first.
__device__ __forceinline__ uint32_t add_sq_bf16x2(uint32_t acc, uint32_t lo, uint32_t hi) {
  uint32_t r;
  asm("{\n\t.reg .b32 t;\n\tcvt.rn.bf16x2.f32 t, %2, %1;\n\t"
      "fma.rn.bf16x2 %0, t, t, %3;\n\t}"
      : "=r"(r)
      : "r"(lo), "r"(hi), "r"(acc));
  return r;
}

template <int R>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}

// True when rounding s to bf16 may differ from rounding the exact value, given
// |exact - s| <= margin.  The bf16 rounding boundaries of |s| in [lo, lo + ulp)
// are lo - ulp/2 (or lo - ulp/4 when lo is a power of two) and lo + ulp/2.
__device__ __forceinline__ bool near_bf16_boundary(float s, float margin) {
  const uint32_t u = __float_as_uint(s) & 0x7FFFFFFFu;
  const uint32_t e = u >> 23;
  if (e <= 8u) return margin > 0.0f;  // |s| < 2^-118 (or zero): recompute
  const float ulp = __uint_as_float((e - 7u) << 23);        // bf16 ulp at |s|
  const float mid = __uint_as_float((u & 0xFFFF0000u) | 0x8000u);
  return margin >= 0.25f * ulp || fabsf(__uint_as_float(u) - mid) <= margin;
}

template <int N>
__global__ void __launch_bounds__(LdCfg<N>::THREADS, 1)
    latent_down_kernel(const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_w, const LatentDown g) {
  using C = LdCfg<N>;
  constexpr int COLS = C::COLS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tfull = bars + 2 * C::STAGES;
  uint64_t* tempty = tfull + C::BUFS;
  uint64_t* drain = tempty + C::BUFS;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint32_t* s_issued = s_tmem + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
      s_issued[s] = 0;
    }
    for (int b = 0; b < C::BUFS; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 2 * LD_EPI_WARPS);  // the epilogue warps of both CTAs
    }
    mbar_init(smem_u32(drain), 1);
    *s_abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(s_tmem), 512);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_wait();

  const int n_rt = (g.T + 2 * LD_ROWS - 1) / (2 * LD_ROWS);
  const int n_ct = g.L / N;
  const int n_tiles = n_rt * n_ct;
  const int KB = g.H / LD_EL;               // K stages per tile
  const int NCH = KB / kChunkStages;        // chunks per tile
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;

  if (warp < C::EPI0) {
    // the first warp group (all four warps together) hands registers over
    if (C::WIDE) regs_dec<C::LOW_REGS>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = cluster; tile < n_tiles && ok && !*s_abort; tile += n_clusters) {
        const int rt = tile / n_ct, ct = tile - rt * n_ct;
        const int row0 = rt * 2 * LD_ROWS + LD_ROWS * (int)rank;
        const int wrow0 = ct * N + (N / 2) * (int)rank;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, g.err, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t st = smem_u32(smem + stage * C::STAGE);
          const uint32_t fb_leader = mapa_shared(smem_u32(&full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(smem_u32(&full[stage]), 2 * C::STAGE);
          tma_load_2d_pair(st, &tm_x, kb * LD_EL, row0, fb_leader);
          tma_load_2d_pair(st + LD_A_BYTES, &tm_w, kb * LD_EL, wrow0, fb_leader);
          s_issued[stage] = phase + 1u;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*s_abort && leader) {  // the pair's loads complete on the even CTA's barriers
        for (int s = 0; s < C::STAGES; ++s)
          if (s_issued[s]) mbar_wait_drain(smem_u32(&full[s]), s_issued[s] - 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      int stage = 0, chunk = 0;
      uint32_t phase = 0;
      bool issued_any = false, ok = true;
      const uint32_t idesc = ld_idesc<N>();
      for (int tile = cluster; tile < n_tiles && ok && !*s_abort; tile += n_clusters) {
        for (int c = 0; c < NCH && ok; ++c, ++chunk) {
          const int buf = chunk % C::BUFS;
          const uint32_t bphase = (uint32_t)(chunk / C::BUFS) & 1u;
          if (!mbar_wait(smem_u32(&tempty[buf]), bphase ^ 1u, g.err, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + buf * N;
          for (int s = 0; s < kChunkStages; ++s) {
            if (!mbar_wait(smem_u32(&full[stage]), phase, g.err, s_abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(smem + stage * C::STAGE);
            const uint32_t b0 = a0 + LD_A_BYTES;
#pragma unroll
            for (int kk = 0; kk < LD_BK / LD_UMMA_B; ++kk)
              mma_bf16_pair(d, smem_desc_sw128(a0 + kk * LD_UMMA_B),
                            smem_desc_sw128(b0 + kk * LD_UMMA_B), idesc, (s | kk) ? 1u : 0u);
            issued_any = true;
            mma_commit_pair(smem_u32(&empty[stage]), 0x3);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) mma_commit_pair(smem_u32(&tfull[buf]), 0x3);
        }
      }
      if (*s_abort && issued_any) {
        mma_commit_pair(smem_u32(drain), 0x1);
        mbar_wait_drain(smem_u32(drain), 0);
      }
    }
  }
  } else {
    // ------------------------------------------------------------ epilogue
    if (C::WIDE) regs_inc<C::HIGH_REGS>();
    const int ew = warp - C::EPI0;
    const int q = warp & 3;          // tensor-memory lane quarter this warp may read
    const int half = ew >> 2;        // which half of the tile's columns
    const uint32_t tempty_leader0 = mapa_shared(smem_u32(&tempty[0]), 0);
    int chunk = 0;
    bool ok = true;
    for (int tile = cluster; tile < n_tiles && ok; tile += n_clusters) {
      const int rt = tile / n_ct, ct = tile - rt * n_ct;
      uint64_t S[COLS / 2];  // fp32 sums of columns 2j, 2j + 1
      uint32_t Q[COLS / 2];  // bf16 sums of partial^2 (only a margin: 8 bits suffice)
#pragma unroll
      for (int j = 0; j < COLS / 2; ++j) {
        S[j] = 0ull;
        Q[j] = 0u;
      }
      for (int c = 0; c < NCH; ++c, ++chunk) {
        const int buf = chunk % C::BUFS;
        const uint32_t bphase = (uint32_t)(chunk / C::BUFS) & 1u;
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait(smem_u32(&tfull[buf]), bphase, g.err, s_abort) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + buf * N + half * COLS;
        // 32 columns per wait (registers are the limit); the buffer goes back
        // once the last group has landed
#pragma unroll
        for (int r = 0; r < COLS / 32; ++r) {
          uint32_t v[32];
          tmem_ld16(tb + 32 * r, *reinterpret_cast<uint32_t(*)[16]>(v));
          tmem_ld16(tb + 32 * r + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
          tmem_ld_wait();
          if (r == COLS / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader0 + buf * 8);
          }
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            add_f32x2(S[16 * r + (j >> 1)], v[j], v[j + 1]);
            Q[16 * r + (j >> 1)] = add_sq_bf16x2(Q[16 * r + (j >> 1)], v[j], v[j + 1]);
          }
        }
      }
      if (!ok) break;
      const int row = rt * 2 * LD_ROWS + LD_ROWS * (int)rank + q * 32 + lane;
      if (row < g.T) {
        const int col0 = ct * N + half * COLS;
        uint32_t fw[COLS / 32];
#pragma unroll
        for (int i = 0; i < COLS / 32; ++i) fw[i] = 0u;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(g.z) + (size_t)row * g.L + col0);
#pragma unroll
        for (int j0 = 0; j0 < COLS; j0 += 8) {
          uint32_t pk[4];
#pragma unroll
          for (int j = j0; j < j0 + 8; j += 2) {
            // margin from the partials' root sum of squares (the chunks'
            // rounding errors add like independent terms of their size)
            const float m0 = (MOE_ZFLAG_ULPS * 0x1p-23f) * sqrtf(__uint_as_float(Q[j >> 1] << 16));
            const float m1 =
                (MOE_ZFLAG_ULPS * 0x1p-23f) * sqrtf(__uint_as_float(Q[j >> 1] & 0xFFFF0000u));
            float s0, s1;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(S[j >> 1]));
            if (near_bf16_boundary(s0, m0)) fw[j >> 5] |= 1u << (j & 31);
            if (near_bf16_boundary(s1, m1)) fw[(j + 1) >> 5] |= 1u << ((j + 1) & 31);
            __nv_bfloat162 b = __floats2bfloat162_rn(s0, s1);
            pk[(j - j0) >> 1] = *reinterpret_cast<uint32_t*>(&b);
          }
          dst[j0 / 8] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        uint32_t* fdst = g.flags + (size_t)row * (g.L / 32) + col0 / 32;
#pragma unroll
        for (int i = 0; i < COLS / 32; ++i) fdst[i] = fw[i];
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while its peer may still signal it
  pdl_release();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// ---------------------------------------------------------------- exact fixup
// s + e == a + b exactly (Knuth's TwoSum; no ordering of |a|, |b| needed).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float aa = __fsub_rn(s, bb);
  e = __fadd_rn(__fsub_rn(a, aa), __fsub_rn(b, bb));
}

// Packed pairs of fp32 (.x in the low word): two independent IEEE
// round-to-nearest operations per instruction.
__device__ __forceinline__ uint64_t f2_pack(uint32_t x, uint32_t y) {
  return (uint64_t)x | ((uint64_t)y << 32);
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Nearest-even bf16 of the exact value hi + lo, where (hi, lo) = TwoSum output
// (|lo| <= ulp(hi) / 2).  Every bf16 rounding boundary is an fp32 value, so
// hi + lo lies on hi's side of it unless hi is the boundary itself; then lo's
// sign decides, and lo == 0 is an exact tie (to even).
__device__ __forceinline__ uint16_t bf16_of_sum(float hi, float lo) {
  const uint32_t u = __float_as_uint(hi);
  uint32_t r = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;  // nearest-even of hi
  if ((u & 0xFFFFu) == 0x8000u && lo != 0.0f) {
    const bool up_mag = (lo > 0.0f) == (hi > 0.0f);  // |hi + lo| beyond the midpoint
    r = up_mag ? (u >> 16) + 1u : (u >> 16);
  }
  return (uint16_t)r;
}

constexpr int FX_THREADS = 256;
constexpr int FX_SMEM_MAX = 160 * 1024;  // x row (bf16) + flagged-column list: 2 H + 2 L bytes
constexpr int FX_AHEAD = 8;              // 16-byte weight loads a lane issues ahead of its sums

// One block per token: x[t] goes to shared memory (bf16), then each warp
// takes flagged elements in turn.  Lane j sums the products of columns
// 8 (j + 32 m) .. 8 (j + 32 m) + 7 (m ascending) with TwoSum in two chains,
// even and odd columns, run as packed fp32 pairs (six instructions per
// product instead of ten, though the fp32 pipe does the same work: T=4096,
// H=7168, L=3584, 0.5% of z flagged: 152 -> 130 us); the lane joins its
// chains and the warp combines the lanes' (hi, lo) pairs.
__global__ void __launch_bounds__(FX_THREADS)
    latent_fix_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wd,
                      uint16_t* __restrict__ z, const uint32_t* __restrict__ flags, int T, int H,
                      int L) {
  extern __shared__ uint4 fx_smem[];
  uint16_t* list = reinterpret_cast<uint16_t*>(fx_smem + H / 8);  // flagged columns of this token
  __shared__ int n_list;
  pdl_wait();
  const int t = blockIdx.x;
  if (t >= T) return;
  const int W = L / 32;
  if (threadIdx.x == 0) n_list = 0;
  __syncthreads();
  for (int w = threadIdx.x; w < W; w += FX_THREADS) {
    uint32_t bits = flags[(size_t)t * W + w];
    while (bits) {
      const int j = __ffs(bits) - 1;
      bits &= bits - 1u;
      list[atomicAdd(&n_list, 1)] = (uint16_t)(32 * w + j);
    }
  }
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  for (int i = threadIdx.x; i < H / 8; i += FX_THREADS) fx_smem[i] = xr[i];
  __syncthreads();
  const int n = n_list;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C8 = H / 8;  // 16-byte chunks of a row
  for (int i = warp; i < n; i += FX_THREADS / 32) {
    const int l = list[i];
    const uint4* wr = reinterpret_cast<const uint4*>(wd + (size_t)l * H);
    // Two TwoSum chains per lane in packed pairs: .x takes the even products
    // (the low bf16 of every word), .y the odd ones; the lane's chunks
    // c = lane + 32 m in ascending m, FX_AHEAD weight loads in flight before
    // the sums that need them.
    uint64_t hi2 = 0, lo2 = 0;
    for (int c0 = lane; c0 < C8; c0 += 32 * FX_AHEAD) {
      uint4 wv[FX_AHEAD];
#pragma unroll
      for (int u = 0; u < FX_AHEAD; ++u)
        wv[u] = c0 + 32 * u < C8 ? __ldg(wr + c0 + 32 * u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < FX_AHEAD; ++u) {
        if (c0 + 32 * u >= C8) break;
        const uint4 xv = fx_smem[c0 + 32 * u];
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t ww[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          // products of bf16 values: 16 significant bits, exact in fp32
          const uint64_t p = f2_mul(f2_pack(xw[q] << 16, xw[q] & 0xFFFF0000u),
                                    f2_pack(ww[q] << 16, ww[q] & 0xFFFF0000u));
          const uint64_t sm = f2_add(hi2, p);  // TwoSum(hi2, p), both halves at once
          const uint64_t bb = f2_sub(sm, hi2);
          const uint64_t aa = f2_sub(sm, bb);
          lo2 = f2_add(lo2, f2_add(f2_sub(hi2, aa), f2_sub(p, bb)));
          hi2 = sm;
        }
      }
    }
    float hi, lo;
    {
      float sm, e;
      two_sum(__uint_as_float((uint32_t)hi2), __uint_as_float((uint32_t)(hi2 >> 32)), sm, e);
      hi = sm;
      lo = __fadd_rn(__fadd_rn(__uint_as_float((uint32_t)lo2), __uint_as_float((uint32_t)(lo2 >> 32))),
                     e);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
      const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
      float sm, e;
      two_sum(hi, h2, sm, e);
      hi = sm;
      lo = __fadd_rn(__fadd_rn(lo, l2), e);
    }
    if (lane == 0) {
      float sm, e;
      two_sum(hi, lo, sm, e);  // renormalise: |e| <= ulp(sm) / 2
      z[(size_t)t * L + l] = bf16_of_sum(sm, e);
    }
  }
  pdl_release();
}

bool ld_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  const auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)LD_EL, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// True when the kernel was built with exactly the per-thread register count
// its setmaxnreg split assumes: a block launched with fewer registers could
// never complete the split.
bool wide_kernel_usable() {
  static const bool ok = [] {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, latent_down_kernel<256>) == cudaSuccess &&
           fa.numRegs == LdCfg<256>::LAUNCH_REGS;
  }();
  return ok;
}

template <int N>
cudaError_t launch_down_gemm(const void* x, const void* wd, const LatentDown& g, cudaStream_t s) {
  using C = LdCfg<N>;
  CUtensorMap tx, tw;
  if (!ld_map(&tx, x, g.H, g.T, LD_ROWS) || !ld_map(&tw, wd, g.H, g.L, N / 2))
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_max_smem<latent_down_kernel<N>>(C::SMEM);
  if (e != cudaSuccess) return e;
  const int tiles = ((g.T + 2 * LD_ROWS - 1) / (2 * LD_ROWS)) * (g.L / N);
  const int clusters = std::min(device_sm_count() / 2, tiles);
  count_launch();
  return launch_kernel(latent_down_kernel<N>, dim3(2 * clusters), dim3(C::THREADS), C::SMEM, s,
                       2, tx, tw, g);
}

}  // namespace

size_t latent_down_flag_bytes(int T, int L) { return (size_t)T * (L / 32) * 4; }

cudaError_t launch_latent_down(const void* x, const void* wd, void* z, uint32_t* flags, int T,
                               int H, int L, int* err, cudaStream_t s) {
  if (T <= 0 || H % (LD_EL * kChunkStages) || L % 128 || !flags) return cudaErrorInvalidValue;
  LatentDown g{T, H, L, z, flags, err};
  // never launch a register split the build cannot complete (it would wait forever)
  if (L % 256 || !wide_kernel_usable()) return cudaErrorInvalidDeviceFunction;
  cudaError_t e = launch_down_gemm<256>(x, wd, g, s);
  if (e != cudaSuccess) return e;
  const size_t fx_smem = (size_t)H * 2 + (size_t)L * 2;
  if (fx_smem > (size_t)FX_SMEM_MAX) return cudaErrorInvalidValue;
  e = ensure_max_smem<latent_fix_kernel>(FX_SMEM_MAX);
  if (e != cudaSuccess) return e;
  count_launch();
  e = launch_kernel(latent_fix_kernel, dim3(T), dim3(FX_THREADS), fx_smem, s, 1,
                    static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(wd),
                    static_cast<uint16_t*>(z), static_cast<const uint32_t*>(flags), T, H, L);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
