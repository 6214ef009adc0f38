// ffn_gemm.cu -- S5/S6: grouped fp8 SwiGLU expert GEMMs on tcgen05.
//
// What is computed ("Optimising Ling-2.6-1T on TPU with SGLang-JAX", s.1 cost
// model FFN1/FFN2 and s.5 "per-channel direct_scaled_dot"): for each routed
// row r of expert e,
//   FFN1  g[n] = (sum_k xq[r,k] W1_e[n,k]) * xs[r] * s13_e[n]
//         u[n] = (sum_k xq[r,k] W3_e[n,k]) * xs[r] * s13_e[I+n]
//         h[r,n] = bf16(silu(g) * u)
//   FFN2  y[r,m] = bf16(row_w[r] * (sum_n hq[r,n] W2_e[m,n]) * hs[r] * s2_e[m])
// e4m3 x e4m3 products are summed in fp32 by the tensor core over the full K;
// the per-token and per-channel scales are applied after the reduction, which
// is what makes one long-K contraction possible (the write-up contrasts this
// with block-wise scales that force K into short pieces).
//
// How (GB300-specific; the TPU kernel of the write-up is prior art only):
//   * Work list: items {group, row0, rows<=BN} over expert-contiguous rows
//     (group E = the shared expert, whose rows follow the routed ones); a tile
//     is (item, 128-wide output block).  One persistent CTA per SM walks tiles
//     blockIdx.x, +gridDim.x, ...
//   * Swap-AB: the MMA's M=128 runs over weight rows (output features) and N
//     over the item's token rows (N = rows rounded up to 16, <= BN), so decode
//     batches of ~16 rows per expert still issue full-height MMAs and every
//     weight byte is streamed once.  D[feature, row] lives in tensor memory.
//   * Warp roles: warp 0 = TMA producer (W tiles through a 3-D map
//     [E][rows][K], activation rows through a 2-D map, 128-byte swizzle),
//     warp 1 = MMA issuer (tcgen05.mma kind::f8f6f4, commit to mbarriers),
//     warps 2-5 = epilogue (tcgen05.ld, scales, SiLU*gate or routing weight,
//     bf16 stores).  A smem ring of at most four stages + double-buffered
//     accumulators (the write-up's "weight double-buffering" becomes this
//     ring; deeper rings streamed the weights more slowly).
//   * Block-wise fp8 weights (one fp32 scale per 128 x 128 block, the format
//     tpu-inference requires, "Kimi K3 ... feasibility analysis" s.3.7): the
//     scale changes every 128 K, so the K-sum cannot run in one accumulator.
//     With BLK the MMAs write each stage's partial sum into one of four (FFN1)
//     or eight (FFN2) tensor-memory buffers (restarted per stage), and the
//     epilogue warps add s[nb][kb] * partial into fp32 registers, stage by
//     stage, before applying
//     the per-token scale and the activation at the end of the tile (tiles of
//     at most 64 token rows, the registers' limit).
//   * Row gather (FFN1, opt-in): the activations arrive as one fp8 row per
//     token, and the producer warp's 32 lanes copy each tile's rows
//     (routed row r -> token src[r]) with 16-byte cp.async into the swizzled
//     layout; each lane's completion arrives on the stage's full barrier and
//     the MMA thread fences the generic proxy before reading the stage
//     ("Optimising Ling-2.6-1T ...", s.4: tokens gathered inside the kernel).
//   * Programmatic dependent launch: the producer issues the weight loads of
//     its first ring stages before griddepcontrol.wait, so the weight stream
//     starts while the previous kernel still runs.
//   * Every pipeline wait is bounded; on timeout the CTA records
//     MOE_ERR_TIMEOUT, drains its own TMA loads and MMAs and frees its tensor
//     memory before returning.
#include <cudaTypedefs.h>

#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int BM = 128;     // output features per tile (MMA M)
constexpr int BK = 128;     // K bytes per stage (= one 128-byte swizzle row)
constexpr int UMMA_K = 32;  // K per tcgen05.mma for 8-bit operands
constexpr int kThreads = 192;
constexpr int kSmemBudget = 221 * 1024;

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <bool FFN1, int BN, bool BLK>
struct Cfg {
  static constexpr int A_BYTES = BM * BK;  // one weight box, 16 KB
  // two 128-row weight blocks per stage sharing the activation tile: W1 and
  // W3 block nb (FFN1), W2 blocks 2nb and 2nb+1 (FFN2)
  static constexpr int NA = 2;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int STAGE_BYTES = NA * A_BYTES + B_BYTES;
  // At most four stages (32 KB of weights each) in flight: with five or six
  // the weight stream ran slower (T=512, H=8192, I=2048, E=256: FFN2 0.65 vs
  // 0.69 ms with 32-row tiles, FFN1 1.23 vs 1.26 ms with 64-row tiles;
  // block-wise scales, 32-row tiles: layer 2.07 ms with four stages, 2.12
  // with five, 2.20 with six), and with three slower again.
  static constexpr int STAGES = cmin(kSmemBudget / STAGE_BYTES, 4);
  static constexpr int ACC_COLS = NA * BN;
  // accumulators per tile, or (BLK) per-stage partial-sum buffers, so the MMAs
  // can run that many stages ahead of the warps that scale and add them: four
  // for FFN1's 32 KB stages, eight for FFN2's 16 KB ones (measured best)
  static constexpr int ACC_STAGES = BLK ? (FFN1 ? 4 : cmin(8, 512 / ACC_COLS))
                                        : (2 * ACC_COLS <= 512) ? 2 : 1;
  static constexpr int ACC_BUFS = ACC_STAGES;
  static constexpr int MAX_KB = 128;  // BLK: scale rows held in registers (K <= 16384)
  static_assert(!BLK || BN <= 64, "block-wise tiles keep their sums in registers");
  static constexpr int TMEM_COLS = pow2_at_least(ACC_BUFS * ACC_COLS);
  static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_STAGES + 1;
  // + the tile's token list (FFN1 row gather)
  static constexpr int SMEM =
      1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16 + STAGES * 4 + BN * 4;
  static_assert(B_BYTES % 1024 == 0, "operand tiles must keep 1024-byte alignment");
  static_assert(ACC_BUFS * ACC_COLS <= 512, "tensor memory holds 512 columns");
  static_assert(STAGES >= 2, "need at least two pipeline stages");
};

__device__ __forceinline__ uint32_t f32_bits_to_bf16(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

// Block-wise epilogue helpers.  Scale rows [.. / 128][KB] of a tile: W1 and W3
// block rows nb and I/128 + nb (FFN1), W2 block row nb (FFN2); lane l holds
// entries l, l+32, l+64, l+96 (KB <= 128).
constexpr int kHeld = 4;

// 128-row block index of weight block b (0, 1) of tile column nb.
template <bool FFN1>
__device__ __forceinline__ int wblock(const GroupedFfnArgs& a, int b, int nb) {
  return FFN1 ? (b == 0 ? nb : a.I / BM + nb) : 2 * nb + b;
}

template <bool FFN1>
__device__ __forceinline__ void load_block_scales(const GroupedFfnArgs& a, int item, int nb,
                                                  int KB, int lane, float (&held)[2][kHeld]) {
  constexpr int NA = 2;
  const int4 it = a.items[item];
  const bool shared = it.x >= a.E;
  const int wrow_blocks = FFN1 ? 2 * a.I / BM : a.K / BM;
  const float* sbase = FFN1 ? (shared ? a.sw13_scale : a.w13_scale + (size_t)it.x * wrow_blocks * KB)
                            : (shared ? a.sw2_scale : a.w2_scale + (size_t)it.x * wrow_blocks * KB);
#pragma unroll
  for (int b = 0; b < NA; ++b) {
    const int blk = wblock<FFN1>(a, b, nb);
    const float* srow = sbase + (size_t)blk * KB;
    const bool have = blk < wrow_blocks;  // FFN2 with K % 256 == 128: no second block
#pragma unroll
    for (int i = 0; i < kHeld; ++i) {
      const int kb = i * 32 + lane;
      held[b][i] = (have && kb < KB) ? __ldg(srow + kb) : 0.0f;
    }
  }
}

// Stage by stage, acc += s[kb] * partial; at the end of the tile the per-token
// scale, activation / routing weight and bf16 store.  The next tile's scale
// rows are loaded into held_next while this tile runs, and lane l loads the
// per-row scalars of rows l and l + 32 once, for the final pass to shuffle.
template <bool FFN1, int BN, int ACC_COLS, int PBUF>
__device__ __forceinline__ bool block_epilogue(const GroupedFfnArgs& a, uint32_t tmem, int q,
                                               int lane, int item, int nb, int KB,
                                               const float (&held)[2][kHeld],
                                               int next_item, int next_nb,
                                               float (&held_next)[2][kHeld],
                                               uint64_t* tfull, uint64_t* tempty,
                                               volatile int* s_abort, int& pcount) {
  constexpr int NA = 2;
  constexpr int RL = (BN + 31) / 32;  // rows per lane for the per-row scalars
  const int4 it = a.items[item];
  const bool shared = it.x >= a.E;
  const int row0 = it.y, rows = it.z;
  float rs[RL], rw[RL];  // xs (FFN1) or hs (FFN2), and the routing weight (FFN2)
#pragma unroll
  for (int i = 0; i < RL; ++i) {
    const int r = i * 32 + lane, row = row0 + r;
    const bool ok = r < rows && (unsigned)row < (unsigned)a.rows_total;
    rs[i] = ok ? (FFN1 ? a.xscale[row] : a.hs[row]) : 0.0f;
    rw[i] = (ok && !FFN1 && !shared && a.row_w) ? a.row_w[row] : 1.0f;
  }
  if (next_item >= 0) load_block_scales<FFN1>(a, next_item, next_nb, KB, lane, held_next);
  float acc[NA][BN];
#pragma unroll
  for (int b = 0; b < NA; ++b)
#pragma unroll
    for (int j = 0; j < BN; ++j) acc[b][j] = 0.0f;
  for (int kb = 0; kb < KB; ++kb, ++pcount) {
    const int pb = pcount % PBUF;
    const uint32_t ph = (uint32_t)(pcount / PBUF) & 1u;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_u32(&tfull[pb]), ph, a.err, s_abort) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) return false;
    tc_fence_after();
    float sk[NA];
#pragma unroll
    for (int b = 0; b < NA; ++b) {
      float v = held[b][0];
#pragma unroll
      for (int i = 1; i < kHeld; ++i) v = (kb >> 5) == i ? held[b][i] : v;
      sk[b] = __shfl_sync(0xffffffffu, v, kb & 31);
    }
    const uint32_t pbase = tmem + ((uint32_t)(q * 32) << 16) + pb * ACC_COLS;
#pragma unroll
    for (int c = 0; c < BN / 16; ++c) {
      if (c * 16 < rows) {  // warp-uniform
        uint32_t v[NA][16];
        __syncwarp();
#pragma unroll
        for (int b = 0; b < NA; ++b) tmem_ld16(pbase + b * BN + c * 16, v[b]);
        tmem_ld_wait();
#pragma unroll
        for (int b = 0; b < NA; ++b)
#pragma unroll
          for (int j = 0; j < 16; ++j)
            acc[b][c * 16 + j] = fmaf(sk[b], __uint_as_float(v[b][j]), acc[b][c * 16 + j]);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&tempty[pb]));
  }
  const int f = nb * BM + q * 32 + lane;        // FFN1: feature
  const int f2 = 2 * nb * BM + q * 32 + lane;   // FFN2: output channel of block 0
#pragma unroll
  for (int j = 0; j < BN; ++j) {
    const float sj = __shfl_sync(0xffffffffu, rs[j / 32], j % 32);
    const float wj = __shfl_sync(0xffffffffu, rw[j / 32], j % 32);
    const int row = row0 + j;
    if (j < rows && (unsigned)row < (unsigned)a.rows_total) {
      if (FFN1) {
        const float hv = gated_act(a.act, acc[0][j] * sj, acc[NA - 1][j] * sj);
        static_cast<uint16_t*>(a.h)[(size_t)row * a.I + f] = (uint16_t)f32_bits_to_bf16(hv);
      } else {  // output channels f (block 2nb) and f + 128 (block 2nb + 1)
        uint16_t* yr = static_cast<uint16_t*>(a.y) + (size_t)row * a.K;
        yr[f2] = (uint16_t)f32_bits_to_bf16((acc[0][j] * sj) * wj);
        if (f2 + BM < a.K) yr[f2 + BM] = (uint16_t)f32_bits_to_bf16((acc[1][j] * sj) * wj);
      }
    }
  }
  return true;
}

template <bool FFN1, int BN, bool BLK>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_ffn_kernel(const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_ws,
                       const __grid_constant__ CUtensorMap tm_x, const GroupedFfnArgs a) {
  using C = Cfg<FFN1, BN, BLK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tfull = bars + 2 * C::STAGES;
  uint64_t* tempty = tfull + C::ACC_STAGES;
  uint64_t* drain = tempty + C::ACC_STAGES;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint32_t* s_issued = s_tmem + 4;  // per stage: 0 = never, else phase + 1
  int* s_tok = reinterpret_cast<int*>(s_issued + C::STAGES);  // [BN] tokens of the tile's rows

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // FFN1 row gather: the producer warp's 32 lanes copy the activation rows, each
  // lane's cp.async completion arriving on the stage's full barrier
  const bool gat = FFN1 && !BLK && a.gather;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), gat ? 1 + 32 : 1);
      mbar_init(smem_u32(&empty[s]), 1);
      s_issued[s] = 0;
    }
    for (int s = 0; s < C::ACC_STAGES; ++s) {
      mbar_init(smem_u32(&tfull[s]), 1);
      mbar_init(smem_u32(&tempty[s]), 4);  // one arrive per epilogue warp
    }
    mbar_init(smem_u32(drain), 1);
    *s_abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_ws);
    tma_prefetch_desc(&tm_x);
  }
  if (warp == 1) tmem_alloc(smem_u32(s_tmem), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  // (with programmatic dependent launch the tile list is final here: it is
  // written by an index kernel that releases its dependents only at its end,
  // at least one launch before this one; everything else the previous
  // kernel writes is read only after pdl_wait)

  const int NB = FFN1 ? a.I / BM : (a.K + 2 * BM - 1) / (2 * BM);  // tiles per item
  const int KB = FFN1 ? a.K / BK : a.I / BK;  // K stages per tile
  const int n_items = min(*a.n_items, a.max_items);
  const int n_tiles = n_items * NB;

  auto load_weights = [&](int tile, int kb, uint32_t st, uint32_t fb) {
    const int4 it = a.items[tile / NB];
    const int nb = tile % NB;
    const bool shared = it.x >= a.E;
    const CUtensorMap* tw = shared ? &tm_ws : &tm_w;
    const int gc = shared ? 0 : it.x;
    // (rows past the last block, FFN2 with K % 256 == 128, read as zeros)
    if (a.packed) {  // tile-major weights: tile (row block, k block) is contiguous
      tma_load_3d(st, tw, 0, BM * (wblock<FFN1>(a, 0, nb) * KB + kb), gc, fb);
      tma_load_3d(st + C::A_BYTES, tw, 0, BM * (wblock<FFN1>(a, 1, nb) * KB + kb), gc, fb);
    } else {
      tma_load_3d(st, tw, kb * BK, wblock<FFN1>(a, 0, nb) * BM, gc, fb);
      tma_load_3d(st + C::A_BYTES, tw, kb * BK, wblock<FFN1>(a, 1, nb) * BM, gc, fb);
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (gat || lane == 0) {  // the whole warp when it gathers rows, else lane 0
      // The weights of the first STAGES stages do not depend on the previous
      // kernel: their loads start before pdl_wait (while that kernel still
      // runs); the activation rows of those stages follow after it.
      int pre = 0;
      if (lane == 0) {
        int tile = blockIdx.x, kb = 0;
        for (; pre < C::STAGES && tile < n_tiles; ++pre) {
          const uint32_t fb = smem_u32(&full[pre]);
          mbar_arrive_expect_tx(fb, gat ? C::NA * C::A_BYTES : C::STAGE_BYTES);
          load_weights(tile, kb, smem_u32(smem + pre * C::STAGE_BYTES), fb);
          s_issued[pre] = 1u;
          if (++kb == KB) {
            kb = 0;
            tile += gridDim.x;
          }
        }
      }
      if (gat) pre = __shfl_sync(0xffffffffu, pre, 0);
      pdl_wait();  // the previous kernel's outputs are complete and visible
      int seq = 0;  // stages handled so far
      int stage = 0;
      uint32_t phase = 0;
      const uint8_t* xtok = static_cast<const uint8_t*>(a.xq);
      for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        int stop = lane == 0 ? *s_abort : 0;
        if (gat) stop = __shfl_sync(0xffffffffu, stop, 0);
        if (stop) break;
        const int item = tile / NB;
        const int4 it = a.items[item];
        const bool shared = it.x >= a.E;
        const int n = min(BN, (it.z + 15) & ~15);  // rows the MMAs read
        if (gat) {
          // token of each row the MMAs read; the padding rows repeat a real one
          for (int i = lane; i < n; i += 32) {
            const int r = it.y + min(i, it.z - 1);
            int t = shared ? r - a.R : a.src[r];
            s_tok[i] = (unsigned)t < (unsigned)a.T ? t : 0;
          }
          __syncwarp();
        }
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++seq) {
          const uint32_t st = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t fb = smem_u32(&full[stage]);
          if (seq >= pre) {  // (the first stages' weights are already on their way)
            int got = 1;
            if (lane == 0)
              got = mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, a.err, s_abort) ? 1 : 0;
            if (gat) got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
              ok = false;
              break;
            }
            if (lane == 0) {
              mbar_arrive_expect_tx(fb, gat ? C::NA * C::A_BYTES : C::STAGE_BYTES);
              load_weights(tile, kb, st, fb);
            }
          }
          if (lane == 0) {
            if (!gat) tma_load_2d(st + C::NA * C::A_BYTES, &tm_x, kb * BK, it.y, fb);
            s_issued[stage] = phase + 1u;
          }
          if (gat) {
            // row i of the 128-byte-swizzled tile: 16-byte chunk c at chunk c ^ (i % 8)
            const uint32_t b0 = st + C::NA * C::A_BYTES;
            for (int qc = lane; qc < n * 8; qc += 32) {
              const int i = qc >> 3, c = qc & 7;
              cp_async16(b0 + i * BK + ((c ^ (i & 7)) << 4),
                         xtok + (size_t)s_tok[i] * a.K + kb * BK + c * 16);
            }
            cp_async_arrive_noinc(fb);
            __syncwarp();
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (gat) __syncwarp();  // s_tok is rewritten for the next tile
      }
      if (gat) cp_async_wait_all();  // no copy into this CTA's shared memory outlives it
      if (lane == 0 && *s_abort) {  // let our own copies land before the CTA can exit
        for (int s = 0; s < C::STAGES; ++s)
          if (s_issued[s]) mbar_wait_drain(smem_u32(&full[s]), s_issued[s] - 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    pdl_wait();
    if (lane == 0 && BLK) {
      // one partial sum per stage, into buffer pcount % ACC_STAGES
      int stage = 0, pcount = 0;
      uint32_t phase = 0;
      bool issued_any = false, ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok && !*s_abort; tile += gridDim.x) {
        const int rows = a.items[tile / NB].z;
        const uint32_t idesc = idesc_e4m3_f32(BM, min(BN, (rows + 15) & ~15));
        for (int kb = 0; kb < KB; ++kb, ++pcount) {
          const int pb = pcount % C::ACC_STAGES;
          if (!mbar_wait(smem_u32(&tempty[pb]), ((uint32_t)(pcount / C::ACC_STAGES) & 1u) ^ 1u,
                         a.err, s_abort) ||
              !mbar_wait(smem_u32(&full[stage]), phase, a.err, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d0 = tmem + pb * C::ACC_COLS;
          const uint32_t a0 = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b0 = a0 + C::NA * C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            const uint64_t bdesc = smem_desc_sw128(b0 + kk * UMMA_K);
            const uint32_t accum = kk ? 1u : 0u;
            mma_f8f6f4(d0, smem_desc_sw128(a0 + kk * UMMA_K), bdesc, idesc, accum);
            mma_f8f6f4(d0 + BN, smem_desc_sw128(a0 + C::A_BYTES + kk * UMMA_K), bdesc, idesc,
                       accum);
          }
          issued_any = true;
          mma_commit(smem_u32(&empty[stage]));
          mma_commit(smem_u32(&tfull[pb]));
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*s_abort && issued_any) {
        mma_commit(smem_u32(drain));
        mbar_wait_drain(smem_u32(drain), 0);
      }
    } else if (lane == 0) {
      int stage = 0, it_local = 0;
      uint32_t phase = 0;
      bool issued_any = false;
      for (int tile = blockIdx.x; tile < n_tiles && !*s_abort; tile += gridDim.x, ++it_local) {
        const int item = tile / NB;
        const int rows = a.items[item].z;
        const int n = min(BN, (rows + 15) & ~15);
        const uint32_t idesc = idesc_e4m3_f32(BM, n);
        const int acc = it_local % C::ACC_STAGES;
        const uint32_t acc_phase = (uint32_t)(it_local / C::ACC_STAGES) & 1u;
        if (!mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, a.err, s_abort)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + acc * C::ACC_COLS;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(smem_u32(&full[stage]), phase, a.err, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (gat) fence_proxy_async_smem();  // gathered rows came through the generic proxy
          const uint32_t a0 = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b0 = a0 + C::NA * C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            const uint64_t bdesc = smem_desc_sw128(b0 + kk * UMMA_K);
            const uint32_t accum = (kb | kk) ? 1u : 0u;
            mma_f8f6f4(d0, smem_desc_sw128(a0 + kk * UMMA_K), bdesc, idesc, accum);
            mma_f8f6f4(d0 + BN, smem_desc_sw128(a0 + C::A_BYTES + kk * UMMA_K), bdesc, idesc,
                       accum);
          }
          issued_any = true;
          mma_commit(smem_u32(&empty[stage]));  // frees the stage once these MMAs finish
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&tfull[acc]));  // accumulator ready for the epilogue
      }
      if (*s_abort && issued_any) {  // wait for our MMAs before tensor memory is freed
        mma_commit(smem_u32(drain));
        mbar_wait_drain(smem_u32(drain), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();
    const int q = warp & 3;  // tensor-memory lane quarter this warp may access
    int it_local = 0;
    if (BLK) {
      int pcount = 0;
      float h0[C::NA][kHeld], h1[C::NA][kHeld];  // scale rows, this tile's and the next's
      if (blockIdx.x < n_tiles)
        load_block_scales<FFN1>(a, blockIdx.x / NB, blockIdx.x % NB, KB, lane, h0);
      // tiles in pairs so that the two scale buffers swap roles without indexing
      for (int tile = blockIdx.x; tile < n_tiles;) {
        int nt = tile + gridDim.x;
        if (!block_epilogue<FFN1, BN, C::ACC_COLS, C::ACC_STAGES>(
                a, tmem, q, lane, tile / NB, tile % NB, KB, h0, nt < n_tiles ? nt / NB : -1,
                nt % NB, h1, tfull, tempty, s_abort, pcount))
          break;
        tile = nt;
        if (tile >= n_tiles) break;
        nt = tile + gridDim.x;
        if (!block_epilogue<FFN1, BN, C::ACC_COLS, C::ACC_STAGES>(
                a, tmem, q, lane, tile / NB, tile % NB, KB, h1, nt < n_tiles ? nt / NB : -1,
                nt % NB, h0, tfull, tempty, s_abort, pcount))
          break;
        tile = nt;
      }
    }
    for (int tile = blockIdx.x; !BLK && tile < n_tiles; tile += gridDim.x, ++it_local) {
      const int item = tile / NB, nb = tile - item * NB;
      const int4 it = a.items[item];
      const bool shared = it.x >= a.E;
      const int row0 = it.y, rows = it.z;
      const int acc = it_local % C::ACC_STAGES;
      const uint32_t acc_phase = (uint32_t)(it_local / C::ACC_STAGES) & 1u;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(smem_u32(&tfull[acc]), acc_phase, a.err, s_abort) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + acc * C::ACC_COLS;
      const int f = nb * BM + q * 32 + lane;  // feature (FFN1)
      if (FFN1) {
        const float* sc = shared ? a.sw13_scale : a.w13_scale + (size_t)it.x * 2 * a.I;
        const float sg = sc[f], su = sc[a.I + f];
        uint16_t* hout = static_cast<uint16_t*>(a.h);
        for (int c0 = 0; c0 < rows; c0 += 16) {
          uint32_t vg[16], vu[16];
          __syncwarp();
          tmem_ld16(tbase + c0, vg);
          tmem_ld16(tbase + BN + c0, vu);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = c0 + j;
            const int row = row0 + r;
            if (r < rows && (unsigned)row < (unsigned)a.rows_total) {
              const float xs = gat ? a.xscale[shared ? row - a.R : a.src[row]] : a.xscale[row];
              const float g = (__uint_as_float(vg[j]) * xs) * sg;
              const float u = (__uint_as_float(vu[j]) * xs) * su;
              const float hv = gated_act(a.act, g, u);
              hout[(size_t)row * a.I + f] = (uint16_t)f32_bits_to_bf16(hv);
            }
          }
        }
      } else {  // output channels f2 (block 2nb) and f2 + 128 (block 2nb + 1)
        const int f2 = 2 * nb * BM + q * 32 + lane;
        const bool two = f2 + BM < a.K;
        const float* sc = shared ? a.sw2_scale : a.w2_scale + (size_t)it.x * a.K;
        const float s2a = sc[f2], s2b = two ? sc[f2 + BM] : 0.0f;
        uint16_t* yout = static_cast<uint16_t*>(a.y);
        for (int c0 = 0; c0 < rows; c0 += 16) {
          uint32_t va[16], vb[16];
          __syncwarp();
          tmem_ld16(tbase + c0, va);
          tmem_ld16(tbase + BN + c0, vb);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = c0 + j;
            const int row = row0 + r;
            if (r < rows && (unsigned)row < (unsigned)a.rows_total) {
              const float rw = (!shared && a.row_w) ? a.row_w[row] : 1.0f;
              const float hs = a.hs[row];
              const float ya = ((__uint_as_float(va[j]) * hs) * s2a) * rw;
              const float yb = ((__uint_as_float(vb[j]) * hs) * s2b) * rw;
              if (a.out_acc) {  // fused combine: add into the token's fp32 sum
                const int tok = shared ? row - a.R : a.src[row];
                if ((unsigned)tok < (unsigned)a.T) {
                  float* acc_r = a.out_acc + (size_t)tok * a.K;
                  atomicAdd(acc_r + f2, ya);
                  if (two) atomicAdd(acc_r + f2 + BM, yb);
                }
              } else {
                uint16_t* yr = yout + (size_t)row * a.K;
                yr[f2] = (uint16_t)f32_bits_to_bf16(ya);
                if (two) yr[f2 + BM] = (uint16_t)f32_bits_to_bf16(yb);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  pdl_release();  // the next kernel may start launching: this one is done
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Byte tensor map with a 128-byte-wide, 128-byte-swizzled box.  rank 3:
// {inner K, rows, groups} with box {128, box_rows, 1} (weights, one group per
// expert; a single group still uses rank 3 because the loads are 3-D);
// rank 2: {inner K, rows} with box {128, box_rows} (activation rows).
bool make_map(CUtensorMap* m, int rank, const void* base, uint64_t inner, uint64_t rows,
              uint64_t groups, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc || !base) return false;
  cuuint64_t dims[3] = {inner, rows, groups};
  cuuint64_t strides[2] = {inner, inner * rows};
  cuuint32_t box[3] = {(cuuint32_t)BK, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool FFN1, int BN, bool BLK>
cudaError_t launch_impl(const GroupedFfnArgs& a, cudaStream_t s) {
  using C = Cfg<FFN1, BN, BLK>;
  const int K = FFN1 ? a.K : a.I;      // reduction width
  const int Wrows = FFN1 ? 2 * a.I : a.K;
  const void* w = FFN1 ? a.w13 : a.w2;
  const void* ws = FFN1 ? a.sw13 : a.sw2;
  const void* x = FFN1 ? a.xq : a.hq;
  CUtensorMap tw, tws, tx;
  // tile-major weights are [group][tiles * 128 rows][128 bytes]
  const uint64_t winner = a.packed ? BK : K;
  const uint64_t wrows = a.packed ? (uint64_t)Wrows * (K / BK) : Wrows;
  if (!make_map(&tw, 3, w, winner, wrows, a.E, BM)) return cudaErrorInvalidValue;
  if (!make_map(&tws, 3, ws ? ws : w, winner, wrows, 1, BM)) return cudaErrorInvalidValue;
  if (!make_map(&tx, 2, x, K, a.rows_total, 1, BN)) return cudaErrorInvalidValue;
  if (BLK && (K / BK > C::MAX_KB || (FFN1 ? a.I : a.K) % BM)) return cudaErrorInvalidValue;
  cudaError_t e = ensure_max_smem<grouped_ffn_kernel<FFN1, BN, BLK>>(C::SMEM);
  if (e != cudaSuccess) return e;
  count_launch();
  e = launch_kernel(grouped_ffn_kernel<FFN1, BN, BLK>, dim3(device_sm_count()), dim3(kThreads),
                    C::SMEM, s, 1, tw, tws, tx, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool FFN1>
cudaError_t launch_bn(const GroupedFfnArgs& a, cudaStream_t s) {
  if (a.blockwise) {
    switch (a.BN) {
      case 32: return launch_impl<FFN1, 32, true>(a, s);
      case 64: return launch_impl<FFN1, 64, true>(a, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.BN) {
    case 32: return launch_impl<FFN1, 32, false>(a, s);
    case 64: return launch_impl<FFN1, 64, false>(a, s);
    case 128: return launch_impl<FFN1, 128, false>(a, s);
    case 256: return launch_impl<FFN1, 256, false>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_ffn1(const GroupedFfnArgs& a, cudaStream_t s) { return launch_bn<true>(a, s); }
cudaError_t launch_ffn2(const GroupedFfnArgs& a, cudaStream_t s) { return launch_bn<false>(a, s); }

}  // namespace moe
