// ffn_gemm_2cta.cu -- GEMMs on pairs of SMs (tcgen05 cta_group::2).
//
// One pipeline, used for
//   * S5/S6 of large batches: the grouped fp8 expert GEMMs (same arithmetic as
//     ffn_gemm.cu: "Optimising Ling-2.6-1T on TPU with SGLang-JAX", s.5
//     per-channel direct_scaled_dot; FFN1/FFN2 of the s.1 cost model), when
//     experts hold hundreds of rows (prefill);
//   * S9 of the LatentMoE block ("Kimi K3 ... feasibility analysis", s.2.4):
//     the bf16 dense GEMMs z = x Wd^T, the shared expert's gate/up with the
//     SwiGLU epilogue, and out = yn Wu^T + h_s W2s^T as one accumulation over
//     two K segments (up_proj and the shared expert's down projection).
//
// A cluster of two CTAs computes a 256-row x 256-column tile with one MMA
// stream.  Each CTA stages half of the activation rows (A, 128 rows x 128 B
// per K step) and half of the weight rows (B, 128 rows x 128 B), so every SM
// moves 32 KB per K step for 4.2 M (fp8) or 2.1 M (bf16) multiply-adds; the
// tile's accumulator (128 rows x 256 fp32 columns per CTA) is double-buffered
// in tensor memory.
//
// Epilogues (thread = one activation row, 16 columns per tcgen05.ld; the
// tile's channel scales staged once in shared memory; each warp's 32 rows x 32
// output columns transposed through a 64-byte-swizzled shared-memory buffer so
// that four lanes store one row's 64 contiguous bytes):
//   SWIGLU: columns 0..127 = g (weight rows f0.., staged by CTA 0), columns
//           128..255 = u (rows I+f0.., staged by CTA 1); h = bf16(silu(g) u),
//           with the fp8 per-row and per-channel scales when the operands are fp8.
//   DOWN:   y = bf16(((acc * hs[row]) * s[c]) * row_w[row])   (fp8 FFN2)
//   STORE:  out = bf16(acc)                                   (bf16 dense)
//
// Roles per CTA (192 threads): warp 0 TMA producer, warp 1 MMA issuer (even
// CTA only; the odd CTA's warp 1 only joins the tensor-memory allocation),
// warps 2-5 epilogue.  Both CTAs' TMA loads complete on the even CTA's `full`
// barrier; the even CTA's commits arrive on both CTAs' `empty` / `tfull`
// barriers; both epilogues release an accumulator on the even CTA's `tempty`
// barrier (a relaxed arrive: the warp's tensor-memory loads have completed, its
// output stores need not have).  All waits are bounded as in ffn_gemm.cu.
//
// Grouped items of at most 128 rows run as M = 128 MMAs (64 activation rows
// per CTA), so an expert's small last item is not padded to 256 rows; see
// is_small() for the accumulator layout of those tiles.
//
// Row gather (FFN1, opt-in, tuning().ffn1_gather): the activations arrive as
// one fp8 row per token; the producer warp's lanes each copy four of the
// tile's rows per stage with one TMA tile::gather4 (a map whose box is one row
// high; rows past the item read out-of-range zeros), straight into the
// swizzled stage, completing on the even CTA's barrier like the other loads.
// Correct, but the gathered stages arrive far slower than one 128-row box
// (prefill FFN1 12.06 vs 3.70 ms), so permuted rows stay the default.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>

#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int P_ROWS = 128;   // activation rows per CTA (M = 256 per pair)
constexpr int P_N = 256;      // output columns per tile
constexpr int P_BK = 128;     // K bytes per stage
constexpr int P_UMMA_B = 32;  // K bytes per tcgen05.mma (32 fp8 or 16 bf16)
constexpr int P_THREADS = 192;
constexpr int P_A_BYTES = P_ROWS * P_BK;       // 16 KB
constexpr int P_B_BYTES = (P_N / 2) * P_BK;    // 16 KB (this CTA's half of N)
constexpr int P_STAGE = P_A_BYTES + P_B_BYTES;  // 32 KB
// six stages: compute-bound tiles want the deeper ring (four stages: prefill
// 7.97 vs 7.75 ms, LatentMoE dense GEMMs 12% slower), unlike the single-SM
// weight stream
constexpr int P_STAGES = 6;
constexpr int P_ACC_STAGES = 2;
constexpr int P_TMEM_COLS = 512;
constexpr int P_NUM_BARS = 2 * P_STAGES + 2 * P_ACC_STAGES + 1;
constexpr int P_STG_ROW = 64;                   // transposed output: 32 bf16 columns per row
constexpr int P_STG_BUF = 32 * P_STG_ROW;       // one epilogue warp's 32 rows
constexpr int P_STG = 4 * 2 * P_STG_BUF;        // 4 epilogue warps, double-buffered (16 KB)
constexpr int P_SCL = 2 * P_N * 4;              // a tile's channel scales, double-buffered
constexpr int P_EPI_BAR = 1;                    // named barrier of the 4 epilogue warps
constexpr int P_SMEM =
    1024 + P_STAGES * P_STAGE + P_STG + P_SCL + P_NUM_BARS * 8 + 16 + P_STAGES * 4;

enum { KIND_FP8 = 0, KIND_BF16 = 1 };
enum { EPI_SWIGLU = 0, EPI_DOWN = 1, EPI_STORE = 2, EPI_F32 = 3 };

// One launch: the tiles, the K segments and the epilogue's operands.
struct PairGemm {
  const int4* items;      // grouped work list {group, row0, rows, 0}; nullptr = dense
  const int32_t* n_items;
  int max_items;
  int dense_rows;         // dense: rows of A, tiled in 256-row items
  int E;                  // grouped: group E reads the shared-expert weight map
  int nb;                 // output blocks per item
  int kb1, kb2;           // K stages from (x, w) and from (x2, w2)
  int I;                  // SWIGLU: first row of the up-projection block
  int packed;             // first-segment weights in tile-major order (pack.cu)
  int act;                // SwiGLU epilogue: 0 SwiGLU, 1 SiTU
  int rows_total;         // rows of A (and of the output)
  int small;              // grouped: items of <= 128 rows run as M = 128 tiles
  const float* xscale;    // fp8 SWIGLU: per-row activation scale
  const float* w_scale;   // fp8: per-channel scale of group 0 (stride scale_stride)
  const float* ws_scale;  // fp8: per-channel scale of the shared expert
  int scale_stride;
  const float* hs;        // DOWN: per-row scale of h
  const float* row_w;     // DOWN: routing weight per row (nullptr = 1)
  void* out;              // bf16 output, row stride ldo elements
  int ldo;
  int gather;             // fp8 SWIGLU: tm_x holds one row per token (box one row
                          // high); the producer gathers row r of a tile from token
                          // src[r] (r < R) or r - R (shared expert), and the
                          // epilogue takes that token's activation scale
  const int32_t* src;     // [R] token of each routed row (gather only)
  int R, T;               // routed rows, tokens (gather only)
  int a_period;           // dense: A's K stage is kb % a_period (0: kb), so one A
                          // row block meets several consecutive K blocks of B
  int n_valid;            // EPI_F32: output columns that exist (ldo >= n_valid)
  int ksplit;             // dense EPI_F32: K cut into this many stage ranges (0, 1:
                          // none), range s stored as its own fp32 block at
                          // out + s * split_stride, so a grid of few tiles still
                          // fills the GPU; each range is non-empty
  size_t split_stride;
  int* err;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);  // a -> low half
  return *reinterpret_cast<uint32_t*>(&p);
}

__device__ __forceinline__ int4 tile_item(const PairGemm& g, int item) {
  if (g.items) return g.items[item];
  const int row0 = item * 2 * P_ROWS;
  return make_int4(0, row0, min(2 * P_ROWS, g.dense_rows - row0), 0);
}

// Tile t -> (item, output block).  Dense launches and groups without the
// count in the item's fourth field go item by item (t = item * NB + nb).  A
// group's items carry {index within the group, items in the group} there, and
// its tiles go output block by output block instead: the group's n items of
// one block are n consecutive tiles, which neighbouring SM pairs run at the
// same time, so they stream the same expert weights while those are in L2.
// (A group cut short by the end of the list keeps the item-by-item order.)
__device__ __forceinline__ int2 tile_coords(const PairGemm& g, int tile, int NB, int n_items) {
  int item = tile / NB, nb = tile - item * NB;
  if (g.items) {
    const int w = g.items[item].w;
    const int first = item - (w & 0xFFFF), n = w >> 16;
    if (w && first >= 0 && first + n <= n_items) {
      const int local = tile - first * NB;
      item = first + local % n;
      nb = local / n;
    }
  }
  return make_int2(item, nb);
}

// Grouped items of at most 128 rows run as M = 128 tiles: each CTA stages 64
// activation rows, and the tile's accumulator lands in tensor-memory columns
// 0..127 of the pair: lanes 0..63 hold rows 0..63 of the CTA's half for output
// columns 0..127, lanes 64..127 the same rows for columns 128..255 (read back
// from the hardware; an M = 256 tile puts row i in lane i, all 256 columns).
__device__ __forceinline__ bool is_small(const PairGemm& g, const int4& it) {
  return g.small && g.items && it.z <= 2 * 64;
}

template <int KIND>
__device__ __forceinline__ uint32_t pair_idesc(int M = 2 * P_ROWS) {
  // f32 accumulate, K-major A and B, M = 256 (or 128) for the pair, N = 256
  const uint32_t fmt = KIND == KIND_FP8 ? 0u : 1u;  // e4m3 (kind::f8f6f4) / bf16 (kind::f16)
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(P_N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

template <int KIND>
__device__ __forceinline__ void pair_mma(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t acc) {
  if (KIND == KIND_FP8) {
    mma_f8f6f4_pair(d, adesc, bdesc, idesc, acc);
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
  }
}

template <int KIND, int EPI>
__global__ void __launch_bounds__(P_THREADS, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_ws,
                     const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_w2,
                     const __grid_constant__ CUtensorMap tm_x2,
                     const __grid_constant__ CUtensorMap tm_xh,
                     const __grid_constant__ CUtensorMap tm_wh,
                     const __grid_constant__ CUtensorMap tm_wsh, const PairGemm g) {
  constexpr int EL = KIND == KIND_FP8 ? P_BK : P_BK / 2;  // K elements per stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stg = smem + P_STAGES * P_STAGE;  // output transpose buffers
  float* s_scl = reinterpret_cast<float*>(stg + P_STG);
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg + P_STG + P_SCL);
  uint64_t* full = bars;
  uint64_t* empty = bars + P_STAGES;
  uint64_t* tfull = bars + 2 * P_STAGES;
  uint64_t* tempty = tfull + P_ACC_STAGES;
  uint64_t* drain = tempty + P_ACC_STAGES;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + P_NUM_BARS);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint32_t* s_issued = s_tmem + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
      s_issued[s] = 0;
    }
    for (int s = 0; s < P_ACC_STAGES; ++s) {
      mbar_init(smem_u32(&tfull[s]), 1);
      mbar_init(smem_u32(&tempty[s]), 8);  // 4 epilogue warps in each CTA
    }
    mbar_init(smem_u32(drain), 1);
    *s_abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_ws);
    tma_prefetch_desc(&tm_x);
    if (g.kb2) {
      tma_prefetch_desc(&tm_w2);
      tma_prefetch_desc(&tm_x2);
    }
    if (g.small) {
      tma_prefetch_desc(&tm_xh);
      tma_prefetch_desc(&tm_wh);
      tma_prefetch_desc(&tm_wsh);
    }
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(s_tmem), P_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_wait();  // the previous kernel's outputs are complete and visible

  const int NB = g.nb;
  const int KB = g.kb1 + g.kb2;
  const int n_items = g.items ? min(*g.n_items, g.max_items)
                              : (g.dense_rows + 2 * P_ROWS - 1) / (2 * P_ROWS);
  // dense split-K: tile t is K range t % S of output tile t / S
  const int S = (!g.items && EPI == EPI_F32 && g.ksplit > 1) ? g.ksplit : 1;
  const int KBs = (KB + S - 1) / S;
  const int n_tiles = n_items * NB * S;
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // With the row gather the whole warp works: lane 0 waits, arms the stage
    // and loads the weights, and every lane gathers four activation rows.
    const bool gat = KIND == KIND_FP8 && EPI == EPI_SWIGLU && g.gather;
    if (gat || lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = cluster; tile < n_tiles; tile += n_clusters) {
        int stop = lane == 0 ? *s_abort : 0;
        if (gat) stop = __shfl_sync(0xffffffffu, stop, 0);
        if (stop) break;
        const int sk = tile % S;
        const int k0 = sk * KBs, k1 = min(KB, k0 + KBs);
        const int2 tc = tile_coords(g, tile / S, NB, n_items);
        const int item = tc.x, nb = tc.y;
        const int4 it = tile_item(g, item);
        const bool shared = g.items && it.x >= g.E;
        const CUtensorMap* tw = shared ? &tm_ws : &tm_w;
        const int gc = shared ? 0 : it.x;
        const int wrow = EPI == EPI_SWIGLU ? (rank == 0 ? nb * 128 : g.I + nb * 128)
                                           : nb * P_N + 128 * (int)rank;
        // M = 128 tile: 64 activation rows per CTA; for SWIGLU each CTA stages
        // the W1 and the W3 half-block of its 64 features (so g and u of a
        // feature meet in one tensor-memory lane half)
        const bool small = is_small(g, it);
        const CUtensorMap* twh = shared ? &tm_wsh : &tm_wh;
        auto load_w = [&](uint32_t dst, const CUtensorMap* m, int row, int kb, uint32_t fb) {
          if (g.packed)  // tile-major weights: (row block, k block) is contiguous
            tma_load_3d_pair(dst, m, 0, 128 * ((row / 128) * g.kb1 + kb) + row % 128, gc, fb);
          else
            tma_load_3d_pair(dst, m, kb * EL, row, gc, fb);
        };
        // gather: the tokens of this CTA's rows 4 lane .. 4 lane + 3 (rows past
        // the item read token T: out of range, so zeros)
        const int cta_rows = small ? 64 : 128;
        int tok[4] = {0, 0, 0, 0};
        if (gat) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int local = cta_rows * (int)rank + 4 * lane + j;  // row within the item
            const int r = it.y + local;
            int t = g.T;
            if (4 * lane + j < cta_rows && local < it.z && (unsigned)r < (unsigned)g.rows_total) {
              t = r < g.R ? g.src[r] : r - g.R;
              if ((unsigned)t >= (unsigned)g.T) t = g.T;
            }
            tok[j] = t;
          }
        }
        bool ok = true;
        for (int kb = k0; kb < k1; ++kb) {
          int got = 1;
          if (lane == 0) got = mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, g.err, s_abort);
          if (gat) got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) {
            ok = false;
            break;
          }
          const uint32_t st = smem_u32(smem + stage * P_STAGE);
          const uint32_t fb_leader = mapa_shared(smem_u32(&full[stage]), 0);
          if (gat) {
            if (lane == 0) {
              if (leader)
                mbar_arrive_expect_tx(smem_u32(&full[stage]),
                                      small ? 2 * (P_A_BYTES / 2 + P_B_BYTES) : 2 * P_STAGE);
              if (small) {
                load_w(st + P_A_BYTES, twh, nb * 128 + 64 * (int)rank, kb, fb_leader);
                load_w(st + P_A_BYTES + P_B_BYTES / 2, twh, g.I + nb * 128 + 64 * (int)rank, kb,
                       fb_leader);
              } else {
                load_w(st + P_A_BYTES, tw, wrow, kb, fb_leader);
              }
              s_issued[stage] = phase + 1u;
            }
            // four 128-byte rows per copy, landing at rows 4 lane .. 4 lane + 3
            // of the swizzled tile (the swizzle follows the shared address)
            if (4 * lane < cta_rows)
              tma_gather4_pair(st + 512 * lane, &tm_x, kb * EL, tok, fb_leader);
            if (++stage == P_STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (leader)
            mbar_arrive_expect_tx(smem_u32(&full[stage]),
                                  small ? 2 * (P_A_BYTES / 2 + P_B_BYTES) : 2 * P_STAGE);
          if (small) {
            tma_load_2d_pair(st, &tm_xh, kb * EL, it.y + 64 * (int)rank, fb_leader);
            if (EPI == EPI_SWIGLU) {
              load_w(st + P_A_BYTES, twh, nb * 128 + 64 * (int)rank, kb, fb_leader);
              load_w(st + P_A_BYTES + P_B_BYTES / 2, twh, g.I + nb * 128 + 64 * (int)rank, kb,
                     fb_leader);
            } else {
              load_w(st + P_A_BYTES, tw, wrow, kb, fb_leader);
            }
          } else if (kb < g.kb1) {
            tma_load_2d_pair(st, &tm_x, (g.a_period ? kb % g.a_period : kb) * EL,
                             it.y + 128 * (int)rank, fb_leader);
            load_w(st + P_A_BYTES, tw, wrow, kb, fb_leader);
          } else {
            const int k2 = (kb - g.kb1) * EL;
            tma_load_2d_pair(st, &tm_x2, k2, it.y + 128 * (int)rank, fb_leader);
            tma_load_3d_pair(st + P_A_BYTES, &tm_w2, k2, wrow, 0, fb_leader);
          }
          s_issued[stage] = phase + 1u;
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (lane == 0 && *s_abort && leader) {  // the pair's loads complete on the even CTA's barriers
        for (int s = 0; s < P_STAGES; ++s)
          if (s_issued[s]) mbar_wait_drain(smem_u32(&full[s]), s_issued[s] - 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      int stage = 0, it_local = 0;
      uint32_t phase = 0;
      bool issued_any = false;
      const uint32_t idesc256 = pair_idesc<KIND>(), idesc128 = pair_idesc<KIND>(128);
      for (int tile = cluster; tile < n_tiles && !*s_abort; tile += n_clusters, ++it_local) {
        const uint32_t idesc =
            is_small(g, tile_item(g, tile_coords(g, tile / S, NB, n_items).x)) ? idesc128 : idesc256;
        const int k0 = (tile % S) * KBs, k1 = min(KB, k0 + KBs);
        const int acc = it_local % P_ACC_STAGES;
        const uint32_t acc_phase = (uint32_t)(it_local / P_ACC_STAGES) & 1u;
        if (!mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, g.err, s_abort)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * P_N;
        bool ok = true;
        for (int kb = k0; kb < k1; ++kb) {
          if (!mbar_wait(smem_u32(&full[stage]), phase, g.err, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * P_STAGE);
          const uint32_t b0 = a0 + P_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < P_BK / P_UMMA_B; ++kk)
            pair_mma<KIND>(d, smem_desc_sw128(a0 + kk * P_UMMA_B),
                           smem_desc_sw128(b0 + kk * P_UMMA_B), idesc,
                           ((kb - k0) | kk) ? 1u : 0u);
          issued_any = true;
          mma_commit_pair(smem_u32(&empty[stage]), 0x3);
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(smem_u32(&tfull[acc]), 0x3);
      }
      if (*s_abort && issued_any) {
        mma_commit_pair(smem_u32(drain), 0x1);
        mbar_wait_drain(smem_u32(drain), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int lrow = q * 32 + lane;  // this thread's row within the CTA's half
    const uint32_t tempty_leader0 = mapa_shared(smem_u32(&tempty[0]), 0);
    const uint32_t stg_w = smem_u32(stg + q * 2 * P_STG_BUF);
    const uint32_t swz = (uint32_t)((lane >> 1) & 3);  // 64-byte swizzle of this row's chunks
    int grp = 0;  // groups stored by this warp (transpose buffer = grp & 1)
    int it_local = 0;
    for (int tile = cluster; tile < n_tiles; tile += n_clusters, ++it_local) {
      const int2 tc = tile_coords(g, tile / S, NB, n_items);
      const int item = tc.x, nb = tc.y;
      const int4 it = tile_item(g, item);
      const bool shared = g.items && it.x >= g.E;
      const size_t part = (size_t)(tile % S) * g.split_stride;  // split-K: this range's block
      const int acc = it_local % P_ACC_STAGES;
      const uint32_t acc_phase = (uint32_t)(it_local / P_ACC_STAGES) & 1u;
      // this tile's channel scales: two per thread, read before the wait
      constexpr bool SCALED = KIND == KIND_FP8 && EPI != EPI_STORE;
      const int cs = EPI == EPI_SWIGLU ? nb * 128 : nb * P_N;  // first scale column
      const int cs2 = EPI == EPI_SWIGLU ? g.I + nb * 128 : nb * P_N + 128;
      float sv0 = 0.0f, sv1 = 0.0f;
      if (SCALED) {
        const float* sc = shared ? g.ws_scale : g.w_scale + (size_t)it.x * g.scale_stride;
        sv0 = __ldg(sc + cs + lrow);
        sv1 = __ldg(sc + cs2 + lrow);
      }
      int ok = 1;
      if (lane == 0) ok = mbar_wait(smem_u32(&tfull[acc]), acc_phase, g.err, s_abort) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      float* scl = s_scl + (it_local & 1) * P_N;
      if (SCALED) {
        scl[lrow] = sv0;
        scl[128 + lrow] = sv1;
      }
      // the four warps agree on going on, and the scales are visible to all
      if (!bar_and(P_EPI_BAR, 128, ok)) break;
      tc_fence_after();
      // M = 128 tiles: warps 0, 1 hold rows 0..63 of this CTA's half for the
      // first 128 output columns, warps 2, 3 the same rows for the last 128
      const bool small = is_small(g, it);
      const int hq = q >> 1;
      const int wr0 = small ? 64 * (int)rank + 32 * (q & 1)  // this warp's first row
                            : 128 * (int)rank + q * 32;     // within the item
      const int r = wr0 + lane;
      const int row = it.y + r;
      const bool valid = r < it.z && (unsigned)row < (unsigned)g.rows_total;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + acc * P_N;
      // 32 bf16 columns of each of the warp's rows at output column `col`: lane
      // l writes its row's four 16-byte chunks (chunk i at i ^ swz), then reads
      // chunk l % 4 of rows l / 4 + 8i, so each store covers 8 rows x 64 bytes
      auto put = [&](const uint32_t (&packed)[16], int col) {
        const uint32_t buf = stg_w + (uint32_t)(grp & 1) * P_STG_BUF;
        ++grp;
        const uint32_t ra = buf + lane * P_STG_ROW;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_shared_v4(ra + (((uint32_t)i ^ swz) << 4), packed[4 * i], packed[4 * i + 1],
                       packed[4 * i + 2], packed[4 * i + 3]);
        __syncwarp();
        const int ch = lane & 3;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = 8 * i + (lane >> 2);
          const uint4 v = ld_shared_v4(buf + rr * P_STG_ROW +
                                       (((uint32_t)ch ^ ((uint32_t)(rr >> 1) & 3u)) << 4));
          const int orow_i = it.y + wr0 + rr;
          if (wr0 + rr < it.z && (unsigned)orow_i < (unsigned)g.rows_total)
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(g.out) + (size_t)orow_i * g.ldo +
                                      col + 8 * ch) = v;
        }
      };
      // fp32 output (EPI_F32): 16 columns of the warp's 32 rows at output
      // column `col` through the same staging buffer, 16-byte stores of four
      // columns (row stride and valid columns multiples of four)
      auto put32 = [&](const uint32_t (&vals)[16], int col) {
        const uint32_t buf = stg_w + (uint32_t)(grp & 1) * P_STG_BUF;
        ++grp;
        const uint32_t ra = buf + lane * P_STG_ROW;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_shared_v4(ra + (((uint32_t)i ^ swz) << 4), vals[4 * i], vals[4 * i + 1],
                       vals[4 * i + 2], vals[4 * i + 3]);
        __syncwarp();
        const int ch = lane & 3;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = 8 * i + (lane >> 2);
          const uint4 v = ld_shared_v4(buf + rr * P_STG_ROW +
                                       (((uint32_t)ch ^ ((uint32_t)(rr >> 1) & 3u)) << 4));
          const int orow_i = it.y + wr0 + rr;
          const int colx = col + 4 * ch;
          if (wr0 + rr < it.z && (unsigned)orow_i < (unsigned)g.rows_total && colx < g.n_valid)
            *reinterpret_cast<uint4*>(static_cast<float*>(g.out) + part + (size_t)orow_i * g.ldo +
                                      colx) = v;
        }
      };
      // Columns in groups of 32 (two tcgen05.ld x16 per operand), software
      // pipelined: the next group's tensor-memory loads are in flight while this
      // group is scaled and stored, so the load latency is paid once per tile.
      if (EPI == EPI_SWIGLU) {
        const int f0 = nb * 128;
        const int uo = small ? 64 : 128;     // tensor-memory column of u after g
        const int co = small ? 64 * hq : 0;  // this thread's first feature in the tile
        const int ncol = small ? 64 : 128;
        float xs = 1.0f;
        if (KIND == KIND_FP8) {
          xs = 0.0f;
          if (valid && g.gather) {  // one scale per token
            const int t = row < g.R ? g.src[row] : row - g.R;
            if ((unsigned)t < (unsigned)g.T) xs = g.xscale[t];
          } else if (valid) {
            xs = g.xscale[row];
          }
        }
        uint32_t va[4][16], vb[4][16];  // g lo, g hi, u lo, u hi
        auto load = [&](uint32_t (&v)[4][16], int c) {
          __syncwarp();
          tmem_ld16(tbase + c, v[0]);
          tmem_ld16(tbase + c + 16, v[1]);
          tmem_ld16(tbase + uo + c, v[2]);
          tmem_ld16(tbase + uo + c + 16, v[3]);
        };
        auto emit = [&](const uint32_t (&v)[4][16], int c) {
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float4 sg = make_float4(1.0f, 1.0f, 1.0f, 1.0f), su = sg;
            if (KIND == KIND_FP8) {
              sg = *reinterpret_cast<const float4*>(scl + co + c + j);
              su = *reinterpret_cast<const float4*>(scl + 128 + co + c + j);
            }
            const float sgv[4] = {sg.x, sg.y, sg.z, sg.w}, suv[4] = {su.x, su.y, su.z, su.w};
            float hv[4];
#pragma unroll
            for (int u2 = 0; u2 < 4; ++u2) {
              const int jj = j + u2;
              float gg = __uint_as_float(v[jj >> 4][jj & 15]);
              float uu = __uint_as_float(v[2 + (jj >> 4)][jj & 15]);
              if (KIND == KIND_FP8) {
                gg = (gg * xs) * sgv[u2];
                uu = (uu * xs) * suv[u2];
              }
              hv[u2] = gated_act(g.act, gg, uu);
            }
            packed[j / 2] = pack_bf16x2(hv[0], hv[1]);
            packed[j / 2 + 1] = pack_bf16x2(hv[2], hv[3]);
          }
          put(packed, f0 + co + c);
        };
        load(va, 0);
        tmem_ld_wait();
        for (int c = 0; c < ncol; c += 64) {
          load(vb, c + 32);
          emit(va, c);
          tmem_ld_wait();
          if (c + 64 < ncol) load(va, c + 64);
          emit(vb, c + 32);
          tmem_ld_wait();
        }
      } else {
        const int c0 = nb * P_N;
        const int co = small ? 128 * hq : 0;  // this thread's first output column in the tile
        const int ncol = small ? 128 : P_N;
        const float hs = EPI == EPI_DOWN ? (valid ? g.hs[row] : 0.0f) : 1.0f;
        const float rw = (EPI == EPI_DOWN && valid && !shared && g.row_w) ? g.row_w[row] : 1.0f;
        uint32_t va[2][16], vb[2][16];
        auto load = [&](uint32_t (&v)[2][16], int c) {
          __syncwarp();
          tmem_ld16(tbase + c, v[0]);
          tmem_ld16(tbase + c + 16, v[1]);
        };
        auto emit = [&](const uint32_t (&v)[2][16], int c) {
          if constexpr (EPI == EPI_F32) {
            if (g.ldo % 4 == 0 && g.n_valid % 4 == 0) {
              put32(v[0], c0 + co + c);
              put32(v[1], c0 + co + c + 16);
              return;
            }
            if (valid) {  // fp32 out, row by row
              float* orow = static_cast<float*>(g.out) + part + (size_t)row * g.ldo;
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                const int col = c0 + co + c + jj;
                if (col < g.n_valid) orow[col] = __uint_as_float(v[jj >> 4][jj & 15]);
              }
            }
          } else {
            uint32_t packed[16];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              float4 s4 = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
              if (EPI == EPI_DOWN) s4 = *reinterpret_cast<const float4*>(scl + co + c + j);
              const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
              float yv[4];
#pragma unroll
              for (int u2 = 0; u2 < 4; ++u2) {
                const int jj = j + u2;
                float y0 = __uint_as_float(v[jj >> 4][jj & 15]);
                if (EPI == EPI_DOWN) y0 = ((y0 * hs) * sv[u2]) * rw;
                yv[u2] = y0;
              }
              packed[j / 2] = pack_bf16x2(yv[0], yv[1]);
              packed[j / 2 + 1] = pack_bf16x2(yv[2], yv[3]);
            }
            put(packed, c0 + co + c);
          }
        };
        load(va, 0);
        tmem_ld_wait();
        for (int c = 0; c < ncol; c += 64) {
          load(vb, c + 32);
          emit(va, c);
          tmem_ld_wait();
          if (c + 64 < ncol) load(va, c + 64);
          emit(vb, c + 32);
          tmem_ld_wait();
        }
      }
      tc_fence_before();
      __syncwarp();
      // the accumulator is free once this warp's tensor-memory loads are done
      // (waited above); the output stores need not be complete
      if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader0 + acc * 8);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while its peer may still signal it
  pdl_release();  // the next kernel may start launching: this one is done
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, P_TMEM_COLS);
  }
}

// Grouped items of <= 128 rows as M = 128 tiles unless tuning().pair_small is 0.
bool pair_small_tiles() { return tuning().pair_small != 0; }

// Map over a row-major [groups][rows][inner] tensor of 1-byte (fp8) or
// 2-byte (bf16) elements; box = 128 bytes x box_rows rows (128, or 64 for the
// halves of M = 128 tiles), 128-byte swizzle.
bool pair_map(CUtensorMap* m, int kind, int rank, const void* base, uint64_t inner,
              uint64_t rows, uint64_t groups, uint32_t box_rows = P_ROWS) {
  auto enc = tensor_map_encoder();
  if (!enc || !base) return false;
  const int es = kind == KIND_FP8 ? 1 : 2;
  cuuint64_t dims[3] = {inner, rows, groups};
  cuuint64_t strides[2] = {inner * es, inner * rows * es};
  cuuint32_t box[3] = {(cuuint32_t)(P_BK / es), box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, kind == KIND_FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
             rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND, int EPI>
cudaError_t launch_pair_gemm(const CUtensorMap& tw, const CUtensorMap& tws, const CUtensorMap& tx,
                             const CUtensorMap& tw2, const CUtensorMap& tx2,
                             const CUtensorMap& txh, const CUtensorMap& twh,
                             const CUtensorMap& twsh, const PairGemm& g, cudaStream_t s) {
  cudaError_t e = ensure_max_smem<pair_gemm_kernel<KIND, EPI>>(P_SMEM);
  if (e != cudaSuccess) return e;
  count_launch();
  e = launch_kernel(pair_gemm_kernel<KIND, EPI>, dim3((device_sm_count() / 2) * 2), dim3(P_THREADS),
                    P_SMEM, s, 2, tw, tws, tx, tw2, tx2, txh, twh, twsh, g);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool FFN1>
cudaError_t launch_grouped_pair(const GroupedFfnArgs& a, cudaStream_t s) {
  const int K = FFN1 ? a.K : a.I;
  const int Wrows = FFN1 ? 2 * a.I : a.K;
  const void* w = FFN1 ? a.w13 : a.w2;
  const void* ws = FFN1 ? a.sw13 : a.sw2;
  const void* x = FFN1 ? a.xq : a.hq;
  CUtensorMap tw, tws, tx;
  const uint64_t winner = a.packed ? P_BK : K;
  const uint64_t wrows = a.packed ? (uint64_t)Wrows * (K / P_BK) : Wrows;
  CUtensorMap twh, twsh, txh;
  const bool gather = FFN1 && a.gather;
  // gathered rows: one row per token, read by four-row gathers (box one row high)
  const bool xmap = gather ? pair_map(&tx, KIND_FP8, 2, x, K, a.T, 1, 1)
                           : pair_map(&tx, KIND_FP8, 2, x, K, a.rows_total, 1);
  if (!pair_map(&tw, KIND_FP8, 3, w, winner, wrows, a.E) ||
      !pair_map(&tws, KIND_FP8, 3, ws ? ws : w, winner, wrows, 1) || !xmap ||
      !pair_map(&twh, KIND_FP8, 3, w, winner, wrows, a.E, 64) ||
      !pair_map(&twsh, KIND_FP8, 3, ws ? ws : w, winner, wrows, 1, 64) ||
      !pair_map(&txh, KIND_FP8, 2, x, K, a.rows_total, 1, 64))
    return cudaErrorInvalidValue;
  PairGemm g{};
  g.items = a.items;
  g.n_items = a.n_items;
  g.max_items = a.max_items;
  g.E = a.E;
  g.nb = FFN1 ? a.I / 128 : a.K / P_N;
  g.kb1 = K / P_BK;
  g.kb2 = 0;
  g.I = a.I;
  g.packed = a.packed;
  g.act = a.act;
  g.rows_total = a.rows_total;
  g.small = pair_small_tiles() ? 1 : 0;
  g.xscale = a.xscale;
  g.w_scale = FFN1 ? a.w13_scale : a.w2_scale;
  g.ws_scale = FFN1 ? a.sw13_scale : a.sw2_scale;
  g.scale_stride = FFN1 ? 2 * a.I : a.K;
  g.hs = a.hs;
  g.row_w = a.row_w;
  g.out = FFN1 ? a.h : a.y;
  g.ldo = FFN1 ? a.I : a.K;
  g.gather = gather ? 1 : 0;
  g.src = a.src;
  g.R = a.R;
  g.T = a.T;
  g.err = a.err;
  if (FFN1) return launch_pair_gemm<KIND_FP8, EPI_SWIGLU>(tw, tws, tx, tw, tx, txh, twh, twsh, g, s);
  return launch_pair_gemm<KIND_FP8, EPI_DOWN>(tw, tws, tx, tw, tx, txh, twh, twsh, g, s);
}

}  // namespace

cudaError_t launch_ffn1_pair(const GroupedFfnArgs& a, cudaStream_t s) {
  return launch_grouped_pair<true>(a, s);
}
cudaError_t launch_ffn2_pair(const GroupedFfnArgs& a, cudaStream_t s) {
  return launch_grouped_pair<false>(a, s);
}

cudaError_t launch_dense_bf16(const DenseGemmArgs& d, cudaStream_t s) {
  // A rows [rows, K1] (+ A2 [rows, K2]); B rows [N, K1] (+ B2 [N, K2]); bf16.
  if (d.K1 % 64 || d.K2 % 64 || (d.swiglu ? d.N % 128 : d.N % P_N)) return cudaErrorInvalidValue;
  CUtensorMap tw, tx, tw2, tx2;
  const int wrows = d.swiglu ? 2 * d.N : d.N;
  if (!pair_map(&tw, KIND_BF16, 3, d.w, d.K1, wrows, 1) ||
      !pair_map(&tx, KIND_BF16, 2, d.x, d.K1, d.rows, 1))
    return cudaErrorInvalidValue;
  if (d.K2) {
    if (!pair_map(&tw2, KIND_BF16, 3, d.w2, d.K2, d.N, 1) ||
        !pair_map(&tx2, KIND_BF16, 2, d.x2, d.K2, d.rows, 1))
      return cudaErrorInvalidValue;
  } else {
    tw2 = tw;
    tx2 = tx;
  }
  PairGemm g{};
  g.items = nullptr;
  g.dense_rows = d.rows;
  g.nb = d.swiglu ? d.N / 128 : d.N / P_N;
  g.kb1 = d.K1 / 64;
  g.kb2 = d.K2 / 64;
  g.I = d.N;
  g.rows_total = d.rows;
  g.act = d.act;
  g.out = d.out;
  g.ldo = d.N;
  g.err = d.err;
  // dense launches have no small tiles: the half-box maps are never read
  if (d.swiglu) return launch_pair_gemm<KIND_BF16, EPI_SWIGLU>(tw, tw, tx, tw2, tx2, tx, tw, tw, g, s);
  return launch_pair_gemm<KIND_BF16, EPI_STORE>(tw, tw, tx, tw2, tx2, tx, tw, tw, g, s);
}

int dense_split_k(int rows, int N, int Kw) {
  // enough K ranges for every SM pair to take one when the output has few
  // tiles, each range at least eight stages of 64 K; none for larger outputs
  const long tiles = (long)((rows + 255) / 256) * ((N + P_N - 1) / P_N);
  const long pairs = device_sm_count() / 2;
  const int KB = Kw / 64;
  if (tiles <= 0 || tiles * 2 > pairs || KB < 16) return 1;  // (an empty batch: none)
  int S = (int)(pairs / tiles);
  S = S < KB / 8 ? S : KB / 8;
  const int KBs = (KB + S - 1) / S;
  return (KB + KBs - 1) / KBs;  // every range non-empty
}

cudaError_t launch_dense_bf16_f32(const void* x, int Kx, const void* w, int Kw, int rows, int N,
                                  float* out, int ksplit, int* err, cudaStream_t s) {
  // out[rows, N] fp32 = sum over Kw of x[:, k mod Kx] w[:, k]; Kx, Kw multiples of 64;
  // with ksplit > 1 (dense_split_k's value), ksplit partial blocks [rows, N]
  // back to back whose sum is out
  if (Kx % 64 || Kw % Kx || N <= 0 || rows <= 0 || ksplit < 1) return cudaErrorInvalidValue;
  if (reinterpret_cast<uintptr_t>(out) % 16) return cudaErrorInvalidValue;  // 16-byte stores
  if (ksplit > 1) {
    const int KB = Kw / 64, KBs = (KB + ksplit - 1) / ksplit;
    if ((ksplit - 1) * KBs >= KB) return cudaErrorInvalidValue;  // an empty range
  }
  CUtensorMap tw, tx;
  if (!pair_map(&tw, KIND_BF16, 3, w, Kw, N, 1) || !pair_map(&tx, KIND_BF16, 2, x, Kx, rows, 1))
    return cudaErrorInvalidValue;
  PairGemm g{};
  g.items = nullptr;
  g.dense_rows = rows;
  g.nb = (N + P_N - 1) / P_N;  // rows of w past N read as zeros; their columns are not stored
  g.kb1 = Kw / 64;
  g.kb2 = 0;
  g.a_period = Kx / 64;
  g.rows_total = rows;
  g.out = out;
  g.ldo = N;
  g.n_valid = N;
  g.ksplit = ksplit;
  g.split_stride = (size_t)rows * N;
  g.err = err;
  return launch_pair_gemm<KIND_BF16, EPI_F32>(tw, tw, tx, tw, tx, tx, tw, tw, g, s);
}

}  // namespace moe
