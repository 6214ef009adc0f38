// ffn_gemm_mx.cu -- S5/S6 with MXFP4 expert weights: grouped e2m1 x e4m3
// GEMMs with hardware block scaling (tcgen05.mma kind::mxf8f6f4.block_scale).
//
// What is computed ("Kimi K3 ... feasibility analysis", s.2.5: MXFP4 routed
// experts, group size 32, uint8 e8m0 scales; "Implementation gaps: advanced
// optimisations", s.4: two e2m1 values per byte plus a shared e8m0 scale):
//   w[n,k] = e2m1(nibble) * 2^(e8m0[n, k/32] - 127)    (low nibble = even k)
//   FFN1  g[n] = (sum_k xq[r,k] W1[n,k]) * xs[r],  u likewise with W3,
//         h[r,n] = bf16(silu(g) * u)
//   FFN2  y[r,m] = bf16(row_w[r] * (sum_n hq[r,n] W2[m,n]) * hs[r])
// The block scales are applied inside the tensor core, per 32-element block,
// so the packed weights stream from HBM at 4.25 bits per element and are never
// expanded in software.
//
// Structure as ffn_gemm.cu (persistent, one CTA per SM, swap-AB: M = 128
// weight rows, N = the item's token rows rounded up to 16):
//   warp 0      producer.  Lane 0 waits for a free stage and issues the TMA
//               loads: weights through a 16U4_ALIGN16B map (each 16 packed e2m1
//               land in 16 bytes of shared memory, the operand layout
//               kind::f8f6f4 reads; the transaction is counted in packed bytes)
//               and activation rows through a byte map, 128-byte swizzle.
//               The stage's e8m0 weight scales go to shared memory in the image
//               tcgen05.cp reads (lane l, 32-bit column c = the four k-block
//               scales of row 32c + l): with scales from moe_pack_weights that
//               image is one contiguous 512-byte block per weight block, fetched
//               by lane 0 with one bulk copy counted on the stage's transaction
//               bytes; with row-major scales all 32 lanes fetch it with 4-byte
//               cp.async whose completion arrives on the stage's full barrier
//               (cp.async.mbarrier.arrive.noinc).  No warp waits on a scale load.
//   Each stage carries two 128-row weight blocks that share the activation
//   tile: W1 and W3 rows of one output block (FFN1), or two adjacent W2 output
//   blocks (FFN2), so every stage streams 16 KB of packed weights.
//   With moe_pack_weights' order the two blocks of a stage are one 256-row
//   TMA box and their scales one 1 KB bulk copy: a stage costs the producer
//   three copies, which keeps its issue rate off the critical path.  Each next
//   tile's scales are prefetched into L2 a tile ahead.
//   warp 1      MMA issuer: per stage, a proxy fence (row-major scales are
//               written through the generic proxy), tcgen05.cp of each weight block's
//               scales into its tensor-memory slot (32x128b replicated to the
//               four lane quarters), then 4 MMAs of K=32 per block, the scale
//               byte picked by the descriptor's scale-factor id.  tcgen05.cp and
//               tcgen05.mma from one thread execute in issue order.  The
//               activation scales are a constant 2^0, copied once.
//   warps 2-5   epilogue.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>

#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int MX_BM = 128;         // weight rows per tile
constexpr int MX_BK = 128;         // K elements per stage
constexpr int MX_A_SMEM = MX_BM * MX_BK;          // 16 KB unpacked in shared memory
constexpr int MX_A_TX = MX_BM * MX_BK / 2;        // 8 KB packed from global memory
constexpr int MX_THREADS = 192;
constexpr int MX_SF_SLOT = 512;  // one weight block's scales for one stage: 32 lanes x 16 B
constexpr int MX_SMEM_BUDGET = 220 * 1024;

constexpr int mx_min(int a, int b) { return a < b ? a : b; }

template <bool FFN1, int BN>
struct MxCfg {
  static constexpr int NA = 2;  // 128-row weight blocks per stage: W1|W3 (FFN1), two W2 blocks (FFN2)
  static constexpr int B_BYTES = BN * MX_BK;
  static constexpr int STAGE_SMEM = NA * MX_A_SMEM + B_BYTES;
  static constexpr int STAGE_TX = NA * MX_A_TX + B_BYTES;
  static constexpr int STAGES = mx_min(MX_SMEM_BUDGET / STAGE_SMEM, 8);
  static constexpr int ACC_COLS = NA * BN;
  static constexpr int ACC_STAGES = 2;
  static constexpr int SFB_COL = ACC_STAGES * ACC_COLS;      // 8 columns of 2^0
  static constexpr int SFA_COL = SFB_COL + 8;                // NA x 4 columns per stage
  static constexpr int TMEM_USED = SFA_COL + STAGES * NA * 4;
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_STAGES + 1;
  static constexpr int SF_BYTES = STAGES * NA * MX_SF_SLOT + MX_SF_SLOT;  // + the 2^0 block
  static constexpr int SMEM = 1024 + STAGES * STAGE_SMEM + SF_BYTES + NUM_BARS * 8 + 16 + STAGES * 4;
  static_assert(TMEM_USED <= TMEM_COLS, "tensor memory budget");
  static_assert(B_BYTES % 1024 == 0, "operand tiles keep 1024-byte alignment");
  static_assert(SMEM <= 232448, "dynamic shared memory per block");
};

// kind::mxf8f6f4 block-scaled instruction descriptor: A = e2m1 (5), B = e4m3
// (0), both K-major, N >> 3 at bits 17-22, e8m0 scales (bit 23), M >> 4 at
// bits 24-28; scale-factor byte ids for B (bits 4-5) and A (bits 29-30).
__device__ __forceinline__ uint32_t idesc_mx(uint32_t M, uint32_t N, uint32_t sf_id) {
  return (sf_id << 4) | (5u << 7) | (0u << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24) |
         (sf_id << 29);
}

__device__ __forceinline__ void mma_mx(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

// 4-byte asynchronous global -> shared copy (both addresses 4-byte aligned).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}


// Shared-memory descriptor of a 32-row x 16-byte scale block, no swizzle: 8-row
// core matrices of 128 contiguous bytes, 128 bytes apart (both offset fields).
__device__ __forceinline__ uint64_t sf_desc(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 16) |
         ((uint64_t)(128 >> 4) << 32) | (1ull << 46);
}

// The same for one block of a stage's scales in moe_pack_weights' order
// ([4 j][2 blocks][8 rows][16 B]): its 8-row core matrices are 256 bytes apart.
__device__ __forceinline__ uint64_t sf_desc_g256(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(256 >> 4) << 16) |
         ((uint64_t)(256 >> 4) << 32) | (1ull << 46);
}

// Both blocks' scales of a stage as one 128-row x 32-byte source (the 1 KB
// of moe_pack_weights' order once per lane quarter): 8-row core matrices 256
// bytes apart (stride offset), the second block's 16 bytes of each row 128
// bytes on (leading offset).
__device__ __forceinline__ uint64_t sf_desc_pair(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 16) |
         ((uint64_t)(256 >> 4) << 32) | (1ull << 46);
}

// Copy a 32-row x 128-bit block from shared memory to tensor memory columns
// [taddr, taddr + 4) of all four lane quarters (row l -> lane l of each quarter).
__device__ __forceinline__ void tmem_cp_32x128_x4(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

template <bool FFN1, int BN>
__global__ void __launch_bounds__(MX_THREADS, 1)
    grouped_mx_kernel(const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_x, const GroupedFfnArgs a) {
  using C = MxCfg<FFN1, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sf = smem + C::STAGES * C::STAGE_SMEM;  // [STAGES][NA][512 B], then the 2^0 block
  uint64_t* bars = reinterpret_cast<uint64_t*>(sf + C::SF_BYTES);
  uint64_t* full = bars;                    // weights, activations and scales landed
  uint64_t* empty = bars + C::STAGES;       // MMAs done with the stage
  uint64_t* tfull = bars + 2 * C::STAGES;
  uint64_t* tempty = tfull + C::ACC_STAGES;
  uint64_t* drain = tempty + C::ACC_STAGES;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint32_t* s_issued = s_tmem + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  {
    // activation scale block: every byte e8m0 127 = 2^0
    uint32_t* one = reinterpret_cast<uint32_t*>(sf + C::STAGES * C::NA * MX_SF_SLOT);
    for (int i = threadIdx.x; i < MX_SF_SLOT / 4; i += blockDim.x) one[i] = 0x7F7F7F7Fu;
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // TMA expect_tx (+ one cp.async arrival per producer lane for row-major scales)
      mbar_init(smem_u32(&full[s]), a.packed ? 1 : 1 + 32);
      mbar_init(smem_u32(&empty[s]), 1);
      s_issued[s] = 0;
    }
    for (int s = 0; s < C::ACC_STAGES; ++s) {
      mbar_init(smem_u32(&tfull[s]), 1);
      mbar_init(smem_u32(&tempty[s]), 4);
    }
    mbar_init(smem_u32(drain), 1);
    *s_abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
  }
  if (warp == 1) tmem_alloc(smem_u32(s_tmem), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_wait();  // the previous kernel's outputs are complete and visible

  const int NB = FFN1 ? a.I / MX_BM : a.K / (2 * MX_BM);  // tiles per item
  const int Kel = FFN1 ? a.K : a.I;  // reduction width in elements
  const int KB = Kel / MX_BK;
  const int n_items = min(*a.n_items, a.max_items);
  const int n_tiles = n_items * NB;
  // first weight row of block blk (0, 1) of tile column nb
  auto block_row = [&](int blk, int nb) {
    return FFN1 ? blk * a.I + nb * MX_BM : (2 * nb + blk) * MX_BM;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // e8m0 scales [E][rows][K/32] (passed through the fp32 scale fields)
    const uint8_t* scales = reinterpret_cast<const uint8_t*>(FFN1 ? a.w13_scale : a.w2_scale);
    const int wrows = FFN1 ? 2 * a.I : a.K;  // weight rows per expert
    const int sbytes = Kel / 32;             // scale bytes per weight row
    const bool sf_pf_ok = (reinterpret_cast<uintptr_t>(scales) & 15) == 0;  // bulk prefetch alignment
    // packed (moe_pack_weights): weights [E][NB][KB][2 blocks][128 rows][64 B] and
    // scales [E][NB][KB][4][2 blocks][8][16 B], so a stage is one 256-row box + 1 KB
    auto sf_packed = [&](int e, int nb, int kb) {
      return scales + (((size_t)e * NB + nb) * KB + kb) * (C::NA * MX_SF_SLOT);
    };
    int stage = 0;
    uint32_t phase = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
      // the whole warp takes the abort decision lane 0 reads (shuffles below need all lanes)
      if (__shfl_sync(0xffffffffu, lane == 0 ? *s_abort : 0, 0)) break;
      const int item = tile / NB, nb = tile - item * NB;
      const int4 it = a.items[item];
      const uint8_t* sb = scales + (size_t)it.x * wrows * sbytes;
      // L2 lookahead: the next tile's item, and its scale rows (one contiguous
      // 128 x K/32-byte range per weight block) fetched a whole tile early
      const int ntile = tile + gridDim.x;
      const bool has_next = ntile < n_tiles;
      const int nnb = has_next ? ntile % NB : 0;
      const int4 itn = has_next ? a.items[ntile / NB] : it;
      if (lane == 0 && has_next && sf_pf_ok) {
#pragma unroll
        for (int blk = 0; blk < C::NA; ++blk) {
          if (a.packed) {
            if (blk == 0)
              prefetch_l2(sf_packed(itn.x, nnb, 0), (uint32_t)(KB * C::NA * MX_SF_SLOT));
          } else
            prefetch_l2(scales + ((size_t)itn.x * wrows + block_row(blk, nnb)) * sbytes,
                        (uint32_t)(MX_BM * sbytes));
        }
      }
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        int got = 1;
        if (lane == 0) got = mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, a.err, s_abort) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&full[stage]);
        const uint32_t sfs = smem_u32(sf + stage * C::NA * MX_SF_SLOT);
        if (!a.packed) {
          // row-major scales: lane l copies rows 32c + l of each block (4 bytes
          // each) into moe_pack_weights' order, word (l / 8, blk, l % 8, c)
#pragma unroll
          for (int blk = 0; blk < C::NA; ++blk) {
            const uint8_t* src = sb + (size_t)(block_row(blk, nb) + lane) * sbytes + kb * 4;
            const uint32_t dst = sfs + (lane >> 3) * 256 + blk * 128 + (lane & 7) * 16;
#pragma unroll
            for (int c = 0; c < 4; ++c) cp_async4(dst + c * 4, src + (size_t)(32 * c) * sbytes);
          }
          cp_async_arrive_noinc(fb);
        }
        if (lane == 0) {
          const uint32_t st = smem_u32(smem + stage * C::STAGE_SMEM);
          mbar_arrive_expect_tx(fb, C::STAGE_TX + (a.packed ? C::NA * MX_SF_SLOT : 0));
          if (a.packed) {
            bulk_load(sfs, sf_packed(it.x, nb, kb), C::NA * MX_SF_SLOT, fb);
            tma_load_3d(st, &tm_w, 0, C::NA * MX_BM * (nb * KB + kb), it.x, fb);  // both blocks
          } else {
            tma_load_3d(st, &tm_w, kb * MX_BK, block_row(0, nb), it.x, fb);
            tma_load_3d(st + MX_A_SMEM, &tm_w, kb * MX_BK, block_row(1, nb), it.x, fb);
          }
          tma_load_2d(st + C::NA * MX_A_SMEM, &tm_x, kb * MX_BK, it.y, fb);
          s_issued[stage] = phase + 1u;
        }
        __syncwarp();
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
    cp_async_wait_all();  // no copy into this CTA's shared memory outlives it
    if (lane == 0 && *s_abort) {
      for (int s = 0; s < C::STAGES; ++s)
        if (s_issued[s]) mbar_wait_drain(smem_u32(&full[s]), s_issued[s] - 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, it_local = 0;
      uint32_t phase = 0;
      bool issued_any = false;
      const uint32_t sfb = tmem + C::SFB_COL;
      {
        const uint64_t one = sf_desc(smem_u32(sf + C::STAGES * C::NA * MX_SF_SLOT));
        tmem_cp_32x128_x4(sfb, one);
        tmem_cp_32x128_x4(sfb + 4, one);
      }
      for (int tile = blockIdx.x; tile < n_tiles && !*s_abort; tile += gridDim.x, ++it_local) {
        const int item = tile / NB;
        const int rows = a.items[item].z;
        const int n = min(BN, (rows + 15) & ~15);
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
          fence_proxy_async_smem();
          const uint32_t a0 = smem_u32(smem + stage * C::STAGE_SMEM);
          const uint32_t b0 = a0 + C::NA * MX_A_SMEM;
          const uint32_t sfa = tmem + C::SFA_COL + stage * C::NA * 4;
          const uint32_t sfs = smem_u32(sf + stage * C::NA * MX_SF_SLOT);
#pragma unroll
          for (int blk = 0; blk < C::NA; ++blk)
            tmem_cp_32x128_x4(sfa + blk * 4, sf_desc_g256(sfs + blk * 128));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t idesc = idesc_mx(MX_BM, n, kk);
            const uint64_t bdesc = smem_desc_sw128(b0 + kk * 32);
            const uint32_t accum = (kb | kk) ? 1u : 0u;
            mma_mx(d0, smem_desc_sw128(a0 + kk * 32), bdesc, idesc, sfa, sfb, accum);
            mma_mx(d0 + BN, smem_desc_sw128(a0 + MX_A_SMEM + kk * 32), bdesc, idesc, sfa + 4, sfb,
                   accum);
          }
          issued_any = true;
          mma_commit(smem_u32(&empty[stage]));
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&tfull[acc]));
      }
      if (*s_abort && issued_any) {
        mma_commit(smem_u32(drain));
        mbar_wait_drain(smem_u32(drain), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    int it_local = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it_local) {
      const int item = tile / NB, nb = tile - item * NB;
      const int4 it = a.items[item];
      const int row0 = it.y, rows = it.z;
      const int acc = it_local % C::ACC_STAGES;
      const uint32_t acc_phase = (uint32_t)(it_local / C::ACC_STAGES) & 1u;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(smem_u32(&tfull[acc]), acc_phase, a.err, s_abort) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + acc * C::ACC_COLS;
      const int f = nb * MX_BM + q * 32 + lane;            // FFN1: h column
      const int f2 = 2 * nb * MX_BM + q * 32 + lane;       // FFN2: y column of block 0
      if (FFN1) {
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
              const float xs = a.xscale[row];
              const float g = __uint_as_float(vg[j]) * xs;
              const float u = __uint_as_float(vu[j]) * xs;
              hout[(size_t)row * a.I + f] = (uint16_t)f32_to_bf16_bits(gated_act(a.act, g, u));
            }
          }
        }
      } else {
        uint16_t* yout = static_cast<uint16_t*>(a.y);
        for (int c0 = 0; c0 < rows; c0 += 16) {
          uint32_t v0[16], v1[16];
          __syncwarp();
          tmem_ld16(tbase + c0, v0);
          tmem_ld16(tbase + BN + c0, v1);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = c0 + j;
            const int row = row0 + r;
            if (r < rows && (unsigned)row < (unsigned)a.rows_total) {
              const float rw = a.row_w ? a.row_w[row] : 1.0f;
              const float hs = a.hs[row];
              uint16_t* yr = yout + (size_t)row * a.K + f2;
              yr[0] = (uint16_t)f32_to_bf16_bits((__uint_as_float(v0[j]) * hs) * rw);
              yr[MX_BM] = (uint16_t)f32_to_bf16_bits((__uint_as_float(v1[j]) * hs) * rw);
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

// ---------------------------------------------------------------- SM pairs
// The same tiles on pairs of SMs (tcgen05 cta_group::2).  The pair's MMAs
// cover 256 weight rows, 128 from each CTA's shared memory and tensor memory,
// and the item's N token rows, N/2 staged by each CTA: each SM stages half of
// the activation tile that the single-SM kernel stages whole, so a stage moves
// ~15% fewer bytes through shared memory (the bound of the single-SM kernel).
// CTA r of a pair runs what would be the single-SM tile column 2p + r (FFN1:
// W1 and W3 blocks 2p + r; FFN2: W2 blocks 2(2p + r) and 2(2p + r) + 1): it
// loads that tile's 256-row weight box and its two scale images, and runs that
// tile's epilogue on its own tensor memory.  Weights and scales must be in
// moe_pack_weights' order; every copy is a TMA load counted on the even CTA's
// full barrier.  Each CTA loads a stage's 1 KB of scales once per
// tensor-memory lane quarter, and the even CTA's warp 1 copies both blocks'
// scales of both CTAs into their tensor memory with one
// tcgen05.cp.cta_group::2.128x256b per stage (each CTA's from its own shared
// memory, same offsets), then issues the pair's MMAs; its commits arrive on
// both CTAs' barriers; both epilogues release accumulators on the even CTA's
// barrier.  All waits are bounded as in the single-SM kernel.
//
// What bounds it: the weight loads and the MMAs together, neither alone.  A
// block-scaled K = 32 MMA holds the tensor pipe a fixed time whatever its N
// (155 cycles for 128 rows per SM and N = 16 to 256 in a timing probe), a
// tcgen05.cp ~60-90 cycles whatever its shape, hence one 128x256b copy per
// stage rather than one 32x128b.warpx4 copy per block (FFN1 2.13 -> 2.02 ms,
// FFN2 1.07 -> 1.02 ms).  Timing-only variants on T=4096, L=3584, I=3072,
// E=896 top-16, FFN1: no MMAs and no scale copies 1.65 ms; copies only 1.66;
// MMAs only 1.89; MMAs and two copies per stage 2.13; one weight block per
// stage (4 MMAs, 1 copy) 1.70; N = 16 2.04; one copy per stage 2.01.  With
// the operands swapped on single SMs (128 token rows as A, the stage's 256
// weight rows as N: four MMAs per stage instead of eight, parity-green) FFN1
// took 2.01-2.05 ms and FFN2 1.10: halving the instructions changes nothing,
// since either way a stage moves 85-100 KB through shared memory (the e2m1
// operand lands unpacked, 32 KB per 16 KB from HBM, and the MMAs read it all
// back).  Changes that did not help: packed weight loads instead of unpacked
// ones, or an L2 prefetch 4 or 8 stages ahead (no change); each stage's
// copies issued one stage ahead, after waiting for that stage's data (2.40:
// the MMAs wait one load longer); the scales written by four more warps with
// tcgen05.st instead of tcgen05.cp (3.98: the stores wait for the MMAs in
// flight, so every stage drains the pipe).
template <bool FFN1, int BN>
struct MxPairCfg {
  static constexpr int NA = 2;
  static constexpr int BH = BN / 2;  // activation rows staged per CTA
  static constexpr int B_BYTES = BH * MX_BK;
  static constexpr int STAGE_SMEM = NA * MX_A_SMEM + B_BYTES;
  static constexpr int SF_STAGE = 4 * NA * MX_SF_SLOT;  // the stage's 1 KB once per lane quarter
  static constexpr int STAGE_TX = NA * MX_A_TX + B_BYTES + SF_STAGE;  // per CTA
  static constexpr int STAGES = mx_min((MX_SMEM_BUDGET - MX_SF_SLOT) / (STAGE_SMEM + SF_STAGE), 8);
  static constexpr int ACC_COLS = NA * BN;
  static constexpr int ACC_STAGES = 2;
  static constexpr int SFB_COL = ACC_STAGES * ACC_COLS;
  static constexpr int SFA_COL = SFB_COL + 8;
  static constexpr int TMEM_USED = SFA_COL + STAGES * NA * 4;
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_STAGES + 1;
  static constexpr int SF_BYTES = STAGES * SF_STAGE + MX_SF_SLOT;
  static constexpr int SMEM = 1024 + STAGES * STAGE_SMEM + SF_BYTES + NUM_BARS * 8 + 16 + STAGES * 4;
  static_assert(TMEM_USED <= TMEM_COLS, "tensor memory budget");
  static_assert(B_BYTES % 1024 == 0, "operand tiles keep 1024-byte alignment");
  static_assert(SMEM <= 232448, "dynamic shared memory per block");
};

__device__ __forceinline__ void mma_mx_pair(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                            uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

// Both CTAs: a 128-row x 256-bit block from each CTA's shared memory (same
// offset) into tensor-memory lanes 0..127, columns [taddr, taddr + 8).
__device__ __forceinline__ void tmem_cp_128x256_pair(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

// Both CTAs: a 32-row x 128-bit block from each CTA's shared memory (same
// offset) into its own tensor memory, replicated to the four lane quarters.
__device__ __forceinline__ void tmem_cp_32x128_x4_pair(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}

template <bool FFN1, int BN>
__global__ void __launch_bounds__(MX_THREADS, 1)
    grouped_mx_pair_kernel(const __grid_constant__ CUtensorMap tm_w,
                           const __grid_constant__ CUtensorMap tm_x,
                           const __grid_constant__ CUtensorMap tm_s, const GroupedFfnArgs a) {
  using C = MxPairCfg<FFN1, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sf = smem + C::STAGES * C::STAGE_SMEM;  // [STAGES][4 quarters][1 KB], then the 2^0 block
  uint64_t* bars = reinterpret_cast<uint64_t*>(sf + C::SF_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tfull = bars + 2 * C::STAGES;
  uint64_t* tempty = tfull + C::ACC_STAGES;
  uint64_t* drain = tempty + C::ACC_STAGES;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint32_t* s_issued = s_tmem + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  {
    uint32_t* one = reinterpret_cast<uint32_t*>(sf + C::STAGES * C::SF_STAGE);
    for (int i = threadIdx.x; i < MX_SF_SLOT / 4; i += blockDim.x) one[i] = 0x7F7F7F7Fu;
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
      s_issued[s] = 0;
    }
    for (int s = 0; s < C::ACC_STAGES; ++s) {
      mbar_init(smem_u32(&tfull[s]), 1);
      mbar_init(smem_u32(&tempty[s]), 8);  // 4 epilogue warps in each CTA
    }
    mbar_init(smem_u32(drain), 1);
    *s_abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_s);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(s_tmem), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers and the 2^0 blocks of both CTAs exist before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_wait();  // the previous kernel's outputs are complete and visible

  const int NB = FFN1 ? a.I / MX_BM : a.K / (2 * MX_BM);  // single-SM tile columns per item
  const int NP = NB / 2;                                 // pair tiles per item
  const int Kel = FFN1 ? a.K : a.I;
  const int KB = Kel / MX_BK;
  const int n_items = min(*a.n_items, a.max_items);
  const int n_tiles = n_items * NP;
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = cluster; tile < n_tiles && !*s_abort; tile += n_clusters) {
        const int item = tile / NP, nb = 2 * (tile - item * NP) + (int)rank;
        const int4 it = a.items[item];
        const int half = min(BN, (it.z + 15) & ~15) / 2;  // this item's N / 2
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, a.err, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t st = smem_u32(smem + stage * C::STAGE_SMEM);
          const uint32_t sfs = smem_u32(sf + stage * C::SF_STAGE);
          const uint32_t fb_leader = mapa_shared(smem_u32(&full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(smem_u32(&full[stage]), 2 * C::STAGE_TX);
          tma_load_3d_pair(st, &tm_w, 0, C::NA * MX_BM * (nb * KB + kb), it.x, fb_leader);
          tma_load_2d_pair(st + C::NA * MX_A_SMEM, &tm_x, kb * MX_BK, it.y + (int)rank * half,
                           fb_leader);
#pragma unroll
          for (int q = 0; q < 4; ++q)  // the stage's scales once per tensor-memory lane quarter
            tma_load_2d_pair(sfs + q * C::NA * MX_SF_SLOT, &tm_s, 0,
                             ((it.x * NB + nb) * KB + kb) * C::NA, fb_leader);
          s_issued[stage] = phase + 1u;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (*s_abort && leader) {  // the pair's loads complete on the even CTA's barriers
        for (int s = 0; s < C::STAGES; ++s)
          if (s_issued[s]) mbar_wait_drain(smem_u32(&full[s]), s_issued[s] - 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      int stage = 0, it_local = 0;
      uint32_t phase = 0;
      bool issued_any = false;
      const uint32_t sfb = tmem + C::SFB_COL;
      {
        const uint64_t one = sf_desc(smem_u32(sf + C::STAGES * C::SF_STAGE));
        tmem_cp_32x128_x4_pair(sfb, one);
        tmem_cp_32x128_x4_pair(sfb + 4, one);
      }
      for (int tile = cluster; tile < n_tiles && !*s_abort; tile += n_clusters, ++it_local) {
        const int item = tile / NP;
        const int n = min(BN, (a.items[item].z + 15) & ~15);
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
          const uint32_t a0 = smem_u32(smem + stage * C::STAGE_SMEM);
          const uint32_t b0 = a0 + C::NA * MX_A_SMEM;
          const uint32_t sfa = tmem + C::SFA_COL + stage * C::NA * 4;
          // both blocks' scales in one copy: lanes 32q + l, columns sfa .. sfa + 7
          tmem_cp_128x256_pair(sfa, sf_desc_pair(smem_u32(sf + stage * C::SF_STAGE)));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t idesc = idesc_mx(2 * MX_BM, n, kk);
            const uint64_t bdesc = smem_desc_sw128(b0 + kk * 32);
            const uint32_t accum = (kb | kk) ? 1u : 0u;
            mma_mx_pair(d0, smem_desc_sw128(a0 + kk * 32), bdesc, idesc, sfa, sfb, accum);
            mma_mx_pair(d0 + BN, smem_desc_sw128(a0 + MX_A_SMEM + kk * 32), bdesc, idesc, sfa + 4,
                        sfb, accum);
          }
          issued_any = true;
          mma_commit_pair(smem_u32(&empty[stage]), 0x3);
          if (++stage == C::STAGES) {
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
    const uint32_t tempty_leader0 = mapa_shared(smem_u32(&tempty[0]), 0);
    int it_local = 0;
    for (int tile = cluster; tile < n_tiles; tile += n_clusters, ++it_local) {
      const int item = tile / NP, nb = 2 * (tile - item * NP) + (int)rank;
      const int4 it = a.items[item];
      const int row0 = it.y, rows = it.z;
      const int acc = it_local % C::ACC_STAGES;
      const uint32_t acc_phase = (uint32_t)(it_local / C::ACC_STAGES) & 1u;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(smem_u32(&tfull[acc]), acc_phase, a.err, s_abort) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + acc * C::ACC_COLS;
      const int f = nb * MX_BM + q * 32 + lane;       // FFN1: h column
      const int f2 = 2 * nb * MX_BM + q * 32 + lane;  // FFN2: y column of block 0
      if (FFN1) {
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
              const float xs = a.xscale[row];
              const float g = __uint_as_float(vg[j]) * xs;
              const float u = __uint_as_float(vu[j]) * xs;
              hout[(size_t)row * a.I + f] = (uint16_t)f32_to_bf16_bits(gated_act(a.act, g, u));
            }
          }
        }
      } else {
        uint16_t* yout = static_cast<uint16_t*>(a.y);
        for (int c0 = 0; c0 < rows; c0 += 16) {
          uint32_t v0[16], v1[16];
          __syncwarp();
          tmem_ld16(tbase + c0, v0);
          tmem_ld16(tbase + BN + c0, v1);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = c0 + j;
            const int row = row0 + r;
            if (r < rows && (unsigned)row < (unsigned)a.rows_total) {
              const float rw = a.row_w ? a.row_w[row] : 1.0f;
              const float hs = a.hs[row];
              uint16_t* yr = yout + (size_t)row * a.K + f2;
              yr[0] = (uint16_t)f32_to_bf16_bits((__uint_as_float(v0[j]) * hs) * rw);
              yr[MX_BM] = (uint16_t)f32_to_bf16_bits((__uint_as_float(v1[j]) * hs) * rw);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      // the accumulator is free once this warp's tensor-memory loads are done
      // (each group waited above); the output stores need not be complete
      if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader0 + acc * 8);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while its peer may still read its shared memory
  pdl_release();  // the next kernel may start launching: this one is done
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

template <bool FFN1, int BN>
cudaError_t launch_mx_impl(const GroupedFfnArgs& a, cudaStream_t s) {
  using C = MxCfg<FFN1, BN>;
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorInvalidValue;
  const int Kel = FFN1 ? a.K : a.I;
  const int Wrows = FFN1 ? 2 * a.I : a.K;
  const void* w = FFN1 ? a.w13 : a.w2;
  const void* x = FFN1 ? a.xq : a.hq;
  const void* sc = FFN1 ? a.w13_scale : a.w2_scale;
  // 4-byte cp.async (row-major scales) or 16-byte bulk copies (packed scales)
  if (reinterpret_cast<uintptr_t>(sc) % (a.packed ? 16 : 4)) return cudaErrorInvalidValue;
  if (!FFN1 && a.K % (2 * MX_BM)) return cudaErrorInvalidValue;           // two W2 blocks per tile
  CUtensorMap tw, tx;
  {
    // packed e2m1 weights [E][rows][Kel/2 bytes], unpacked to 16 bytes per 16 values;
    // moe_pack_weights' order is [E][rows/256 * Kel/128 * 256 rows][64 bytes], read as
    // one box of both blocks of a stage
    const cuuint64_t inner = a.packed ? MX_BK : Kel;
    const cuuint64_t wr = a.packed ? (cuuint64_t)Wrows * (Kel / MX_BK) : Wrows;
    cuuint64_t dims[3] = {inner, wr, (cuuint64_t)a.E};
    cuuint64_t strides[2] = {inner / 2, inner / 2 * wr};
    cuuint32_t box[3] = {MX_BK, (cuuint32_t)(a.packed ? 2 * MX_BM : MX_BM), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(w), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)Kel, (cuuint64_t)a.rows_total};
    cuuint64_t strides[1] = {(cuuint64_t)Kel};
    cuuint32_t box[2] = {MX_BK, (cuuint32_t)BN};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e = ensure_max_smem<grouped_mx_kernel<FFN1, BN>>(C::SMEM);
  if (e != cudaSuccess) return e;
  count_launch();
  e = launch_kernel(grouped_mx_kernel<FFN1, BN>, dim3(device_sm_count()), dim3(MX_THREADS), C::SMEM,
                    s, 1, tw, tx, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool FFN1, int BN>
cudaError_t launch_mx_pair_impl(const GroupedFfnArgs& a, cudaStream_t s) {
  using C = MxPairCfg<FFN1, BN>;
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorInvalidValue;
  const int Kel = FFN1 ? a.K : a.I;
  const int Wrows = FFN1 ? 2 * a.I : a.K;
  const int NB = FFN1 ? a.I / MX_BM : a.K / (2 * MX_BM);
  const void* w = FFN1 ? a.w13 : a.w2;
  const void* x = FFN1 ? a.xq : a.hq;
  const void* sc = FFN1 ? a.w13_scale : a.w2_scale;
  if (!a.packed || NB % 2 || (!FFN1 && a.K % (2 * MX_BM)) ||
      reinterpret_cast<uintptr_t>(sc) % 16)
    return cudaErrorInvalidValue;
  CUtensorMap tw, tx, ts;
  {
    // moe_pack_weights' order [E][rows/256 * Kel/128 * 256 rows][64 bytes]: one
    // 256-row box per stage, each 16 packed e2m1 unpacked to 16 bytes
    const cuuint64_t wr = (cuuint64_t)Wrows * (Kel / MX_BK);
    cuuint64_t dims[3] = {MX_BK, wr, (cuuint64_t)a.E};
    cuuint64_t strides[2] = {MX_BK / 2, MX_BK / 2 * wr};
    cuuint32_t box[3] = {MX_BK, 2 * MX_BM, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(w), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // activation rows: half of the item's rows per CTA
    cuuint64_t dims[2] = {(cuuint64_t)Kel, (cuuint64_t)a.rows_total};
    cuuint64_t strides[1] = {(cuuint64_t)Kel};
    cuuint32_t box[2] = {MX_BK, (cuuint32_t)C::BH};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // packed scale images [E][NB][KB][2][512 B] as rows of 128 words; a
    // stage's two images are one 2-row box
    cuuint64_t dims[2] = {MX_SF_SLOT / 4, (cuuint64_t)a.E * NB * (Kel / MX_BK) * C::NA};
    cuuint64_t strides[1] = {MX_SF_SLOT};
    cuuint32_t box[2] = {MX_SF_SLOT / 4, (cuuint32_t)C::NA};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(sc), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e = ensure_max_smem<grouped_mx_pair_kernel<FFN1, BN>>(C::SMEM);
  if (e != cudaSuccess) return e;
  count_launch();
  e = launch_kernel(grouped_mx_pair_kernel<FFN1, BN>, dim3((device_sm_count() / 2) * 2),
                    dim3(MX_THREADS), C::SMEM, s, 2, tw, tx, ts, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool FFN1>
cudaError_t launch_mx_bn(const GroupedFfnArgs& a, cudaStream_t s) {
  if (mx_pair_eligible(a, FFN1)) {
    switch (a.BN) {
      case 32: return launch_mx_pair_impl<FFN1, 32>(a, s);
      case 64: return launch_mx_pair_impl<FFN1, 64>(a, s);
      case 96: return launch_mx_pair_impl<FFN1, 96>(a, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.BN) {
    case 32: return launch_mx_impl<FFN1, 32>(a, s);
    case 64: return launch_mx_impl<FFN1, 64>(a, s);
    case 96: return launch_mx_impl<FFN1, 96>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// SM pairs need moe_pack_weights' order and an even number of single-SM tile
// columns; tuning().mx_1cta forces the single-SM kernel.
bool mx_pair_eligible(const GroupedFfnArgs& a, bool ffn1) {
  if (tuning().mx_1cta) return false;
  const int nb = ffn1 ? a.I / MX_BM : a.K / (2 * MX_BM);
  return a.packed && nb % 2 == 0 && (ffn1 || a.K % (2 * MX_BM) == 0);
}

cudaError_t launch_ffn1_mx(const GroupedFfnArgs& a, cudaStream_t s) { return launch_mx_bn<true>(a, s); }
cudaError_t launch_ffn2_mx(const GroupedFfnArgs& a, cudaStream_t s) { return launch_mx_bn<false>(a, s); }

}  // namespace moe
