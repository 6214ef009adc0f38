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
// weight rows, N = the item's token rows rounded up to 16), plus four
// scale-writer warps:
//   warp 0      TMA producer: weights through a 16U4_ALIGN16B map (each 16
//               packed e2m1 land in 16 bytes of shared memory, the operand
//               layout kind::f8f6f4 reads; the transaction is counted in packed
//               bytes), activation rows through a byte map; 128-byte swizzle.
//   warp 1      MMA issuer: 4 MMAs of K=32 per 128-element stage, scale byte
//               k selected by the descriptor's scale-factor ids.
//   warps 2-5   epilogue.
//   warps 6-9   scale writers: for each stage, the e8m0 scales of the stage's
//               weight rows go to tensor memory with tcgen05.st (row r of the
//               128-row block at lane r mod 32 of every lane quarter, column
//               r / 32, byte = k-block within the stage); the activation
//               scales are a constant 2^0.
#include <cudaTypedefs.h>

#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int MX_BM = 128;         // weight rows per tile
constexpr int MX_BK = 128;         // K elements per stage
constexpr int MX_A_SMEM = MX_BM * MX_BK;          // 16 KB unpacked in shared memory
constexpr int MX_A_TX = MX_BM * MX_BK / 2;        // 8 KB packed from global memory
constexpr int MX_THREADS = 320;
constexpr int MX_SMEM_BUDGET = 220 * 1024;

constexpr int mx_min(int a, int b) { return a < b ? a : b; }

template <bool FFN1, int BN>
struct MxCfg {
  static constexpr int NA = FFN1 ? 2 : 1;
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
  static constexpr int NUM_BARS = 3 * STAGES + 2 * ACC_STAGES + 1;
  static constexpr int SMEM = 1024 + STAGES * STAGE_SMEM + NUM_BARS * 8 + 16 + STAGES * 4;
  static_assert(TMEM_USED <= TMEM_COLS, "tensor memory budget");
  static_assert(B_BYTES % 1024 == 0, "operand tiles keep 1024-byte alignment");
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

__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
               : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
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
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_SMEM);
  uint64_t* full = bars;                    // TMA data landed
  uint64_t* sfull = bars + C::STAGES;       // scales in tensor memory
  uint64_t* empty = bars + 2 * C::STAGES;   // MMAs done with the stage
  uint64_t* tfull = bars + 3 * C::STAGES;
  uint64_t* tempty = tfull + C::ACC_STAGES;
  uint64_t* drain = tempty + C::ACC_STAGES;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint32_t* s_issued = s_tmem + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&sfull[s]), 4);
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

  const int NB = FFN1 ? a.I / MX_BM : a.K / MX_BM;
  const int Kel = FFN1 ? a.K : a.I;  // reduction width in elements
  const int KB = Kel / MX_BK;
  const int n_items = min(*a.n_items, a.max_items);
  const int n_tiles = n_items * NB;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < n_tiles && !*s_abort; tile += gridDim.x) {
        const int item = tile / NB, nb = tile - item * NB;
        const int4 it = a.items[item];
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, a.err, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t st = smem_u32(smem + stage * C::STAGE_SMEM);
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, C::STAGE_TX);
          tma_load_3d(st, &tm_w, kb * MX_BK, nb * MX_BM, it.x, fb);
          if (FFN1) tma_load_3d(st + MX_A_SMEM, &tm_w, kb * MX_BK, a.I + nb * MX_BM, it.x, fb);
          tma_load_2d(st + C::NA * MX_A_SMEM, &tm_x, kb * MX_BK, it.y, fb);
          s_issued[stage] = phase + 1u;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (*s_abort) {
        for (int s = 0; s < C::STAGES; ++s)
          if (s_issued[s]) mbar_wait_drain(smem_u32(&full[s]), s_issued[s] - 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, it_local = 0;
      uint32_t phase = 0;
      bool issued_any = false;
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
          if (!mbar_wait(smem_u32(&full[stage]), phase, a.err, s_abort) ||
              !mbar_wait(smem_u32(&sfull[stage]), phase, a.err, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * C::STAGE_SMEM);
          const uint32_t b0 = a0 + C::NA * MX_A_SMEM;
          const uint32_t sfa = tmem + C::SFA_COL + stage * C::NA * 4;
          const uint32_t sfb = tmem + C::SFB_COL;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t idesc = idesc_mx(MX_BM, n, kk);
            const uint64_t bdesc = smem_desc_sw128(b0 + kk * 32);
            const uint32_t accum = (kb | kk) ? 1u : 0u;
            mma_mx(d0, smem_desc_sw128(a0 + kk * 32), bdesc, idesc, sfa, sfb, accum);
            if (FFN1)
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
  } else if (warp >= 6) {
    // ------------------------------------------------------------ scale writers
    const int q = warp & 3;
    const uint32_t lq = (uint32_t)(q * 32) << 16;
    {
      const uint32_t one[4] = {0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu};
      tmem_st4(tmem + lq + C::SFB_COL, one);
      tmem_st4(tmem + lq + C::SFB_COL + 4, one);
    }
    // e8m0 scales [E][rows][K/32] (passed through the fp32 scale fields)
    const uint8_t* scales = reinterpret_cast<const uint8_t*>(FFN1 ? a.w13_scale : a.w2_scale);
    const int wrows = FFN1 ? 2 * a.I : a.K;  // weight rows per expert
    const int sbytes = Kel / 32;             // scale bytes per weight row
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      const int item = tile / NB, nb = tile - item * NB;
      const int4 it = a.items[item];
      const uint8_t* sb = scales + (size_t)it.x * wrows * sbytes;
      for (int kb = 0; kb < KB; ++kb) {
        int got = 1;
        if (lane == 0) got = mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, a.err, s_abort) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int blk = 0; blk < C::NA; ++blk) {
          const int r0 = (blk == 0 ? 0 : a.I) + nb * MX_BM;
          uint32_t v[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            v[c] = __ldg(reinterpret_cast<const uint32_t*>(sb + (size_t)(r0 + lane + 32 * c) * sbytes +
                                                           kb * 4));
          tmem_st4(tmem + lq + C::SFA_COL + stage * C::NA * 4 + blk * 4, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sfull[stage]));
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
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
      const int f = nb * MX_BM + q * 32 + lane;
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
              hout[(size_t)row * a.I + f] = (uint16_t)f32_to_bf16_bits(g / (1.0f + expf(-g)) * u);
            }
          }
        }
      } else {
        uint16_t* yout = static_cast<uint16_t*>(a.y);
        for (int c0 = 0; c0 < rows; c0 += 16) {
          uint32_t v[16];
          __syncwarp();
          tmem_ld16(tbase + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = c0 + j;
            const int row = row0 + r;
            if (r < rows && (unsigned)row < (unsigned)a.rows_total) {
              const float rw = a.row_w ? a.row_w[row] : 1.0f;
              yout[(size_t)row * a.K + f] =
                  (uint16_t)f32_to_bf16_bits((__uint_as_float(v[j]) * a.hs[row]) * rw);
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
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 mx_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

template <bool FFN1, int BN>
cudaError_t launch_mx_impl(const GroupedFfnArgs& a, cudaStream_t s) {
  using C = MxCfg<FFN1, BN>;
  auto enc = mx_encoder();
  if (!enc) return cudaErrorInvalidValue;
  const int Kel = FFN1 ? a.K : a.I;
  const int Wrows = FFN1 ? 2 * a.I : a.K;
  const void* w = FFN1 ? a.w13 : a.w2;
  const void* x = FFN1 ? a.xq : a.hq;
  CUtensorMap tw, tx;
  {
    // packed e2m1 weights [E][rows][Kel/2 bytes], unpacked to 16 bytes per 16 values
    cuuint64_t dims[3] = {(cuuint64_t)Kel, (cuuint64_t)Wrows, (cuuint64_t)a.E};
    cuuint64_t strides[2] = {(cuuint64_t)Kel / 2, (cuuint64_t)Kel / 2 * Wrows};
    cuuint32_t box[3] = {MX_BK, MX_BM, 1};
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
  cudaError_t e = cudaFuncSetAttribute(grouped_mx_kernel<FFN1, BN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  count_launch();
  grouped_mx_kernel<FFN1, BN><<<device_sm_count(), MX_THREADS, C::SMEM, s>>>(tw, tx, a);
  return cudaGetLastError();
}

template <bool FFN1>
cudaError_t launch_mx_bn(const GroupedFfnArgs& a, cudaStream_t s) {
  switch (a.BN) {
    case 32: return launch_mx_impl<FFN1, 32>(a, s);
    case 64: return launch_mx_impl<FFN1, 64>(a, s);
    case 96: return launch_mx_impl<FFN1, 96>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_ffn1_mx(const GroupedFfnArgs& a, cudaStream_t s) { return launch_mx_bn<true>(a, s); }
cudaError_t launch_ffn2_mx(const GroupedFfnArgs& a, cudaStream_t s) { return launch_mx_bn<false>(a, s); }

}  // namespace moe
