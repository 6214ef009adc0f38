// ffn_gemm_2cta.cu -- S5/S6 for large batches: the grouped fp8 expert GEMMs
// on pairs of SMs (tcgen05 cta_group::2).
//
// Same arithmetic as ffn_gemm.cu ("Optimising Ling-2.6-1T on TPU with
// SGLang-JAX", s.5 per-channel direct_scaled_dot; FFN1/FFN2 of the s.1 cost
// model), different shape, chosen when experts hold hundreds of rows
// (prefill): a cluster of two CTAs computes a 256-row x 256-column tile with
// one MMA stream.  Each CTA stages half of the token rows (A, 128 x 128 B per
// K step) and half of the weight rows (B, 128 x 128 B), so every SM moves 32 KB
// per 4.2 M multiply-adds instead of 48-64 KB for a single-SM tile of the same
// depth; the tile's accumulator (128 rows x 256 fp32 columns per CTA) is
// double-buffered in tensor memory.
//
//   FFN1: columns 0..127 = g (W1 rows f0..f0+127, staged by CTA 0),
//         columns 128..255 = u (W3 rows I+f0.., staged by CTA 1), so each
//         epilogue thread holds g and u of one token row and writes 128
//         contiguous bf16 of h.
//   FFN2: columns = 256 output channels (W2 rows c0.., 128 per CTA).
//
// Roles per CTA (192 threads): warp 0 TMA producer, warp 1 MMA issuer (even
// CTA only; the odd CTA's warp 1 only joins the tensor-memory allocation),
// warps 2-5 epilogue (thread = token row, 16 columns per tcgen05.ld).  Both
// CTAs' TMA loads complete on the even CTA's `full` barrier; the even CTA's
// commits arrive on both CTAs' `empty` / `tfull` barriers; both epilogues
// release an accumulator on the even CTA's `tempty` barrier.  All waits are
// bounded as in ffn_gemm.cu.
#include <cudaTypedefs.h>

#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int P_ROWS = 128;   // token rows per CTA (M = 256 per pair)
constexpr int P_N = 256;      // output columns per tile
constexpr int P_BK = 128;     // K bytes per stage
constexpr int P_UMMA_K = 32;  // K per tcgen05.mma for 8-bit operands
constexpr int P_THREADS = 192;
constexpr int P_A_BYTES = P_ROWS * P_BK;       // 16 KB
constexpr int P_B_BYTES = (P_N / 2) * P_BK;    // 16 KB (this CTA's half of N)
constexpr int P_STAGE = P_A_BYTES + P_B_BYTES;  // 32 KB
constexpr int P_STAGES = 6;
constexpr int P_ACC_STAGES = 2;
constexpr int P_TMEM_COLS = 512;
constexpr int P_NUM_BARS = 2 * P_STAGES + 2 * P_ACC_STAGES + 1;
constexpr int P_SMEM = 1024 + P_STAGES * P_STAGE + P_NUM_BARS * 8 + 16 + P_STAGES * 4;

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);  // a -> low half
  return *reinterpret_cast<uint32_t*>(&p);
}

template <bool FFN1>
__global__ void __launch_bounds__(P_THREADS, 1)
    grouped_ffn_pair_kernel(const __grid_constant__ CUtensorMap tm_w,
                            const __grid_constant__ CUtensorMap tm_ws,
                            const __grid_constant__ CUtensorMap tm_x, const GroupedFfnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P_STAGES * P_STAGE);
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
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(s_tmem), P_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  const int NB = FFN1 ? a.I / 128 : a.K / P_N;  // output blocks per item
  const int KB = FFN1 ? a.K / P_BK : a.I / P_BK;
  const int n_items = min(*a.n_items, a.max_items);
  const int n_tiles = n_items * NB;
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = cluster; tile < n_tiles && !*s_abort; tile += n_clusters) {
        const int item = tile / NB, nb = tile - item * NB;
        const int4 it = a.items[item];
        const bool shared = it.x >= a.E;
        const CUtensorMap* tw = shared ? &tm_ws : &tm_w;
        const int gc = shared ? 0 : it.x;
        const int wrow = FFN1 ? (rank == 0 ? nb * 128 : a.I + nb * 128) : nb * P_N + 128 * (int)rank;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, a.err, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t st = smem_u32(smem + stage * P_STAGE);
          const uint32_t fb_leader = mapa_shared(smem_u32(&full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(smem_u32(&full[stage]), 2 * P_STAGE);
          tma_load_2d_pair(st, &tm_x, kb * P_BK, it.y + 128 * (int)rank, fb_leader);
          tma_load_3d_pair(st + P_A_BYTES, tw, kb * P_BK, wrow, gc, fb_leader);
          s_issued[stage] = phase + 1u;
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (*s_abort && leader) {  // the pair's loads complete on the even CTA's barriers
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
      const uint32_t idesc = idesc_e4m3_f32(2 * P_ROWS, P_N);
      for (int tile = cluster; tile < n_tiles && !*s_abort; tile += n_clusters, ++it_local) {
        const int acc = it_local % P_ACC_STAGES;
        const uint32_t acc_phase = (uint32_t)(it_local / P_ACC_STAGES) & 1u;
        if (!mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, a.err, s_abort)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * P_N;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(smem_u32(&full[stage]), phase, a.err, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * P_STAGE);
          const uint32_t b0 = a0 + P_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < P_BK / P_UMMA_K; ++kk)
            mma_f8f6f4_pair(d, smem_desc_sw128(a0 + kk * P_UMMA_K),
                            smem_desc_sw128(b0 + kk * P_UMMA_K), idesc, (kb | kk) ? 1u : 0u);
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
    int it_local = 0;
    for (int tile = cluster; tile < n_tiles; tile += n_clusters, ++it_local) {
      const int item = tile / NB, nb = tile - item * NB;
      const int4 it = a.items[item];
      const bool shared = it.x >= a.E;
      const int acc = it_local % P_ACC_STAGES;
      const uint32_t acc_phase = (uint32_t)(it_local / P_ACC_STAGES) & 1u;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(smem_u32(&tfull[acc]), acc_phase, a.err, s_abort) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int r = lrow + 128 * (int)rank;
      const int row = it.y + r;
      const bool valid = r < it.z && (unsigned)row < (unsigned)a.rows_total;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + acc * P_N;
      if (FFN1) {
        const float* sc = shared ? a.sw13_scale : a.w13_scale + (size_t)it.x * 2 * a.I;
        const int f0 = nb * 128;
        const float xs = valid ? a.xscale[row] : 0.0f;
        uint16_t* hrow = static_cast<uint16_t*>(a.h) + (size_t)(valid ? row : 0) * a.I + f0;
#pragma unroll 1
        for (int c = 0; c < 128; c += 16) {
          uint32_t vg[16], vu[16];
          __syncwarp();
          tmem_ld16(tbase + c, vg);
          tmem_ld16(tbase + 128 + c, vu);
          tmem_ld_wait();
          uint32_t packed[8];
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            float hv[2];
#pragma unroll
            for (int u2 = 0; u2 < 2; ++u2) {
              const float sg = __ldg(sc + f0 + c + j + u2), su = __ldg(sc + a.I + f0 + c + j + u2);
              const float g = (__uint_as_float(vg[j + u2]) * xs) * sg;
              const float u = (__uint_as_float(vu[j + u2]) * xs) * su;
              hv[u2] = g / (1.0f + expf(-g)) * u;
            }
            packed[j / 2] = pack_bf16x2(hv[0], hv[1]);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(hrow + c);
            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
          }
        }
      } else {
        const float* sc = shared ? a.sw2_scale : a.w2_scale + (size_t)it.x * a.K;
        const int c0 = nb * P_N;
        const float hs = valid ? a.hs[row] : 0.0f;
        const float rw = (valid && !shared && a.row_w) ? a.row_w[row] : 1.0f;
        uint16_t* yrow = static_cast<uint16_t*>(a.y) + (size_t)(valid ? row : 0) * a.K + c0;
#pragma unroll 1
        for (int c = 0; c < P_N; c += 16) {
          uint32_t v[16];
          __syncwarp();
          tmem_ld16(tbase + c, v);
          tmem_ld_wait();
          uint32_t packed[8];
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const float y0 = ((__uint_as_float(v[j]) * hs) * __ldg(sc + c0 + c + j)) * rw;
            const float y1 = ((__uint_as_float(v[j + 1]) * hs) * __ldg(sc + c0 + c + j + 1)) * rw;
            packed[j / 2] = pack_bf16x2(y0, y1);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(yrow + c);
            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader0 + acc * 8);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, P_TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

bool pair_map(CUtensorMap* m, int rank, const void* base, uint64_t inner, uint64_t rows,
              uint64_t groups) {
  auto enc = encoder();
  if (!enc || !base) return false;
  cuuint64_t dims[3] = {inner, rows, groups};
  cuuint64_t strides[2] = {inner, inner * rows};
  cuuint32_t box[3] = {(cuuint32_t)P_BK, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool FFN1>
cudaError_t launch_pair(const GroupedFfnArgs& a, cudaStream_t s) {
  const int K = FFN1 ? a.K : a.I;
  const int Wrows = FFN1 ? 2 * a.I : a.K;
  const void* w = FFN1 ? a.w13 : a.w2;
  const void* ws = FFN1 ? a.sw13 : a.sw2;
  const void* x = FFN1 ? a.xq : a.hq;
  CUtensorMap tw, tws, tx;
  if (!pair_map(&tw, 3, w, K, Wrows, a.E) || !pair_map(&tws, 3, ws ? ws : w, K, Wrows, 1) ||
      !pair_map(&tx, 2, x, K, a.rows_total, 1))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(grouped_ffn_pair_kernel<FFN1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((device_sm_count() / 2) * 2);
  cfg.blockDim = dim3(P_THREADS);
  cfg.dynamicSmemBytes = P_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  e = cudaLaunchKernelEx(&cfg, grouped_ffn_pair_kernel<FFN1>, tw, tws, tx, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn1_pair(const GroupedFfnArgs& a, cudaStream_t s) { return launch_pair<true>(a, s); }
cudaError_t launch_ffn2_pair(const GroupedFfnArgs& a, cudaStream_t s) { return launch_pair<false>(a, s); }

}  // namespace moe
