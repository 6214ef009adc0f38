// permute.cu -- routing metadata, scatter and gather kernels.
//
// S3  per-expert counts, offsets and a stable rank of every (token, slot) pair
//     ("Optimising Ling-2.6-1T on TPU with SGLang-JAX", s.6: the metadata block
//     holds the token->expert map, per-expert offsets/counts and the
//     scatter/gather indices; it moves little data).
// S4  dynamic per-token fp8 quantisation applied before the scatter (same
//     write-up, s.5 "activation quantisation"), then 16-byte row copies into
//     expert-contiguous order.  On one GPU the ICI scatter is this local copy.
// S6a per-row fp8 requantisation of the bf16 intermediate.
// S7  weighted gather back to token order plus the shared-expert rows
//     (s.1 "gather results"; s.5 in-kernel shared expert).
//
// Determinism: counts are order-independent; the rank of a pair inside its
// 32-token chunk comes from a per-warp bitmask table (popcount of the lanes
// below), and chunk bases from a prefix scan, so every row index is fixed.
#include <algorithm>

#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kWarps = 8;  // warps per block in the index kernels

// Build, for the warp's 32-token chunk, bits[e] = mask of lanes whose token
// picked expert e.  Returns false for the lane if its token is out of range.
__device__ __forceinline__ void build_chunk_bits(const int32_t* __restrict__ idx, uint32_t* bits,
                                                 int t, int T, int E, int k, int lane, int* err) {
  for (int e = lane; e < E; e += 32) bits[e] = 0u;
  __syncwarp();
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      int e = idx[(size_t)t * k + j];
      if ((unsigned)e < (unsigned)E)
        atomicOr(&bits[e], 1u << lane);
      else
        record_error(err, kErrInvalidArg);
    }
  }
  __syncwarp();
}

__global__ void __launch_bounds__(kWarps * 32)
    count_kernel(const int32_t* __restrict__ idx, int32_t* __restrict__ cc, int32_t* ticket,
                 int T, int E, int k, int nch, int* err) {
  pdl_wait();  // the previous kernel's outputs are complete and visible
  pdl_release();
  extern __shared__ uint32_t s_bits[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0;  // scan_kernel's completion count
  const int c = blockIdx.x * kWarps + warp;
  if (c >= nch) return;  // whole warp leaves together
  uint32_t* bits = s_bits + warp * E;
  build_chunk_bits(idx, bits, c * kChunk + lane, T, E, k, lane, err);
  for (int e = lane; e < E; e += 32) cc[(size_t)e * nch + c] = __popc(bits[e]);
}

__global__ void __launch_bounds__(kWarps * 32)
    rank_kernel(const int32_t* __restrict__ idx, const float* __restrict__ topk_w,
                const int32_t* __restrict__ off, const int32_t* __restrict__ cbase,
                int32_t* __restrict__ perm, int32_t* __restrict__ src, float* __restrict__ row_w,
                int T, int E, int k, int nch) {
  pdl_wait();  // the previous kernel's outputs are complete and visible
  pdl_release();
  extern __shared__ uint32_t s_bits[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * kWarps + warp;
  if (c >= nch) return;
  uint32_t* bits = s_bits + warp * E;
  const int t = c * kChunk + lane;
  build_chunk_bits(idx, bits, t, T, E, k, lane, nullptr);
  if (t >= T) return;
  const uint32_t below = (1u << lane) - 1u;
  for (int j = 0; j < k; ++j) {
    int e = idx[(size_t)t * k + j];
    if ((unsigned)e >= (unsigned)E) continue;
    int row = off[e] + cbase[(size_t)e * nch + c] + __popc(bits[e] & below);
    perm[(size_t)t * k + j] = row;
    src[row] = t;
    if (row_w) row_w[row] = topk_w[(size_t)t * k + j];
  }
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
    int z = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    s_warp[lane] = z - w;  // exclusive warp base
    if (lane == 31) s_warp[32] = z;
  }
  __syncthreads();
  int res = s_warp[warp] + x - v;
  *total = s_warp[32];
  __syncthreads();
  return res;
}

// Tile work list over groups 0..E-1 (offsets) and, when shared_rows > 0, one
// more group for the shared expert.  Items are {group, row0, rows, w} with
// rows <= BN, in group order; w = (items in the group) << 16 | (index of the
// item within it) for groups of at most four items, else 0: the SM-pair GEMMs
// run such a group's tiles output block by output block, so the few items of
// an expert stream its weights together (T=2048, H=8192, I=2048, E=32: FFN1
// DRAM reads 1.31 vs 1.50 GB, 1.26 GB algorithmic).  Groups of many items
// (the skewed batch's hot experts, 32 items) keep the item-by-item order,
// which was 3% faster there (FFN1 1.53 vs 1.57 ms).  Called by every thread
// of a 1024-thread block.
__device__ void build_items(const int32_t* off, int E, int BN, int shared_row0, int shared_rows,
                            int4* items, int32_t* n_items, int max_items, int* s_warp) {
  const int G = E + (shared_rows > 0 ? 1 : 0);
  int carry = 0;
  for (int base = 0; base < G; base += blockDim.x) {
    const int g = base + threadIdx.x;
    int n = 0, start = 0, rows = 0;
    if (g < G) {
      if (g < E) {
        start = off[g];
        rows = off[g + 1] - start;
      } else {
        start = shared_row0;
        rows = shared_rows;
      }
      n = (rows + BN - 1) / BN;
    }
    int total;
    const int ex = block_exclusive_scan(n, s_warp, &total);
    for (int i = 0; i < n; ++i) {
      int id = carry + ex + i;
      const int w = n <= 4 ? (n << 16) | i : 0;
      if (id < max_items) items[id] = make_int4(g, start + i * BN, min(BN, rows - i * BN), w);
    }
    carry += total;
  }
  if (threadIdx.x == 0) *n_items = min(carry, max_items);
}

// One warp per expert (32 per block): the exclusive scan of its per-chunk
// counts gives the chunk bases, eight chunk counts per lane loaded before the
// scans that use them.  The block that finishes last (a ticket taken after
// every block's writes are fenced; no block waits for another) turns the
// expert totals into offsets and the tile list.
__global__ void __launch_bounds__(1024)
    scan_kernel(const int32_t* __restrict__ cc, int32_t* __restrict__ cbase, int32_t* cnt,
                int32_t* off, int32_t* ticket, int E, int nch, int R, int4* items,
                int32_t* n_items, int max_items, int BN, int shared_row0, int shared_rows) {
  pdl_wait();  // the previous kernel's outputs are complete and visible
  __shared__ int s_cnt[kMaxExperts + 1];
  __shared__ int s_warp[33];
  __shared__ bool s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + warp;
  if (e < E) {
    const int32_t* row = cc + (size_t)e * nch;
    int32_t* base = cbase + (size_t)e * nch;
    int run = 0;
    for (int c0 = 0; c0 < nch; c0 += 32 * 8) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + 32 * u + lane;
        v[u] = c < nch ? row[c] : 0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        int x = v[u];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        const int c = c0 + 32 * u + lane;
        if (c < nch) base[c] = run + x - v[u];
        run += __shfl_sync(0xffffffffu, x, 31);
      }
    }
    if (lane == 0) cnt[e] = run;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (s_last) {
    __threadfence();
    const int v = threadIdx.x < E ? __ldcg(cnt + threadIdx.x) : 0;
    int total;
    const int ex = block_exclusive_scan(v, s_warp, &total);
    if (threadIdx.x < E) {
      off[threadIdx.x] = ex;
      s_cnt[threadIdx.x] = ex;
    }
    if (threadIdx.x == 0) {
      off[E] = total;  // == R when every index was valid
      s_cnt[E] = total;
    }
    __syncthreads();
    if (items) build_items(s_cnt, E, BN, shared_row0, shared_rows, items, n_items, max_items, s_warp);
    // the tile list is final and visible before the next kernels may launch:
    // the expert GEMMs read it before their pdl_wait
    __threadfence();
    __syncthreads();
  }
  pdl_release();
}

// S3 for small batches in one block of 1024 threads (up to 1024 tokens fit;
// the layer uses it below 512): the per-chunk expert masks, the per-expert
// chunk scans, the expert offsets, the tile list and the stable ranks of
// count_kernel, scan_kernel and rank_kernel, with the masks and chunk bases in
// shared memory ([nch][E] words each) and one launch instead of three.  Warp c owns chunk c and lane l its token, whose
// top-k indices and weights are loaded once, up front, into registers.  Same
// results bit for bit.  KMAX >= k bounds the per-lane register arrays.
template <int KMAX>
__global__ void __launch_bounds__(1024)
    index_small_kernel(const int32_t* __restrict__ idx, const float* __restrict__ topk_w,
                       int32_t* __restrict__ cnt, int32_t* __restrict__ off,
                       int32_t* __restrict__ perm, int32_t* __restrict__ src,
                       float* __restrict__ row_w, int T, int E, int k, int nch, int4* items,
                       int32_t* n_items, int max_items, int BN, int shared_row0,
                       int shared_rows, int* err) {
  pdl_wait();  // the previous kernel's outputs are complete and visible
  extern __shared__ uint32_t s_dyn[];
  uint32_t* bits = s_dyn;                                   // [nch][E] lane masks
  int* cb = reinterpret_cast<int*>(s_dyn + (size_t)nch * E);  // [nch][E] chunk bases
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_warp[33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = warp;  // nch <= 32: one chunk per warp at most
  const int t = c * kChunk + lane;
  const bool mine = c < nch && t < T;
  int ev[KMAX];
  float wv[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    ev[j] = (mine && j < k) ? idx[(size_t)t * k + j] : -1;
    wv[j] = (mine && j < k && row_w) ? topk_w[(size_t)t * k + j] : 0.0f;
  }
  if (c < nch) {
    uint32_t* b = bits + (size_t)c * E;
    for (int e = lane; e < E; e += 32) b[e] = 0u;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j >= k || !mine) continue;
      if ((unsigned)ev[j] < (unsigned)E)
        atomicOr(&b[ev[j]], 1u << lane);
      else
        record_error(err, kErrInvalidArg);
    }
  }
  __syncthreads();
  for (int e = warp; e < E; e += 32) {
    const int v = lane < nch ? __popc(bits[(size_t)lane * E + e]) : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < nch) cb[(size_t)lane * E + e] = x - v;
    if (lane == 31) s_off[e] = x;
  }
  __syncthreads();
  const int v = threadIdx.x < E ? s_off[threadIdx.x] : 0;
  int total;
  const int ex = block_exclusive_scan(v, s_warp, &total);
  if (threadIdx.x < E) {
    cnt[threadIdx.x] = v;
    off[threadIdx.x] = ex;
    s_off[threadIdx.x] = ex;
  }
  if (threadIdx.x == 0) {
    off[E] = total;
    s_off[E] = total;
  }
  __syncthreads();
  if (items) build_items(s_off, E, BN, shared_row0, shared_rows, items, n_items, max_items, s_warp);
  // the tile list is final and visible before the next kernels may launch:
  // the expert GEMMs read it before their pdl_wait
  __threadfence();
  __syncthreads();
  pdl_release();
  if (!mine) return;
  const uint32_t below = (1u << lane) - 1u;
  const uint32_t* b = bits + (size_t)c * E;
  const int* base = cb + (size_t)c * E;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    if (j >= k) break;
    const int e = ev[j];
    if ((unsigned)e >= (unsigned)E) continue;
    const int row = s_off[e] + base[e] + __popc(b[e] & below);
    perm[(size_t)t * k + j] = row;
    src[row] = t;
    if (row_w) row_w[row] = wv[j];
  }
}

__global__ void __launch_bounds__(1024)
    items_kernel(const int32_t* __restrict__ off, int E, int4* items, int32_t* n_items,
                 int max_items, int BN) {
  pdl_wait();  // the previous kernel's outputs are complete and visible
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_warp[33];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = off[e];
  __syncthreads();
  build_items(s_off, E, BN, 0, 0, items, n_items, max_items, s_warp);
  // the tile list is final and visible before the next kernels may launch:
  // the expert GEMMs read it before their pdl_wait
  __threadfence();
  __syncthreads();
  pdl_release();
}

// Block-wide max of non-negative floats (blockDim.x == 256).
__device__ __forceinline__ float block_max256(float v, float* s_red) {
  v = warp_max(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float w = lane < 8 ? s_red[lane] : 0.0f;
    w = warp_max(w);
    if (lane == 0) s_red[8] = w;
  }
  __syncthreads();
  float r = s_red[8];
  __syncthreads();
  return r;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
    f[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
}

// e4m3 codes of four values (round-to-nearest-even, saturating), the first
// in the low byte; two values per conversion instruction.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// q = e4m3(v / s) for 8 values (fp32 IEEE division, round-to-nearest-even).
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float s) {
  return make_uint2(e4m3x4(f[0] / s, f[1] / s, f[2] / s, f[3] / s),
                    e4m3x4(f[4] / s, f[5] / s, f[6] / s, f[7] / s));
}

__global__ void __launch_bounds__(256)
    quant_scatter_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                         uint8_t* __restrict__ xq, float* __restrict__ xscale, int H, int k,
                         int shared_row0, int R, int* err, float* __restrict__ acc_zero) {
  pdl_wait();  // the previous kernel's outputs are complete and visible
  pdl_release();
  __shared__ float s_red[9];
  __shared__ int s_rows[kMaxTopK + 1];
  const int t = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  const int nv = H / 8;
  float amax = 0.0f;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    float f[8];
    unpack_bf16x8(xr[v], f);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
  amax = block_max256(amax, s_red);
  const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
  const int nrows = k + (shared_row0 >= 0 ? 1 : 0);
  if (threadIdx.x < k) {
    // rows come from the rank pass; anything outside [0, R) (possible only for
    // invalid expert indices) is dropped rather than written
    int row = perm[(size_t)t * k + threadIdx.x];
    if ((unsigned)row >= (unsigned)R) {
      record_error(err, kErrInvalidArg);
      row = -1;
    }
    s_rows[threadIdx.x] = row;
  }
  if (threadIdx.x == k && shared_row0 >= 0) s_rows[k] = shared_row0 + t;
  __syncthreads();
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    float f[8];
    unpack_bf16x8(xr[v], f);
    const uint2 q = quant8(f, s);
    for (int j = 0; j < nrows; ++j)
      if (s_rows[j] >= 0) *reinterpret_cast<uint2*>(xq + (size_t)s_rows[j] * H + (size_t)v * 8) = q;
  }
  if (threadIdx.x < nrows && s_rows[threadIdx.x] >= 0) xscale[s_rows[threadIdx.x]] = s;
  if (acc_zero) {  // the fused combine's fp32 sum of this token starts at zero
    float4* ar = reinterpret_cast<float4*>(acc_zero + (size_t)t * H);
    for (int v = threadIdx.x; v < H / 4; v += blockDim.x) ar[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__global__ void __launch_bounds__(256)
    requant_kernel(const uint16_t* __restrict__ h, uint8_t* __restrict__ hq, float* __restrict__ hs,
                   int I) {
  pdl_wait();  // the previous kernel's outputs are complete and visible
  pdl_release();
  __shared__ float s_red[9];
  const size_t r = blockIdx.x;
  const uint4* hr = reinterpret_cast<const uint4*>(h + r * I);
  const int nv = I / 8;
  float amax = 0.0f;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    float f[8];
    unpack_bf16x8(hr[v], f);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
  amax = block_max256(amax, s_red);
  const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    float f[8];
    unpack_bf16x8(hr[v], f);
    *reinterpret_cast<uint2*>(hq + r * I + (size_t)v * 8) = quant8(f, s);
  }
  if (threadIdx.x == 0) hs[r] = s;
}

// The same per-row requantisation with one warp per row: the row (I <= 32 *
// 8 * MAXV elements) stays in registers between the max and the quantisation,
// and the max is a shuffle reduction, so many rows are in flight per SM.
template <int MAXV>
__global__ void __launch_bounds__(256)
    requant_warp_kernel(const uint16_t* __restrict__ h, uint8_t* __restrict__ hq,
                        float* __restrict__ hs, int rows, int I) {
  pdl_wait();  // the previous kernel's outputs are complete and visible
  pdl_release();
  const int r = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const uint4* hr = reinterpret_cast<const uint4*>(h + (size_t)r * I);
  const int nv = I / 8;
  uint4 v[MAXV];
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    const int i = lane + 32 * j;
    if (i < nv) {
      v[j] = __ldcs(hr + i);
      float f[8];
      unpack_bf16x8(v[j], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
    }
  }
  amax = warp_max(amax);
  const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    const int i = lane + 32 * j;
    if (i < nv) {
      float f[8];
      unpack_bf16x8(v[j], f);
      *reinterpret_cast<uint2*>(hq + (size_t)r * I + (size_t)i * 8) = quant8(f, s);
    }
  }
  if (lane == 0) hs[r] = s;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);  // a -> low half
  return *reinterpret_cast<uint32_t*>(&p);
}

// out = bf16(acc), eight elements per thread and step.
__global__ void __launch_bounds__(256)
    acc_to_bf16_kernel(const float4* __restrict__ acc, uint4* __restrict__ out, size_t n8) {
  pdl_wait();  // the previous kernel's outputs are complete and visible
  pdl_release();
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = acc[2 * i], b = acc[2 * i + 1];
    uint4 u;
    u.x = pack_bf16x2(a.x, a.y);
    u.y = pack_bf16x2(a.z, a.w);
    u.z = pack_bf16x2(b.x, b.y);
    u.w = pack_bf16x2(b.z, b.w);
    out[i] = u;
  }
}

// One thread per 8 output columns; the grid covers (token, column slice) so a
// decode-sized batch still fills the GPU.  All k rows of the thread's columns
// are loaded before the fp32 sum (j ascending, shared expert last), so the
// loads overlap.
template <int KMAX>
__global__ void __launch_bounds__(256)
    combine_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ perm,
                   const uint16_t* __restrict__ shared, uint16_t* __restrict__ out, int H, int k,
                   int R, int* err) {
  pdl_wait();  // the previous kernel's outputs are complete and visible
  pdl_release();
  const int t = blockIdx.x;
  const int v = blockIdx.y * blockDim.x + threadIdx.x;  // 16-byte column group
  const int nv = H / 8;
  int rows[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    int row = -1;
    if (j < k) {
      row = __ldg(perm + (size_t)t * k + j);
      if ((unsigned)row >= (unsigned)R) {  // invalid permutation entry: contributes nothing
        if (v == 0) record_error(err, kErrInvalidArg);
        row = -1;
      }
    }
    rows[j] = row;
  }
  if (v >= nv) return;
  uint4 raw[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    if (rows[j] >= 0) raw[j] = __ldcs(reinterpret_cast<const uint4*>(y + (size_t)rows[j] * H) + v);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    if (rows[j] < 0) continue;
    float f[8];
    unpack_bf16x8(raw[j], f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += f[i];
  }
  if (shared) {
    float f[8];
    unpack_bf16x8(reinterpret_cast<const uint4*>(shared + (size_t)t * H)[v], f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += f[i];
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  reinterpret_cast<uint4*>(out + (size_t)t * H)[v] = o;
}

// LatentMoE: the routed combine feeds RMSNorm on the latent ("Kimi K3 ...
// feasibility analysis", s.2.4: routed experts -> routed_expert_norm ->
// up_proj).  acc = sum_j y[perm[t,j]] in fp32 (j ascending), then
// yn = bf16(acc / sqrt(mean(acc^2) + eps) * gamma).
template <int KMAX>
__global__ void __launch_bounds__(256)
    combine_rmsnorm_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ perm,
                           const uint16_t* __restrict__ gamma, uint16_t* __restrict__ yn, int L,
                           int k, int R, float eps, int* err) {
  pdl_wait();  // the previous kernel's outputs are complete and visible
  pdl_release();
  extern __shared__ float s_acc[];  // [L]
  __shared__ int s_rows[kMaxTopK];
  __shared__ float s_red[9];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    int row = perm[(size_t)t * k + threadIdx.x];
    if ((unsigned)row >= (unsigned)R) {
      record_error(err, kErrInvalidArg);
      row = -1;
    }
    s_rows[threadIdx.x] = row;
  }
  __syncthreads();
  const int nv = L / 8;
  float sq = 0.0f;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    // all k row loads in flight before the sum (j ascending, as in the gather)
    uint4 raw[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k && s_rows[j] >= 0)
        raw[j] = __ldcs(reinterpret_cast<const uint4*>(y + (size_t)s_rows[j] * L) + v);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j >= k || s_rows[j] < 0) continue;
      float f[8];
      unpack_bf16x8(raw[j], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += f[i];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s_acc[v * 8 + i] = acc[i];
      sq += acc[i] * acc[i];
    }
  }
  // block sum of squares (non-negative: reuse the max helper's layout with adds)
  sq = [&] {
    float x = sq;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) s_red[warp] = x;
    __syncthreads();
    if (warp == 0) {
      float w = lane < 8 ? s_red[lane] : 0.0f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
      if (lane == 0) s_red[8] = w;
    }
    __syncthreads();
    return s_red[8];
  }();
  const float scale = 1.0f / sqrtf(sq / (float)L + eps);
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    float g[8];
    unpack_bf16x8(reinterpret_cast<const uint4*>(gamma)[v], g);
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = s_acc[v * 8 + i] * scale * g[i];
    uint4 u;
    u.x = pack_bf16x2(o[0], o[1]);
    u.y = pack_bf16x2(o[2], o[3]);
    u.z = pack_bf16x2(o[4], o[5]);
    u.w = pack_bf16x2(o[6], o[7]);
    reinterpret_cast<uint4*>(yn + (size_t)t * L)[v] = u;
  }
}

}  // namespace

cudaError_t launch_combine_rmsnorm(const void* y, const int32_t* perm, const void* gamma, void* yn,
                                   int T, int L, int k, float eps, int* err, cudaStream_t s) {
  const size_t smem = (size_t)L * sizeof(float);
  auto go = [&](auto kern) {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
      if (e != cudaSuccess) return e;
    }
    count_launch();
    return launch_kernel(kern, dim3(T), dim3(256), smem, s, 1, static_cast<const uint16_t*>(y),
                         perm, static_cast<const uint16_t*>(gamma), static_cast<uint16_t*>(yn), L,
                         k, T * k, eps, err);
  };
  if (k <= 4) return go(combine_rmsnorm_kernel<4>);
  if (k <= 8) return go(combine_rmsnorm_kernel<8>);
  if (k <= 16) return go(combine_rmsnorm_kernel<16>);
  return go(combine_rmsnorm_kernel<kMaxTopK>);
}

cudaError_t launch_count(const int32_t* idx, int32_t* cc, int32_t* ticket, int T, int E, int k,
                         int* err, cudaStream_t s) {
  const int nch = num_chunks(T);
  const int blocks = (nch + kWarps - 1) / kWarps;
  const size_t smem = (size_t)kWarps * E * sizeof(uint32_t);
  count_launch();
  return launch_kernel(count_kernel, dim3(blocks), dim3(kWarps * 32), smem, s, 1, idx, cc, ticket,
                       T, E, k, nch, err);
}

cudaError_t launch_scan(const int32_t* cc, int32_t* cbase, int32_t* cnt, int32_t* off,
                        int32_t* ticket, int T, int E, int k, int4* items, int32_t* n_items,
                        int max_items, int BN, int shared_row0, int shared_rows, cudaStream_t s) {
  if (E <= 0 || E > kMaxExperts) return cudaErrorInvalidValue;
  count_launch();
  return launch_kernel(scan_kernel, dim3((E + 31) / 32), dim3(1024), 0, s, 1, cc, cbase, cnt, off,
                       ticket, E, num_chunks(T), T * k, items, n_items, max_items, BN, shared_row0,
                       shared_rows);
}

bool index_small_fits(int T, int E) {
  return num_chunks(T) <= 32 &&
         (size_t)num_chunks(T) * E * 2 * sizeof(uint32_t) <= kIndexSmallSmem;
}

cudaError_t launch_index_small(const int32_t* idx, const float* topk_w, int32_t* cnt, int32_t* off,
                               int32_t* perm, int32_t* src, float* row_w, int T, int E, int k,
                               int4* items, int32_t* n_items, int max_items, int BN,
                               int shared_row0, int shared_rows, int* err, cudaStream_t s) {
  const int nch = num_chunks(T);
  const size_t smem = (size_t)nch * E * 2 * sizeof(uint32_t);
  if (nch > 32 || smem > kIndexSmallSmem) return cudaErrorInvalidValue;
  auto go = [&](auto kern) {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kIndexSmallSmem);
      if (e != cudaSuccess) return e;
    }
    count_launch();
    return launch_kernel(kern, dim3(1), dim3(1024), smem, s, 1, idx, topk_w, cnt, off, perm, src,
                         row_w, T, E, k, nch, items, n_items, max_items, BN, shared_row0,
                         shared_rows, err);
  };
  if (k <= 8) return go(index_small_kernel<8>);
  if (k <= 16) return go(index_small_kernel<16>);
  return go(index_small_kernel<kMaxTopK>);
}

cudaError_t launch_items_from_offsets(const int32_t* off, int E, int4* items, int32_t* n_items,
                                      int max_items, int BN, cudaStream_t s) {
  count_launch();
  return launch_kernel(items_kernel, dim3(1), dim3(1024), 0, s, 1, off, E, items, n_items, max_items,
                       BN);
}

cudaError_t launch_rank(const int32_t* idx, const float* topk_w, const int32_t* off,
                        const int32_t* cbase, int32_t* perm, int32_t* src, float* row_w, int T,
                        int E, int k, cudaStream_t s) {
  const int nch = num_chunks(T);
  const int blocks = (nch + kWarps - 1) / kWarps;
  const size_t smem = (size_t)kWarps * E * sizeof(uint32_t);
  count_launch();
  return launch_kernel(rank_kernel, dim3(blocks), dim3(kWarps * 32), smem, s, 1, idx, topk_w, off,
                       cbase, perm, src, row_w, T, E, k, nch);
}

cudaError_t launch_quant_scatter(const void* x, const int32_t* perm, void* xq, float* xscale,
                                 int T, int H, int k, int shared_row0, int* err, cudaStream_t s,
                                 float* acc_zero) {
  count_launch();
  return launch_kernel(quant_scatter_kernel, dim3(T), dim3(256), 0, s, 1,
                       static_cast<const uint16_t*>(x), perm, static_cast<uint8_t*>(xq), xscale, H, k,
                       shared_row0, T * k, err, acc_zero);
}

cudaError_t launch_acc_to_bf16(const float* acc, void* out, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  count_launch();
  const size_t n8 = n / 8;
  const int blocks = (int)std::min<size_t>((n8 + 255) / 256, (size_t)device_sm_count() * 8);
  return launch_kernel(acc_to_bf16_kernel, dim3(blocks), dim3(256), 0, s, 1,
                       reinterpret_cast<const float4*>(acc), static_cast<uint4*>(out), n8);
}

cudaError_t launch_requant(const void* h, void* hq, float* hs, int rows, int I, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  count_launch();
  const auto* hp = static_cast<const uint16_t*>(h);
  auto* qp = static_cast<uint8_t*>(hq);
  const unsigned warps_blocks = (unsigned)(((size_t)rows * 32 + 255) / 256);
  const int per_lane = (I / 8 + 31) / 32;  // 16-byte vectors per lane
  if (per_lane <= 4)
    return launch_kernel(requant_warp_kernel<4>, dim3(warps_blocks), dim3(256), 0, s, 1, hp, qp, hs,
                         rows, I);
  else if (per_lane <= 8)
    return launch_kernel(requant_warp_kernel<8>, dim3(warps_blocks), dim3(256), 0, s, 1, hp, qp, hs,
                         rows, I);
  else if (per_lane <= 12)  // I = 3072: fewer registers, more rows per SM
    return launch_kernel(requant_warp_kernel<12>, dim3(warps_blocks), dim3(256), 0, s, 1, hp, qp, hs,
                         rows, I);
  else if (per_lane <= 16)
    return launch_kernel(requant_warp_kernel<16>, dim3(warps_blocks), dim3(256), 0, s, 1, hp, qp, hs,
                         rows, I);
  else
    return launch_kernel(requant_kernel, dim3(rows), dim3(256), 0, s, 1, hp, qp, hs, I);
}

cudaError_t launch_combine(const void* y, const int32_t* perm, const void* shared, void* out,
                           int T, int H, int k, int* err, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  count_launch();
  const dim3 grid(T, (H / 8 + 255) / 256);
  const auto* yp = static_cast<const uint16_t*>(y);
  const auto* sp = static_cast<const uint16_t*>(shared);
  auto* op = static_cast<uint16_t*>(out);
  if (k <= 4)
    return launch_kernel(combine_kernel<4>, grid, dim3(256), 0, s, 1, yp, perm, sp, op, H, k, T * k,
                         err);
  else if (k <= 8)
    return launch_kernel(combine_kernel<8>, grid, dim3(256), 0, s, 1, yp, perm, sp, op, H, k, T * k,
                         err);
  else if (k <= 16)
    return launch_kernel(combine_kernel<16>, grid, dim3(256), 0, s, 1, yp, perm, sp, op, H, k, T * k,
                         err);
  else
    return launch_kernel(combine_kernel<32>, grid, dim3(256), 0, s, 1, yp, perm, sp, op, H, k, T * k,
                         err);
}

}  // namespace moe
