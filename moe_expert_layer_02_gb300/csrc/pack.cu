// pack.cu -- one-time repack of expert weights into the order the grouped
// GEMMs stream them.
//
// The fp8 grouped GEMMs read each expert's weights as 128-row x 128-byte tiles
// (one per pipeline stage).  In the row-major layout a tile is 128 separate
// 128-byte pieces, one per weight row; stored tile-major,
// [group][row_block][k_block][128 rows][128 bytes], every stage reads one
// contiguous 16 KB block.  MXFP4 stages read two 128-row blocks and their e8m0
// scales together; their packed order (below) makes that one TMA box plus one
// bulk copy per stage.  This is the usual load-time weight processing step;
// bytes are only permuted.
#include "../../include/moe.h"
#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

// src [G][R][Cb] bytes -> dst [G][R/128][Cb/tb][128][tb]; one thread per 4 bytes.
__global__ void pack_tiles_kernel(const uint32_t* __restrict__ src, uint32_t* __restrict__ dst,
                                  int64_t words, int R, int Cb, int tb) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= words) return;
  const int64_t byte = i * 4;
  const int64_t per_group = (int64_t)R * Cb;
  const int64_t g = byte / per_group;
  int64_t rem = byte - g * per_group;
  const int KB = Cb / tb;
  const int64_t tile = rem / (128 * tb);  // rb * KB + kb
  rem -= tile * (128 * tb);
  const int r = (int)(rem / tb), c = (int)(rem - (int64_t)r * tb);
  const int rb = (int)(tile / KB), kb = (int)(tile - (int64_t)rb * KB);
  const int64_t s = g * per_group + (int64_t)(rb * 128 + r) * Cb + (int64_t)kb * tb + c;
  dst[i] = src[s / 4];
}

// MXFP4 stages read two 128-row weight blocks at once: W1 and W3 block p of
// w13 (block rows p*128 and I + p*128), or W2 blocks 2p and 2p + 1 of w2.  The
// packed order keeps each stage's two tiles adjacent,
//   weights [G][P][KB][2][128 rows][64 bytes]       (one 256-row TMA box), and
//   scales  [G][P][KB][4 j][2 blk][8 i][4 c] words  (1 KB per stage),
// where word (j, blk, i, c) holds the four e8m0 bytes of k-stage kb of row
// 32c + 8j + i of block blk.  Block-scaled MMAs (M = 128 per CTA) read a
// block's scales from tensor memory as lane l = 8j + i, column c, in every
// lane quarter; in this order one stage's 1 KB, repeated once per lane
// quarter, is the 128-row x 32-byte source of a single tcgen05.cp.128x256b
// (8-row groups 256 bytes apart, the second block 128 bytes along each row)
// that fills both blocks' columns.
// Source row of (p, blk, r): p * 128 * pstep + blk * bstep + r.
__global__ void pack_mx_weights_kernel(const uint32_t* __restrict__ src,
                                       uint32_t* __restrict__ dst, int64_t words, int R, int KB,
                                       int pstep, int bstep) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= words) return;
  const int w = (int)(i & 15);            // 16 words = 64 bytes per tile row
  const int r = (int)((i >> 4) & 127);
  const int blk = (int)((i >> 11) & 1);
  const int64_t t = i >> 12;              // (g, p, kb)
  const int kb = (int)(t % KB);
  const int64_t gp = t / KB;
  const int P = R / 256;
  const int64_t g = gp / P;
  const int p = (int)(gp - g * P);
  const int64_t row = (int64_t)g * R + (int64_t)p * 128 * pstep + (int64_t)blk * bstep + r;
  dst[i] = src[row * (KB * 16) + kb * 16 + w];
}

__global__ void pack_mx_scales_kernel(const uint32_t* __restrict__ src, uint32_t* __restrict__ dst,
                                      int64_t words, int R, int KB, int pstep, int bstep) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= words) return;
  const int c = (int)(i & 3), ii = (int)((i >> 2) & 7);
  const int blk = (int)((i >> 5) & 1), j = (int)((i >> 6) & 3);
  const int l = 8 * j + ii;
  const int64_t t = i >> 8;  // (g, p, kb)
  const int kb = (int)(t % KB);
  const int64_t gp = t / KB;
  const int P = R / 256;
  const int64_t g = gp / P;
  const int p = (int)(gp - g * P);
  const int64_t row =
      (int64_t)g * R + (int64_t)p * 128 * pstep + (int64_t)blk * bstep + 32 * c + l;
  dst[i] = src[row * KB + kb];
}

// One MXFP4 matrix [G][R][K]: weights (K/2 bytes per row) and e8m0 scales
// (K/32 bytes per row), R a multiple of 256.
cudaError_t pack_mx(const void* w, void* wp, const void* sc, void* scp, int G, int R, int K,
                    int pstep, int bstep, cudaStream_t s) {
  const int KB = K / 128;
  const int64_t ww = (int64_t)G * R * K / 8, sw = (int64_t)G * R * KB;
  count_launch();
  pack_mx_weights_kernel<<<(unsigned)((ww + 255) / 256), 256, 0, s>>>(
      static_cast<const uint32_t*>(w), static_cast<uint32_t*>(wp), ww, R, KB, pstep, bstep);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launch();
  pack_mx_scales_kernel<<<(unsigned)((sw + 255) / 256), 256, 0, s>>>(
      static_cast<const uint32_t*>(sc), static_cast<uint32_t*>(scp), sw, R, KB, pstep, bstep);
  return cudaGetLastError();
}

cudaError_t pack_tiles(const void* src, void* dst, int G, int R, int Cb, int tb, cudaStream_t s) {
  if (!src || !dst) return cudaSuccess;
  const int64_t words = (int64_t)G * R * Cb / 4;
  const int64_t blocks = (words + 255) / 256;
  count_launch();
  pack_tiles_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint32_t*>(src),
                                                     static_cast<uint32_t*>(dst), words, R, Cb, tb);
  return cudaGetLastError();
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_pack_weights(const moe_problem* p, const void* w13, const void* w2,
                                const void* w13_scale, const void* w2_scale, void* w13_packed,
                                void* w2_packed, void* w13_scale_packed, void* w2_scale_packed,
                                void* stream) {
  if (!p || p->E <= 0 || p->I <= 0 || p->I % 128 || p->H <= 0 || p->H % 128 || p->latent < 0 ||
      p->latent % 128)
    return MOE_ERR_INVALID_ARG;
  if (p->wfmt != MOE_W_FP8_E4M3_PER_CHANNEL && p->wfmt != MOE_W_MXFP4_E2M1_E8M0_B32 &&
      p->wfmt != MOE_W_FP8_E4M3_BLOCK128)
    return MOE_ERR_INVALID_ARG;
  if (!w13 || !w2 || !w13_packed || !w2_packed) return MOE_ERR_INVALID_ARG;
  if (w13 == w13_packed || w2 == w2_packed) return MOE_ERR_INVALID_ARG;
  const uintptr_t al = reinterpret_cast<uintptr_t>(w13) | reinterpret_cast<uintptr_t>(w2) |
                       reinterpret_cast<uintptr_t>(w13_packed) |
                       reinterpret_cast<uintptr_t>(w2_packed);
  if (al % 16) return MOE_ERR_INVALID_ARG;
  const int E = p->E, I = p->I, K = p->latent > 0 ? p->latent : p->H;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool mx = p->wfmt == MOE_W_MXFP4_E2M1_E8M0_B32;
  if (mx) {
    if (!w13_scale || !w2_scale || !w13_scale_packed || !w2_scale_packed) return MOE_ERR_INVALID_ARG;
    if (w13_scale == w13_scale_packed || w2_scale == w2_scale_packed) return MOE_ERR_INVALID_ARG;
    const uintptr_t sa = reinterpret_cast<uintptr_t>(w13_scale) |
                         reinterpret_cast<uintptr_t>(w2_scale) |
                         reinterpret_cast<uintptr_t>(w13_scale_packed) |
                         reinterpret_cast<uintptr_t>(w2_scale_packed);
    if (sa % 16) return MOE_ERR_INVALID_ARG;
  }
  cudaError_t e;
  if (mx) {
    if (K % 256) return MOE_ERR_INVALID_ARG;
    // w13: block pair p = (W1 rows p*128.., W3 rows I + p*128..); w2: rows p*256..
    e = pack_mx(w13, w13_packed, w13_scale, w13_scale_packed, E, 2 * I, K, 1, I, s);
    if (e == cudaSuccess) e = pack_mx(w2, w2_packed, w2_scale, w2_scale_packed, E, K, I, 2, 128, s);
  } else {
    // w13 [E][2I][K], w2 [E][K][I]; tiles of 128 rows x 128 bytes
    e = pack_tiles(w13, w13_packed, E, 2 * I, K, 128, s);
    if (e == cudaSuccess) e = pack_tiles(w2, w2_packed, E, K, I, 128, s);
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
