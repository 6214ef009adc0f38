// pack.cu -- one-time repack of expert weights into tile-major order.
//
// The fp8 grouped GEMMs stream each expert's weights as 128-row x 128-byte
// tiles (one per pipeline stage).  In the row-major layout a tile is 128
// separate 128-byte pieces, one per weight row.  Stored tile-major,
// [group][row_block][k_block][128 rows][128 bytes], every stage reads one
// contiguous 16 KB block.  This is the usual load-time weight processing step;
// the bytes are only permuted.  MXFP4 weights stay row-major: their stages are
// half the bytes and the tile order measured slower for them.
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
  if (p->wfmt != MOE_W_FP8_E4M3_PER_CHANNEL) return MOE_ERR_UNSUPPORTED;
  if (!w13 || !w2 || !w13_packed || !w2_packed) return MOE_ERR_INVALID_ARG;
  if (w13 == w13_packed || w2 == w2_packed) return MOE_ERR_INVALID_ARG;
  const uintptr_t al = reinterpret_cast<uintptr_t>(w13) | reinterpret_cast<uintptr_t>(w2) |
                       reinterpret_cast<uintptr_t>(w13_packed) |
                       reinterpret_cast<uintptr_t>(w2_packed);
  if (al % 16) return MOE_ERR_INVALID_ARG;
  const int E = p->E, I = p->I, K = p->latent > 0 ? p->latent : p->H;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  (void)w13_scale, (void)w2_scale, (void)w13_scale_packed, (void)w2_scale_packed;
  // w13 [E][2I][K], w2 [E][K][I]; tiles of 128 rows x 128 bytes
  cudaError_t e = pack_tiles(w13, w13_packed, E, 2 * I, K, 128, s);
  if (e == cudaSuccess) e = pack_tiles(w2, w2_packed, E, K, I, 128, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
