// permute_static.cu -- moe_permute for callers that cannot allocate.
//
// moe_permute needs two small scratch tables (per 32-token chunk and expert:
// how many rows, and where the chunk's rows start), which it carves from the
// caller's workspace.  Some callers have no workspace to lend: a host that
// plans every byte of device memory up front and only hands a plugin its input
// and output buffers, or a latency-critical loop where cudaMalloc is not
// allowed because it can synchronise the device.  moe_permute_static serves
// them: the two tables live in a fixed array in this library's own device
// memory (kStaticTableInts int32 each, 4 MiB in total, plus one word the scan
// counts its finished blocks on; held on every GPU that loads the library
// until the process exits), so the caller passes only inputs and outputs.
//
// Limits and sharing: a problem needs E * ceil(T / 32) <= kStaticTableInts
// entries per table; larger problems are rejected with MOE_ERR_WORKSPACE.  All
// calls on a device share the array and it keeps the last call's contents.
// Nothing in it has to start at zero (each call writes every entry it later
// reads), but two calls whose kernels overlap on the GPU (different streams,
// or different host threads) race on the array: serialise them.
#include <mutex>

#include "../../include/moe.h"
#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int64_t kStaticTableInts = int64_t(1) << 19;  // 2 MiB per table

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) int32_t g_permute_scratch[2 * kStaticTableInts + 64];

constexpr int kMaxDev = 64;
int32_t* g_scratch_addr[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of g_permute_scratch on the current device, looked up once per
// device (with that device current) and cached; nullptr on failure.
int32_t* scratch_address() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_addr[d] = static_cast<int32_t*>(p);
  }
  return g_scratch_addr[d];
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_permute_static(const moe_problem* p, const int32_t* topk_idx, const void* x,
                                  int32_t* counts, int32_t* offsets, int32_t* perm,
                                  int32_t* src_row, void* xq_perm, float* xscale_perm,
                                  void* stream) {
  const int st = check_problem(p);  // the same checks as moe_permute
  if (st) return st;
  if (!topk_idx || !x || !counts || !offsets || !perm || !src_row || !xq_perm || !xscale_perm)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(xq_perm)) % 16)
    return MOE_ERR_INVALID_ARG;
  const int T = p->T, E = p->E, k = p->top_k;
  const int K = p->latent > 0 ? p->latent : p->H;
  const int64_t table = (int64_t)E * num_chunks(T);
  if (table > kStaticTableInts) return MOE_ERR_WORKSPACE;  // beyond the fixed scratch
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  int32_t* scratch = scratch_address();
  int* err = device_error_word();
  if (!scratch || !err) return MOE_ERR_CUDA;
  int32_t* cc = scratch;                       // per-chunk counts  [E, nch]
  int32_t* cbase = scratch + kStaticTableInts;  // per-chunk bases   [E, nch]
  int32_t* ticket = scratch + 2 * kStaticTableInts;  // the scan's completion count
  if (launch_count(topk_idx, cc, ticket, T, E, k, err, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_scan(cc, cbase, counts, offsets, ticket, T, E, k, nullptr, nullptr, 0, 32, 0, 0, s) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_rank(topk_idx, nullptr, offsets, cbase, perm, src_row, nullptr, T, E, k, s) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_quant_scatter(x, perm, xq_perm, xscale_perm, T, K, k, -1, err, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
