// watchdog.cu -- self-test of the bounded pipeline waits.
//
// Every producer / MMA / epilogue wait in the tcgen05 + TMA kernels goes
// through mbar_wait (device.cuh): it gives up after kWaitTimeoutNs, records
// MOE_ERR_TIMEOUT in the per-device error word and raises the CTA's abort
// flag, so that the other roles stop waiting and the CTA can free its tensor
// memory and return with the context intact.  This kernel runs that machinery
// on a CTA laid out like the GEMMs (one warp holding tensor memory, others
// waiting on pipeline barriers) whose barriers nothing ever arrives on: no
// copy or MMA is in flight, so the expiry is the only way out of the waits.
#include "../../include/moe.h"
#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kRoles = 4;  // warps

__global__ void __launch_bounds__(kRoles * 32, 1)
    watchdog_selftest_kernel(int* err, int32_t* role_status) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_flag;
  volatile int* s_abort = &s_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    *s_abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(&s_tmem), 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  // warp 0 plays the producer waiting for a free slot, warps 1..3 the MMA and
  // epilogue roles waiting for data; nobody arrives on either barrier.
  const uint32_t bar = smem_u32(&bars[warp == 0 ? 0 : 1]);
  const bool ok = mbar_wait(bar, 0u, err, s_abort);
  __syncwarp();
  if (lane == 0 && role_status) role_status[warp] = ok ? 1 : 0;

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_watchdog_selftest(int32_t* role_status, void* stream) {
  int* err = device_error_word();
  if (!err) return MOE_ERR_CUDA;
  count_launch();
  watchdog_selftest_kernel<<<1, kRoles * 32, 0, static_cast<cudaStream_t>(stream)>>>(err,
                                                                                   role_status);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
