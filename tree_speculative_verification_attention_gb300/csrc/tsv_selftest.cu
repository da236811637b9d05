// tsv_selftest.cu — a self-test of the bounded device-side wait that every
// kernel of the library uses (mbar_wait in tsv_device.cuh).
//
// One CTA of two warps sets up two mbarriers and waits on both, one per warp,
// through the same helper the attention and verification kernels call.  With
// `arrive` set, thread 0 completes both barriers first and the waits return at
// once.  Without it nothing ever arrives: the first wait to reach the time
// limit raises the CTA's abort flag, the other wait sees the flag and gives up
// too, and the kernel records TSV_ERR_TIMEOUT and returns normally.  This is
// how a caller can check, on its own device, that a stalled wait ends in an
// error status (and a usable context) rather than a hang; it needs no fault.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tsv.h"
#include "tsv_device.cuh"

namespace tsv {
namespace {

__global__ void __launch_bounds__(64, 1)
    bounded_wait_selftest_kernel(int32_t arrive, int32_t* status, int64_t* elapsed_ns) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  volatile int* abort_v = &abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const uint64_t t0 = global_timer_ns();
  if (tid == 0 && arrive) {
    mbar_arrive(&bars[0]);
    mbar_arrive(&bars[1]);
  }
  bool ok = true;
  if (lane == 0) ok = mbar_wait(&bars[warp], 0, abort_v);
  // An abort raised by either warp fails the whole CTA, as in the kernels.
  const bool timed_out = __syncthreads_or(lane == 0 && !ok) || *abort_v;
  if (tid == 0) {
    *status = timed_out ? TSV_ERR_TIMEOUT : TSV_OK;
    if (elapsed_ns != nullptr) *elapsed_ns = (int64_t)(global_timer_ns() - t0);
  }
}

}  // namespace
}  // namespace tsv

extern "C" tsv_status tsv_selftest_bounded_wait(tsv_handle h, int32_t arrive, int32_t* status_d,
                                                int64_t* elapsed_ns_d, void* stream) {
  if (!h || !status_d) return TSV_ERR_INVALID_ARG;
  tsv::bounded_wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(
      arrive, status_d, elapsed_ns_d);
  return cudaGetLastError() == cudaSuccess ? TSV_OK : TSV_ERR_CUDA;
}
