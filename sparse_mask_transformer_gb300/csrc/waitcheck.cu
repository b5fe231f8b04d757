// Diagnostic of this library's failure handling (no counterpart in the
// paper): every pipeline wait in the attention kernels is an mbarrier wait
// bounded in wall time (sm100_ptx.cuh, mbar_wait), after which the kernel
// reports STOF_DEVERR_PIPE_TIMEOUT in a device error word and finishes
// instead of hanging.  stof_check_bounded_wait() runs that same wait on an
// mbarrier that nothing ever arrives on, so a test can watch it give up and
// report, and check that the context stays usable afterwards.
#include <cuda_runtime.h>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace stof {

namespace {

__global__ void bounded_wait_kernel(int64_t* err, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  // phase 0 of bar never completes: the wait can only run out
  if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, &abort_flag, timeout_ns))
    atomicOr(reinterpret_cast<unsigned long long*>(err), static_cast<unsigned long long>(STOF_DEVERR_PIPE_TIMEOUT));
}

}  // namespace

}  // namespace stof

extern "C" stof_status stof_check_bounded_wait(int64_t* device_error, double seconds, void* stream) {
  if (!device_error || !(seconds > 0.0) || seconds > 10.0) return STOF_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(device_error) % 8) return STOF_ERR_ALIGNMENT;
  const unsigned long long ns = static_cast<unsigned long long>(seconds * 1e9);
  stof::bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(device_error, ns);
  return stof::record_cuda(cudaGetLastError()) == cudaSuccess ? STOF_OK : STOF_ERR_CUDA;
}
