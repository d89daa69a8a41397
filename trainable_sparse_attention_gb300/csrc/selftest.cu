// Self-test of the failure path of the bounded device waits, with no fault.
//
// One CTA waits on a shared-memory mbarrier that no thread ever arrives on,
// with the same bounded wait (tc::mbar_wait) that every pipeline of the
// library uses.  The wait gives up after its time limit, the CTA raises
// TSA_FLAG_TIMEOUT in the library's flag word and returns normally, so the
// CUDA context stays usable; the host reads the flag with tsa_read_flags.
#include "kernels.cuh"
#include "tc.cuh"

namespace tsa {

namespace {

__global__ void __launch_bounds__(32, 1) bounded_wait_selftest_kernel(unsigned int* flags) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);  // one expected arrival that never comes
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  // phase 0 of a fresh barrier completes only on an arrival, so every lane waits out the limit
  const bool done = tc::mbar_wait(&bar, 0, &abort_flag);
  if (!__any_sync(0xffffffffu, done) && threadIdx.x == 0) raise_flag(flags, TSA_FLAG_TIMEOUT);
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(unsigned int* flags, cudaStream_t stream) {
  if (flags == nullptr) return cudaErrorInvalidValue;
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(flags);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tsa
