// mnw_selftest.cu -- a self-test of the library's failure detection on the GPU.
//
// Every wait inside the library's kernels is bounded (bounded_wait in
// mnw_ptx.cuh): when one runs out it ORs MNW_DEVERR_TIMEOUT into the caller's
// error word and raises the CTA's abort flag, and every other role of the CTA
// leaves its own wait when it sees the flag.  This entry point exercises
// exactly that code without any fault: one CTA of two warps, each waiting on
// an mbarrier phase that nothing completes.  Warp 0 waits with the caller's
// short limit and times out; warp 1 waits with the library's full limit and
// must leave early through the abort flag.  The kernel then returns normally,
// so the context stays usable.
#include "mnw_internal.h"
#include "mnw_ptx.cuh"

namespace mnw {
namespace {

__global__ void __launch_bounds__(64, 1) wait_timeout_kernel(uint64_t limit_ns, uint32_t* err, uint32_t* left_early) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane != 0) return;
  // phase 0 of both barriers never completes: nobody arrives
  if (warp == 0) {
    bounded_wait_for(&bars[0], 0, abort, err, limit_ns);
  } else {
    const uint64_t t0 = globaltimer();
    const bool done = bounded_wait(&bars[1], 0, abort, err);
    if (!done && globaltimer() - t0 < kWaitLimitNs / 2) atomicOr(left_early, 1u);
  }
}

// One thread waits, with the caller's limit, for *counter >= need: the wait a
// dependent launch uses for a token tile released by the launch before it.
__global__ void __launch_bounds__(32, 1) counter_timeout_kernel(const uint32_t* counter, uint32_t need,
                                                                uint64_t limit_ns, uint32_t* err) {
  if (threadIdx.x == 0) bounded_poll_ge_for(counter, need, nullptr, err, limit_ns);
}

}  // namespace
}  // namespace mnw

extern "C" int mnw_moe_selftest_wait_timeout(uint32_t limit_us, uint32_t* err, uint32_t* left_early,
                                             mnw_stream stream) {
  if (!err || !left_early || limit_us == 0 || limit_us > 1000000u) return MNW_E_INVALID_ARG;
  mnw::wait_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint64_t>(limit_us) * 1000u,
                                                                            err, left_early);
  if (cudaGetLastError() != cudaSuccess) return MNW_E_CUDA;
  mnw::note_launch();
  return MNW_OK;
}

extern "C" int mnw_moe_selftest_counter_timeout(uint32_t limit_us, const uint32_t* counter, uint32_t need,
                                                uint32_t* err, mnw_stream stream) {
  if (!counter || !err || limit_us == 0 || limit_us > 1000000u) return MNW_E_INVALID_ARG;
  mnw::counter_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      counter, need, static_cast<uint64_t>(limit_us) * 1000u, err);
  if (cudaGetLastError() != cudaSuccess) return MNW_E_CUDA;
  mnw::note_launch();
  return MNW_OK;
}
