// lion_debug.cu -- the bound on device-side waits, and a probe that makes one
// run out.
//
// Every warp-specialised tensor-core kernel of this library hands work
// between its warps through mbarriers and waits on them with
// mbar_wait_or_abort: a wait that has not completed after the bound records
// a timeout in the library's status word, makes every other wait of the CTA
// give up, and the CTA unwinds (its copies and matrix products in flight are
// waited for, its tensor memory freed) instead of spinning forever.  The
// bound is a launch parameter of those kernels, taken from
// wait_limit_cycles() at each launch.
//
// lion_debug_wait_timeout runs that same wait on an mbarrier that nothing
// ever arrives at, in a one-warp kernel with no copy and no matrix product
// in flight, so that the timeout path can be exercised on a GPU without a
// hang: the wait gives up after the bound, the kernel records the timeout
// and returns, and the next lion_sync_status reports LION_ERR_TIMEOUT.
#include <atomic>

#include "../../include/lion.h"
#include "lion_common.cuh"
#include "lion_internal.h"
#include "tc_ptx.cuh"

namespace lion {
namespace {

constexpr long long kDefaultWaitCycles = 2000000000LL;   // about 1 s at 2 GHz
std::atomic<long long> g_wait_cycles{kDefaultWaitCycles};

__global__ void __launch_bounds__(32) lion_wait_probe_kernel(int* status, long long limit) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);   // one arrival would complete phase 0; none comes
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncwarp();
  const bool done = tc::mbar_wait_or_abort(&bar, 0, limit, 2000u, &abort_flag);
  __syncwarp();
  if (threadIdx.x == 0 && (!done || abort_flag)) atomicExch(status, kStatusTimeout);
}

}  // namespace

long long wait_limit_cycles() { return g_wait_cycles.load(std::memory_order_relaxed); }

}  // namespace lion

extern "C" {

lion_status lion_debug_set_wait_cycles(long long cycles) {
  if (cycles < 0) return LION_ERR_INVALID_ARG;
  lion::g_wait_cycles.store(cycles == 0 ? lion::kDefaultWaitCycles : cycles, std::memory_order_relaxed);
  return LION_OK;
}

lion_status lion_debug_wait_timeout(cudaStream_t stream) {
  int* status = lion::device_status_ptr();
  if (!status) return LION_ERR_CUDA;
  lion::lion_wait_probe_kernel<<<1, 32, 0, stream>>>(status, lion::wait_limit_cycles());
  return cudaGetLastError() == cudaSuccess ? LION_OK : LION_ERR_CUDA;
}

}  // extern "C"
