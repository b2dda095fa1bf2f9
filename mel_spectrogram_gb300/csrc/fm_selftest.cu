// fm_selftest_wait_timeout: the bounded wait of the mel kernels, run out on
// purpose, so the timeout path can be tested without faulting or hanging a
// GPU. One CTA of two groups of 64 threads waits on two mbarriers with the
// kernels' own waits and exit vote (group_sync_or): group 1's barrier
// completes by an arrival, group 0's by nothing, so group 0 gives up after its
// polls, records FM_ERR_KERNEL_TIMEOUT in the plan's error word and leaves
// through its OR-vote barrier while group 1 finishes normally. Kind 0 is the
// groups' wait for a staged tile (mbar_wait_polls: blocking try_wait polls),
// kind 1 the producer warp's wait for a free staging area (non-blocking
// test_wait with idle_backoff).
#include <cuda_runtime.h>

#include <mutex>

#include "fm_host.h"
#include "fm_kernel_x2.cuh"
#include "fm_mel.h"

namespace fm {

// groups of the self-test CTA that passed their wait (read back by the host)
static __device__ unsigned g_selftest_completed;

__global__ void __launch_bounds__(128, 1) wait_timeout_kernel(unsigned* err, int kind, int polls) {
  __shared__ unsigned long long bar[2];
  const int tid = threadIdx.x, grp = tid >> 6, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (grp == 1 && (tid & 63) == 0) mbar_arrive(&bar[1]);  // nothing arrives on bar[0]
  bool ok;
  if (kind == 0 || grp == 1) {
    // the groups' wait for a staged tile
    ok = mbar_wait_polls(&bar[grp], 0u, err, polls);
  } else {
    // the producer warp's wait for a free staging area: non-blocking tests
    // with back-off, the warp agreeing through lane 0 as the producer does
    int idle = 0;
    for (;;) {
      int ready = mbar_test_wait(&bar[0], 0u) ? 1 : 0;
      ready = __shfl_sync(0xffffffffu, ready, 0);
      if (ready) break;
      if (!idle_backoff(idle, polls)) {
        if (lane == 0) atomicExch(err, (unsigned)FM_ERR_KERNEL_TIMEOUT);
        break;
      }
    }
    ok = idle <= polls;
  }
  if (group_sync_or(1 + grp, 64, !ok)) return;  // the group leaves together, error recorded
  if ((tid & 63) == 0) atomicAdd(&g_selftest_completed, 1u);
}

}  // namespace fm

namespace {
std::mutex g_selftest_mu;  // one self-test at a time per process (one counter per device)
}

extern "C" fm_status fm_selftest_wait_timeout(const fm_plan* plan, int kind, int log2_polls, fm_stream_t stream,
                                              int* groups_completed, double* elapsed_us) {
  if (plan == nullptr || (kind != 0 && kind != 1)) return FM_ERR_INVALID_ARG;
  if (log2_polls < 0 || log2_polls > (kind == 0 ? fm::kWaitLog2Polls : fm::kIdleLog2Polls)) return FM_ERR_INVALID_ARG;
  fm_plan_info info;
  fm_status st = fm_plan_get_info(plan, &info);
  if (st != FM_OK) return st;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != info.device) return FM_ERR_CUDA;
  unsigned* err = fm::plan_error_word(plan);
  if (err == nullptr) return FM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_selftest_mu);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const unsigned zero = 0;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(fm::g_selftest_completed, &zero, sizeof(zero), 0,
                                                    cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaEventRecord(e0, s);
  if (e == cudaSuccess) {
    fm::wait_timeout_kernel<<<1, 128, 0, s>>>(err, kind, 1 << log2_polls);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaEventRecord(e1, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  unsigned done = 0;
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&done, fm::g_selftest_completed, sizeof(done));
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (e != cudaSuccess) return FM_ERR_CUDA;
  if (groups_completed) *groups_completed = (int)done;
  if (elapsed_us) *elapsed_us = 1e3 * (double)ms;
  return FM_OK;
}
