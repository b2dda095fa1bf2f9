// fm_mel_forward_host_noalloc: the host-buffer entry point with its device
// staging in a fixed, statically allocated array instead of caller buffers.
//
// Some callers hold their audio in host memory and cannot allocate device
// memory when they want a spectrogram: a real-time audio callback, where
// cudaMalloc's implicit device synchronisation and unbounded latency would
// miss the deadline, or a process whose device memory belongs to another
// framework's allocator. fm_mel_forward_host needs two device buffers from
// them; this entry point needs none. It stages the input and the output in
// one array of FM_NOALLOC_MAX_BYTES that every GPU loading this library holds
// until the process exits, and calls no allocating routine.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "fm_mel.h"

namespace {

constexpr size_t kStagingBytes = FM_NOALLOC_MAX_BYTES;
constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;

// Input samples at offset 0, the spectrogram at the next 256-byte boundary.
// Neither part needs clearing between calls: the host-to-device copy
// overwrites every input byte a call reads and the kernel writes every output
// element the call copies back.
static __device__ __align__(256) unsigned char g_staging[kStagingBytes];

std::mutex g_setup_mu;
// device address of g_staging per device, and the context it was looked up in
unsigned char* g_staging_addr[kMaxDevices];
CUcontext g_staging_ctx[kMaxDevices];

// cuCtxGetCurrent from the driver, resolved once through the runtime (no link
// against libcuda); null if unavailable.
PFN_cuCtxGetCurrent_v4000 ctx_getter() {
  static const PFN_cuCtxGetCurrent_v4000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_cuCtxGetCurrent_v4000) nullptr;
    return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  }();
  return fn;
}

// The array's device address on `dev` (the current device). It is looked up
// the first time a context of `dev` is current here, and again whenever the
// current context differs from the one it was looked up in (a context
// created by the caller, or the primary context after cudaDeviceReset), so a
// stale address is never used. In host code g_staging names a host-side
// shadow, never device memory.
fm_status staging_address(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return FM_ERR_UNSUPPORTED;
  const PFN_cuCtxGetCurrent_v4000 get_ctx = ctx_getter();
  if (get_ctx == nullptr) return FM_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return FM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  // no context bound to this thread yet (ctx null): the look-up binds the
  // device's primary context, which is then read back
  if (ctx == nullptr || g_staging_addr[dev] == nullptr || g_staging_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_staging) != cudaSuccess || p == nullptr) return FM_ERR_CUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return FM_ERR_CUDA;
    g_staging_addr[dev] = static_cast<unsigned char*>(p);
    g_staging_ctx[dev] = ctx;
  }
  *out = g_staging_addr[dev];
  return FM_OK;
}

size_t dtype_bytes(int dt) { return dt == FM_F32 ? 4 : 2; }

}  // namespace

extern "C" fm_status fm_mel_forward_host_noalloc(const fm_plan* plan, const void* h_in, int64_t B, int64_t T,
                                                 void* h_out, fm_stream_t stream) {
  if (plan == nullptr || B < 0) return FM_ERR_INVALID_ARG;
  if (B == 0) return FM_OK;
  if (h_in == nullptr || h_out == nullptr) return FM_ERR_INVALID_ARG;
  fm_plan_info info;
  fm_status st = fm_plan_get_info(plan, &info);
  if (st != FM_OK) return st;
  const int64_t n_frames = fm_n_frames(plan, T);  // -1 if T is too short for the plan's framing
  if (n_frames < 1) return FM_ERR_INVALID_ARG;
  // sizes, checked against the array before any product can overflow
  const int64_t cap = (int64_t)kStagingBytes;
  if (B > cap || T > cap / B) return FM_ERR_INVALID_ARG;
  if (n_frames > cap / B || (int64_t)info.n_mels > cap / (B * n_frames)) return FM_ERR_INVALID_ARG;
  const size_t in_bytes = (size_t)B * (size_t)T * dtype_bytes(info.in_dtype);
  const size_t out_bytes = (size_t)B * (size_t)info.n_mels * (size_t)n_frames * dtype_bytes(info.out_dtype);
  const size_t out_off = (in_bytes + kAlign - 1) / kAlign * kAlign;
  if (out_off > kStagingBytes || out_bytes > kStagingBytes - out_off) return FM_ERR_INVALID_ARG;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != info.device) return FM_ERR_CUDA;
  unsigned char* base = nullptr;
  st = staging_address(dev, &base);
  if (st != FM_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(base, h_in, in_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return FM_ERR_CUDA;
  st = fm_mel_forward(plan, base, B, T, base + out_off, stream);
  if (st != FM_OK) return st;
  if (cudaMemcpyAsync(h_out, base + out_off, out_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FM_ERR_CUDA;
  return FM_OK;
}
