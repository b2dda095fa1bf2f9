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
#include <cuda_runtime.h>

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
unsigned char* g_staging_addr[kMaxDevices];  // device address of g_staging, per device

// The array's device address on `dev` (the current device), looked up once.
// In host code g_staging names a host-side shadow, never device memory.
fm_status staging_address(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return FM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_staging_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_staging) != cudaSuccess || p == nullptr) return FM_ERR_CUDA;
    g_staging_addr[dev] = static_cast<unsigned char*>(p);
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
