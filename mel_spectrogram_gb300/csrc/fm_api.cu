// C-ABI layer: plan creation (validation, host tables, device upload) and the
// launch of the fused kernel. See include/fm_mel.h for the contract.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <cudaTypedefs.h>

#include "fm_host.h"
#include "fm_internal.h"
#include "fm_kernel_big.cuh"
#include "fm_kernel_c2c.cuh"
#include "fm_mel.h"

namespace fm {
extern const Variant kVariant64, kVariant128, kVariant256, kVariant400, kVariant400h160, kVariant512x2, kVariant512,
    kVariant1024, kVariant2048, kVariant4096, kVariant8192, kVariant16384;
extern const Variant kVariant256g2, kVariant256g1, kVariant400g2, kVariant400g1, kVariant512g1;
extern const Variant kVariant64odd, kVariant128odd, kVariant256odd, kVariant400odd, kVariant512odd,
    kVariant1024odd, kVariant2048odd;
extern const Variant kVariant400c2c, kVariant400h160x2h;
extern const Variant kVariant400h100, kVariant400h200, kVariant128h32, kVariant256h64, kVariant512h128;
extern const Variant kVariant1024big, kVariant2048big;
extern const Variant kVariant4096dif, kVariant8192dif, kVariant16384dif;

// The kernels for (n_fft, hop), in order: a build for exactly this hop if
// there is one, then those for its parity (even hops stage and read aligned
// sample pairs: the packed two-frame kernel, with fewer tile groups per CTA
// for longer hops, ahead of the one-frame kernel; odd hops take the generic
// kernel's contiguous staging), then those for any hop (the large-transform
// kernels: at n_fft 8192 and 16384 the decimation-in-frequency build ahead
// of the three-pass one; last at 1024 and 2048, where the three-pass build
// takes the hops the others have no shared memory for).
const Variant* find_variant(int n_fft, int hop, const Variant* after) {
  static const Variant* all[] = {&kVariant400h160, &kVariant400h100, &kVariant400h200, &kVariant128h32,
                                 &kVariant256h64,  &kVariant512h128, &kVariant64,      &kVariant128,
                                 &kVariant256,     &kVariant256g2,   &kVariant256g1,   &kVariant400,
                                 &kVariant400g2,   &kVariant400g1,   &kVariant512x2,   &kVariant512g1,
                                 &kVariant512,     &kVariant1024,    &kVariant2048,    &kVariant4096,
                                 &kVariant8192dif, &kVariant8192,    &kVariant16384dif, &kVariant16384,
                                 &kVariant64odd,   &kVariant128odd,
                                 &kVariant256odd,  &kVariant400odd,  &kVariant512odd,  &kVariant1024odd,
                                 &kVariant2048odd, &kVariant1024big, &kVariant2048big};
  const bool even = hop % 2 == 0;
  // diagnostic A/B switches: the paired-frame complex transform at n_fft 400
  // (even hops) instead of the two-frame packed kernel; the
  // decimation-in-frequency build of the large-transform kernel at 4096, the
  // three-pass build at 8192 and 16384
  if (after == nullptr && n_fft == 400 && even) {
    const char* k = std::getenv("FM_MEL_N400_KERNEL");
    if (k != nullptr && std::strcmp(k, "c2c") == 0) return &kVariant400c2c;
    if (k != nullptr && std::strcmp(k, "x2h") == 0 && hop == 160) return &kVariant400h160x2h;
  }
  if (after == nullptr && (n_fft == 4096 || n_fft == 8192 || n_fft == 16384)) {
    const char* k = std::getenv("FM_MEL_BIG_KERNEL");
    if (k != nullptr && std::strcmp(k, "dif") == 0 && n_fft == 4096) return &kVariant4096dif;
    if (k != nullptr && std::strcmp(k, "passes") == 0 && n_fft != 4096)
      return n_fft == 8192 ? &kVariant8192 : &kVariant16384;
  }
  // up to and including `after` (a diagnostic choice falls back to the list)
  bool skip = after != nullptr && after != &kVariant400c2c && after != &kVariant400h160x2h &&
              after != &kVariant4096dif;
  for (const Variant* v : all) {
    if (skip) {
      skip = v != after;
      continue;
    }
    if (v->n_fft != n_fft) continue;
    if (v->hop > 0 ? v->hop == hop : (v->hop == kAnyHop || (v->hop == kEvenHops) == even)) return v;
  }
  return nullptr;
}
}  // namespace fm

// Copy-in / kernel / copy-out pipeline of fm_mel_forward_host: three
// streams and the events that chain one call's chunks; the enqueue of one
// call holds the mutex, so calls from several host threads do not interleave
// their use of the events.
constexpr int kHostChunks = 4;
constexpr size_t kHostChunkMinBytes = (size_t)2 << 20;  // input + output bytes of one chunk, at least
struct HostPipe {
  std::mutex mu;
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in_done[kHostChunks] = {}, comp_done[kHostChunks] = {};
};

struct fm_plan {
  int device;
  int sr, n_fft, hop, win_length, n_mels;
  int center, pad_mode, zpad, normalized;  // framing options (fm_plan_create_ex)
  double f_min, f_max, power;
  int mel_scale, norm, in_dtype, out_dtype, power_mode;
  const fm::Variant* var;
  int nnz;
  size_t smem;
  int blocks_per_sm, grid_limit, num_sms;
  void* dmem;
  float4* p1;
  float2* tw_half;
  float2* tw_full;
  int4* mel;
  float* mel_w;
  unsigned* err;
  float* win;        // the window, for the large-transform kernel (inside dmem)
  fm::X2Tables* x2;  // device tables of the two-frames-per-thread kernel (inside dmem)
  mutable HostPipe pipe;  // streams and events of fm_mel_forward_host
  int x2_slots;         // its mel chunk slots
  int big_span;         // large-transform kernel: samples staged per tile (0: loads from global memory)
  int mel_taps;         // decimation-in-frequency large-transform kernel: the mel mapping (KernelParams)
  float2* c2c;          // paired-frame kernel: its pass-1 table, then W_400^j (inside dmem)
};

namespace {

int dtype_size(int dt) { return dt == FM_F32 ? 4 : 2; }

// Mel mapping of the decimation-in-frequency large-transform kernel (16
// warps, F frames a tile), from the filters' tap counts ml: the estimated
// critical path of one tile's projection in SM cycles under each mapping,
// the cheaper one wins. A lane per filter and frame (mel_project_lanes): a
// warp's filters run side by side, so a warp takes its widest filter's taps,
// about 33 cycles each; a warp per filter (mel_project_taps): about 40 cycles
// per 32 taps plus 300 per filter (its shuffle sum and store). Measured on
// GB300, a warp per filter was the faster mapping on every configuration
// tried: 272.5 against 281.6 us at n_fft 16384 with 256 filters to 22.05 kHz
// (16 x 30 s, hop 4096), 69.8 against 86.2 us at 16384 and 69.3 against
// 70.9 us at 8192 with 128 filters to 8 kHz (32 x 10 s, hop n_fft / 4); with
// these constants the estimate agrees on all three and leaves the lanes to
// banks of a few narrow filters. FM_MEL_BIG_MEL=taps or lanes overrides it.
bool choose_mel_taps(const std::vector<int>& ml, int F) {
  const char* k = std::getenv("FM_MEL_BIG_MEL");
  if (k != nullptr && std::strcmp(k, "taps") == 0) return true;
  if (k != nullptr && std::strcmp(k, "lanes") == 0) return false;
  constexpr int kWarps = fm::kBigThreads / 32;
  const int n = (int)ml.size(), subs = 32 / F;
  long long lanes = 0, taps = 0;
  for (int w = 0; w < kWarps; ++w) {
    long long tl = 0, tt = 0;
    for (int base = w * subs; base < n; base += kWarps * subs) {
      int widest = 0;
      for (int s = 0; s < subs && base + s < n; ++s) widest = std::max(widest, ml[base + s]);
      tl += widest;
    }
    for (int m = w; m < n; m += kWarps) tt += 40LL * ((ml[m] + 31) / 32) + 300;
    lanes = std::max(lanes, 33 * tl);
    taps = std::max(taps, tt);
  }
  return taps < lanes;
}

// Mel schedule of the two-frames-per-thread kernel: four chunk streams per
// warp (one per quarter-warp). Each filter is padded to an even length
// L >= 2 (zero weights; a run that would pass bin M is shifted left) and cut
// into L/2 two-bin chunks; filters are dealt to streams to balance their
// chunk counts (largest first onto the least loaded stream), and the four
// streams of a warp are padded with no-op chunks to one length, a multiple of
// the kernel's unroll. Layout as in X2Tables.
struct X2Schedule {
  std::vector<int> warp_begin;
  std::vector<int2> desc;   // 4 per slot
  std::vector<float4> w4;   // 4 per slot
};

X2Schedule build_x2_schedule(int M, int n_mels, int n_warps, const std::vector<int>& ms, const std::vector<int>& ml,
                             const std::vector<int>& mo, const std::vector<float>& mw) {
  struct Chunk { int2 d; float4 w; };
  auto chunks_of = [&](int m) {
    int L = ml[m] + (ml[m] & 1);
    L = L < 2 ? 2 : L;
    int start = ms[m], lead = 0;
    if (start + L > M + 1) {
      lead = start + L - (M + 1);
      start -= lead;
    }
    auto weight = [&](int j) {
      const int k2 = j - lead;
      return (k2 >= 0 && k2 < ml[m]) ? mw[mo[m] + k2] : 0.0f;
    };
    std::vector<Chunk> out;
    for (int c = 0; c < L / 2; ++c) {
      const float w0 = weight(2 * c), w1 = weight(2 * c + 1);
      out.push_back({make_int2((start + 2 * c) * 16 * (int)sizeof(float2), c == L / 2 - 1 ? m : -1),
                     make_float4(w0, w0, w1, w1)});
    }
    return out;
  };
  const int n_streams = 4 * n_warps;
  std::vector<int> order(n_mels);
  for (int m = 0; m < n_mels; ++m) order[m] = m;
  auto n_chunks = [&](int m) { return ml[m] < 2 ? 1 : (ml[m] + 1) / 2; };
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return n_chunks(a) > n_chunks(b); });
  std::vector<std::vector<Chunk>> stream(n_streams);
  for (int m : order) {
    int s = 0;
    for (int k = 1; k < n_streams; ++k)
      if (stream[k].size() < stream[s].size()) s = k;
    const std::vector<Chunk> c = chunks_of(m);
    stream[s].insert(stream[s].end(), c.begin(), c.end());
  }
  const Chunk noop = {make_int2(0, -1), make_float4(0.0f, 0.0f, 0.0f, 0.0f)};
  X2Schedule S;
  S.warp_begin.push_back(0);
  for (int w = 0; w < n_warps; ++w) {
    size_t len = 0;
    for (int h = 0; h < 4; ++h) len = std::max(len, stream[4 * w + h].size());
    len = (len + fm::kX2Unroll - 1) / fm::kX2Unroll * fm::kX2Unroll;
    for (size_t c = 0; c < len; ++c)
      for (int h = 0; h < 4; ++h) {
        const std::vector<Chunk>& st = stream[4 * w + h];
        const Chunk& k = c < st.size() ? st[c] : noop;
        S.desc.push_back(k.d);
        S.w4.push_back(k.w);
      }
    S.warp_begin.push_back(S.warp_begin.back() + (int)len);
  }
  return S;
}

// cuTensorMapEncodeTiled from the driver, resolved once through the runtime
// (no link against libcuda); null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// The packed kernel's tensor map over the input (see KernelParams::tmap):
// per signal, rows of one staged line starting at the sample where tile rows
// start (-pad mod line), each row wholly inside the signal; the box is a
// whole staged tile at the padded pitch. Left unset (tmap_ok = 0) when the
// layout does not allow it; the kernel then copies line by line.
void encode_input_map(const fm_plan* plan, const void* d_in, int64_t B, int64_t T, fm::KernelParams& prm) {
  prm.tmap_ok = 0;
  prm.tmap_off = 0;
  prm.tmap_rows = 0;
  const fm::Variant* v = plan->var;
  if (v->kind != 1) return;
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return;
  const int64_t esize = dtype_size(plan->in_dtype);
  const int kh = v->hop > 0 ? 2 : 1;
  const int64_t line = (int64_t)kh * plan->hop;
  const int64_t pitch = (int64_t)fm::in_row_stride_x2((int)line, (int)esize) * esize;  // bytes per staged row
  const int64_t rows = fm::x2_lines(plan->n_fft, plan->hop, kh);
  const int64_t lead = (plan->center ? plan->n_fft / 2 : 0) + plan->zpad;  // padding before sample 0
  const int64_t off = ((-lead) % line + line) % line;
  const uintptr_t base = reinterpret_cast<uintptr_t>(d_in) + (uintptr_t)(off * esize);
  if ((line * esize) % 16 != 0 || (T * esize) % 16 != 0 || base % 16 != 0) return;
  if (pitch / 8 > 256 || rows > 256 || B > ((int64_t)1 << 31) || T - off < line) return;
  const int64_t per_signal = (T - off) / line;
  if (per_signal > ((int64_t)1 << 31)) return;
  const cuuint64_t dims[3] = {(cuuint64_t)(line * esize / 8), (cuuint64_t)per_signal, (cuuint64_t)B};
  const cuuint64_t strides[2] = {(cuuint64_t)(line * esize), (cuuint64_t)(T * esize)};
  const cuuint32_t box[3] = {(cuuint32_t)(pitch / 8), (cuuint32_t)rows, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  if (encode(&prm.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, reinterpret_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return;
  prm.tmap_ok = 1;
  prm.tmap_off = (int)off;
  prm.tmap_rows = (int)per_signal;
}

fm_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return FM_OK;
  if (e == cudaErrorMemoryAllocation) return FM_ERR_OOM;
  return FM_ERR_CUDA;
}

void destroy_pipe(HostPipe& p) {
  for (cudaStream_t* st : {&p.in, &p.comp, &p.out})
    if (*st) cudaStreamDestroy(*st), *st = nullptr;
  for (cudaEvent_t* ev : {&p.start, &p.end})
    if (*ev) cudaEventDestroy(*ev), *ev = nullptr;
  for (int i = 0; i < kHostChunks; ++i) {
    if (p.in_done[i]) cudaEventDestroy(p.in_done[i]), p.in_done[i] = nullptr;
    if (p.comp_done[i]) cudaEventDestroy(p.comp_done[i]), p.comp_done[i] = nullptr;
  }
}

cudaError_t create_pipe(HostPipe& p) {
  cudaError_t e = cudaSuccess;
  for (cudaStream_t* st : {&p.in, &p.comp, &p.out})
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking);
  for (cudaEvent_t* ev : {&p.start, &p.end})
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  for (int i = 0; i < kHostChunks && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&p.in_done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.comp_done[i], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) destroy_pipe(p);
  return e;
}

}  // namespace

extern "C" fm_status fm_plan_create(fm_plan** out, int sr, int n_fft, int hop, int win_length, int n_mels,
                                    double f_min, double f_max, double power, fm_mel_scale mel_scale,
                                    fm_norm norm, fm_dtype in_dtype, fm_dtype out_dtype) {
  fm_plan_params p;
  p.sr = sr;
  p.n_fft = n_fft;
  p.hop = hop;
  p.win_length = win_length;
  p.n_mels = n_mels;
  p.f_min = f_min;
  p.f_max = f_max;
  p.power = power;
  p.mel_scale = mel_scale;
  p.norm = norm;
  p.in_dtype = in_dtype;
  p.out_dtype = out_dtype;
  p.center = 1;
  p.pad_mode = FM_PAD_REFLECT;
  p.pad = 0;
  p.normalized = FM_NORMALIZED_NONE;
  return fm_plan_create_ex(out, &p);
}

extern "C" fm_status fm_plan_create_ex(fm_plan** out, const fm_plan_params* params) {
  if (out == nullptr) return FM_ERR_INVALID_ARG;
  *out = nullptr;
  if (params == nullptr) return FM_ERR_INVALID_ARG;
  const int sr = params->sr, n_fft = params->n_fft, hop = params->hop, n_mels = params->n_mels;
  int win_length = params->win_length;
  const double f_min = params->f_min, power = params->power;
  double f_max = params->f_max;
  const fm_mel_scale mel_scale = params->mel_scale;
  const fm_norm norm = params->norm;
  const fm_dtype in_dtype = params->in_dtype, out_dtype = params->out_dtype;
  const int center = params->center ? 1 : 0, pad_mode = (int)params->pad_mode, zpad = params->pad;
  const int normalized = (int)params->normalized;
  if (pad_mode < FM_PAD_REFLECT || pad_mode > FM_PAD_CIRCULAR) return FM_ERR_INVALID_ARG;
  if (zpad < 0 || zpad > (1 << 20)) return FM_ERR_INVALID_ARG;
  if (normalized < FM_NORMALIZED_NONE || normalized > FM_NORMALIZED_FRAME_LENGTH) return FM_ERR_INVALID_ARG;
  if (win_length == 0) win_length = n_fft;
  if (sr <= 0 || n_fft <= 0 || hop <= 0 || n_mels <= 0) return FM_ERR_INVALID_ARG;
  if (win_length < 0 || win_length > n_fft) return FM_ERR_INVALID_ARG;
  if (!std::isfinite(power) || !(power > 0.0)) return FM_ERR_INVALID_ARG;
  if (in_dtype != FM_F32 && in_dtype != FM_I16 && in_dtype != FM_F16) return FM_ERR_INVALID_ARG;
  if (out_dtype != FM_F32 && out_dtype != FM_F16) return FM_ERR_INVALID_ARG;
  fm_status st = fm::check_filter_args(sr, n_fft, n_mels, f_min, &f_max, mel_scale, norm);
  if (st != FM_OK) return st;
  if (!fm::is_supported_nfft(n_fft) || n_mels > 256) return FM_ERR_UNSUPPORTED;
  if (fm::find_variant(n_fft, hop) == nullptr) return FM_ERR_UNSUPPORTED;

  // host tables (double precision, rounded to float)
  std::vector<int> ms, ml, mo;
  std::vector<float> mw, win;
  std::vector<float2> twh, twf;
  try {
    fm::build_filterbank(sr, n_fft, n_mels, f_min, f_max, mel_scale == FM_MEL_SLANEY, norm == FM_NORM_SLANEY, ms,
                         ml, mo, mw);
    // the STFT normalisation is folded into the window (README "How it works")
    fm::build_window(n_fft, win_length, normalized, win);
    fm::build_twiddles(n_fft / 2, n_fft / 2, twh);
    fm::build_twiddles(n_fft, n_fft / 2 + 1, twf);
  } catch (const std::bad_alloc&) {
    return FM_ERR_OOM;
  }
  const int nnz = (int)mw.size();

  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess) return FM_ERR_CUDA;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FM_ERR_CUDA;
  const int in_esize = in_dtype == FM_F32 ? 4 : 2;
  // the first kernel for (n_fft, hop) whose tables and shared memory fit
  const fm::Variant* var = nullptr;
  X2Schedule x2s;
  int x2_slots = 0;
  size_t smem_total = 0, dyn_max = 0;
  for (const fm::Variant* v = fm::find_variant(n_fft, hop); v != nullptr && var == nullptr;
       v = fm::find_variant(n_fft, hop, v)) {
    // warps per tile group of the packed kernel (its CTA adds the producer warp)
    const int x2_warps = v->kind == 1 ? (v->threads / 32 - fm::kX2ProducerWarps) / v->groups : 0;
    X2Schedule sched;
    if (v->kind == 1) sched = build_x2_schedule(n_fft / 2, n_mels, x2_warps, ms, ml, mo, mw);
    const int slots = v->kind == 1 ? sched.warp_begin.back() : 0;
    if (v->kind == 1 && (n_fft / 2 > fm::kX2MaxM || slots > fm::kX2MaxSlots || x2_warps > fm::kX2MaxWarps))
      continue;
    const size_t need =
        v->kind == 1   ? fm::smem_layout_x2(n_fft, hop, v->hop > 0 ? 2 : 1, slots, in_esize, v->groups).total
        : v->kind == 2 ? fm::big_layout(n_fft, n_mels, nnz, v->P > 0).st
        : v->kind == 3 ? fm::smem_layout_c2c(hop, n_mels, nnz, in_esize).total
                       : fm::smem_layout(n_fft, hop, n_mels, nnz, v->frames_per_tile, in_esize, v->in_buffers).total;
    // the kernel's static shared memory comes out of the same per-block limit
    cudaFuncAttributes fattr;
    if (cudaFuncGetAttributes(&fattr, v->fn) != cudaSuccess) return FM_ERR_CUDA;
    const size_t avail = prop.sharedMemPerBlockOptin > fattr.sharedSizeBytes
                             ? prop.sharedMemPerBlockOptin - fattr.sharedSizeBytes
                             : 0;
    if (need > avail) continue;
    var = v;
    x2s = std::move(sched);
    x2_slots = slots;
    smem_total = need;
    dyn_max = avail;
  }
  if (var == nullptr) return FM_ERR_UNSUPPORTED;
  // three-pass large-transform kernel: a staging buffer for the next tile's
  // samples, when one tile's span fits beside the transform buffer
  int big_span = 0;
  if (var->kind == 2 && var->P == 0) {
    // one staging buffer per tile group
    const int F = var->frames_per_tile, GB = var->groups > 0 ? var->groups : 1;
    const size_t st_bytes = fm::big_staging_bytes(F, n_fft, hop, in_esize);
    if (fm::big_span(F, n_fft, hop) < (1 << 24) && smem_total + GB * st_bytes <= dyn_max) {
      big_span = (int)fm::big_span(F, n_fft, hop);
      smem_total += GB * st_bytes;
    }
  }
  // allow the device maximum once, so plans of different sizes never undercut each other
  if (cudaFuncSetAttribute(var->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_max) != cudaSuccess)
    return FM_ERR_CUDA;
  int bps = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, var->fn, var->threads, smem_total) != cudaSuccess)
    return FM_ERR_CUDA;
  if (bps <= 0) return FM_ERR_UNSUPPORTED;

  fm_plan* p = new (std::nothrow) fm_plan();
  if (p == nullptr) return FM_ERR_OOM;
  p->x2 = nullptr;
  p->device = dev;
  p->center = center;
  p->pad_mode = pad_mode;
  p->zpad = zpad;
  p->normalized = normalized;
  p->sr = sr;
  p->n_fft = n_fft;
  p->hop = hop;
  p->win_length = win_length;
  p->n_mels = n_mels;
  p->f_min = f_min;
  p->f_max = f_max;
  p->power = power;
  p->mel_scale = mel_scale;
  p->norm = norm;
  p->in_dtype = in_dtype;
  p->out_dtype = out_dtype;
  p->power_mode = power == 2.0 ? 0 : power == 1.0 ? 1 : 2;
  p->var = var;
  p->nnz = nnz;
  p->x2_slots = x2_slots;
  p->big_span = big_span;
  p->mel_taps = var->kind == 2 && var->P > 0 ? (int)choose_mel_taps(ml, var->frames_per_tile) : 0;
  p->smem = smem_total;
  p->blocks_per_sm = bps;
  p->num_sms = prop.multiProcessorCount;
  p->grid_limit = bps * prop.multiProcessorCount;

  // pass-1 table: role p, step q -> window at 2n, 2n+1 (n = p + P q) and the
  // tile offset of sample 2n (rows of hop samples, stride in_row_stride)
  const int M = n_fft / 2;
  const int S = var->kind == 1 ? fm::in_row_stride_x2(hop, in_esize) : fm::in_row_stride(hop);
  const float in_scale = in_dtype == FM_I16 ? 1.0f / 32768.0f : 1.0f;  // exact power of two
  std::vector<float4> p1(M);
  for (int pp = 0; pp < var->P && var->kind < 2; ++pp)  // the other kernels have their own tables
    for (int q = 0; q < var->Q; ++q) {
      const int j = 2 * (pp + var->P * q);
      const int off = (j / hop) * S + (j % hop);
      float4 e;
      e.x = win[j] * in_scale;
      e.y = win[j + 1] * in_scale;
      std::memcpy(&e.z, &off, sizeof(int));
      e.w = 0.0f;
      p1[pp * var->Q + q] = e;
    }
  std::vector<int4> mel(n_mels);
  for (int m = 0; m < n_mels; ++m) mel[m] = make_int4(ms[m], ml[m], mo[m], 0);
  // packed copies for the two-frames-per-thread kernel
  std::vector<float4> twh4(M), twf4(M + 1);
  for (int j = 0; j < M; ++j) twh4[j] = make_float4(twh[j].x, twh[j].x, twh[j].y, twh[j].y);
  for (int j = 0; j <= M; ++j) twf4[j] = make_float4(twf[j].x, twf[j].x, twf[j].y, twf[j].y);

  // one device blob: p1 | tw_half | tw_full | mel | weights | packed-kernel tables | err | window
  size_t o = 0;
  const size_t o_p1 = o;   o = fm::align16(o + sizeof(float4) * M);
  const size_t o_twh = o;  o = fm::align16(o + sizeof(float2) * M);
  const size_t o_twf = o;  o = fm::align16(o + sizeof(float2) * (M + 1));
  const size_t o_mel = o;  o = fm::align16(o + sizeof(int4) * n_mels);
  const size_t o_mw = o;   o = fm::align16(o + sizeof(float) * (nnz > 0 ? nnz : 1));
  const size_t o_x2 = o;   o = fm::align16(o + (var->kind == 1 ? sizeof(fm::X2Tables) : 0));
  const size_t o_err = o;  o = fm::align16(o + sizeof(unsigned) * 4);
  const size_t o_win = o;  o = fm::align16(o + sizeof(float) * (var->kind == 2 ? n_fft : 0));
  const size_t o_c2c = o;  o = fm::align16(o + sizeof(float2) * (var->kind == 3 ? 2 * fm::kC2cN : 0));
  std::vector<unsigned char> blob(o, 0);
  if (var->kind == 1) {
    fm::X2Tables* t = reinterpret_cast<fm::X2Tables*>(blob.data() + o_x2);
    std::memcpy(t->p1, p1.data(), sizeof(float4) * M);
    // pass-1 twiddles by role: [p * Q + k2] = W_M^{p k2}
    for (int pp = 0; pp < var->P; ++pp)
      for (int k2 = 0; k2 < var->Q; ++k2) t->tw_half[pp * var->Q + k2] = twh4[pp * k2];
    std::memcpy(t->tw_full, twf4.data(), sizeof(float4) * (M + 1));
    for (size_t i = 0; i < x2s.warp_begin.size(); ++i) t->warp_begin[i] = x2s.warp_begin[i];
    std::memcpy(t->desc, x2s.desc.data(), sizeof(int2) * x2s.desc.size());
    std::memcpy(t->w4, x2s.w4.data(), sizeof(float4) * x2s.w4.size());
  }
  std::memcpy(blob.data() + o_p1, p1.data(), sizeof(float4) * M);
  std::memcpy(blob.data() + o_twh, twh.data(), sizeof(float2) * M);
  std::memcpy(blob.data() + o_twf, twf.data(), sizeof(float2) * (M + 1));
  std::memcpy(blob.data() + o_mel, mel.data(), sizeof(int4) * n_mels);
  if (nnz > 0) std::memcpy(blob.data() + o_mw, mw.data(), sizeof(float) * nnz);
  if (var->kind == 3) {
    // paired-frame kernel: per (role p, step q) the window at n = p + P q
    // (with the split's 1/2 and the int16 scale) and the tile offset of
    // sample n (rows of hop samples, stride in_row_stride); then W_N^j, j < N
    float2* tab = reinterpret_cast<float2*>(blob.data() + o_c2c);
    for (int pp = 0; pp < fm::kC2cP; ++pp)
      for (int q = 0; q < fm::kC2cQ; ++q) {
        const int n = pp + fm::kC2cP * q;
        const int off = (n / hop) * S + (n % hop);
        tab[pp * fm::kC2cQ + q].x = win[n] * in_scale;
        std::memcpy(&tab[pp * fm::kC2cQ + q].y, &off, sizeof(int));
      }
    std::vector<float2> tw400;
    fm::build_twiddles(fm::kC2cN, fm::kC2cN, tw400);
    std::memcpy(tab + fm::kC2cN, tw400.data(), sizeof(float2) * fm::kC2cN);
  }
  if (var->kind == 2) {  // the window with the int16 scale, for the large-transform kernel
    float* wd = reinterpret_cast<float*>(blob.data() + o_win);
    for (int j = 0; j < n_fft; ++j) wd[j] = win[j] * in_scale;
  }

  cudaError_t e = cudaMalloc(&p->dmem, o);
  if (e != cudaSuccess) {
    delete p;
    return from_cuda(e);
  }
  e = cudaMemcpy(p->dmem, blob.data(), o, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = create_pipe(p->pipe);
  if (e != cudaSuccess) {
    cudaFree(p->dmem);
    delete p;
    return from_cuda(e);
  }
  unsigned char* base = static_cast<unsigned char*>(p->dmem);
  p->p1 = reinterpret_cast<float4*>(base + o_p1);
  p->tw_half = reinterpret_cast<float2*>(base + o_twh);
  p->tw_full = reinterpret_cast<float2*>(base + o_twf);
  p->mel = reinterpret_cast<int4*>(base + o_mel);
  p->mel_w = reinterpret_cast<float*>(base + o_mw);
  p->err = reinterpret_cast<unsigned*>(base + o_err);
  p->win = reinterpret_cast<float*>(base + o_win);
  p->x2 = var->kind == 1 ? reinterpret_cast<fm::X2Tables*>(base + o_x2) : nullptr;
  p->c2c = reinterpret_cast<float2*>(base + o_c2c);
  *out = p;
  return FM_OK;
}

extern "C" fm_status fm_plan_destroy(fm_plan* plan) {
  if (plan == nullptr) return FM_OK;
  cudaError_t e = cudaSuccess;
  destroy_pipe(plan->pipe);
  if (plan->dmem) e = cudaFree(plan->dmem);
  delete plan;
  return e == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

// Frames for T samples under the plan's framing, or -1 if T is too short for
// it: with T' = T + 2 pad, centred reflect needs T' > n_fft/2 (a mirror cannot
// reach further), centred circular T' >= n_fft/2, centred constant and
// replicate T >= 1, uncentred T' >= n_fft.
static int64_t frames_for(const fm_plan* plan, int64_t T) {
  if (plan == nullptr || T < 1 || T > ((int64_t)1 << 61)) return -1;
  const int64_t Tp = T + 2 * (int64_t)plan->zpad, c = plan->n_fft / 2;
  if (!plan->center) return Tp >= plan->n_fft ? 1 + (Tp - plan->n_fft) / plan->hop : -1;
  if (plan->pad_mode == FM_PAD_REFLECT && Tp <= c) return -1;
  if (plan->pad_mode == FM_PAD_CIRCULAR && Tp < c) return -1;
  return 1 + Tp / plan->hop;
}

extern "C" int64_t fm_n_frames(const fm_plan* plan, int64_t T) { return frames_for(plan, T); }

static fm_status check_forward(const fm_plan* plan, const void* in, int64_t B, int64_t T, const void* out) {
  if (plan == nullptr || B < 0) return FM_ERR_INVALID_ARG;
  if (B == 0) return FM_OK;
  if (in == nullptr || out == nullptr) return FM_ERR_INVALID_ARG;
  const int64_t nf = frames_for(plan, T);
  if (nf < 1 || nf > INT_MAX) return FM_ERR_INVALID_ARG;
  const int64_t lim = (int64_t)1 << 62;
  if (T > lim / B) return FM_ERR_INVALID_ARG;
  if (nf * plan->n_mels > lim / B) return FM_ERR_INVALID_ARG;
  return FM_OK;
}

extern "C" fm_status fm_mel_forward(const fm_plan* plan, const void* d_in, int64_t B, int64_t T, void* d_out,
                                    fm_stream_t stream) {
  fm_status st = check_forward(plan, d_in, B, T, d_out);
  if (st != FM_OK || B == 0) return st;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->device) return FM_ERR_CUDA;

  const fm::Variant* v = plan->var;
  fm::KernelParams prm;
  prm.in = d_in;
  prm.out = d_out;
  prm.B = B;
  prm.T = T;
  prm.n_frames = (int)frames_for(plan, T);
  prm.hop = plan->hop;
  prm.cpad = plan->center ? plan->n_fft / 2 : 0;
  prm.zpad = plan->zpad;
  prm.lead = prm.cpad + prm.zpad;
  prm.pad_mode = plan->pad_mode;
  prm.in_dtype = plan->in_dtype;
  prm.out_dtype = plan->out_dtype;
  prm.n_mels = plan->n_mels;
  prm.nnz = plan->nnz;
  prm.x2_slots = plan->x2_slots;
  prm.power_mode = plan->power_mode;
  prm.power = (float)plan->power;
  prm.tiles_per_signal = (prm.n_frames + v->frames_per_tile - 1) / v->frames_per_tile;
  prm.total_tiles = (long long)B * prm.tiles_per_signal;
  prm.p1 = plan->p1;
  prm.tw_half = plan->tw_half;
  prm.tw_full = plan->tw_full;
  prm.mel = plan->mel;
  prm.mel_w = plan->mel_w;
  prm.err = plan->err;
  prm.win = plan->win;
  prm.big_span = plan->big_span;
  prm.mel_taps = plan->mel_taps;
  prm.c2c_tab = plan->c2c;
  prm.c2c_tw = plan->c2c + fm::kC2cN;

  const long long grid = prm.total_tiles < plan->grid_limit ? prm.total_tiles : plan->grid_limit;
  prm.x2 = plan->x2;
  // two-frames-per-thread kernel: move the signals' first and last tiles (the
  // slow ones to stage) into the last group's first slots, when there are at
  // most as many as CTAs and every slot they take holds an interior tile
  prm.perm_edges = 0;
  prm.perm_t0 = 0;
  if (v->kind == 1) {
    const long long tps = prm.tiles_per_signal, n_edge = 2 * B, t0 = (long long)(v->groups - 1) * grid;
    if (tps >= 3 && n_edge <= grid && t0 + n_edge <= prm.total_tiles) {
      bool ok = true;
      for (long long i = 0; i < n_edge && ok; ++i) {
        const long long tt = (t0 + i) % tps;
        ok = tt != 0 && tt != tps - 1;
      }
      if (ok) {
        prm.perm_edges = (int)n_edge;
        prm.perm_t0 = t0;
      }
    }
  }
  encode_input_map(plan, d_in, B, T, prm);
  void* args[] = {&prm};
  // programmatic dependent launch: the kernel waits (griddepcontrol.wait) for
  // the previous kernel in the stream before it reads d_in or writes d_out, so
  // only set-up overlaps; a predecessor that did not opt in is waited for in full
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(v->threads);
  cfg.dynamicSmemBytes = plan->smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelExC(&cfg, v->fn, args);
  return e == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

extern "C" fm_status fm_mel_forward_host(const fm_plan* plan, const void* h_in, int64_t B, int64_t T,
                                         void* h_out, void* d_in_scratch, void* d_out_scratch,
                                         fm_stream_t stream) {
  fm_status st = check_forward(plan, h_in, B, T, h_out);
  if (st != FM_OK || B == 0) return st;
  if (d_in_scratch == nullptr || d_out_scratch == nullptr) return FM_ERR_INVALID_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->device) return FM_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t in_row = (size_t)T * dtype_size(plan->in_dtype);
  const size_t out_row = (size_t)plan->n_mels * (size_t)frames_for(plan, T) * dtype_size(plan->out_dtype);
  const unsigned char* hin = static_cast<const unsigned char*>(h_in);
  unsigned char* hout = static_cast<unsigned char*>(h_out);
  unsigned char* din = static_cast<unsigned char*>(d_in_scratch);
  unsigned char* dout = static_cast<unsigned char*>(d_out_scratch);
  // Signals in up to kHostChunks chunks of at least kHostChunkMinBytes:
  // copy in (pipe.in), kernel (pipe.comp), copy out (pipe.out), chained by
  // events, so one chunk's upload, another's kernel and a third's download
  // overlap; the three streams start after the work already queued on
  // `stream`, which then waits for the last download. A call that makes one
  // chunk runs on `stream` itself.
  const int64_t C = std::min<int64_t>(
      std::min<int64_t>(B, kHostChunks),
      std::max<int64_t>(1, (int64_t)((size_t)B * (in_row + out_row) / kHostChunkMinBytes)));
  if (C == 1) {
    if (cudaMemcpyAsync(din, hin, (size_t)B * in_row, cudaMemcpyHostToDevice, s) != cudaSuccess) return FM_ERR_CUDA;
    st = fm_mel_forward(plan, din, B, T, dout, stream);
    if (st != FM_OK) return st;
    if (cudaMemcpyAsync(hout, dout, (size_t)B * out_row, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return FM_ERR_CUDA;
    return FM_OK;
  }
  HostPipe& P = plan->pipe;
  std::lock_guard<std::mutex> lock(P.mu);
  if (cudaEventRecord(P.start, s) != cudaSuccess) return FM_ERR_CUDA;
  cudaError_t e = cudaStreamWaitEvent(P.in, P.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(P.comp, P.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.start, 0);
  for (int c = 0; c < C && e == cudaSuccess && st == FM_OK; ++c) {
    const int64_t b0 = B * c / C, nb = B * (c + 1) / C - b0;
    e = cudaMemcpyAsync(din + b0 * in_row, hin + b0 * in_row, nb * in_row, cudaMemcpyHostToDevice, P.in);
    if (e == cudaSuccess) e = cudaEventRecord(P.in_done[c], P.in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.comp, P.in_done[c], 0);
    if (e != cudaSuccess) break;
    st = fm_mel_forward(plan, din + b0 * in_row, nb, T, dout + b0 * out_row, reinterpret_cast<fm_stream_t>(P.comp));
    if (st != FM_OK) break;
    e = cudaEventRecord(P.comp_done[c], P.comp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.comp_done[c], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(hout + b0 * out_row, dout + b0 * out_row, nb * out_row, cudaMemcpyDeviceToHost, P.out);
  }
  // join even after a failure, so that `stream` never runs ahead of queued
  // work; after one, an upload or kernel may be queued that no download
  // follows, so the download stream first waits for the other two
  cudaError_t j = cudaSuccess;
  if (e != cudaSuccess || st != FM_OK) {
    j = cudaEventRecord(P.in_done[0], P.in);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(P.out, P.in_done[0], 0);
    if (j == cudaSuccess) j = cudaEventRecord(P.comp_done[0], P.comp);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(P.out, P.comp_done[0], 0);
  }
  if (j == cudaSuccess) j = cudaEventRecord(P.end, P.out);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(s, P.end, 0);
  if (st != FM_OK) return st;
  return (e == cudaSuccess && j == cudaSuccess) ? FM_OK : FM_ERR_CUDA;
}

extern "C" fm_status fm_plan_get_info(const fm_plan* plan, fm_plan_info* info) {
  if (plan == nullptr || info == nullptr) return FM_ERR_INVALID_ARG;
  info->n_fft = plan->n_fft;
  info->hop = plan->hop;
  info->win_length = plan->win_length;
  info->n_mels = plan->n_mels;
  info->n_freqs = plan->n_fft / 2 + 1;
  info->in_dtype = plan->in_dtype;
  info->out_dtype = plan->out_dtype;
  info->nnz = plan->nnz;
  info->frames_per_tile = plan->var->frames_per_tile;
  info->threads_per_block = plan->var->threads;
  info->blocks_per_sm = plan->blocks_per_sm;
  info->grid_limit = plan->grid_limit;
  info->smem_bytes = (int)plan->smem;
  info->device = plan->device;
  info->center = plan->center;
  info->pad_mode = plan->pad_mode;
  info->pad = plan->zpad;
  info->normalized = plan->normalized;
  return FM_OK;
}

unsigned* fm::plan_error_word(const fm_plan* plan) { return plan ? plan->err : nullptr; }

// err[0] is the error word the kernels write; err[1] receives its value when
// fm_plan_poll_error takes and clears it in one atomic exchange.
__global__ void take_error_word(unsigned* err) { err[1] = atomicExch(err, 0u); }

extern "C" fm_status fm_plan_poll_error(const fm_plan* plan) {
  if (plan == nullptr) return FM_ERR_INVALID_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->device) return FM_ERR_CUDA;
  take_error_word<<<1, 1>>>(plan->err);
  if (cudaGetLastError() != cudaSuccess) return FM_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, plan->err + 1, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return FM_ERR_CUDA;
  if (word == 0) return FM_OK;
  return word <= FM_ERR_BOUNDS ? (fm_status)word : FM_ERR_KERNEL_TIMEOUT;
}

extern "C" const char* fm_status_string(fm_status status) {
  switch (status) {
    case FM_OK: return "FM_OK";
    case FM_ERR_INVALID_ARG: return "FM_ERR_INVALID_ARG";
    case FM_ERR_UNSUPPORTED: return "FM_ERR_UNSUPPORTED";
    case FM_ERR_CUDA: return "FM_ERR_CUDA";
    case FM_ERR_OOM: return "FM_ERR_OOM";
    case FM_ERR_KERNEL_TIMEOUT: return "FM_ERR_KERNEL_TIMEOUT";
    case FM_ERR_BOUNDS: return "FM_ERR_BOUNDS";
  }
  return "FM_ERR_UNKNOWN";
}
