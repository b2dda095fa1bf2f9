/*
 * fm_mel.h -- C ABI of the GB300 (sm_103a) batched mel spectrogram.
 *
 * The operation is torchaudio's MelSpectrogram as the flashmel 0.1.0 page
 * states it (README, "Usage" and "How it works"; filters.py, make_window and
 * pack_fbank):
 *
 *   out[b, m, t] = sum_k F[m, k] * |X_{b,t}[k]|^power
 *   X_{b,t}[k]   = sum_{n < n_fft} xp_b[t*hop + n] * w[n] * exp(-2 pi i k n / n_fft)
 *
 * with xp_b the signal padded for framing (by default reflect-padded by
 * n_fft/2 on both sides, torchaudio's center=True, pad_mode="reflect";
 * fm_plan_create_ex selects the other torchaudio framings), w the periodic
 * Hann window of win_length samples zero-padded and centred to n_fft (scaled
 * by the chosen STFT normalisation), k = 0 .. n_fft/2, t over the frames, and F
 * the triangular mel filterbank (HTK or Slaney mel scale, optional Slaney
 * area norm) over bins at frequency k*sr/n_fft.
 *
 * Conventions for every call:
 *   - Errors are returned as fm_status; nothing is thrown or printed, and a
 *     failing call has no side effects.
 *   - "device pointer" means memory the current CUDA device can address
 *     (cudaMalloc / torch CUDA tensors); "host pointer" means CPU memory.
 *   - All arrays are dense and row-major.
 *
 * This header needs no CUDA header: fm_stream_t is ABI-identical to
 * cudaStream_t / CUstream (a pointer to the opaque CUstream_st); pass NULL
 * for the legacy default stream.
 */
#ifndef FM_MEL_H
#define FM_MEL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fm_stream_t;
typedef struct fm_plan fm_plan; /* opaque; owns its device tables */

typedef enum {
  FM_OK = 0,
  FM_ERR_INVALID_ARG = 1,    /* a NULL pointer, a size or a parameter out of range */
  FM_ERR_UNSUPPORTED = 2,    /* valid for torchaudio, but not built here (see fm_plan_create) */
  FM_ERR_CUDA = 3,           /* a CUDA runtime call failed (no device, launch failure, ...) */
  FM_ERR_OOM = 4,            /* device or host allocation failed */
  FM_ERR_KERNEL_TIMEOUT = 5, /* a bounded device-side wait gave up (reported by fm_plan_poll_error) */
  FM_ERR_BOUNDS = 6          /* debug build only (libfm_mel_check.so, -DFM_BOUNDS_CHECK): an index check
                                found an access outside its buffer and skipped it (fm_plan_poll_error) */
} fm_status;

typedef enum { FM_MEL_HTK = 0, FM_MEL_SLANEY = 1 } fm_mel_scale;
typedef enum { FM_NORM_NONE = 0, FM_NORM_SLANEY = 1 } fm_norm;
typedef enum { FM_F32 = 0, FM_I16 = 1, FM_F16 = 2 } fm_dtype;
/* torch's pad modes for the centre padding: mirror without repeating the
 * edge sample, zeros, repeat the edge sample, wrap around the signal */
typedef enum { FM_PAD_REFLECT = 0, FM_PAD_CONSTANT = 1, FM_PAD_REPLICATE = 2, FM_PAD_CIRCULAR = 3 } fm_pad_mode;
/* STFT normalisation, folded into the window (flashmel filters.py
 * make_window): none, divide by sqrt(sum w^2) (normalized=True / "window"),
 * or by sqrt(win_length) ("frame_length"; torch.stft's sqrt(n_fft) when
 * win_length = n_fft) */
typedef enum { FM_NORMALIZED_NONE = 0, FM_NORMALIZED_WINDOW = 1, FM_NORMALIZED_FRAME_LENGTH = 2 } fm_normalized;

/*
 * fm_plan_create -- validate the transform parameters and build its tables.
 *
 * flashmel README "Usage" (torchaudio arguments, input dtype f32 or int16
 * PCM scaled by 1/32768, output dtype f32 or f16) and "How it works" (window
 * and sparse filterbank built once on the host); filters.py make_window /
 * pack_fbank. f16 input (computed in fp32) is this library's addition.
 *
 *   out        : receives the new plan (host pointer to a pointer). Set to
 *                NULL on failure.
 *   sr         : sample rate in Hz, > 0.
 *   n_fft      : DFT size. Supported: 400 and the powers of two 64 .. 16384
 *                (README "Usage": "400 or a power of 2 in [64, 16384]").
 *   hop        : frame advance in samples, > 0 (odd hops run a kernel that
 *                stages each tile as one contiguous run of samples; the plan
 *                takes the first kernel for its n_fft and hop whose staged
 *                tiles fit shared memory, so long hops run builds with fewer
 *                tiles in flight per CTA).
 *   win_length : Hann length, 1 .. n_fft; 0 means n_fft.
 *   n_mels     : number of mel filters, 1 .. 256.
 *   f_min      : lowest filter edge in Hz, >= 0.
 *   f_max      : highest filter edge in Hz, f_min < f_max <= sr/2;
 *                f_max <= 0 means sr/2.
 *   power      : exponent on |X|, finite and > 0 (2 = power, 1 = magnitude).
 *   mel_scale  : FM_MEL_HTK or FM_MEL_SLANEY.
 *   norm       : FM_NORM_NONE or FM_NORM_SLANEY (filter m scaled by
 *                2 / (f[m+2] - f[m]), i.e. unit area).
 *   in_dtype   : storage type of the input samples (FM_F32, FM_I16, FM_F16).
 *   out_dtype  : FM_F32 or FM_F16 (round-to-nearest-even at the store;
 *                accumulation is always fp32).
 *
 * Builds the window, the DFT twiddles and the per-filter CSR (start, length,
 * offset, weights) in float64 on the host, rounds them to fp32 and copies them
 * to memory on the current CUDA device, which the plan owns until
 * fm_plan_destroy. The plan is read-only afterwards: it may be used from
 * several host threads and streams at once, on the device it was created on.
 *
 * Errors: FM_ERR_INVALID_ARG (out NULL or a parameter out of range, including
 * out_dtype == FM_I16); FM_ERR_UNSUPPORTED (n_fft not in the supported set,
 * n_mels > 256, or a hop whose staged tile does not fit shared memory);
 * FM_ERR_CUDA (no usable device); FM_ERR_OOM.
 */
fm_status fm_plan_create(fm_plan** out, int sr, int n_fft, int hop, int win_length, int n_mels,
                         double f_min, double f_max, double power, fm_mel_scale mel_scale,
                         fm_norm norm, fm_dtype in_dtype, fm_dtype out_dtype);

/*
 * fm_plan_create_ex -- fm_plan_create with the framing options too.
 *
 * flashmel README "Usage": every torchaudio.transforms.MelSpectrogram
 * argument except window_fn / wkwargs, including pad, center, pad_mode and
 * normalized; "How it works": the padding (pad, center, all four pad modes)
 * is applied as index arithmetic and the normalized modes are folded into
 * the window on the host.
 *
 * The first twelve fields mean what fm_plan_create's arguments of the same
 * names mean. Then:
 *   center     : nonzero pads n_fft/2 samples on both sides by pad_mode
 *                before framing (frames = 1 + floor(T' / hop)); zero frames
 *                the signal as it is (frames = 1 + floor((T' - n_fft) / hop)),
 *                with T' = T + 2 * pad.
 *   pad_mode   : fm_pad_mode of the centre padding (ignored without center).
 *   pad        : zeros added on both sides of every signal before the centre
 *                padding (torchaudio's `pad`), 0 .. 2^20.
 *   normalized : fm_normalized.
 * fm_plan_create(...) is fm_plan_create_ex with center = 1, FM_PAD_REFLECT,
 * pad = 0 and FM_NORMALIZED_NONE. `params` is read during the call only.
 * Errors: as fm_plan_create, plus FM_ERR_INVALID_ARG for NULL params or an
 * option out of range.
 */
typedef struct {
  int sr, n_fft, hop, win_length, n_mels;
  double f_min, f_max, power;
  fm_mel_scale mel_scale;
  fm_norm norm;
  fm_dtype in_dtype, out_dtype;
  int center;
  fm_pad_mode pad_mode;
  int pad;
  fm_normalized normalized;
} fm_plan_params;

fm_status fm_plan_create_ex(fm_plan** out, const fm_plan_params* params);

/* fm_plan_destroy -- free the plan's device tables. NULL is accepted (no-op).
 * The pages have no counterpart (flashmel keeps its per-configuration
 * modules and filter buffers in process-wide caches, README "How it works");
 * here the plan owns them and this call releases them.
 * Work already queued with the plan must have finished (e.g. synchronise the
 * streams first). Returns FM_OK, or FM_ERR_CUDA if freeing failed. */
fm_status fm_plan_destroy(fm_plan* plan);

/* fm_n_frames -- frames per signal for T samples: with T' = T + 2 * pad,
 * 1 + floor(T' / hop) when centred, 1 + floor((T' - n_fft) / hop) when not.
 * flashmel README "Usage": the output is (..., n_mels, n_frames) like
 * torchaudio's, e.g. 480000 samples at hop 160, centred, give 3001 frames.
 * Returns -1 if plan is NULL or T is too short for the plan's framing (see
 * fm_mel_forward). */
int64_t fm_n_frames(const fm_plan* plan, int64_t T);

/*
 * fm_mel_forward -- the whole path in one kernel launch, asynchronously on
 * `stream` (README "How it works": pad, frame, window, R2C DFT, |X|^power and
 * the sparse mel projection fused; launched on the caller's stream).
 *
 *   d_in   : device pointer, [B][T] samples of the plan's in_dtype,
 *            contiguous, any alignment of the element type. Not modified.
 *   B      : number of signals, >= 0. B == 0 returns FM_OK and does nothing
 *            (d_in / d_out may then be NULL).
 *   T      : samples per signal, >= 1. With T' = T + 2 * pad: centred
 *            reflect padding needs T' > n_fft/2 and circular T' >= n_fft/2
 *            (a mirror or a wrap cannot reach further); without centring
 *            T' >= n_fft (one whole frame).
 *   d_out  : device pointer, [B][n_mels][fm_n_frames(T)] of the plan's
 *            out_dtype, contiguous, element-aligned; fully overwritten. Must
 *            not overlap d_in.
 *   stream : the CUDA stream to run on (NULL = legacy default stream).
 *
 * Allocates nothing and does not synchronise. Both buffers are owned by the
 * caller and must stay valid until the stream reaches this work.
 * Errors: FM_ERR_INVALID_ARG (NULL plan or pointer with B > 0, B < 0,
 * T too short for the framing, B*T or the output size beyond 2^62
 * elements); FM_ERR_CUDA
 * (launch failed, or called on another device than the plan's).
 */
fm_status fm_mel_forward(const fm_plan* plan, const void* d_in, int64_t B, int64_t T, void* d_out,
                         fm_stream_t stream);

/*
 * fm_mel_forward_host -- fm_mel_forward for inputs and outputs in host memory.
 *
 * Copies h_in [B][T] into d_in_scratch, runs the kernel and copies
 * d_out_scratch into h_out [B][n_mels][n_frames]. The caller supplies both
 * device buffers (at least B*T and B*n_mels*n_frames elements) so the call
 * allocates nothing; pinned host memory makes the copies asynchronous.
 * Ordering: the work starts after everything already queued on `stream`,
 * and `stream` waits for all of it, so the caller synchronises `stream`
 * before reading h_out. Inside, the signals go in up to four chunks of at
 * least 2 MiB (input plus output bytes) through three streams that the plan
 * owns (upload, kernel, download), so one chunk's upload overlaps another's
 * kernel and a third's download; a call too small for two chunks runs on
 * `stream` alone. Calls on one plan from several host threads are
 * serialised while they queue work. Calls that share scratch buffers must
 * be ordered by the caller, as for fm_mel_forward.
 * The current device must be the plan's device (else FM_ERR_CUDA).
 * Errors: as fm_mel_forward, plus FM_ERR_INVALID_ARG for NULL buffers.
 */
fm_status fm_mel_forward_host(const fm_plan* plan, const void* h_in, int64_t B, int64_t T,
                              void* h_out, void* d_in_scratch, void* d_out_scratch,
                              fm_stream_t stream);

/* Size in bytes of the device staging array behind
 * fm_mel_forward_host_noalloc (32 MiB). */
#define FM_NOALLOC_MAX_BYTES ((size_t)32 << 20)

/*
 * fm_mel_forward_host_noalloc -- fm_mel_forward_host without caller-supplied
 * device buffers. The pages have no counterpart: this entry point is for
 * callers that hold audio in host memory but cannot allocate device memory
 * when they need a spectrogram -- a real-time audio callback, where
 * cudaMalloc's implicit device synchronisation and unbounded latency would
 * miss the deadline, or a process whose device memory is owned by another
 * framework's allocator.
 *
 * Queues on `stream`: a copy of h_in [B][T] (plan's in_dtype) into a staging
 * array in device memory, the kernel, and a copy of the spectrogram into
 * h_out [B][n_mels][n_frames] (plan's out_dtype). The staging array is a
 * static device array of FM_NOALLOC_MAX_BYTES that every GPU loading this
 * library holds until the process exits; the call allocates nothing.
 *
 * Limit: the input bytes, rounded up to 256, plus the output bytes must fit
 * in FM_NOALLOC_MAX_BYTES (the B = 8 x 480000 f32 speech batch with 128 mels,
 * 27.7 MB, does); larger calls return FM_ERR_INVALID_ARG before any CUDA work.
 * Sharing: every call on a device uses the same array and the array keeps the
 * last call's contents. Calls queued on one stream run in order and are safe;
 * calls that overlap on the GPU (other streams, other host threads, or two
 * plans on one device) race on the array and must be serialised by the caller.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, which may make the CUDA runtime load this library's
 * module on that device); make that first call before any stream capture.
 * The address is looked up again when the current context of the device is
 * not the one it was looked up in (after cudaDeviceReset, or under a context
 * the caller made current), so that call too belongs outside a capture.
 * The caller synchronises `stream` before reading h_out; pinned host memory
 * makes the copies asynchronous.
 * Errors: as fm_mel_forward_host, plus FM_ERR_INVALID_ARG for sizes beyond
 * the limit and FM_ERR_CUDA if the address look-up fails.
 */
fm_status fm_mel_forward_host_noalloc(const fm_plan* plan, const void* h_in, int64_t B, int64_t T,
                                      void* h_out, fm_stream_t stream);

/*
 * fm_selftest_wait_timeout -- diagnostic: runs out, on purpose, one of the
 * bounded waits of the kernels, so that the timeout path can be exercised
 * without faulting or hanging the GPU. The pages have no counterpart
 * (flashmel's kernels have no device-side waits).
 *
 * One CTA of two groups of 64 threads; each group waits, with the kernels'
 * own wait code and exit vote, on its own mbarrier for 2^log2_polls polls.
 * Group 1's barrier completes by an arrival; nothing arrives on group 0's, so
 * group 0 gives up, records FM_ERR_KERNEL_TIMEOUT in the plan's error word
 * (read it with fm_plan_poll_error, as after a real kernel) and leaves, while
 * group 1 finishes normally. The call synchronises `stream`.
 *   kind            : 0 = a tile group's wait for its staged tile (blocking
 *                     mbarrier.try_wait polls); 1 = the producer warp's wait
 *                     for a free staging area (non-blocking test_wait polls
 *                     with a short sleep between them).
 *   log2_polls      : 0 .. the kernels' own limit for that wait.
 *   groups_completed: host int, may be NULL; receives the number of groups
 *                     that passed their wait (1 when the path works).
 *   elapsed_us      : host double, may be NULL; the kernel's duration by CUDA
 *                     events, from which the time per poll follows.
 * Calls are serialised within the process; the plan must be on the current
 * device. Errors: FM_ERR_INVALID_ARG for a NULL plan, another kind or
 * log2_polls out of range; FM_ERR_CUDA if a CUDA call fails.
 */
fm_status fm_selftest_wait_timeout(const fm_plan* plan, int kind, int log2_polls, fm_stream_t stream,
                                   int* groups_completed, double* elapsed_us);

/*
 * fm_mel_filterbank_csr -- the plan's filterbank, computed on the host only
 * (no CUDA call), for inspection and tests.
 *
 * filters.py pack_fbank: a triangular filter has contiguous support, so row
 * m is stored as start[m], len[m] and len[m] weights beginning at off[m] in
 * `weights` (off[m+1] = off[m] + len[m]). An empty filter has len 0.
 *
 *   start, len : host int32 arrays of n_mels entries (may be NULL to query).
 *   off        : host int32 array of n_mels + 1 entries (may be NULL).
 *   weights    : host float array with room for *nnz floats (may be NULL).
 *   nnz        : in: capacity of `weights`; out: entries needed. Required.
 * Returns FM_ERR_INVALID_ARG for bad parameters (same rules as
 * fm_plan_create) or if weights is non-NULL and its capacity is too small.
 */
fm_status fm_mel_filterbank_csr(int sr, int n_fft, int n_mels, double f_min, double f_max,
                                fm_mel_scale mel_scale, fm_norm norm, int32_t* start, int32_t* len,
                                int32_t* off, float* weights, int64_t* nnz);

/* Facts about a plan, for sizing buffers and computing roofline figures. */
typedef struct {
  int n_fft, hop, win_length, n_mels, n_freqs;
  int in_dtype, out_dtype;
  int64_t nnz;            /* filterbank non-zeros */
  int frames_per_tile;    /* frames one CTA processes per tile */
  int threads_per_block;  /* CTA size of the kernel */
  int blocks_per_sm;      /* resident CTAs per SM (occupancy) */
  int grid_limit;         /* persistent grid size = SMs x blocks_per_sm */
  int smem_bytes;         /* dynamic shared memory per CTA */
  int device;             /* CUDA device the plan lives on */
  int center, pad_mode, pad, normalized;  /* the framing options (fm_plan_create_ex) */
} fm_plan_info;

/* fm_plan_get_info -- fill *info. FM_ERR_INVALID_ARG on NULL arguments. */
fm_status fm_plan_get_info(const fm_plan* plan, fm_plan_info* info);

/*
 * fm_plan_poll_error -- read and clear the plan's device error word. The
 * pages have no counterpart (flashmel's kernels wait on nothing that can be
 * lost); this is the report channel of the bounded waits below.
 * Kernels that wait on a device-side
 * barrier give up after a bounded number of polls, about a second on GB300
 * (a tile group's wait for its staged tile: 2^18 mbarrier.try_wait polls of
 * about 3.8 us; the producer warp's wait for a free staging area: 2^22
 * test_wait polls of about 0.1 us). They then record FM_ERR_KERNEL_TIMEOUT
 * there and return instead of hanging. The word is read and cleared in one
 * atomic exchange on the device (a one-thread kernel on the legacy default
 * stream), then copied back, so a code that a kernel still running records
 * in between is kept for the next poll rather than lost. The result covers
 * the kernels that have finished: call it after synchronising every stream
 * that used the plan to see all of them. Returns FM_OK if nothing was
 * recorded, FM_ERR_CUDA if the exchange or the copy failed.
 */
fm_status fm_plan_poll_error(const fm_plan* plan);

/* fm_status_string -- a static, human-readable name for a status code
 * ("FM_OK", "FM_ERR_INVALID_ARG", ...; "FM_ERR_UNKNOWN" for any other value).
 * The pages have no counterpart: flashmel raises Python exceptions, and
 * errors cross this C ABI as status codes instead. */
const char* fm_status_string(fm_status status);

#ifdef __cplusplus
}
#endif

#endif /* FM_MEL_H */
