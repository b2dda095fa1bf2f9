// Fused mel-spectrogram kernel for sm_103a.
//
// One launch runs the whole path of the flashmel README ("How it works"):
// centre reflect padding and framing as index arithmetic, the periodic Hann
// window, the n_fft-point real DFT, |X|^power and the sparse triangular mel
// projection, with coalesced stores of [B][n_mels][n_frames].
//
// Work split. A tile is G consecutive frames of one signal. A persistent grid
// of CTAs walks the tiles round-robin. Thread (role, g), g = tid % G, owns
// frame g of the tile and plays `role` = tid / G in each phase, so every
// role-dependent constant (window slice, twiddles, filter row) is the same for
// the G lanes that share it and is read as a shared-memory broadcast.
//
// Staging. Each tile's samples (G frames plus the (n_fft - hop) overlap) are
// copied raw into shared memory as rows of `hop` samples with cp.async (8- or
// 4-byte pieces), double-buffered so the next tile lands while this one
// computes. Tiles that touch a signal edge (reflect padding) or whose source
// is not 2-sample aligned are gathered with plain loads instead.
//
// The real n_fft-point DFT of frame y is the complex M = n_fft/2 point DFT of
// z[n] = (y[2n] + i y[2n+1]) / 2, split four-step as M = P * Q:
//   pass 1 : role p takes z[p + P q], q < Q, does a Q-point DFT in registers
//            and multiplies output k2 by W_M^{p k2};
//   pass 2 : role t does P-point DFTs over p for its k2 values, which gives
//            Z[k2 + Q k1];
//   split  : X[k] = S + U and X[M-k] = conj(S - U) with S = Z[k] + conj Z[M-k]
//            and U = -i W_N^k (Z[k] - conj Z[M-k]) (the 1/2 sits in the window).
// When Q = 2P, role t holds k2 = t and Q - t, so both members of every pair
// (k, M - k) are in its registers and the split needs no exchange.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fm_fft.cuh"
#include "fm_internal.h"

namespace fm {

// ---------------------------------------------------------------------------
// asynchronous global -> shared copies (Ampere-style cp.async, L1-allocating)
// ---------------------------------------------------------------------------
template <int BYTES>
__device__ __forceinline__ void cp_async(void* smem_dst, const void* gsrc) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n" ::"r"(d), "l"(gsrc), "n"(BYTES) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// Make mbarrier `bar` track this thread's cp.async copies issued so far: its
// pending count goes up by one now and comes down (an arrival) once they have
// landed, so a waiter on the phase sees the copied bytes without the issuing
// thread blocking on them.
__device__ __forceinline__ void cp_async_mbar_arrive(unsigned long long* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];\n" ::"r"((unsigned)__cvta_generic_to_shared(bar))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// ---------------------------------------------------------------------------
// TMA bulk copies (cp.async.bulk) completing on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned smem_addr(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// order earlier generic-proxy accesses of shared memory before later async-proxy (TMA) writes
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// global -> shared bulk copy of `bytes` (multiple of 16, both ends 16-byte aligned)
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, unsigned bytes, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// one box of a 3-D tensor map (coordinates x, y, z) into shared memory
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];\n" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// add `bytes` to the transaction count of the current phase (no arrival)
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// plain arrival (count 1, no transaction bytes) with release semantics
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}
// non-blocking test of phase `parity`
__device__ __forceinline__ bool mbar_test_wait(unsigned long long* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for phase `parity` of an mbarrier: gives up after `polls`
// try_wait polls, records FM_ERR_KERNEL_TIMEOUT in *err and returns false, so
// a lost transfer never hangs the GPU.
__device__ __forceinline__ bool mbar_wait_polls(unsigned long long* bar, unsigned parity, unsigned* err, int polls) {
  for (int i = 0; i < polls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  if (err) atomicExch(err, (unsigned)FM_ERR_KERNEL_TIMEOUT);
  return false;
}
// The kernels' wait for a staged tile: 2^18 try_wait polls. A poll that finds
// the phase incomplete suspends the thread for about 3.8 us on GB300
// (measured), so the wait gives up after about a second, some 10^4 times
// longer than any staged copy takes.
constexpr int kWaitLog2Polls = 18;
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* bar, unsigned parity, unsigned* err) {
  return mbar_wait_polls(bar, parity, err, 1 << kWaitLog2Polls);
}
// Back-off of a polling loop built on non-blocking tests (the producer warp's
// wait for a free staging area): sleeps briefly and returns true while the
// loop has been idle for at most `polls` rounds, false once it should give up.
// 2^22 rounds of about 100 ns (measured on GB300) give up after ~0.4 s.
constexpr int kIdleLog2Polls = 22;
__device__ __forceinline__ bool idle_backoff(int& idle, int polls) {
  if (++idle > polls) return false;
  __nanosleep(32);
  return true;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// CTAs (as SM slots free up) and do its own set-up while this one runs; and,
// before touching any caller buffer, wait until the previous kernel in the
// stream has completed and its memory is visible. Both are no-ops when the
// launch did not opt in.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// a pair of consecutive samples (2n, 2n+1) from the staged tile, as floats
__device__ __forceinline__ float2 load_pair(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 load_pair(const short* p) {
  const int w = *reinterpret_cast<const int*>(p);
  return make_float2((float)(short)(w & 0xffff), (float)(w >> 16));  // int16 scale is in the window
}
__device__ __forceinline__ float2 load_pair(const __half* p) {
  return __half22float2(*reinterpret_cast<const __half2*>(p));
}

// the same pair where it may start on an odd sample (odd hops): two scalar loads
__device__ __forceinline__ float2 load_pair_odd(const float* p) { return make_float2(p[0], p[1]); }
__device__ __forceinline__ float2 load_pair_odd(const short* p) { return make_float2((float)p[0], (float)p[1]); }
__device__ __forceinline__ float2 load_pair_odd(const __half* p) {
  return make_float2(__half2float(p[0]), __half2float(p[1]));
}

__device__ __forceinline__ float load_one(const float* p) { return __ldg(p); }
__device__ __forceinline__ short load_one(const short* p) { return __ldg(p); }
__device__ __forceinline__ __half load_one(const __half* p) { return __ldg(p); }

template <typename Raw>
__device__ __forceinline__ Raw raw_zero() {
  if constexpr (std::is_same<Raw, __half>::value) return __float2half_rn(0.0f);
  else return Raw(0);
}

// Framing of one signal outside its samples [0, T): zpad zeros on each side
// (torchaudio's `pad`), then cpad samples of centre padding by mode.
struct PadSpec {
  int zpad, cpad, mode;
};

// The signal index whose sample stands at position s (< 0 or >= T) of the
// padded signal, or -1 for a zero: one of the `pad` zeros, constant centre
// padding, or a position past the padded signal (no valid frame reads it).
// With T' = T + 2 zpad and j = s + zpad the index in the zero-padded signal:
// reflect mirrors j about its first / last sample without repeating it,
// replicate repeats the edge, circular wraps by T' (torch's pad modes).
__device__ __forceinline__ long long padded_source(long long s, long long T, const PadSpec& ps) {
  if (s >= 0 && s < T) return s;
  const long long Tp = T + 2 * (long long)ps.zpad;
  long long j = s + ps.zpad;
  if (j >= 0 && j < Tp) return -1;
  if (j < -(long long)ps.cpad || j >= Tp + ps.cpad) return -1;
  if (ps.mode == FM_PAD_REFLECT) j = j < 0 ? -j : 2 * (Tp - 1) - j;
  else if (ps.mode == FM_PAD_REPLICATE) j = j < 0 ? 0 : Tp - 1;
  else if (ps.mode == FM_PAD_CIRCULAR) j = j < 0 ? j + Tp : j - Tp;
  else return -1;
  const long long src = j - ps.zpad;
  return (src >= 0 && src < T) ? src : -1;
}

// The length in elements of the buffer a guarded access touches, and the
// plan's error word: what the debug build's index checks (FM_IN) compare
// against. The normal build never reads it.
struct Cap {
  int n;
  unsigned* err;
};

// Element i of a row that starts at element `off` of a buffer of cap.n
// elements: stored / loaded only if it lies inside the buffer (checked in the
// debug build; a plain access otherwise).
template <typename T>
__device__ __forceinline__ void put(T* row, int off, int i, const T& v, Cap cap) {
  if (FM_IN(off + i >= 0 && off + i < cap.n, cap.err)) row[i] = v;
}
template <typename T>
__device__ __forceinline__ T get(const T* row, int off, int i, Cap cap) {
  return FM_IN(off + i >= 0 && off + i < cap.n, cap.err) ? row[i] : T{};
}

// The general staging path of stage_tile: rows [0, rows) of hop samples from
// signal index gstart, in-range aligned pairs as one cp.async, every other
// sample through padded_source. Positions from the end of the padded signal
// (T + zpad + cpad) on are left untouched: no valid frame reads them. Kept
// out of line: only tiles at the signal edges (or with misaligned rows) take
// it, and its code then stays out of the kernels' hot loops.
template <typename Raw>
__device__ __noinline__ void stage_rows_padded(const Raw* __restrict__ src, long long T, long long gstart, int rows,
                                               int hop, int S, Raw* dst, int warp, int nwarps, int lane,
                                               PadSpec ps, Cap cap) {
  const bool aligned = ((reinterpret_cast<uintptr_t>(src + gstart)) % (2 * sizeof(Raw))) == 0;
  const int pairs = hop / 2;
  const long long end = T + ps.zpad + ps.cpad;  // one past the padded signal
  // the default framing (centre reflect, no `pad` zeros) maps by mirroring alone
  const bool plain_reflect = ps.zpad == 0 && ps.mode == FM_PAD_REFLECT;
  for (int r = warp; r < rows; r += nwarps) {
    Raw* d = dst + r * S;
    const long long s0 = gstart + (long long)r * hop;
    if (s0 >= end) break;
    const long long left = (end - s0 + 1) / 2;  // pairs that start inside the padded signal
    const int c2_end = left < pairs ? (int)left : pairs;
    for (int c2 = lane; c2 < c2_end; c2 += 32) {
      const long long s = s0 + 2 * c2;
      if (aligned && s >= 0 && s + 1 < T) {
        if (FM_IN(r * S + 2 * c2 + 1 < cap.n, cap.err)) cp_async<2 * sizeof(Raw)>(d + 2 * c2, src + s);
        continue;
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        long long se = s + e;
        if (plain_reflect) {
          if (se < 0) se = -se;                   // mirror about the first sample
          else if (se >= T) se = 2 * T - 2 - se;  // mirror about the last sample
          if (se >= T) se = -1;                   // past the padded signal (not read)
        } else {
          se = padded_source(se, T, ps);
        }
        Raw* de = d + 2 * c2 + e;
        if (!FM_IN(r * S + 2 * c2 + e < cap.n && se < T, cap.err)) continue;
        if (se < 0) {
          *de = raw_zero<Raw>();
        } else if constexpr (sizeof(Raw) == 4) {
          cp_async<4>(de, src + se);
        } else {
          *de = load_one(src + se);
        }
      }
    }
  }
}

// Stage rows [0, rows) of hop samples starting at signal index gstart of
// signal row `src` (length T) into dst (row stride S elements), as
// asynchronous copies wherever possible: aligned in-range sample pairs as one
// 8- or 4-byte cp.async; otherwise element by element through
// padded_source (the padding of `ps`), f32 still by 4-byte cp.async and
// 16-bit samples by plain loads (only the few padded or misaligned ones).
// The caller commits the group, waits for it and then synchronises the CTA.
template <typename Raw, int NWARPS>
__device__ __forceinline__ void stage_tile(const Raw* __restrict__ src, long long T, long long gstart, int rows,
                                           int hop, int S, Raw* dst, int warp, int lane, const PadSpec& ps,
                                           Cap cap) {
  const bool interior = gstart >= 0 && gstart + (long long)rows * hop <= T;
  const bool aligned = ((reinterpret_cast<uintptr_t>(src + gstart)) % (2 * sizeof(Raw))) == 0;
  const int pairs = hop / 2;
  if (interior && aligned) {
    for (int r = warp; r < rows; r += NWARPS) {
      const Raw* s = src + gstart + (long long)r * hop;
      Raw* d = dst + r * S;
      for (int c2 = lane; c2 < pairs; c2 += 32)
        if (FM_IN(r * S + 2 * c2 + 1 < cap.n && gstart + (long long)r * hop + 2 * c2 + 1 < T, cap.err))
          cp_async<2 * sizeof(Raw)>(d + 2 * c2, s + 2 * c2);
    }
    return;
  }
  stage_rows_padded<Raw>(src, T, gstart, rows, hop, S, dst, warp, NWARPS, lane, ps, cap);
}

// Staging for odd hops, where rows of one hop cannot keep sample pairs
// aligned: the tile is one contiguous run of `len` samples from signal index
// gstart (frame g starts at element g * hop). In-range samples arrive by
// cp.async: f32 one per copy, 16-bit samples two per copy when the run starts
// on a 4-byte boundary of the signal, else by plain loads. Padding goes
// through padded_source; positions past the padded signal are left
// untouched (no valid frame reads them). The caller commits, waits and
// synchronises as for stage_tile.
template <typename Raw>
__device__ __noinline__ void stage_run(const Raw* __restrict__ src, long long T, long long gstart, int len, Raw* dst,
                                       int tid, int nthreads, PadSpec ps, Cap cap) {
  const long long end = T + ps.zpad + ps.cpad;  // one past the padded signal
  if constexpr (sizeof(Raw) == 2) {
    const bool pairs_ok = gstart >= 0 && gstart + len <= T && (reinterpret_cast<uintptr_t>(src + gstart) & 3) == 0;
    if (pairs_ok) {
      for (int i = 2 * tid; i + 1 < len; i += 2 * nthreads)
        if (FM_IN(i + 1 < cap.n, cap.err)) cp_async<4>(dst + i, src + gstart + i);
      if ((len & 1) && tid == 0 && FM_IN(len - 1 < cap.n, cap.err)) dst[len - 1] = load_one(src + gstart + len - 1);
      return;
    }
  }
  for (int i = tid; i < len; i += nthreads) {
    const long long s = gstart + i;
    if (s >= end) break;  // s only grows with i
    const long long se = (s >= 0 && s < T) ? s : padded_source(s, T, ps);
    if (!FM_IN(i < cap.n && se < T, cap.err)) continue;
    if (se < 0) {
      dst[i] = raw_zero<Raw>();
    } else if constexpr (sizeof(Raw) == 4) {
      cp_async<4>(dst + i, src + se);
    } else {
      dst[i] = load_one(src + se);
    }
  }
}

// Pass 1 for role p and frame g: windowed Q-point DFT of z[p + P q] and the
// four-step twiddle W_M^{p k2}; writes row g of the exchange buffer at
// [k2 * P + p]. frame_off / xoff: the frame's and the row's offsets in the
// staging and exchange buffers (for the debug build's index checks).
template <int P, int Q, bool ODD, typename Raw>
__device__ __forceinline__ void pass1(const Raw* __restrict__ frame_base, const float4* __restrict__ s_p1,
                                      const float2* __restrict__ s_twh, float2* xrow, int p, int frame_off,
                                      Cap in_cap, int xoff, Cap x_cap) {
  float2 z[Q];
  const float4* tab = s_p1 + p * Q;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const float4 e = tab[q];
    const int o = __float_as_int(e.z);
    const Raw* src = frame_base + o;
    float2 v = make_float2(0.0f, 0.0f);
    if (FM_IN(frame_off + o >= 0 && frame_off + o + 1 < in_cap.n, in_cap.err))
      v = ODD ? load_pair_odd(src) : load_pair(src);
    z[q] = make_float2(v.x * e.x, v.y * e.y);
  }
  dft<Q>(z);
  if (FM_IN(xoff + p < x_cap.n, x_cap.err)) xrow[p] = z[0];
#pragma unroll
  for (int k2 = 1; k2 < Q; ++k2)
    if (FM_IN(xoff + k2 * P + p < x_cap.n, x_cap.err)) xrow[k2 * P + p] = cmul(z[k2], s_twh[p * k2]);
}

// Copy `bytes` (a multiple of 8, both ends 8-byte aligned) from global to
// shared memory with cp.async, 16 bytes per copy where alignment allows.
__device__ __forceinline__ void copy_table_async(void* dst, const void* src, int bytes, int tid, int nthreads) {
  unsigned char* d = static_cast<unsigned char*>(dst);
  const unsigned char* s = static_cast<const unsigned char*>(src);
  if (((reinterpret_cast<uintptr_t>(d) | reinterpret_cast<uintptr_t>(s)) & 15) == 0 && (bytes & 15) == 0) {
    for (int i = tid * 16; i < bytes; i += nthreads * 16) cp_async<16>(d + i, s + i);
  } else {
    for (int i = tid * 8; i < bytes; i += nthreads * 8) cp_async<8>(d + i, s + i);
  }
}

// tile -> (signal b, tile index within the signal), without a 64-bit divide:
// a float reciprocal gives the quotient to within one, then one correction.
struct TileSplitter {
  int tps;
  float inv;
  __device__ explicit TileSplitter(int tiles_per_signal) : tps(tiles_per_signal), inv(1.0f / (float)tiles_per_signal) {}
  __device__ __forceinline__ void operator()(long long tile, long long& b, int& tt) const {
    if (tile < (1LL << 22)) {
      const int t = (int)tile;
      int q = (int)((float)t * inv);
      int r = t - q * tps;
      if (r < 0) {
        r += tps;
        --q;
      } else if (r >= tps) {
        r -= tps;
        ++q;
      }
      b = q;
      tt = r;
    } else {
      b = tile / tps;
      tt = (int)(tile - b * tps);
    }
  }
};

template <int MODE>
__device__ __forceinline__ float power_of(float2 x, float p) {
  const float m2 = fmaf(x.x, x.x, x.y * x.y);
  if constexpr (MODE == 0) return m2;
  else if constexpr (MODE == 1) return sqrtf(m2);
  else return powf(m2, 0.5f * p);
}

// |X[k]|^p and |X[M-k]|^p from Z[k], Z[M-k] and W_N^k.
template <int MODE>
__device__ __forceinline__ void split_pair(float2 zk, float2 zm, float2 w, float p, float& out_k, float& out_mk) {
  const float2 s = make_float2(zk.x + zm.x, zk.y - zm.y);
  const float2 d = make_float2(zk.x - zm.x, zk.y + zm.y);
  const float2 u = mul_neg_i(cmul(d, w));
  out_k = power_of<MODE>(cadd(s, u), p);
  out_mk = power_of<MODE>(csub(s, u), p);
}

// Pass 2 and split when Q = 2P. Role t >= 1 holds k2 = t and Q - t; role 0
// holds k2 = 0 and Q/2, whose pairs (k, M - k) fall inside each set. Ends
// with the power values written into prow (which aliases the exchange
// buffer: the barrier inside separates all reads from all writes).
template <int N, int P, int Q, int MODE>
__device__ __forceinline__ void pass2_split_paired(const float2* xrow, float* prow, const float2* __restrict__ s_twf,
                                                   int t, float pw, int xoff, Cap x_cap, int poff, Cap p_cap) {
  constexpr int M = N / 2;
  static_assert(Q == 2 * P && P % 2 == 0, "paired split needs Q = 2P with P even");
  const int kA = t;                      // 0 for role 0
  const int kB = (t == 0) ? Q / 2 : Q - t;
  float2 a[P], b[P];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    a[p] = get(xrow, xoff, kA * P + p, x_cap);
    b[p] = get(xrow, xoff, kB * P + p, x_cap);
  }
  dft<P>(a);  // a[k1] = Z[kA + Q k1]
  dft<P>(b);  // b[k1] = Z[kB + Q k1]
  __syncthreads();
  if (t != 0) {
    // Z[t + Q k1] pairs with Z[(Q - t) + Q (P - 1 - k1)]
#pragma unroll
    for (int k1 = 0; k1 < P; ++k1) {
      const int k = t + Q * k1;
      float lo, hi;
      split_pair<MODE>(a[k1], b[P - 1 - k1], s_twf[k], pw, lo, hi);
      put(prow, poff, k, lo, p_cap);
      put(prow, poff, M - k, hi, p_cap);
    }
  } else {
    // k = Q k1 pairs with Q (P - k1); k1 = 0 gives X[0] and X[M]
#pragma unroll
    for (int k1 = 0; k1 <= P / 2; ++k1) {
      const int k = Q * k1;
      float lo, hi;
      split_pair<MODE>(a[k1], a[(P - k1) % P], s_twf[k], pw, lo, hi);
      put(prow, poff, k, lo, p_cap);
      put(prow, poff, M - k, hi, p_cap);
    }
    // k = Q/2 + Q k1 pairs with Q/2 + Q (P - 1 - k1)
#pragma unroll
    for (int k1 = 0; k1 < P / 2; ++k1) {
      const int k = Q / 2 + Q * k1;
      float lo, hi;
      split_pair<MODE>(b[k1], b[P - 1 - k1], s_twf[k], pw, lo, hi);
      put(prow, poff, k, lo, p_cap);
      put(prow, poff, M - k, hi, p_cap);
    }
  }
}

// Pass 2 and split when Q = P: role t does the P-point DFT for k2 = t, Z goes
// back through shared memory, and role t then splits the pairs k = t + P j.
template <int N, int P, int Q, int MODE>
__device__ __forceinline__ void pass2_split_exchange(float2* xrow, float* prow, const float2* __restrict__ s_twf,
                                                     int t, float pw, int xoff, Cap x_cap, int poff, Cap p_cap) {
  constexpr int M = N / 2;
  constexpr int PAIRS = M / 2 + 1;  // k = 0 .. M/2
  constexpr int PPR = (PAIRS + P - 1) / P;
  static_assert(Q == P, "exchange split is for Q = P");
  float2 y[P];
#pragma unroll
  for (int p = 0; p < P; ++p) y[p] = get(xrow, xoff, t * P + p, x_cap);
  dft<P>(y);
  __syncthreads();
#pragma unroll
  for (int k1 = 0; k1 < P; ++k1) put(xrow, xoff, t + Q * k1, y[k1], x_cap);
  __syncthreads();
  float lo[PPR], hi[PPR];
#pragma unroll
  for (int i = 0; i < PPR; ++i) {
    const int k = t + i * P;
    lo[i] = hi[i] = 0.0f;
    if (k <= M / 2)
      split_pair<MODE>(get(xrow, xoff, k, x_cap), get(xrow, xoff, k == 0 ? 0 : M - k, x_cap), s_twf[k], pw, lo[i],
                       hi[i]);
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < PPR; ++i) {
    const int k = t + i * P;
    if (k <= M / 2) {
      put(prow, poff, k, lo[i], p_cap);
      put(prow, poff, M - k, hi[i], p_cap);
    }
  }
}

template <int N, int P, int Q, int MODE>
__device__ __forceinline__ void pass2_split(float2* xrow, float* prow, const float2* s_twf, int t, float pw, int xoff,
                                            Cap x_cap, int poff, Cap p_cap) {
  if constexpr (Q == 2 * P) pass2_split_paired<N, P, Q, MODE>(xrow, prow, s_twf, t, pw, xoff, x_cap, poff, p_cap);
  else pass2_split_exchange<N, P, Q, MODE>(xrow, prow, s_twf, t, pw, xoff, x_cap, poff, p_cap);
}

__device__ __forceinline__ void store_out(float* o, float v) { *o = v; }
__device__ __forceinline__ void store_out(__half* o, float v) { *o = __float2half_rn(v); }

// Sparse mel projection: lane = frame, G lanes per mel, warp-uniform filter
// rows read as broadcasts; stores of consecutive frames are coalesced.
// p_cap: the power tile's floats; nnz: the filter weights; out_left: output
// elements from out_tile to the end of the output (debug-build checks).
template <int G, int NWARPS, int PS, typename OutT>
__device__ __forceinline__ void mel_project(const float* s_pw, const int4* __restrict__ s_mel,
                                            const float* __restrict__ s_mw, OutT* out_tile, int n_valid,
                                            int n_mels, long long n_frames, int warp, int lane, Cap p_cap,
                                            int nnz, long long out_left) {
  constexpr int SUBS = 32 / G;
  const int gg = lane % G, sub = lane / G;
  const float* prow = s_pw + gg * PS;
  const bool valid = gg < n_valid;
  OutT* o = out_tile + gg;
  for (int m = warp * SUBS + sub; m < n_mels; m += NWARPS * SUBS) {
    const int4 md = s_mel[m];
    const float* pr = prow + md.x;
    const float* wr = s_mw + md.z;
    float acc = 0.0f;
#pragma unroll 4
    for (int j = 0; j < md.y; ++j)
      if (FM_IN(gg * PS + md.x + j >= 0 && gg * PS + md.x + j < p_cap.n && md.z + j >= 0 && md.z + j < nnz,
                p_cap.err))
        acc = fmaf(wr[j], pr[j], acc);
    if (valid && FM_IN(gg + (long long)m * n_frames < out_left, p_cap.err)) store_out(o + (long long)m * n_frames, acc);
  }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int N, int P, int Q, int G, int NBUF, bool ODD, typename Raw>
__device__ __forceinline__ void run_tiles(const KernelParams& prm, unsigned char* smem, const SmemLayout& lay) {
  constexpr int M = N / 2;
  constexpr int THREADS = P * G;
  constexpr int NWARPS = THREADS / 32;
  constexpr int GS = M + 1;  // complex stride between frames in the exchange buffer (odd)
  constexpr int PS = M + 1;  // float stride between frames in the power tile (odd)
  const float4* s_p1 = reinterpret_cast<const float4*>(smem + lay.p1);
  const float2* s_twh = reinterpret_cast<const float2*>(smem + lay.tw_half);
  const float2* s_twf = reinterpret_cast<const float2*>(smem + lay.tw_full);
  const int4* s_mel = reinterpret_cast<const int4*>(smem + lay.mel);
  const float* s_mw = reinterpret_cast<const float*>(smem + lay.mel_w);
  float2* s_x = reinterpret_cast<float2*>(smem + lay.xbuf);
  float* s_pw = reinterpret_cast<float*>(smem + lay.xbuf);  // aliases s_x after pass 2

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = tid % G, role = tid / G;
  const int hop = prm.hop, S = in_row_stride(hop), rows = in_rows(N, hop, G);
  const Raw* in = static_cast<const Raw*>(prm.in);
  const long long T = prm.T;
  const TileSplitter split(prm.tiles_per_signal);
  const PadSpec pads = {prm.zpad, prm.cpad, prm.pad_mode};
  auto in_buf = [&](int i) { return reinterpret_cast<Raw*>(smem + lay.in_tile + (size_t)i * lay.in_tile_bytes); };
  // buffer sizes for the debug build's index checks
  const Cap in_cap = {(int)(lay.in_tile_bytes / sizeof(Raw)), prm.err};
  const Cap x_cap = {G * GS, prm.err}, p_cap = {G * PS, prm.err};
  const long long out_total = prm.B * (long long)prm.n_mels * prm.n_frames;
  auto stage = [&](long long tile, int buf) {
    long long b;
    int tt;
    split(tile, b, tt);
    const long long t0 = (long long)tt * G;
    if constexpr (ODD)  // rows of one odd hop, back to back (S == hop)
      stage_run<Raw>(in + b * T, T, t0 * hop - prm.lead, rows * hop, in_buf(buf), tid, THREADS, pads, in_cap);
    else
      stage_tile<Raw, NWARPS>(in + b * T, T, t0 * hop - prm.lead, rows, hop, S, in_buf(buf), warp, lane, pads,
                              in_cap);
    cp_async_commit();
  };

  long long tile = blockIdx.x;
  int buf = 0;
  if (tile < prm.total_tiles) stage(tile, 0);
  for (; tile < prm.total_tiles; tile += gridDim.x) {
    cp_async_wait_all();
    __syncthreads();  // this tile's samples are visible; the previous tile is fully done
    const long long next = tile + gridDim.x;
    if (NBUF == 2 && next < prm.total_tiles) stage(next, buf ^ 1);

    float2* xrow = s_x + g * GS;
    pass1<P, Q, ODD, Raw>(in_buf(buf) + g * S, s_p1, s_twh, xrow, role, g * S, in_cap, g * GS, x_cap);
    __syncthreads();
    if (NBUF == 1 && next < prm.total_tiles) stage(next, 0);  // pass 1 was the last reader

    float* prow = s_pw + g * PS;
    switch (prm.power_mode) {
      case 0: pass2_split<N, P, Q, 0>(xrow, prow, s_twf, role, prm.power, g * GS, x_cap, g * PS, p_cap); break;
      case 1: pass2_split<N, P, Q, 1>(xrow, prow, s_twf, role, prm.power, g * GS, x_cap, g * PS, p_cap); break;
      default: pass2_split<N, P, Q, 2>(xrow, prow, s_twf, role, prm.power, g * GS, x_cap, g * PS, p_cap); break;
    }
    __syncthreads();

    long long b;
    int tt;
    split(tile, b, tt);
    const int t0 = tt * G;
    const int n_valid = min(G, prm.n_frames - t0);
    const long long obase = b * prm.n_mels * (long long)prm.n_frames + t0;
    if (prm.out_dtype == FM_F32)
      mel_project<G, NWARPS, PS>(s_pw, s_mel, s_mw, static_cast<float*>(prm.out) + obase, n_valid, prm.n_mels,
                                 prm.n_frames, warp, lane, p_cap, prm.nnz, out_total - obase);
    else
      mel_project<G, NWARPS, PS>(s_pw, s_mel, s_mw, static_cast<__half*>(prm.out) + obase, n_valid, prm.n_mels,
                                 prm.n_frames, warp, lane, p_cap, prm.nnz, out_total - obase);
    if (NBUF == 2) buf ^= 1;
    // The next iteration's barrier orders these power-tile reads before the
    // next pass 1 overwrites the exchange buffer.
  }
  cp_async_commit();  // nothing may stay in flight past the end of the CTA
  cp_async_wait_all();
}

template <int N, int P, int Q, int G, int NBUF, bool ODD>
__global__ void __launch_bounds__(P* G) mel_kernel(const KernelParams prm) {
  constexpr int M = N / 2;
  constexpr int THREADS = P * G;
  static_assert(P * Q == M && (Q == P || Q == 2 * P), "bad FFT split");
  static_assert(G == 32 || G == 16, "frames per tile must be 16 or 32");
  static_assert(THREADS % 32 == 0, "CTA must be whole warps");
  extern __shared__ __align__(16) unsigned char smem[];
  const int esize = prm.in_dtype == FM_F32 ? 4 : 2;
  const SmemLayout lay = smem_layout(N, prm.hop, prm.n_mels, prm.nnz, G, esize, NBUF);

  pdl_launch_dependents();
  // per-CTA constant tables, fetched once (the grid is persistent) in the same
  // cp.async group as the first tile, so one wait covers both
  const int tid = threadIdx.x;
  copy_table_async(smem + lay.p1, prm.p1, (int)sizeof(float4) * M, tid, THREADS);
  copy_table_async(smem + lay.tw_half, prm.tw_half, (int)sizeof(float2) * M, tid, THREADS);
  copy_table_async(smem + lay.tw_full, prm.tw_full, (int)sizeof(float2) * (M + 1) + ((M + 1) & 1) * 8, tid, THREADS);
  copy_table_async(smem + lay.mel, prm.mel, (int)sizeof(int4) * prm.n_mels, tid, THREADS);
  copy_table_async(smem + lay.mel_w, prm.mel_w, (int)align16(sizeof(float) * (prm.nnz > 0 ? prm.nnz : 1)), tid, THREADS);
  pdl_wait();  // caller buffers only after the previous kernel in the stream is done
  // (the first barrier inside run_tiles publishes the tables)

  if (prm.in_dtype == FM_F32) run_tiles<N, P, Q, G, NBUF, ODD, float>(prm, smem, lay);
  else if (prm.in_dtype == FM_I16) run_tiles<N, P, Q, G, NBUF, ODD, short>(prm, smem, lay);
  else run_tiles<N, P, Q, G, NBUF, ODD, __half>(prm, smem, lay);
}

}  // namespace fm

// Instantiate one variant: FM_DEFINE_VARIANT(name, N, P, Q, G, NBUF) for even
// hops, FM_DEFINE_VARIANT_ODD(...) for odd ones
#define FM_DEFINE_VARIANT_HOPS(NAME, N, P, Q, G, NBUF, ODD, HOPS)                                      \
  namespace fm {                                                                                        \
  template __global__ void mel_kernel<N, P, Q, G, NBUF, ODD>(const KernelParams);                     \
  extern const Variant NAME = {N,    P, Q, G, P * G, NBUF, 0, (const void*)&mel_kernel<N, P, Q, G, NBUF, ODD>, \
                               HOPS};                                                                   \
  }
#define FM_DEFINE_VARIANT(NAME, N, P, Q, G, NBUF) FM_DEFINE_VARIANT_HOPS(NAME, N, P, Q, G, NBUF, false, kEvenHops)
#define FM_DEFINE_VARIANT_ODD(NAME, N, P, Q, G, NBUF) FM_DEFINE_VARIANT_HOPS(NAME, N, P, Q, G, NBUF, true, kOddHops)
