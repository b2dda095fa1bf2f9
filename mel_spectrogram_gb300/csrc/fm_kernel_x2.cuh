// Two-frames-per-thread variant of the fused mel kernel (sm_103a), for the
// splits with Q = 2P (n_fft = 400, 256, 64) and Q = P (n_fft = 128, 512).
//
// Same path and same four-step real FFT as fm_kernel.cuh, but a tile holds 32
// frames and thread (role, g), g < 16, carries frames g and g + 16 through
// every phase as packed pairs (see fm_fft2.cuh):
//   staging : raw samples in lines of two hops (one when the hop is a
//             runtime value) in the upper half of the exchange buffer,
//             which is free from the end of pass 2 (the power tile uses the
//             lower half) to the start of the next pass 1: the next tile
//             lands during the split and the mel projection. A producer
//             warp stages every group's tiles: one tensor-map TMA copy per
//             interior tile, line copies plus cp.async element copies at the
//             signal edges;
//   tables  : window/offset, twiddles and filters are copied once per CTA
//             into shared memory and read as broadcasts;
//   pass 1  : two 8-byte pair loads per step, the window multiply scatters
//             them into the packed layout; Q-point DFT; twiddle W_M^{p k2};
//             {re_a, re_b, im_a, im_b} per value as two 8-byte stores;
//   pass 2  : P-point DFTs for k2 = t and Q - t (role 0: 0 and Q/2), then the
//             real-FFT split and |X|^p, still packed;
//   power   : tile rows P[k] of 32 frames, 16 bytes per 4 frames;
//   mel     : quarter-warps on four filters, lane = 4 frames, two packed
//             FMAs per filter weight.
#pragma once

#include "fm_fft2.cuh"
#include "fm_kernel.cuh"

namespace fm {

constexpr int kX2Lanes = 16;   // lanes per role
constexpr int kX2Frames = 32;  // frames per tile

// Barrier over one tile group (named barrier `id`, `n` threads), and the same
// with an OR vote over the group's threads.
__device__ __forceinline__ void group_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ bool group_sync_or(int id, int n, bool v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((int)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Pass 1, load half: the windowed pairs z[q] = (y[2n], y[2n+1]) / 2 with
// n = p + P q, for frames g and g + 16. HOP > 0: the hop is a compile-time
// multiple of 2P and the tile is staged in lines of two hops, frame g starting
// at line g / 2, column (g % 2) HOP; base points at sample 2p of frame g and
// base_o is base plus one line pad for odd g. The line crossings of sample
// 2Pq + 2p do not depend on p, so every load is a compile-time offset from
// base or base_o (frame g + 16 is 8 lines further). HOP = 0: lines of one hop,
// frame g on line g, and the offsets come from the table.
// A sample pair of the staged tile, read only if it lies inside the staging
// area that starts at s_in (checked in the debug build).
template <typename Raw>
__device__ __forceinline__ float2 staged_pair(const Raw* p, const Raw* s_in, Cap cap) {
  const long long o = p - s_in;
  return FM_IN(o >= 0 && o + 1 < cap.n, cap.err) ? load_pair(p) : make_float2(0.0f, 0.0f);
}

template <int P, int Q, int HOP, typename Raw>
__device__ __forceinline__ void pass1_load_x2(const Raw* __restrict__ base, const Raw* __restrict__ base_o, int S,
                                              const float4* __restrict__ s_p1, int p, cx2 (&z)[Q], const Raw* s_in,
                                              Cap in_cap) {
  const float4* tab = s_p1 + p * Q;
  if constexpr (HOP > 0) {
    static_assert(HOP % (2 * P) == 0, "compile-time hop must be a multiple of 2P");
    constexpr int SC = in_row_stride_x2_c(2 * HOP, (int)sizeof(Raw));
    constexpr int PAD = SC - 2 * HOP;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const float2 w = *reinterpret_cast<const float2*>(tab + q);
      const int j = 2 * P * q;
      const int ce = j / (2 * HOP), co = (HOP + j) / (2 * HOP);  // lines crossed, even / odd g
      const Raw* b = co != ce ? base_o : base;
      const int off = j + ce * PAD;
      const float2 va = staged_pair(b + off, s_in, in_cap);
      const float2 vb = staged_pair(b + off + (kX2Lanes / 2) * SC, s_in, in_cap);
      z[q].re = make_float2(va.x * w.x, vb.x * w.x);
      z[q].im = make_float2(va.y * w.y, vb.y * w.y);
    }
  } else {
    const Raw* base_b = base + kX2Lanes * S;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const float4 e = tab[q];
      const int off = __float_as_int(e.z);
      const float2 va = staged_pair(base + off, s_in, in_cap);
      const float2 vb = staged_pair(base_b + off, s_in, in_cap);
      z[q].re = make_float2(va.x * e.x, vb.x * e.x);
      z[q].im = make_float2(va.y * e.y, vb.y * e.y);
    }
  }
}

__device__ __forceinline__ cx2 load_cx2(const float4* p) {
  const float4 v = *p;
  return {make_float2(v.x, v.y), make_float2(v.z, v.w)};
}

template <int MODE>
__device__ __forceinline__ float2 power2(float2 re, float2 im, float pw) {
  const float2 m2 = fma2(re, re, mul2(im, im));
  if constexpr (MODE == 0) return m2;
  else if constexpr (MODE == 1) return make_float2(sqrtf(m2.x), sqrtf(m2.y));
  else return make_float2(powf(m2.x, 0.5f * pw), powf(m2.y, 0.5f * pw));
}

// (|X[k]|^p, |X[M-k]|^p) for both frames from Z[k], Z[M-k] and W_N^k.
template <int MODE>
__device__ __forceinline__ void split_pair_x2(cx2 zk, cx2 zm, float4 w, float pw, float2& out_k, float2& out_mk) {
  const cx2 s = {add2(zk.re, zm.re), sub2(zk.im, zm.im)};
  const cx2 d = {sub2(zk.re, zm.re), add2(zk.im, zm.im)};
  const cx2 v = cmul(d, make_float2(w.x, w.y), make_float2(w.z, w.w));
  // X[k] = s - i v, conj X[M-k] = s + i v
  out_k = power2<MODE>(add2(s.re, v.im), sub2(s.im, v.re), pw);
  out_mk = power2<MODE>(sub2(s.re, v.im), add2(s.im, v.re), pw);
}

// Pass 2 for Q = 2P: role t >= 1 holds k2 = t and Q - t, role 0 holds k2 = 0
// and Q/2; P-point DFTs over p give a[k1] = Z[kA + Q k1], b[k1] = Z[kB + Q k1].
template <int P, int Q>
__device__ __forceinline__ void pass2_x2(const float4* xq_row, int t, cx2 (&a)[P], cx2 (&b)[P], int xoff, Cap x_cap) {
  static_assert(Q == 2 * P && P % 2 == 0, "paired split needs Q = 2P with P even");
  const int kA = t;
  const int kB = (t == 0) ? Q / 2 : Q - t;
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const float4 va = get(xq_row, xoff, kA * P + p, x_cap), vb = get(xq_row, xoff, kB * P + p, x_cap);
    a[p] = {make_float2(va.x, va.y), make_float2(va.z, va.w)};
    b[p] = {make_float2(vb.x, vb.y), make_float2(vb.z, vb.w)};
  }
  dft<P>(a);
  dft<P>(b);
}

__device__ __forceinline__ cx2 sel(bool c, const cx2& a, const cx2& b) { return c ? a : b; }

// Real-FFT split of pass 2's outputs: both members of every pair (k, M - k)
// are in this thread's registers; power pairs go to pw_col[k * 16] (float2,
// 128-byte bin rows).
//   role t >= 1: pairs (a[j], b[P-1-j]) at k = t + Q j, j < P;
//   role 0:      pairs (a[j], a[(P-j) % P]) at k = Q j, j <= P/2 (j = 0 gives
//                X[0] and X[M]), and (b[i], b[P-1-i]) at k = Q/2 + Q i, i < P/2.
// The warp holding role 0 (with role 1 beside it) runs both as one stream of
// P + 1 slots with the operands chosen by selects, so it does not execute two
// divergent paths while the other warps wait at the next barrier.
template <int N, int P, int Q, int MODE>
__device__ __forceinline__ void split_x2(const cx2 (&a)[P], const cx2 (&b)[P], float2* pw_col,
                                         const float4* __restrict__ s_twf4, int t, float pw, bool merged, int poff,
                                         Cap p_cap) {
  constexpr int M = N / 2;
  if (!merged) {
#pragma unroll
    for (int k1 = 0; k1 < P; ++k1) {
      const int k = t + Q * k1;
      float2 lo, hi;
      split_pair_x2<MODE>(a[k1], b[P - 1 - k1], s_twf4[k], pw, lo, hi);
      put(pw_col, poff, k * kX2Lanes, lo, p_cap);
      put(pw_col, poff, (M - k) * kX2Lanes, hi, p_cap);
    }
    return;
  }
  const bool r0 = (t == 0);
#pragma unroll
  for (int j = 0; j <= P; ++j) {
    cx2 u, v;
    int k;
    if (j <= P / 2) {
      u = a[j];
      v = sel(r0, a[(P - j) % P], b[P - 1 - j]);
      k = t + Q * j;
    } else if (j < P) {
      u = sel(r0, b[j - P / 2 - 1], a[j]);
      v = sel(r0, b[3 * P / 2 - j], b[P - 1 - j]);
      k = r0 ? Q / 2 + Q * (j - P / 2 - 1) : t + Q * j;
    } else {  // the one extra pair of role 0
      u = b[P / 2 - 1];
      v = b[P / 2];
      k = Q / 2 + Q * (P / 2 - 1);
    }
    if (j < P || r0) {
      float2 lo, hi;
      split_pair_x2<MODE>(u, v, s_twf4[k], pw, lo, hi);
      put(pw_col, poff, k * kX2Lanes, lo, p_cap);
      put(pw_col, poff, (M - k) * kX2Lanes, hi, p_cap);
    }
  }
}

// Pass 2 and split when Q = P (n_fft 128, 512): role t does the P-point DFT over p
// for k2 = t, Z[t + Q k1] goes back through the exchange buffer in natural
// order, and role t then splits the pairs (k, M - k), k = t + P i <= M/2
// (k = 0 gives X[0] and X[M]). The power values stay in registers until every
// thread has read its Z, since the power tile and the next staged tile
// overwrite the buffer; `freed` then releases the staging area.
template <int N, int P, int MODE, typename Freed>
__device__ __forceinline__ void pass2_split_exchange_x2(float4* xq_row, float2* pw_col, const float4* __restrict__ s_twf4,
                                                        int t, float pw, int xoff, Cap x_cap, int poff, Cap p_cap,
                                                        int bar_id, int threads, Freed freed) {
  constexpr int M = N / 2, Q = P;
  constexpr int PER = (M / 2) / P + 1;
  cx2 y[P];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const float4 v = get(xq_row, xoff, t * P + p, x_cap);
    y[p] = {make_float2(v.x, v.y), make_float2(v.z, v.w)};
  }
  dft<P>(y);
  group_sync(bar_id, threads);  // every pass-1 value read before Z overwrites the rows
#pragma unroll
  for (int k1 = 0; k1 < P; ++k1)
    put(xq_row, xoff, t + Q * k1, make_float4(y[k1].re.x, y[k1].re.y, y[k1].im.x, y[k1].im.y), x_cap);
  group_sync(bar_id, threads);
  float2 lo[PER], hi[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int k = t + P * i;
    lo[i] = hi[i] = make_float2(0.0f, 0.0f);
    if (k <= M / 2) {
      const float4 a = get(xq_row, xoff, k, x_cap), b = get(xq_row, xoff, (M - k) % M, x_cap);
      split_pair_x2<MODE>({make_float2(a.x, a.y), make_float2(a.z, a.w)}, {make_float2(b.x, b.y), make_float2(b.z, b.w)},
                          s_twf4[k], pw, lo[i], hi[i]);
    }
  }
  group_sync(bar_id, threads);  // every Z read: the power tile and the next staged tile may land
  freed();
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int k = t + P * i;
    if (k <= M / 2) {
      put(pw_col, poff, k * kX2Lanes, lo[i], p_cap);
      put(pw_col, poff, (M - k) * kX2Lanes, hi[i], p_cap);
    }
  }
}

// Mel projection over this warp's four chunk streams (see X2Tables). Lane
// (h, l), h = lane / 8, runs stream h for frames l, l + 16, l + 8 and l + 24,
// which one 16-byte load of a power-tile row gives (see split_x2): a chunk is
// two such loads, one weight broadcast {w0, w0, w1, w1} and four packed FMAs.
// The loop has no data-dependent bounds; it runs kX2Unroll chunks per
// iteration with all their loads in flight. A chunk that ends its filter
// stores the four sums (8 consecutive frames per quarter-warp per store) and
// restarts them.
template <typename OutT>
__device__ __forceinline__ void mel_project_x2(const unsigned char* s_pw, const int2* __restrict__ s_desc,
                                               const float4* __restrict__ s_w4, OutT* out_tile, int n_valid,
                                               long long n_frames, int c_begin, int c_end, int lane, int pw_bytes,
                                               int n_slots, long long out_left, unsigned* err) {
  const int l = lane & 7, h = lane >> 3;
  const unsigned char* pcol = s_pw + l * (int)sizeof(float4);
  const bool v0 = l < n_valid, v1 = l + 16 < n_valid, v2 = l + 8 < n_valid, v3 = l + 24 < n_valid;
  constexpr int kRow = kX2Lanes * (int)sizeof(float2);  // bytes per power-tile bin row
  float2 a01 = make_float2(0.0f, 0.0f), a23 = make_float2(0.0f, 0.0f);
  const int2* dp = s_desc + 4 * c_begin + h;
  const float4* wp = s_w4 + 4 * c_begin + h;
  for (int c = c_begin; c < c_end; c += kX2Unroll, dp += 4 * kX2Unroll, wp += 4 * kX2Unroll) {
    int2 d[kX2Unroll];
    float4 w[kX2Unroll], p0[kX2Unroll], p1[kX2Unroll];
#pragma unroll
    for (int u = 0; u < kX2Unroll; ++u)
      d[u] = FM_IN(c + u >= 0 && c + u < n_slots, err) ? dp[4 * u] : make_int2(0, -1);
#pragma unroll
    for (int u = 0; u < kX2Unroll; ++u) {
      w[u] = wp[4 * u];
      const bool in = FM_IN(d[u].x >= 0 && l * (int)sizeof(float4) + d[u].x + kRow + (int)sizeof(float4) <= pw_bytes,
                            err);
      p0[u] = in ? *reinterpret_cast<const float4*>(pcol + d[u].x) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      p1[u] = in ? *reinterpret_cast<const float4*>(pcol + d[u].x + kRow) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
#pragma unroll
    for (int u = 0; u < kX2Unroll; ++u) {
      const float2 w0 = make_float2(w[u].x, w[u].y), w1 = make_float2(w[u].z, w[u].w);
      a01 = fma2(w0, make_float2(p0[u].x, p0[u].y), a01);
      a23 = fma2(w0, make_float2(p0[u].z, p0[u].w), a23);
      a01 = fma2(w1, make_float2(p1[u].x, p1[u].y), a01);
      a23 = fma2(w1, make_float2(p1[u].z, p1[u].w), a23);
      if (d[u].y >= 0) {
        const long long oi = (long long)d[u].y * n_frames + l;  // element offset from out_tile
        OutT* o = out_tile + oi;
        if (v0 && FM_IN(oi < out_left, err)) store_out(o, a01.x);
        if (v1 && FM_IN(oi + 16 < out_left, err)) store_out(o + 16, a01.y);
        if (v2 && FM_IN(oi + 8 < out_left, err)) store_out(o + 8, a23.x);
        if (v3 && FM_IN(oi + 24 < out_left, err)) store_out(o + 24, a23.y);
        a01 = make_float2(0.0f, 0.0f);
        a23 = make_float2(0.0f, 0.0f);
      }
    }
  }
}

// Tile k of tile group g of this CTA (GR groups): groups take the grid's tile
// slots in turn, so group g runs tiles blockIdx.x + gridDim.x * (g + GR k).
template <int GR>
__device__ __forceinline__ long long x2_tile(int g, int k) {
  return (long long)blockIdx.x + (long long)gridDim.x * (g + (long long)GR * k);
}

// The tile that slot p processes. A signal's first and last tiles take
// padding and are the slowest to stage; the host may swap them (perm_edges)
// with interior tiles of the slots [perm_t0, perm_t0 + perm_edges), which it
// sets to the last group's first tiles: that group has the fewest tiles, so
// a late start costs it nothing, and no later round then waits behind an
// edge tile. Edge tile 2b is signal b's first, 2b + 1 its last.
__device__ __forceinline__ long long x2_logical(const KernelParams& prm, const TileSplitter& split, long long p) {
  if (prm.perm_edges == 0) return p;
  const long long i = p - prm.perm_t0;
  const long long tps = prm.tiles_per_signal;
  if (i >= 0 && i < prm.perm_edges) return (i >> 1) * tps + (i & 1) * (tps - 1);
  long long b;
  int tt;
  split(p, b, tt);
  if (tt == 0) return prm.perm_t0 + 2 * b;
  if (tt == tps - 1) return prm.perm_t0 + 2 * b + 1;
  return p;
}

// Geometry of the staged tile: lines of KH hops (two for a compile-time hop,
// else one), `rows` lines with a stride of S samples.
template <int N, int HOP, typename Raw>
struct X2Staging {
  static constexpr int KH = HOP > 0 ? 2 : 1;
  int hop, line, S, rows;
  __device__ explicit X2Staging(int runtime_hop) {
    hop = HOP > 0 ? HOP : runtime_hop;
    line = KH * hop;
    S = in_row_stride_x2(line, (int)sizeof(Raw));
    rows = x2_lines(N, hop, KH);
  }
};

// Lines [r0, r1) of a staged tile (line r starts at signal index
// gstart + r L) under the default framing, centre reflect padding with no
// `pad` zeros: sample s comes from -s before the signal, s inside it and
// 2 T - 2 - s in the cpad samples after it; positions from T + cpad on are
// left untouched (no valid frame reads them). One warp, 32-bit offsets within
// the lines, each sample by one 4-byte cp.async (f32 only).
template <typename Raw>
__device__ __forceinline__ void stage_lines_reflect(const Raw* __restrict__ sig, long long T, long long gstart,
                                                    int r0, int r1, int L, int S, int cpad, Raw* dst, int lane,
                                                    Cap cap) {
  static_assert(sizeof(Raw) == 4, "4-byte samples only");
  const long long base = gstart + (long long)r0 * L;
  const int n = (r1 - r0) * L;
  const auto clamp_n = [n](long long v) { return (int)(v < 0 ? 0 : (v > n ? n : v)); };
  const int a = clamp_n(-base);           // i < a: before the signal
  const int b = clamp_n(T - base);        // a <= i < b: inside it
  const int c = clamp_n(T + cpad - base);  // b <= i < c: mirrored after it
  for (int r = 0, i0 = 0; r < r1 - r0 && i0 < c; ++r, i0 += L) {
    Raw* d = dst + (r0 + r) * S;
    for (int col = lane; col < L && i0 + col < c; col += 32) {
      const int i = i0 + col;
      const long long src = i < a ? -(base + i) : (i < b ? base + i : 2 * T - 2 - (base + i));
      if (FM_IN((r0 + r) * S + col < cap.n && src >= 0 && src < T, cap.err)) cp_async<4>(d + col, sig + src);
    }
  }
}

// The producer warp: stages every tile of the CTA's groups into the group's
// staging area (the upper half of its exchange buffer). Lines that lie inside
// the signal arrive by TMA bulk copies, one line per lane, when the signal's
// lines start on 16-byte boundaries; their bytes are registered on the group's
// "staged" mbarrier. The other lines (the reflect-padded edges, or every line
// of an unaligned signal) are gathered by the warp's lanes with cp.async
// element copies, mirrored about the first / last sample; lines that start
// past the padded signal are skipped (no valid frame reads them). Every lane
// hands its element copies to the mbarrier (cp.async.mbarrier.arrive: a
// pending arrival that lands with them) and lane 0 then arrives, so the phase
// completes once both kinds of copies have landed while the warp already
// serves the next group. A group's next tile is staged once the group reports its
// staging area free (its "free" mbarrier, after pass 2 has read the exchange
// buffer); the warp serves whichever group is ready first. Waits are bounded:
// if no group frees its area for ~2^22 polls the warp records
// FM_ERR_KERNEL_TIMEOUT and stops staging (the waiting groups then time out).
template <int N, int GR, int HOP, typename Raw>
__device__ __forceinline__ void produce_x2(const KernelParams& prm, unsigned char* smem, const SmemLayoutX2& lay,
                                           int lane) {
  const X2Staging<N, HOP, Raw> st(prm.hop);
  const int esize = (int)sizeof(Raw);
  const Raw* in = static_cast<const Raw*>(prm.in);
  const long long T = prm.T;
  const TileSplitter split(prm.tiles_per_signal);
  const PadSpec pads = {prm.zpad, prm.cpad, prm.pad_mode};
  unsigned long long* full = reinterpret_cast<unsigned long long*>(smem + lay.bars);
  unsigned long long* empty = full + GR;
  // The tensor map's rows are lines of L samples starting at signal index
  // tmap_off, and lead + tmap_off is a multiple of L, so tile tt's first line
  // is tensor row tt * kX2Frames / KH - y_lead.
  const int y_lead = (prm.lead + prm.tmap_off) / st.line;
  // the default framing (centre reflect, no `pad` zeros) with f32 samples; its
  // edge tiles take stage_lines_reflect (16-bit samples keep stage_tile's
  // pairwise cp.async)
  const bool plain_reflect = sizeof(Raw) == 4 && prm.zpad == 0 && prm.pad_mode == FM_PAD_REFLECT;
  int2* slots = reinterpret_cast<int2*>(smem + lay.slots);
  const Cap in_cap = {(int)(lay.in_tile_bytes / sizeof(Raw)), prm.err};  // one group's staging area
  auto stage = [&](int g, long long tile, int k) {
    long long b;
    int tt;
    split(tile, b, tt);
    if (lane == 0) slots[2 * g + (k & 1)] = make_int2((int)b, tt);  // published by the arrival below
    const long long gstart = (long long)tt * kX2Frames * st.hop - prm.lead;
    const Raw* sig = in + b * T;
    Raw* dst = reinterpret_cast<Raw*>(smem + lay.in_tile + g * lay.group_stride);
    const int L = st.line, rows = st.rows;
    const long long span = (long long)rows * L;
    // lines [r_lo, r_hi) lie inside [0, T); lines from r_end on start past
    // the padded signal (T + zpad + cpad). Clamped to the tile's rows, every
    // count fits 32 bits, so no 64-bit division is needed.
    int r_lo = gstart >= 0 ? 0 : ((int)(-gstart) + L - 1) / L;  // -gstart <= lead
    const long long avail = T - gstart;
    int r_hi = avail >= span ? rows : (avail <= 0 ? 0 : (int)avail / L);
    const long long avail_p = T + prm.zpad + prm.cpad - gstart;
    const int r_end = avail_p >= span ? rows : (avail_p <= 0 ? 0 : ((int)avail_p + L - 1) / L);
    r_hi = r_hi < r_end ? r_hi : r_end;
    const bool tma_ok = ((L * esize) & 15) == 0 && (reinterpret_cast<uintptr_t>(sig + gstart) & 15) == 0;
    if (!tma_ok || r_lo >= r_hi) r_lo = r_hi = 0;
    // an interior tile whose rows all lie in the tensor map: one tensor copy
    const int y0 = tt * (kX2Frames / X2Staging<N, HOP, Raw>::KH) - y_lead;
    bool one_copy = prm.tmap_ok && y0 >= 0 && y0 + rows <= prm.tmap_rows && (smem_addr(dst) & 127u) == 0;
    // debug build: a copy that would not fit the staging area is not issued
    // (and its bytes are not expected), so the checks never leave a wait open
    if (one_copy && !FM_IN(st.rows * st.S <= in_cap.n, prm.err)) one_copy = false;
    if (r_hi > r_lo && !FM_IN((r_hi - 1) * st.S + L <= in_cap.n && gstart + (long long)r_lo * L >= 0 &&
                                  gstart + (long long)r_hi * L <= T,
                              prm.err))
      r_lo = r_hi = 0;
    int r_stop = r_end;
    if (one_copy) r_lo = r_hi = r_stop = 0;
    // the consumers' generic accesses of the area were ordered before this
    // warp by the "free" mbarrier; order them before the async-proxy writes
    if (lane == 0) {
      fence_proxy_async();
      if (one_copy) {
        mbar_expect_tx(full + g, (unsigned)(st.rows * st.S * esize));
        tma_load_3d(dst, &prm.tmap, 0, (int)y0, (int)b, full + g);
      } else if (r_hi > r_lo) {
        mbar_expect_tx(full + g, (unsigned)((r_hi - r_lo) * L * esize));
      }
    }
    __syncwarp();
    for (int r = r_lo + lane; r < r_hi; r += 32)
      tma_load_1d(dst + r * st.S, sig + gstart + (long long)r * L, (unsigned)(L * esize), full + g);
    const int r_tail = r_hi > r_lo ? r_hi : r_lo;
    // a tile that reaches past an edge of the signal mirrors its padding with
    // stage_lines_reflect; the others keep stage_tile's pairwise copies
    const bool mirror = plain_reflect && (gstart < 0 || avail < span);
    if constexpr (sizeof(Raw) == 4) {
      if (mirror) {
        if (r_lo > 0) stage_lines_reflect<Raw>(sig, T, gstart, 0, r_lo, L, st.S, prm.cpad, dst, lane, in_cap);
        if (r_stop > r_tail)
          stage_lines_reflect<Raw>(sig, T, gstart, r_tail, r_stop, L, st.S, prm.cpad, dst, lane, in_cap);
      }
    }
    if (!mirror) {
      if (r_lo > 0) stage_tile<Raw, 1>(sig, T, gstart, r_lo, L, st.S, dst, 0, lane, pads, in_cap);
      if (r_stop > r_tail)
        stage_tile<Raw, 1>(sig, T, gstart + (long long)r_tail * L, r_stop - r_tail, L, st.S, dst + r_tail * st.S,
                           0, lane, pads, Cap{in_cap.n - r_tail * st.S, in_cap.err});
    }
    // each lane's element copies arrive on the group's barrier when they land,
    // so the warp goes on to the next group instead of waiting for DRAM here
    cp_async_mbar_arrive(full + g);
    __syncwarp();  // every lane's pending arrival is registered before lane 0's
    if (lane == 0) mbar_arrive(full + g);
  };
  int next_k[GR];
  unsigned phase[GR];
#pragma unroll
  for (int g = 0; g < GR; ++g) {
    phase[g] = 0u;
    next_k[g] = 0;
    if (x2_tile<GR>(g, 0) < prm.total_tiles) {
      stage(g, x2_logical(prm, split, x2_tile<GR>(g, 0)), 0);
      next_k[g] = 1;
    }
  }
  for (int idle = 0;;) {
    int ready = -1;
    bool left = false;
#pragma unroll
    for (int g = 0; g < GR; ++g) {
      if (x2_tile<GR>(g, next_k[g]) >= prm.total_tiles) continue;
      left = true;
      if (ready < 0 && mbar_test_wait(empty + g, phase[g])) ready = g;
    }
    ready = __shfl_sync(0xffffffffu, ready, 0);
    if (!left) break;
    if (ready < 0) {
      if (!idle_backoff(idle, 1 << kIdleLog2Polls)) {
        if (lane == 0) atomicExch(prm.err, (unsigned)FM_ERR_KERNEL_TIMEOUT);
        break;
      }
      continue;
    }
    idle = 0;
    phase[ready] ^= 1u;
    stage(ready, x2_logical(prm, split, x2_tile<GR>(ready, next_k[ready])), next_k[ready]);
    ++next_k[ready];
  }
  cp_async_wait_all();  // no copy of this warp stays in flight past its exit
}

// The tile loop of one group (P x 16 threads on named barrier 1 + grp, its
// own exchange buffer and staging area). Per tile:
//   wait for the staged samples (every thread, on the group's mbarrier);
//   pass 1 in registers (loads, window, Q-point DFT, twiddles);
//   barrier: every staged sample has been read and the previous tile's mel
//            phase has finished reading the power tile;
//   pass-1 stores; barrier; pass 2 (loads, P-point DFTs); barrier: the
//   exchange buffer is free, so the producer may stage the next tile into
//   its upper half while the split writes the power tile into the lower half;
//   split and |X|^p; barrier; mel projection and stores.
// A warp that finishes its mel work early runs the next tile's pass 1 while
// the others finish theirs.
template <int N, int P, int Q, int GR, int HOP, typename Raw>
__device__ __forceinline__ void consume_x2(const KernelParams& prm, unsigned char* smem, const SmemLayoutX2& lay,
                                           int grp) {
  constexpr int M = N / 2;
  constexpr int THREADS = P * kX2Lanes;  // per group
  constexpr int GS4 = M + 1;  // float4 stride between frame pairs in the exchange buffer (odd)
  const float4* s_p1 = reinterpret_cast<const float4*>(smem + lay.p1);
  const float4* s_twh4 = reinterpret_cast<const float4*>(smem + lay.tw_half);
  const float4* s_twf4 = reinterpret_cast<const float4*>(smem + lay.tw_full);
  const int2* s_desc = reinterpret_cast<const int2*>(smem + lay.desc);
  const float4* s_w4 = reinterpret_cast<const float4*>(smem + lay.w4);
  unsigned char* s_x = smem + lay.xbuf + grp * lay.group_stride;
  float4* s_xq = reinterpret_cast<float4*>(s_x);
  const int bar_id = 1 + grp;
  unsigned long long* full = reinterpret_cast<unsigned long long*>(smem + lay.bars) + grp;
  unsigned long long* empty = full + GR;

  const int tid = threadIdx.x - grp * THREADS, warp = tid >> 5, lane = tid & 31;
  const int g = tid % kX2Lanes, role = tid / kX2Lanes;
  // Power tile, aliasing s_xq after pass 2: bin rows of 128 bytes; within a
  // row, 16 bytes per l < 8 hold frames {l, l + 16, l + 8, l + 24}, so thread
  // g writes its pair (g, g + 16) at float2 slot 2 (g % 8) + g / 8.
  const unsigned char* s_pw = s_x;
  float2* pw_col = reinterpret_cast<float2*>(s_x) + 2 * (g & 7) + (g >> 3);
  const X2Staging<N, HOP, Raw> st(prm.hop);
  const int s_begin = __ldg(&prm.x2->warp_begin[warp]), s_end = __ldg(&prm.x2->warp_begin[warp + 1]);
  const Raw* s_in = reinterpret_cast<const Raw*>(smem + lay.in_tile + grp * lay.group_stride);
  // frame g's first sample (HOP > 0: plus 2p, the role's first pair)
  const Raw* fbase = HOP > 0 ? s_in + (g >> 1) * st.S + (g & 1) * st.hop + 2 * role : s_in + g * st.S;
  const Raw* fbase_o = fbase + ((HOP > 0 && (g & 1)) ? st.S - st.line : 0);
  float4* xq_row = s_xq + g * GS4;
  const float4* tw = s_twh4 + role * Q;  // this role's W_M^{p k2}, k2 < Q
  unsigned phase = 0u;
  // buffer sizes for the debug build's index checks: the staging area, the
  // exchange buffer (float4), the power tile (float2 and bytes), the output
  const Cap in_cap = {(int)(lay.in_tile_bytes / sizeof(Raw)), prm.err};
  const Cap x_cap = {kX2Lanes * GS4, prm.err}, p_cap = {(M + 1) * kX2Lanes, prm.err};
  const int pw_off = 2 * (g & 7) + (g >> 3);
  const long long out_total = prm.B * (long long)prm.n_mels * prm.n_frames;

  for (int k = 0;; ++k) {
    const long long tile = x2_tile<GR>(grp, k);
    if (tile >= prm.total_tiles) break;
    const bool ok = mbar_wait_bounded(full, phase, prm.err);
    phase ^= 1u;

    cx2 z[Q];
    pass1_load_x2<P, Q, HOP, Raw>(fbase, fbase_o, st.S, s_p1, role, z, s_in, in_cap);
    dft<Q>(z);
#pragma unroll
    for (int k2 = 1; k2 < Q; ++k2) {
      const float4 w = tw[k2];
      z[k2] = cmul(z[k2], make_float2(w.x, w.y), make_float2(w.z, w.w));
    }
    // staged samples all read, previous power tile no longer needed
    if (group_sync_or(bar_id, THREADS, !ok)) return;  // staging never arrived (error recorded)
    // {re_a, re_b, im_a, im_b} per value, as two 8-byte stores of the register
    // pairs the packed math left them in (one 16-byte store would first copy
    // them into an aligned quad)
#pragma unroll
    for (int k2 = 0; k2 < Q; ++k2) {
      float2* dst = reinterpret_cast<float2*>(xq_row + k2 * P + role);
      if (FM_IN(g * GS4 + k2 * P + role < x_cap.n, prm.err)) {
        dst[0] = z[k2].re;
        dst[1] = z[k2].im;
      }
    }
    group_sync(bar_id, THREADS);

    // the staging area (upper half) is free for the next tile once the
    // exchange buffer has been read for the last time
    const auto freed = [&] {
      if (tid == 0) {
        fence_proxy_async();  // the group's generic accesses before the producer's TMA writes
        mbar_arrive(empty);
      }
    };
    if constexpr (Q == 2 * P) {
      cx2 za[P], zb[P];
      pass2_x2<P, Q>(xq_row, role, za, zb, g * GS4, x_cap);
      group_sync(bar_id, THREADS);  // exchange reads done
      freed();
      const bool merged = role < 2;  // the warp that holds role 0 (and role 1)
      switch (prm.power_mode) {
        case 0: split_x2<N, P, Q, 0>(za, zb, pw_col, s_twf4, role, prm.power, merged, pw_off, p_cap); break;
        case 1: split_x2<N, P, Q, 1>(za, zb, pw_col, s_twf4, role, prm.power, merged, pw_off, p_cap); break;
        default: split_x2<N, P, Q, 2>(za, zb, pw_col, s_twf4, role, prm.power, merged, pw_off, p_cap); break;
      }
    } else {
      switch (prm.power_mode) {
        case 0:
          pass2_split_exchange_x2<N, P, 0>(xq_row, pw_col, s_twf4, role, prm.power, g * GS4, x_cap, pw_off, p_cap,
                                           bar_id, THREADS, freed);
          break;
        case 1:
          pass2_split_exchange_x2<N, P, 1>(xq_row, pw_col, s_twf4, role, prm.power, g * GS4, x_cap, pw_off, p_cap,
                                           bar_id, THREADS, freed);
          break;
        default:
          pass2_split_exchange_x2<N, P, 2>(xq_row, pw_col, s_twf4, role, prm.power, g * GS4, x_cap, pw_off, p_cap,
                                           bar_id, THREADS, freed);
          break;
      }
    }
    group_sync(bar_id, THREADS);

    // the tile's place, as the producer staged it (slot k % 2 is rewritten
    // only for tile k + 2, after this group has freed its area twice more)
    const int2 bt = reinterpret_cast<const int2*>(smem + lay.slots)[2 * grp + (k & 1)];
    const long long b = bt.x;
    const int tt = bt.y;
    const int t0 = tt * kX2Frames;
    const int n_valid = min(kX2Frames, prm.n_frames - t0);
    const long long obase = b * prm.n_mels * (long long)prm.n_frames + t0;
    if (prm.out_dtype == FM_F32)
      mel_project_x2(s_pw, s_desc, s_w4, static_cast<float*>(prm.out) + obase, n_valid, prm.n_frames, s_begin,
                     s_end, lane, p_cap.n * (int)sizeof(float2), prm.x2_slots, out_total - obase, prm.err);
    else
      mel_project_x2(s_pw, s_desc, s_w4, static_cast<__half*>(prm.out) + obase, n_valid, prm.n_frames, s_begin,
                     s_end, lane, p_cap.n * (int)sizeof(float2), prm.x2_slots, out_total - obase, prm.err);
  }
}

// GR tile groups of P x 16 threads, each running its own tile loop on its own
// exchange buffer, and one producer warp that stages all their tiles; the
// tables are shared. As many CTAs per SM as fit (one at n_fft 256-512).
template <int N, int P, int Q, int GR, int HOP>
__global__ void __launch_bounds__(GR* P* kX2Lanes + 32 * kX2ProducerWarps, 1)
    mel_kernel_x2(const __grid_constant__ KernelParams prm) {
  constexpr int M = N / 2;
  constexpr int GROUP = P * kX2Lanes;
  constexpr int CONSUMERS = GR * GROUP;
  static_assert(P * Q == M && (Q == 2 * P || Q == P) && M <= kX2MaxM, "x2 kernel needs Q = 2P or P and M <= 256");
  static_assert(GR >= 1 && GR <= 14, "named barriers 1..GR + 1");
  static_assert(GROUP % 32 == 0, "a group must be whole warps");
  static_assert(kX2ProducerWarps == 1, "one producer warp");
  // (its own name: a translation unit that also holds the one-frame kernel
  // declares that kernel's dynamic shared array with 16-byte alignment)
  extern __shared__ __align__(128) unsigned char smem_x2[];
  unsigned char* const smem = smem_x2;
  const int esize = prm.in_dtype == FM_F32 ? 4 : 2;
  const SmemLayoutX2 lay = smem_layout_x2(N, prm.hop, HOP > 0 ? 2 : 1, prm.x2_slots, esize, GR);
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  if (tid == CONSUMERS) {
    unsigned long long* bars = reinterpret_cast<unsigned long long*>(smem + lay.bars);
    for (int i = 0; i < 2 * GR; ++i) mbar_init(bars + i, 1);
    fence_mbar_init();
  }
  // tables, fetched once per CTA by the consumer threads
  if (tid < CONSUMERS) {
    const X2Tables* t = prm.x2;
    copy_table_async(smem + lay.p1, t->p1, (int)sizeof(float4) * M, tid, CONSUMERS);
    copy_table_async(smem + lay.tw_half, t->tw_half, (int)sizeof(float4) * M, tid, CONSUMERS);
    copy_table_async(smem + lay.tw_full, t->tw_full, (int)sizeof(float4) * (M + 1), tid, CONSUMERS);
    copy_table_async(smem + lay.desc, t->desc, (int)sizeof(int2) * 4 * prm.x2_slots, tid, CONSUMERS);
    copy_table_async(smem + lay.w4, t->w4, (int)sizeof(float4) * 4 * prm.x2_slots, tid, CONSUMERS);
  }
  pdl_wait();       // caller buffers only after the previous kernel in the stream is done
  __syncthreads();  // the mbarriers exist before anyone uses them
  if (tid >= CONSUMERS) {
    if (prm.in_dtype == FM_F32) produce_x2<N, GR, HOP, float>(prm, smem, lay, tid & 31);
    else if (prm.in_dtype == FM_I16) produce_x2<N, GR, HOP, short>(prm, smem, lay, tid & 31);
    else produce_x2<N, GR, HOP, __half>(prm, smem, lay, tid & 31);
    return;
  }
  cp_async_wait_all();
  asm volatile("bar.sync %0, %1;" ::"r"(1 + GR), "r"(CONSUMERS) : "memory");  // tables visible
  // warp-uniform (a group is whole warps); reading it through a shuffle lets
  // the compiler keep the group's base addresses in uniform registers
  const int grp = __shfl_sync(0xffffffffu, tid / GROUP, 0);
  if (prm.in_dtype == FM_F32) consume_x2<N, P, Q, GR, HOP, float>(prm, smem, lay, grp);
  else if (prm.in_dtype == FM_I16) consume_x2<N, P, Q, GR, HOP, short>(prm, smem, lay, grp);
  else consume_x2<N, P, Q, GR, HOP, __half>(prm, smem, lay, grp);
}

}  // namespace fm

// Instantiate one two-frames-per-thread variant:
// FM_DEFINE_VARIANT_X2(name, N, P, Q, GR, HOP), GR tile groups per CTA, HOP = 0
// for any even hop
#define FM_DEFINE_VARIANT_X2(NAME, N, P, Q, GR, HOP)                                                    \
  namespace fm {                                                                                        \
  template __global__ void mel_kernel_x2<N, P, Q, GR, HOP>(const __grid_constant__ KernelParams);     \
  extern const Variant NAME = {N, P, Q, kX2Frames, GR * P * kX2Lanes + 32 * kX2ProducerWarps,          \
                               2, 1, (const void*)&mel_kernel_x2<N, P, Q, GR, HOP>, HOP, GR};           \
  }
