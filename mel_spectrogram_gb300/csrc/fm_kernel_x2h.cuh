// Lane-pair variant of the two-frame packed kernel (n_fft 400, compile-time
// hop; sm_103a). Same staging, tables, power tile and mel projection as
// fm_kernel_x2.cuh, but every DFT of the four-step split is shared by the two
// lanes g and g + 16 of a warp (half h = lane / 16), so a thread holds half
// the values and a group has twice the warps:
//   pass 1 : warp = role p. Half h takes z[p + P (2 i + h)], i < Q/2 (the
//            even or odd steps), does a Q/2-point DFT, and half 1 multiplies
//            output k by W_Q^k; the halves swap their outputs through one
//            shuffle per value and form X[k + (Q/2) h] = E[k] +- W_Q^k O[k]
//            (radix 2 by decimation in time), then the twiddle W_M^{p k2};
//   pass 2 : warp = t. Half 0 does the P-point DFT for k2 = t, half 1 for
//            k2 = Q - t (Q/2 for t = 0);
//   split  : the pairs (k, M - k) of warp t >= 1 have one member in each
//            half; each half takes P/2 of them and receives the other
//            member by shuffle. Warp 0's pairs lie inside each half.
#pragma once

#include "fm_kernel_x2.cuh"

namespace fm {

// the value of the partner lane (lane ^ 16): the other half of the pair
__device__ __forceinline__ cx2 shfl_half(cx2 v) {
  return {make_float2(__shfl_xor_sync(0xffffffffu, v.re.x, 16), __shfl_xor_sync(0xffffffffu, v.re.y, 16)),
          make_float2(__shfl_xor_sync(0xffffffffu, v.im.x, 16), __shfl_xor_sync(0xffffffffu, v.im.y, 16))};
}

// Pass 1 loads of one half: z[i] = the windowed pairs at n = p + P (2 i + h)
// of frames g and g + 16. base and base_o point at sample 2 (p + P h) of
// frame g (base_o: one line pad further, for odd g), tab at the role's window
// entry of step h; steps 2 i + h then sit 4 P i samples on, and with the hop
// a multiple of 4 P the line crossings do not depend on h.
template <int P, int Q, int HOP, typename Raw>
__device__ __forceinline__ void pass1_load_x2h(const Raw* __restrict__ base, const Raw* __restrict__ base_o,
                                               const float4* __restrict__ tab, cx2 (&z)[Q / 2], const Raw* s_in,
                                               Cap in_cap) {
  static_assert(HOP > 0 && HOP % (4 * P) == 0, "compile-time hop, a multiple of 4P");
  constexpr int SC = in_row_stride_x2_c(2 * HOP, (int)sizeof(Raw));
  constexpr int PAD = SC - 2 * HOP;
#pragma unroll
  for (int i = 0; i < Q / 2; ++i) {
    const float2 w = *reinterpret_cast<const float2*>(tab + 2 * i);
    const int j = 4 * P * i;
    const int ce = j / (2 * HOP), co = (HOP + j) / (2 * HOP);  // lines crossed, even / odd g
    const Raw* b = co != ce ? base_o : base;
    const int off = j + ce * PAD;
    const float2 va = staged_pair(b + off, s_in, in_cap);
    const float2 vb = staged_pair(b + off + (kX2Lanes / 2) * SC, s_in, in_cap);
    z[i].re = make_float2(va.x * w.x, vb.x * w.x);
    z[i].im = make_float2(va.y * w.y, vb.y * w.y);
  }
}

// The tile loop of one group (P warps, named barrier 1 + grp): as
// consume_x2, with the lane-pair passes above.
template <int N, int P, int Q, int GR, int HOP, int MODE, typename Raw>
__device__ __forceinline__ void consume_x2h(const KernelParams& prm, unsigned char* smem, const SmemLayoutX2& lay,
                                            int grp) {
  constexpr int M = N / 2, H = Q / 2;
  constexpr int THREADS = P * 32;  // per group: warp = role, lane = g + 16 h
  constexpr int GS4 = M + 1;
  static_assert(Q == 2 * P && P % 2 == 0, "lane pairs split Q = 2P");
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
  const int g = lane & 15, h = lane >> 4, role = warp;
  const unsigned char* s_pw = s_x;
  float2* pw_col = reinterpret_cast<float2*>(s_x) + 2 * (g & 7) + (g >> 3);
  const X2Staging<N, HOP, Raw> st(prm.hop);
  const int s_begin = __ldg(&prm.x2->warp_begin[warp]), s_end = __ldg(&prm.x2->warp_begin[warp + 1]);
  const Raw* s_in = reinterpret_cast<const Raw*>(smem + lay.in_tile + grp * lay.group_stride);
  const Raw* fbase = s_in + (g >> 1) * st.S + (g & 1) * st.hop + 2 * (role + P * h);
  const Raw* fbase_o = fbase + ((g & 1) ? st.S - st.line : 0);
  float4* xq_row = s_xq + g * GS4;
  const float4* tw = s_twh4 + role * Q + H * h;  // W_M^{p k2}, k2 = k + H h
  const float4* tab = s_p1 + role * Q + h;        // window entries of steps 2 i + h
  const float2 sgn = h ? make_float2(-1.0f, -1.0f) : make_float2(1.0f, 1.0f);
  // pass 2: this half's k2, and the split's partner pairs
  const int t = role;
  const int k2p = h ? (t == 0 ? Q / 2 : Q - t) : t;
  unsigned phase = 0u;
  const Cap in_cap = {(int)(lay.in_tile_bytes / sizeof(Raw)), prm.err};
  const Cap x_cap = {kX2Lanes * GS4, prm.err}, p_cap = {(M + 1) * kX2Lanes, prm.err};
  const int pw_off = 2 * (g & 7) + (g >> 3);
  const long long out_total = prm.B * (long long)prm.n_mels * prm.n_frames;

  for (int k = 0;; ++k) {
    const long long tile = x2_tile<GR>(grp, k);
    if (tile >= prm.total_tiles) break;
    const bool ok = mbar_wait_bounded(full, phase, prm.err);
    phase ^= 1u;

    cx2 z[H];
    pass1_load_x2h<P, Q, HOP, Raw>(fbase, fbase_o, tab, z, s_in, in_cap);
    dft<H>(z);  // E[k] (h = 0) or O[k] (h = 1)
#pragma unroll
    for (int j = 1; j < H; ++j) {  // O[k] W_Q^k = O[k] W_N^{(N/Q) k}; half 0 multiplies by 1
      const float4 w = h ? s_twf4[(N / Q) * j] : make_float4(1.0f, 1.0f, 0.0f, 0.0f);
      z[j] = cmul(z[j], make_float2(w.x, w.y), make_float2(w.z, w.w));
    }
#pragma unroll
    for (int j = 0; j < H; ++j) {  // X[j + H h] = partner +- mine
      const cx2 o = shfl_half(z[j]);
      z[j] = {fma2(z[j].re, sgn, o.re), fma2(z[j].im, sgn, o.im)};
      const float4 w = tw[j];
      z[j] = cmul(z[j], make_float2(w.x, w.y), make_float2(w.z, w.w));
    }
    if (group_sync_or(bar_id, THREADS, !ok)) return;  // staged samples read, previous power tile done
#pragma unroll
    for (int j = 0; j < H; ++j) {
      float2* dst = reinterpret_cast<float2*>(xq_row + (j + H * h) * P + role);
      if (FM_IN(g * GS4 + (j + H * h) * P + role < x_cap.n, prm.err)) {
        dst[0] = z[j].re;
        dst[1] = z[j].im;
      }
    }
    group_sync(bar_id, THREADS);

    cx2 y[P];
#pragma unroll
    for (int p = 0; p < P; ++p) {
      const float4 v = get(xq_row, g * GS4, k2p * P + p, x_cap);
      y[p] = {make_float2(v.x, v.y), make_float2(v.z, v.w)};
    }
    dft<P>(y);  // y[k1] = Z[k2p + Q k1]
    group_sync(bar_id, THREADS);  // exchange reads done: the staging area is free
    if (tid == 0) {
      fence_proxy_async();
      mbar_arrive(empty);
    }
    if (t != 0) {
      // half 0 holds a[k1] = Z[t + Q k1], half 1 b[k1] = Z[Q - t + Q k1];
      // a[k1] pairs with b[P - 1 - k1] at k = t + Q k1; half h takes
      // k1 = j + (P/2) h
#pragma unroll
      for (int j = 0; j < P / 2; ++j) {
        const cx2 send = h ? y[P - 1 - j] : y[P / 2 + j];
        const cx2 recv = shfl_half(send);
        const cx2 zk = h ? recv : y[j];
        const cx2 zm = h ? y[P / 2 - 1 - j] : recv;
        const int kk = t + Q * (j + (P / 2) * h);
        float2 lo, hi;
        split_pair_x2<MODE>(zk, zm, s_twf4[kk], prm.power, lo, hi);
        put(pw_col, pw_off, kk * kX2Lanes, lo, p_cap);
        put(pw_col, pw_off, (M - kk) * kX2Lanes, hi, p_cap);
      }
    } else {
      // half 0: pairs (a[j], a[(P - j) % P]) at k = Q j, j <= P/2 (j = 0:
      // X[0] and X[M]); half 1: (b[j], b[P - 1 - j]) at k = Q/2 + Q j, j < P/2
#pragma unroll
      for (int j = 0; j <= P / 2; ++j) {
        if (j < P / 2 || h == 0) {
          const cx2 zm = h ? y[(P - 1 - j) % P] : y[(P - j) % P];
          const int kk = h ? Q / 2 + Q * j : Q * j;
          float2 lo, hi;
          split_pair_x2<MODE>(y[j], zm, s_twf4[kk], prm.power, lo, hi);
          put(pw_col, pw_off, kk * kX2Lanes, lo, p_cap);
          put(pw_col, pw_off, (M - kk) * kX2Lanes, hi, p_cap);
        }
      }
    }
    group_sync(bar_id, THREADS);

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

template <int N, int P, int Q, int GR, int HOP, typename Raw>
__device__ __forceinline__ void consume_x2h_mode(const KernelParams& prm, unsigned char* smem,
                                                 const SmemLayoutX2& lay, int grp) {
  switch (prm.power_mode) {
    case 0: consume_x2h<N, P, Q, GR, HOP, 0, Raw>(prm, smem, lay, grp); break;
    case 1: consume_x2h<N, P, Q, GR, HOP, 1, Raw>(prm, smem, lay, grp); break;
    default: consume_x2h<N, P, Q, GR, HOP, 2, Raw>(prm, smem, lay, grp); break;
  }
}

// GR groups of P warps and one producer warp per CTA, one CTA per SM.
template <int N, int P, int Q, int GR, int HOP>
__global__ void __launch_bounds__(GR* P * 32 + 32 * kX2ProducerWarps, 1)
    mel_kernel_x2h(const __grid_constant__ KernelParams prm) {
  constexpr int M = N / 2;
  constexpr int CONSUMERS = GR * P * 32;
  static_assert(P * Q == M && Q == 2 * P && M <= kX2MaxM && GR >= 1 && GR <= 14, "lane-pair split");
  extern __shared__ __align__(128) unsigned char smem_x2h[];
  unsigned char* const smem = smem_x2h;
  const int esize = prm.in_dtype == FM_F32 ? 4 : 2;
  const SmemLayoutX2 lay = smem_layout_x2(N, prm.hop, 2, prm.x2_slots, esize, GR);
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  if (tid == CONSUMERS) {
    unsigned long long* bars = reinterpret_cast<unsigned long long*>(smem + lay.bars);
    for (int i = 0; i < 2 * GR; ++i) mbar_init(bars + i, 1);
    fence_mbar_init();
  }
  if (tid < CONSUMERS) {
    const X2Tables* t = prm.x2;
    copy_table_async(smem + lay.p1, t->p1, (int)sizeof(float4) * M, tid, CONSUMERS);
    copy_table_async(smem + lay.tw_half, t->tw_half, (int)sizeof(float4) * M, tid, CONSUMERS);
    copy_table_async(smem + lay.tw_full, t->tw_full, (int)sizeof(float4) * (M + 1), tid, CONSUMERS);
    copy_table_async(smem + lay.desc, t->desc, (int)sizeof(int2) * 4 * prm.x2_slots, tid, CONSUMERS);
    copy_table_async(smem + lay.w4, t->w4, (int)sizeof(float4) * 4 * prm.x2_slots, tid, CONSUMERS);
  }
  pdl_wait();
  __syncthreads();
  if (tid >= CONSUMERS) {
    if (prm.in_dtype == FM_F32) produce_x2<N, GR, HOP, float>(prm, smem, lay, tid & 31);
    else if (prm.in_dtype == FM_I16) produce_x2<N, GR, HOP, short>(prm, smem, lay, tid & 31);
    else produce_x2<N, GR, HOP, __half>(prm, smem, lay, tid & 31);
    return;
  }
  cp_async_wait_all();
  asm volatile("bar.sync %0, %1;" ::"r"(1 + GR), "r"(CONSUMERS) : "memory");
  const int grp = __shfl_sync(0xffffffffu, tid / (P * 32), 0);
  if (prm.in_dtype == FM_F32) consume_x2h_mode<N, P, Q, GR, HOP, float>(prm, smem, lay, grp);
  else if (prm.in_dtype == FM_I16) consume_x2h_mode<N, P, Q, GR, HOP, short>(prm, smem, lay, grp);
  else consume_x2h_mode<N, P, Q, GR, HOP, __half>(prm, smem, lay, grp);
}

}  // namespace fm

// FM_DEFINE_VARIANT_X2H(name, N, P, Q, GR, HOP): HOP a compile-time multiple of 4P
#define FM_DEFINE_VARIANT_X2H(NAME, N, P, Q, GR, HOP)                                                   \
  namespace fm {                                                                                       \
  template __global__ void mel_kernel_x2h<N, P, Q, GR, HOP>(const __grid_constant__ KernelParams);    \
  extern const Variant NAME = {N, P, Q, kX2Frames, GR * P * 32 + 32 * kX2ProducerWarps,               \
                               2, 1, (const void*)&mel_kernel_x2h<N, P, Q, GR, HOP>, HOP, GR};         \
  }
