// Batched lossless speculative-decoding verify step for sm_103a.
//
// Rule ([SD §2.1-§2.2] "Speculative decoding, the founding scheme";
// [SSD §2.4, §4.3] "Self-speculative decoding with layer skip and KV reuse";
// [FS §2.3, §3.2, §5.4] "FlashSpec speculative decoding in practice"):
// position i of a sequence is accepted iff u_i < p_i(x_i)/q_i(x_i); the first
// rejection j draws from norm(max(0, p_j - q_j)); if all k are accepted the
// bonus is drawn from p_k; greedy rows compare the draft with the target
// argmax instead.
//
// Work decomposition.  One "item" is a (sequence b, position i) pair: the
// target row i and, for i < k_b on a sampled row, the draft row i.  An item
// runs on a thread-block cluster of C CTAs; CTA r owns the vocabulary slice
// [r*L, (r+1)*L) of both rows and streams it through a 3-stage ring in shared
// memory fed by the bulk-copy engine (one mbarrier per stage).  Each row is
// reduced in ONE pass: the running max, and the sum of 2^(z*c - R) where the
// reference exponent R is an integer that only grows; when it grows the
// partial sum is rescaled by an exact power of two, so the online pass adds
// no rounding beyond the exponentials themselves.  The cluster combines the
// per-slice results through distributed shared memory.
//
// Items are launched position-major (all sequences' position 0 first).  Each
// item publishes {done, rejected, error} bits for its position in one 64-bit
// word per sequence.  An item that starts after an earlier position of its
// sequence has been rejected exits without reading its rows: those rows
// cannot change the result.  The item whose publication completes the
// prefix 0..j (j = first rejection, or k_b when all were accepted) is the
// sequence's finisher: it streams row(s) j again (usually still in L2) to
// sum the residual max(0, p - q) (or p for the bonus) per chunk, then reads
// back the one chunk that holds the inverse-CDF point.  No item ever waits
// for another one.
#include <cstdint>
#include <cstdio>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kCmax = 16;
constexpr int kChunkUnits = 256;                   // 16-byte units of one row per chunk
constexpr int kHalfBytes = kChunkUnits * 16;       // 4 KB of one row
constexpr int kStageBytes = 2 * kHalfBytes;        // target half + draft half
constexpr int kStages = 3;
constexpr int kMaxChunks = 32;                     // slice <= 128 KB of a row per CTA
constexpr int kUnitsPerThread = kChunkUnits / kThreads;
constexpr int kWordBits = 21;                      // positions per field of the sequence word

struct ItemStats {
  float m_t, R_t, st_hi, st_lo;
  float m_d, R_d, sd_hi, sd_lo;
  int argmax;
  uint32_t errbits;
};

struct VerifyParams {
  const char* tgt;
  long long t_seq, t_pos;  // bytes
  const char* drf;
  long long d_seq, d_pos;  // bytes
  int B, K, V;
  const int32_t* tokens;
  const int32_t* kpr;
  const float* temp;
  float top_p;
  const float* unif;
  const uint8_t* mode;
  int32_t* out;
  int32_t* nacc;
  float* diag;
  uint32_t* flags;
  unsigned long long* words;
  ItemStats* stats;
  int slice_len;  // elements per CTA slice
};

// ---------------------------------------------------------------------------
// One CTA's slice [e0, e1) of one logit row, in 16-byte units: unit u holds
// global bytes [base16 + 16u, base16 + 16u + 16).  Units inside the aligned
// body [a0, a1) are fully valid and arrive by bulk copy; the (at most two)
// partial units at the ends are read element by element from global memory.
// ---------------------------------------------------------------------------
template <int ES>
struct RowSlice {
  const char* row;
  int e0, e1;
  uintptr_t base16, a0, a1;
  int n_units, ebase0, n_chunks;

  __device__ void init(const char* row_, int e0_, int e1_) {
    row = row_;
    e0 = e0_;
    e1 = e1_;
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(row) + (uintptr_t)e0 * ES;
    const uintptr_t g1 = reinterpret_cast<uintptr_t>(row) + (uintptr_t)e1 * ES;
    base16 = g0 & ~uintptr_t(15);
    a0 = (g0 + 15) & ~uintptr_t(15);
    a1 = g1 & ~uintptr_t(15);
    if (a1 < a0) a1 = a0;
    n_units = e1 > e0 ? (int)((g1 - base16 + 15) / 16) : 0;
    ebase0 = e0 - (int)((g0 & 15) / ES);
    n_chunks = (n_units + kChunkUnits - 1) / kChunkUnits;
  }
  __device__ __forceinline__ bool unit_bulk(int u) const {
    const uintptr_t a = base16 + 16 * (uintptr_t)u;
    return a >= a0 && a + 16 <= a1;
  }
    // units [ub0, ub1) are fully inside the aligned body
  __device__ __forceinline__ int ub0() const { return (int)((a0 - base16) / 16); }
  __device__ __forceinline__ int ub1() const { return (int)((a1 - base16) / 16); }
  // bulk-copied byte range of chunk c
  __device__ __forceinline__ void chunk_body(int c, uintptr_t* lo, uintptr_t* hi) const {
    const uintptr_t c0 = base16 + (uintptr_t)c * kHalfBytes, c1 = c0 + kHalfBytes;
    *lo = c0 > a0 ? c0 : a0;
    *hi = c1 < a1 ? c1 : a1;
    if (*hi < *lo) *hi = *lo;
  }
  __device__ __forceinline__ float elem(int e) const {  // from global memory
    return ES == 2 ? bf16_lo(*reinterpret_cast<const uint16_t*>(row + (size_t)e * 2))
                   : *reinterpret_cast<const float*>(row + (size_t)e * 4);
  }
};

template <int ES>
__device__ __forceinline__ float unit_elem(const uint4& v, int j) {
  if (ES == 4) {
    uint32_t w = j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
    return __uint_as_float(w);
  } else {
    uint32_t w = (j >> 1) == 0 ? v.x : (j >> 1) == 1 ? v.y : (j >> 1) == 2 ? v.z : v.w;
    return (j & 1) ? bf16_hi(w) : bf16_lo(w);
  }
}

// max that propagates NaN (one instruction)
__device__ __forceinline__ float nanmax(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// "no finite element yet" value of the reference exponent R: finite, so that
// z*c - R stays -inf (never NaN) for z = -inf, and far below any real R.
constexpr float kRnone = -3.0e38f;

// max of a full unit, NaN-propagating
template <int ES>
__device__ __forceinline__ float unit_max(const uint4& v) {
  if (ES == 2) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
    __nv_bfloat162 m2 = __hmax2_nan(__hmax2_nan(p[0], p[1]), __hmax2_nan(p[2], p[3]));
    return nanmax(__low2float(m2), __high2float(m2));
  } else {
    float a = __uint_as_float(v.x), b = __uint_as_float(v.y), c = __uint_as_float(v.z),
          d = __uint_as_float(v.w);
    return nanmax(nanmax(a, b), nanmax(c, d));
  }
}

// c = log2(e)/T as chi + clo with chi <= c (so clo > 0), from float operations
// only: q1 = hi/T, then the quotient of the exact remainder.  exp((z - m)/T)
// is then 2^(z*chi + z*clo - m*c), and no rounded reciprocal of T enters it.
constexpr float kLog2eHi = 1.44269502162933349609375f;
constexpr float kLog2eLo = 1.925963033500011079e-08f;

struct Expo {
  float chi, clo;
};

__device__ __forceinline__ Expo make_expo(float T) {
  const float q1 = __fdiv_rn(kLog2eHi, T);
  const float r = __fadd_rn(__fmaf_rn(-q1, T, kLog2eHi), kLog2eLo);
  const float q2 = __fdiv_rn(r, T);
  float hi = __fadd_rn(q1, q2);
  float lo = __fsub_rn(q2, __fsub_rn(hi, q1));
  if (lo < 0.f) {  // step hi one ulp down so that lo is positive
    const float h2 = __int_as_float(__float_as_int(hi) - 1);
    lo = __fadd_rn(lo, __fsub_rn(hi, h2));
    hi = h2;
  }
  if (!(lo > 0.f)) lo = 1e-30f;  // keeps -inf * lo = -inf (never NaN)
  return Expo{hi, lo};
}

// base-2 exponent of element z against reference R: z*c - R, one rounding
// for the large part (FMA), the small correction z*clo added after.
__device__ __forceinline__ float earg(float z, const Expo& x, float R) {
  return __fmaf_rn(z, x.clo, __fmaf_rn(z, x.chi, -R));
}

// 2^k for an integer-valued k <= 0; 0 below 2^-126.
__device__ __forceinline__ float pow2i(float k) {
  if (!(k >= -126.f)) return 0.f;
  return __int_as_float((127 + (int)k) << 23);
}

// ---------------------------------------------------------------------------
// Per-thread row accumulator
// ---------------------------------------------------------------------------
struct RowAcc {
  float mx;  // running max of the raw logits (NaN propagates)
  float R;   // integer reference exponent, kRnone until a finite element
  DF s;      // sum of 2^(z*c - R)
  int amax;  // index of the first maximum (greedy rows)
};

__device__ __forceinline__ RowAcc acc_init() {
  return RowAcc{-INFINITY, kRnone, DF{0.f, 0.f}, 0x7fffffff};
}

__device__ __forceinline__ void acc_raise(RowAcc& a, float Rn) {
  const float p = pow2i(a.R - Rn);  // exact power of two (0 from kRnone)
  a.s.hi *= p;
  a.s.lo *= p;
  a.R = Rn;
}

__device__ __forceinline__ float e2(float z, const Expo& x, float nR) {
  return ex2(__fmaf_rn(z, x.clo, __fmaf_rn(z, x.chi, nR)));
}

// 2^(z*c - R) for a pair of logits held as an f32x2 (same arithmetic as e2)
__device__ __forceinline__ F2 e2x2(F2 z, F2 C, F2 L, F2 N) {
  float p, q;
  f2_unpack(f2_fma(z, L, f2_fma(z, C, N)), p, q);
  return f2_pack(ex2(p), ex2(q));
}

__device__ __forceinline__ F2 bf16x2_to_f2(uint32_t w) { return f2_pack(bf16_lo(w), bf16_hi(w)); }

template <int ES>
__device__ __forceinline__ void sampled_unit(RowAcc& a, const uint4& v, const Expo& x) {
  const float g = unit_max<ES>(v);
  a.mx = nanmax(a.mx, g);
  const float gc = g * x.chi;
  if (gc > a.R) acc_raise(a, ceilf(gc));
  const F2 C = f2_pack(x.chi, x.chi), L = f2_pack(x.clo, x.clo);
  const F2 N = f2_pack(-a.R, -a.R);
  F2 s;
  if (ES == 2) {
    const F2 e0 = e2x2(bf16x2_to_f2(v.x), C, L, N), e1 = e2x2(bf16x2_to_f2(v.y), C, L, N);
    const F2 e2_ = e2x2(bf16x2_to_f2(v.z), C, L, N), e3 = e2x2(bf16x2_to_f2(v.w), C, L, N);
    s = f2_add(f2_add(e0, e1), f2_add(e2_, e3));
  } else {
    const F2 e0 = e2x2(f2_pack(__uint_as_float(v.x), __uint_as_float(v.y)), C, L, N);
    const F2 e1 = e2x2(f2_pack(__uint_as_float(v.z), __uint_as_float(v.w)), C, L, N);
    s = f2_add(e0, e1);
  }
  float sx, sy;
  f2_unpack(s, sx, sy);
  df_acc(a.s, sx + sy);
}

__device__ __forceinline__ void sampled_elem(RowAcc& a, float z, const Expo& x) {
  a.mx = nanmax(a.mx, z);
  const float zc = z * x.chi;
  if (zc > a.R) acc_raise(a, ceilf(zc));
  df_acc(a.s, e2(z, x, -a.R));
}

template <int ES>
__device__ __forceinline__ void greedy_unit(RowAcc& a, const uint4& v, int eb) {
  constexpr int EPU = 16 / ES;
  const float g = unit_max<ES>(v);
  if (g != g) {
    a.mx = g;
  } else if (g > a.mx) {  // strict: the first occurrence in index order stays
    int first = EPU - 1;
#pragma unroll
    for (int j = EPU - 1; j >= 0; --j)
      if (unit_elem<ES>(v, j) == g) first = j;
    a.mx = g;
    a.amax = eb + first;
  }
}

__device__ __forceinline__ void greedy_elem(RowAcc& a, float z, int e) {
  if (z != z) {
    a.mx = z;
  } else if (z > a.mx) {
    a.mx = z;
    a.amax = e;
  }
}

template <int ES>
__device__ __forceinline__ void row_unit(RowAcc& a, const RowSlice<ES>& rs, const char* half, int c,
                                         int u, int ub0, int ub1, bool greedy, const Expo& x) {
  constexpr int EPU = 16 / ES;
  const int eb = rs.ebase0 + u * EPU;
  if (u >= ub0 && u < ub1) {
    const uint4 v = *reinterpret_cast<const uint4*>(half + 16 * (u - c * kChunkUnits));
    if (greedy)
      greedy_unit<ES>(a, v, eb);
    else
      sampled_unit<ES>(a, v, x);
  } else if (u < rs.n_units) {
    for (int j = 0; j < EPU; ++j) {
      const int e = eb + j;
      if (e < rs.e0 || e >= rs.e1) continue;
      const float z = rs.elem(e);
      if (greedy)
        greedy_elem(a, z, e);
      else
        sampled_elem(a, z, x);
    }
  }
}

// Combine row accumulators over the lanes of a warp (lanes with valid ==
// false contribute nothing).  The butterfly leaves the same bits on every
// lane, so every CTA that combines the same values gets the same result.
__device__ __forceinline__ float warp_maxf(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_nanmax(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = nanmax(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ RowAcc lanes_combine(RowAcc v, bool valid, bool greedy) {
  if (!valid) v = acc_init();
  const float m = warp_nanmax(v.mx);
  if (greedy) {
    const int cand = (v.mx == m) ? v.amax : 0x7fffffff;
    return RowAcc{m, -INFINITY, DF{0.f, 0.f}, warp_min(cand)};
  }
  const float Rw = warp_maxf(v.R);
  DF s = DF{0.f, 0.f};
  if (v.R > kRnone && Rw > kRnone) {
    const float p = pow2i(v.R - Rw);
    s = DF{v.s.hi * p, v.s.lo * p};
  }
  s = df_warp_sum(s);
  return RowAcc{m, Rw, s, 0x7fffffff};
}

__device__ __forceinline__ DF df_shfl(DF v, int src) {
  return DF{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

// Inclusive prefix over lanes in double-float.
__device__ __forceinline__ DF df_warp_scan(DF v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    DF n = DF{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
    if (lane >= o) v = df_add(v, n);
  }
  return v;
}

// ---------------------------------------------------------------------------
// Residual / bonus weights: w = max(0, e_t - rho * e_d) with e = 2^(z*c - R)
// and rho = S_t / S_d (hi + lo), or e_t alone ("p only": the bonus, or the
// all-zero residual fallback).  w / S_t = max(0, p - q).
// ---------------------------------------------------------------------------
struct Weight {
  Expo x;
  float Rt, Rd, rho_hi, rho_lo;
  bool p_only;
  __device__ __forceinline__ float operator()(float zt, float zd) const {
    const float a = e2(zt, x, -Rt);
    if (p_only) return a;
    const float b = e2(zd, x, -Rd);
    return fmaxf(0.f, __fmaf_rn(-rho_lo, b, __fmaf_rn(-rho_hi, b, a)));
  }
  __device__ __forceinline__ float pair(float zt, float zd) const {
    const float a = e2(zt, x, -Rt), b = e2(zd, x, -Rd);
    return fmaxf(0.f, __fmaf_rn(-rho_lo, b, __fmaf_rn(-rho_hi, b, a)));
  }
  // two elements at once (f32x2), lane by lane the same arithmetic as pair()
  __device__ __forceinline__ float pair2(F2 zt, F2 zd, F2 C, F2 L, F2 Nt, F2 Nd, F2 RH,
                                         F2 RL) const {
    const F2 a = e2x2(zt, C, L, Nt), b = e2x2(zd, C, L, Nd);
    float w0, w1;
    f2_unpack(f2_fma(RL, b, f2_fma(RH, b, a)), w0, w1);
    return fmaxf(0.f, w0) + fmaxf(0.f, w1);
  }
};

// Sum of the weights of unit u (target units), with the draft read from its
// own half when both rows share the 16-byte phase, else element-wise.
template <int ES>
__device__ __forceinline__ float unit_wsum(const RowSlice<ES>& st, const RowSlice<ES>& sd,
                                           const char* ht, const char* hd, int c, int u,
                                           const Weight& W, bool same_phase) {
  constexpr int EPU = 16 / ES;
  if (u >= st.n_units) return 0.f;
  const int eb = st.ebase0 + u * EPU;
  if (st.unit_bulk(u) && (W.p_only || same_phase)) {
    const int off = 16 * (u - c * kChunkUnits);
    const uint4 vt = *reinterpret_cast<const uint4*>(ht + off);
    if (W.p_only) {
      const float nR = -W.Rt;
      if (ES == 2) {
        const float e0 = e2(bf16_lo(vt.x), W.x, nR), e1 = e2(bf16_hi(vt.x), W.x, nR);
        const float f0 = e2(bf16_lo(vt.y), W.x, nR), f1 = e2(bf16_hi(vt.y), W.x, nR);
        const float g0 = e2(bf16_lo(vt.z), W.x, nR), g1 = e2(bf16_hi(vt.z), W.x, nR);
        const float h0 = e2(bf16_lo(vt.w), W.x, nR), h1 = e2(bf16_hi(vt.w), W.x, nR);
        return ((e0 + e1) + (f0 + f1)) + ((g0 + g1) + (h0 + h1));
      }
      const float e0 = e2(__uint_as_float(vt.x), W.x, nR), e1 = e2(__uint_as_float(vt.y), W.x, nR);
      const float f0 = e2(__uint_as_float(vt.z), W.x, nR), f1 = e2(__uint_as_float(vt.w), W.x, nR);
      return (e0 + e1) + (f0 + f1);
    }
    const uint4 vd = *reinterpret_cast<const uint4*>(hd + off);
    const F2 C = f2_pack(W.x.chi, W.x.chi), L = f2_pack(W.x.clo, W.x.clo);
    const F2 Nt = f2_pack(-W.Rt, -W.Rt), Nd = f2_pack(-W.Rd, -W.Rd);
    const F2 RH = f2_pack(-W.rho_hi, -W.rho_hi), RL = f2_pack(-W.rho_lo, -W.rho_lo);
    if (ES == 2) {
      const float e = W.pair2(bf16x2_to_f2(vt.x), bf16x2_to_f2(vd.x), C, L, Nt, Nd, RH, RL);
      const float f = W.pair2(bf16x2_to_f2(vt.y), bf16x2_to_f2(vd.y), C, L, Nt, Nd, RH, RL);
      const float g = W.pair2(bf16x2_to_f2(vt.z), bf16x2_to_f2(vd.z), C, L, Nt, Nd, RH, RL);
      const float h = W.pair2(bf16x2_to_f2(vt.w), bf16x2_to_f2(vd.w), C, L, Nt, Nd, RH, RL);
      return (e + f) + (g + h);
    }
    const float e = W.pair2(f2_pack(__uint_as_float(vt.x), __uint_as_float(vt.y)),
                            f2_pack(__uint_as_float(vd.x), __uint_as_float(vd.y)), C, L, Nt, Nd, RH, RL);
    const float f = W.pair2(f2_pack(__uint_as_float(vt.z), __uint_as_float(vt.w)),
                            f2_pack(__uint_as_float(vd.z), __uint_as_float(vd.w)), C, L, Nt, Nd, RH, RL);
    return e + f;
  }
  float acc = 0.f;
  for (int j = 0; j < EPU; ++j) {
    const int e = eb + j;
    if (e < st.e0 || e >= st.e1) continue;
    acc += W(st.elem(e), W.p_only ? 0.f : sd.elem(e));
  }
  return acc;
}

// weight of element e of unit u (same reads as unit_wsum)
template <int ES>
__device__ __forceinline__ float elem_w(const RowSlice<ES>& st, const RowSlice<ES>& sd,
                                        const char* ht, const char* hd, int c, int u, int e,
                                        const Weight& W, bool same_phase) {
  constexpr int EPU = 16 / ES;
  if (st.unit_bulk(u) && (W.p_only || same_phase)) {
    const int off = 16 * (u - c * kChunkUnits);
    const uint4 vt = *reinterpret_cast<const uint4*>(ht + off);
    const uint4 vd = W.p_only ? vt : *reinterpret_cast<const uint4*>(hd + off);
    const int j = e - (st.ebase0 + u * EPU);
    return W(unit_elem<ES>(vt, j), unit_elem<ES>(vd, j));
  }
  return W(st.elem(e), W.p_only ? 0.f : sd.elem(e));
}

struct Shared {
  uint64_t full[kStages];
  // all-gather slots, indexed by the writing CTA's rank
  RowAcc g_t[kCmax], g_d[kCmax];
  DF g_w[kCmax];
  // per-warp partials
  RowAcc r_t[kWarps], r_d[kWarps];
  DF tw[kMaxChunks][kWarps];
  DF scan[2][kWarps];
  int r_i[kWarps];
  // item scalars, written by warp 0 and read by the whole CTA
  RowAcc row_t, row_d;
  DF S_w;
  int skip, skip_seen;
  int fin, fin_j, fin_err;
  int owner, csel;
  DF rem;
  int timeout;
  int x;
  float u_i, zt_x, zd_x;
};

__device__ __forceinline__ bool resolvable(unsigned long long w, int kb, int* j_out, bool* err) {
  const unsigned long long mask = (1ull << kWordBits) - 1;
  const unsigned long long D = w & mask;
  const unsigned long long Rj = (w >> kWordBits) & mask;
  const unsigned long long E = (w >> (2 * kWordBits)) & mask;
  const unsigned long long R = Rj | E;
  const int j = R ? __ffsll((long long)R) - 1 : kb;
  const unsigned long long need = (j + 1 >= 64) ? ~0ull : ((1ull << (j + 1)) - 1);
  *j_out = j;
  *err = (E >> j) & 1;
  return (D & need) == need;
}

__device__ void write_outputs(const VerifyParams& P, int b, int n, int y, bool err) {
  int32_t* o = P.out + (size_t)b * (P.K + 1);
  for (int t = 0; t <= P.K; ++t) {
    int v = -1;
    if (!err) v = t < n ? P.tokens[(size_t)b * P.K + t] : (t == n ? y : -1);
    o[t] = v;
  }
  P.nacc[b] = err ? 0 : n;
}

// ---------------------------------------------------------------------------
// The ring: chunk c of the current pass is ring entry q = q0 + c, stage
// q % kStages, mbarrier phase (q / kStages) & 1.  Thread 0 issues the bulk
// copies and waits; the others sleep at the CTA barrier.
// ---------------------------------------------------------------------------
template <int ES>
__device__ __forceinline__ void ring_issue(Shared& sh, char* ring, uint32_t q, int c,
                                           const RowSlice<ES>& st, bool with_d,
                                           const RowSlice<ES>& sd) {
  const int s = q % kStages;
  char* stage = ring + s * kStageBytes;
  uintptr_t tl = 0, th = 0, dl = 0, dh = 0;
  if (c < st.n_chunks) st.chunk_body(c, &tl, &th);
  if (with_d && c < sd.n_chunks) sd.chunk_body(c, &dl, &dh);
  mbar_arrive_expect_tx(&sh.full[s], (uint32_t)((th - tl) + (dh - dl)));
  if (th > tl)
    bulk_copy_g2s(stage + (tl - (st.base16 + (uintptr_t)c * kHalfBytes)),
                  reinterpret_cast<const void*>(tl), (uint32_t)(th - tl), &sh.full[s]);
  if (dh > dl)
    bulk_copy_g2s(stage + kHalfBytes + (dl - (sd.base16 + (uintptr_t)c * kHalfBytes)),
                  reinterpret_cast<const void*>(dl), (uint32_t)(dh - dl), &sh.full[s]);
}

// Stream chunks 0..NC-1 of (st[, sd]) and call body(c, stage) for each, with
// every thread.  Returns false if a bounded wait ran out (the caller reports
// SV_FLAG_TIMEOUT and treats the data as invalid).
template <int ES, typename Body>
__device__ __forceinline__ bool ring_pass(Shared& sh, char* ring, uint32_t& q0, int NC,
                                          const RowSlice<ES>& st, bool with_d,
                                          const RowSlice<ES>& sd, Body body) {
  const int tid = threadIdx.x;
  if (tid == 0)
    for (int c = 0; c < NC && c < kStages; ++c) ring_issue<ES>(sh, ring, q0 + c, c, st, with_d, sd);
  bool ok_all = true;
  for (int c = 0; c < NC; ++c) {
    const uint32_t q = q0 + c;
    const int s = q % kStages;
    const uint32_t par = (q / kStages) & 1;
    bool ok = true;
    if (tid == 0) ok = mbar_wait_bounded(&sh.full[s], par);
    // everyone is done with chunk c-1 and chunk c has landed
    if (__syncthreads_or(!ok)) {
      ok_all = false;
      break;
    }
    if (tid == 0 && c >= 1 && c - 1 + kStages < NC)
      ring_issue<ES>(sh, ring, q + kStages - 1, c - 1 + kStages, st, with_d, sd);
    mbar_try_wait(&sh.full[s], par);  // this thread's acquire of the landed data
    body(c, ring + s * kStageBytes);
  }
  __syncthreads();
  q0 += NC;
  return ok_all;
}

template <int ES>
__global__ void __launch_bounds__(kThreads, 8) verify_kernel(const VerifyParams P) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int item = blockIdx.x / C;
  const int i = item / P.B, b = item % P.B;

  extern __shared__ __align__(128) char ring[];
  __shared__ Shared sh;

  // ---- per-row parameters (identical in every CTA of the cluster) ----
  const int kb = P.kpr ? P.kpr[b] : P.K;
  const int md = P.mode ? (int)P.mode[b] : 0;
  const float T = P.temp ? P.temp[b] : 1.0f;
  uint32_t seq_err = 0;
  if (kb < 0 || kb > P.K) seq_err |= SV_FLAG_BAD_K;
  else if (md != 0 && md != 1) seq_err |= SV_FLAG_BAD_MODE;
  else if (md == 0 && !(T > 0.f && T < INFINITY)) seq_err |= SV_FLAG_BAD_TEMPERATURE;
  else if (md == 0 && kb > 0 && P.drf == nullptr) seq_err |= SV_FLAG_BAD_MODE;  // no draft rows
  if (seq_err) {
    if (i == 0 && rank == 0 && tid == 0) {
      write_outputs(P, b, 0, -1, true);
      atomicOr(P.flags, seq_err);
    }
    return;
  }
  if (i > kb) return;
  const bool greedy = md == 1;
  const bool has_draft = !greedy && i < kb;
  const Expo X = greedy ? Expo{1.f, 1e-30f} : make_expo(T);

  // ---- set-up; rank 0 reads the sequence word ----
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&sh.full[s], 1);
    fence_mbar_init();
    if (rank == 0) {
      const unsigned long long w = __ldcg(P.words + b);
      const unsigned long long R =
          ((w >> kWordBits) | (w >> (2 * kWordBits))) & ((1ull << kWordBits) - 1);
      sh.skip = (R & ((1ull << i) - 1)) != 0;
    }
  }
  // every CTA is running (distributed shared memory is safe) and rank 0's
  // skip flag is visible to all of them
  cluster.sync();
  if (tid == 0) sh.skip_seen = *cluster.map_shared_rank(&sh.skip, 0);
  __syncthreads();
  if (sh.skip_seen) {
    cluster.sync();  // rank 0 stays until every CTA has read its flag
    return;
  }
  // decision inputs, fetched by one thread of warp 1 while the rows stream
  if (rank == 0 && tid == 32) {
    int x = -1;
    float u = 0.f, zt = 0.f, zd = 0.f;
    if (i < kb) {
      x = P.tokens[(size_t)b * P.K + i];
      if (!greedy) u = P.unif[(size_t)b * (P.K + 1) + i];
      if (x >= 0 && x < P.V) {
        const char* rt = P.tgt + (long long)b * P.t_seq + (long long)i * P.t_pos;
        zt = ES == 2 ? bf16_lo(*reinterpret_cast<const uint16_t*>(rt + (size_t)x * 2))
                     : *reinterpret_cast<const float*>(rt + (size_t)x * 4);
        if (has_draft) {
          const char* rd = P.drf + (long long)b * P.d_seq + (long long)i * P.d_pos;
          zd = ES == 2 ? bf16_lo(*reinterpret_cast<const uint16_t*>(rd + (size_t)x * 2))
                       : *reinterpret_cast<const float*>(rd + (size_t)x * 4);
        }
      }
    }
    sh.x = x;
    sh.u_i = u;
    sh.zt_x = zt;
    sh.zd_x = zd;
  }

  // ---- stream the slices: one pass per row ----
  const int e0 = min(P.V, rank * P.slice_len), e1 = min(P.V, e0 + P.slice_len);
  RowSlice<ES> st, sd;
  st.init(P.tgt + (long long)b * P.t_seq + (long long)i * P.t_pos, e0, e1);
  if (has_draft) sd.init(P.drf + (long long)b * P.d_seq + (long long)i * P.d_pos, e0, e1);
  else sd = st;
  uint32_t q0 = 0;
  RowAcc at = acc_init(), ad = acc_init();
  const int NC = has_draft ? max(st.n_chunks, sd.n_chunks) : st.n_chunks;
  const int tb0 = st.ub0(), tb1 = st.ub1(), db0 = sd.ub0(), db1 = sd.ub1();
  const bool ok = ring_pass<ES>(sh, ring, q0, NC, st, has_draft, sd, [&](int c, const char* stage) {
#pragma unroll
    for (int h = 0; h < kUnitsPerThread; ++h) {
      const int u = c * kChunkUnits + h * kThreads + tid;
      row_unit<ES>(at, st, stage, c, u, tb0, tb1, greedy, X);
      if (has_draft) row_unit<ES>(ad, sd, stage + kHalfBytes, c, u, db0, db1, false, X);
    }
  });
  if (!ok && tid == 0) atomicOr(P.flags, (uint32_t)SV_FLAG_TIMEOUT);

  // ---- combine: warps -> CTA -> cluster (warp 0 of every CTA) ----
  {
    const RowAcc wt = lanes_combine(at, true, greedy);
    const RowAcc wd = has_draft ? lanes_combine(ad, true, false) : acc_init();
    if (lane == 0) {
      sh.r_t[warp] = wt;
      sh.r_d[warp] = wd;
    }
  }
  __syncthreads();
  if (warp == 0) {
    RowAcc ct = lanes_combine(lane < kWarps ? sh.r_t[lane] : acc_init(), lane < kWarps, greedy);
    const RowAcc cd = lanes_combine(lane < kWarps ? sh.r_d[lane] : acc_init(), lane < kWarps, false);
    if (!ok) ct.mx = __int_as_float(0x7fc00000);  // a timed-out slice poisons the row
    if (lane < C) {
      *cluster.map_shared_rank(&sh.g_t[rank], lane) = ct;
      *cluster.map_shared_rank(&sh.g_d[rank], lane) = cd;
    }
  }
  cluster.sync();
  if (warp == 0) {
    const RowAcc rt = lanes_combine(lane < C ? sh.g_t[lane] : acc_init(), lane < C, greedy);
    const RowAcc rd = lanes_combine(lane < C ? sh.g_d[lane] : acc_init(), lane < C, false);
    if (lane == 0) {
      sh.row_t = rt;
      sh.row_d = rd;
    }
  }
  __syncthreads();
  const RowAcc row_t = sh.row_t, row_d = sh.row_d;
  // Row validity: no NaN, no +inf, not all -inf, exponent range finite.
  const bool bad_t = !(row_t.mx > -INFINITY && row_t.mx < INFINITY) ||
                     (!greedy && !(row_t.R > kRnone && row_t.R < INFINITY));
  const bool bad_d = has_draft && (!(row_d.mx > -INFINITY && row_d.mx < INFINITY) ||
                                   !(row_d.R > kRnone && row_d.R < INFINITY));

  // ---- decision and publication (rank 0, one thread) ----
  if (rank == 0 && tid == 0) {
    const int x = sh.x;
    const float u_i = sh.u_i, zt_x = sh.zt_x, zd_x = sh.zd_x;
    uint32_t errbits = 0;
    if (bad_t || bad_d) errbits |= SV_FLAG_NONFINITE;
    if (i < kb && (x < 0 || x >= P.V)) errbits |= SV_FLAG_BAD_TOKEN;
    bool reject = false;
    float diag_px = NAN, diag_qx = NAN, diag_r = NAN;
    if (greedy) {
      if (i < kb && !errbits) reject = (x != row_t.amax);
    } else if (has_draft) {
      if (!(u_i >= 0.f && u_i < 1.f)) errbits |= SV_FLAG_BAD_UNIFORM;
      if (!errbits) {
        // p(x)/q(x) = 2^((z_t - z_d)*c + R_d - R_t) * S_d / S_t, formed in the
        // exponent domain so that neither factor underflows on its own;
        // zero where the exact probability underflows double precision.
        const float lt = (zt_x - row_t.mx) * X.chi, ld = (zd_x - row_d.mx) * X.chi;
        float r;
        if (!(ld > -1074.f) || !(lt > -1074.f)) {
          r = 0.f;
        } else {
          const float a = zt_x - zd_x;
          const float ex = __fmaf_rn(a, X.chi, a * X.clo) + (row_d.R - row_t.R);
          r = ex2(ex) * df_to_float(df_div(row_d.s, row_t.s));
        }
        diag_px = ex2(earg(zt_x, X, row_t.R)) / row_t.s.hi;
        diag_qx = ex2(earg(zd_x, X, row_d.R)) / row_d.s.hi;
        diag_r = r;
        reject = !(u_i < r);
      }
    }
    ItemStats s;
    s.m_t = row_t.mx;
    s.R_t = row_t.R;
    s.st_hi = row_t.s.hi;
    s.st_lo = row_t.s.lo;
    s.m_d = row_d.mx;
    s.R_d = row_d.R;
    s.sd_hi = row_d.s.hi;
    s.sd_lo = row_d.s.lo;
    s.argmax = row_t.amax;
    s.errbits = errbits;
    P.stats[(size_t)b * (P.K + 1) + i] = s;
    if (P.diag) {
      float* dg = P.diag + ((size_t)b * (P.K + 1) + i) * SV_DIAG_FIELDS;
      dg[SV_DIAG_M_T] = row_t.mx;
      if (greedy) {
        dg[SV_DIAG_ARGMAX] = (float)row_t.amax;
      } else if (!bad_t) {
        // normaliser relative to the row max: S_R * 2^(R - m*c)
        dg[SV_DIAG_S_T] = df_to_float(row_t.s) * ex2(-earg(row_t.mx, X, row_t.R));
        dg[SV_DIAG_MASS_T] = 1.f;
        if (has_draft && !bad_d) {
          dg[SV_DIAG_M_D] = row_d.mx;
          dg[SV_DIAG_S_D] = df_to_float(row_d.s) * ex2(-earg(row_d.mx, X, row_d.R));
          dg[SV_DIAG_MASS_D] = 1.f;
          dg[SV_DIAG_P_X] = diag_px;
          dg[SV_DIAG_Q_X] = diag_qx;
          dg[SV_DIAG_RATIO] = diag_r;
        }
      }
    }
    __threadfence();
    unsigned long long bits = 1ull << i;
    if (errbits) bits |= 1ull << (2 * kWordBits + i);
    else if (reject) bits |= 1ull << (kWordBits + i);
    const unsigned long long old = atomicOr(P.words + b, bits);
    __threadfence();
    int j0, j1;
    bool e0_, e1_;
    const bool was = resolvable(old, kb, &j0, &e0_);
    const bool now = resolvable(old | bits, kb, &j1, &e1_);
    const int fin = (!was && now) ? 1 : 0;
    for (int r = 0; r < C; ++r) {
      Shared* rs = cluster.map_shared_rank(&sh, r);
      rs->fin = fin;
      rs->fin_j = j1;
      rs->fin_err = e1_ ? 1 : 0;
    }
  }
  cluster.sync();
  if (!sh.fin) return;

  // ======================= finisher =======================
  const int j = sh.fin_j;
  if (sh.fin_err) {
    if (rank == 0 && tid == 0) {
      const uint32_t eb = __ldcg(&P.stats[(size_t)b * (P.K + 1) + j].errbits);
      write_outputs(P, b, 0, -1, true);
      atomicOr(P.flags, eb);
    }
    return;
  }
  if (greedy) {
    if (rank == 0 && tid == 0) {
      const int a = j == i ? row_t.amax : __ldcg(&P.stats[(size_t)b * (P.K + 1) + j].argmax);
      write_outputs(P, b, j, a, false);
    }
    return;
  }
  const float uK = P.unif[(size_t)b * (P.K + 1) + P.K];
  if (!(uK >= 0.f && uK < 1.f)) {
    if (rank == 0 && tid == 0) {
      write_outputs(P, b, 0, -1, true);
      atomicOr(P.flags, SV_FLAG_BAD_UNIFORM);
    }
    return;
  }
  const bool bonus = (j == kb);
  float Rt = row_t.R, Rd = row_d.R;
  DF S_t = row_t.s, S_d = row_d.s;
  if (j != i) {
    const ItemStats* sj = P.stats + (size_t)b * (P.K + 1) + j;
    Rt = __ldcg(&sj->R_t);
    Rd = __ldcg(&sj->R_d);
    S_t = DF{__ldcg(&sj->st_hi), __ldcg(&sj->st_lo)};
    S_d = DF{__ldcg(&sj->sd_hi), __ldcg(&sj->sd_lo)};
  }
  st.init(P.tgt + (long long)b * P.t_seq + (long long)j * P.t_pos, e0, e1);
  if (!bonus) sd.init(P.drf + (long long)b * P.d_seq + (long long)j * P.d_pos, e0, e1);
  else sd = st;
  const bool same_phase = st.ebase0 == sd.ebase0;
  const bool load_d = !bonus && same_phase;  // else the draft is read element-wise
  Weight W;
  W.x = X;
  W.Rt = Rt;
  W.Rd = Rd;
  W.p_only = bonus;
  {
    const DF rho = bonus ? DF{0.f, 0.f} : df_div(S_t, S_d);
    W.rho_hi = rho.hi;
    W.rho_lo = rho.lo;
  }
  const int NCj = st.n_chunks;
  DF slice_w{0.f, 0.f};
  for (int pass = 0; pass < 2; ++pass) {
    if (pass) cluster.sync();  // every CTA has read the first pass's slots
    const bool okp = ring_pass<ES>(sh, ring, q0, NCj, st, load_d && !W.p_only, sd,
                                   [&](int c, const char* stage) {
      float v = 0.f;
#pragma unroll
      for (int h = 0; h < kUnitsPerThread; ++h)
        v += unit_wsum<ES>(st, sd, stage, stage + kHalfBytes, c, c * kChunkUnits + h * kThreads + tid,
                           W, same_phase);
      const DF wsum = df_warp_sum(DF{v, 0.f});
      if (lane == 0) sh.tw[c][warp] = wsum;
    });
    if (!okp && tid == 0) atomicOr(P.flags, (uint32_t)SV_FLAG_TIMEOUT);
    if (warp == 0) {
      DF a{0.f, 0.f};
      if (lane < NCj)
        for (int w = 0; w < kWarps; ++w) a = df_add(a, sh.tw[lane][w]);
      a = df_warp_sum(a);
      if (lane < C) *cluster.map_shared_rank(&sh.g_w[rank], lane) = a;
    }
    cluster.sync();
    if (warp == 0) {
      const DF tot = df_warp_sum(lane < C ? sh.g_w[lane] : DF{0.f, 0.f});
      if (lane == 0) sh.S_w = tot;
    }
    __syncthreads();
    const DF tot = sh.S_w;
    if (df_pos(tot) || W.p_only) {
      slice_w = tot;
      break;
    }
    W.p_only = true;  // residual all zero: draw from p  [SSD §4.3]
  }
  // ---- locate u * total: rank, then chunk (warp 0), then unit, element ----
  const DF tgt = df_mul_f(slice_w, uK);
  if (warp == 0) {
    const DF v = lane < C ? sh.g_w[lane] : DF{0.f, 0.f};
    const DF inc = df_warp_scan(v, lane);
    const unsigned hit = __ballot_sync(0xffffffffu, lane < C && df_pos(v) && df_gt(inc, tgt));
    const unsigned pos = __ballot_sync(0xffffffffu, lane < C && df_pos(v));
    const int owner = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    const DF v_own = df_shfl(v, owner);
    // past the end by rounding: the last positive slice, just inside its end
    DF rem = hit ? df_sub(tgt, df_sub(df_shfl(inc, owner), v_own)) : df_mul_f(v_own, 0.999999f);
    if (rank == 0 && lane == 0 && P.diag) {
      float* dg = P.diag + ((size_t)b * (P.K + 1) + j) * SV_DIAG_FIELDS;
      dg[SV_DIAG_S_W] = W.p_only ? 1.f : df_to_float(df_div(slice_w, S_t));
    }
    if (owner == rank) {
      DF cv{0.f, 0.f};
      if (lane < NCj)
        for (int w = 0; w < kWarps; ++w) cv = df_add(cv, sh.tw[lane][w]);
      const DF cinc = df_warp_scan(cv, lane);
      const unsigned ch = __ballot_sync(0xffffffffu, lane < NCj && df_pos(cv) && df_gt(cinc, rem));
      const unsigned cp = __ballot_sync(0xffffffffu, lane < NCj && df_pos(cv));
      const int csel = ch ? __ffs(ch) - 1 : (cp ? 31 - __clz(cp) : 0);
      const DF cv_sel = df_shfl(cv, csel);
      rem = ch ? df_sub(rem, df_sub(df_shfl(cinc, csel), cv_sel)) : df_mul_f(cv_sel, 0.999999f);
      if (lane == 0) {
        sh.csel = csel;
        sh.rem = rem;
      }
    }
    if (lane == 0) sh.owner = owner;
  }
  __syncthreads();
  if (sh.owner != rank) return;
  // read back chunk csel and scan its units in index order
  const int csel = sh.csel;
  const DF rem = sh.rem;
  const int s_last = q0 % kStages;
  const uint32_t par_last = (q0 / kStages) & 1;
  const char* stage = ring + s_last * kStageBytes;
  if (tid == 0) {
    ring_issue<ES>(sh, ring, q0, csel, st, load_d && !W.p_only, sd);
    if (!mbar_wait_bounded(&sh.full[s_last], par_last)) {
      atomicOr(P.flags, (uint32_t)SV_FLAG_TIMEOUT);
      sh.timeout = 1;
    } else {
      sh.timeout = 0;
    }
  }
  __syncthreads();
  if (sh.timeout) {
    if (tid == 0) write_outputs(P, b, 0, -1, true);
    return;
  }
  mbar_try_wait(&sh.full[s_last], par_last);
  const int ubase = csel * kChunkUnits;
  float v[kUnitsPerThread];
#pragma unroll
  for (int h = 0; h < kUnitsPerThread; ++h)
    v[h] = unit_wsum<ES>(st, sd, stage, stage + kHalfBytes, csel, ubase + h * kThreads + tid, W,
                         same_phase);
  // block-wide inclusive prefix of the unit sums, units 0..255 in order:
  // half h holds units h*kThreads + tid
  DF inc[kUnitsPerThread];
  DF carry{0.f, 0.f};
#pragma unroll
  for (int h = 0; h < kUnitsPerThread; ++h) {
    const DF wi = df_warp_scan(DF{v[h], 0.f}, lane);
    if (lane == 31) sh.scan[h & 1][warp] = wi;
    __syncthreads();
    DF before = carry;
    for (int w = 0; w < warp; ++w) before = df_add(before, sh.scan[h & 1][w]);
    DF total = carry;
    for (int w = 0; w < kWarps; ++w) total = df_add(total, sh.scan[h & 1][w]);
    inc[h] = df_add(before, wi);
    carry = total;
  }
  int cand = 0x7fffffff, lastpos = -1;
#pragma unroll
  for (int h = kUnitsPerThread - 1; h >= 0; --h) {
    const int uo = h * kThreads + tid;  // unit offset in the chunk
    if (v[h] > 0.f) {
      lastpos = max(lastpos, uo);
      if (df_gt(inc[h], rem)) cand = uo;
    }
  }
  cand = warp_min(cand);
  lastpos = -warp_min(-lastpos);
  if (lane == 0) sh.r_i[warp] = cand;
  __syncthreads();
  int usel = 0x7fffffff;
  for (int w = 0; w < kWarps; ++w) usel = min(usel, sh.r_i[w]);
  __syncthreads();
  if (lane == 0) sh.r_i[warp] = lastpos;
  __syncthreads();
  bool past_end = false;
  if (usel == 0x7fffffff) {  // rounding: the last positive unit
    past_end = true;
    usel = -1;
    for (int w = 0; w < kWarps; ++w) usel = max(usel, sh.r_i[w]);
    if (usel < 0) usel = 0;
  }
  const int hsel = usel / kThreads, tsel = usel % kThreads;
  if (tid != tsel) return;
  constexpr int EPU = 16 / ES;
  const int u = ubase + usel;
  DF cum = past_end ? DF{0.f, 0.f} : df_sub(inc[hsel], DF{v[hsel], 0.f});
  int y = -1, ylast = -1;
  const int eb = st.ebase0 + u * EPU;
  for (int q = 0; q < EPU; ++q) {
    const int e = eb + q;
    if (e < st.e0 || e >= st.e1) continue;
    const float wv = elem_w<ES>(st, sd, stage, stage + kHalfBytes, csel, u, e, W, same_phase);
    if (wv > 0.f) ylast = e;
    cum = df_add(cum, DF{wv, 0.f});
    if (!past_end && wv > 0.f && df_gt(cum, rem)) {
      y = e;
      break;
    }
  }
  if (y < 0) y = ylast;
  write_outputs(P, b, j, y, false);
}

__global__ void verify_init_kernel(uint32_t* flags, unsigned long long* words, int B) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t == 0) *flags = 0u;
  for (int b = t; b < B; b += gridDim.x * blockDim.x) words[b] = 0ull;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

size_t ws_layout(int B, int K, size_t* words_off, size_t* stats_off) {
  size_t off = 256;
  *words_off = off;
  off += ((size_t)B * 8 + 255) / 256 * 256;
  *stats_off = off;
  off += (size_t)B * (K + 1) * sizeof(ItemStats);
  return (off + 255) / 256 * 256;
}

static int g_configured[2] = {0, 0};

template <int ES>
static cudaError_t configure() {
  return cudaFuncSetAttribute(verify_kernel<ES>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int ES>
static cudaError_t launch(const VerifyParams& P0, int C, int items, cudaStream_t stream) {
  VerifyParams P = P0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)items * (unsigned)C, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kStages * kStageBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_kernel<ES>, P);
}

// Cluster width: about 32 KB of each row per CTA, at most 16 CTAs.
static void choose_geometry(int V, int ES, int* C_out, int* slice_out) {
  const long long row_bytes = (long long)V * ES;
  int C = (int)((row_bytes + 32767) / 32768);
  if (C < 1) C = 1;
  if (C > kCmax) C = kCmax;
  int slice = (V + C - 1) / C;
  slice = (slice + 7) / 8 * 8;
  C = (V + slice - 1) / slice;
  if (C < 1) C = 1;
  *C_out = C;
  *slice_out = slice;
}

int verify_launch(const VerifyLaunch& L, std::string* err) {
  const int ES = L.dtype == SV_BF16 ? 2 : 4;
  int C, slice;
  choose_geometry(L.V, ES, &C, &slice);
  if ((long long)slice * ES + 32 > (long long)kMaxChunks * kHalfBytes) {
    *err = "vocabulary too large for the cluster slice layout";
    return SV_ERR_SHAPE;
  }
  cudaError_t e;
  const int gi = ES == 2 ? 0 : 1;
  if (!g_configured[gi]) {
    e = ES == 2 ? configure<2>() : configure<4>();
    if (e != cudaSuccess) {
      *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return SV_ERR_CUDA;
    }
    g_configured[gi] = 1;
  }
  size_t words_off, stats_off;
  ws_layout(L.B, L.K, &words_off, &stats_off);
  char* ws = static_cast<char*>(L.workspace);
  VerifyParams P;
  P.tgt = static_cast<const char*>(L.target);
  P.t_seq = L.t_seq * ES;
  P.t_pos = L.t_pos * ES;
  P.drf = static_cast<const char*>(L.draft);
  P.d_seq = L.d_seq * ES;
  P.d_pos = L.d_pos * ES;
  P.B = L.B;
  P.K = L.K;
  P.V = L.V;
  P.tokens = L.tokens;
  P.kpr = L.kpr;
  P.temp = L.temp;
  P.top_p = L.top_p;
  P.unif = L.unif;
  P.mode = L.mode;
  P.out = L.out;
  P.nacc = L.nacc;
  P.diag = L.diag;
  P.flags = reinterpret_cast<uint32_t*>(ws);
  P.words = reinterpret_cast<unsigned long long*>(ws + words_off);
  P.stats = reinterpret_cast<ItemStats*>(ws + stats_off);
  P.slice_len = slice;
  cudaStream_t stream = static_cast<cudaStream_t>(L.stream);

  const int ib = (L.B + 255) / 256;
  verify_init_kernel<<<ib < 1 ? 1 : ib, 256, 0, stream>>>(P.flags, P.words, L.B);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("init launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  const int items = (L.K + 1) * L.B;
  e = ES == 2 ? launch<2>(P, C, items, stream) : launch<4>(P, C, items, stream);
  if (e != cudaSuccess) {
    *err = std::string("verify launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

size_t verify_workspace_bytes(int B, int K) {
  size_t a, b;
  return ws_layout(B, K, &a, &b);
}

}  // namespace sv
