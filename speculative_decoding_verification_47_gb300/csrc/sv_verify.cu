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
// [r*L, (r+1)*L) of both rows.  Each thread keeps two steps of 16-byte units
// of both rows in flight in its own shared-memory slots (cp.async) and
// reduces the oldest step.  Each row is reduced in ONE pass: the running max,
// and the sum of 2^(z*c - R) where the reference exponent R is an integer
// that only grows; when it grows the partial sum is rescaled by an exact
// power of two, so the online pass adds no rounding beyond the exponentials
// themselves.  The cluster combines the per-slice results through
// distributed shared memory.
//
// Items are launched position-major (all sequences' position 0 first).  Each
// item publishes {done, rejected, error} bits for its position in one 64-bit
// word per sequence.  An item whose sequence already has an earlier rejection
// (seen at its start, or while it streams) drops out: those rows cannot
// change the result.  Every CTA of the cluster computes the item's verdict;
// rank 0 publishes it.  A sampled item that rejects x_i, or the bonus item
// i = k_b, then draws its token at once from norm(max(0, p - q)) (or p):
// one more pass over its rows sums the residual per warp and round, and one
// warp re-reads the 32 units around the inverse-CDF point.  The sequence's
// outputs are written by whichever comes last of the item that completes the
// prefix 0..j (j = first rejection, or k_b) and the draw at j, met through a
// second per-sequence word.  No item ever waits for another one.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCmax = 16;
static_assert((kWarps & (kWarps - 1)) == 0 && kCmax <= 16, "butterfly widths are powers of two up to 16");
constexpr int kLoadsInFlight = 2;                  // 16-byte units per row per thread per step
constexpr int kRingStages = 2;                     // steps of units in flight ahead of the one reduced
constexpr int kSampleRingStages = 2;               // the draft sampler's (one row): more stages cost
                                                   // a CTA per SM, which is slower
constexpr int kRingBytes = kRingStages * 2 * kLoadsInFlight * kThreads * 16;  // 32 KB
constexpr int kMaxRounds = 64;                     // slice <= 64 * 256 units = 256 KB of a row
constexpr int kWordBits = 21;                      // positions per field of the sequence word

// What an item leaves for the one that writes its sequence's outputs.
struct ItemStats {
  int argmax;        // first maximum of the target row (greedy rows)
  uint32_t errbits;  // SV_FLAG_* bits of this position's error, 0 if none
  int y;             // this position's draw (resample or bonus), kYBad if its uniform was bad
  int pad;
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
  uint32_t* words2;  // per sequence: bit 0 prefix resolved, bit 1+i draw of position i stored
  int topp_draft;    // top_p < 1: also truncate the draft rows (1) or only the target rows (0)
  ItemStats* stats;
  int slice_len;  // elements per CTA slice
};

// ---------------------------------------------------------------------------
// One CTA's slice [e0, e1) of one logit row, in 16-byte units: unit u holds
// global bytes [base16 + 16u, base16 + 16u + 16).  Units inside the aligned
// body [a0, a1) are fully valid and are read as 16-byte vectors (cp.async
// into shared memory in the row pass, plain loads in the others); the (at most
// two) partial units at the ends are read element by element.
// ---------------------------------------------------------------------------
template <int ES>
struct RowSlice {
  const char* row;
  int e0, e1;
  uintptr_t base16, a0, a1;
  int n_units, ebase0;

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
  }
    // units [ub0, ub1) are fully inside the aligned body
  __device__ __forceinline__ int ub0() const { return (int)((a0 - base16) / 16); }
  __device__ __forceinline__ int ub1() const { return (int)((a1 - base16) / 16); }
  __device__ __forceinline__ float elem(int e) const {  // from global memory
    return ES == 2 ? bf16_lo(*reinterpret_cast<const uint16_t*>(row + (size_t)e * 2))
                   : *reinterpret_cast<const float*>(row + (size_t)e * 4);
  }
  __device__ __forceinline__ uint32_t bits(int e) const {  // bit pattern, from global memory
    return ES == 2 ? (uint32_t)*reinterpret_cast<const uint16_t*>(row + (size_t)e * 2)
                   : *reinterpret_cast<const uint32_t*>(row + (size_t)e * 4);
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

// largest non-NaN logit of a unit (-inf if none)
template <int ES>
__device__ __forceinline__ float unit_max_num(const uint4& v) {
  if (ES == 2) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
    __nv_bfloat162 m2 = __hmax2(__hmax2(p[0], p[1]), __hmax2(p[2], p[3]));
    return fmaxf(__low2float(m2), __high2float(m2));
  } else {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
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
// Top-p order [FS §3.2]: tokens ranked by (probability desc, index asc) are
// the tokens ranked by (logit desc, index asc), because the temperature
// softmax is increasing in the logit.  A logit is identified by the
// order-preserving unsigned key of its bit pattern (-0 taken as +0), so
// "ranked before" is "larger key, or the same key at a smaller index".
// ---------------------------------------------------------------------------
template <int ES>
__device__ __forceinline__ uint32_t okey(uint32_t b) {
  if (ES == 2) {
    b &= 0xffffu;
    if (b == 0x8000u) b = 0u;
    return (b & 0x8000u) ? (~b & 0xffffu) : (b | 0x8000u);
  } else {
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
}

// inverse of okey: the bit pattern of a key
template <int ES>
__device__ __forceinline__ uint32_t key_bits(uint32_t k) {
  if (ES == 2) return (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
  return (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
}

template <int ES>
__device__ __forceinline__ float bits_val(uint32_t b) {
  return ES == 2 ? __uint_as_float(b << 16) : __uint_as_float(b);
}

// bit pattern of a value that is exactly representable in the row's type
template <int ES>
__device__ __forceinline__ uint32_t val_bits(float v) {
  return ES == 2 ? (__float_as_uint(v) >> 16) : __float_as_uint(v);
}

// bit pattern of the largest representable value <= v
template <int ES>
__device__ __forceinline__ uint32_t floor_bits(float v) {
  return ES == 2 ? (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rd(v)) : __float_as_uint(v);
}

// bit pattern of the smallest representable value >= v
template <int ES>
__device__ __forceinline__ uint32_t ceil_bits(float v) {
  return ES == 2 ? (uint32_t)__bfloat16_as_ushort(__float2bfloat16_ru(v)) : __float_as_uint(v);
}

// element j of a 16-byte unit as its bit pattern
template <int ES>
__device__ __forceinline__ uint32_t unit_bits(const uint4& v, int j) {
  if (ES == 4) return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
  const uint32_t w = (j >> 1) == 0 ? v.x : (j >> 1) == 1 ? v.y : (j >> 1) == 2 ? v.z : v.w;
  return (j & 1) ? (w >> 16) : (w & 0xffffu);
}

// kept by the cut (key kk, first dropped index kc among the tokens of key kk)
__device__ __forceinline__ bool topp_kept(uint32_t key, int idx, uint32_t kk, int kc) {
  return key > kk || (key == kk && idx < kc);
}

// ---------------------------------------------------------------------------
// Per-thread row accumulator
// ---------------------------------------------------------------------------
struct RowAcc {
  float mx;      // running max of the raw logits (NaN propagates)
  float R;       // integer reference exponent, kRnone until a finite element
  DF s;          // sum of 2^(z*c - R)
  int amax;      // index of the first maximum (greedy rows)
  float pend;    // unit sums not yet added into s (same reference R)
  uint32_t mx2;  // bf16 sampled rows: running max as a packed bf16x2
};

constexpr uint32_t kBf16x2NegInf = 0xff80ff80u;

__device__ __forceinline__ RowAcc acc_init() {
  return RowAcc{-INFINITY, kRnone, DF{0.f, 0.f}, 0x7fffffff, 0.f, kBf16x2NegInf};
}

__device__ __forceinline__ void acc_raise(RowAcc& a, float Rn) {
  const float p = pow2i(a.R - Rn);  // exact power of two (0 from kRnone)
  a.s.hi *= p;
  a.s.lo *= p;
  a.pend *= p;
  a.R = Rn;
}

// A unit of 8 or fewer weights whose sum exceeds 8 has an element above the
// reference (2^(z*c - R) > 1): the reference is raised to ceil(max*c) and the
// unit recomputed.  So R stays within 3 of the thread's largest z*c, and the
// heaviest weights are formed from arguments in [-1, 3]: the rounding of
// z*c - R to float grows with its magnitude, and a reference lagging the
// maximum by ~20 made those weights ~10x less precise, which moved draws that
// fall within ~1e-8 of a CDF boundary.  (A raise happens once per new
// running maximum of the thread; the first unit always raises from kRnone.)
constexpr float kRaiseAbove = 8.f;

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// move pending unit sums into the compensated total
__device__ __forceinline__ void acc_flush(RowAcc& a) {
  df_acc(a.s, a.pend);
  a.pend = 0.f;
}

// running max of a sampled row as a float (after the pass)
template <int ES>
__device__ __forceinline__ void acc_finish_max(RowAcc& a) {
  if (ES == 2) {
    const float lo = bf16_lo(a.mx2), hi = bf16_hi(a.mx2);
    a.mx = nanmax(a.mx, nanmax(lo, hi));
  }
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

// sum over a full unit of 2^(z*c - R) (f32x2 lanes)
template <int ES>
__device__ __forceinline__ float unit_sumexp(const uint4& v, const Expo& x, float R) {
  const F2 C = f2_pack(x.chi, x.chi), L = f2_pack(x.clo, x.clo);
  const F2 N = f2_pack(-R, -R);
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
  return sx + sy;
}

// Adds a full unit to the row accumulator.  With MAX it returns the unit's
// max (NaN if it holds one), which callers that keep per-thread candidate
// lists compare; without, it returns 0 and forms the max only when the
// reference exponent must rise.
template <int ES, bool MAX = false>
__device__ __forceinline__ float sampled_unit(RowAcc& a, const uint4& v, const Expo& x) {
  uint32_t um = 0;
  if (ES == 2) {
    um = bf16x2_max_nan(bf16x2_max_nan(v.x, v.y), bf16x2_max_nan(v.z, v.w));
    a.mx2 = bf16x2_max_nan(a.mx2, um);
  } else {
    a.mx = nanmax(a.mx, unit_max<ES>(v));
  }
  float g = 0.f;
  if (MAX) g = ES == 2 ? nanmax(bf16_lo(um), bf16_hi(um)) : unit_max<ES>(v);
  float us = unit_sumexp<ES>(v, x, a.R);
  if (!(us <= kRaiseAbove)) {
    if (!MAX) g = ES == 2 ? nanmax(bf16_lo(um), bf16_hi(um)) : unit_max<ES>(v);
    const float gc = g * x.chi;
    if (gc > a.R) {
      acc_raise(a, ceilf(gc));
      us = unit_sumexp<ES>(v, x, a.R);
    }
  }
  a.pend += us;
  return g;
}

__device__ __forceinline__ void sampled_elem(RowAcc& a, float z, const Expo& x) {
  a.mx = nanmax(a.mx, z);
  const float zc = z * x.chi;
  if (zc > a.R) acc_raise(a, ceilf(zc));
  a.pend += e2(z, x, -a.R);
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

// ---------------------------------------------------------------------------
// Loads: 16-byte units, read-only path, straight into registers or (the row
// pass) copied asynchronously into the thread's own shared-memory slots
// (cp.async: the bytes in flight hold no registers).  Units outside the
// aligned body [ub0, ub1) are read element by element.
// ---------------------------------------------------------------------------
// Brings [a, a + bytes) of global memory into L2 with the bulk-copy engine
// (a and bytes multiples of 16; nothing is written to shared memory).
__device__ __forceinline__ void l2_prefetch_bulk(uintptr_t a, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(bytes) : "memory");
}

// The aligned body of a slice back into L2, 16 KB per lane of the calling
// warp (every lane calls).
template <int ES>
__device__ __forceinline__ void l2_prefetch_slice(const RowSlice<ES>& rs, int lane) {
  constexpr uint32_t kPiece = 16384;
  const uintptr_t n = rs.a1 - rs.a0;  // (a multiple of 16)
  for (uintptr_t o = (uintptr_t)lane * kPiece; o < n; o += 32 * (uintptr_t)kPiece)
    l2_prefetch_bulk(rs.a0 + o, (uint32_t)(n - o < kPiece ? n - o : kPiece));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int ES>
__device__ __forceinline__ uint4 ldg_unit(const RowSlice<ES>& rs, int u) {
  return __ldg(reinterpret_cast<const uint4*>(rs.base16 + 16 * (uintptr_t)u));
}

// ---------------------------------------------------------------------------
// Per-thread unit lists (top-p instances).  During the row pass each thread
// keeps, per row, the kListLen units of its slice with the largest maxima
// (the max's key and the unit's index, keys descending; key 0 = empty slot)
// in shared memory, slot k of row r at lst[(r * kListLen + k) * kThreads +
// tid].  A unit is recorded only if its max is strictly larger than the
// thread's last entry (once the list is full) and than the CTA's floor T
// (sh.lth[r]): the largest last-entry key any full list of the CTA has had,
// raised with atomicMax as lists fill.  T only grows, so every unit left out
// (or pushed out later) has a max key <= the final T; with theta = the
// largest final T over the cluster's CTAs, every token of the row whose key
// exceeds theta lies in a recorded unit.  The selection re-reads just those
// units to collect the candidates above theta (at most kListLen units per
// thread and row).
// ---------------------------------------------------------------------------
constexpr int kListLen = 4;

// value of a key, -inf for key 0 (no floor yet)
template <int ES>
__device__ __forceinline__ float key_val(uint32_t k) {
  return k ? bits_val<ES>(key_bits<ES>(k)) : -INFINITY;
}


// Combine row accumulators over groups of W lanes of a warp (W a power of
// two; lanes with valid == false contribute nothing): xor butterflies over
// offsets W/2 .. 1.  Every lane of a group ends with the group's result, and
// every CTA that combines the same values in the same lanes gets the same
// bits.
__device__ __forceinline__ float lanes_maxf(float v, int W) {
#pragma unroll
  for (int o = W >> 1; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float lanes_nanmax(float v, int W) {
#pragma unroll
  for (int o = W >> 1; o > 0; o >>= 1) v = nanmax(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int lanes_min(int v, int W) {
#pragma unroll
  for (int o = W >> 1; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ DF lanes_dfsum(DF v, int W) {
#pragma unroll
  for (int o = W >> 1; o > 0; o >>= 1) v = df_add(v, df_shfl_xor(v, o));
  return v;
}

__device__ __forceinline__ int warp_min(int v) { return lanes_min(v, 32); }

// Lane 0's accumulator on every lane of the warp.
__device__ __forceinline__ RowAcc acc_bcast0(const RowAcc& v) {
  RowAcc r;
  r.mx = __shfl_sync(0xffffffffu, v.mx, 0);
  r.R = __shfl_sync(0xffffffffu, v.R, 0);
  r.s.hi = __shfl_sync(0xffffffffu, v.s.hi, 0);
  r.s.lo = __shfl_sync(0xffffffffu, v.s.lo, 0);
  r.amax = __shfl_sync(0xffffffffu, v.amax, 0);
  r.pend = 0.f;
  r.mx2 = kBf16x2NegInf;
  return r;
}

__device__ __forceinline__ RowAcc lanes_combine(RowAcc v, bool valid, bool greedy, int W = 32) {
  if (!valid) v = acc_init();
  const float m = lanes_nanmax(v.mx, W);
  if (greedy) {
    const int cand = (v.mx == m) ? v.amax : 0x7fffffff;
    return RowAcc{m, -INFINITY, DF{0.f, 0.f}, lanes_min(cand, W)};
  }
  const float Rw = lanes_maxf(v.R, W);
  DF s = DF{0.f, 0.f};
  if (v.R > kRnone && Rw > kRnone) {
    const float p = pow2i(v.R - Rw);
    s = DF{v.s.hi * p, v.s.lo * p};
  }
  s = lanes_dfsum(s, W);
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
  // top-p cuts of the two rows (every token kept: key 0, index INT_MAX);
  // vkt = value of key kt (-inf without a cut): below it no target token is kept
  uint32_t kt, kd;
  int ct, cd;
  float vkt;
  // weight of element e with logits (zt, zd) and keys (yt, yd), top-p masks applied
  __device__ __forceinline__ float masked(float zt, float zd, uint32_t yt, uint32_t yd,
                                          int e) const {
    const float a = topp_kept(yt, e, kt, ct) ? e2(zt, x, -Rt) : 0.f;
    if (p_only) return a;
    const float b = topp_kept(yd, e, kd, cd) ? e2(zd, x, -Rd) : 0.f;
    return fmaxf(0.f, __fmaf_rn(-rho_lo, b, __fmaf_rn(-rho_hi, b, a)));
  }
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

// Weight sum of one full unit (both rows hold the same elements in it).
template <int ES>
__device__ __forceinline__ float wsum_full(const uint4& vt, const uint4& vd, const Weight& W) {
  if (W.p_only) {  // w = e_t: the row pass's unit sum (packed f32x2 arithmetic)
    (void)vd;
    return unit_sumexp<ES>(vt, W.x, W.Rt);
  }
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

// Masked weight sum of one full unit (out of line: reached only by the units
// that hold a kept target token).
template <int ES>
__device__ __noinline__ float masked_unit(const Weight& W, uint4 vt, uint4 vd, int eb) {
  constexpr int EPU = 16 / ES;
  float acc = 0.f;
#pragma unroll 1
  for (int j = 0; j < EPU; ++j) {
    const uint32_t bt = unit_bits<ES>(vt, j), bd = W.p_only ? 0u : unit_bits<ES>(vd, j);
    acc += W.masked(bits_val<ES>(bt), bits_val<ES>(bd), okey<ES>(bt), okey<ES>(bd), eb + j);
  }
  return acc;
}

// The rows of a drawing item as the draw reads them a second time (from L2
// when they are still there).  Full units of both rows are read as 16-byte
// vectors when the rows share their 16-byte phase, else element by element.
template <int ES>
struct PairRead {
  RowSlice<ES> st, sd;
  int ub0, ub1;
  bool vec;
  __device__ __forceinline__ bool full(int u) const { return vec && u >= ub0 && u < ub1; }
  __device__ __forceinline__ void load(int u, const Weight& W, uint4& vt, uint4& vd) const {
    if (full(u)) {
      vt = ldg_unit(st, u);
      if (!W.p_only) vd = ldg_unit(sd, u);
    }
  }
  template <bool TOPP>
  __device__ __forceinline__ float value(int u, const Weight& W, const uint4& vt,
                                         const uint4& vd) const {
    constexpr int EPU = 16 / ES;
    if (u >= st.n_units) return 0.f;
    const int eb = st.ebase0 + u * EPU;
    if (full(u)) {
      if (!TOPP) return wsum_full<ES>(vt, W.p_only ? vt : vd, W);
      // no kept target token: max(0, 0 - rho q') = 0 for every element
      if (unit_max<ES>(vt) < W.vkt) return 0.f;
      return masked_unit<ES>(W, vt, vd, eb);
    }
    float acc = 0.f;
    for (int j = 0; j < EPU; ++j) {
      const int e = eb + j;
      if (e < st.e0 || e >= st.e1) continue;
      acc += elem_w<TOPP>(e, W);
    }
    return acc;
  }
  template <bool TOPP>
  __device__ __forceinline__ float elem_w(int e, const Weight& W) const {
    if (!TOPP) return W(st.elem(e), W.p_only ? 0.f : sd.elem(e));
    const uint32_t bt = st.bits(e), bd = W.p_only ? 0u : sd.bits(e);
    return W.masked(bits_val<ES>(bt), bits_val<ES>(bd), okey<ES>(bt), okey<ES>(bd), e);
  }
};

// ---------------------------------------------------------------------------
// Top-p selection state of one row.  The cut is searched in the key window
// [lo, hi].  Every pass sums the mass of the tokens above the window exactly
// (in registers).  A "count" pass (window of at most kNB keys) histograms
// exact token counts per key, so a key's mass is count * 2^(z*c - R) with no
// summation error; it settles the cut when the cut lies in the window.  A
// wider window first
// takes a "locator" pass: float masses over kNB bins, which only choose the
// bin that most likely holds the cut (their order of accumulation does not
// change the result, which comes from exact counts).  Locator bins are
// uniform in log-probability (z*c - R), so the many tokens of a long tail
// spread over many bins; when that cannot narrow a window (keys too close in
// value), bins of 2^shift consecutive keys are used instead.
// If a pass finds the cut outside its window (a locator misled by rounding),
// the feasible key range [flo, fhi] shrinks to the side that holds it and
// the search continues there.
// ---------------------------------------------------------------------------
constexpr int kNB = 2048;
constexpr int kSlotLt = kNB;         // count pass: tokens of key kx before the draft token
constexpr int kSlotAbove = kNB + 2;  // count pass: double-float mass above the window
constexpr int kHistRowBytes = 8448;  // >= (kNB + 4) * 4
constexpr int kHistBytes = 2 * kHistRowBytes;
constexpr int kSelLoads = 4;  // units per thread per step of a selection pass
constexpr int kStageBytes = kThreads * kSelLoads * 16;  // each thread's units of a step
constexpr int kSelSmemBytes = kHistBytes + kStageBytes;
// candidate lists (top-p instances): after the row pass's ring and the
// selection's histograms and staging, alive from the row pass to the cut
constexpr int kListOff = ((kSelSmemBytes > kRingBytes ? kSelSmemBytes : kRingBytes) + 255) / 256 * 256;
constexpr int kListBytes = 2 * kListLen * kThreads * 8;
constexpr int kToppSmemBytes = kListOff + kListBytes;
// the draft sampler without top-p: a ring of the target slots, then the unit sums
constexpr int kSampleSumsOff = kSampleRingStages * kLoadsInFlight * kThreads * 16;
// candidates above the cluster's floor (top-p instances): this CTA's at the
// start of the dynamic area, the cluster's gathered after them, and the
// cluster's in rank order over the unit lists once those are read
constexpr int kUOwn = 512;   // candidates one CTA may contribute per row
constexpr int kUCap = 1024;  // candidates per row over the cluster
constexpr int kUAllOff = 2 * kUOwn * 8;
static_assert(kUAllOff + 2 * kUCap * 8 <= kListOff && 2 * kUCap * 8 <= kListBytes, "candidate areas");
// local ranking of one row's candidates: counts and slot starts of
// kRankBins value bins, between the gathered candidates and the lists
constexpr int kRankBins = 1024;
constexpr int kRankOff = kUAllOff + 2 * kUCap * 8;
constexpr int kRankGroupMax = 64;  // the most candidates one bin may hold
static_assert(kRankOff + 2 * kRankBins * 4 <= kListOff, "ranking area");
constexpr int kMaxSelPasses = 12;

struct TopSel {
  uint32_t lth;       // the cluster's list floor: the lists hold every key above it
  uint32_t lo, hi;    // window of the next pass
  uint32_t flo, fhi;  // keys that may still hold the cut
  int mode;           // 0 resolved, 1 count pass next, 2 locator pass next
  int shift;          // locator over key bins: bin = (key - lo) >> shift
  int vbins;          // locator over value bins: bin = kNB-1 - (int)((tmax - t(z)) * inv)
  float tmax, inv;    //   with t(z) = z*chi - R
  float chi;          // log2(e) / T (leading part)
  float R;            // the row's reference exponent
  DF S, thr;          // row normaliser and top_p * S
  DF A;               // mass above hi (exact, summed by the last pass)
  uint32_t kx;        // key of the draft token's logit in this row
  // result
  uint32_t kstar;  // cut key
  int cstar;       // tokens with the cut key
  int nk;          // of which the first nk in index order are kept
  int lt;          // tokens with key kx and an index below the draft token's
  DF E;            // kept mass
};

struct Shared {
  // top-p
  TopSel ts[2];
  int selbin[2], lowbin[2], sel_cnt[2];
  DF sel_excl[2];
  DF wab[2][kWarps];
  RowAcc w_t[kWarps], w_d[kWarps];  // per-warp partials of the row pass
  uint32_t rcnt[kMaxRounds];
  uint32_t ccnt[kCmax];
  int tcut, rrem, xtok;
  // all-gather slots, indexed by the writing CTA's rank
  RowAcc g_t[kCmax], g_d[kCmax];
  DF g_w[kCmax];
  int g_m[kCmax];
  // per-warp partials
  DF rtot[kMaxRounds];
  DF scan[kWarps];
  int r_i[kWarps];
  float wR[kWarps];  // draft sampler: each warp's reference exponent after the row pass
  // item scalars, written by one thread and read by the whole CTA
  RowAcc row_t, row_d;
  DF S_w, rem;
  int skip, moot;
  uint32_t lth[2];          // this CTA's floor of the unit lists, per row
  uint32_t g_th[kCmax][2];  // all-gather of every CTA's lth
  // candidates above the cluster's floor (top-p): this CTA's count, every
  // CTA's offset, the total, whether the exact cut came from them, the cut's
  // rank and the key range of the cut key; the draw's location
  uint32_t ucnt[2], uoff[2][kCmax], utot[2], ukmax[2];
  int uok[2], ubelow[2], ucut[2], ua[2], ub[2], ult[2];
  DF uE[2];
  int ypos, ylast;
  int fin;
  int owner, rsel;
  int x;
  float u_i, zt_x, zd_x, uK;
  float dq[3];  // p'(x), q'(x) and their ratio, for the diagnostics
  uint32_t eb;  // the item's verdict: error bits, rejection
  int rej;
  // the item's two row slices (the same in every thread of the CTA), for the
  // out-of-line selection and tie helpers: read through a pointer, they take
  // no per-thread stack copies; both element sizes share one layout
  RowSlice<4> rsl[2];
};

// An earlier position of the sequence has been rejected (or failed) in the
// sequence word w: item i cannot change the result.
__device__ __forceinline__ bool word_moot(unsigned long long w, int i) {
  const unsigned long long R = ((w >> kWordBits) | (w >> (2 * kWordBits))) & ((1ull << kWordBits) - 1);
  return (R & ((1ull << i) - 1)) != 0;
}

__device__ bool resolvable(unsigned long long w, int kb, int* j_out, bool* err) {
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

constexpr int kYBad = -2;  // a draw whose uniform was outside [0, 1)

__device__ void write_outputs(const VerifyParams& P, int b, int n, int y, bool err);

// Outputs of sampled sequence b with the draw y at its cut j (error outputs
// if the draw's uniform was bad).
__device__ void emit_sampled(const VerifyParams& P, int b, int j, int y);

__device__ __forceinline__ uint32_t or_acqrel32(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.or.b32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ unsigned long long or_acqrel64(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.or.b64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

__device__ __forceinline__ unsigned long long or_acq64(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acquire.gpu.global.or.b64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

__device__ bool resolvable(unsigned long long w, int kb, int* j_out, bool* err);

// A sampled sequence's outputs need its prefix resolved (bit 0 of its second
// word, set by the item whose publication completed the prefix) and the draw
// at its cut j stored (bit 1 + j, set by item j after its draw).  Each side
// sets its bit with one atomic; the one that finds the other bit already set
// writes the outputs, so exactly one does.
__device__ void prefix_resolved(const VerifyParams& P, int b, int j) {
  const uint32_t old = or_acqrel32(P.words2 + b, 1u);
  if (old & (1u << (1 + j))) emit_sampled(P, b, j, __ldcg(&P.stats[(size_t)b * (P.K + 1) + j].y));
}

__device__ void draw_ready(const VerifyParams& P, int b, int i, int kb, int y) {
  P.stats[(size_t)b * (P.K + 1) + i].y = y;
  const uint32_t old = or_acqrel32(P.words2 + b, 1u << (1 + i));
  if (old & 1u) {  // prefix already resolved: emit if this position is the cut
    int j;
    bool err;
    const unsigned long long w = or_acqrel64(P.words + b, 0ull);
    if (resolvable(w, kb, &j, &err) && !err && j == i) emit_sampled(P, b, i, y);
  }
}

__device__ void emit_sampled(const VerifyParams& P, int b, int j, int y) {
  if (y == kYBad) {
    write_outputs(P, b, 0, -1, true);
    atomicOr(P.flags, SV_FLAG_BAD_UNIFORM);
  } else {
    write_outputs(P, b, j, y, false);
  }
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
// Cluster helpers (a cluster of one CTA synchronises and addresses locally)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void csync(cg::cluster_group& cluster, int C) {
  if (C > 1) cluster.sync();
  else __syncthreads();
}

template <typename T>
__device__ __forceinline__ T* remote(cg::cluster_group& cluster, int C, T* p, int q) {
  return C > 1 ? cluster.map_shared_rank(p, q) : p;
}

// ---------------------------------------------------------------------------
// Top-p selection [FS §3.2]: keep a token iff the mass ranked strictly before
// it is at most top_p * S.  The mass ranked before a token is the mass of all
// larger keys plus that of the equal keys at smaller indices, so the kept set
// is every key above a cut key k*, and the first nk tokens (index order) of
// key k*.  The search narrows a key window by passes over the row (re-read
// from L2), every CTA of the cluster counting its own slice.
//
// First window: [key(tau0 point), key(max)], where tau0 = (1 - top_p) S / (2V)
// in e units.  A token whose e lies below tau0 has, ranked before it, every
// token above tau0, of mass > S - V tau0 > top_p S: it is never kept.
// ---------------------------------------------------------------------------
template <int ES>
__device__ __forceinline__ void sel_set_mode(TopSel& t, bool value_bins) {
  const uint32_t span = t.hi - t.lo;
  t.vbins = 0;
  if (span < (uint32_t)kNB) {
    t.mode = 1;
    t.shift = 0;
  } else {
    t.mode = 2;
    t.shift = (32 - __clz(span)) - 11;  // (span >> shift) < kNB
    if (value_bins) {
      const float tmax = __fmaf_rn(bits_val<ES>(key_bits<ES>(t.hi)), t.chi, -t.R);
      const float tmin = __fmaf_rn(bits_val<ES>(key_bits<ES>(t.lo)), t.chi, -t.R);
      const float inv = __fdiv_rn((float)(kNB - 1), tmax - tmin);
      if (tmax > tmin && inv > 0.f && inv < INFINITY) {
        t.vbins = 1;
        t.tmax = tmax;
        t.inv = inv;
      }
    }
  }
}

// Pass parameters of one row, in registers.
struct SelP {
  uint32_t lo, span, kx;
  int shift;
  bool counts, vbins;
  float R, chi, tmax, inv;
  float vfloor;  // value of key lo
  uint32_t floor2;  // bf16: vfloor in both halves
};

__device__ __forceinline__ SelP sel_params(const TopSel& t, int ES) {
  SelP p;
  p.lo = t.lo;
  p.span = t.hi - t.lo;
  p.kx = t.kx;
  p.shift = t.shift;
  p.counts = t.mode == 1;
  p.vbins = t.vbins != 0;
  p.R = t.R;
  p.chi = t.chi;
  p.tmax = t.tmax;
  p.inv = t.inv;
  p.vfloor = ES == 2 ? bits_val<2>(key_bits<2>(t.lo)) : bits_val<4>(key_bits<4>(t.lo));
  const uint32_t fb = ES == 2 ? key_bits<2>(t.lo) : 0u;
  p.floor2 = fb | (fb << 16);
  return p;
}

// Mask of the unit's elements whose value is at least the window's floor
// (bit j = slot j): they are in the window or above it.
template <int ES>
__device__ __forceinline__ uint32_t window_mask(const uint4& v, const SelP& p) {
  if (ES == 2) {
    const __nv_bfloat162 f = *reinterpret_cast<const __nv_bfloat162*>(&p.floor2);
    const uint32_t m0 = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&v.x), f);
    const uint32_t m1 = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&v.y), f);
    const uint32_t m2 = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&v.z), f);
    const uint32_t m3 = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&v.w), f);
    const uint32_t m = (m0 & 0x10001u) | ((m1 & 0x10001u) << 2) | ((m2 & 0x10001u) << 4) |
                       ((m3 & 0x10001u) << 6);
    return (m | (m >> 15)) & 0xffu;
  } else {
    return (__uint_as_float(v.x) >= p.vfloor ? 1u : 0u) | (__uint_as_float(v.y) >= p.vfloor ? 2u : 0u) |
           (__uint_as_float(v.z) >= p.vfloor ? 4u : 0u) | (__uint_as_float(v.w) >= p.vfloor ? 8u : 0u);
  }
}

// The unit's elements in `mask` (slot 0 = element eb): add the mass of the
// ones above the window to *above.  Count pass: count their keys in the
// window, return how many have the draft token's key at a smaller index.
// Locator pass: add their masses to the bins.
// One element (bit pattern, index) of a selection pass: its mass goes to
// *above if its key lies above the window; in the window it is counted (count
// pass) or its mass binned (locator pass).  Returns 1 if a count pass saw the
// draft token's key at a smaller index.
template <int ES>
__device__ __forceinline__ uint32_t sel_key(const SelP& p, unsigned char* h, uint32_t bits, int idx,
                                            int x, const Expo& X, DF* above) {
  const uint32_t key = okey<ES>(bits);
  const uint32_t d = key - p.lo;
  const float z = bits_val<ES>(bits);
  if (d > p.span) {
    if (key > p.lo) df_acc(*above, e2(z, X, -p.R));
  } else if (p.counts) {
    atomicAdd(reinterpret_cast<uint32_t*>(h) + d, 1u);
  } else {
    int bin = (int)(d >> p.shift);
    if (p.vbins)  // bins numbered upward in value, like key bins
      bin = max(0, kNB - 1 - (int)((p.tmax - __fmaf_rn(z, p.chi, -p.R)) * p.inv));
    atomicAdd(reinterpret_cast<float*>(h) + bin, e2(z, X, -p.R));
  }
  return (p.counts && key == p.kx && idx < x) ? 1u : 0u;
}

template <int ES>
__device__ __forceinline__ uint32_t sel_bits(const SelP& p, unsigned char* h, const uint4& v, int eb,
                                             uint32_t mask, int x, const Expo& X, DF* above) {
  uint32_t lt = 0;
  while (mask) {
    const int j = __ffs(mask) - 1;
    mask &= mask - 1u;
    lt += sel_key<ES>(p, h, unit_bits<ES>(v, j), eb + j, x, X, above);
  }
  return lt;
}


// A partial unit at a slice end, as a 16-byte unit: the slots of elements in
// [e0, e1) are set in *valid, the others are zero.
template <int ES>
__device__ __forceinline__ uint4 edge_unit(const RowSlice<ES>& rs, int eb, uint32_t* valid) {
  constexpr int EPU = 16 / ES;
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < EPU; ++j) {
    const int e = eb + j;
    if (e < rs.e0 || e >= rs.e1) continue;
    m |= 1u << j;
    const uint32_t b = rs.bits(e);
    if (ES == 4) w[j] = b;
    else w[j >> 1] |= (j & 1) ? (b << 16) : b;
  }
  *valid = m;
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One selection pass of this thread's warp over one row slice (out of line:
// one copy of the code, with registers of its own).  Each thread marks the
// elements of its units in flight that reach the window; the warp then
// takes the marked elements of all its lanes 32 at a time (the units are
// staged in shared memory), so sparse windows keep every lane busy.
// Returns this thread's lt count and adds its mass above the window to
// *above.
template <int ES>
__device__ __noinline__ uint32_t sel_stream(const TopSel* tp, unsigned char* h, uint4* stage,
                                            const RowSlice<ES> rs, int x, float chi, float clo,
                                            DF* above) {
  constexpr int EPU = 16 / ES;
  static_assert(kSelLoads * EPU <= 32, "one 32-bit mask for the units in flight");
  const SelP p = sel_params(*tp, ES);
  const Expo X{chi, clo};
  const int lane = threadIdx.x & 31;
  uint4* mine = stage + threadIdx.x * kSelLoads;
  const unsigned char* wstage = reinterpret_cast<const unsigned char*>(stage + (threadIdx.x - lane) * kSelLoads);
  const int NU = rs.n_units, b0 = rs.ub0(), b1 = rs.ub1();
  uint32_t lt = 0;
  DF ab = *above;
  // (every lane runs the same number of steps: the shuffles below need all 32)
  const int steps = (NU + kThreads * kSelLoads - 1) / (kThreads * kSelLoads);
  for (int it = 0; it < steps; ++it) {
    const int u0 = threadIdx.x + it * kThreads * kSelLoads;
    uint4 v[kSelLoads];
    uint32_t mall = 0;
#pragma unroll
    for (int k = 0; k < kSelLoads; ++k) {
      const int u = u0 + k * kThreads;
      if (u >= b0 && u < b1) {
        v[k] = ldg_unit(rs, u);
      } else if (u < NU) {  // a partial unit at a slice end
        uint32_t valid;
        v[k] = edge_unit<ES>(rs, rs.ebase0 + u * EPU, &valid);
        mall |= valid << (k * EPU);
      } else {
        v[k] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int k = 0; k < kSelLoads; ++k) {
      const int u = u0 + k * kThreads;
      if (u >= b0 && u < b1) mall |= window_mask<ES>(v[k], p) << (k * EPU);
    }
    // exclusive prefix of the marked counts over the warp
    const int c = __popc(mall);
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += n;
    }
    const int total = __shfl_sync(0xffffffffu, inc, 31);
    if (total == 0) continue;  // (warp-uniform)
    const int ex = inc - c;
    if (mall) {
#pragma unroll
      for (int k = 0; k < kSelLoads; ++k) mine[k] = v[k];
    }
    __syncwarp();
    for (int base = 0; base < total; base += 32) {
      const int q = base + lane;
      // source lane: the last lane whose prefix is <= q
      int L = 0;
#pragma unroll
      for (int step = 16; step >= 1; step >>= 1) {
        const int e_ = __shfl_sync(0xffffffffu, ex, L + step);
        if (e_ <= q) L += step;
      }
      const uint32_t mL = __shfl_sync(0xffffffffu, mall, L);
      const int exL = __shfl_sync(0xffffffffu, ex, L);
      if (q < total) {
        const int bit = (int)__fns(mL, 0u, q - exL + 1);
        const int k = bit / EPU, j = bit % EPU;
        const unsigned char* src = wstage + (size_t)L * kSelLoads * 16 + bit * ES;
        const uint32_t bits = ES == 2 ? (uint32_t)*reinterpret_cast<const uint16_t*>(src)
                                      : *reinterpret_cast<const uint32_t*>(src);
        const int eb = rs.ebase0 + (u0 - lane + L + k * kThreads) * EPU;
        lt += sel_bits<ES>(p, h, make_uint4(bits, 0u, 0u, 0u), eb + j, 1u, x, X, &ab);
      }
    }
    __syncwarp();  // staged units are read before the next step overwrites them
  }
  *above = ab;
  return lt;
}

// Thread t gathers bins [8t, 8t+8) of one row's histogram from every CTA of
// the cluster, in rank order (so every CTA holds the same totals); thread 0
// also gathers the mass above the window and the count pass's lt count.
__device__ __forceinline__ void sel_reduce(cg::cluster_group& cluster, int C, unsigned char* h,
                                           bool counts, uint32_t (&w)[8], uint32_t* lt, DF* above) {
  const int tid = threadIdx.x;
  if (counts) {
    uint32_t a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int q = 0; q < C; ++q) {
      const uint4* p = remote(cluster, C, reinterpret_cast<uint4*>(h) + 2 * tid, q);
      const uint4 x = p[0], y = p[1];
      a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
      a[4] += y.x; a[5] += y.y; a[6] += y.z; a[7] += y.w;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = a[k];
  } else {
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int q = 0; q < C; ++q) {
      const float4* p = remote(cluster, C, reinterpret_cast<float4*>(h) + 2 * tid, q);
      const float4 x = p[0], y = p[1];
      a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
      a[4] += y.x; a[5] += y.y; a[6] += y.z; a[7] += y.w;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(a[k]);
  }
  if (tid == 0) {
    uint32_t l = 0;
    DF ab{0.f, 0.f};
    for (int q = 0; q < C; ++q) {
      uint32_t* r = remote(cluster, C, reinterpret_cast<uint32_t*>(h), q);
      l += r[kSlotLt];
      ab = df_add(ab, DF{__uint_as_float(r[kSlotAbove]), __uint_as_float(r[kSlotAbove + 1])});
    }
    *lt = l;
    *above = ab;
  }
}

// Sum of v over the threads above this one (threadIdx greater), in
// double-float; the same bits in every CTA that scans the same values.
__device__ __forceinline__ DF block_suffix_excl(DF v, DF* wtot, int lane, int warp) {
  DF s = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF n = DF{__shfl_down_sync(0xffffffffu, s.hi, o), __shfl_down_sync(0xffffffffu, s.lo, o)};
    if (lane + o < 32) s = df_add(s, n);
  }
  DF ex = DF{__shfl_down_sync(0xffffffffu, s.hi, 1), __shfl_down_sync(0xffffffffu, s.lo, 1)};
  if (lane == 31) ex = DF{0.f, 0.f};
  if (lane == 0) wtot[warp] = s;
  __syncthreads();
  DF above = DF{0.f, 0.f};
  for (int w = kWarps - 1; w > warp; --w) above = df_add(above, wtot[w]);
  return df_add(above, ex);
}

// The cut lies under the window (or above it): search the rest of the
// feasible range on that side.
template <int ES>
__device__ __forceinline__ void sel_go_below(TopSel& t) {
  t.fhi = t.lo - 1u;
  t.lo = t.flo;
  t.hi = t.fhi;
  sel_set_mode<ES>(t, true);
}

template <int ES>
__device__ __forceinline__ void sel_go_above(TopSel& t) {
  t.flo = t.hi + 1u;
  t.lo = t.flo;
  t.hi = t.fhi;
  sel_set_mode<ES>(t, true);
}

// After a count pass: fix the cut key and how many of its tokens are kept, or
// move to the side of the window that holds the cut.  After a locator pass:
// narrow the window to the bin whose (approximate) mass interval holds
// top_p S; if none does, to the end of the window nearest to it.
template <int ES>
__device__ void sel_resolve(Shared& sh, int r, const uint32_t (&w)[8], uint32_t lt_tot,
                            const Expo& X) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const TopSel s = sh.ts[r];
  const bool cm = s.mode == 1;
  DF m[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    m[q] = DF{0.f, 0.f};
    if (cm) {
      if (w[q]) {
        const uint32_t key = s.lo + (uint32_t)(8 * tid + q);
        const float e = e2(bits_val<ES>(key_bits<ES>(key)), X, -s.R);
        m[q] = df_mul_f(DF{e, 0.f}, (float)w[q]);
      }
    } else {
      m[q] = DF{__uint_as_float(w[q]), 0.f};
    }
  }
  DF T = DF{0.f, 0.f};
#pragma unroll
  for (int q = 0; q < 8; ++q) T = df_add(T, m[q]);
  const DF above = df_add(s.A, block_suffix_excl(T, sh.scan, lane, warp));
  DF run = above;
  int cand = -1, low = 0x7fffffff;
#pragma unroll
  for (int q = 7; q >= 0; --q) {
    if (df_pos(m[q])) {
      const DF inc = df_add(run, m[q]);
      const int g = 8 * tid + q;
      if (cand < 0 && df_gt(inc, s.thr) && !df_gt(run, s.thr)) cand = g;
      low = g;
      run = inc;
    }
  }
  if (cand >= 0) atomicMax(&sh.selbin[r], cand);
  if (low != 0x7fffffff) atomicMin(&sh.lowbin[r], low);
  __syncthreads();
  int bs = sh.selbin[r];
  const bool above_w = df_gt(s.A, s.thr) && s.hi < s.fhi;  // cut above the window
  const bool below = cm && bs < 0 && s.lo > s.flo;          // cut under the window
  if (bs < 0 && !below)  // count pass: nothing below, keep the whole window;
    bs = sh.lowbin[r];   // locator: its lowest bin (the cut is there or lower)
  if (bs >= 0 && bs != 0x7fffffff && bs / 8 == tid) {
    DF run2 = above;
#pragma unroll
    for (int q = 7; q >= 0; --q) {
      if (df_pos(m[q])) {
        if (8 * tid + q == bs) {
          sh.sel_excl[r] = run2;
          sh.sel_cnt[r] = cm ? (int)w[q] : 0;
        }
        run2 = df_add(run2, m[q]);
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    TopSel& t = sh.ts[r];
    if (above_w) {
      // the cut lies above the window (its keys all rank after mass > top_p S)
      sel_go_above<ES>(t);
    } else if (below) {
      sel_go_below<ES>(t);
    } else if (bs < 0 || bs == 0x7fffffff) {
      // no mass where the cut should be (not reachable for a finite row)
      t.mode = 0;
      t.kstar = 0u;
      t.cstar = 0;
      t.nk = 0x7fffffff;
      t.lt = 0;
      t.E = t.S;
    } else if (cm) {
      const uint32_t kk = t.lo + (uint32_t)bs;
      const float es = e2(bits_val<ES>(key_bits<ES>(kk)), X, -t.R);
      const DF excl = sh.sel_excl[r];
      const int c = sh.sel_cnt[r];
      // token n (0-based, index order) of key kk has mass excl + n*es ranked
      // before it: kept iff n <= (thr - excl) / es
      const DF q = df_div(df_sub(t.thr, excl), DF{es, 0.f});
      float f = floorf(q.hi);
      if (f == q.hi && q.lo < 0.f) f -= 1.f;
      const int nk = (f + 1.f >= (float)c) ? c : (f >= 0.f ? (int)f + 1 : 1);
      t.kstar = kk;
      t.cstar = c;
      t.nk = nk;
      t.E = df_add(excl, df_mul_f(DF{es, 0.f}, (float)nk));
      t.lt = (int)lt_tot;
      t.mode = 0;
    } else if (t.vbins) {
      // keys of bin bs with half a bin of margin on each side (the bin edges
      // are recomputed, not stored), one key wider still
      const float rk = (float)(kNB - 1 - bs);  // bin rank from the top of the window
      const float z_top = __fdiv_rn(t.tmax - (rk - 0.5f) / t.inv + t.R, t.chi);
      const float z_bot = __fdiv_rn(t.tmax - (rk + 1.5f) / t.inv + t.R, t.chi);
      uint32_t nhi = t.hi, nlo = t.lo;
      if (z_top < bits_val<ES>(key_bits<ES>(t.hi))) nhi = min(t.hi, okey<ES>(ceil_bits<ES>(z_top)) + 1u);
      if (z_bot > bits_val<ES>(key_bits<ES>(t.lo))) nlo = max(t.lo, okey<ES>(floor_bits<ES>(z_bot)) - 1u);
      if (nlo > nhi) {
        nlo = t.lo;
        nhi = t.hi;
      }
      const bool narrowed = (nhi - nlo) < (t.hi - t.lo) / 2u;
      t.lo = nlo;
      t.hi = nhi;
      sel_set_mode<ES>(t, narrowed);
    } else {
      const unsigned long long nlo = (unsigned long long)t.lo + ((unsigned long long)bs << t.shift);
      unsigned long long nhi = nlo + (1ull << t.shift) - 1ull;
      if (nhi > (unsigned long long)t.hi) nhi = t.hi;
      t.lo = (uint32_t)nlo;
      t.hi = (uint32_t)nhi;
      sel_set_mode<ES>(t, true);
    }
  }
  __syncthreads();
}

// Rank order of candidates (key, index): by key descending, then index
// ascending; "ranked before" is a larger composite.
__device__ __forceinline__ unsigned long long cand_order(uint2 e) {
  return ((unsigned long long)e.x << 32) | (unsigned long long)(~e.y);
}

// Exact top-p cut of each row from its candidates: every token whose key
// exceeds the cluster's list floor theta (sh.ts[r].lth).  Each CTA collects
// the candidates of its slice from the units its threads recorded, every CTA
// gathers all of them (at most kUCap per row), ranks them by (key desc, index
// asc) and walks their masses from the top [FS §3.2]: the first candidate
// whose mass ranked before it exceeds top_p * S is the first dropped token.
// Rows resolved this way get mode 0 and keep the ranked candidates (the kept
// ones are ranks 0 .. ucut - 1) for the draw.  A row whose candidates overflow
// keeps its full window; a row whose candidates are all kept (the cut lies
// at or below theta) gets the window [flo, theta]; both go to the passes.
template <int ES>
__device__ __noinline__ void topp_candidates(const VerifyParams& P, Shared& sh, unsigned char* dyn, int C,
                                             int nrows, const Expo X) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  constexpr int EPU = 16 / ES;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint2* own = reinterpret_cast<uint2*>(dyn);
  uint2* all = reinterpret_cast<uint2*>(dyn + kUAllOff);
  uint2* srt = reinterpret_cast<uint2*>(dyn + kListOff);  // (the unit lists until step 4)
  const uint2* lst = srt;
  if (tid < 2) {
    sh.ucnt[tid] = 0u;
    sh.ukmax[tid] = 0u;
    sh.ucut[tid] = 0x7fffffff;
    sh.ua[tid] = 0x7fffffff;
    sh.ub[tid] = 0;
    sh.ult[tid] = 0;
    sh.uok[tid] = 0;
    sh.ubelow[tid] = 0;
  }
  __syncthreads();
  // 1. the elements above the floor in this thread's recorded units (all of
  //    them are requested before any is examined)
  uint2 e[2][kListLen];
  uint4 v[2][kListLen];
  uint32_t valid[2][kListLen];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint32_t th = sh.ts[r].lth;
    const RowSlice<ES>& rs = *reinterpret_cast<const RowSlice<ES>*>(&sh.rsl[r]);
#pragma unroll
    for (int k = 0; k < kListLen; ++k) {
      e[r][k] = r < nrows ? lst[(r * kListLen + k) * kThreads + tid] : make_uint2(0u, 0u);  // (keys descend; 0 = empty)
      valid[r][k] = 0u;
      v[r][k] = make_uint4(0u, 0u, 0u, 0u);
      const int u = (int)e[r][k].y;
      if (e[r][k].x > th && u >= rs.ub0() && u < rs.ub1()) {
        v[r][k] = ldg_unit(rs, u);
        valid[r][k] = (1u << EPU) - 1u;
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint32_t th = sh.ts[r].lth;
    const RowSlice<ES>& rs = *reinterpret_cast<const RowSlice<ES>*>(&sh.rsl[r]);
    // which elements qualify (bit 8k + j: element j of unit k), then one
    // atomic per warp reserves the warp's places
    uint32_t m[kListLen];
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < kListLen; ++k) {
      m[k] = 0u;
      if (e[r][k].x <= th) continue;
      const int u = (int)e[r][k].y;
      if (!(u >= rs.ub0() && u < rs.ub1())) v[r][k] = edge_unit<ES>(rs, rs.ebase0 + u * EPU, &valid[r][k]);
#pragma unroll
      for (int j = 0; j < EPU; ++j)
        if (((valid[r][k] >> j) & 1u) && okey<ES>(unit_bits<ES>(v[r][k], j)) > th) m[k] |= 1u << j;
      cnt += __popc(m[k]);
    }
    int inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nb = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += nb;
    }
    uint32_t base = 0u;
    if (lane == 31 && inc) base = atomicAdd(&sh.ucnt[r], (uint32_t)inc);
    base = __shfl_sync(0xffffffffu, base, 31) + (uint32_t)(inc - cnt);
#pragma unroll
    for (int k = 0; k < kListLen; ++k) {
      const int eb = rs.ebase0 + (int)e[r][k].y * EPU;
      uint32_t mk = m[k];
      while (mk) {
        const int j = __ffs(mk) - 1;
        mk &= mk - 1u;
        if (base < (uint32_t)kUOwn)
          own[r * kUOwn + base] = make_uint2(okey<ES>(unit_bits<ES>(v[r][k], j)), (uint32_t)(eb + j));
        ++base;
      }
    }
  }
  csync(cluster, C);  // every CTA's candidates are complete
  // 2. every CTA's count: offsets, total, overflow (the same in every CTA)
  if (tid < nrows) {
    uint32_t tot = 0u;
    bool ovf = false;
    for (int q = 0; q < C; ++q) {
      const uint32_t c = *remote(cluster, C, &sh.ucnt[tid], q);
      sh.uoff[tid][q] = tot;
      tot += c;
      ovf |= c > (uint32_t)kUOwn;
    }
    sh.utot[tid] = tot;
    sh.uok[tid] = (!ovf && tot <= (uint32_t)kUCap) ? 1 : 0;
  }
  __syncthreads();
  // 3. gather every CTA's candidates (in rank order of the CTAs; padded with
  //    key 0, which no candidate has, to an even count)
  for (int r = 0; r < nrows; ++r) {
    if (!sh.uok[r]) continue;
    const int n = (int)sh.utot[r], n32 = (n + 1) & ~1;
    for (int i0 = tid; i0 < n32; i0 += kThreads * 2) {
      uint2 got[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // two remote loads in flight per thread
        const int i = i0 + h * kThreads;
        got[h] = make_uint2(0u, 0u);
        if (i < n) {
          int q = 0;
          while (q + 1 < C && (uint32_t)i >= sh.uoff[r][q + 1]) ++q;
          got[h] = remote(cluster, C, own, q)[r * kUOwn + (i - (int)sh.uoff[r][q])];
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h)
        if (i0 + h * kThreads < n32) all[r * kUCap + i0 + h * kThreads] = got[h];
      atomicMax(&sh.ukmax[r], max(got[0].x, got[1].x));  // (padding: key 0)
    }
  }
  __syncthreads();
  // 4. rank: the tokens ranked before a candidate have a larger key, or the
  //    same key at a smaller index; each candidate goes to its rank in srt
  //    (the lists are read: their area takes it).
  //    Every CTA holds all the candidates and ranks them itself with a
  //    counting sort: kRankBins bins uniform in value over (theta, max] (bin
  //    0 the largest values; a bin never holds a candidate ranked after one
  //    of a later bin, since rounding is monotone), their counts and prefix,
  //    each candidate placed in its bin's range of slots, then its place in
  //    the range from a count of the range's candidates ranked before it.
  //    No DSMEM traffic and no cluster barrier.  A row with a bin of more
  //    than kRankGroupMax candidates (or a value range that overflows) takes
  //    the distributed count below.  All of it is decided from values that
  //    are the same in every CTA.
  bool loc[2] = {false, false};
  bool need_dist = false;
  for (int r = 0; r < nrows; ++r) {
    if (!sh.uok[r]) continue;  // (uniform in the cluster)
    const int n = (int)sh.utot[r];
    if (n == 0) {
      loc[r] = true;
      continue;
    }
    const uint32_t kmax = sh.ukmax[r], th = sh.ts[r].lth;
    const float vmax = bits_val<ES>(key_bits<ES>(kmax)), vth = bits_val<ES>(key_bits<ES>(th));
    const float inv = (float)(kRankBins - 1) / (vmax - vth);
    if (kmax <= th || !(inv > 0.f && inv < INFINITY)) {
      need_dist = true;
      continue;
    }
    constexpr int R = kRankBins;
    auto bin_of = [&](uint32_t key) {
      const int b_ = (int)((vmax - bits_val<ES>(key_bits<ES>(key))) * inv);
      return min(max(b_, 0), R - 1);
    };
    uint32_t* cnt = reinterpret_cast<uint32_t*>(dyn + kRankOff);
    uint32_t* st = cnt + kRankBins;
    const uint2* a = all + r * kUCap;
    uint2* out = srt + r * kUCap;
    for (int b_ = tid; b_ < R; b_ += kThreads) cnt[b_] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) atomicAdd(&cnt[bin_of(a[i].x)], 1u);
    __syncthreads();
    bool big = false;
    for (int b_ = tid; b_ < R; b_ += kThreads) big |= cnt[b_] > (uint32_t)kRankGroupMax;
    if (__syncthreads_or(big)) {
      need_dist = true;
      continue;
    }
    {  // exclusive prefix of the counts: thread t takes bins 4t .. 4t+3
      uint32_t v[4], tot_ = 0u;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int b_ = 4 * tid + q;
        v[q] = b_ < R ? cnt[b_] : 0u;
        tot_ += v[q];
      }
      uint32_t inc = tot_;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane == 31) sh.r_i[warp] = (int)inc;
      __syncthreads();
      uint32_t off = inc - tot_;
      for (int w = 0; w < warp; ++w) off += (uint32_t)sh.r_i[w];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int b_ = 4 * tid + q;
        if (b_ < R) st[b_] = off;
        off += v[q];
      }
    }
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {  // (st[b] ends at the end of b's range)
      const uint2 e_ = a[i];
      out[atomicAdd(&st[bin_of(e_.x)], 1u)] = e_;
    }
    __syncthreads();
    // within a bin's range, the rank of a candidate is the count of the
    // range's candidates ranked before it; the ranked row goes through the
    // gathered array (no longer needed) and back
    uint2* tmp = all + r * kUCap;
    for (int x1 = tid; x1 < n; x1 += kThreads) {
      const uint2 v_ = out[x1];
      const unsigned long long cv = cand_order(v_);
      const int b_ = bin_of(v_.x), g = (int)cnt[b_], s0 = (int)st[b_] - g;
      int w_ = s0;
      for (int y = s0; y < s0 + g; ++y) w_ += cand_order(out[y]) > cv ? 1 : 0;
      tmp[w_] = v_;
    }
    __syncthreads();
    for (int x1 = tid; x1 < n; x1 += kThreads) out[x1] = tmp[x1];
    __syncthreads();
    loc[r] = true;
  }
  if (need_dist) {
    // this CTA's candidates of the remaining rows, G adjacent threads each
    // (G divides 32), each counting over a share of the gathered ones
    int cr[2], orr[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int n = (int)sh.utot[r];
      const bool d = r < nrows && sh.uok[r] && !loc[r];
      orr[r] = d ? (int)sh.uoff[r][rank] : 0;
      cr[r] = d ? (rank + 1 < C ? (int)sh.uoff[r][rank + 1] : n) - orr[r] : 0;
    }
    const int items = cr[0] + cr[1];
    int G = 1;
    while (G < 8 && items * G * 2 <= kThreads) G <<= 1;
    for (int base = 0; base < items * G; base += kThreads) {  // (uniform in the CTA)
      const int wi = base + tid, item = wi / G, part = wi % G;
      const bool act = item < items;
      const int r = (act && item >= cr[0]) ? 1 : 0;
      const int n = (int)sh.utot[r], n2 = (n + 1) >> 1, chunk = (n2 + G - 1) / G;
      uint2 e_ = make_uint2(0u, 0u);
      int before = 0;
      if (act) {
        e_ = all[r * kUCap + orr[r] + (r ? item - cr[0] : item)];
        const unsigned long long ce = cand_order(e_);
        const uint4* a2 = reinterpret_cast<const uint4*>(all + r * kUCap);  // two candidates per load
        const int j1 = min(n2, (part + 1) * chunk);
#pragma unroll 4
        for (int j = part * chunk; j < j1; ++j) {
          const uint4 f = a2[j];
          before += cand_order(make_uint2(f.x, f.y)) > ce ? 1 : 0;
          before += cand_order(make_uint2(f.z, f.w)) > ce ? 1 : 0;  // (padding: key 0, never before)
        }
      }
      for (int o = 1; o < G; o <<= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
      if (act && part == 0 && before < n)  // (always < n: the candidates are distinct)
        for (int q = 0; q < C; ++q) remote(cluster, C, srt, q)[r * kUCap + before] = e_;
    }
    csync(cluster, C);  // every rank is placed in every CTA
  }
  // 5. masses in rank order: the first candidate whose exclusive prefix
  //    exceeds top_p * S is the first dropped token
  const int x = sh.xtok;
  for (int r = 0; r < nrows; ++r) {
    if (!sh.uok[r]) continue;  // (uniform in the cluster)
    const int n = (int)sh.utot[r];
    const TopSel& t = sh.ts[r];
    const uint2* a = srt + r * kUCap;
    const int c = kThreads - 1 - tid;  // chunk: ranks 4c .. 4c+3 (the suffix over threads is the prefix over chunks)
    float m[4];
    DF loc{0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = 4 * c + q;
      m[q] = i < n ? e2(bits_val<ES>(key_bits<ES>(a[i].x)), X, -t.R) : 0.f;
      df_acc(loc, m[q]);
    }
    const DF pre = block_suffix_excl(loc, sh.scan, lane, warp);
    DF run = pre;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = 4 * c + q;
      if (i < n && df_gt(run, t.thr)) {
        atomicMin(&sh.ucut[r], i);
        break;
      }
      run = df_add(run, DF{m[q], 0.f});
    }
    __syncthreads();
    const int rc = sh.ucut[r];
    if (rc != 0x7fffffff) {
      const uint32_t kk = a[rc].x;
      if (rc >= 4 * c && rc < 4 * c + 4) {  // this thread's chunk holds the cut: its kept mass
        DF ex = pre;
        for (int q = 0; q < rc - 4 * c; ++q) ex = df_add(ex, DF{m[q], 0.f});
        sh.uE[r] = ex;
      }
      for (int i = tid; i < n; i += kThreads) {
        const uint2 e = a[i];
        if (e.x == kk) {
          atomicMin(&sh.ua[r], i);
          atomicMax(&sh.ub[r], i + 1);
        }
        if (x >= 0 && e.x == t.kx && (int)e.y < x) atomicAdd(&sh.ult[r], 1);
      }
    }
    __syncthreads();
    if (tid == 0) {
      TopSel& w = sh.ts[r];
      if (rc == 0x7fffffff) {  // every candidate kept: the cut lies at or below theta
        sh.uok[r] = 0;
        sh.ubelow[r] = 1;
      } else {
        w.kstar = a[rc].x;
        w.cstar = sh.ub[r] - sh.ua[r];
        w.nk = rc - sh.ua[r];
        w.lt = sh.ult[r];
        w.E = sh.uE[r];
        w.mode = 0;
      }
    }
    __syncthreads();
  }
  csync(cluster, C);  // every CTA has read this CTA's candidates
}

// Top-p cut of the target row (and of the draft row when `two`) of one item.
// Every CTA of the cluster ends with the same sh.ts[] results.
template <int ES>
__device__ __noinline__ void topp_select(const VerifyParams& P, Shared& sh, unsigned char* hist,
                                         int C, int b, int i, int kb, bool two, const Expo X,
                                         const RowAcc& row_t, const RowAcc& row_d) {
  const RowSlice<ES>& st = *reinterpret_cast<const RowSlice<ES>*>(&sh.rsl[0]);
  const RowSlice<ES>& sd = *reinterpret_cast<const RowSlice<ES>*>(&sh.rsl[1]);
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < 2 && (tid == 0 || two)) {
    const int r = tid;
    int x = -1;  // the draft token and its logits, as warp 1 fetched them while the rows streamed
    if (i < kb) {
      x = sh.x;
      if (x < 0 || x >= P.V) x = -1;
    }
    if (r == 0) sh.xtok = x;
    const RowAcc& row = r ? row_d : row_t;
    const RowSlice<ES>& rs = r ? sd : st;
    TopSel t;
    t.lth = 0u;
    for (int q = 0; q < C; ++q) t.lth = max(t.lth, sh.g_th[q][r]);
    t.R = row.R;
    t.S = row.s;
    t.thr = df_mul_f(row.s, P.top_p);
    t.A = DF{0.f, 0.f};
    t.hi = okey<ES>(val_bits<ES>(row.mx));
    const float tau0 = 0.5f * (1.f - P.top_p) * (row.s.hi / (float)P.V);
    const float z0 = __fdiv_rn(__log2f(tau0) + row.R, X.chi);
    uint32_t lo;
    if (!(z0 < row.mx)) lo = t.hi;
    else if (!(z0 > -INFINITY)) lo = 0u;
    else lo = okey<ES>(floor_bits<ES>(z0));
    t.lo = min(lo, t.hi);
    t.flo = t.lo;
    t.fhi = t.hi;
    t.chi = X.chi;
    sel_set_mode<ES>(t, true);
    t.kx = x >= 0 ? okey<ES>(val_bits<ES>(r ? sh.zd_x : sh.zt_x)) : 0u;
    t.kstar = 0u;
    t.cstar = 0;
    t.nk = 0x7fffffff;
    t.lt = 0;
    t.E = row.s;
    sh.ts[r] = t;
  }
  __syncthreads();
  // The exact cut from the candidates above the lists' floor; the rows it
  // leaves open search by passes over the slices.
  topp_candidates<ES>(P, sh, hist, C, two ? 2 : 1, X);
  if (tid < 2 && (tid == 0 || two) && !sh.uok[tid]) {
    TopSel& t = sh.ts[tid];
    if (sh.ubelow[tid] && t.lth >= t.flo && t.lth < t.fhi) {  // every candidate kept: the cut is at or below theta
      t.fhi = t.lth;
      t.hi = t.lth;
    }
    t.lo = t.flo;
    sel_set_mode<ES>(t, true);
  }
  __syncthreads();
  for (int pass = 0; pass < kMaxSelPasses; ++pass) {
    const bool a0 = sh.ts[0].mode != 0, a1 = two && sh.ts[1].mode != 0;
    if (!a0 && !a1) break;
    for (int k = tid; k < kHistBytes / 16; k += kThreads)
      reinterpret_cast<uint4*>(hist)[k] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
      sh.selbin[0] = sh.selbin[1] = -1;
      sh.lowbin[0] = sh.lowbin[1] = 0x7fffffff;
    }
    __syncthreads();
    const int x = sh.xtok;
    const bool c0 = a0 && sh.ts[0].mode == 1, c1 = a1 && sh.ts[1].mode == 1;
    uint32_t l0 = 0, l1 = 0;
    DF ab0{0.f, 0.f}, ab1{0.f, 0.f};
    unsigned char* h1 = hist + kHistRowBytes;
    uint4* stage = reinterpret_cast<uint4*>(hist + kHistBytes);
    if (a0) l0 = sel_stream<ES>(&sh.ts[0], hist, stage, st, x, X.chi, X.clo, &ab0);
    if (a1) l1 = sel_stream<ES>(&sh.ts[1], h1, stage, sd, x, X.chi, X.clo, &ab1);
    // the CTA's lt count (count passes) and mass above the window (fixed order)
    if (c0 && l0) atomicAdd(reinterpret_cast<uint32_t*>(hist) + kSlotLt, l0);
    if (c1 && l1) atomicAdd(reinterpret_cast<uint32_t*>(h1) + kSlotLt, l1);
    ab0 = df_warp_sum(ab0);
    ab1 = df_warp_sum(ab1);
    if (lane == 0) {
      sh.wab[0][warp] = ab0;
      sh.wab[1][warp] = ab1;
    }
    __syncthreads();
    if (tid < 2 && (tid == 0 ? a0 : a1)) {
      DF a{0.f, 0.f};
      for (int q = 0; q < kWarps; ++q) a = df_add(a, sh.wab[tid][q]);
      uint32_t* hc = reinterpret_cast<uint32_t*>(tid ? h1 : hist);
      hc[kSlotAbove] = __float_as_uint(a.hi);
      hc[kSlotAbove + 1] = __float_as_uint(a.lo);
    }
    csync(cluster, C);  // every CTA's histograms are complete
    // one row at a time: gather its totals, then resolve (only this CTA's
    // state changes, so other CTAs may still be reading its histograms)
#pragma unroll 1
    for (int r = 0; r < 2; ++r) {
      if (!(r ? a1 : a0)) continue;  // (uniform in the cluster)
      uint32_t w[8], lt = 0;
      DF A{0.f, 0.f};
      sel_reduce(cluster, C, r ? h1 : hist, r ? c1 : c0, w, &lt, &A);
      if (tid == 0) sh.ts[r].A = A;  // exact mass above the window
      __syncthreads();
      sel_resolve<ES>(sh, r, w, lt, X);
    }
    csync(cluster, C);  // every CTA has read every histogram before they are cleared
  }
}

// Index of token nk (0-based, index order) among the tokens of key kk in a
// row: the first one the top-p cut drops.  Each CTA counts the key per unit
// of its slice; the CTA holding token nk finds its round, unit and element
// and writes the index into every CTA.  0x7fffffff if the row has <= nk.
template <int ES>
__device__ __noinline__ int tie_cut(Shared& sh, uint32_t* iv, int C, int rank, int which,
                                    uint32_t kk, int nk) {
  cg::cluster_group cluster = cg::this_cluster();
  const RowSlice<ES>& rs = *reinterpret_cast<const RowSlice<ES>*>(&sh.rsl[which]);
  constexpr int EPU = 16 / ES;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NU = rs.n_units, rounds = (NU + kThreads - 1) / kThreads;
  const int ub0 = rs.ub0(), ub1 = rs.ub1();
  const float vk = bits_val<ES>(key_bits<ES>(kk));  // units entirely below it hold no token of key kk
  for (int u = tid; u < rounds * kThreads; u += kThreads) {
    uint32_t c = 0;
    if (u >= ub0 && u < ub1) {
      const uint4 v = ldg_unit(rs, u);
      if (unit_max<ES>(v) >= vk) {
#pragma unroll
        for (int j = 0; j < EPU; ++j) c += okey<ES>(unit_bits<ES>(v, j)) == kk ? 1u : 0u;
      }
    } else if (u < NU) {
      const int eb = rs.ebase0 + u * EPU;
      for (int j = 0; j < EPU; ++j) {
        const int e = eb + j;
        if (e >= rs.e0 && e < rs.e1 && okey<ES>(rs.bits(e)) == kk) ++c;
      }
    }
    iv[u] = c;
  }
  __syncthreads();
  for (int r = warp; r < rounds; r += kWarps) {
    uint32_t a = 0;
    for (int t = lane; t < kThreads; t += 32) a += iv[r * kThreads + t];
    a = __reduce_add_sync(0xffffffffu, a);
    if (lane == 0) sh.rcnt[r] = a;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t a = 0;
    for (int r = lane; r < rounds; r += 32) a += sh.rcnt[r];
    a = __reduce_add_sync(0xffffffffu, a);
    if (lane < C) *remote(cluster, C, &sh.ccnt[rank], lane) = a;
  }
  if (tid == 0) sh.tcut = 0x7fffffff;
  csync(cluster, C);
  uint32_t off = 0;
  for (int q = 0; q < rank; ++q) off += sh.ccnt[q];
  const uint32_t mine = sh.ccnt[rank];
  if ((uint32_t)nk >= off && (uint32_t)nk - off < mine) {  // (uniform inside this CTA)
    if (tid == 0) {
      uint32_t rem = (uint32_t)nk - off;
      int r = 0;
      for (; r < rounds - 1; ++r) {
        if (rem < sh.rcnt[r]) break;
        rem -= sh.rcnt[r];
      }
      sh.rsel = r;
      sh.rrem = (int)rem;
    }
    __syncthreads();
    const int r = sh.rsel;
    const uint32_t rem = (uint32_t)sh.rrem;
    const uint32_t v = iv[r * kThreads + tid];
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += n;
    }
    if (lane == 31) sh.r_i[warp] = (int)inc;
    __syncthreads();
    for (int w = 0; w < warp; ++w) inc += (uint32_t)sh.r_i[w];
    if (v > 0 && inc > rem && inc - v <= rem) {
      uint32_t left = rem - (inc - v);  // tokens of key kk to pass over inside this unit
      const int eb = rs.ebase0 + (r * kThreads + tid) * EPU;
      int idx = 0x7fffffff;
      for (int j = 0; j < EPU; ++j) {
        const int e = eb + j;
        if (e < rs.e0 || e >= rs.e1 || okey<ES>(rs.bits(e)) != kk) continue;
        if (left == 0) {
          idx = e;
          break;
        }
        --left;
      }
      for (int q = 0; q < C; ++q) *remote(cluster, C, &sh.tcut, q) = idx;
    }
  }
  csync(cluster, C);
  return sh.tcut;
}

// ---------------------------------------------------------------------------
// Draw of a top-p item whose cuts came from the candidates (one CTA): the
// kept target tokens are the target's ranked candidates 0 .. ucut[0] - 1, so
// the residual max(0, p' - q') (or p' alone) is non-zero on them only.  Each
// takes its weight w = max(0, e_t - rho * e_d) as the row draw computes it
// (e_d from the draft's logit at the token, 0 if the draft's cut drops it),
// and the draw is the inverse CDF of w in index order with the uniform uK.
// ---------------------------------------------------------------------------
template <int ES, bool SAMPLE>
__device__ __noinline__ void draw_candidates(const VerifyParams& P, Shared& sh, unsigned char* dyn, int b,
                                             int kb, int j, float uK, float T, float Rt, float Rd, DF S_t,
                                             DF S_d) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool bonus = (j == kb);
  const Expo X = make_expo(T);
  const uint2* srt = reinterpret_cast<const uint2*>(dyn + kListOff);
  float* wv = reinterpret_cast<float*>(dyn);         // weight of kept candidate i (rank order)
  uint2* byi = reinterpret_cast<uint2*>(dyn + 4 * kUCap);  // (index, weight) in index order
  const int n = sh.ucut[0];
  bool p_only = bonus;
  float rho_hi = 0.f, rho_lo = 0.f;
  if (!p_only) {
    const DF rho = df_div(S_t, S_d);
    rho_hi = rho.hi;
    rho_lo = rho.lo;
  }
  // the draft's cut: key kd, and the first dropped index cd among its tokens
  const bool dcut = !p_only && P.topp_draft;
  const uint32_t kd = dcut ? sh.ts[1].kstar : 0u;
  const int cd = dcut ? (int)srt[kUCap + sh.ucut[1]].y : 0x7fffffff;
  const char* drow = p_only ? nullptr : P.drf + (long long)b * P.d_seq + (long long)j * P.d_pos;
  DF loc{0.f, 0.f};
  for (int i = tid; i < n; i += kThreads) {
    const uint2 e = srt[i];
    const float a = e2(bits_val<ES>(key_bits<ES>(e.x)), X, -Rt);
    float w = a;
    if (!p_only && e.y < (uint32_t)P.V) {
      const uint32_t bd = ES == 2 ? (uint32_t)*reinterpret_cast<const uint16_t*>(drow + (size_t)e.y * 2)
                                  : *reinterpret_cast<const uint32_t*>(drow + (size_t)e.y * 4);
      const uint32_t kyd = okey<ES>(bd);
      const bool keptd = !dcut || kyd > kd || (kyd == kd && (int)e.y < cd);
      const float q = keptd ? e2(bits_val<ES>(bd), X, -Rd) : 0.f;
      w = fmaxf(0.f, __fmaf_rn(-rho_lo, q, __fmaf_rn(-rho_hi, q, a)));
    }
    wv[i] = w;
    df_acc(loc, w);
  }
  DF tot = df_warp_sum(loc);
  if (lane == 0) sh.scan[warp] = tot;
  __syncthreads();
  tot = DF{0.f, 0.f};
  for (int w_ = 0; w_ < kWarps; ++w_) tot = df_add(tot, sh.scan[w_]);
  if (!df_pos(tot) && !p_only) {  // residual all zero: draw from p  [SSD §4.3]
    p_only = true;
    loc = DF{0.f, 0.f};
    __syncthreads();  // (every thread has read sh.scan)
    for (int i = tid; i < n; i += kThreads) {
      const float a = e2(bits_val<ES>(key_bits<ES>(srt[i].x)), X, -Rt);
      wv[i] = a;
      df_acc(loc, a);
    }
    tot = df_warp_sum(loc);
    if (lane == 0) sh.scan[warp] = tot;
    __syncthreads();
    tot = DF{0.f, 0.f};
    for (int w_ = 0; w_ < kWarps; ++w_) tot = df_add(tot, sh.scan[w_]);
  }
  // index order: the position of candidate i among the kept ones
  for (int i = tid; i < n; i += kThreads) {
    const uint32_t v = srt[i].y;
    int before = 0;
#pragma unroll 4
    for (int k = 0; k < n; ++k) before += srt[k].y < v ? 1 : 0;
    byi[before] = make_uint2(v, __float_as_uint(wv[i]));
  }
  if (tid == 0) {
    sh.ypos = 0x7fffffff;
    sh.ylast = -1;
  }
  __syncthreads();
  // inclusive prefix in index order; y = the first token whose prefix passes u * sum(w)
  const DF tgt = df_mul_f(tot, uK);
  const int c = kThreads - 1 - tid;  // chunk: positions 4c .. 4c+3
  float wq[4];
  DF lsum{0.f, 0.f};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = 4 * c + q;
    wq[q] = i < n ? __uint_as_float(byi[i].y) : 0.f;
    df_acc(lsum, wq[q]);
  }
  DF run = block_suffix_excl(lsum, sh.scan, lane, warp);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = 4 * c + q;
    if (i < n && wq[q] > 0.f) {
      run = df_add(run, DF{wq[q], 0.f});
      atomicMax(&sh.ylast, i);
      if (df_gt(run, tgt)) {
        atomicMin(&sh.ypos, i);
        break;
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    int pos = sh.ypos;
    if (pos == 0x7fffffff) pos = sh.ylast;  // past the end by rounding: the last positive weight
    const int y = pos >= 0 ? (int)byi[pos].x : -1;
    if (!SAMPLE && P.diag) {
      float* dg = P.diag + ((size_t)b * (P.K + 1) + j) * SV_DIAG_FIELDS;
      dg[SV_DIAG_S_W] = p_only ? 1.f : df_to_float(df_div(tot, S_t));
    }
    if (SAMPLE) P.out[(size_t)b * P.K + j] = y;
    else draw_ready(P, b, j, kb, y);
  }
}

// The round that holds rem among sh.rtot[0 .. rounds) (first round whose
// inclusive prefix exceeds rem; rounds of zero mass never chosen), found by
// warp 0 with one double-float warp scan per 32 rounds.  Writes sh.rsel and
// the remainder inside that round to sh.rem.  Past the end by rounding: the
// last positive round, just inside its end.  Every lane of warp 0 calls it
// with the same rem.
__device__ __forceinline__ void locate_round(Shared& sh, int rounds, DF rem, int lane) {
  int rsel = -1, rlast = -1;
  DF vlast{0.f, 0.f};
  for (int r0 = 0; r0 < rounds && rsel < 0; r0 += 32) {
    const int r = r0 + lane;
    const DF v = r < rounds ? sh.rtot[r] : DF{0.f, 0.f};
    const DF inc = df_warp_scan(v, lane);
    const unsigned hit = __ballot_sync(0xffffffffu, r < rounds && df_pos(v) && df_gt(inc, rem));
    const unsigned pos = __ballot_sync(0xffffffffu, r < rounds && df_pos(v));
    if (hit) {
      const int l = __ffs(hit) - 1;
      rsel = r0 + l;
      rem = df_sub(rem, df_sub(df_shfl(inc, l), df_shfl(v, l)));
    } else {
      if (pos) {
        const int l = 31 - __clz(pos);
        rlast = r0 + l;
        vlast = df_shfl(v, l);
      }
      rem = df_sub(rem, df_shfl(inc, 31));
    }
  }
  if (rsel < 0) {
    rsel = rlast < 0 ? 0 : rlast;
    rem = df_mul_f(vlast, 0.999999f);
  }
  if (lane == 0) {
    sh.rsel = rsel;
    sh.rem = rem;
  }
}

// ---------------------------------------------------------------------------
// Draw of the resample (or bonus) token of sequence b at position j with the
// uniform uK, made by item j itself right after its verdict.  Every CTA of
// the cluster takes part.  One pass over both rows puts each thread's unit
// sums in shared memory in index order (round r holds units
// r*kThreads .. r*kThreads + kThreads-1); then round totals, the cluster-wide
// owner of u*total, the round, the unit and the element.  The token is
// stored for the sequence's outputs.
// ---------------------------------------------------------------------------
template <int ES, bool TOPP, bool SAMPLE = false>
__device__ __noinline__ void finish(const VerifyParams& P, Shared& sh, float* vals, int C, int rank,
                                    int b, int kb,
                                    float T, int j, float uK, int e0, int e1, float Rt, float Rd,
                                    DF S_t, DF S_d, uint32_t kt, int nkt, int cntt, uint32_t kd,
                                    int nkd, int cntd) {
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool bonus = (j == kb);
  if (TOPP && sh.uok[0] && (bonus || !P.topp_draft || sh.uok[1])) {
    // the cuts came from the candidates, which hold every kept token: one CTA
    // draws from them (no row is read again)
    if (rank == 0)
      draw_candidates<ES, SAMPLE>(P, sh, reinterpret_cast<unsigned char*>(vals), b, kb, j, uK, T, Rt, Rd,
                                  S_t, S_d);
    return;
  }
  const Expo X = make_expo(T);
  PairRead<ES> pr;
  pr.st.init(P.tgt + (long long)b * P.t_seq + (long long)j * P.t_pos, e0, e1);
  if (!bonus) pr.sd.init(P.drf + (long long)b * P.d_seq + (long long)j * P.d_pos, e0, e1);
  else pr.sd = pr.st;
  pr.ub0 = pr.st.ub0();
  pr.ub1 = pr.st.ub1();
  const bool same_phase = pr.st.ebase0 == pr.sd.ebase0;
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
  W.kt = W.kd = 0u;
  W.ct = W.cd = 0x7fffffff;
  W.vkt = -INFINITY;
  if (TOPP) {  // (S_t, S_d are the kept masses here)
    uint32_t* iv = reinterpret_cast<uint32_t*>(vals);
    if (tid == 0) {
      sh.rsl[0] = *reinterpret_cast<const RowSlice<4>*>(&pr.st);
      sh.rsl[1] = *reinterpret_cast<const RowSlice<4>*>(&pr.sd);
    }
    __syncthreads();
    W.kt = kt;
    if (kt != 0u) W.vkt = bits_val<ES>(key_bits<ES>(kt));
    if (nkt < cntt) W.ct = tie_cut<ES>(sh, iv, C, rank, 0, kt, nkt);
    if (!bonus) {
      W.kd = kd;
      if (nkd < cntd) W.cd = tie_cut<ES>(sh, iv, C, rank, 1, kd, nkd);
    }
  }
  const int NU = pr.st.n_units;
  const int rounds = (NU + kThreads - 1) / kThreads;
  DF slice_w{0.f, 0.f};
  for (int pass = 0; pass < 2; ++pass) {
    if (pass) cluster.sync();  // every CTA has read the first pass's slots
    pr.vec = W.p_only || same_phase;
    for (int u0 = tid; u0 < rounds * kThreads; u0 += kThreads * kLoadsInFlight) {
      uint4 vt[kLoadsInFlight], vd[kLoadsInFlight];
#pragma unroll
      for (int k = 0; k < kLoadsInFlight; ++k) {
        vt[k] = vd[k] = make_uint4(0, 0, 0, 0);
        pr.load(u0 + k * kThreads, W, vt[k], vd[k]);
      }
#pragma unroll
      for (int k = 0; k < kLoadsInFlight; ++k) {
        const int u = u0 + k * kThreads;
        if (u < rounds * kThreads) vals[u] = pr.template value<TOPP>(u, W, vt[k], vd[k]);
      }
    }
    __syncthreads();
    for (int r = warp; r < rounds; r += kWarps) {
      DF a{0.f, 0.f};
      for (int t = lane; t < kThreads; t += 32) df_acc(a, vals[r * kThreads + t]);
      a = df_warp_sum(a);
      if (lane == 0) sh.rtot[r] = a;
    }
    __syncthreads();
    if (warp == 0) {
      DF a{0.f, 0.f};
      for (int r = lane; r < rounds; r += 32) a = df_add(a, sh.rtot[r]);
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
  // ---- locate u * total: slice and round (warp 0), unit (block scan), element ----
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
    if (lane == 0) sh.owner = owner;
    if (owner == rank) locate_round(sh, rounds, rem, lane);  // (owner: uniform in the warp)
  }
  __syncthreads();
  if (sh.owner != rank) return;  // (uniform inside this CTA)
  const int rsel = sh.rsel;
  const DF rem = sh.rem;
  // block-wide inclusive prefix of round rsel's unit sums (thread order)
  const float v = vals[rsel * kThreads + tid];
  const DF wi = df_warp_scan(DF{v, 0.f}, lane);
  if (lane == 31) sh.scan[warp] = wi;
  __syncthreads();
  DF inc = wi;
  for (int w = 0; w < warp; ++w) inc = df_add(sh.scan[w], inc);
  int cand = (v > 0.f && df_gt(inc, rem)) ? tid : 0x7fffffff;
  int lastpos = v > 0.f ? tid : -1;
  cand = warp_min(cand);
  lastpos = -warp_min(-lastpos);
  __syncthreads();
  if (lane == 0) {
    sh.r_i[warp] = cand;
    sh.scan[warp].hi = __int_as_float(lastpos);
  }
  __syncthreads();
  int tsel = 0x7fffffff, tlast = -1;
  for (int w = 0; w < kWarps; ++w) {
    tsel = min(tsel, sh.r_i[w]);
    tlast = max(tlast, __float_as_int(sh.scan[w].hi));
  }
  const bool past_end = tsel == 0x7fffffff;  // rounding: the last positive unit
  if (past_end) tsel = tlast < 0 ? 0 : tlast;
  if (tid != tsel) return;
  constexpr int EPU = 16 / ES;
  const int u = rsel * kThreads + tid;
  DF cum = past_end ? DF{0.f, 0.f} : df_sub(inc, DF{v, 0.f});
  int y = -1, ylast = -1;
  const int eb = pr.st.ebase0 + u * EPU;
  for (int q = 0; q < EPU; ++q) {
    const int e = eb + q;
    if (e < pr.st.e0 || e >= pr.st.e1) continue;
    const float wv = pr.template elem_w<TOPP>(e, W);
    if (wv > 0.f) ylast = e;
    cum = df_add(cum, DF{wv, 0.f});
    if (!past_end && wv > 0.f && df_gt(cum, rem)) {
      y = e;
      break;
    }
  }
  if (y < 0) y = ylast;
  if (SAMPLE) P.out[(size_t)b * P.K + j] = y;  // a draft token: written at once
  else draw_ready(P, b, j, kb, y);
}

// Verdict of one item: its error bits and whether x_i is rejected.  Every
// CTA of the cluster computes it (thread 0) from values that are identical in
// all of them, and gets the same answer; *dq receives p'(x), q'(x) and the
// ratio for the diagnostics.
template <int ES, bool TOPP>
__device__ __noinline__ void judge(const VerifyParams& P, Shared& sh, int i, int kb, bool greedy,
                                   bool has_draft, const Expo X, const RowAcc& row_t,
                                   const RowAcc& row_d, bool bad_t, bool bad_d, float* dq) {
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
      // Under top-p, S is the kept mass and a dropped token has probability 0.
      DF Et = row_t.s, Ed = row_d.s;
      bool keep_t = true, keep_d = true;
      if (TOPP) {
        const TopSel& a = sh.ts[0];
        Et = a.E;
        keep_t = a.kx > a.kstar || (a.kx == a.kstar && a.lt < a.nk);
        if (P.topp_draft) {  // (else the draft keeps its untruncated softmax)
          const TopSel& d = sh.ts[1];
          Ed = d.E;
          keep_d = d.kx > d.kstar || (d.kx == d.kstar && d.lt < d.nk);
        }
      }
      const float lt = (zt_x - row_t.mx) * X.chi, ld = (zd_x - row_d.mx) * X.chi;
      float r;
      if (!keep_t || !keep_d || !(ld > -1074.f) || !(lt > -1074.f)) {
        r = 0.f;
      } else {
        const float a = zt_x - zd_x;
        const float ex = __fmaf_rn(a, X.chi, a * X.clo) + (row_d.R - row_t.R);
        r = ex2(ex) * df_to_float(df_div(Ed, Et));
      }
      diag_px = keep_t ? ex2(earg(zt_x, X, row_t.R)) / Et.hi : 0.f;
      diag_qx = keep_d ? ex2(earg(zd_x, X, row_d.R)) / Ed.hi : 0.f;
      diag_r = r;
      reject = !(u_i < r);
    }
  }
  sh.eb = errbits;
  sh.rej = reject ? 1 : 0;
  dq[0] = diag_px;
  dq[1] = diag_qx;
  dq[2] = diag_r;
}

// Publication of an item's verdict in the sequence word (rank 0, thread 0).
// Returns 1 if it completes the sequence's prefix, with the cut position and
// whether it is an error in *j_out / *err_out; *moot_out tells whether an
// earlier position had already been rejected or failed.
template <bool TOPP>
__device__ __noinline__ int publish(const VerifyParams& P, Shared& sh, int i, int b, int kb,
                                    bool greedy, bool has_draft, const Expo X,
                                    const RowAcc& row_t, const RowAcc& row_d, bool bad_t,
                                    bool bad_d, uint32_t errbits, bool reject, const float* dq,
                                    int* j_out, int* err_out, bool* moot_out) {
  // Only a position that can be the cut (an error, a rejection, or k_b) has
  // statistics that another item reads; the others publish without release.
  const bool cut_here = errbits != 0u || reject || i == kb;
  if (cut_here) {
    ItemStats s;
    s.argmax = row_t.amax;
    s.errbits = errbits;
    s.y = -1;
    s.pad = 0;
    P.stats[(size_t)b * (P.K + 1) + i] = s;
  }
  const bool sel = TOPP && !greedy && !bad_t && !bad_d;
  if (P.diag) {
    float* dg = P.diag + ((size_t)b * (P.K + 1) + i) * SV_DIAG_FIELDS;
    dg[SV_DIAG_M_T] = row_t.mx;
    if (greedy) {
      dg[SV_DIAG_ARGMAX] = (float)row_t.amax;
    } else if (!bad_t) {
      // normaliser relative to the row max: S_R * 2^(R - m*c)
      dg[SV_DIAG_S_T] = df_to_float(row_t.s) * ex2(-earg(row_t.mx, X, row_t.R));
      dg[SV_DIAG_MASS_T] = sel ? df_to_float(df_div(sh.ts[0].E, row_t.s)) : 1.f;
      if (has_draft && !bad_d) {
        dg[SV_DIAG_M_D] = row_d.mx;
        dg[SV_DIAG_S_D] = df_to_float(row_d.s) * ex2(-earg(row_d.mx, X, row_d.R));
        dg[SV_DIAG_MASS_D] = sel && P.topp_draft ? df_to_float(df_div(sh.ts[1].E, row_d.s)) : 1.f;
        dg[SV_DIAG_P_X] = dq[0];
        dg[SV_DIAG_Q_X] = dq[1];
        dg[SV_DIAG_RATIO] = dq[2];
      }
    }
  }
  unsigned long long bits = 1ull << i;
  if (errbits) bits |= 1ull << (2 * kWordBits + i);
  else if (reject) bits |= 1ull << (kWordBits + i);
  // release: this item's statistics are visible before its bits; acquire:
  // the outputs then see the statistics every earlier item released
  const unsigned long long old = cut_here ? or_acqrel64(P.words + b, bits) : or_acq64(P.words + b, bits);
  *moot_out = word_moot(old, i);
  int j0, j1;
  bool e0_, e1_;
  const bool was = resolvable(old, kb, &j0, &e0_);
  const bool now = resolvable(old | bits, kb, &j1, &e1_);
  *j_out = j1;
  *err_out = e1_ ? 1 : 0;
  return (!was && now) ? 1 : 0;
}

// Record unit u, whose max has key `key`, in this thread's list of row r; a
// full list's floor goes to the CTA's floor T.  Returns the thread's new
// admission threshold (value).
template <int ES>
__device__ __forceinline__ float list_unit(Shared& sh, uint2* lst, int r, uint32_t key, int u, float thr) {
  uint2 cur = make_uint2(key, (uint32_t)u);
  uint2* base = lst + (size_t)r * kListLen * kThreads + threadIdx.x;
#pragma unroll
  for (int k = 0; k < kListLen; ++k) {  // insertion from the top (empty slots hold key 0)
    const uint2 e = base[k * kThreads];
    if (cur.x > e.x) {
      base[k * kThreads] = cur;
      cur = e;
    }
  }
  const uint32_t f = base[(kListLen - 1) * kThreads].x;
  if (f) {
    atomicMax(&sh.lth[r], f);
    thr = fmaxf(thr, key_val<ES>(f));
  }
  return thr;
}

template <int ES, bool LISTS = false>
__device__ __forceinline__ void row_unit_v(RowAcc& a, const RowSlice<ES>& rs, int u, int ub0,
                                           int ub1, const uint4& v, bool greedy, const Expo& x,
                                           Shared* sh = nullptr, uint2* lst = nullptr, int r = 0,
                                           float* thr = nullptr) {
  constexpr int EPU = 16 / ES;
  const int eb = rs.ebase0 + u * EPU;
  if (u >= ub0 && u < ub1) {
    if (greedy) {
      greedy_unit<ES>(a, v, eb);
    } else {
      const float g = sampled_unit<ES, LISTS>(a, v, x);
      if (LISTS && g > *thr) *thr = list_unit<ES>(*sh, lst, r, okey<ES>(val_bits<ES>(g)), u, *thr);
    }
  } else if (u < rs.n_units) {
    float g = -INFINITY;  // (a partial unit's max over its valid elements)
    for (int j = 0; j < EPU; ++j) {
      const int e = eb + j;
      if (e < rs.e0 || e >= rs.e1) continue;
      const float z = rs.elem(e);
      if (greedy) {
        greedy_elem(a, z, e);
      } else {
        sampled_elem(a, z, x);
        g = fmaxf(g, z);
      }
    }
    if (LISTS && !greedy && g > *thr) *thr = list_unit<ES>(*sh, lst, r, okey<ES>(val_bits<ES>(g)), u, *thr);
  }
}

// Seeds the reference exponent of a sampled row, before anything is summed,
// from the largest logit among the warp's first-step units (kLoadsInFlight
// aligned units per lane, in this lane's slots).  Each lane raises its own
// reference whenever one of its units goes above it; started from kRnone, a
// lane would raise at most of its first units (a new running maximum is
// frequent early), and a warp runs the raise path whenever any of its lanes
// takes it.  From the warp's maximum over 64 units, a later unit rises above
// the reference rarely.  Every lane of the warp must call this.
template <int ES>
__device__ __forceinline__ void seed_reference(RowAcc& a, const uint4* slot, int u0, int ub0, int ub1,
                                               const Expo& x) {
  float g = -INFINITY;
#pragma unroll
  for (int k = 0; k < kLoadsInFlight; ++k) {
    const int u = u0 + k * kThreads;
    if (u >= ub0 && u < ub1) g = fmaxf(g, unit_max_num<ES>(slot[k * kThreads]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) g = fmaxf(g, __shfl_xor_sync(0xffffffffu, g, o));
  const float gc = g * x.chi;
  if (gc > -INFINITY && gc < INFINITY) a.R = ceilf(gc);  // (else kRnone: the units raise it)
}

// Streams this CTA's slices of both rows through the per-thread cp.async ring
// and reduces them into at / ad (row pass of a1 and a3).  With MOOT, every
// other step each thread looks at the sequence word and stops reading once
// an earlier position of the sequence is rejected (it then sets sh.moot).
// With LISTS (top-p instances, sampled rows), each thread also keeps its
// candidate lists in lst, and sh.lth[r] ends as the CTA's floor of row r.
template <int ES, bool MOOT, bool LISTS = false>
__device__ __forceinline__ void stream_slices(const VerifyParams& P, Shared& sh, float* vals,
                                              const RowSlice<ES>& st, const RowSlice<ES>& sd,
                                              bool has_draft, bool greedy, bool skip, const Expo& X,
                                              int b, int i, RowAcc& at, RowAcc& ad,
                                              uint2* lst = nullptr) {
  const int tid = threadIdx.x;
  const bool lists = LISTS && !greedy;
  // list admission thresholds (values); the draft row keeps no list when
  // the call leaves the draft untruncated
  float thr0 = -INFINITY, thr1 = P.topp_draft ? -INFINITY : INFINITY;
  if (lists) {
#pragma unroll
    for (int k = 0; k < 2 * kListLen; ++k) lst[k * kThreads + tid] = make_uint2(0u, 0u);
  }
  {
    // Each thread keeps NS steps of its units in flight in its own
    // shared-memory slots (slot k of stage s: ring[(s*2L + k)*kThreads + tid],
    // k < L target, k >= L draft) and reduces the oldest step from there.
    constexpr int L = kLoadsInFlight;
    constexpr int kStep = kThreads * L;
    constexpr int kStage = 2 * L * kThreads;  // slots per stage
    constexpr int NS = kRingStages;           // stages
    uint4* ring = reinterpret_cast<uint4*>(vals);
    const int NU = has_draft ? max(st.n_units, sd.n_units) : st.n_units;
    const int tb0 = st.ub0(), tb1 = st.ub1(), db0 = sd.ub0(), db1 = sd.ub1();
    const int nsteps = (!skip && NU > tid) ? (NU - tid + kStep - 1) / kStep : 0;
    // Interior steps (every unit of the step inside the aligned bodies of
    // both rows) take a path without per-unit bounds checks.
    const int in0 = has_draft ? max(tb0, db0) : tb0, in1 = has_draft ? min(tb1, db1) : tb1;
    const char* gt = reinterpret_cast<const char*>(st.base16) + 16 * (size_t)tid;
    const char* gd = reinterpret_cast<const char*>(sd.base16) + 16 * (size_t)tid;
    auto interior = [&](int u0) { return u0 >= in0 && u0 + (L - 1) * kThreads < in1; };
    auto issue = [&](int n) {  // copies of step n into stage n % NS (one group)
      const int u0 = tid + n * kStep;
      uint4* slot = ring + (size_t)(n % NS) * kStage + tid;
      if (interior(u0)) {
        const char* pt = gt + (size_t)n * kStep * 16;
#pragma unroll
        for (int k = 0; k < L; ++k) cp_async16(slot + k * kThreads, pt + (size_t)k * kThreads * 16);
        if (has_draft) {
          const char* pd = gd + (size_t)n * kStep * 16;
#pragma unroll
          for (int k = 0; k < L; ++k)
            cp_async16(slot + (L + k) * kThreads, pd + (size_t)k * kThreads * 16);
        }
      } else {
#pragma unroll
        for (int k = 0; k < L; ++k) {
          const int u = u0 + k * kThreads;
          if (u >= tb0 && u < tb1)
            cp_async16(slot + k * kThreads, reinterpret_cast<const void*>(st.base16 + 16 * (uintptr_t)u));
          if (has_draft && u >= db0 && u < db1)
            cp_async16(slot + (L + k) * kThreads, reinterpret_cast<const void*>(sd.base16 + 16 * (uintptr_t)u));
        }
      }
      cp_async_commit();
    };
    if (!skip) {
#pragma unroll
      for (int n = 0; n < NS; ++n) issue(n);
      // (every lane is here: the references start from the warp's first step)
      cp_async_wait<NS - 1>();
      if (!greedy) seed_reference<ES>(at, ring + tid, tid, tb0, tb1, X);
      if (has_draft) seed_reference<ES>(ad, ring + L * kThreads + tid, tid, db0, db1, X);
    }
    // the sequence word, read two steps before it is looked at (no stall)
    unsigned long long wseen = (MOOT && i > 0 && !skip) ? __ldcg(P.words + b) : 0ull;
    for (int n = 0; n < nsteps; ++n) {
      if (LISTS && lists) {  // the CTA's floors may have risen: admit only above them
        thr0 = fmaxf(thr0, key_val<ES>(sh.lth[0]));
        thr1 = fmaxf(thr1, key_val<ES>(sh.lth[1]));
      }
      // every other step each thread looks again whether an earlier
      // position has been rejected meanwhile; if so it stops reading (the
      // item is then moot, and the cluster drops it after the combine).  A
      // plain per-thread load: the lanes of a warp may leave this loop at
      // different steps, so no warp-synchronous operation may sit in it.
      if (MOOT && i > 0 && (n & 1)) {
        if (word_moot(wseen, i)) {
          sh.moot = 1;  // (a plain store: read after the barriers below)
          break;
        }
        wseen = __ldcg(P.words + b);
      }
      cp_async_wait<NS - 1>();  // this thread's step n has landed
      const int u0 = tid + n * kStep;
      const uint4* slot = ring + (size_t)(n % NS) * kStage + tid;
      // units are read from the slots one at a time (the ring, not registers,
      // holds the step)
      if (interior(u0)) {
        constexpr int EPU = 16 / ES;
#pragma unroll
        for (int k = 0; k < L; ++k) {
          const uint4 vt = slot[k * kThreads];
          if (greedy) {
            greedy_unit<ES>(at, vt, st.ebase0 + (u0 + k * kThreads) * EPU);
          } else {
            const float g = sampled_unit<ES, LISTS>(at, vt, X);
            if (LISTS && g > thr0) thr0 = list_unit<ES>(sh, lst, 0, okey<ES>(val_bits<ES>(g)), u0 + k * kThreads, thr0);
          }
        }
        if (has_draft) {
#pragma unroll
          for (int k = 0; k < L; ++k) {
            const uint4 vd = slot[(L + k) * kThreads];
            const float g = sampled_unit<ES, LISTS>(ad, vd, X);
            if (LISTS && g > thr1) thr1 = list_unit<ES>(sh, lst, 1, okey<ES>(val_bits<ES>(g)), u0 + k * kThreads, thr1);
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < L; ++k) {
          const int u = u0 + k * kThreads;
          const uint4 vt = (u >= tb0 && u < tb1) ? slot[k * kThreads] : make_uint4(0, 0, 0, 0);
          row_unit_v<ES, LISTS>(at, st, u, tb0, tb1, vt, greedy, X, &sh, lst, 0, &thr0);
          if (has_draft) {
            const uint4 vd = (u >= db0 && u < db1) ? slot[(L + k) * kThreads] : make_uint4(0, 0, 0, 0);
            row_unit_v<ES, LISTS>(ad, sd, u, db0, db1, vd, false, X, &sh, lst, 1, &thr1);
          }
        }
      }
      if (!greedy) acc_flush(at);
      if (has_draft) acc_flush(ad);
      issue(n + NS);  // (the slots were consumed above)
    }
    cp_async_wait_all();
  }
  if (!greedy) acc_finish_max<ES>(at);
  if (has_draft) acc_finish_max<ES>(ad);
  if (lists) {  // the recorded units come back in the selection: have them in L2
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const RowSlice<ES>& rs = r ? sd : st;
#pragma unroll
      for (int k = 0; k < kListLen; ++k) {
        const uint2 e = lst[(r * kListLen + k) * kThreads + tid];
        if (e.x != 0u && (r == 0 || has_draft) && (int)e.y >= rs.ub0() && (int)e.y < rs.ub1())
          asm volatile("prefetch.global.L2 [%0];" ::"l"(rs.base16 + 16 * (uintptr_t)e.y));
      }
    }
  }
}

// Combines the row accumulators: lanes, warps, then the CTAs of the cluster
// (every CTA ends with the same bits in sh.row_t / sh.row_d).  Returns true,
// uniformly in the cluster, if any CTA skipped or stopped its rows because an
// earlier position of the sequence was rejected.
__device__ __forceinline__ bool combine_rows(Shared& sh, cg::cluster_group& cluster, int C, int rank,
                                             const RowAcc& at, const RowAcc& ad, bool greedy,
                                             bool has_draft, bool skip) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // ---- combine: lanes -> warps (butterflies) -> CTA (warp 0) -> cluster ----
  // (a CTA that skipped its rows has nothing to combine; skip is uniform in
  // the CTA)
  if (!skip) {
    const RowAcc wt = lanes_combine(at, true, greedy);
    const RowAcc wd = has_draft ? lanes_combine(ad, true, false) : acc_init();
    if (lane == 0) {
      sh.w_t[warp] = wt;
      sh.w_d[warp] = wd;
    }
    __syncthreads();
  }
  if (warp == 0) {
    RowAcc ct = acc_init(), cd = acc_init();
    if (!skip) {
      // (the butterfly covers lanes 0..kWarps-1; lane 0's result goes to
      // every lane, since lane q sends it to CTA q below)
      ct = acc_bcast0(lanes_combine(lane < kWarps ? sh.w_t[lane] : acc_init(), lane < kWarps, greedy, kWarps));
      if (has_draft)
        cd = acc_bcast0(lanes_combine(lane < kWarps ? sh.w_d[lane] : acc_init(), lane < kWarps, false, kWarps));
    }
    // this CTA's moot flag: the word it saw at the start, or at the last
    // step it looked (any thread)
    const int m = (sh.skip | sh.moot) ? 1 : 0;
    const uint32_t th0 = sh.lth[0], th1 = sh.lth[1];  // (complete: the barrier above)
    if (C > 1) {
      if (lane < C) {
        *cluster.map_shared_rank(&sh.g_t[rank], lane) = ct;
        *cluster.map_shared_rank(&sh.g_d[rank], lane) = cd;
        *cluster.map_shared_rank(&sh.g_m[rank], lane) = m;
        uint32_t* g = cluster.map_shared_rank(&sh.g_th[rank][0], lane);
        g[0] = th0;
        g[1] = th1;
      }
    } else if (lane == 0) {
      sh.row_t = ct;
      sh.row_d = cd;
      sh.g_m[0] = m;
      sh.g_th[0][0] = th0;
      sh.g_th[0][1] = th1;
    }
  }
  if (C > 1) cluster.sync();
  else __syncthreads();
  {
    // moot if any CTA saw an earlier rejection (the same OR in every CTA)
    int m = 0;
    for (int r = 0; r < C; ++r) m |= sh.g_m[r];
    if (m) return true;  // (uniform in the cluster; no distributed access follows)
  }
  if (C > 1) {
    if (warp == 0) {
      const int W = C <= 2 ? 2 : C <= 4 ? 4 : C <= 8 ? 8 : 16;  // lanes of the butterfly
      const RowAcc rt = lanes_combine(lane < C ? sh.g_t[lane] : acc_init(), lane < C, greedy, W);
      const RowAcc rd = has_draft ? lanes_combine(lane < C ? sh.g_d[lane] : acc_init(), lane < C, false, W)
                                  : acc_init();
      if (lane == 0) {
        sh.row_t = rt;
        sh.row_d = rd;
      }
    }
    __syncthreads();
  }
  return false;
}

template <int ES, bool TOPP>
__global__ void __launch_bounds__(kThreads, 4) verify_kernel(const __grid_constant__ VerifyParams P) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int item = blockIdx.x / C;
  const int i = item / P.B, b = item % P.B;

  extern __shared__ __align__(16) float vals[];  // cp.async ring; draw's unit sums; top-p histograms
  __shared__ Shared sh;

  // ---- per-row parameters (identical in every CTA of the cluster) ----
  const int kb = P.kpr ? P.kpr[b] : P.K;
  const int md = P.mode ? (int)P.mode[b] : 0;
  const float T = P.temp ? P.temp[b] : 1.0f;
  // The launch may overlap the init kernel that clears the sequence words and
  // the flag word: nothing of the workspace or the outputs is touched before
  // this.  The kernel after this one may start launching meanwhile.
  pdl_wait();
  pdl_launch_dependents();
  // the sequence word (thread 0 of every CTA); its latency overlaps the
  // parameter checks
  const unsigned long long w0 = (tid == 0 && i > 0) ? __ldcg(P.words + b) : 0ull;
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

  // ---- an earlier rejection already makes this item moot: no streaming ----
  // Each CTA looks for itself.  The CTAs of a cluster may see different words,
  // so the flag only decides whether this CTA streams; the cluster-wide
  // verdict is the OR of every CTA's flag, formed in the combine below.
  if (tid == 0) {
    sh.skip = word_moot(w0, i) ? 1 : 0;
    sh.moot = 0;
    sh.lth[0] = sh.lth[1] = 0u;
  }
  __syncthreads();
  const bool skip = sh.skip != 0;

  // ---- stream the slices: one pass per row, through the cp.async ring ----
  const int e0 = min(P.V, rank * P.slice_len), e1 = min(P.V, e0 + P.slice_len);
  RowSlice<ES> st, sd;
  st.init(P.tgt + (long long)b * P.t_seq + (long long)i * P.t_pos, e0, e1);
  if (has_draft) sd.init(P.drf + (long long)b * P.d_seq + (long long)i * P.d_pos, e0, e1);
  else sd = st;
  // warp 1 of every CTA: the decision's inputs, fetched while the rows stream
  if (tid == 32 && !skip) {
    int x = -1;
    float u = 0.f, zt = 0.f, zd = 0.f;
    sh.uK = greedy ? 0.f : P.unif[(size_t)b * (P.K + 1) + P.K];
    if (i < kb) {
      x = P.tokens[(size_t)b * P.K + i];
      if (!greedy) u = P.unif[(size_t)b * (P.K + 1) + i];
      if (x >= 0 && x < P.V) {
        zt = st.elem(x);
        if (has_draft) zd = sd.elem(x);
      }
    }
    sh.x = x;
    sh.u_i = u;
    sh.zt_x = zt;
    sh.zd_x = zd;
  }
  RowAcc at = acc_init(), ad = acc_init();
  stream_slices<ES, true, TOPP>(P, sh, vals, st, sd, has_draft, greedy, skip, X, b, i, at, ad,
                                reinterpret_cast<uint2*>(reinterpret_cast<char*>(vals) + kListOff));
  if (combine_rows(sh, cluster, C, rank, at, ad, greedy, has_draft, skip)) return;  // (moot: uniform)
  // Row validity: no NaN, no +inf, not all -inf, exponent range finite.  (The
  // row statistics are read from shared memory from here on: nothing of them
  // stays in registers across the out-of-line calls below.)
  const bool bad_t = !(sh.row_t.mx > -INFINITY && sh.row_t.mx < INFINITY) ||
                     (!greedy && !(sh.row_t.R > kRnone && sh.row_t.R < INFINITY));
  const bool bad_d = has_draft && (!(sh.row_d.mx > -INFINITY && sh.row_d.mx < INFINITY) ||
                                   !(sh.row_d.R > kRnone && sh.row_d.R < INFINITY));
  if (TOPP && !greedy && !bad_t && !bad_d) {
    if (tid == 0) {
      sh.rsl[0] = *reinterpret_cast<const RowSlice<4>*>(&st);
      sh.rsl[1] = *reinterpret_cast<const RowSlice<4>*>(&sd);
    }
    __syncthreads();
    topp_select<ES>(P, sh, reinterpret_cast<unsigned char*>(vals), C, b, i, kb,
                    has_draft && P.topp_draft, X, sh.row_t, sh.row_d);
  }

  // ---- verdict (every CTA), publication (rank 0, one thread) ----
  if (tid == 0) judge<ES, TOPP>(P, sh, i, kb, greedy, has_draft, X, sh.row_t, sh.row_d, bad_t, bad_d, sh.dq);
  __syncthreads();
  const uint32_t eb_i = sh.eb;
  const bool rej = sh.rej != 0;
  // The draw this item owes on a sampled row: the resample at its own
  // rejection, or the bonus at k_b.  It is made now, while the item's rows
  // may still be in L2; it goes unused if an earlier position turns out
  // rejected, and is skipped if one already was when this item published.
  const bool cand = !greedy && eb_i == 0u && (rej || i == kb);
  // A draw reads this CTA's slices again (both rows, or the target's for a
  // bonus).  Streamed a while ago, they have mostly left L2: warp 1 starts a
  // bulk prefetch of the whole slice now, while rank 0 publishes, where the
  // draw's own loads would take one DRAM round trip per step.  (Top-p draws
  // from the kept candidates read no row again.)
  if (!TOPP && cand && (tid >> 5) == 1) {
    l2_prefetch_slice<ES>(st, tid & 31);
    if (i < kb) l2_prefetch_slice<ES>(sd, tid & 31);
  }
  if (rank == 0 && tid == 0) {
    int j1, e1_;
    bool moot_pub;
    const int fin = publish<TOPP>(P, sh, i, b, kb, greedy, has_draft, X, sh.row_t, sh.row_d, bad_t,
                                  bad_d, eb_i, rej, sh.dq, &j1, &e1_, &moot_pub);
    if (fin) {  // this publication resolved the sequence's prefix, cut at j1
      if (e1_) {
        const uint32_t ebj = __ldcg(&P.stats[(size_t)b * (P.K + 1) + j1].errbits);
        write_outputs(P, b, 0, -1, true);
        atomicOr(P.flags, ebj);
      } else if (greedy) {
        const int a = j1 == i ? sh.row_t.amax : __ldcg(&P.stats[(size_t)b * (P.K + 1) + j1].argmax);
        write_outputs(P, b, j1, a, false);
      } else {
        prefix_resolved(P, b, j1);
      }
    }
    if (cand) {
      int draw = moot_pub ? 0 : 1;
      if (draw && !(sh.uK >= 0.f && sh.uK < 1.f)) {
        draw_ready(P, b, i, kb, kYBad);
        draw = 0;
      }
      for (int r = 0; r < C; ++r) *remote(cluster, C, &sh.fin, r) = draw;
    }
  }
  if (!cand) return;  // (uniform in the cluster: no distributed access follows)
  csync(cluster, C);
  if (!sh.fin) return;

  // ======================= this item's draw =======================
  const float uK = sh.uK;
  DF S_t = sh.row_t.s, S_d = sh.row_d.s;
  uint32_t kt = 0u, kd = 0u;
  int nkt = 0x7fffffff, cntt = 0, nkd = 0x7fffffff, cntd = 0;
  if (TOPP) {  // kept masses and cuts of this item's rows
    S_t = sh.ts[0].E;
    kt = sh.ts[0].kstar;
    nkt = sh.ts[0].nk;
    cntt = sh.ts[0].cstar;
    if (i < kb && P.topp_draft) {
      S_d = sh.ts[1].E;
      kd = sh.ts[1].kstar;
      nkd = sh.ts[1].nk;
      cntd = sh.ts[1].cstar;
    }
  }
  finish<ES, TOPP>(P, sh, vals, C, rank, b, kb, T, i, uK, e0, e1, sh.row_t.R, sh.row_d.R, S_t, S_d,
                   kt, nkt, cntt, kd, nkd, cntd);
}

// ---------------------------------------------------------------------------
// The draft sampler's row pass (no top-p): this CTA's slice of one row
// through the per-thread cp.async ring, as in stream_slices, keeping the sum
// 2^(z*c - R) of every pair of adjacent units.  Unit u = tid + n*kStep +
// k*kThreads, so units 2p and 2p+1 are read by lanes 2j and 2j+1 of one warp
// in the same step: the even lane adds its partner's sum (one shuffle) and
// stores pair p = u/2 in uv.  The warp keeps one reference exponent R, so the
// two sums of a pair share it: it is seeded from the warp's first step and
// raised for every lane at once when a unit of any lane sums above
// kRaiseAbove (to ceil(c * the warp's largest value)), which rescales the
// pairs the warp stored before.  (One reference per lane pair rounds the
// weights' arguments a little more finely, but its divergent raise path
// measured 40% slower.)  Every lane takes the same number of steps (units
// past the slice are empty), so the warp's shuffles and votes are converged.
// The warp's final R goes to sh.wR[warp].  Greedy rows keep only their first
// maximum.
// ---------------------------------------------------------------------------
template <int ES>
__device__ __forceinline__ void stream_pairs(Shared& sh, float* vals, const RowSlice<ES>& st, bool greedy,
                                             const Expo& X, RowAcc& at, float* uv) {
  const int tid = threadIdx.x, lane = tid & 31;
  constexpr int L = kLoadsInFlight;
  constexpr int kStep = kThreads * L;
  constexpr int NS = kSampleRingStages;
  constexpr int kStage = L * kThreads;
  constexpr int EPU = 16 / ES;
  uint4* ring = reinterpret_cast<uint4*>(vals);
  const int NU = st.n_units;
  const int nslots = ((NU + 1) / 2 + kThreads - 1) / kThreads * kThreads;
  for (int q = tid; q < nslots; q += kThreads) uv[q] = 0.f;  // (pairs past the slice stay 0)
  const int tb0 = st.ub0(), tb1 = st.ub1();
  const int nsteps = (NU + kStep - 1) / kStep;
  auto issue = [&](int n) {
    uint4* slot = ring + (size_t)(n % NS) * kStage + tid;
#pragma unroll
    for (int k = 0; k < L; ++k) {
      const int u = tid + n * kStep + k * kThreads;
      if (u >= tb0 && u < tb1)
        cp_async16(slot + k * kThreads, reinterpret_cast<const void*>(st.base16 + 16 * (uintptr_t)u));
    }
    cp_async_commit();
  };
#pragma unroll
  for (int n = 0; n < NS; ++n) issue(n);
  cp_async_wait<NS - 1>();
  if (!greedy) seed_reference<ES>(at, ring + tid, tid, tb0, tb1, X);  // (the same R in every lane)
  // the sum of unit u (valid elements only) against reference R
  auto usum = [&](int u, bool full, const uint4& v, float R) {
    if (full) return unit_sumexp<ES>(v, X, R);
    float a = 0.f;
    if (u < NU) {
      const int eb = st.ebase0 + u * EPU;
      for (int j = 0; j < EPU; ++j) {
        const int e = eb + j;
        if (e >= st.e0 && e < st.e1) a += e2(st.elem(e), X, -R);
      }
    }
    return a;
  };
  for (int n = 0; n < nsteps; ++n) {
    cp_async_wait<NS - 1>();  // this thread's step n has landed
    const uint4* slot = ring + (size_t)(n % NS) * kStage + tid;
#pragma unroll
    for (int k = 0; k < L; ++k) {
      const int u = tid + n * kStep + k * kThreads;
      const bool full = u >= tb0 && u < tb1;
      const uint4 v = full ? slot[k * kThreads] : make_uint4(0u, 0u, 0u, 0u);
      if (greedy) {  // (uniform in the CTA)
        if (full) {
          greedy_unit<ES>(at, v, st.ebase0 + u * EPU);
        } else if (u < NU) {
          const int eb = st.ebase0 + u * EPU;
          for (int j = 0; j < EPU; ++j) {
            const int e = eb + j;
            if (e >= st.e0 && e < st.e1) greedy_elem(at, st.elem(e), e);
          }
        }
        continue;
      }
      // the running max (NaN propagates) and the unit's sum
      if (full) {
        if (ES == 2) at.mx2 = bf16x2_max_nan(at.mx2, bf16x2_max_nan(bf16x2_max_nan(v.x, v.y), bf16x2_max_nan(v.z, v.w)));
        else at.mx = nanmax(at.mx, unit_max<ES>(v));
      } else if (u < NU) {
        const int eb = st.ebase0 + u * EPU;
        for (int j = 0; j < EPU; ++j) {
          const int e = eb + j;
          if (e >= st.e0 && e < st.e1) at.mx = nanmax(at.mx, st.elem(e));
        }
      }
      float us = usum(u, full, v, at.R);
      if (__any_sync(0xffffffffu, !(us <= kRaiseAbove))) {  // some lane is above R (rare)
        float g = -INFINITY;
        if (full) {
          g = unit_max_num<ES>(v);
        } else if (u < NU) {
          const int eb = st.ebase0 + u * EPU;
          for (int j = 0; j < EPU; ++j) {
            const int e = eb + j;
            if (e >= st.e0 && e < st.e1) g = fmaxf(g, st.elem(e));
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) g = fmaxf(g, __shfl_xor_sync(0xffffffffu, g, o));
        const float gc = g * X.chi;
        if (gc > at.R) {  // (uniform in the warp)
          const float p = pow2i(at.R - ceilf(gc));
          acc_raise(at, ceilf(gc));
          if (!(lane & 1))  // this lane's pairs so far (slots tid/2 mod kThreads/2)
            for (int q = tid >> 1; q < nslots; q += kThreads / 2) uv[q] *= p;
          us = usum(u, full, v, at.R);
        }
      }
      at.pend += us;
      const float pv = us + __shfl_xor_sync(0xffffffffu, us, 1);
      if (!(lane & 1) && u < NU) uv[u >> 1] = pv;
    }
    if (!greedy) acc_flush(at);
    issue(n + NS);  // (the slots were consumed above)
  }
  cp_async_wait_all();
  if (!greedy) acc_finish_max<ES>(at);
  if (lane == 0) sh.wR[tid >> 5] = at.R;
}

// ---------------------------------------------------------------------------
// The draft sampler's draw without top-p (weights p' alone).  The row pass
// left the sums 2^(z*c - R) of the slice's unit pairs in uv (R: the
// reference of the warp that stored the pair, sh.wR), and the combine left
// every CTA's slice accumulator in sh.g_t.  Every CTA finds, from the same
// values, the slice that holds u*S; the others return at once (nothing
// distributed follows the combine).  The owner brings its sums to the row's
// reference Rrow, then finds the round of kThreads pairs (a warp scan over
// the round totals, 32 rounds at a time), the pair (a block scan of the
// round) and the element (the pair's two units read again, their weights
// 2^(z*c - Rrow) in index order).  The token goes to *out.
// ---------------------------------------------------------------------------
// (the slice comes as scalars: row, [e0, e1), n_units, ebase0 as in RowSlice;
// a struct passed to a call that is not inlined would go through local memory)
template <int ES>
__device__ __noinline__ void sample_draw(Shared& sh, float* uv, int C, int rank, const char* row, int e0,
                                         int e1, int n_units, int ebase0, float chi, float clo, float Rrow,
                                         float uK, int32_t* out) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Expo X{chi, clo};
  if (warp == 0) {  // the owner of u*S among the slices, in rank order
    DF v{0.f, 0.f};
    if (lane < C) {
      const RowAcc g = C > 1 ? sh.g_t[lane] : sh.row_t;
      if (g.R > kRnone) {
        const float p = pow2i(g.R - Rrow);
        v = DF{g.s.hi * p, g.s.lo * p};
      }
    }
    const DF inc = df_warp_scan(v, lane);
    const DF tgt = df_mul_f(df_shfl(inc, 31), uK);
    const unsigned hit = __ballot_sync(0xffffffffu, lane < C && df_pos(v) && df_gt(inc, tgt));
    const unsigned pos = __ballot_sync(0xffffffffu, lane < C && df_pos(v));
    const int owner = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    const DF v_own = df_shfl(v, owner), inc_own = df_shfl(inc, owner);
    // past the end by rounding: the last positive slice, just inside its end
    const DF rem = hit ? df_sub(tgt, df_sub(inc_own, v_own)) : df_mul_f(v_own, 0.999999f);
    if (lane == 0) {
      sh.owner = owner;
      sh.rem = rem;
    }
  }
  __syncthreads();
  if (sh.owner != rank) return;  // (uniform inside this CTA)
  const int rounds = ((n_units + 1) / 2 + kThreads - 1) / kThreads;
  {  // slots r*kThreads + tid, stored by warp (tid mod 128) / 16: against the row's reference
    const float Rw = sh.wR[(tid & (kThreads / 2 - 1)) >> 4];
    const float f = Rw > kRnone ? pow2i(Rw - Rrow) : 0.f;
    if (f != 1.f)
      for (int r = 0; r < rounds; ++r) uv[r * kThreads + tid] *= f;
  }
  __syncthreads();
  for (int r = warp; r < rounds; r += kWarps) {
    DF a{0.f, 0.f};
    for (int t = lane; t < kThreads; t += 32) df_acc(a, uv[r * kThreads + t]);
    a = df_warp_sum(a);
    if (lane == 0) sh.rtot[r] = a;
  }
  __syncthreads();
  if (warp == 0) {  // the round
    const DF rem = sh.rem;
    __syncwarp();  // (every lane has read sh.rem before lane 0 rewrites it)
    locate_round(sh, rounds, rem, lane);
  }
  __syncthreads();
  const int rsel = sh.rsel;
  const DF rem = sh.rem;
  // block-wide inclusive prefix of round rsel's unit sums (thread order)
  const float v = uv[rsel * kThreads + tid];
  const DF wi = df_warp_scan(DF{v, 0.f}, lane);
  if (lane == 31) sh.scan[warp] = wi;
  __syncthreads();
  DF inc = wi;
  for (int w = 0; w < warp; ++w) inc = df_add(sh.scan[w], inc);
  int cand = (v > 0.f && df_gt(inc, rem)) ? tid : 0x7fffffff;
  int lastpos = v > 0.f ? tid : -1;
  cand = warp_min(cand);
  lastpos = -warp_min(-lastpos);
  __syncthreads();
  if (lane == 0) {
    sh.r_i[warp] = cand;
    sh.scan[warp].hi = __int_as_float(lastpos);
  }
  __syncthreads();
  int tsel = 0x7fffffff, tlast = -1;
  for (int w = 0; w < kWarps; ++w) {
    tsel = min(tsel, sh.r_i[w]);
    tlast = max(tlast, __float_as_int(sh.scan[w].hi));
  }
  const bool past_end = tsel == 0x7fffffff;  // rounding: the last positive unit
  if (past_end) tsel = tlast < 0 ? 0 : tlast;
  if (tid != tsel) return;
  constexpr int EPU = 16 / ES;
  const int pr = rsel * kThreads + tid;  // the pair: units 2pr and 2pr+1
  DF cum = past_end ? DF{0.f, 0.f} : df_sub(inc, DF{v, 0.f});
  int y = -1, ylast = -1;
  const int eb = ebase0 + 2 * pr * EPU;
  for (int q = 0; q < 2 * EPU; ++q) {
    const int e = eb + q;
    if (e < e0 || e >= e1) continue;
    const float z = ES == 2 ? bf16_lo(*reinterpret_cast<const uint16_t*>(row + (size_t)e * 2))
                            : *reinterpret_cast<const float*>(row + (size_t)e * 4);
    const float wv = e2(z, X, -Rrow);
    if (wv > 0.f) ylast = e;
    cum = df_add(cum, DF{wv, 0.f});
    if (!past_end && wv > 0.f && df_gt(cum, rem)) {
      y = e;
      break;
    }
  }
  if (y < 0) y = ylast;
  // (a pair whose rescaled sum is positive but whose weights against Rrow all
  // flush to zero holds mass below 2^-126 of the row: its first element)
  if (y < 0) y = max(eb, e0);
  *out = y;
}

// ---------------------------------------------------------------------------
// Draft-side sampler: item (b, i), i < k_b, draws draft token i of sequence b
// from its row of draft logits with the verify step's processing - the
// temperature softmax, top-p truncation (a2) and the inverse CDF in index
// order (a5's draw, with w = p') - or takes the argmax on a greedy row.
// Items are independent: no sequence words, no early exit.  Position-major,
// P.K positions per sequence; uniforms and outputs are [B][K].
// ---------------------------------------------------------------------------
template <int ES, bool TOPP>
__global__ void __launch_bounds__(kThreads, 4) sample_kernel(const __grid_constant__ VerifyParams P) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int item = blockIdx.x / C;
  const int i = item / P.B, b = item % P.B;

  extern __shared__ __align__(16) float vals[];  // cp.async ring; draw's unit sums; top-p histograms
  __shared__ Shared sh;

  const int kb = P.kpr ? P.kpr[b] : P.K;
  const int md = P.mode ? (int)P.mode[b] : 0;
  const float T = P.temp ? P.temp[b] : 1.0f;
  pdl_wait();  // (the flag word is cleared by the kernel before this one)
  pdl_launch_dependents();
  int32_t* out = P.out + (size_t)b * P.K + i;
  uint32_t seq_err = 0;
  if (kb < 0 || kb > P.K) seq_err |= SV_FLAG_BAD_K;
  else if (md != 0 && md != 1) seq_err |= SV_FLAG_BAD_MODE;
  else if (md == 0 && !(T > 0.f && T < INFINITY)) seq_err |= SV_FLAG_BAD_TEMPERATURE;
  if (seq_err || i >= kb) {  // padding, or a sequence with bad knobs
    if (rank == 0 && tid == 0) {
      *out = -1;
      if (seq_err && i == 0) atomicOr(P.flags, seq_err);
    }
    return;
  }
  const bool greedy = md == 1;
  const Expo X = greedy ? Expo{1.f, 1e-30f} : make_expo(T);
  const int e0 = min(P.V, rank * P.slice_len), e1 = min(P.V, e0 + P.slice_len);
  RowSlice<ES> st;
  st.init(P.tgt + (long long)b * P.t_seq + (long long)i * P.t_pos, e0, e1);
  if (tid == 0) {
    sh.skip = 0;
    sh.moot = 0;
    sh.lth[0] = sh.lth[1] = 0u;
  }
  if (tid == 32) sh.uK = greedy ? 0.f : P.unif[(size_t)b * P.K + i];
  __syncthreads();
  RowAcc at = acc_init(), ad = acc_init();
  // without top-p the row pass keeps its unit-pair sums for the draw (after
  // a ring of the row's slots only)
  float* uv = reinterpret_cast<float*>(reinterpret_cast<char*>(vals) + kSampleSumsOff);
  if (TOPP)
    stream_slices<ES, false, TOPP>(P, sh, vals, st, st, false, greedy, false, X, b, i, at, ad,
                                   reinterpret_cast<uint2*>(reinterpret_cast<char*>(vals) + kListOff));
  else
    stream_pairs<ES>(sh, vals, st, greedy, X, at, uv);
  combine_rows(sh, cluster, C, rank, at, ad, greedy, false, false);  // (never moot here)
  const RowAcc row_t = sh.row_t;
  const bool bad = !(row_t.mx > -INFINITY && row_t.mx < INFINITY) ||
                   (!greedy && !(row_t.R > kRnone && row_t.R < INFINITY));
  const float u = sh.uK;
  // (every condition below is uniform in the cluster)
  if (bad || greedy || !(u >= 0.f && u < 1.f)) {
    if (rank == 0 && tid == 0) {
      *out = (bad || !greedy) ? -1 : row_t.amax;
      if (bad) atomicOr(P.flags, SV_FLAG_NONFINITE);
      else if (!greedy) atomicOr(P.flags, SV_FLAG_BAD_UNIFORM);
    }
    return;
  }
  if (!TOPP) {  // the unit sums are in uv: no row is read again
    sample_draw<ES>(sh, uv, C, rank, st.row, st.e0, st.e1, st.n_units, st.ebase0, X.chi, X.clo, row_t.R,
                    u, out);
    return;
  }
  DF S_t = row_t.s;
  uint32_t kt = 0u;
  int nkt = 0x7fffffff, cntt = 0;
  if (TOPP) {  // (kb = i: no draft token of this row enters the tie count)
    if (tid == 0) {
      sh.rsl[0] = *reinterpret_cast<const RowSlice<4>*>(&st);
      sh.rsl[1] = sh.rsl[0];
    }
    __syncthreads();
    topp_select<ES>(P, sh, reinterpret_cast<unsigned char*>(vals), C, b, i, i, false, X, sh.row_t,
                    sh.row_d);
    S_t = sh.ts[0].E;
    kt = sh.ts[0].kstar;
    nkt = sh.ts[0].nk;
    cntt = sh.ts[0].cstar;
  }
  // j = k_b = i: the draw's weights are p' alone, as for a bonus token
  finish<ES, TOPP, true>(P, sh, vals, C, rank, b, i, T, i, u, e0, e1, row_t.R, row_t.R, S_t,
                         S_t, kt, nkt, cntt, 0u, 0x7fffffff, 0);
}

// Clears the flag word and the sequence words before a verify (or sampler)
// kernel.  It is launched as a programmatic dependent of whatever kernel
// precedes it on the stream, so its launch overlaps that kernel's end; it
// writes nothing until that kernel has completed (griddepcontrol.wait), which
// may be the previous call on the same workspace.
__global__ void verify_init_kernel(uint32_t* flags, unsigned long long* words, uint32_t* words2,
                                   int B) {
  pdl_wait();
  pdl_launch_dependents();  // the verify kernel may start launching
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t == 0) *flags = 0u;
  for (int b = t; b < B; b += gridDim.x * blockDim.x) {
    words[b] = 0ull;
    words2[b] = 0u;
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

size_t ws_layout(int B, int K, size_t* words_off, size_t* words2_off, size_t* stats_off) {
  size_t off = 256;
  *words_off = off;
  off += ((size_t)B * 8 + 255) / 256 * 256;
  *words2_off = off;
  off += ((size_t)B * 4 + 255) / 256 * 256;
  *stats_off = off;
  off += (size_t)B * (K + 1) * sizeof(ItemStats);
  return (off + 255) / 256 * 256;
}

// Launch state per device: the kernels' shared-memory and cluster attributes
// and the SM count are per device in CUDA, so each device is set up by the
// first call made on it.
struct DeviceLaunchState {
  std::atomic<int> configured[4], configured_sample[4], sms;
};
static DeviceLaunchState g_launch[kMaxDevices];

template <int ES, bool TOPP, bool SAMPLE = false>
static cudaError_t configure() {
  auto k = SAMPLE ? sample_kernel<ES, TOPP> : verify_kernel<ES, TOPP>;
  constexpr int kSums = kMaxRounds * kThreads * (int)sizeof(float);
  constexpr int kMax = (kSums > kRingBytes ? kSums : kRingBytes) + (SAMPLE ? kSampleSumsOff : 0);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kMax);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int ES, bool TOPP, bool SAMPLE = false>
static cudaError_t launch(const VerifyParams& P0, int C, int items, size_t smem, cudaStream_t stream) {
  VerifyParams P = P0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)items * (unsigned)C, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may overlap the init kernel before it (the kernel waits for it)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, SAMPLE ? sample_kernel<ES, TOPP> : verify_kernel<ES, TOPP>, P);
}

static int sm_count() {
  const int d = current_device();
  if (d < 0) return 148;
  int n = g_launch[d].sms.load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n < 1) n = 148;
    g_launch[d].sms.store(n, std::memory_order_relaxed);
  }
  return n;
}

// Cluster width: enough CTAs per position level (B items each) to give every
// SM about three, but no slice under 32 KB of a row (narrower slices spend
// more time in the per-item combine and decision than in streaming), and at
// least wide enough that a slice fits kMaxRounds rounds; at most 16 CTAs.
static cudaError_t launch_init(uint32_t* flags, unsigned long long* words, uint32_t* words2, int B,
                               int blocks, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_init_kernel, flags, words, words2, B);
}

static void choose_geometry(int V, int ES, int B, int* C_out, int* slice_out, int max_rounds = kMaxRounds) {
  const long long row_bytes = (long long)V * ES;
  const long long max_slice = (long long)max_rounds * kThreads * 16 - 64;
  int C = (3 * sm_count() + B - 1) / (B > 0 ? B : 1);
  const int cwide = (int)((row_bytes + 32767) / 32768);
  if (C > cwide) C = cwide;
  const int cmin = (int)((row_bytes + max_slice - 1) / max_slice);
  if (C < cmin) C = cmin;
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
  choose_geometry(L.V, ES, L.B, &C, &slice);
  const long long units = ((long long)slice * ES + 30) / 16 + 1;
  const long long rounds = (units + kThreads - 1) / kThreads;
  if (rounds > kMaxRounds) {
    *err = "vocabulary too large for the cluster slice layout";
    return SV_ERR_SHAPE;
  }
  const bool topp = L.top_p < 1.0f;
  size_t smem = (size_t)rounds * kThreads * sizeof(float);  // the draw's unit sums
  if (smem < (size_t)kRingBytes) smem = kRingBytes;          // the row pass's ring
  if (topp && smem < (size_t)kToppSmemBytes) smem = kToppSmemBytes;
  cudaError_t e;
  const int gi = (ES == 2 ? 0 : 1) + (topp ? 2 : 0);
  const int dev = current_device();
  if (dev < 0) {
    *err = "no current CUDA device, or its ordinal is past the library's limit";
    return SV_ERR_CUDA;
  }
  if (!g_launch[dev].configured[gi].load(std::memory_order_acquire)) {
    e = ES == 2 ? (topp ? configure<2, true>() : configure<2, false>())
                : (topp ? configure<4, true>() : configure<4, false>());
    if (e != cudaSuccess) {
      *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return SV_ERR_CUDA;
    }
    g_launch[dev].configured[gi].store(1, std::memory_order_release);
  }
  size_t words_off, words2_off, stats_off;
  ws_layout(L.B, L.K, &words_off, &words2_off, &stats_off);
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
  P.words2 = reinterpret_cast<uint32_t*>(ws + words2_off);
  P.topp_draft = L.topp_draft;
  P.stats = reinterpret_cast<ItemStats*>(ws + stats_off);
  P.slice_len = slice;
  cudaStream_t stream = static_cast<cudaStream_t>(L.stream);

  const int ib = (L.B + 255) / 256;
  e = launch_init(P.flags, P.words, P.words2, L.B, ib < 1 ? 1 : ib, stream);
  if (e != cudaSuccess) {
    *err = std::string("init launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  const int items = (L.K + 1) * L.B;
  if (ES == 2)
    e = topp ? launch<2, true>(P, C, items, smem, stream) : launch<2, false>(P, C, items, smem, stream);
  else
    e = topp ? launch<4, true>(P, C, items, smem, stream) : launch<4, false>(P, C, items, smem, stream);
  if (e != cudaSuccess) {
    *err = std::string("verify launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

size_t verify_workspace_bytes(int B, int K) {
  size_t a, b;
  size_t c;
  return ws_layout(B, K, &a, &c, &b);
}

int sample_launch(const SampleLaunch& L, std::string* err) {
  const int ES = L.dtype == SV_BF16 ? 2 : 4;
  // every item is independent: clusters as narrow as the slice limit allows
  // (without top-p the draw keeps a sum per unit pair, 32 KB for 64 rounds
  // of units; with top-p, 32 rounds)
  const bool topp = L.top_p < 1.0f;
  int C, slice;
  choose_geometry(L.V, ES, L.B * L.K, &C, &slice, topp ? 32 : kMaxRounds);
  const long long units = ((long long)slice * ES + 30) / 16 + 1;
  const long long rounds = (units + kThreads - 1) / kThreads;
  if (rounds > kMaxRounds) {
    *err = "vocabulary too large for the cluster slice layout";
    return SV_ERR_SHAPE;
  }
  size_t smem = (size_t)rounds * kThreads * sizeof(float);
  if (smem < (size_t)kRingBytes) smem = kRingBytes;
  if (topp && smem < (size_t)kToppSmemBytes) smem = kToppSmemBytes;
  if (!topp)  // ring + pair sums
    smem = (size_t)kSampleSumsOff + (size_t)(((units + 1) / 2 + kThreads - 1) / kThreads) * kThreads * sizeof(float);
  cudaError_t e;
  const int gi = (ES == 2 ? 0 : 1) + (topp ? 2 : 0);
  const int dev = current_device();
  if (dev < 0) {
    *err = "no current CUDA device, or its ordinal is past the library's limit";
    return SV_ERR_CUDA;
  }
  if (!g_launch[dev].configured_sample[gi].load(std::memory_order_acquire)) {
    e = ES == 2 ? (topp ? configure<2, true, true>() : configure<2, false, true>())
                : (topp ? configure<4, true, true>() : configure<4, false, true>());
    if (e != cudaSuccess) {
      *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return SV_ERR_CUDA;
    }
    g_launch[dev].configured_sample[gi].store(1, std::memory_order_release);
  }
  VerifyParams P = {};
  P.tgt = static_cast<const char*>(L.logits);
  P.t_seq = L.l_seq * ES;
  P.t_pos = L.l_pos * ES;
  P.B = L.B;
  P.K = L.K;
  P.V = L.V;
  P.kpr = L.kpr;
  P.temp = L.temp;
  P.top_p = L.top_p;
  P.unif = L.unif;
  P.mode = L.mode;
  P.out = L.out;
  P.flags = static_cast<uint32_t*>(L.workspace);
  P.slice_len = slice;
  cudaStream_t stream = static_cast<cudaStream_t>(L.stream);
  e = launch_init(P.flags, nullptr, nullptr, 0, 1, stream);  // the flag word only
  if (e != cudaSuccess) {
    *err = std::string("init launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  const int items = L.K * L.B;
  if (items > 0) {
    if (ES == 2)
      e = topp ? launch<2, true, true>(P, C, items, smem, stream) : launch<2, false, true>(P, C, items, smem, stream);
    else
      e = topp ? launch<4, true, true>(P, C, items, smem, stream) : launch<4, false, true>(P, C, items, smem, stream);
    if (e != cudaSuccess) {
      *err = std::string("sample launch: ") + cudaGetErrorString(e);
      return SV_ERR_CUDA;
    }
  }
  return SV_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the verify step's scratch (flag word, per-sequence
// words, per-position statistics) lives in this fixed device array instead of
// a caller-provided workspace.  Every GPU that loads the library holds the
// array until the process exits.  All calls share it: each call's first
// kernel zeroes the flag word and the sequence words it will use (the
// statistics are written before they are read), so consecutive calls on one
// stream are independent, but calls whose kernels overlap on the GPU (other
// streams, other host threads) race on it.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mutex;
static void* g_noalloc_addr[kMaxDevices];

int verify_launch_noalloc(const VerifyLaunch& L, std::string* err) {
  const size_t need = verify_workspace_bytes(L.B, L.K);
  if (need > kNoAllocScratchBytes) {
    *err = "sv_spec_verify_noalloc: B=" + std::to_string(L.B) + ", K=" + std::to_string(L.K) +
           " needs " + std::to_string(need) + " bytes of scratch; the built-in buffer holds " +
           std::to_string(kNoAllocScratchBytes) + " (use sv_spec_verify with a workspace)";
    return SV_ERR_WORKSPACE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = std::string("sv_spec_verify_noalloc: no usable current device: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
      // Host code cannot use the array's name as a device address: ask the
      // runtime for the address of this device's copy (once per device).
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        *err = std::string("sv_spec_verify_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e);
        return SV_ERR_CUDA;
      }
      g_noalloc_addr[dev] = p;
    }
    scratch = g_noalloc_addr[dev];
  }
  VerifyLaunch L2 = L;
  L2.workspace = scratch;
  return verify_launch(L2, err);
}

}  // namespace sv
