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
// [r*L, (r+1)*L) of both rows and keeps it resident in its shared memory
// (bulk-copy engine loads, one mbarrier per row).  Passes over a row (max;
// exp-sum with the exact max; residual CDF) then read shared memory, and the
// cluster combines per-slice partials through distributed shared memory.
//
// Items are launched position-major (all sequences' position 0 first).  Each
// item publishes {done, rejected, error} bits for its position in one 64-bit
// word per sequence.  An item that starts after an earlier position of its
// sequence has been rejected exits without reading its rows: those rows
// cannot change the result.  The item whose publication completes the
// prefix 0..j (j = first rejection, or k_b when all were accepted) is the
// sequence's finisher: it draws the resample / bonus token, from its own
// resident slices when j is its own position, else after loading row(s) j.
// No item ever waits for another one.
#include <cstdint>
#include <cstdio>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCmax = 16;
constexpr int kMaxTiles = 24;  // slice <= 24 * 256 units of 16 B
constexpr int kWordBits = 21;  // positions per field of the sequence word

struct ItemStats {
  float m_t, st_hi, st_lo, m_d;
  float sd_hi, sd_lo;
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
  int slice_len;      // elements per CTA slice
  int rowbuf_bytes;   // shared-memory bytes per row buffer
};

// ---------------------------------------------------------------------------
// One CTA's slice of one logit row, mapped to 16-byte units in shared memory.
// Unit u holds global bytes [base16 + 16u, base16 + 16u + 16); element e of
// the row lies in unit (e*ES + row - base16) / 16.
// ---------------------------------------------------------------------------
template <int ES>
struct SliceMap {
  const char* row;  // row start (global)
  int e0, e1;       // elements owned by this CTA
  uintptr_t g0, g1, base16, a0, a1;
  int n_units;
  int ebase0;  // element index of the first lane of unit 0 (may be < e0)

  __device__ void init(const char* row_, int e0_, int e1_) {
    row = row_;
    e0 = e0_;
    e1 = e1_;
    g0 = reinterpret_cast<uintptr_t>(row) + (uintptr_t)e0 * ES;
    g1 = reinterpret_cast<uintptr_t>(row) + (uintptr_t)e1 * ES;
    base16 = g0 & ~uintptr_t(15);
    a0 = (g0 + 15) & ~uintptr_t(15);
    a1 = g1 & ~uintptr_t(15);
    if (a1 < a0) a1 = a0;
    n_units = e1 > e0 ? (int)((g1 - base16 + 15) / 16) : 0;
    ebase0 = e0 - (int)((g0 & 15) / ES);
  }
};

// Issue the loads of a slice into `buf`: the 16-byte-aligned body with bulk
// copies on `bar` (thread 0), the unaligned head and tail with plain loads
// (all threads).  Returns nothing; consumers wait on `bar` and a
// __syncthreads() that follows this call.
template <int ES>
__device__ void issue_slice(const SliceMap<ES>& s, char* buf, uint64_t* bar) {
  const int tid = threadIdx.x;
  const uint32_t body = (uint32_t)(s.a1 - s.a0);
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, body);
    constexpr uint32_t kChunk = 8192;
    for (uint32_t off = 0; off < body; off += kChunk) {
      uint32_t n = body - off < kChunk ? body - off : kChunk;
      bulk_copy_g2s(buf + (s.a0 - s.base16) + off, reinterpret_cast<const void*>(s.a0 + off), n,
                    bar);
    }
  }
  // head [g0, a0) and tail [a1, g1) (or everything when there is no body)
  const int n_head = (int)((body ? s.a0 : s.g1) - s.g0) / ES;
  const int n_tail = body ? (int)(s.g1 - s.a1) / ES : 0;
  for (int k = tid; k < n_head + n_tail; k += kThreads) {
    uintptr_t ga = k < n_head ? s.g0 + (uintptr_t)k * ES : s.a1 + (uintptr_t)(k - n_head) * ES;
    char* dst = buf + (ga - s.base16);
    if (ES == 2)
      *reinterpret_cast<uint16_t*>(dst) = *reinterpret_cast<const uint16_t*>(ga);
    else
      *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(ga);
  }
}

// element j (0..16/ES-1) of a 16-byte unit as float
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

__device__ __forceinline__ float nanmax(float a, float b) {
  return (a != a || b != b) ? __int_as_float(0x7fc00000) : fmaxf(a, b);
}

// Row max of a slice held in shared memory (NaN propagates).
template <int ES>
__device__ float slice_max(const SliceMap<ES>& s, const char* buf) {
  constexpr int EPU = 16 / ES;
  float m = -__int_as_float(0x7f800000);
  if (ES == 2) {
    __nv_bfloat162 m2 = __floats2bfloat162_rn(-INFINITY, -INFINITY);
    for (int u = threadIdx.x; u < s.n_units; u += kThreads) {
      uint4 v = *reinterpret_cast<const uint4*>(buf + 16 * u);
      int eb = s.ebase0 + u * EPU;
      if (eb >= s.e0 && eb + EPU <= s.e1) {
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
        m2 = __hmax2_nan(m2, __hmax2_nan(__hmax2_nan(p[0], p[1]), __hmax2_nan(p[2], p[3])));
      } else {
        for (int j = 0; j < EPU; ++j)
          if (eb + j >= s.e0 && eb + j < s.e1) m = nanmax(m, unit_elem<ES>(v, j));
      }
    }
    m = nanmax(m, nanmax(__low2float(m2), __high2float(m2)));
  } else {
    bool nan = false;
    for (int u = threadIdx.x; u < s.n_units; u += kThreads) {
      uint4 v = *reinterpret_cast<const uint4*>(buf + 16 * u);
      int eb = s.ebase0 + u * EPU;
#pragma unroll
      for (int j = 0; j < EPU; ++j) {
        float z = unit_elem<ES>(v, j);
        bool ok = eb + j >= s.e0 && eb + j < s.e1;
        if (ok) {
          nan |= (z != z);
          m = fmaxf(m, z);
        }
      }
    }
    if (nan) m = __int_as_float(0x7fc00000);
  }
  return m;
}

// exp((z - m)/T) as 2^((z - m) * c) with c = log2(e)/T held as hi + lo, so
// the temperature is applied without a rounded reciprocal.  d is clamped at
// dmin (where the result underflows anyway) so that -inf logits give 0.
struct Expo {
  float m, chi, clo, dmin;
  __device__ __forceinline__ float operator()(float z) const {
    float d = fmaxf(z - m, dmin);
    return ex2(fmaf(d, chi, d * clo));
  }
  __device__ __forceinline__ double arg_exact(float z) const {
    return ((double)z - (double)m) * ((double)chi + (double)clo);
  }
};

__device__ Expo make_expo(float m, float T) {
  double c = 1.4426950408889634074 / (double)T;
  Expo e;
  e.m = m;
  e.chi = (float)c;
  e.clo = (float)(c - (double)e.chi);
  e.dmin = -256.0f / e.chi;
  return e;
}

// Sum of exp over a slice (double-float).
template <int ES>
__device__ DF slice_sumexp(const SliceMap<ES>& s, const char* buf, const Expo& ex) {
  constexpr int EPU = 16 / ES;
  DF acc{0.f, 0.f};
  for (int u = threadIdx.x; u < s.n_units; u += kThreads) {
    uint4 v = *reinterpret_cast<const uint4*>(buf + 16 * u);
    int eb = s.ebase0 + u * EPU;
    float e[EPU];
    if (eb >= s.e0 && eb + EPU <= s.e1) {
#pragma unroll
      for (int j = 0; j < EPU; ++j) e[j] = ex(unit_elem<ES>(v, j));
    } else {
#pragma unroll
      for (int j = 0; j < EPU; ++j)
        e[j] = (eb + j >= s.e0 && eb + j < s.e1) ? ex(unit_elem<ES>(v, j)) : 0.f;
    }
    float us;
    if (EPU == 8)
      us = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
    else
      us = (e[0] + e[1]) + (e[2] + e[3]);
    df_acc(acc, us);
  }
  return acc;
}

// Residual / bonus weight of one element: w' = max(0, e_t - rho * e_d) with
// rho = S_t/S_d (hi + lo), or e_t alone when rho_hi < 0 marks "p only".
struct Weight {
  Expo et, ed;
  float rho_hi, rho_lo;
  bool p_only;
  __device__ __forceinline__ float operator()(float zt, float zd) const {
    float a = et(zt);
    if (p_only) return a;
    float b = ed(zd);
    return fmaxf(0.f, fmaf(-rho_lo, b, fmaf(-rho_hi, b, a)));
  }
};

// Element e of a slice read back from shared memory one at a time (used when
// the draft row's 16-byte phase differs from the target row's).
template <int ES>
__device__ __forceinline__ float slice_elem(const SliceMap<ES>& s, const char* buf, int e) {
  const char* p = buf + (s.g0 - s.base16) + (size_t)(e - s.e0) * ES;
  return ES == 2 ? bf16_lo(*reinterpret_cast<const uint16_t*>(p))
                 : *reinterpret_cast<const float*>(p);
}

// Target and draft slices of one position: unit u of the target buffer holds
// elements [ebase0 + u*EPU, ...).  When both rows start at the same offset
// modulo 16 bytes the draft buffer's unit u holds the same elements.
template <int ES>
struct PairMap {
  const SliceMap<ES>* st;
  const SliceMap<ES>* sd;
  bool same_phase;
};

template <int ES>
__device__ __forceinline__ float unit_weight_sum(const PairMap<ES>& pm, const char* bt,
                                                 const char* bd, int u, const Weight& W) {
  constexpr int EPU = 16 / ES;
  const SliceMap<ES>& s = *pm.st;
  if (u >= s.n_units) return 0.f;
  uint4 vt = *reinterpret_cast<const uint4*>(bt + 16 * u);
  const bool vec_d = W.p_only || pm.same_phase;
  uint4 vd = vec_d ? (W.p_only ? vt : *reinterpret_cast<const uint4*>(bd + 16 * u)) : vt;
  int eb = s.ebase0 + u * EPU;
  float e[EPU];
  bool full = eb >= s.e0 && eb + EPU <= s.e1;
#pragma unroll
  for (int j = 0; j < EPU; ++j) {
    bool ok = full || (eb + j >= s.e0 && eb + j < s.e1);
    float zd = 0.f;
    if (ok) zd = vec_d ? unit_elem<ES>(vd, j) : slice_elem<ES>(*pm.sd, bd, eb + j);
    e[j] = ok ? W(unit_elem<ES>(vt, j), zd) : 0.f;
  }
  if (EPU == 8) return ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
  return (e[0] + e[1]) + (e[2] + e[3]);
}

// Per-tile (256 units), per-warp partial sums of the weights of a slice.
template <int ES>
__device__ void slice_weight_partials(const PairMap<ES>& pm, const char* bt, const char* bd,
                                      const Weight& W, DF (*tw)[kWarps]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = (pm.st->n_units + kThreads - 1) / kThreads;
  for (int t = 0; t < tiles; ++t) {
    float us = unit_weight_sum<ES>(pm, bt, bd, t * kThreads + threadIdx.x, W);
    DF v = df_warp_sum(DF{us, 0.f});
    if (lane == 0) tw[t][warp] = v;
  }
}

struct Shared {
  uint64_t bar[2];
  uint32_t bar_phase[2];
  // all-gather slots, indexed by the writing CTA's rank
  float g_mt[kCmax], g_md[kCmax];
  DF g_st[kCmax], g_sd[kCmax], g_w[kCmax];
  int g_amax[kCmax];
  // block reduction scratch
  float r_f[kWarps][2];
  DF r_df[kWarps][2];
  int r_i[kWarps];
  DF tw[kMaxTiles][kWarps];
  // broadcast values
  int skip;
  int fin, fin_j, fin_err;
  float bc_f[4];
};

__device__ __forceinline__ bool resolvable(unsigned long long w, int kb, int* j_out, bool* err) {
  const unsigned long long mask = (1ull << kWordBits) - 1;
  unsigned long long D = w & mask;
  unsigned long long Rj = (w >> kWordBits) & mask;
  unsigned long long E = (w >> (2 * kWordBits)) & mask;
  unsigned long long R = Rj | E;
  int j = R ? __ffsll((long long)R) - 1 : kb;
  unsigned long long need = (j + 1 >= 64) ? ~0ull : ((1ull << (j + 1)) - 1);
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

template <int ES>
__global__ void __launch_bounds__(kThreads) verify_kernel(const VerifyParams P) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int item = blockIdx.x / C;
  const int i = item / P.B, b = item % P.B;

  extern __shared__ __align__(128) char dyn[];
  char* buf_t = dyn;
  char* buf_d = dyn + P.rowbuf_bytes;
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

  // Every CTA of the cluster must be running before any distributed
  // shared-memory access: arrive now, wait after the local set-up.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (tid == 0) {
    mbar_init(&sh.bar[0], 1);
    mbar_init(&sh.bar[1], 1);
    sh.bar_phase[0] = sh.bar_phase[1] = 0;
    fence_mbar_init();
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  // ---- agree on skipping: an earlier position already rejected ----
  if (rank == 0 && tid == 0) {
    unsigned long long w = __ldcg(P.words + b);
    unsigned long long R = ((w >> kWordBits) | (w >> (2 * kWordBits))) & ((1ull << kWordBits) - 1);
    int skip = (R & ((1ull << i) - 1)) != 0;
    for (int r = 0; r < C; ++r) *cluster.map_shared_rank(&sh.skip, r) = skip;
  }
  cluster.sync();
  if (sh.skip) return;

  // ---- load the slices ----
  const int e0 = min(P.V, rank * P.slice_len), e1 = min(P.V, e0 + P.slice_len);
  SliceMap<ES> st, sd;
  st.init(P.tgt + (long long)b * P.t_seq + (long long)i * P.t_pos, e0, e1);
  issue_slice<ES>(st, buf_t, &sh.bar[0]);
  if (has_draft) {
    sd.init(P.drf + (long long)b * P.d_seq + (long long)i * P.d_pos, e0, e1);
    issue_slice<ES>(sd, buf_d, &sh.bar[1]);
  }
  __syncthreads();
  bool timed_out = false;
  timed_out |= !mbar_wait_bounded(&sh.bar[0], 0);
  if (has_draft) timed_out |= !mbar_wait_bounded(&sh.bar[1], 0);
  if (timed_out && tid == 0) atomicOr(P.flags, (uint32_t)SV_FLAG_TIMEOUT);
  if (tid == 0) {
    sh.bar_phase[0] = 1;
    if (has_draft) sh.bar_phase[1] = 1;
  }

  // ---- pass 1: row maxima ----
  float mt = slice_max<ES>(st, buf_t);
  float mdx = has_draft ? slice_max<ES>(sd, buf_d) : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mt = nanmax(mt, __shfl_xor_sync(0xffffffffu, mt, o));
    mdx = nanmax(mdx, __shfl_xor_sync(0xffffffffu, mdx, o));
  }
  if (lane == 0) {
    sh.r_f[warp][0] = mt;
    sh.r_f[warp][1] = mdx;
  }
  __syncthreads();
  if (tid < C) {
    float a = sh.r_f[0][0], d = sh.r_f[0][1];
    for (int w = 1; w < kWarps; ++w) {
      a = nanmax(a, sh.r_f[w][0]);
      d = nanmax(d, sh.r_f[w][1]);
    }
    if (timed_out) a = __int_as_float(0x7fc00000);
    *cluster.map_shared_rank(&sh.g_mt[rank], tid) = a;
    *cluster.map_shared_rank(&sh.g_md[rank], tid) = d;
  }
  cluster.sync();
  float m_t = sh.g_mt[0], m_d = sh.g_md[0];
  for (int r = 1; r < C; ++r) {
    m_t = nanmax(m_t, sh.g_mt[r]);
    m_d = nanmax(m_d, sh.g_md[r]);
  }
  // Row validity: no NaN, no +inf, not all -inf.
  const bool bad_t = !(m_t > -INFINITY && m_t < INFINITY);
  const bool bad_d = has_draft && !(m_d > -INFINITY && m_d < INFINITY);
  // (a bounded-wait timeout poisoned its CTA's max with NaN above)

  uint32_t errbits = 0;
  if (bad_t || bad_d) errbits |= SV_FLAG_NONFINITE;
  int x = -1;
  if (i < kb) {
    x = P.tokens[(size_t)b * P.K + i];
    if (x < 0 || x >= P.V) errbits |= SV_FLAG_BAD_TOKEN;
  }
  bool reject = false;
  int amax = -1;
  float diag_px = NAN, diag_qx = NAN, diag_r = NAN;
  DF S_t{0.f, 0.f}, S_d{0.f, 0.f};
  Expo ext{}, exd{};

  if (greedy) {
    // ---- pass 2 (greedy): lowest index holding the max ----
    int best = 0x7fffffff;
    if (!bad_t) {
      constexpr int EPU = 16 / ES;
      for (int u = tid; u < st.n_units && best == 0x7fffffff; u += kThreads) {
        uint4 v = *reinterpret_cast<const uint4*>(buf_t + 16 * u);
        int eb = st.ebase0 + u * EPU;
        for (int j = 0; j < EPU; ++j) {
          int e = eb + j;
          if (e >= st.e0 && e < st.e1 && unit_elem<ES>(v, j) == m_t) {
            best = e;
            break;
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, o));
    if (lane == 0) sh.r_i[warp] = best;
    __syncthreads();
    if (tid < C) {
      int a = sh.r_i[0];
      for (int w = 1; w < kWarps; ++w) a = min(a, sh.r_i[w]);
      *cluster.map_shared_rank(&sh.g_amax[rank], tid) = a;
    }
    cluster.sync();
    amax = sh.g_amax[0];
    for (int r = 1; r < C; ++r) amax = min(amax, sh.g_amax[r]);
    if (i < kb && !errbits) reject = (x != amax);
  } else {
    // ---- pass 2 (sampled): normalisers with the exact row max ----
    float u_i = 0.f;
    if (i < kb) {
      u_i = P.unif[(size_t)b * (P.K + 1) + i];
      if (!(u_i >= 0.f && u_i < 1.f)) errbits |= SV_FLAG_BAD_UNIFORM;
    }
    ext = make_expo(bad_t ? 0.f : m_t, T);
    exd = make_expo(bad_d ? 0.f : m_d, T);
    DF at = bad_t ? DF{0.f, 0.f} : slice_sumexp<ES>(st, buf_t, ext);
    DF ad = (has_draft && !bad_d) ? slice_sumexp<ES>(sd, buf_d, exd) : DF{0.f, 0.f};
    at = df_warp_sum(at);
    ad = df_warp_sum(ad);
    if (lane == 0) {
      sh.r_df[warp][0] = at;
      sh.r_df[warp][1] = ad;
    }
    __syncthreads();
    if (tid < C) {
      DF a = sh.r_df[0][0], d = sh.r_df[0][1];
      for (int w = 1; w < kWarps; ++w) {
        a = df_add(a, sh.r_df[w][0]);
        d = df_add(d, sh.r_df[w][1]);
      }
      *cluster.map_shared_rank(&sh.g_st[rank], tid) = a;
      *cluster.map_shared_rank(&sh.g_sd[rank], tid) = d;
    }
    cluster.sync();
    S_t = sh.g_st[0];
    S_d = sh.g_sd[0];
    for (int r = 1; r < C; ++r) {
      S_t = df_add(S_t, sh.g_st[r]);
      S_d = df_add(S_d, sh.g_sd[r]);
    }
    if (has_draft && !errbits) {
      // ratio p(x)/q(x) = 2^(a_t - a_d) * S_d / S_t, in the exponent domain so
      // that neither factor underflows on its own; q(x) = 0 only where the
      // exact value underflows double precision.
      const char* rt = P.tgt + (long long)b * P.t_seq + (long long)i * P.t_pos;
      const char* rd = P.drf + (long long)b * P.d_seq + (long long)i * P.d_pos;
      float zt = ES == 2 ? bf16_lo(*reinterpret_cast<const uint16_t*>(rt + (size_t)x * 2))
                         : *reinterpret_cast<const float*>(rt + (size_t)x * 4);
      float zd = ES == 2 ? bf16_lo(*reinterpret_cast<const uint16_t*>(rd + (size_t)x * 2))
                         : *reinterpret_cast<const float*>(rd + (size_t)x * 4);
      double at_x = ext.arg_exact(zt), ad_x = exd.arg_exact(zd);
      float r;
      if (!(ad_x > -1074.0) || !(at_x > -1074.0)) {
        r = 0.f;
      } else {
        float ratio_s = (float)(df_to_double(S_d) / df_to_double(S_t));
        r = ex2((float)(at_x - ad_x)) * ratio_s;
      }
      diag_px = ext(zt) / S_t.hi;
      diag_qx = exd(zd) / S_d.hi;
      diag_r = r;
      reject = !(u_i < r);
    }
  }

  // ---- publish; find out whether this item finishes the sequence ----
  if (rank == 0 && tid == 0) {
    ItemStats s;
    s.m_t = m_t;
    s.st_hi = S_t.hi;
    s.st_lo = S_t.lo;
    s.m_d = m_d;
    s.sd_hi = S_d.hi;
    s.sd_lo = S_d.lo;
    s.argmax = amax;
    s.errbits = errbits;
    P.stats[(size_t)b * (P.K + 1) + i] = s;
    if (P.diag) {
      float* dg = P.diag + ((size_t)b * (P.K + 1) + i) * SV_DIAG_FIELDS;
      dg[SV_DIAG_M_T] = m_t;
      if (greedy) {
        dg[SV_DIAG_ARGMAX] = (float)amax;
      } else {
        dg[SV_DIAG_S_T] = S_t.hi + S_t.lo;
        dg[SV_DIAG_MASS_T] = 1.f;
        if (has_draft) {
          dg[SV_DIAG_M_D] = m_d;
          dg[SV_DIAG_S_D] = S_d.hi + S_d.lo;
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
    unsigned long long old = atomicOr(P.words + b, bits);
    __threadfence();
    int j0, j1;
    bool e0_, e1_;
    bool was = resolvable(old, kb, &j0, &e0_);
    bool now = resolvable(old | bits, kb, &j1, &e1_);
    int fin = (!was && now) ? 1 : 0;
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
      uint32_t eb = j == i ? errbits : __ldcg(&P.stats[(size_t)b * (P.K + 1) + j].errbits);
      write_outputs(P, b, 0, -1, true);
      atomicOr(P.flags, eb);
    }
    return;
  }
  if (greedy) {
    if (rank == 0 && tid == 0) {
      int a = j == i ? amax : __ldcg(&P.stats[(size_t)b * (P.K + 1) + j].argmax);
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
  // statistics and resident rows of position j
  Weight W;
  if (j != i) {
    const ItemStats* sj = P.stats + (size_t)b * (P.K + 1) + j;
    float jm_t = __ldcg(&sj->m_t), jm_d = __ldcg(&sj->m_d);
    S_t = DF{__ldcg(&sj->st_hi), __ldcg(&sj->st_lo)};
    S_d = DF{__ldcg(&sj->sd_hi), __ldcg(&sj->sd_lo)};
    ext = make_expo(jm_t, T);
    exd = make_expo(jm_d, T);
    __syncthreads();  // everyone is done with the old contents
    st.init(P.tgt + (long long)b * P.t_seq + (long long)j * P.t_pos, e0, e1);
    issue_slice<ES>(st, buf_t, &sh.bar[0]);
    if (!bonus) {
      sd.init(P.drf + (long long)b * P.d_seq + (long long)j * P.d_pos, e0, e1);
      issue_slice<ES>(sd, buf_d, &sh.bar[1]);
    }
    __syncthreads();
    bool ok = mbar_wait_bounded(&sh.bar[0], sh.bar_phase[0]);
    if (!bonus) ok &= mbar_wait_bounded(&sh.bar[1], sh.bar_phase[1]);
    if (!ok && tid == 0) atomicOr(P.flags, SV_FLAG_TIMEOUT);
  }
  W.et = ext;
  W.ed = exd;
  W.p_only = bonus;
  {
    double rho = df_to_double(S_t) / df_to_double(S_d);
    W.rho_hi = (float)rho;
    W.rho_lo = (float)(rho - (double)W.rho_hi);
  }
  const int tiles = (st.n_units + kThreads - 1) / kThreads;
  PairMap<ES> pm;
  pm.st = &st;
  pm.sd = &sd;
  pm.same_phase = bonus || st.ebase0 == sd.ebase0;
  DF slice_w{0.f, 0.f};
  for (int pass = 0; pass < 2; ++pass) {
    if (pass) cluster.sync();  // every CTA has read the first pass's slots
    slice_weight_partials<ES>(pm, buf_t, buf_d, W, sh.tw);
    __syncthreads();
    if (tid < C) {
      DF a{0.f, 0.f};
      for (int t = 0; t < tiles; ++t)
        for (int w = 0; w < kWarps; ++w) a = df_add(a, sh.tw[t][w]);
      *cluster.map_shared_rank(&sh.g_w[rank], tid) = a;
    }
    cluster.sync();
    DF tot = sh.g_w[0];
    for (int r = 1; r < C; ++r) tot = df_add(tot, sh.g_w[r]);
    if (tot.hi > 0.f || W.p_only) {
      slice_w = tot;
      break;
    }
    W.p_only = true;  // residual all zero: draw from p  [SSD §4.3]
    __syncthreads();
  }
  // locate the owner of u * total (ranks in order, then tiles, warps, lanes)
  const double total = df_to_double(slice_w);
  const double tgt = (double)uK * total;
  double pre = 0.0;
  int owner = -1, last_pos = 0;
  for (int r = 0; r < C; ++r) {
    double v = df_to_double(sh.g_w[r]);
    if (v > 0.0) last_pos = r;
    if (owner < 0 && pre + v > tgt && v > 0.0) owner = r;
    if (owner < 0) pre += v;
  }
  if (owner < 0) {
    owner = last_pos;
    pre = 0.0;
    for (int r = 0; r < last_pos; ++r) pre += df_to_double(sh.g_w[r]);
  }
  if (rank == 0 && tid == 0 && P.diag) {
    float* dg = P.diag + ((size_t)b * (P.K + 1) + j) * SV_DIAG_FIELDS;
    dg[SV_DIAG_S_W] = W.p_only ? 1.f : (float)(total / df_to_double(S_t));
  }
  if (rank != owner) return;
  // tile and warp inside the owner (everyone computes the same answer)
  double rem = tgt - pre;
  int tsel = -1, wsel = 0, tlast = 0, wlast = 0;
  for (int t = 0; t < tiles && tsel < 0; ++t)
    for (int w = 0; w < kWarps; ++w) {
      double v = df_to_double(sh.tw[t][w]);
      if (v > 0.0) {
        tlast = t;
        wlast = w;
      }
      if (v > rem && v > 0.0) {
        tsel = t;
        wsel = w;
        break;
      }
      rem -= v;
    }
  if (tsel < 0) {  // rounding pushed the target past the end: last positive
    tsel = tlast;
    wsel = wlast;
    rem = df_to_double(sh.tw[tlast][wlast]);
    rem = rem > 0.0 ? rem * 0.999999 : 0.0;
  }
  if (warp != wsel) return;
  // lanes of the selected warp: inclusive scan of their unit sums
  const int u = tsel * kThreads + wsel * 32 + lane;
  float us = unit_weight_sum<ES>(pm, buf_t, buf_d, u, W);
  double inc = (double)us;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    double n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  const double exc = inc - (double)us;
  unsigned hit = __ballot_sync(0xffffffffu, inc > rem && us > 0.f);
  unsigned pos = __ballot_sync(0xffffffffu, us > 0.f);
  int sel = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
  if (lane == sel && u < st.n_units) {
    constexpr int EPU = 16 / ES;
    uint4 vt = *reinterpret_cast<const uint4*>(buf_t + 16 * u);
    const bool vec_d = W.p_only || pm.same_phase;
    uint4 vd = vec_d ? (W.p_only ? vt : *reinterpret_cast<const uint4*>(buf_d + 16 * u)) : vt;
    int eb = st.ebase0 + u * EPU;
    double c = exc;
    int y = -1, ylast = -1;
    for (int q = 0; q < EPU; ++q) {
      int e = eb + q;
      if (e < st.e0 || e >= st.e1) continue;
      float zd = vec_d ? unit_elem<ES>(vd, q) : slice_elem<ES>(sd, buf_d, e);
      float wv = W(unit_elem<ES>(vt, q), zd);
      if (wv > 0.f) ylast = e;
      c += (double)wv;
      if (wv > 0.f && c > rem) {
        y = e;
        break;
      }
    }
    if (y < 0) y = ylast;
    write_outputs(P, b, j, y, false);
  }
}

__global__ void verify_init_kernel(uint32_t* flags, unsigned long long* words, int B) {
  int t = blockIdx.x * blockDim.x + threadIdx.x;
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
static cudaError_t configure(size_t max_smem) {
  cudaError_t e = cudaFuncSetAttribute(verify_kernel<ES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(verify_kernel<ES>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int ES>
static cudaError_t launch(const VerifyParams& P0, int C, size_t smem, int items,
                          cudaStream_t stream) {
  VerifyParams P = P0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)items * (unsigned)C, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
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

// Cluster width: about 16 KB of each row per CTA, at most 16 CTAs.
static void choose_geometry(int V, int ES, int* C_out, int* slice_out, int* rowbuf_out) {
  const long long row_bytes = (long long)V * ES;
  int C = (int)((row_bytes + 16383) / 16384);
  if (C < 1) C = 1;
  if (C > kCmax) C = kCmax;
  int slice = (V + C - 1) / C;
  slice = (slice + 7) / 8 * 8;
  C = (V + slice - 1) / slice;
  if (C < 1) C = 1;
  *C_out = C;
  *slice_out = slice;
  *rowbuf_out = (int)(((long long)slice * ES + 32 + 127) / 128 * 128);
}

int verify_launch(const VerifyLaunch& L, std::string* err) {
  const int ES = L.dtype == SV_BF16 ? 2 : 4;
  int C, slice, rowbuf;
  choose_geometry(L.V, ES, &C, &slice, &rowbuf);
  if ((long long)slice * ES > (long long)kMaxTiles * kThreads * 16 - 32) {
    *err = "vocabulary too large for the cluster slice layout";
    return SV_ERR_SHAPE;
  }
  const size_t smem = 2 * (size_t)rowbuf;
  const size_t max_smem = 2 * (size_t)(((long long)kMaxTiles * kThreads * 16 + 32 + 127) / 128 * 128);
  cudaError_t e;
  int gi = ES == 2 ? 0 : 1;
  if (!g_configured[gi]) {
    e = ES == 2 ? configure<2>(max_smem) : configure<4>(max_smem);
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
  P.rowbuf_bytes = rowbuf;
  cudaStream_t stream = static_cast<cudaStream_t>(L.stream);

  int ib = (L.B + 255) / 256;
  verify_init_kernel<<<ib < 1 ? 1 : ib, 256, 0, stream>>>(P.flags, P.words, L.B);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("init launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  const int items = (L.K + 1) * L.B;
  e = ES == 2 ? launch<2>(P, C, smem, items, stream) : launch<4>(P, C, smem, items, stream);
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
