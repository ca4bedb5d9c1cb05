// Fused final RMSNorm + LM head for sm_103a: the draft-logit producer of
// layer-skip self-speculation [SSD §3.1, §4.2] ("Self-speculative decoding
// with layer skip and KV reuse"): a draft that leaves the stack at layer L
// still passes through the model's final RMSNorm before the output head.
//
//   y[m][k]      = bf16( h[m][k] * rsqrt(mean_k h[m][k]^2 + eps) * w[k] )
//   logits[m][n] = sum_k y[m][k] * W[k][n]            (fp32 accumulation)
//
// Two kernels on the caller's stream:
//  1. rmsnorm_kernel: one CTA per row writes the normalised, weighted bf16
//     row y into the workspace (4 MB at M=512, H=4096: L2-resident for 2.).
//  2. lmhead_gemm_kernel: persistent, one CTA per SM, 128 x BN output tiles
//     on the 5th-generation tensor cores (BN in 128..256, chosen per shape for
//     the fewest waves).  A 4-stage ring in shared memory is filled by the TMA
//     engine (cp.async.bulk.tensor, 128-byte swizzle): y tiles K-major (128
//     rows x 64 k), W tiles N-major (64 k x 64 n, up to four per stage).  One
//     thread issues tcgen05.mma (M=128, N=BN, K=16, bf16 in, fp32 accumulator
//     in tensor memory) and tcgen05.commit frees each stage once its MMAs are
//     done; two accumulators let four epilogue warps read one tile back
//     (tcgen05.ld) and store bf16 (or fp32) logits while the next tile
//     accumulates.  Tiles are numbered M-fastest, so the row tiles that share
//     a W column block run side by side and W streams from HBM about once.
#include <cuda.h>  // CUtensorMap and the encoder's signature (resolved at run time)

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {
namespace lmh {

constexpr int BM = 128, BN = 256, BK = 64;        // BK: one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr int kPrefetch = 8;  // k blocks of W pulled into L2 ahead of the ring
constexpr int kABytes = BM * BK * 2;                // 16 KB
constexpr int kBAtomBytes = BK * 64 * 2;            // 8 KB: BK rows x 64 columns of W
constexpr int kBBytes = (BN / 64) * kBAtomBytes;    // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;      // 48 KB
constexpr int kSmemBytes = kStages * kStageBytes + 1024;  // + slack to align to 1 KB

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits 4-5
// = 1), A and B bf16 (bits 7-9 and 10-12 = 1), A K-major (bit 15 = 0), B
// N-major (bit 16 = 1), N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                            ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (all >> 4), descriptor version 1 (bits 46-48),
// swizzle mode 2 = 128 B (bits 61-63).  Atoms are 1 KB aligned, so the base
// offset field (bits 49-51) stays 0.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// The address of `p` (in this CTA's shared memory) in the CTA of cluster rank
// `rank`, as a shared::cluster address.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

// A box into THIS CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (bar: shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Pull a box into L2 ahead of its shared-memory load (hides HBM latency that
// the shared-memory ring alone is too short to cover).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t tmem, uint64_t adesc, uint64_t bdesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(acc)
      : "memory");
}

// mbarrier arrival once every tcgen05 operation this thread issued is done
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// Pair form: one arrival on the barrier at shared::cluster address `bar` (in
// either CTA of the pair) once every tcgen05 operation this thread issued is
// done.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Arrival on a barrier of another CTA of the cluster, releasing this thread's
// earlier operations at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait with acquire at cluster scope (for arrivals from the peer CTA).
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                          uint32_t limit = 2048) {
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(500000u)
        : "memory");
    if (ok) return true;
  }
  return false;
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]),
        "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]),
        "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// ---------------------------------------------------------------------------
// 1. RMSNorm rows into the workspace; block 0 also clears the flag word.
// ---------------------------------------------------------------------------
constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const uint16_t* __restrict__ h,
                                                               const uint16_t* __restrict__ w,
                                                               float eps, uint16_t* __restrict__ y,
                                                               int H, uint32_t* flags) {
  __shared__ float part[kNormThreads / 32];
  pdl_launch_dependents();  // the GEMM may start its set-up meanwhile
  const int m = blockIdx.x, tid = threadIdx.x;
  if (m == 0 && tid == 0) *flags = 0u;
  const uint16_t* hr = h + (size_t)m * H;
  uint16_t* yr = y + (size_t)m * H;
  // the row's first kNormKeep * kNormThreads * 8 elements stay in registers
  // between the sum of squares and the scaling (no second read)
  constexpr int kNormKeep = 2;
  uint4 keep[kNormKeep];
  float ss = 0.f;
#pragma unroll
  for (int it = 0; it < kNormKeep; ++it) {
    const int k = (it * kNormThreads + tid) * 8;
    keep[it] = k < H ? *reinterpret_cast<const uint4*>(hr + k) : make_uint4(0u, 0u, 0u, 0u);
  }
  for (int k = (kNormKeep * kNormThreads + tid) * 8; k < H; k += kNormThreads * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(hr + k);
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(q[j]), b = bf16_hi(q[j]);
      ss = __fmaf_rn(a, a, ss);
      ss = __fmaf_rn(b, b, ss);
    }
  }
#pragma unroll
  for (int it = 0; it < kNormKeep; ++it) {
    const uint32_t q[4] = {keep[it].x, keep[it].y, keep[it].z, keep[it].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(q[j]), b = bf16_hi(q[j]);
      ss = __fmaf_rn(a, a, ss);
      ss = __fmaf_rn(b, b, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) part[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += part[i];
  const float r = rsqrtf(tot / (float)H + eps);
  const bool w16 = (reinterpret_cast<uintptr_t>(w) & 15u) == 0;  // (the weight needs only 2-byte alignment)
  auto scale = [&](const uint4& v, int k) {
    uint32_t wq[4];
    if (w16) {
      const uint4 wv = *reinterpret_cast<const uint4*>(w + k);
      wq[0] = wv.x;
      wq[1] = wv.y;
      wq[2] = wv.z;
      wq[3] = wv.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) wq[j] = (uint32_t)w[k + 2 * j] | ((uint32_t)w[k + 2 * j + 1] << 16);
    }
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = pack_bf16x2(bf16_lo(q[j]) * r * bf16_lo(wq[j]), bf16_hi(q[j]) * r * bf16_hi(wq[j]));
    *reinterpret_cast<uint4*>(yr + k) = make_uint4(o[0], o[1], o[2], o[3]);
  };
#pragma unroll
  for (int it = 0; it < kNormKeep; ++it) {
    const int k = (it * kNormThreads + tid) * 8;
    if (k < H) scale(keep[it], k);
  }
  for (int k = (kNormKeep * kNormThreads + tid) * 8; k < H; k += kNormThreads * 8)
    scale(*reinterpret_cast<const uint4*>(hr + k), k);
}

// Epilogue of one accumulator: this thread's TMEM lane is output row `row`
// (32 lanes per warp), columns n0 .. n0 + BNT - 1, read 32 at a time.
template <int BNT>
__device__ __forceinline__ void store_tile(void* out, int out_f32, int M, int N, int row, int n0,
                                           uint32_t tbase) {
#pragma unroll 1
  for (int c = 0; c < BNT; c += 32) {
    uint32_t v[32];
    tmem_ld32(tbase + (uint32_t)c, v);
    const int n = n0 + c;
    if (row >= M || n >= N) continue;
    if (out_f32) {
      float* o = static_cast<float*>(out) + (size_t)row * N + n;
      if (n + 32 <= N) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          reinterpret_cast<uint4*>(o)[q] = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      } else {
#pragma unroll
        for (int q = 0; q < 32; ++q)
          if (q < N - n) o[q] = __uint_as_float(v[q]);
      }
    } else {
      uint16_t* o = static_cast<uint16_t*>(out) + (size_t)row * N + n;
      uint32_t pk[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) pk[q] = pack_bf16x2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
      if (n + 32 <= N) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          reinterpret_cast<uint4*>(o)[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      } else {
#pragma unroll
        for (int q = 0; q < 32; ++q)
          if (q < N - n) o[q] = (uint16_t)((q & 1) ? (pk[q >> 1] >> 16) : (pk[q >> 1] & 0xffffu));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 2. The tcgen05 GEMM, persistent (one CTA per SM).  Warp 0 streams operand
//    tiles, warp 1 issues the MMAs into one of two TMEM accumulators (512
//    columns: tile i uses half i & 1), warps 2-5 drain the other accumulator
//    to global memory while the next tile accumulates.
//
//    2a. lmhead_gemm_kernel: 128 x BN tiles, one CTA each (M <= 128).
//    2b. lmhead_gemm_pair_kernel: 256 x BN tiles on a CTA pair (a cluster of
//        two).  The pair's leader issues tcgen05.mma.cta_group::2 (M = 256):
//        each CTA stages its own 128 rows of y and HALF of the tile's W
//        columns (BN / 2), and the tensor cores of the two SMs exchange the W
//        halves, so each SM's shared memory feeds half the W operand it
//        would feed alone - the traffic (TMA fill plus operand reads) that
//        capped the single-CTA kernel.  Both CTAs' TMA loads complete on the
//        leader's stage barrier; the leader's commits free the stage in each
//        CTA; each CTA's epilogue reads its own TMEM rows and reports to the
//        leader before its accumulator is reused.
// ---------------------------------------------------------------------------
constexpr int kGemmThreads = 192;
constexpr uint32_t kTmemAlloc = 512;

template <int BNT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    lmhead_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       void* __restrict__ out, int out_f32, int M, int N, int K, uint32_t* flags) {
  static_assert(BNT % 16 == 0 && BNT >= 64 && BNT <= 256, "MMA N");
  constexpr int kAtoms = (BNT + 63) / 64;  // W tiles of 64 columns per stage
  constexpr uint32_t kTx = (uint32_t)(kABytes + kAtoms * kBAtomBytes);
  constexpr uint32_t kIdescT = (kIdesc & ~(0x3Fu << 17)) | ((uint32_t)(BNT >> 3) << 17);
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], accf[2], acce[2];
  __shared__ uint32_t tmem_base;
  __shared__ int issued, consumed, failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = (M + BM - 1) / BM, nt = (N + BNT - 1) / BNT;
  const int tiles = mt * nt;
  const int KB = K / BK;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 4);  // one arrival per epilogue warp
    }
    issued = consumed = failed = 0;
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base)),
                 "r"(kTmemAlloc)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  // The launch may overlap the RMSNorm kernel before it (programmatic stream
  // serialization): its set-up above runs meanwhile; the normalised rows, the
  // flag word and the output are touched only after that kernel completed.
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer: one stage counter across all tiles ----
      int g = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int m0 = (t % mt) * BM, n0 = (t / mt) * BNT;
        for (int kb = 0; kb < kPrefetch && kb < KB; ++kb)  // W boxes of the first k blocks into L2
#pragma unroll
          for (int j = 0; j < kAtoms; ++j) tma_prefetch_2d(&tmB, n0 + 64 * j, kb * BK);
        for (int kb = 0; kb < KB; ++kb, ++g) {
          if (kb + kPrefetch < KB) {
#pragma unroll
            for (int j = 0; j < kAtoms; ++j) tma_prefetch_2d(&tmB, n0 + 64 * j, (kb + kPrefetch) * BK);
          }
          const int s = g % kStages, use = g / kStages;
          if (use > 0 && !mbar_wait_bounded(&empty[s], (uint32_t)((use - 1) & 1))) {
            ok = false;
            break;
          }
          uint8_t* a = smem + s * kStageBytes;
          uint8_t* b = a + kABytes;
          mbar_arrive_expect_tx(&full[s], kTx);
          tma_load_2d(a, &tmA, kb * BK, m0, &full[s]);
#pragma unroll
          for (int j = 0; j < kAtoms; ++j) tma_load_2d(b + j * kBAtomBytes, &tmB, n0 + 64 * j, kb * BK, &full[s]);
        }
      }
      issued = g;
      if (!ok) {
        atomicOr(flags, SV_FLAG_TIMEOUT);
        failed = 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer ----
      int g = 0, i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++i) {
        const int b = i & 1, ub = i >> 1;
        if (ub > 0 && !mbar_wait_bounded(&acce[b], (uint32_t)((ub - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * 256);
        for (int kb = 0; kb < KB; ++kb, ++g) {
          const int s = g % kStages, use = g / kStages;
          if (!mbar_wait_bounded(&full[s], (uint32_t)(use & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_addr(smem + s * kStageBytes);
          const uint32_t bb = a + kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = desc_sw128(a + 32u * kk, 16u, 1024u);
            const uint64_t bd = desc_sw128(bb + 2048u * kk, (uint32_t)kBAtomBytes, 1024u);
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
            asm volatile(
                "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
                "l"(ad), "l"(bd), "r"(kIdescT), "r"(acc)
                : "memory");
          }
          tc_commit(&empty[s]);
        }
        if (!ok) break;
        tc_commit(&accf[b]);  // accumulator b complete
      }
      consumed = g;
      if (!ok) {
        atomicOr(flags, SV_FLAG_TIMEOUT);
        failed = 1;
      }
    }
  } else {
    // ---- epilogue warps 2..5: TMEM lanes 32*(warp % 4) .. +31 ----
    const int lg = warp & 3;
    int i = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
      const int b = i & 1, ub = i >> 1;
      const bool ok = mbar_wait_bounded(&accf[b], (uint32_t)(ub & 1));
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) atomicOr(flags, SV_FLAG_TIMEOUT);
        break;
      }
      tc_fence_after();
      const int m0 = (t % mt) * BM, n0 = (t / mt) * BNT;
      store_tile<BNT>(out, out_f32, M, N, m0 + lg * 32 + lane, n0,
                      tmem + (uint32_t)(b * 256) + ((uint32_t)(lg * 32) << 16));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[b]);  // accumulator b may be overwritten
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && failed) {
    // a wait ran out: let the copies already issued land before the CTA exits
    for (int g = consumed; g < issued; ++g)
      (void)mbar_wait_bounded(&full[g % kStages], (uint32_t)((g / kStages) & 1), 64);
  }
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemAlloc)
                 : "memory");
  }
}

// Pair tiles: MS sub-tiles of 256 rows (MS = 1 or 2) x BNT columns.  Each
// CTA stages, per k block, its 128 rows of every sub-tile and its half of the
// W columns, so a W tile is staged once for up to 512 rows.  TMEM holds two
// 256-column accumulators: two tiles in flight with one sub-tile (the
// epilogue of one overlaps the MMAs of the next), or one tile of two.
constexpr int kPairStageMax = 2 * kABytes + 2 * kBAtomBytes;  // 48 KB
constexpr int kPairSmemBytes = 4 * kPairStageMax + 1024;       // + slack to align to 1 KB

template <int MS>
struct PairShape {
  static constexpr int kStageBytes = MS * kABytes + 2 * kBAtomBytes;
  static constexpr int kStages = (kPairSmemBytes - 1024) / kStageBytes;  // 6 (MS 1) or 4 (MS 2)
  static constexpr int kBufs = 2 / MS;                                   // accumulator sets
};

template <int BNT, int MS>
__global__ void __launch_bounds__(kGemmThreads, 1)
    lmhead_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            void* __restrict__ out, int out_f32, int M, int N, int K, uint32_t* flags) {
  static_assert(BNT % 32 == 0 && BNT >= 128 && BNT <= 256, "pair MMA N (halves of 64..128 columns)");
  static_assert(MS == 1 || MS == 2, "sub-tiles per pair tile");
  using PS = PairShape<MS>;
  constexpr int kSt = PS::kStages, kSB = PS::kStageBytes, NB = PS::kBufs;
  constexpr int BH = BNT / 2;                  // W columns staged by each CTA of the pair
  constexpr int kAtomsH = (BH + 63) / 64;      // W boxes of 64 columns per CTA per stage
  static_assert(MS * kABytes + kAtomsH * kBAtomBytes <= kSB, "stage size");
  constexpr uint32_t kTxPair = 2u * (uint32_t)(MS * kABytes + kAtomsH * kBAtomBytes);  // both CTAs
  // M = 256 (two CTAs of 128 rows), N = BNT
  constexpr uint32_t kIdescP = (kIdesc & ~((0x3Fu << 17) | (0x1Fu << 24))) | ((uint32_t)(BNT >> 3) << 17) |
                               ((uint32_t)(256 >> 4) << 24);
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kSt], empty[kSt], accf[NB], acce[NB];
  __shared__ uint32_t tmem_base;
  __shared__ int issued, consumed, failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t half = blockIdx.x & 1u;  // cluster rank; 0 is the pair's leader
  const int pid = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
  constexpr int TR = MS * 2 * BM;  // rows of a pair tile
  const int mt2 = (M + TR - 1) / TR, nt = (N + BNT - 1) / BNT;
  const int tiles = mt2 * nt;  // pair tiles, numbered M-fastest
  const int KB = K / BK;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  if (tid == 0) {
    for (int s = 0; s < kSt; ++s) {
      mbar_init(&full[s], 1);   // (the leader's: its arrival + both CTAs' bytes)
      mbar_init(&empty[s], 1);  // one commit from the leader's MMA thread
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 8);  // (the leader's: four epilogue warps in each CTA)
    }
    issued = consumed = failed = 0;
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 0) {  // one warp of each CTA of the pair allocates, together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base)),
                 "r"(kTmemAlloc)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cg::this_cluster().sync();  // both CTAs' barriers and TMEM exist before any remote use
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer (both CTAs): own y rows, own half of W ----
      int g = 0;
      bool ok = true;
      for (int t = pid; t < tiles && ok; t += npairs) {
        const int m0 = (t % mt2) * TR + (int)half * BM;  // + 256 per sub-tile
        const int n0 = (t / mt2) * BNT + (int)half * BH;
        for (int kb = 0; kb < kPrefetch && kb < KB; ++kb)
#pragma unroll
          for (int j = 0; j < kAtomsH; ++j) tma_prefetch_2d(&tmB, n0 + 64 * j, kb * BK);
        for (int kb = 0; kb < KB; ++kb, ++g) {
          if (kb + kPrefetch < KB) {
#pragma unroll
            for (int j = 0; j < kAtomsH; ++j) tma_prefetch_2d(&tmB, n0 + 64 * j, (kb + kPrefetch) * BK);
          }
          const int s = g % kSt, use = g / kSt;
          if (use > 0 && !mbar_wait_bounded(&empty[s], (uint32_t)((use - 1) & 1))) {
            ok = false;
            break;
          }
          uint8_t* a = smem + s * kSB;
          uint8_t* b = a + MS * kABytes;
          if (half == 0) mbar_arrive_expect_tx(&full[s], kTxPair);
          const uint32_t fb = cluster_addr(&full[s], 0u);  // the leader's stage barrier
#pragma unroll
          for (int ms = 0; ms < MS; ++ms) tma_load_2d_pair(a + ms * kABytes, &tmA, kb * BK, m0 + ms * 2 * BM, fb);
#pragma unroll
          for (int j = 0; j < kAtomsH; ++j) tma_load_2d_pair(b + j * kBAtomBytes, &tmB, n0 + 64 * j, kb * BK, fb);
        }
      }
      issued = g;
      if (!ok) {
        atomicOr(flags, SV_FLAG_TIMEOUT);
        failed = 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && half == 0) {  // ---- MMA issuer: the leader only ----
      int g = 0, i = 0;
      bool ok = true;
      for (int t = pid; t < tiles && ok; t += npairs, ++i) {
        const int b = i % NB, ub = i / NB;
        if (ub > 0 && !mbar_wait_cluster_bounded(&acce[b], (uint32_t)((ub - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb, ++g) {
          const int s = g % kSt, use = g / kSt;
          if (!mbar_wait_bounded(&full[s], (uint32_t)(use & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_addr(smem + s * kSB);
          const uint32_t bb = a + MS * kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bd = desc_sw128(bb + 2048u * kk, (uint32_t)kBAtomBytes, 1024u);
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
#pragma unroll
            for (int ms = 0; ms < MS; ++ms) {
              const uint64_t ad = desc_sw128(a + (uint32_t)(ms * kABytes) + 32u * kk, 16u, 1024u);
              const uint32_t d = tmem + (uint32_t)((b * MS + ms) * 256);
              asm volatile(
                  "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                  " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
                  "l"(ad), "l"(bd), "r"(kIdescP), "r"(acc)
                  : "memory");
            }
          }
          // the stage is free in both CTAs once these MMAs are done
          tc_commit_pair(cluster_addr(&empty[s], 0u));
          tc_commit_pair(cluster_addr(&empty[s], 1u));
        }
        if (!ok) break;
        tc_commit_pair(cluster_addr(&accf[b], 0u));  // accumulators complete in both CTAs
        tc_commit_pair(cluster_addr(&accf[b], 1u));
      }
      consumed = g;
      if (!ok) {
        atomicOr(flags, SV_FLAG_TIMEOUT);
        failed = 1;
      }
    }
  } else {
    // ---- epilogue warps 2..5 (both CTAs): this CTA's 128 rows of each sub-tile ----
    const int lg = warp & 3;
    int i = 0;
    for (int t = pid; t < tiles; t += npairs, ++i) {
      const int b = i % NB, ub = i / NB;
      const bool ok = mbar_wait_bounded(&accf[b], (uint32_t)(ub & 1));
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) atomicOr(flags, SV_FLAG_TIMEOUT);
        break;
      }
      tc_fence_after();
      const int m0 = (t % mt2) * TR + (int)half * BM, n0 = (t / mt2) * BNT;
#pragma unroll 1
      for (int ms = 0; ms < MS; ++ms)
        store_tile<BNT>(out, out_f32, M, N, m0 + ms * 2 * BM + lg * 32 + lane, n0,
                        tmem + (uint32_t)((b * MS + ms) * 256) + ((uint32_t)(lg * 32) << 16));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(cluster_addr(&acce[b], 0u));  // (the leader's barrier)
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && failed && half == 0) {
    // a wait ran out: let the copies already issued (by both CTAs, counted on
    // the leader's barriers) land before the pair exits
    for (int g = consumed; g < issued; ++g)
      (void)mbar_wait_bounded(&full[g % kSt], (uint32_t)((g / kSt) & 1), 64);
  }
  cg::this_cluster().sync();  // no CTA leaves while its peer may still signal or read it
  tc_fence_after();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemAlloc)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

static std::mutex g_mutex;
static EncodeTiledFn g_encode = nullptr;

// SM count per device (device properties are per device in CUDA)
static int num_sms() {
  static std::atomic<int> cache[sv::kMaxDevices];
  const int d = sv::current_device();
  if (d < 0) return 148;
  int n = cache[d].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n < 1) n = 148;
    cache[d].store(n, std::memory_order_relaxed);
  }
  return n;
}

static EncodeTiledFn encoder(std::string* err) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
      *err = std::string("cuTensorMapEncodeTiled is not available: ") + cudaGetErrorString(e);
      return nullptr;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

// 2-D bf16 tensor map: inner extent `inner` (contiguous), `outer` rows of
// `row_bytes`, box {box_inner, box_outer}, 128-byte swizzle, zero fill.
static bool make_map(EncodeTiledFn enc, CUtensorMap* map, const void* base, uint64_t inner,
                     uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                     std::string* err) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

struct GemmArgs {
  CUtensorMap a, b;
  void* out;
  int out_f32, M, N, K;
  uint32_t* flags;
};

// Launch configuration of the persistent GEMM: clusters of `cm` CTAs (1: no
// cluster; 2: the pair kernel), `smem` dynamic bytes.
static void gemm_cfg(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int grid, int cm, int smem,
                     cudaStream_t st) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = dim3((unsigned)grid, 1, 1);
  cfg->blockDim = dim3(kGemmThreads, 1, 1);
  cfg->dynamicSmemBytes = (size_t)smem;
  cfg->stream = st;
  int n = 0;
  if (cm > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cm;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg->attrs = attr;
  cfg->numAttrs = (unsigned)n;
}

// Work units (CTAs, or CTA pairs for PAIR) that can be resident at once: the
// grid of the persistent kernel.  0 if the query fails.  Queried once per
// device (it also sets the kernel's shared-memory attribute there).
template <int BNT, int MS>  // MS 0: the single-CTA kernel; 1, 2: pair tiles of MS sub-tiles
static int resident_units() {
  constexpr bool PAIR = MS > 0;
  static std::atomic<int> cache[sv::kMaxDevices];  // units + 1; 0: not queried yet
  const int d = sv::current_device();
  if (d < 0) return 0;
  int n = cache[d].load(std::memory_order_acquire) - 1;
  if (n < 0) {
    auto k = PAIR ? lmhead_gemm_pair_kernel<BNT, MS ? MS : 1> : lmhead_gemm_kernel<BNT>;
    const int smem = PAIR ? kPairSmemBytes : kSmemBytes;
    int c = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
      if (PAIR) {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[1];
        gemm_cfg(&cfg, attr, 2 * 64, 2, smem, nullptr);
        if (cudaOccupancyMaxActiveClusters(&c, k, &cfg) != cudaSuccess) c = 0;
      } else {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kGemmThreads, smem) == cudaSuccess)
          c = per_sm * num_sms();
      }
    }
    n = c;
    cache[d].store(c + 1, std::memory_order_release);
  }
  return n;
}

template <int BNT, int MS>
static cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t st, int* grid_out) {
  constexpr bool PAIR = MS > 0;
  const int rows = PAIR ? MS * 2 * BM : BM;
  const int tiles = ((g.M + rows - 1) / rows) * ((g.N + BNT - 1) / BNT);
  int act = resident_units<BNT, MS>();
  if (act <= 0) act = PAIR ? num_sms() / 2 : num_sms();
  const int units = tiles < act ? tiles : act;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  gemm_cfg(&cfg, attr, units * (PAIR ? 2 : 1), PAIR ? 2 : 1, PAIR ? kPairSmemBytes : kSmemBytes, st);
  // the set-up (barriers, TMEM, tensor maps) overlaps the RMSNorm kernel
  attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs += 1;
  *grid_out = units * (PAIR ? 2 : 1);
  return cudaLaunchKernelEx(&cfg, PAIR ? lmhead_gemm_pair_kernel<BNT, MS ? MS : 1> : lmhead_gemm_kernel<BNT>,
                            g.a, g.b, g.out, g.out_f32, g.M, g.N, g.K, g.flags);
}

// Tile width: the fewest rounds of tiles over the resident units, weighted
// by the width (the columns one tile computes), then the widest.
template <int MS>
static cudaError_t launch_widest(const GemmArgs& g, cudaStream_t st, int* grid_out) {
  constexpr bool PAIR = MS > 0;
  const int rows = PAIR ? MS * 2 * BM : BM;
  const int mt = (g.M + rows - 1) / rows;
  const int widths[5] = {256, 224, 192, 160, 128};
  const int acts[5] = {resident_units<256, MS>(), resident_units<224, MS>(), resident_units<192, MS>(),
                       resident_units<160, MS>(), resident_units<128, MS>()};
  int best = 0;
  long long best_cost = -1;
  for (int i = 0; i < 5; ++i) {
    const long long act = acts[i] > 0 ? acts[i] : (PAIR ? num_sms() / 2 : num_sms());
    const long long tiles = (long long)mt * ((g.N + widths[i] - 1) / widths[i]);
    const long long cost = ((tiles + act - 1) / act) * widths[i];
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = i;
    }
  }
  switch (widths[best]) {
    case 224: return launch_gemm<224, MS>(g, st, grid_out);
    case 192: return launch_gemm<192, MS>(g, st, grid_out);
    case 160: return launch_gemm<160, MS>(g, st, grid_out);
    case 128: return launch_gemm<128, MS>(g, st, grid_out);
    default: return launch_gemm<256, MS>(g, st, grid_out);
  }
}

}  // namespace lmh

size_t lmhead_workspace_bytes(int M, int H) { return 256 + (size_t)M * H * 2 + 256; }

int lmhead_launch(const void* hidden, const void* norm_w, float eps, const void* W, void* logits,
                  sv_dtype out_dtype, int M, int H, int V, void* workspace, size_t ws_bytes,
                  void* stream, std::string* err) {
  (void)ws_bytes;
  using namespace lmh;
  EncodeTiledFn enc = encoder(err);
  if (!enc) return SV_ERR_CUDA;
  uint32_t* flags = static_cast<uint32_t*>(workspace);
  uint16_t* y = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + 256);
  GemmArgs g;
  if (!make_map(enc, &g.a, y, (uint64_t)H, (uint64_t)M, (uint64_t)H * 2, BK, BM, err)) return SV_ERR_CUDA;
  if (!make_map(enc, &g.b, W, (uint64_t)V, (uint64_t)H, (uint64_t)V * 2, 64, BK, err)) return SV_ERR_CUDA;
  g.out = logits;
  g.out_f32 = out_dtype == SV_F32 ? 1 : 0;
  g.M = M;
  g.N = V;
  g.K = H;
  g.flags = flags;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rmsnorm_kernel<<<M, kNormThreads, 0, st>>>(static_cast<const uint16_t*>(hidden),
                                             static_cast<const uint16_t*>(norm_w), eps, y, H, flags);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("rmsnorm launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  // more than one row tile: tiles of 256 (M <= 256) or 512 rows on CTA pairs
  // (tcgen05 cta_group::2)
  int grid = 0;
  {
    std::lock_guard<std::mutex> lock(g_mutex);  // one-time attribute setup inside
    e = M > 2 * BM ? launch_widest<2>(g, st, &grid)
                   : (M > BM ? launch_widest<1>(g, st, &grid) : launch_widest<0>(g, st, &grid));
  }
  if (e != cudaSuccess) {
    *err = std::string("lmhead launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

}  // namespace sv
