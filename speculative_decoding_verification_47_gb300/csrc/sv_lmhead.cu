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
//  2. lmhead_gemm_kernel: one CTA per 128 x 256 output tile on the 5th-
//     generation tensor cores.  A 4-stage ring in shared memory is filled by
//     the TMA engine (cp.async.bulk.tensor, 128-byte swizzle): y tiles
//     K-major (128 rows x 64 k), W tiles N-major (64 k x 64 n, four per
//     stage).  One thread issues tcgen05.mma (M=128, N=256, K=16, bf16 in,
//     fp32 accumulator in tensor memory) and tcgen05.commit frees each stage
//     once its MMAs are done; the four warps then read the accumulator back
//     with tcgen05.ld and store bf16 (or fp32) logits.  Tiles are numbered
//     M-fastest, so the four row tiles that share a W column block run side
//     by side and W streams from HBM about once.
#include <cuda.h>  // CUtensorMap and the encoder's signature (resolved at run time)

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
constexpr int kABytes = BM * BK * 2;                // 16 KB
constexpr int kBAtomBytes = BK * 64 * 2;            // 8 KB: BK rows x 64 columns of W
constexpr int kBBytes = (BN / 64) * kBAtomBytes;    // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;      // 48 KB
constexpr int kSmemBytes = kStages * kStageBytes + 1024;  // + slack to align to 1 KB
constexpr int kThreads = 128;                       // one warpgroup: the 128 TMEM lanes
constexpr uint32_t kTmemCols = BN;                  // fp32 accumulator columns

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
  const int m = blockIdx.x, tid = threadIdx.x;
  if (m == 0 && tid == 0) *flags = 0u;
  const uint16_t* hr = h + (size_t)m * H;
  float ss = 0.f;
  for (int k = tid * 8; k < H; k += kNormThreads * 8) {
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
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) part[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += part[i];
  const float r = rsqrtf(tot / (float)H + eps);
  uint16_t* yr = y + (size_t)m * H;
  for (int k = tid * 8; k < H; k += kNormThreads * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(hr + k);
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float w0 = bf16_lo((uint32_t)w[k + 2 * j]), w1 = bf16_lo((uint32_t)w[k + 2 * j + 1]);
      o[j] = pack_bf16x2(bf16_lo(q[j]) * r * w0, bf16_hi(q[j]) * r * w1);
    }
    *reinterpret_cast<uint4*>(yr + k) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ---------------------------------------------------------------------------
// 2. The tcgen05 GEMM.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       void* __restrict__ out, int out_f32, int M, int N, int K, uint32_t* flags) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], done;
  __shared__ uint32_t tmem_base;
  __shared__ int issued, consumed, failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = (M + BM - 1) / BM;
  const int m0 = (blockIdx.x % mt) * BM, n0 = (blockIdx.x / mt) * BN;
  const int KB = K / BK;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    issued = consumed = failed = 0;
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 0) {  // the whole warp allocates the accumulator's TMEM columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer ----
    int kb = 0;
    for (; kb < KB; ++kb) {
      const int s = kb % kStages, use = kb / kStages;
      if (use > 0 && !mbar_wait_bounded(&empty[s], (uint32_t)((use - 1) & 1))) {
        atomicOr(flags, SV_FLAG_TIMEOUT);
        failed = 1;
        break;
      }
      uint8_t* a = smem + s * kStageBytes;
      uint8_t* b = a + kABytes;
      mbar_arrive_expect_tx(&full[s], (uint32_t)kStageBytes);
      tma_load_2d(a, &tmA, kb * BK, m0, &full[s]);
#pragma unroll
      for (int j = 0; j < BN / 64; ++j) tma_load_2d(b + j * kBAtomBytes, &tmB, n0 + 64 * j, kb * BK, &full[s]);
    }
    issued = kb;
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    int kb = 0;
    for (; kb < KB; ++kb) {
      const int s = kb % kStages, use = kb / kStages;
      if (!mbar_wait_bounded(&full[s], (uint32_t)(use & 1))) {
        atomicOr(flags, SV_FLAG_TIMEOUT);
        failed = 1;
        break;
      }
      tc_fence_after();
      const uint32_t a = smem_addr(smem + s * kStageBytes);
      const uint32_t b = a + kABytes;
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        // A: next 16 k = 32 bytes along the swizzled row; B: next 16 k rows
        // = two 8-row groups of 1 KB; B's 64-column atoms are kBAtomBytes apart
        tc_mma(tmem, desc_sw128(a + 32u * kk, 16u, 1024u),
               desc_sw128(b + 2048u * kk, (uint32_t)kBAtomBytes, 1024u), (kb | kk) != 0 ? 1u : 0u);
      }
      tc_commit(&empty[s]);
    }
    consumed = kb;
    tc_commit(&done);  // arrives when every MMA issued above has completed
  }
  __syncwarp();

  // ---- epilogue: TMEM -> registers -> global ----
  const bool ok = mbar_wait_bounded(&done, 0u);
  if (!ok && lane == 0) atomicOr(flags, SV_FLAG_TIMEOUT);
  tc_fence_after();
  const int row = m0 + warp * 32 + lane;
  if (__all_sync(0xffffffffu, ok)) {
    for (int c = 0; c < BN; c += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
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
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && failed) {
    // a wait ran out: let the copies already issued land before the CTA exits
    for (int kb = consumed; kb < issued; ++kb)
      (void)mbar_wait_bounded(&full[kb % kStages], (uint32_t)((kb / kStages) & 1), 64);
  }
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
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
static int g_configured = 0;

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
  CUtensorMap tmA, tmB;
  if (!make_map(enc, &tmA, y, (uint64_t)H, (uint64_t)M, (uint64_t)H * 2, BK, BM, err)) return SV_ERR_CUDA;
  if (!make_map(enc, &tmB, W, (uint64_t)V, (uint64_t)H, (uint64_t)V * 2, 64, BK, err)) return SV_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_configured) {
      const cudaError_t e =
          cudaFuncSetAttribute(lmhead_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) {
        *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
        return SV_ERR_CUDA;
      }
      g_configured = 1;
    }
  }
  rmsnorm_kernel<<<M, kNormThreads, 0, st>>>(static_cast<const uint16_t*>(hidden),
                                             static_cast<const uint16_t*>(norm_w), eps, y, H, flags);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("rmsnorm launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  const int tiles = ((M + BM - 1) / BM) * ((V + BN - 1) / BN);
  lmhead_gemm_kernel<<<tiles, kThreads, kSmemBytes, st>>>(tmA, tmB, logits, out_dtype == SV_F32 ? 1 : 0,
                                                          M, V, H, flags);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("lmhead launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

}  // namespace sv
