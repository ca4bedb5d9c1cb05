// Dynamic draft length ("Self-speculative decoding with layer skip and KV
// reuse", §3.2 and §5.3): each sequence's k follows its acceptance rate over
// the last 64 rounds in which it proposed drafts; k grows by one when that
// rate crosses above 0.85 and shrinks by one when it crosses below 0.7, within
// [2, 8].  An optional cap per sequence (for instance from the context
// length) bounds the k handed to the next round, and below 2 the round does
// not speculate.  One thread per sequence; the state lives in device memory
// between calls.
#include <cstdint>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

constexpr int kWindow = 64;
constexpr int kKMin = 2, kKMax = 8;

// Per-sequence state, structure of arrays in one buffer:
//   int32 k[B], head[B], count[B], acc[B], prop[B], pacc[B], pprop[B];
//   uint8 ring_acc[B][64], ring_prop[B][64].
// pacc/pprop: the window sums after the previous update (pprop < 0: none).
struct DynkState {
  int32_t *k, *head, *count, *acc, *prop, *pacc, *pprop;
  uint8_t *racc, *rprop;
};

__host__ __device__ inline DynkState dynk_view(void* base, int B) {
  char* p = static_cast<char*>(base);
  DynkState s;
  s.k = reinterpret_cast<int32_t*>(p);
  s.head = s.k + B;
  s.count = s.head + B;
  s.acc = s.count + B;
  s.prop = s.acc + B;
  s.pacc = s.prop + B;
  s.pprop = s.pacc + B;
  s.racc = reinterpret_cast<uint8_t*>(s.pprop + B);
  s.rprop = s.racc + (size_t)B * kWindow;
  return s;
}

size_t dynk_state_bytes(int B) {
  return (size_t)B * (7 * sizeof(int32_t) + 2 * kWindow);
}

__global__ void dynk_init_kernel(DynkState s, int B, int k0) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  s.k[b] = k0 < kKMin ? kKMin : (k0 > kKMax ? kKMax : k0);
  s.head[b] = s.count[b] = s.acc[b] = s.prop[b] = s.pacc[b] = 0;
  s.pprop[b] = -1;
}

// exact tests of the window rate against the thresholds
__device__ __forceinline__ bool above(int a, int p) { return p > 0 && 20 * a > 17 * p; }
__device__ __forceinline__ bool below(int a, int p) { return p > 0 && 10 * a < 7 * p; }

__global__ void dynk_update_kernel(DynkState s, int B, const int32_t* __restrict__ n_accepted,
                                   const int32_t* __restrict__ k_used,
                                   const int32_t* __restrict__ cap, int32_t* __restrict__ k_next,
                                   uint32_t* flags) {
  pdl_wait();  // the launch may overlap the kernel that wrote n_accepted
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  int k = s.k[b];
  const int ku = k_used[b], n = n_accepted[b];
  if (ku < 0 || ku > 255 || n < 0 || n > ku) {
    atomicOr(flags, SV_FLAG_BAD_N);  // the round is not recorded
  } else if (ku > 0) {
    int head = s.head[b], count = s.count[b], acc = s.acc[b], prop = s.prop[b];
    uint8_t* ra = s.racc + (size_t)b * kWindow;
    uint8_t* rp = s.rprop + (size_t)b * kWindow;
    if (count == kWindow) {  // the oldest round leaves the window
      acc -= ra[head];
      prop -= rp[head];
    } else {
      ++count;
    }
    ra[head] = (uint8_t)n;
    rp[head] = (uint8_t)ku;
    head = head + 1 == kWindow ? 0 : head + 1;
    acc += n;
    prop += ku;
    const int pa = s.pacc[b], pp = s.pprop[b];
    if (pp >= 0) {
      if (above(acc, prop) && !above(pa, pp)) k = k + 1 > kKMax ? kKMax : k + 1;
      else if (below(acc, prop) && !below(pa, pp)) k = k - 1 < kKMin ? kKMin : k - 1;
    }
    s.k[b] = k;
    s.head[b] = head;
    s.count[b] = count;
    s.acc[b] = acc;
    s.prop[b] = prop;
    s.pacc[b] = acc;
    s.pprop[b] = prop;
  }
  int kn = k;
  if (cap && cap[b] < kn) kn = cap[b];
  k_next[b] = kn >= kKMin ? kn : 0;
}

int dynk_init_launch(void* state, int B, int k0, void* stream, std::string* err) {
  const int threads = 256, blocks = (B + threads - 1) / threads;
  dynk_init_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(dynk_view(state, B), B, k0);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("dynk init launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

int dynk_update_launch(void* state, int B, const int32_t* n_accepted, const int32_t* k_used,
                       const int32_t* cap, int32_t* k_next, uint32_t* flags, void* stream,
                       std::string* err) {
  const int threads = 256, blocks = (B + threads - 1) / threads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, dynk_update_kernel, dynk_view(state, B), B, n_accepted,
                                     k_used, cap, k_next, flags);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("dynk update launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

}  // namespace sv
