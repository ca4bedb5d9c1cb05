// KV write-pointer rollback after verification [SSD §3.3, §4.3] ("Self-
// speculative decoding with layer skip and KV reuse"); [SD §4.3]
// ("Speculative decoding, the founding scheme"): the pointer that stood at the
// round-start length while the drafts were written moves to
// seq_len + n_accepted, and entries at or beyond it are stale.
#include <cstdint>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {

__global__ void kv_commit_kernel(int32_t* __restrict__ seq_lens,
                                 const int32_t* __restrict__ n_accepted,
                                 const int32_t* __restrict__ capacity, int B, int K,
                                 uint32_t* __restrict__ flags) {
  pdl_wait();  // the launch may overlap the kernel that wrote n_accepted
  uint32_t f = 0;
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
    const int n = n_accepted[b];
    if (n < 0 || (K >= 0 && n > K)) {
      f |= SV_FLAG_BAD_N;
      continue;
    }
    const long long nl = (long long)seq_lens[b] + n;
    if ((capacity && nl > capacity[b]) || nl > 0x7fffffffLL) {
      f |= SV_FLAG_CAPACITY;
      continue;
    }
    seq_lens[b] = (int32_t)nl;
  }
  if (f) atomicOr(flags, f);
}

int commit_launch(int32_t* seq_lens, const int32_t* n_accepted, const int32_t* capacity, int B,
                  int K, uint32_t* flags, void* stream, std::string* err) {
  int blocks = (B + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kv_commit_kernel, seq_lens, n_accepted, capacity, B, K, flags);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("kv_commit launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

}  // namespace sv
