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
                                 const int32_t* __restrict__ capacity,
                                 const int32_t* __restrict__ k_per_row, int B, int K,
                                 uint32_t* __restrict__ flags) {
  pdl_wait();  // the launch may overlap the kernel that wrote n_accepted
  uint32_t f = 0;
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
    const int n = n_accepted[b];
    // more accepted than this sequence drafted: the pointer would move past
    // the entries the round wrote
    if (n < 0 || (K >= 0 && n > K) || (k_per_row && n > k_per_row[b])) {
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

int commit_launch(int32_t* seq_lens, const int32_t* n_accepted, const int32_t* capacity,
                  const int32_t* k_per_row, int B, int K, uint32_t* flags, void* stream,
                  std::string* err) {
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, kv_commit_kernel, seq_lens, n_accepted, capacity, k_per_row, B, K,
                                     flags);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("kv_commit launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

// ---------------------------------------------------------------------------
// Paged-KV commit ([SSD §3.3, §4.5]): the cache of sequence b is a block table
// of pages of P tokens.  After verification its length is L' = L + n; pages
// 0 .. ceil(L'/P)-1 stay and every allocated page from index ceil(L'/P) on
// goes back to the free stack (its table entry becomes -1).  Two launches:
// the first checks every sequence and counts the call's releases (and keeps
// the free stack's top as it was), the second applies them all, or none if
// together they would overflow the free stack.  Scratch: workspace words 1
// (release count) and 2 (the top before the call).
// ---------------------------------------------------------------------------

__device__ __forceinline__ bool paged_ok(int L, int n, int k, int max_pages, int P) {
  return k >= 0 && (long long)L + k <= (long long)max_pages * P && n >= 0 && n <= k && L >= 0;
}

// One warp per sequence: the lanes read its block-table row together (lane
// q holds entries q, q + 32, ...), so the row is read coalesced and counted by
// ballots.
__global__ void paged_count_kernel(const int32_t* __restrict__ seq_lens,
                                   const int32_t* __restrict__ n_accepted,
                                   const int32_t* __restrict__ k_per_row,
                                   const int32_t* __restrict__ table, int max_pages, int P, int B,
                                   const int32_t* __restrict__ free_top, uint32_t* ws) {
  pdl_wait();  // the launch may overlap the kernel that wrote n_accepted
  const int lane = threadIdx.x & 31;
  const int b = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (b == 0 && lane == 0) ws[2] = (uint32_t)*free_top;
  if (b >= B) return;  // (whole warps)
  const int L = seq_lens[b], n = n_accepted[b], k = k_per_row[b];
  if (!paged_ok(L, n, k, max_pages, P)) {
    if (lane == 0) atomicOr(ws, SV_FLAG_BAD_N);
    return;
  }
  const int keep = (L + n + P - 1) / P;
  const int32_t* row = table + (size_t)b * max_pages;
  uint32_t c = 0;
  for (int j0 = keep; j0 < max_pages; j0 += 32) {
    const int j = j0 + lane;
    c += __popc(__ballot_sync(0xffffffffu, j < max_pages && row[j] >= 0));
  }
  if (lane == 0 && c) atomicAdd(ws + 1, c);
}

__global__ void paged_apply_kernel(int32_t* __restrict__ seq_lens,
                                   const int32_t* __restrict__ n_accepted,
                                   const int32_t* __restrict__ k_per_row, int32_t* __restrict__ table,
                                   int max_pages, int P, int B, int32_t* __restrict__ free_pages,
                                   int32_t* __restrict__ free_top, int free_capacity, uint32_t* ws) {
  const int lane = threadIdx.x & 31;
  const int b = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if ((long long)ws[2] + ws[1] > (long long)free_capacity) {  // (the same test in every thread)
    if (b == 0 && lane == 0) atomicOr(ws, SV_FLAG_CAPACITY);
    return;
  }
  if (b >= B) return;  // (whole warps)
  const int L = seq_lens[b], n = n_accepted[b], k = k_per_row[b];
  if (!paged_ok(L, n, k, max_pages, P)) return;
  const int keep = (L + n + P - 1) / P;
  int32_t* row = table + (size_t)b * max_pages;
  int c = 0;
  for (int j0 = keep; j0 < max_pages; j0 += 32) {
    const int j = j0 + lane;
    c += __popc(__ballot_sync(0xffffffffu, j < max_pages && row[j] >= 0));
  }
  int pos = 0;
  if (lane == 0 && c) pos = atomicAdd(free_top, c);  // this sequence's places on the stack
  pos = __shfl_sync(0xffffffffu, pos, 0);
  for (int j0 = keep; j0 < max_pages; j0 += 32) {
    const int j = j0 + lane;
    const int32_t id = j < max_pages ? row[j] : -1;
    const unsigned m = __ballot_sync(0xffffffffu, id >= 0);
    if (id >= 0) free_pages[pos + __popc(m & ((1u << lane) - 1u))] = id;
    if (j < max_pages) row[j] = -1;
    pos += __popc(m);
  }
  if (lane == 0) seq_lens[b] = L + n;
}

int paged_commit_launch(int32_t* seq_lens, const int32_t* n_accepted, const int32_t* k_per_row,
                        int32_t* block_table, int max_pages, int page_size, int32_t* free_pages,
                        int32_t* free_top, int free_capacity, int B, uint32_t* ws, void* stream,
                        std::string* err) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws + 1, 0, sizeof(uint32_t), st);  // the release count
  const int threads = 256, blocks = (int)(((long long)B * 32 + threads - 1) / threads);  // a warp per sequence
  if (e == cudaSuccess) {
    paged_count_kernel<<<blocks, threads, 0, st>>>(seq_lens, n_accepted, k_per_row, block_table,
                                                  max_pages, page_size, B, free_top, ws);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    paged_apply_kernel<<<blocks, threads, 0, st>>>(seq_lens, n_accepted, k_per_row, block_table,
                                                  max_pages, page_size, B, free_pages, free_top,
                                                  free_capacity, ws);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    *err = std::string("paged kv_commit launch: ") + cudaGetErrorString(e);
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

}  // namespace sv
