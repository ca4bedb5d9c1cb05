// Host-side interfaces between the C ABI (sv_api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>

#include <cuda_runtime.h>

#include "../../include/specverify.h"

namespace sv {

struct VerifyLaunch {
  const void* target;
  long long t_seq, t_pos;  // elements
  const void* draft;
  long long d_seq, d_pos;  // elements
  sv_dtype dtype;
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
  void* workspace;
  void* stream;
  int topp_draft = 1;  // top_p < 1: truncate the draft rows too (1) or only the target rows (0)
};

// Enqueue the verify step.  Returns an sv_status; fills *err on failure.
int verify_launch(const VerifyLaunch& L, std::string* err);

struct SampleLaunch {
  const void* logits;
  long long l_seq, l_pos;  // elements
  sv_dtype dtype;
  int B, K, V;
  const int32_t* kpr;
  const float* temp;
  float top_p;
  const float* unif;
  const uint8_t* mode;
  int32_t* out;
  void* workspace;
  void* stream;
};

// Enqueue the draft-side sampler.  Returns an sv_status; fills *err on failure.
int sample_launch(const SampleLaunch& L, std::string* err);
size_t verify_workspace_bytes(int B, int K);

// Allocation-free verify: scratch in a fixed device array of this size
// (L.workspace is ignored).
constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;
constexpr int kMaxDevices = 64;

// The calling thread's current device, for state kept per device (kernel
// attributes and device properties are per device in CUDA): -1 if there is
// none or its ordinal is kMaxDevices or more.
inline int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}
int verify_launch_noalloc(const VerifyLaunch& L, std::string* err);

size_t dynk_state_bytes(int B);
int dynk_init_launch(void* state, int B, int k0, void* stream, std::string* err);
int dynk_update_launch(void* state, int B, const int32_t* n_accepted, const int32_t* k_used,
                       const int32_t* cap, int32_t* k_next, uint32_t* flags, void* stream,
                       std::string* err);

int paged_commit_launch(int32_t* seq_lens, const int32_t* n_accepted, const int32_t* k_per_row,
                        int32_t* block_table, int max_pages, int page_size, int32_t* free_pages,
                        int32_t* free_top, int free_capacity, int B, uint32_t* ws, void* stream,
                        std::string* err);

int commit_launch(int32_t* seq_lens, const int32_t* n_accepted, const int32_t* capacity,
                  const int32_t* k_per_row, int B,
                  int K, uint32_t* flags, void* stream, std::string* err);

int lmhead_launch(const void* hidden, const void* norm_w, float eps, const void* W, void* logits,
                  sv_dtype out_dtype, int M, int H, int V, void* workspace, size_t ws_bytes,
                  void* stream, std::string* err);
size_t lmhead_workspace_bytes(int M, int H);

}  // namespace sv
