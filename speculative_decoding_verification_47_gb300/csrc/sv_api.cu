// extern "C" entry points of libspecverify.so: argument checks, workspace
// sizing and error reporting around the kernels' launchers.
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "sv_internal.h"

namespace {

thread_local std::string g_last_error;

sv_status fail(sv_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

constexpr int kMaxK = 20;
constexpr long long kMaxItems = 0x7fffffffLL / 16;  // items per call: the grid is items x <= 16 CTAs
constexpr int kMaxSeqs = 1 << 30;                   // one thread per sequence

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

int sv_version(void) { return 100; }

size_t sv_workspace_size(int B, int K, int V, sv_dtype dt) {
  if (B < 1 || K < 0 || K > kMaxK || V < 1 || (dt != SV_F32 && dt != SV_BF16)) return 0;
  return sv::verify_workspace_bytes(B, K);
}

size_t sv_lmhead_workspace_size(int M, int H) {
  if (M < 1 || H < 1) return 0;
  return sv::lmhead_workspace_bytes(M, H);
}

// Host-checkable arguments of the three verify entry points; fills *L with
// everything but the workspace.
static sv_status verify_args(const void* target_logits, int64_t target_seq_stride,
                             int64_t target_pos_stride, const void* draft_logits,
                             int64_t draft_seq_stride, int64_t draft_pos_stride, sv_dtype dtype,
                             int B, int K, int V, const int32_t* draft_tokens,
                             const int32_t* k_per_row, const float* temperature, float top_p,
                             const float* uniforms, const uint8_t* mode, int32_t* out_tokens,
                             int32_t* n_accepted, float* diag, void* stream,
                             sv::VerifyLaunch* L) {
  if (dtype != SV_F32 && dtype != SV_BF16) return fail(SV_ERR_DTYPE, "dtype must be SV_F32 or SV_BF16");
  if (B < 1 || K < 0 || K > kMaxK || V < 1)
    return fail(SV_ERR_SHAPE, "need B >= 1, 0 <= K <= 20, V >= 1");
  // one cluster of up to 16 CTAs per (sequence, position): the grid must fit 2^31 - 1 blocks
  if ((long long)B * (K + 1) > kMaxItems)
    return fail(SV_ERR_SHAPE, "B * (K + 1) must be at most 134217727");
  if (!target_logits || !uniforms || !out_tokens || !n_accepted)
    return fail(SV_ERR_ARG, "target_logits, uniforms, out_tokens and n_accepted are required");
  if (K > 0 && !draft_tokens) return fail(SV_ERR_ARG, "draft_tokens is required when K > 0");
  if (K > 0 && !draft_logits && !mode)
    return fail(SV_ERR_ARG, "draft_logits may be NULL only when every row is greedy (mode given)");
  if (!(top_p > 0.0f && top_p <= 1.0f)) return fail(SV_ERR_ARG, "top_p must be in (0, 1]");
  const int es = dtype == SV_BF16 ? 2 : 4;
  if (!aligned(target_logits, es) || (draft_logits && !aligned(draft_logits, es)))
    return fail(SV_ERR_ARG, "logit pointers must be aligned to their element size");
  const long long Vl = V;
  const long long ts = target_seq_stride ? target_seq_stride : (long long)(K + 1) * Vl;
  const long long tp = target_pos_stride ? target_pos_stride : Vl;
  const long long ds = draft_seq_stride ? draft_seq_stride : (long long)K * Vl;
  const long long dp = draft_pos_stride ? draft_pos_stride : Vl;
  if (ts < 0 || tp < 0 || ds < 0 || dp < 0) return fail(SV_ERR_SHAPE, "strides must be >= 0");
  if (tp < Vl && K > 0) return fail(SV_ERR_SHAPE, "target position stride is smaller than V");
  if (dp < Vl && K > 1) return fail(SV_ERR_SHAPE, "draft position stride is smaller than V");
  L->target = target_logits;
  L->t_seq = ts;
  L->t_pos = tp;
  L->draft = draft_logits;
  L->d_seq = ds;
  L->d_pos = dp;
  L->dtype = dtype;
  L->B = B;
  L->K = K;
  L->V = V;
  L->tokens = draft_tokens;
  L->kpr = k_per_row;
  L->temp = temperature;
  L->top_p = top_p;
  L->unif = uniforms;
  L->mode = mode;
  L->out = out_tokens;
  L->nacc = n_accepted;
  L->diag = diag;
  L->workspace = nullptr;
  L->stream = stream;
  return SV_OK;
}

static sv_status spec_verify_impl(const void* target_logits, int64_t target_seq_stride,
                                  int64_t target_pos_stride, const void* draft_logits,
                                  int64_t draft_seq_stride, int64_t draft_pos_stride,
                                  sv_dtype dtype, int B, int K, int V, const int32_t* draft_tokens,
                                  const int32_t* k_per_row, const float* temperature, float top_p,
                                  const float* uniforms, const uint8_t* mode, int32_t* out_tokens,
                                  int32_t* n_accepted, float* diag, void* workspace,
                                  size_t workspace_bytes, void* stream, int topp_draft) {
  sv::VerifyLaunch L;
  const sv_status a = verify_args(target_logits, target_seq_stride, target_pos_stride,
                                  draft_logits, draft_seq_stride, draft_pos_stride, dtype, B, K,
                                  V, draft_tokens, k_per_row, temperature, top_p, uniforms, mode,
                                  out_tokens, n_accepted, diag, stream, &L);
  if (a != SV_OK) return a;
  if (!workspace || !aligned(workspace, 256))
    return fail(SV_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
  if (workspace_bytes < sv::verify_workspace_bytes(B, K))
    return fail(SV_ERR_WORKSPACE, "workspace smaller than sv_workspace_size()");
  L.workspace = workspace;
  L.topp_draft = topp_draft;
  std::string err;
  int s = sv::verify_launch(L, &err);
  if (s != SV_OK) return fail(static_cast<sv_status>(s), err);
  return SV_OK;
}

sv_status sv_spec_verify(const void* target_logits, int64_t target_seq_stride,
                         int64_t target_pos_stride, const void* draft_logits,
                         int64_t draft_seq_stride, int64_t draft_pos_stride, sv_dtype dtype,
                         int B, int K, int V, const int32_t* draft_tokens,
                         const int32_t* k_per_row, const float* temperature, float top_p,
                         const float* uniforms, const uint8_t* mode, int32_t* out_tokens,
                         int32_t* n_accepted, float* diag, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return spec_verify_impl(target_logits, target_seq_stride, target_pos_stride, draft_logits,
                          draft_seq_stride, draft_pos_stride, dtype, B, K, V, draft_tokens,
                          k_per_row, temperature, top_p, uniforms, mode, out_tokens, n_accepted,
                          diag, workspace, workspace_bytes, stream, 1);
}

sv_status sv_spec_verify_target_topp(const void* target_logits, int64_t target_seq_stride,
                                     int64_t target_pos_stride, const void* draft_logits,
                                     int64_t draft_seq_stride, int64_t draft_pos_stride,
                                     sv_dtype dtype, int B, int K, int V,
                                     const int32_t* draft_tokens, const int32_t* k_per_row,
                                     const float* temperature, float top_p, const float* uniforms,
                                     const uint8_t* mode, int32_t* out_tokens, int32_t* n_accepted,
                                     float* diag, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  return spec_verify_impl(target_logits, target_seq_stride, target_pos_stride, draft_logits,
                          draft_seq_stride, draft_pos_stride, dtype, B, K, V, draft_tokens,
                          k_per_row, temperature, top_p, uniforms, mode, out_tokens, n_accepted,
                          diag, workspace, workspace_bytes, stream, 0);
}

sv_status sv_spec_verify_noalloc(const void* target_logits, int64_t target_seq_stride,
                                 int64_t target_pos_stride, const void* draft_logits,
                                 int64_t draft_seq_stride, int64_t draft_pos_stride,
                                 sv_dtype dtype, int B, int K, int V, const int32_t* draft_tokens,
                                 const int32_t* k_per_row, const float* temperature, float top_p,
                                 const float* uniforms, const uint8_t* mode, int32_t* out_tokens,
                                 int32_t* n_accepted, float* diag, void* stream) {
  sv::VerifyLaunch L;
  const sv_status a = verify_args(target_logits, target_seq_stride, target_pos_stride,
                                  draft_logits, draft_seq_stride, draft_pos_stride, dtype, B, K,
                                  V, draft_tokens, k_per_row, temperature, top_p, uniforms, mode,
                                  out_tokens, n_accepted, diag, stream, &L);
  if (a != SV_OK) return a;
  std::string err;
  int s = sv::verify_launch_noalloc(L, &err);
  if (s != SV_OK) return fail(static_cast<sv_status>(s), err);
  return SV_OK;
}

sv_status sv_kv_commit(int32_t* seq_lens, const int32_t* n_accepted, const int32_t* capacity,
                       const int32_t* k_per_row, int B, int K, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (B < 1 || B > kMaxSeqs) return fail(SV_ERR_SHAPE, "need 1 <= B <= 2^30");
  if (!seq_lens || !n_accepted) return fail(SV_ERR_ARG, "seq_lens and n_accepted are required");
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < 256)
    return fail(SV_ERR_WORKSPACE, "workspace must be non-NULL, 256-byte aligned, >= 256 bytes");
  std::string err;
  int s = sv::commit_launch(seq_lens, n_accepted, capacity, k_per_row, B, K,
                            static_cast<uint32_t*>(workspace), stream, &err);
  if (s != SV_OK) return fail(static_cast<sv_status>(s), err);
  return SV_OK;
}

sv_status sv_kv_commit_paged(int32_t* seq_lens, const int32_t* n_accepted,
                             const int32_t* k_per_row, int32_t* block_table, int max_pages,
                             int page_size, int32_t* free_pages, int32_t* free_top,
                             int free_capacity, int B, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (B < 1 || B > kMaxSeqs || max_pages < 1 || page_size < 1 || free_capacity < 0)
    return fail(SV_ERR_SHAPE, "need 1 <= B <= 2^30, max_pages >= 1, page_size >= 1, free_capacity >= 0");
  // lengths and page counts are int32 on the device: a full table plus one page must fit
  if ((long long)max_pages * page_size + page_size > 0x7fffffffLL)
    return fail(SV_ERR_SHAPE, "(max_pages + 1) * page_size must fit in int32");
  if (!seq_lens || !n_accepted || !k_per_row || !block_table || !free_pages || !free_top)
    return fail(SV_ERR_ARG, "every array argument is required");
  if (!workspace || workspace_bytes < 16 || !aligned(workspace, 16))
    return fail(SV_ERR_WORKSPACE, "workspace must be non-NULL, 16-byte aligned and >= 16 bytes");
  std::string err;
  const int s = sv::paged_commit_launch(seq_lens, n_accepted, k_per_row, block_table, max_pages,
                                        page_size, free_pages, free_top, free_capacity, B,
                                        static_cast<uint32_t*>(workspace), stream, &err);
  if (s != SV_OK) return fail(static_cast<sv_status>(s), err);
  return SV_OK;
}

size_t sv_dynk_state_size(int B) { return B < 1 || B > kMaxSeqs ? 0 : sv::dynk_state_bytes(B); }

sv_status sv_dynk_init(void* state, int B, int k0, void* stream) {
  if (B < 1 || B > kMaxSeqs) return fail(SV_ERR_SHAPE, "need 1 <= B <= 2^30");
  if (!state || !aligned(state, 16)) return fail(SV_ERR_ARG, "state must be non-NULL and 16-byte aligned");
  std::string err;
  const int s = sv::dynk_init_launch(state, B, k0, stream, &err);
  if (s != SV_OK) return fail(static_cast<sv_status>(s), err);
  return SV_OK;
}

sv_status sv_dynk_update(void* state, int B, const int32_t* n_accepted, const int32_t* k_used,
                         const int32_t* cap, int32_t* k_next, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (B < 1 || B > kMaxSeqs) return fail(SV_ERR_SHAPE, "need 1 <= B <= 2^30");
  if (!state || !aligned(state, 16)) return fail(SV_ERR_ARG, "state must be non-NULL and 16-byte aligned");
  if (!n_accepted || !k_used || !k_next) return fail(SV_ERR_ARG, "n_accepted, k_used and k_next are required");
  if (!workspace || workspace_bytes < 4 || !aligned(workspace, 4))
    return fail(SV_ERR_WORKSPACE, "workspace (its flag word) must be non-NULL, aligned, >= 4 bytes");
  std::string err;
  const int s = sv::dynk_update_launch(state, B, n_accepted, k_used, cap, k_next,
                                       static_cast<uint32_t*>(workspace), stream, &err);
  if (s != SV_OK) return fail(static_cast<sv_status>(s), err);
  return SV_OK;
}

size_t sv_draft_sample_workspace_size(void) { return 256; }

sv_status sv_draft_sample(const void* draft_logits, int64_t seq_stride, int64_t pos_stride,
                          sv_dtype dtype, int B, int K, int V, const int32_t* k_per_row,
                          const float* temperature, float top_p, const float* uniforms,
                          const uint8_t* mode, int32_t* out_tokens, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (dtype != SV_F32 && dtype != SV_BF16) return fail(SV_ERR_DTYPE, "dtype must be SV_F32 or SV_BF16");
  if (B < 1 || K < 1 || V < 1) return fail(SV_ERR_SHAPE, "need B >= 1, K >= 1, V >= 1");
  if ((long long)B * K > kMaxItems) return fail(SV_ERR_SHAPE, "B * K must be at most 134217727");
  if (!draft_logits || !uniforms || !out_tokens)
    return fail(SV_ERR_ARG, "draft_logits, uniforms and out_tokens are required");
  if (!(top_p > 0.0f && top_p <= 1.0f)) return fail(SV_ERR_ARG, "top_p must be in (0, 1]");
  const int es = dtype == SV_BF16 ? 2 : 4;
  if (!aligned(draft_logits, es)) return fail(SV_ERR_ARG, "logits must be aligned to their element size");
  const long long Vl = V;
  const long long ss = seq_stride ? seq_stride : (long long)K * Vl;
  const long long ps = pos_stride ? pos_stride : Vl;
  if (ss < 0 || ps < 0) return fail(SV_ERR_SHAPE, "strides must be >= 0");
  if (ps < Vl && K > 1) return fail(SV_ERR_SHAPE, "position stride is smaller than V");
  if (!workspace || !aligned(workspace, 256))
    return fail(SV_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
  if (workspace_bytes < sv_draft_sample_workspace_size())
    return fail(SV_ERR_WORKSPACE, "workspace smaller than sv_draft_sample_workspace_size()");
  sv::SampleLaunch L;
  L.logits = draft_logits;
  L.l_seq = ss;
  L.l_pos = ps;
  L.dtype = dtype;
  L.B = B;
  L.K = K;
  L.V = V;
  L.kpr = k_per_row;
  L.temp = temperature;
  L.top_p = top_p;
  L.unif = uniforms;
  L.mode = mode;
  L.out = out_tokens;
  L.workspace = workspace;
  L.stream = stream;
  std::string err;
  const int s = sv::sample_launch(L, &err);
  if (s != SV_OK) return fail(static_cast<sv_status>(s), err);
  return SV_OK;
}

sv_status sv_lmhead_rmsnorm(const void* hidden, const void* norm_w, float eps, const void* W,
                            void* logits, sv_dtype out_dtype, int M, int H, int V,
                            void* workspace, size_t workspace_bytes, void* stream) {
  if (out_dtype != SV_F32 && out_dtype != SV_BF16) return fail(SV_ERR_DTYPE, "bad out_dtype");
  if (M < 1 || H < 64 || H % 64 != 0 || V < 16 || V % 16 != 0)
    return fail(SV_ERR_SHAPE, "need M >= 1, H % 64 == 0, V % 16 == 0");
  if (!hidden || !norm_w || !W || !logits) return fail(SV_ERR_ARG, "null pointer");
  if (!(eps >= 0.0f)) return fail(SV_ERR_ARG, "eps must be >= 0");
  if (!aligned(hidden, 16) || !aligned(W, 16) || !aligned(logits, 16) || !aligned(norm_w, 2))
    return fail(SV_ERR_ARG, "hidden, W and logits must be 16-byte aligned");
  if (!workspace || !aligned(workspace, 256))
    return fail(SV_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
  if (workspace_bytes < sv::lmhead_workspace_bytes(M, H))
    return fail(SV_ERR_WORKSPACE, "workspace smaller than sv_lmhead_workspace_size()");
  std::string err;
  int s = sv::lmhead_launch(hidden, norm_w, eps, W, logits, out_dtype, M, H, V, workspace,
                            workspace_bytes, stream, &err);
  if (s != SV_OK) return fail(static_cast<sv_status>(s), err);
  return SV_OK;
}

sv_status sv_read_device_flags(const void* workspace, uint32_t* flags_host, void* stream) {
  if (!workspace || !flags_host) return fail(SV_ERR_ARG, "null pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(flags_host, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, std::string("reading flags: ") + cudaGetErrorString(e));
  if (*flags_host == 0) return SV_OK;
  if (*flags_host & SV_FLAG_TIMEOUT) return fail(SV_ERR_TIMEOUT, "a bounded device wait ran out");
  return fail(SV_ERR_DEVICE_FLAG, "device flag word is non-zero");
}

const char* sv_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
