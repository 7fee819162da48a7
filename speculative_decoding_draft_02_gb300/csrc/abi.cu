// abi.cu — C-ABI glue: argument checks, composition of a1..a4, the sticky
// device status word, error strings and the launch counter.
#include <atomic>

#include "common.cuh"

static std::atomic<uint64_t> g_launches{0};

void dspark_count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int dspark_lm_head_tc(const dspark_dims *, const void *, const void *, void *, cudaStream_t);
int dspark_status_lmhead(int clear);
int dspark_status_markov(int clear);
int dspark_status_verify(int clear);
int dspark_status_sched(int clear);
int dspark_status_sts(int clear);
int dspark_status_selftest(int clear);

extern "C" uint64_t dspark_launch_count(void) { return g_launches.load(); }

extern "C" const char *dspark_error_string(int code) {
  switch (code) {
    case DSPARK_OK: return "ok";
    case DSPARK_ERR_ARG: return "invalid argument";
    case DSPARK_ERR_SPS_SHORT: return "SPS table shorter than R*(gamma+1)";
    case DSPARK_ERR_CUDA: return "CUDA error";
    case DSPARK_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DSPARK_ERR_TOKEN: return "token id outside [0, V)";
    case DSPARK_ERR_LENGTH: return "verify length outside [0, gamma]";
    case DSPARK_ERR_TIMEOUT: return "device-side wait timed out";
    case DSPARK_ERR_TOO_LARGE: return "problem exceeds the library's static scratch";
    default: return "unknown error";
  }
}

extern "C" int dspark_device_status(dspark_stream_t stream, int clear) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  int first = DSPARK_OK;
  const int vals[6] = {dspark_status_lmhead(clear), dspark_status_markov(clear),
                       dspark_status_verify(clear), dspark_status_sched(clear),
                       dspark_status_sts(clear),    dspark_status_selftest(clear)};
  for (int v : vals)
    if (first == DSPARK_OK && v != DSPARK_OK) first = v;
  return first;
}

extern "C" int dspark_lm_head(const dspark_dims *dims, const void *h, const void *W_lm,
                              void *base_logits, dspark_stream_t stream) {
  if (!dspark_dims_ok(dims) || !h || !W_lm || !base_logits) return DSPARK_ERR_ARG;
  if (((uintptr_t)h | (uintptr_t)W_lm | (uintptr_t)base_logits) & 15) return DSPARK_ERR_ARG;
  return dspark_lm_head_tc(dims, h, W_lm, base_logits, stream);
}

extern "C" int dspark_draft(const dspark_dims *dims, const void *h, const int32_t *anchor,
                            const void *W_lm, const void *W1, const void *W2t,
                            const void *w_conf, const float *T, float tau, uint64_t seed,
                            void *base_logits, int32_t *tokens, float *conf, float *logp_d,
                            float *lse_d, void *workspace, size_t workspace_bytes,
                            dspark_stream_t stream) {
  if (!dspark_dims_ok(dims)) return DSPARK_ERR_ARG;
  if (!workspace || workspace_bytes < dspark_markov_workspace_bytes(dims))
    return DSPARK_ERR_WORKSPACE;
  int rc = dspark_lm_head(dims, h, W_lm, base_logits, stream);
  if (rc != DSPARK_OK) return rc;
  return dspark_markov_draft(dims, base_logits, h, anchor, W1, W2t, w_conf, T, tau, seed, tokens,
                             conf, logp_d, lse_d, workspace, workspace_bytes, stream);
}
