// markov.cu — a2-a4: the gamma-step sequential (Markov) head with the
// confidence head.
//
// "DSpark 深度解读" §二 设计一: x_k is sampled from base logits plus the low-rank
// transition bias W1[x_{k-1}] W2; §二 设计二: c_k = sigmoid(w^T [h_k; W1[x_{k-1}]])
// calibrated per position by a temperature T_k.  "DSpark整体架构": the anchor is
// the first prediction position, so x_0 = anchor.
//
// Per step k the library runs: step_prep (gather E = W1[x_{k-1}], confidence
// c_k), one vocabulary pass (bias + base logits + decision, logits stay on
// chip), and row_reduce (combine the per-tile partials into x_k, lse_k, logp_k).
#include "logits_tile.cuh"

DSPARK_DECLARE_STATUS(s_status_markov)

namespace {

// zh[m] = w_h . h[m] for every (request, position) row m; one warp per row.
__global__ void conf_hidden(const bf16 *__restrict__ h, const bf16 *__restrict__ w_conf,
                            float *__restrict__ zh, int rows, int d) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const uint4 *hr = reinterpret_cast<const uint4 *>(h + (size_t)warp * d);
  const uint4 *wr = reinterpret_cast<const uint4 *>(w_conf);
  float acc = 0.f;
  for (int c = lane; c < d / 8; c += 32) {
    const uint4 a = hr[c], b = wr[c];
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      acc = fmaf(bf16_lo(av[t]), bf16_lo(bv[t]), acc);
      acc = fmaf(bf16_hi(av[t]), bf16_hi(bv[t]), acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) zh[warp] = acc;
}

// Step k: E[i] = W1[x_{k-1}], c_k = sigmoid((zh + w_e . E[i]) / T_k); one warp per request.
__global__ void step_prep(const int32_t *__restrict__ anchor, const int32_t *__restrict__ tokens,
                          const bf16 *__restrict__ W1, const bf16 *__restrict__ w_e,
                          const float *__restrict__ zh, const float *__restrict__ T,
                          bf16 *__restrict__ E, float *__restrict__ conf, int R, int gamma,
                          int V, int r, int k) {
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (i >= R) return;
  int prev = (k == 1) ? anchor[i] : tokens[(size_t)i * gamma + k - 2];
  if (prev < 0 || prev >= V) {
    if (lane == 0) dspark_set_status(DSPARK_ERR_TOKEN);
    prev = 0;
  }
  const uint4 *src = reinterpret_cast<const uint4 *>(W1 + (size_t)prev * r);
  uint4 *dst = reinterpret_cast<uint4 *>(E + (size_t)i * r);
  const uint4 *wr = reinterpret_cast<const uint4 *>(w_e);
  float acc = 0.f;
  for (int c = lane; c < r / 8; c += 32) {
    const uint4 a = src[c], b = wr[c];
    dst[c] = a;
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      acc = fmaf(bf16_lo(av[t]), bf16_lo(bv[t]), acc);
      acc = fmaf(bf16_hi(av[t]), bf16_hi(bv[t]), acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) {
    const size_t o = (size_t)i * gamma + k - 1;
    const float z = zh[o] + acc;
    conf[o] = 1.f / (1.f + expf(-z / T[k - 1]));
  }
}

// Combine the vocabulary-tile partials of each row into x_k, lse_k, logp_k.
template <int MODE>
__global__ void row_reduce(const RowPartial *__restrict__ part, int n_tiles, int R, int gamma,
                           int k, int32_t *__restrict__ tokens, float *__restrict__ lse_out,
                           float *__restrict__ logp_out) {
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (i >= R) return;
  float m = -INFINITY, s = 0.f, best = -INFINITY, bs = 0.f;
  int idx = 0x7fffffff;
  for (int t = lane; t < n_tiles; t += 32) {
    const RowPartial p = part[(size_t)i * n_tiles + t];
    lse_merge(m, s, p.m, p.sum);
    if (better(p.best, p.idx, best, idx)) { best = p.best; idx = p.idx; bs = p.best_s; }
  }
  warp_merge(m, s, best, idx, bs);
  if (lane == 0) {
    const size_t o = (size_t)i * gamma + k - 1;
    tokens[o] = idx;
    float lse = 0.f, logp = 0.f;
    if (MODE == MODE_SAMPLE) {
      lse = m + logf(s);
      logp = bs - lse;
    }
    if (lse_out) lse_out[o] = lse;
    if (logp_out) logp_out[o] = logp;
  }
}

struct MarkovWs {
  float *zh;
  bf16 *E;
  RowPartial *part;
  size_t bytes;
};

MarkovWs markov_layout(const dspark_dims *d, char *base) {
  MarkovWs w;
  size_t off = 0;
  w.zh = (float *)(base + off);
  off = dspark_align_up(off + sizeof(float) * (size_t)d->R * d->gamma, 256);
  w.E = (bf16 *)(base + off);
  off = dspark_align_up(off + sizeof(bf16) * (size_t)d->R * d->r, 256);
  w.part = (RowPartial *)(base + off);
  const size_t n_tiles = (d->V + TN - 1) / TN;
  off = dspark_align_up(off + sizeof(RowPartial) * (size_t)d->R * n_tiles, 256);
  w.bytes = off;
  return w;
}

}  // namespace

extern "C" size_t dspark_markov_workspace_bytes(const dspark_dims *dims) {
  if (!dspark_dims_ok(dims)) return 0;
  return markov_layout(dims, nullptr).bytes;
}

extern "C" int dspark_markov_draft(const dspark_dims *dims, const void *base_logits,
                                   const void *h, const int32_t *anchor, const void *W1,
                                   const void *W2t, const void *w_conf, const float *T,
                                   float tau, uint64_t seed, int32_t *tokens, float *conf,
                                   float *logp_d, float *lse_d, void *workspace,
                                   size_t workspace_bytes, dspark_stream_t stream) {
  if (!dspark_dims_ok(dims) || !base_logits || !h || !anchor || !W1 || !W2t || !w_conf || !T ||
      !tokens || !conf || !(tau >= 0.f))
    return DSPARK_ERR_ARG;
  MarkovWs ws = markov_layout(dims, (char *)workspace);
  if (!workspace || workspace_bytes < ws.bytes || ((uintptr_t)workspace & 255))
    return DSPARK_ERR_WORKSPACE;
  const int R = dims->R, G = dims->gamma, V = dims->V, r = dims->r, d = dims->d;
  const int rows = R * G;
  conf_hidden<<<(rows * 32 + 255) / 256, 256, 0, stream>>>((const bf16 *)h, (const bf16 *)w_conf,
                                                          ws.zh, rows, d);
  DSPARK_CHECK_LAUNCH();
  TileArgs ta;
  ta.base = (const bf16 *)base_logits;
  ta.E = ws.E;
  ta.W2t = (const bf16 *)W2t;
  ta.target = nullptr;
  ta.rows = nullptr;
  ta.part = ws.part;
  ta.M = R;
  ta.V = V;
  ta.r = r;
  ta.gamma = G;
  ta.n_tiles = (V + TN - 1) / TN;
  ta.inv_tau = tau > 0.f ? 1.f / tau : 1.f;
  ta.seed = seed;
  const dim3 tgrid(ta.n_tiles, (R + TM - 1) / TM);
  for (int k = 1; k <= G; ++k) {
    step_prep<<<(R * 32 + 255) / 256, 256, 0, stream>>>(
        anchor, tokens, (const bf16 *)W1, (const bf16 *)w_conf + d, ws.zh, T, ws.E, conf, R, G,
        V, r, k);
    DSPARK_CHECK_LAUNCH();
    ta.k = k;
    if (tau > 0.f) {
      logits_tile_simple<MODE_SAMPLE><<<tgrid, 256, 0, stream>>>(ta);
      DSPARK_CHECK_LAUNCH();
      row_reduce<MODE_SAMPLE><<<(R * 32 + 255) / 256, 256, 0, stream>>>(
          ws.part, ta.n_tiles, R, G, k, tokens, lse_d, logp_d);
    } else {
      logits_tile_simple<MODE_GREEDY><<<tgrid, 256, 0, stream>>>(ta);
      DSPARK_CHECK_LAUNCH();
      row_reduce<MODE_GREEDY><<<(R * 32 + 255) / 256, 256, 0, stream>>>(
          ws.part, ta.n_tiles, R, G, k, tokens, lse_d, logp_d);
    }
    DSPARK_CHECK_LAUNCH();
  }
  dspark_count_launches(1 + 3 * (uint64_t)G);
  return DSPARK_OK;
}

int dspark_status_markov(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, s_status_markov, sizeof(int)) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (clear) {
    const int z = 0;
    cudaMemcpyToSymbol(s_status_markov, &z, sizeof(int));
  }
  return v;
}
