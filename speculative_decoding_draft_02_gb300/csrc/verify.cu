// verify.cu — a8: verification of the admitted draft prefixes.
//
// "DSpark整体架构" Fig. 1: the target checks the scheduled prefix in parallel,
// keeps the accepted run and emits one corrected token G* at the first
// rejection; "DSpark 深度解读" §二: the procedure recovers the target
// distribution exactly.  The rule is standard speculative sampling:
//   accept x_j iff u * p_d(x_j) < p_t(x_j); on the first rejection sample
//   norm(max(0, p_t - p_d)); if all l_r drafts pass, sample target row l_r + 1.
// Greedy (tau = 0): accept iff x_j = argmax t_j; emit the argmax of the first
// failing row (or of row l_r + 1).
//
// Pass 1 (verify_rows) scans each target row 1..l_r+1 once: its argmax, its
// log-sum-exp and the drafted token's logit.  Pass 2 (verify_decide) walks each
// request.  Sampling only: pass 3 rebuilds p_d on the rejected row through the
// same fused vocabulary pass as the draft (bias + base logits, on chip) and
// draws the residual, or draws the bonus from the target row.
#include "logits_tile.cuh"

DSPARK_DECLARE_STATUS(s_status_verify)

namespace {

struct __align__(16) RowStat {
  int32_t argmax;  // argmax_v t[v]          (greedy)
  float lse_t;     // logsumexp(t / tau)     (sampling)
  float tx;        // t[x_j] / tau           (sampling, rows with a draft token)
  int32_t pad;
};

__device__ __forceinline__ int clamp_len(const int32_t *len, int i, int gamma) {
  int L = len[i];
  if (L < 0 || L > gamma) {
    dspark_set_status(DSPARK_ERR_LENGTH);
    L = L < 0 ? 0 : gamma;
  }
  return L;
}

// One CTA per (row j, request i) with j <= l_i: argmax or log-sum-exp over V.
template <int MODE>
__global__ void __launch_bounds__(256) verify_rows(const bf16 *__restrict__ target,
                                                   const int32_t *__restrict__ tokens,
                                                   const int32_t *__restrict__ len,
                                                   RowStat *__restrict__ stat, int gamma,
                                                   int V, float inv_tau) {
  const int j = blockIdx.x, i = blockIdx.y;  // j: 0-based row (position j + 1)
  const int L = clamp_len(len, i, gamma);
  if (j > L) return;
  const bf16 *row = target + ((size_t)i * (gamma + 1) + j) * V;
  const uint4 *row4 = reinterpret_cast<const uint4 *>(row);
  float m = -INFINITY, s = 0.f, best = -INFINITY, bs = 0.f;
  int idx = 0x7fffffff;
  for (int c = threadIdx.x; c < V / 8; c += blockDim.x) {
    const uint4 q = row4[c];
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    float vals[8];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      vals[2 * t] = bf16_lo(w[t]);
      vals[2 * t + 1] = bf16_hi(w[t]);
    }
    if (MODE == MODE_GREEDY) {
#pragma unroll
      for (int t = 0; t < 8; ++t)
        if (better(vals[t], c * 8 + t, best, idx)) { best = vals[t]; idx = c * 8 + t; }
    } else {
      float cm = vals[0] * inv_tau;
#pragma unroll
      for (int t = 1; t < 8; ++t) cm = fmaxf(cm, vals[t] * inv_tau);
      float cs = 0.f;
#pragma unroll
      for (int t = 0; t < 8; ++t) cs += __expf(vals[t] * inv_tau - cm);
      lse_merge(m, s, cm, cs);
    }
  }
  warp_merge(m, s, best, idx, bs);
  __shared__ float sm[8], ss[8], sb[8];
  __shared__ int si[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { sm[warp] = m; ss[warp] = s; sb[warp] = best; si[warp] = idx; }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    m = lane < nw ? sm[lane] : -INFINITY;
    s = lane < nw ? ss[lane] : 0.f;
    best = lane < nw ? sb[lane] : -INFINITY;
    idx = lane < nw ? si[lane] : 0x7fffffff;
    warp_merge(m, s, best, idx, bs);
    if (lane == 0) {
      RowStat st;
      st.argmax = idx;
      st.lse_t = m + logf(s);
      st.tx = 0.f;
      st.pad = 0;
      if (MODE != MODE_GREEDY && j < L) {
        int x = tokens[(size_t)i * gamma + j];
        if (x < 0 || x >= V) { dspark_set_status(DSPARK_ERR_TOKEN); x = 0; }
        st.tx = __bfloat162float(row[x]) * inv_tau;
      }
      stat[(size_t)i * (gamma + 1) + j] = st;
    }
  }
}

// Walk each request's admitted prefix; one thread per request.
template <int MODE>
__global__ void verify_decide(const RowStat *__restrict__ stat, const int32_t *__restrict__ anchor,
                              const int32_t *__restrict__ tokens, const int32_t *__restrict__ len,
                              const float *__restrict__ lse_d, const float *__restrict__ logp_d,
                              ResampleRow *__restrict__ rows, int32_t *__restrict__ accepted,
                              int32_t *__restrict__ bonus, int R, int gamma, int V, uint64_t seed) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= R) return;
  const int L = clamp_len(len, i, gamma);
  const RowStat *st = stat + (size_t)i * (gamma + 1);
  const int32_t *x = tokens + (size_t)i * gamma;
  int n = L;
  if (MODE == MODE_GREEDY) {
    for (int j = 1; j <= L; ++j)
      if (x[j - 1] != st[j - 1].argmax) { n = j - 1; break; }
    accepted[i] = n;
    bonus[i] = st[n].argmax;
    return;
  }
  ResampleRow rr;
  rr.kind = KIND_BONUS;
  rr.pos = L + 1;
  rr.prev = 0;
  rr.lse_t = st[L].lse_t;
  rr.lse_d = 0.f;
  rr.pad[0] = rr.pad[1] = rr.pad[2] = 0;
  for (int j = 1; j <= L; ++j) {
    const uint4 w = rng_words4(seed, 0u, (uint32_t)j, (uint32_t)i, RNG_ACCEPT);
    const float u = rng_uniform(w.x);
    const size_t o = (size_t)i * gamma + j - 1;
    const float margin = logf(u) + logp_d[o] - (st[j - 1].tx - st[j - 1].lse_t);
    if (margin < 0.f) continue;  // u * p_d(x_j) < p_t(x_j): accepted
    n = j - 1;
    rr.kind = KIND_RESIDUAL;
    rr.pos = j;
    int prev = (j == 1) ? anchor[i] : x[j - 2];
    if (prev < 0 || prev >= V) { dspark_set_status(DSPARK_ERR_TOKEN); prev = 0; }
    rr.prev = prev;
    rr.lse_t = st[j - 1].lse_t;
    rr.lse_d = lse_d[o];
    break;
  }
  accepted[i] = n;
  rows[i] = rr;
}

// E[i] = W1[x_{j*-1}] for residual rows, zero elsewhere; one warp per request.
__global__ void resample_gather(const ResampleRow *__restrict__ rows, const bf16 *__restrict__ W1,
                                bf16 *__restrict__ E, int R, int r) {
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (i >= R) return;
  const ResampleRow rr = rows[i];
  uint4 *dst = reinterpret_cast<uint4 *>(E + (size_t)i * r);
  const uint4 *src = reinterpret_cast<const uint4 *>(W1 + (size_t)rr.prev * r);
  for (int c = lane; c < r / 8; c += 32)
    dst[c] = rr.kind == KIND_RESIDUAL ? src[c] : make_uint4(0, 0, 0, 0);
}

// Bonus rows: Gumbel-max over target row pos (stream 3), 128 entries per tile;
// one warp per request, 8 requests per CTA.
__global__ void __launch_bounds__(256) bonus_tile(const ResampleRow *__restrict__ rows,
                                                  const bf16 *__restrict__ target,
                                                  RowPartial *__restrict__ part, int R,
                                                  int gamma, int V, int n_tiles, float inv_tau,
                                                  uint64_t seed) {
  const int i = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (i >= R) return;
  const ResampleRow rr = rows[i];
  if (rr.kind != KIND_BONUS) return;
  const bf16 *trow = target + ((size_t)i * (gamma + 1) + rr.pos - 1) * V;
  const int n0 = blockIdx.x * TN;
  float best = -INFINITY, bs = 0.f, m = -INFINITY, s = 0.f;
  int idx = 0x7fffffff;
  // each lane owns 4 consecutive entries: one Philox call per lane
  const int v0 = n0 + lane * 4;
  if (v0 < V) {
    const uint4 w = rng_words4(seed, (uint32_t)(v0 >> 2), (uint32_t)rr.pos, (uint32_t)i, RNG_BONUS);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int v = v0 + t;
      if (v < V) {
        const float sc = __bfloat162float(trow[v]) * inv_tau + rng_gumbel(uint4_get(w, t));
        if (better(sc, v, best, idx)) { best = sc; idx = v; }
      }
    }
  }
  warp_merge(m, s, best, idx, bs);
  if (lane == 0) {
    RowPartial p;
    p.m = -INFINITY; p.sum = 0.f; p.best = best; p.idx = idx; p.best_s = 0.f;
    p.pad0 = -INFINITY; p.pad1 = __int_as_float(0x7fffffff); p.pad2 = 0.f;
    part[(size_t)i * n_tiles + blockIdx.x] = p;
  }
}

// Final residual / bonus token per request.
__global__ void resample_reduce(const ResampleRow *__restrict__ rows,
                                const RowPartial *__restrict__ part, int n_tiles, int R,
                                int32_t *__restrict__ bonus) {
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (i >= R) return;
  if (rows[i].kind == KIND_NONE) return;
  float best = -INFINITY, fb = -INFINITY, d0 = 0.f, d1 = 0.f, d2 = 0.f, e0 = 0.f, e1 = 0.f,
        e2 = 0.f;
  int idx = 0x7fffffff, fidx = 0x7fffffff;
  for (int t = lane; t < n_tiles; t += 32) {
    const RowPartial p = part[(size_t)i * n_tiles + t];
    if (better(p.best, p.idx, best, idx)) { best = p.best; idx = p.idx; }
    const int pi = __float_as_int(p.pad1);
    if (better(p.pad0, pi, fb, fidx)) { fb = p.pad0; fidx = pi; }
  }
  warp_merge(d0, d1, best, idx, d2);
  warp_merge(e0, e1, fb, fidx, e2);
  if (lane == 0) bonus[i] = (best > -INFINITY) ? idx : fidx;
}

struct VerifyWs {
  RowStat *stat;
  ResampleRow *rows;
  bf16 *E;
  RowPartial *part;
  size_t bytes;
};

VerifyWs verify_layout(const dspark_dims *d, char *base) {
  VerifyWs w;
  size_t off = 0;
  w.stat = (RowStat *)(base + off);
  off = dspark_align_up(off + sizeof(RowStat) * (size_t)d->R * (d->gamma + 1), 256);
  w.rows = (ResampleRow *)(base + off);
  off = dspark_align_up(off + sizeof(ResampleRow) * (size_t)d->R, 256);
  w.E = (bf16 *)(base + off);
  off = dspark_align_up(off + sizeof(bf16) * (size_t)d->R * d->r, 256);
  w.part = (RowPartial *)(base + off);
  const size_t n_tiles = (d->V + TN - 1) / TN;
  off = dspark_align_up(off + sizeof(RowPartial) * (size_t)d->R * n_tiles, 256);
  w.bytes = off;
  return w;
}

}  // namespace

extern "C" size_t dspark_verify_workspace_bytes(const dspark_dims *dims) {
  if (!dspark_dims_ok(dims)) return 0;
  return verify_layout(dims, nullptr).bytes;
}

extern "C" int dspark_verify(const dspark_dims *dims, const int32_t *anchor, const int32_t *tokens,
                             const int32_t *len, const void *base_logits, const void *W1,
                             const void *W2t, const float *lse_d, const float *logp_d,
                             const void *target, float tau, uint64_t seed, int32_t *accepted,
                             int32_t *bonus, void *workspace, size_t workspace_bytes,
                             dspark_stream_t stream) {
  if (!dspark_dims_ok(dims) || !tokens || !len || !target || !accepted || !bonus || !(tau >= 0.f))
    return DSPARK_ERR_ARG;
  const bool sample = tau > 0.f;
  if (sample && (!anchor || !base_logits || !W1 || !W2t || !lse_d || !logp_d)) return DSPARK_ERR_ARG;
  VerifyWs ws = verify_layout(dims, (char *)workspace);
  if (!workspace || workspace_bytes < ws.bytes || ((uintptr_t)workspace & 255))
    return DSPARK_ERR_WORKSPACE;
  const int R = dims->R, G = dims->gamma, V = dims->V, r = dims->r;
  const float inv_tau = sample ? 1.f / tau : 1.f;
  const dim3 rgrid(G + 1, R);
  if (!sample) {
    verify_rows<MODE_GREEDY><<<rgrid, 256, 0, stream>>>((const bf16 *)target, tokens, len,
                                                        ws.stat, G, V, inv_tau);
    DSPARK_CHECK_LAUNCH();
    verify_decide<MODE_GREEDY><<<(R + 127) / 128, 128, 0, stream>>>(
        ws.stat, anchor, tokens, len, lse_d, logp_d, ws.rows, accepted, bonus, R, G, V, seed);
    DSPARK_CHECK_LAUNCH();
    dspark_count_launches(2);
    return DSPARK_OK;
  }
  verify_rows<MODE_SAMPLE><<<rgrid, 256, 0, stream>>>((const bf16 *)target, tokens, len, ws.stat,
                                                      G, V, inv_tau);
  DSPARK_CHECK_LAUNCH();
  verify_decide<MODE_SAMPLE><<<(R + 127) / 128, 128, 0, stream>>>(
      ws.stat, anchor, tokens, len, lse_d, logp_d, ws.rows, accepted, bonus, R, G, V, seed);
  DSPARK_CHECK_LAUNCH();
  resample_gather<<<(R * 32 + 255) / 256, 256, 0, stream>>>(ws.rows, (const bf16 *)W1, ws.E, R, r);
  DSPARK_CHECK_LAUNCH();
  TileArgs ta;
  ta.base = (const bf16 *)base_logits;
  ta.E = ws.E;
  ta.W2t = (const bf16 *)W2t;
  ta.target = (const bf16 *)target;
  ta.rows = ws.rows;
  ta.part = ws.part;
  ta.M = R;
  ta.V = V;
  ta.r = r;
  ta.gamma = G;
  ta.k = 0;
  ta.n_tiles = (V + TN - 1) / TN;
  ta.inv_tau = inv_tau;
  ta.seed = seed;
  logits_tile_simple<MODE_RESIDUAL><<<dim3(ta.n_tiles, (R + TM - 1) / TM), 256, 0, stream>>>(ta);
  DSPARK_CHECK_LAUNCH();
  bonus_tile<<<dim3(ta.n_tiles, (R + 7) / 8), 256, 0, stream>>>(ws.rows, (const bf16 *)target,
                                                              ws.part, R, G, V, ta.n_tiles,
                                                              inv_tau, seed);
  DSPARK_CHECK_LAUNCH();
  resample_reduce<<<(R * 32 + 255) / 256, 256, 0, stream>>>(ws.rows, ws.part, ta.n_tiles, R, bonus);
  DSPARK_CHECK_LAUNCH();
  dspark_count_launches(6);
  return DSPARK_OK;
}

int dspark_status_verify(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, s_status_verify, sizeof(int)) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (clear) {
    const int z = 0;
    cudaMemcpyToSymbol(s_status_verify, &z, sizeof(int));
  }
  return v;
}
