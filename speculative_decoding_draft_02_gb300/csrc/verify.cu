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

constexpr int NSEG = 4;  // CTAs per target row in the first pass

// Per (request, row, segment): online log-sum-exp of t / tau (sampling) or the
// argmax (greedy) over one quarter of the vocabulary.
struct __align__(16) SegStat {
  float m, s;      // sampling
  float best;      // greedy
  int32_t idx;     // greedy
};

__device__ __forceinline__ int clamp_len(const int32_t *len, int i, int gamma) {
  int L = len[i];
  if (L < 0 || L > gamma) {
    dspark_set_status(DSPARK_ERR_LENGTH);
    L = L < 0 ? 0 : gamma;
  }
  return L;
}

__device__ __forceinline__ int seg_len(int V) { return ((V + NSEG - 1) / NSEG + 7) / 8 * 8; }

// Pass 1: grid (NSEG * (gamma+1), R).  Greedy scans rows 1..l_r+1 (their
// argmaxes decide acceptance and give the correction or bonus token); sampling
// scans rows 1..l_r (their normalisers enter the acceptance test; the bonus
// row needs none).  Block (0, 0) also clears the residual-row counter.
template <int MODE>
__global__ void __launch_bounds__(256) verify_rows(const bf16 *__restrict__ target,
                                                   const int32_t *__restrict__ len,
                                                   SegStat *__restrict__ stat,
                                                   int *__restrict__ count, int gamma, int V,
                                                   float inv_tau) {
  const int j = blockIdx.x / NSEG, seg = blockIdx.x % NSEG, i = blockIdx.y;
  if (blockIdx.x == 0 && i == 0 && threadIdx.x == 0) *count = 0;
  const int L = clamp_len(len, i, gamma);
  if (MODE == MODE_GREEDY ? j > L : j >= L) return;
  const int sl = seg_len(V), v_beg = seg * sl, v_end = min(V, v_beg + sl);
  const bf16 *row = target + ((size_t)i * (gamma + 1) + j) * V;
  const uint4 *row4 = reinterpret_cast<const uint4 *>(row);
  float m = -INFINITY, s = 0.f, best = -INFINITY, bs = 0.f;
  int idx = 0x7fffffff;
  const float c2 = inv_tau * 1.4426950408889634f;
  auto consume = [&](const uint4 q, int c) {
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
        if (vals[t] > best) { best = vals[t]; idx = c * 8 + t; }  // ids increase per thread
    } else {
      float cm = vals[0];
#pragma unroll
      for (int t = 1; t < 8; ++t) cm = fmaxf(cm, vals[t]);
      cm *= c2;  // log2 units
      if (cm > m) { s *= ex2_fast(m - cm); m = cm; }
#pragma unroll
      for (int t = 0; t < 8; ++t) s += ex2_fast(vals[t] * c2 - m);
    }
  };
  // four independent 16-byte loads in flight per thread
  const int c_end = v_end / 8, step = blockDim.x;
  int c = v_beg / 8 + threadIdx.x;
  for (; c + 3 * step < c_end; c += 4 * step) {
    const uint4 q0 = __ldg(row4 + c), q1 = __ldg(row4 + c + step);
    const uint4 q2 = __ldg(row4 + c + 2 * step), q3 = __ldg(row4 + c + 3 * step);
    consume(q0, c);
    consume(q1, c + step);
    consume(q2, c + 2 * step);
    consume(q3, c + 3 * step);
  }
  for (; c < c_end; c += step) consume(__ldg(row4 + c), c);
  constexpr float LN2 = 0.6931471805599453f;
  m = m > -INFINITY ? m * LN2 : m;  // back to natural units
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
      SegStat st;
      st.m = m; st.s = s; st.best = best; st.idx = idx;
      stat[((size_t)i * (gamma + 1) + j) * NSEG + seg] = st;
    }
  }
}

// Pass 2: walk each request's admitted prefix; one thread per request.
template <int MODE>
__global__ void verify_decide(const SegStat *__restrict__ stat, const bf16 *__restrict__ target,
                              const int32_t *__restrict__ anchor,
                              const int32_t *__restrict__ tokens, const int32_t *__restrict__ len,
                              const float *__restrict__ lse_d, const float *__restrict__ logp_d,
                              ResampleRow *__restrict__ rows, int *__restrict__ list,
                              int *__restrict__ count, int32_t *__restrict__ accepted,
                              int32_t *__restrict__ bonus, int R, int gamma, int V, float inv_tau,
                              uint64_t seed) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= R) return;
  const int L = clamp_len(len, i, gamma);
  const SegStat *st = stat + (size_t)i * (gamma + 1) * NSEG;
  const int32_t *x = tokens + (size_t)i * gamma;
  int n = L;
  if (MODE == MODE_GREEDY) {
    auto row_argmax = [&](int j) {  // 0-based row
      float b = -INFINITY;
      int id = 0x7fffffff;
      for (int g = 0; g < NSEG; ++g)
        if (better(st[j * NSEG + g].best, st[j * NSEG + g].idx, b, id)) {
          b = st[j * NSEG + g].best;
          id = st[j * NSEG + g].idx;
        }
      return id;
    };
    for (int j = 1; j <= L; ++j)
      if (x[j - 1] != row_argmax(j - 1)) { n = j - 1; break; }
    accepted[i] = n;
    bonus[i] = row_argmax(n);
    return;
  }
  ResampleRow rr;
  rr.kind = KIND_BONUS;
  rr.pos = L + 1;
  rr.prev = 0;
  rr.lse_t = 0.f;
  rr.lse_d = 0.f;
  rr.pad[0] = rr.pad[1] = rr.pad[2] = 0;
  for (int j = 1; j <= L; ++j) {
    float m = -INFINITY, s = 0.f;
    for (int g = 0; g < NSEG; ++g) lse_merge(m, s, st[(j - 1) * NSEG + g].m, st[(j - 1) * NSEG + g].s);
    const float lse_t = m + logf(s);
    int xj = x[j - 1];
    if (xj < 0 || xj >= V) { dspark_set_status(DSPARK_ERR_TOKEN); xj = 0; }
    const float tx = __bfloat162float(target[((size_t)i * (gamma + 1) + j - 1) * V + xj]) * inv_tau;
    const uint4 w = rng_words4(seed, 0u, (uint32_t)j, (uint32_t)i, RNG_ACCEPT);
    const float u = rng_uniform(w.x);
    const size_t o = (size_t)i * gamma + j - 1;
    if (logf(u) + logp_d[o] < tx - lse_t) continue;  // u * p_d(x_j) < p_t(x_j): accepted
    n = j - 1;
    rr.kind = KIND_RESIDUAL;
    rr.pos = j;
    int prev = (j == 1) ? anchor[i] : x[j - 2];
    if (prev < 0 || prev >= V) { dspark_set_status(DSPARK_ERR_TOKEN); prev = 0; }
    rr.prev = prev;
    rr.lse_t = lse_t;
    rr.lse_d = lse_d[o];
    list[atomicAdd(count, 1)] = i;  // compacted residual rows (order irrelevant)
    break;
  }
  accepted[i] = n;
  rows[i] = rr;
}

// E[slot] = W1[x_{j*-1}] of the slot's request; fresh shared floor per slot.
__global__ void resample_gather(const ResampleRow *__restrict__ rows, const int *__restrict__ list,
                                const int *__restrict__ count, const bf16 *__restrict__ W1,
                                bf16 *__restrict__ E, float *__restrict__ gfloor, int r) {
  const int slot = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (slot >= *count) return;
  if (lane == 0) gfloor[slot] = -INFINITY;
  const ResampleRow rr = rows[list[slot]];
  uint4 *dst = reinterpret_cast<uint4 *>(E + (size_t)slot * r);
  const uint4 *src = reinterpret_cast<const uint4 *>(W1 + (size_t)rr.prev * r);
  for (int c = lane; c < r / 8; c += 32) dst[c] = src[c];
}

// Residual rows: combine the slice partials into the corrected token; a row
// whose residual came out empty is handed to the plain target sample.  One CTA
// of 256 threads per compacted row, eight partial loads in flight per thread.
__global__ void __launch_bounds__(256) resample_reduce(ResampleRow *__restrict__ rows,
                                                       const int *__restrict__ list,
                                                       const int *__restrict__ count,
                                                       const RowPartial *__restrict__ part,
                                                       int n_parts, int32_t *__restrict__ bonus) {
  const int slot = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (slot >= *count) return;
  float best = -INFINITY, d0 = 0.f, d1 = 0.f, d2 = 0.f;
  int idx = 0x7fffffff;
  const RowPartial *pr = part + (size_t)slot * n_parts;
  for (int t0 = 0; t0 < n_parts; t0 += 8 * 256) {
    float b[8];
    int id[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = t0 + u * 256 + tid;
      b[u] = -INFINITY;
      id[u] = 0x7fffffff;
      if (t < n_parts) {
        const RowPartial p = pr[t];
        b[u] = p.best;
        id[u] = p.idx;
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (better(b[u], id[u], best, idx)) { best = b[u]; idx = id[u]; }
  }
  warp_merge(d0, d1, best, idx, d2);
  __shared__ float sb[8];
  __shared__ int si[8];
  if (lane == 0) { sb[warp] = best; si[warp] = idx; }
  __syncthreads();
  if (warp == 0) {
    best = lane < 8 ? sb[lane] : -INFINITY;
    idx = lane < 8 ? si[lane] : 0x7fffffff;
    warp_merge(d0, d1, best, idx, d2);
    if (lane == 0) {
      const int req = list[slot];
      if (best > -INFINITY) bonus[req] = idx;
      else rows[req].kind = KIND_FALLBACK;
    }
  }
}

// Plain target samples: the bonus row l_r + 1 when every draft passed (stream
// 3), or the rejected row when its residual was empty (stream 2).  Gumbel-max
// over t / tau; one CTA of 512 threads per request.  Entries that cannot beat
// the best score the warp has seen skip their logarithms
// (1 - u >= e^{s - F + 0.01} implies s + g < F).
__global__ void __launch_bounds__(512) bonus_row(const ResampleRow *__restrict__ rows,
                                                 const bf16 *__restrict__ target,
                                                 int32_t *__restrict__ bonus, int gamma, int V,
                                                 float inv_tau, uint64_t seed) {
  const int i = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const ResampleRow rr = rows[i];
  if (rr.kind != KIND_BONUS && rr.kind != KIND_FALLBACK) return;
  const uint32_t stream = rr.kind == KIND_BONUS ? RNG_BONUS : RNG_RESIDUAL;
  const bf16 *trow = target + ((size_t)i * (gamma + 1) + rr.pos - 1) * V;
  const PhiloxKeys keys(seed);
  float best = -INFINITY, bs = 0.f, m = -INFINITY, s = 0.f;
  int idx = 0x7fffffff;
  // warp-uniform trip count: every lane reaches every shuffle; lanes past V are
  // masked.  Each lane takes 8 entries (16 bytes, two Philox calls) per step
  // and the next step's 16 bytes are in flight while the current ones are used.
  constexpr int STEP = 16 * 256;  // 16 warps x 32 lanes x 8 entries
  int base = warp * 256;
  uint4 nq = make_uint4(0, 0, 0, 0);
  if (base + lane * 8 < V) nq = __ldg(reinterpret_cast<const uint4 *>(trow + base + lane * 8));
  for (; base < V; base += STEP) {
    const int v0 = base + lane * 8;
    const bool valid = v0 < V;  // V % 8 == 0: a valid group has all 8 entries
    const uint4 q = nq;
    if (base + STEP + lane * 8 < V)
      nq = __ldg(reinterpret_cast<const uint4 *>(trow + base + STEP + lane * 8));
    float tv[8];
    uint32_t ws[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    {
      const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        tv[2 * t] = valid ? bf16_lo(qw[t]) * inv_tau : -INFINITY;
        tv[2 * t + 1] = valid ? bf16_hi(qw[t]) * inv_tau : -INFINITY;
      }
    }
    if (valid) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 w = keys(make_uint4((uint32_t)((v0 >> 2) + h), (uint32_t)rr.pos, (uint32_t)i,
                                        stream));
        ws[4 * h] = w.x; ws[4 * h + 1] = w.y; ws[4 * h + 2] = w.z; ws[4 * h + 3] = w.w;
      }
    }
    const float F = warp_max(best);
    if (valid) {
      // group test first: with tmax the largest of the 8 scaled logits, every
      // entry needs g > F - tmax; as an integer bound on the words (see the
      // draft epilogue), then per entry
      float tmax = fmaxf(fmaxf(fmaxf(tv[0], tv[1]), fmaxf(tv[2], tv[3])),
                         fmaxf(fmaxf(tv[4], tv[5]), fmaxf(tv[6], tv[7])));
      int w_thr = -1;
      if (F > -INFINITY) {
        const float X = __expf(fminf(tmax - F + 0.01f, 0.f)) * 8388608.f;
        w_thr = X >= 8388607.f ? -1 : 8388607 - (int)ceilf(X);
      }
      uint32_t wmax = 0;
#pragma unroll
      for (int t = 0; t < 8; ++t) wmax = max(wmax, ws[t]);
      if ((int)(wmax >> 9) > w_thr) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const bool cand = !(F > -INFINITY) ||
                            (1.f - rng_uniform(ws[t])) < __expf(tv[t] - F + 0.01f);
          if (cand) {
            const float sc = tv[t] + rng_gumbel(ws[t]);
            if (better(sc, v0 + t, best, idx)) { best = sc; idx = v0 + t; }
          }
        }
      }
    }
  }
  warp_merge(m, s, best, idx, bs);
  __shared__ float sb[16];
  __shared__ int si[16];
  if (lane == 0) { sb[warp] = best; si[warp] = idx; }
  __syncthreads();
  if (warp == 0) {
    best = lane < 16 ? sb[lane] : -INFINITY;
    idx = lane < 16 ? si[lane] : 0x7fffffff;
    warp_merge(m, s, best, idx, bs);
    if (lane == 0) bonus[i] = idx;
  }
}

struct VerifyWs {
  SegStat *stat;
  ResampleRow *rows;
  int *list;
  int *count;
  float *gfloor;
  bf16 *E;
  RowPartial *part;
  size_t bytes;
};

VerifyWs verify_layout(const dspark_dims *d, char *base) {
  VerifyWs w;
  size_t off = 0;
  w.stat = (SegStat *)(base + off);
  off = dspark_align_up(off + sizeof(SegStat) * (size_t)d->R * (d->gamma + 1) * NSEG, 256);
  w.rows = (ResampleRow *)(base + off);
  off = dspark_align_up(off + sizeof(ResampleRow) * (size_t)d->R, 256);
  w.list = (int *)(base + off);
  off = dspark_align_up(off + sizeof(int) * (size_t)d->R, 256);
  w.count = (int *)(base + off);
  off = dspark_align_up(off + sizeof(int), 256);
  w.gfloor = (float *)(base + off);
  off = dspark_align_up(off + sizeof(float) * (size_t)d->R, 256);
  w.E = (bf16 *)(base + off);
  off = dspark_align_up(off + sizeof(bf16) * (size_t)d->R * d->r, 256);
  w.part = (RowPartial *)(base + off);
  off = dspark_align_up(off + sizeof(RowPartial) * (size_t)d->R * logits_parts_max(d->V), 256);
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
  if (((uintptr_t)target | (sample ? ((uintptr_t)W2t | (uintptr_t)W1 | (uintptr_t)base_logits)
                                   : (uintptr_t)0)) & 15)
    return DSPARK_ERR_ARG;  // TMA and 16-byte vector loads
  VerifyWs ws = verify_layout(dims, (char *)workspace);
  if (!workspace || workspace_bytes < ws.bytes || ((uintptr_t)workspace & 255))
    return DSPARK_ERR_WORKSPACE;
  const int R = dims->R, G = dims->gamma, V = dims->V, r = dims->r;
  const float inv_tau = sample ? 1.f / tau : 1.f;
  const dim3 rgrid(NSEG * (G + 1), R);
  const bf16 *tgt = (const bf16 *)target;
  if (!sample) {
    verify_rows<MODE_GREEDY><<<rgrid, 256, 0, stream>>>(tgt, len, ws.stat, ws.count, G, V, inv_tau);
    DSPARK_CHECK_LAUNCH();
    verify_decide<MODE_GREEDY><<<(R + 127) / 128, 128, 0, stream>>>(
        ws.stat, tgt, anchor, tokens, len, lse_d, logp_d, ws.rows, ws.list, ws.count, accepted,
        bonus, R, G, V, inv_tau, seed);
    DSPARK_CHECK_LAUNCH();
    dspark_count_launches(2);
    return DSPARK_OK;
  }
  verify_rows<MODE_SAMPLE><<<rgrid, 256, 0, stream>>>(tgt, len, ws.stat, ws.count, G, V, inv_tau);
  DSPARK_CHECK_LAUNCH();
  verify_decide<MODE_SAMPLE><<<(R + 127) / 128, 128, 0, stream>>>(
      ws.stat, tgt, anchor, tokens, len, lse_d, logp_d, ws.rows, ws.list, ws.count, accepted,
      bonus, R, G, V, inv_tau, seed);
  DSPARK_CHECK_LAUNCH();
  resample_gather<<<(R * 32 + 255) / 256, 256, 0, stream>>>(ws.rows, ws.list, ws.count,
                                                          (const bf16 *)W1, ws.E, ws.gfloor, r);
  DSPARK_CHECK_LAUNCH();
  const int n_parts = logits_parts<MODE_RESIDUAL>(V);
  EpiLogits<MODE_RESIDUAL> epi{(const bf16 *)base_logits, tgt, ws.rows, ws.list, ws.count, ws.part,
                               ws.gfloor, R, V, G, 0, n_parts, inv_tau, seed};
  const int rc = gemm::launch<LogitsCfg<MODE_RESIDUAL>::EPI_WARPS, LogitsCfg<MODE_RESIDUAL>::BN>(ws.E, W2t, R, V, r, epi, stream,
                                                                  ws.count);
  if (rc != DSPARK_OK) return rc;
  resample_reduce<<<R, 256, 0, stream>>>(ws.rows, ws.list, ws.count, ws.part, n_parts, bonus);
  DSPARK_CHECK_LAUNCH();
  bonus_row<<<R, 512, 0, stream>>>(ws.rows, tgt, bonus, G, V, inv_tau, seed);
  DSPARK_CHECK_LAUNCH();
  dspark_count_launches(5);  // + the GEMM, counted by launch()
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
