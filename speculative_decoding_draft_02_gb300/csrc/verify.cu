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
// Pass 1 (verify_rows) scans each target row 1..l_r+1 once: greedy, its
// argmax; sampling, the log-sum-exp of rows 1..l_r (the acceptance test's
// normalisers) and, for row l_r + 1, the first level of the bonus draw (each
// 64-id block's log-mass plus its Gumbel).  The last CTA of each request to
// finish its row then decides the request: the acceptance ballot, and the
// bonus drawn inside the winning block, or (sampling) the request joins the
// rejected rows.  Pass 2 (residual_trials) draws each rejected row's residual
// norm(max(0, p_t - p_d)) by rejection from p_t, which needs p_d at the
// proposed ids only (one W2t row each).  A row none of whose trials keeps its
// proposal (rare unless p_t and p_d nearly agree) takes the explicit route:
// pass 3 rebuilds p_d on the row through the same fused vocabulary pass as the
// draft (bias + base logits, on chip), and pass 4 draws the residual.
#include "logits_tile.cuh"

DSPARK_DECLARE_STATUS(s_status_verify)

namespace {

constexpr int NSEG = 4;  // CTAs per target row in the first pass

// Per (request, row, segment): online log-sum-exp of t / tau (sampling rows
// 1..l_r), the argmax (greedy), or the best block score and its block
// (sampling, the bonus row l_r + 1) over one quarter of the vocabulary.
struct __align__(16) SegStat {
  float m, s;      // sampling: log-sum-exp
  float best;      // greedy: max logit; sampling bonus row: best block score
  int32_t idx;     // its id or block
};

__device__ __forceinline__ int clamp_len(const int32_t *len, int i, int gamma) {
  int L = len[i];
  if (L < 0 || L > gamma) {
    dspark_set_status(DSPARK_ERR_LENGTH);
    L = L < 0 ? 0 : gamma;
  }
  return L;
}

// Segments hold whole groups of four sampler blocks (256 ids), so a block's
// log-mass, and one Philox call's four block words, are one CTA's.
__device__ __forceinline__ int seg_len(int V) {
  return ((V + NSEG - 1) / NSEG + 4 * GUMBEL_BLOCK - 1) / (4 * GUMBEL_BLOCK) * (4 * GUMBEL_BLOCK);
}

__device__ __forceinline__ void block_best_reduce(float &best, int &idx) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    if (better(b2, i2, best, idx)) { best = b2; idx = i2; }
  }
}

// The first level of a two-level draw from softmax(row / tau) over segment
// `seg`'s sampler blocks: G_b = log Z_b + Gumbel(block id b, stream + 4) at
// (pos, req); the best (G_b, b) goes to out->best, out->idx.  Pass 1 leaves
// log Z_b of every block of the segment in s_lz (dynamic shared memory): eight
// lanes take a block (one 16-byte word each), eight words in flight per lane.
// Pass 2 scores them, four blocks per thread from one Philox call (segments
// start on a multiple of four blocks).  Called by a whole CTA of 256.
// log Z_b of sampler blocks [b_lo, b_hi) of a row of logits / tau into
// out[b - b_lo] (-inf for a block with no finite weight): eight lanes take a
// block (one 16-byte word each), eight words in flight per lane.  Called by a
// whole CTA of NT threads; ends with a CTA barrier, after which out is complete.
template <int NT>
__device__ void block_lz(const bf16 *__restrict__ row, int V, int b_lo, int b_hi, float inv_tau,
                         float *out) {
  constexpr float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;
  constexpr int GROUPS = NT / 8, U = 8;
  const int tid = threadIdx.x;
  const int grp = tid >> 3, sub = tid & 7;
  const float c2 = inv_tau * LOG2E;
  // the trip count depends on the block range only: every lane reaches every shuffle
  for (int b0 = b_lo; b0 < b_hi; b0 += GROUPS * U) {
    uint4 w4[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int b = b0 + u * GROUPS + grp, v = b * GUMBEL_BLOCK + sub * 8;
      w4[u] = (b < b_hi && v < V) ? __ldg(reinterpret_cast<const uint4 *>(row + v))
                                  : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int b = b0 + u * GROUPS + grp, v = b * GUMBEL_BLOCK + sub * 8;
      const bool ok = b < b_hi && v < V;  // V % 8 == 0: a word is all inside or all past V
      const uint32_t w[4] = {w4[u].x, w4[u].y, w4[u].z, w4[u].w};
      float x[8];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        x[2 * t] = bf16_lo(w[t]);
        x[2 * t + 1] = bf16_hi(w[t]);
      }
      // the maximum of the raw values, scaled once (c2 > 0 keeps the order)
      float mx = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                       fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
      mx = ok ? mx : -INFINITY;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float ms = mx * c2;  // log2 units
      float sm = 0.f;
      if (ok && mx > -INFINITY) {
#pragma unroll
        for (int t = 0; t < 8; ++t) sm += ex2_fast(fmaf(x[t], c2, -ms));
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
      if (sub == 0 && b < b_hi)
        out[b - b_lo] = mx > -INFINITY ? (ms + __log2f(sm)) * LN2 : -INFINITY;
    }
  }
  __syncthreads();
}

__device__ void seg_block_scores(const bf16 *__restrict__ row, int V, int seg, float inv_tau,
                                 uint64_t seed, int pos, int req, uint32_t stream,
                                 SegStat *out) {
  extern __shared__ float s_lz[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sl = seg_len(V), nb = (V + GUMBEL_BLOCK - 1) / GUMBEL_BLOCK;
  const int b_lo = seg * sl / GUMBEL_BLOCK;
  const int b_hi = min(nb, b_lo + sl / GUMBEL_BLOCK);
  // pass 1: the blocks' log-masses
  block_lz<256>(row, V, b_lo, b_hi, inv_tau, s_lz);
  // pass 2: G_b = log Z_b + Gumbel(block id b, block stream), b_lo % 4 == 0
  float best = -INFINITY;
  int idx = 0x7fffffff;
  for (int q4 = b_lo / 4 + tid; q4 * 4 < b_hi; q4 += 256) {
    const uint4 g4 = rng_words4(seed, (uint32_t)q4, (uint32_t)pos, (uint32_t)req,
                                stream + RNG_BLOCK_OFFSET);
    const uint32_t ws[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int b = 4 * q4 + t;
      if (b < b_hi && s_lz[b - b_lo] > -INFINITY) {
        const float G = s_lz[b - b_lo] + rng_gumbel(ws[t]);
        if (better(G, b, best, idx)) { best = G; idx = b; }
      }
    }
  }
  block_best_reduce(best, idx);
  __shared__ float sb[8];
  __shared__ int si[8];
  if (lane == 0) { sb[warp] = best; si[warp] = idx; }
  __syncthreads();
  if (warp == 0) {
    best = lane < 8 ? sb[lane] : -INFINITY;
    idx = lane < 8 ? si[lane] : 0x7fffffff;
    block_best_reduce(best, idx);
    if (lane == 0) {
      SegStat st;
      st.m = -INFINITY; st.s = 0.f; st.best = best; st.idx = idx;
      *out = st;
    }
  }
  __syncthreads();  // s_lz, sb, si are free for the next call
}

// Dynamic shared memory of seg_block_scores: log Z_b of one segment's blocks.
static inline size_t seg_lz_bytes(int V) {
  const int sl = ((V + NSEG - 1) / NSEG + 4 * GUMBEL_BLOCK - 1) / (4 * GUMBEL_BLOCK) *
                 (4 * GUMBEL_BLOCK);
  return sizeof(float) * (size_t)(sl / GUMBEL_BLOCK);
}
constexpr size_t SEG_LZ_MAX = 200 * 1024;  // V up to about 13 million

__device__ __forceinline__ void bonus_blocks(const bf16 *__restrict__ row, int V, int seg,
                                             float inv_tau, uint64_t seed, int pos, int req,
                                             SegStat *out) {
  seg_block_scores(row, V, seg, inv_tau, seed, pos, req, RNG_BONUS, out);
}

// Arguments of the first pass (and of the decision its last CTA per request takes).
struct VerifyArgs {
  const bf16 *target;           // [R, gamma + 1, V]
  const int32_t *len;           // [R]
  const int32_t *anchor;        // [R]
  const int32_t *tokens;        // [R, gamma]
  const float *lse_d, *logp_d;  // [R, gamma]
  const bf16 *base;             // [R * gamma, V]
  const bf16 *W1, *W2t;         // [V, r]
  SegStat *stat;                // [R, gamma + 1, NSEG]
  int *done;                    // [R]  arrivals of a request's row CTAs (zeroed per call)
  int *count;                   // rejected requests
  int *list;                    // [R]  those requests, compacted
  ResampleRow *rows;            // [R]
  int32_t *accepted, *bonus;    // [R]
  int R, gamma, V, r;
  float inv_tau;
  uint64_t seed;
};

// The decision of request i from its rows' statistics, by the last CTA of the
// request to finish its row: warp 0 tests admitted position j on lane j - 1
// and a ballot finds the first failure.  Greedy: the argmaxes decide.
// Sampling: every draft passed, the bonus is drawn inside the bonus row's
// winning block; else the request joins the rejected rows of the trial pass.
template <int MODE>
__device__ void decide_request(const VerifyArgs &a, int i, int L) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gamma = a.gamma, V = a.V;
  const SegStat *st = a.stat + (size_t)i * (gamma + 1) * NSEG;
  const int32_t *x = a.tokens + (size_t)i * gamma;
  const int j = lane + 1;  // this lane's 1-based position (gamma <= 32)
  auto load = [&](int k) {  // another CTA's statistics: from L2
    SegStat v;
    const float4 f = __ldcg(reinterpret_cast<const float4 *>(st + k));
    v.m = f.x; v.s = f.y; v.best = f.z; v.idx = __float_as_int(f.w);
    return v;
  };
  if (MODE == MODE_GREEDY) {
    if (warp != 0) return;
    auto row_argmax = [&](int jr) {  // 0-based row
      float b = -INFINITY;
      int id = 0x7fffffff;
      for (int g = 0; g < NSEG; ++g) {
        const SegStat v = load(jr * NSEG + g);
        if (better(v.best, v.idx, b, id)) { b = v.best; id = v.idx; }
      }
      return id;
    };
    const bool fail = j <= L && x[j - 1] != row_argmax(j - 1);
    const unsigned bal = __ballot_sync(0xffffffffu, fail);
    const int n = bal ? __ffs(bal) - 1 : L;  // first failing position - 1
    const int tok = row_argmax(n);
    if (lane == 0) {
      a.accepted[i] = n;
      a.bonus[i] = tok;
    }
    return;
  }
  if (warp == 0) {
    // sampling: accept x_j iff u * p_d(x_j) < p_t(x_j), tested in logs
    bool fail = false;
    float lse_t = 0.f;
    if (j <= L) {
      float m = -INFINITY, s = 0.f;
      for (int g = 0; g < NSEG; ++g) {
        const SegStat v = load((j - 1) * NSEG + g);
        lse_merge(m, s, v.m, v.s);
      }
      lse_t = m + logf(s);
      int xj = x[j - 1];
      if (xj < 0 || xj >= V) { dspark_set_status(DSPARK_ERR_TOKEN); xj = 0; }
      const float tx =
          __bfloat162float(a.target[((size_t)i * (gamma + 1) + j - 1) * V + xj]) * a.inv_tau;
      const uint4 w = rng_words4(a.seed, 0u, (uint32_t)j, (uint32_t)i, RNG_ACCEPT);
      const float u = rng_uniform(w.x);
      fail = !(logf(u) + a.logp_d[(size_t)i * gamma + j - 1] < tx - lse_t);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, fail);
    const int jf = bal ? __ffs(bal) : 0;  // first rejected position (1-based), 0 if none
    const int src = jf ? jf - 1 : 0;
    if (lane == src) {
      ResampleRow rr;
      rr.pad[0] = rr.pad[1] = rr.pad[2] = 0;
      if (jf) {
        rr.kind = KIND_RESIDUAL;
        rr.pos = jf;
        int prev = (jf == 1) ? a.anchor[i] : x[jf - 2];
        if (prev < 0 || prev >= V) { dspark_set_status(DSPARK_ERR_TOKEN); prev = 0; }
        rr.prev = prev;
        rr.lse_t = lse_t;
        rr.lse_d = a.lse_d[(size_t)i * gamma + jf - 1];
        a.list[atomicAdd(a.count, 1)] = i;  // compacted rejected rows (order irrelevant)
      } else {
        rr.kind = KIND_BONUS;
        rr.pos = L + 1;
        rr.prev = 0;
        rr.lse_t = 0.f;
        rr.lse_d = 0.f;
      }
      a.accepted[i] = jf ? jf - 1 : L;
      a.rows[i] = rr;
    }
    if (!jf) {  // warp-uniform: every draft passed, the bonus comes from row l_r + 1
      // the winning block of the bonus row's block scores, then the ids inside
      // it: t / tau + Gumbel(id, bonus stream) at position l_r + 1
      float gb = -INFINITY;
      int b = 0x7fffffff;
      for (int g = 0; g < NSEG; ++g) {
        const SegStat v = load(L * NSEG + g);
        if (better(v.best, v.idx, gb, b)) { gb = v.best; b = v.idx; }
      }
      const int nb = (V + GUMBEL_BLOCK - 1) / GUMBEL_BLOCK;
      if (!(gb > -INFINITY) || b >= nb) {  // non-finite target row
        if (lane == 0) dspark_set_status(DSPARK_ERR_TOKEN);
        b = 0;
      }
      __shared__ float s_score[GUMBEL_BLOCK];
      const bf16 *trow = a.target + ((size_t)i * (gamma + 1) + L) * V;
      for (int e = lane; e < GUMBEL_BLOCK; e += 32) {
        const int v = b * GUMBEL_BLOCK + e;
        s_score[e] = v < V ? __bfloat162float(trow[v]) * a.inv_tau : -INFINITY;
      }
      __syncwarp();
      const int tok =
          block_pick(s_score, b, V, a.seed, (uint32_t)(L + 1), (uint32_t)i, RNG_BONUS);
      if (lane == 0) a.bonus[i] = tok >= 0 ? tok : b * GUMBEL_BLOCK;
    }
  }
}

// Pass 1: grid (NSEG * (gamma+1), R).  Greedy scans rows 1..l_r+1 (their
// argmaxes decide acceptance and give the correction or bonus token); sampling
// scans rows 1..l_r (their normalisers enter the acceptance test) and the
// bonus row l_r + 1 (block scores: the bonus draw's first level, on the bonus
// stream).  Each CTA then counts itself in for its request; the last of the
// request's NSEG (l_r + 1) CTAs takes the request's decision (decide_request),
// so the decision of one request overlaps the scans of the others and no CTA
// ever waits for another.
template <int MODE>
__global__ void __launch_bounds__(256) verify_rows(const __grid_constant__ VerifyArgs a) {
  const int j = blockIdx.x / NSEG, seg = blockIdx.x % NSEG, i = blockIdx.y;
  const int gamma = a.gamma, V = a.V;
  const float inv_tau = a.inv_tau;
  pdl_trigger();
  pdl_wait();  // len comes from the scheduler
  const int L = clamp_len(a.len, i, gamma);
  if (j > L) return;
  SegStat *out = a.stat + ((size_t)i * (gamma + 1) + j) * NSEG + seg;
  if (MODE == MODE_SAMPLE && j == L) {
    bonus_blocks(a.target + ((size_t)i * (gamma + 1) + j) * V, V, seg, inv_tau, a.seed, j + 1,
                 i, out);
  } else {
    const int sl = seg_len(V), v_beg = seg * sl, v_end = min(V, v_beg + sl);
    const bf16 *row = a.target + ((size_t)i * (gamma + 1) + j) * V;
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
    // eight independent 16-byte loads in flight per thread
    const int c_end = v_end / 8, step = blockDim.x;
    int c = v_beg / 8 + threadIdx.x;
    for (; c + 7 * step < c_end; c += 8 * step) {
      uint4 q[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) q[u] = __ldg(row4 + c + u * step);
#pragma unroll
      for (int u = 0; u < 8; ++u) consume(q[u], c + u * step);
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
        *out = st;
      }
    }
  }
  // thread 0 wrote this CTA's statistics: it makes them visible, then counts
  // the CTA in; the last of the request's CTAs decides
  __shared__ int s_last;
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(a.done + i, 1) == NSEG * (L + 1) - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();  // the other CTAs' statistics, read below through L2
  decide_request<MODE>(a, i, L);
}

// Pass 4, the rows no trial settled: the block scores of the slices pick a block of 64 ids; inside
// it the residual q = max(0, p_t - p_d) is rebuilt (target row, base logits and
// the Markov bias W1[x_{j*-1}] . W2t[v]) and the corrected token is drawn from
// log q + Gumbel.  A row whose residual came out empty is drawn from p_t
// instead.  One CTA of 256 threads per compacted row, eight partial loads in
// flight per thread.
__global__ void __launch_bounds__(256) resample_reduce(
    ResampleRow *__restrict__ rows, const int *__restrict__ list, const int *__restrict__ count,
    const RowPartial *__restrict__ part, int n_parts, const bf16 *__restrict__ base,
    const bf16 *__restrict__ target, const bf16 *__restrict__ E, const bf16 *__restrict__ W2t,
    int gamma, int V, int r, float inv_tau, uint64_t seed, int32_t *__restrict__ bonus) {
  const int slot = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();  // the residual pass's partials
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
  __shared__ float sb[8], s_logit[GUMBEL_BLOCK], s_score[GUMBEL_BLOCK];
  __shared__ int si[8], s_blk;
  if (lane == 0) { sb[warp] = best; si[warp] = idx; }
  __syncthreads();
  if (warp == 0) {
    best = lane < 8 ? sb[lane] : -INFINITY;
    idx = lane < 8 ? si[lane] : 0x7fffffff;
    warp_merge(d0, d1, best, idx, d2);
    if (lane == 0) s_blk = best > -INFINITY ? idx : -1;
  }
  __syncthreads();
  const int req = list[slot];
  const ResampleRow rr = rows[req];
  const bf16 *trow = target + ((size_t)req * (gamma + 1) + rr.pos - 1) * V;
  const int nb = (V + GUMBEL_BLOCK - 1) / GUMBEL_BLOCK;
  __shared__ int s_fb;
  const int b = s_blk;
  bool fallback = b < 0 || b >= nb;  // every block's residual empty (CTA-uniform)
  if (!fallback) {
    block_logits<256>(base + ((size_t)req * gamma + rr.pos - 1) * V, E + (size_t)slot * r, W2t,
                      b, V, r, s_logit);
    if (warp == 0) {
      for (int j = lane; j < GUMBEL_BLOCK; j += 32) {
        const int v = b * GUMBEL_BLOCK + j;
        float sc = -INFINITY;
        if (v < V) {
          const float pt = __expf(__bfloat162float(trow[v]) * inv_tau - rr.lse_t);
          const float pd = __expf(s_logit[j] * inv_tau - rr.lse_d);
          if (pt > pd) sc = __logf(pt - pd);
        }
        s_score[j] = sc;
      }
      __syncwarp();
      const int tok = block_pick(s_score, b, V, seed, (uint32_t)rr.pos, (uint32_t)req, RNG_RESIDUAL);
      if (lane == 0) {
        if (tok >= 0) bonus[req] = tok;
        s_fb = tok < 0;  // the block's mass was rounding only
      }
    }
    __syncthreads();
    fallback = s_fb;
  }
  if (fallback) {
    // the residual max(0, p_t - p_d) is empty in floating point (impossible in
    // exact arithmetic): the row is drawn from p_t itself, on the residual
    // stream, in the same two levels (block scores over the whole row, then
    // the ids of the winning block)
    __shared__ SegStat s_seg[NSEG];
    if (tid == 0) rows[req].kind = KIND_FALLBACK;
    for (int g = 0; g < NSEG; ++g)
      seg_block_scores(trow, V, g, inv_tau, seed, rr.pos, req, RNG_RESIDUAL, &s_seg[g]);
    if (warp == 0) {
      float gb = -INFINITY;
      int bb = 0x7fffffff;
      for (int g = 0; g < NSEG; ++g)
        if (better(s_seg[g].best, s_seg[g].idx, gb, bb)) { gb = s_seg[g].best; bb = s_seg[g].idx; }
      if (!(gb > -INFINITY) || bb >= nb) {  // non-finite target row
        if (lane == 0) dspark_set_status(DSPARK_ERR_TOKEN);
        bb = 0;
      }
      for (int j = lane; j < GUMBEL_BLOCK; j += 32) {
        const int v = bb * GUMBEL_BLOCK + j;
        s_score[j] = v < V ? __bfloat162float(trow[v]) * inv_tau : -INFINITY;
      }
      __syncwarp();
      const int tok = block_pick(s_score, bb, V, seed, (uint32_t)rr.pos, (uint32_t)req,
                                 RNG_RESIDUAL);
      if (lane == 0) bonus[req] = tok >= 0 ? tok : bb * GUMBEL_BLOCK;
    }
  }
}

// Rejection trials from p_t per rejected row before the explicit residual.
constexpr int RESIDUAL_TRIALS = 64;
constexpr int TRIAL_WARPS = 32;  // trials in flight per row (one per warp)
constexpr int TRIAL_THREADS = 32 * TRIAL_WARPS;
constexpr int TRIAL_SUPER = 16;  // sampler blocks per first-level block of a proposal

// Pass 2, one CTA per rejected row (compacted by the decisions of pass 1): the
// residual norm(max(0, p_t - p_d)) by rejection from p_t.  The row's
// log-masses over sampler blocks and over super-blocks of TRIAL_SUPER of them
// go to lz once; then rounds of TRIAL_WARPS trials, one per warp: trial q
// draws y_q ~ p_t in three levels (super-block by log Z_S + Gumbel(S) on
// stream RNG_TRIAL0 + 8q + RNG_SUPER_OFFSET, sampler block inside it by
// log Z_b + Gumbel(b) on RNG_TRIAL0 + 8q + RNG_BLOCK_OFFSET, id inside that by
// t_v / tau + Gumbel(v) on RNG_TRIAL0 + 8q) and keeps it iff
// u_q < 1 - p_d(y_q) / p_t(y_q), u_q on RNG_TRIAL0 + 8q + 1, where p_d(y)
// needs only the base logit, W1[x_{j*-1}] . W2t[y] and lse_d.  The first kept
// trial in q order is the corrected token.  A row that keeps none of its
// RESIDUAL_TRIALS goes to the explicit residual pass: compacted into list_fb,
// with E_fb = W1[x_{j*-1}] as its A operand.
__global__ void __launch_bounds__(TRIAL_THREADS) residual_trials(
    ResampleRow *__restrict__ rows, const int *__restrict__ list, const int *__restrict__ count,
    const bf16 *__restrict__ base, const bf16 *__restrict__ target, const bf16 *__restrict__ W1,
    const bf16 *__restrict__ W2t, float *__restrict__ lz, int gamma, int V, int r,
    float inv_tau, uint64_t seed, int32_t *__restrict__ bonus, int *__restrict__ list_fb,
    int *__restrict__ count_fb, bf16 *__restrict__ E_fb) {
  const int slot = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();  // the compacted rows of pass 1
  if (slot >= *count) return;
  const int req = list[slot];
  const ResampleRow rr = rows[req];
  const int nb = (V + GUMBEL_BLOCK - 1) / GUMBEL_BLOCK;
  const int ns = (nb + TRIAL_SUPER - 1) / TRIAL_SUPER;
  const uint32_t pos = (uint32_t)rr.pos;
  const bf16 *trow = target + ((size_t)req * (gamma + 1) + rr.pos - 1) * V;
  const bf16 *brow = base + ((size_t)req * gamma + rr.pos - 1) * V;
  const uint4 *e4 = reinterpret_cast<const uint4 *>(W1 + (size_t)rr.prev * r);
  // the log-masses of the sampler blocks, then of super-blocks of TRIAL_SUPER of them
  float *lz64 = lz + (size_t)slot * (nb + ns), *lzs = lz64 + nb;
  block_lz<TRIAL_THREADS>(trow, V, 0, nb, inv_tau, lz64);  // ends with a CTA barrier
  for (int c = tid; c < ns; c += TRIAL_THREADS) {
    const int t1 = min(nb, TRIAL_SUPER * c + TRIAL_SUPER);
    float m = -INFINITY;
    for (int t = TRIAL_SUPER * c; t < t1; ++t) m = fmaxf(m, lz64[t]);
    float sm = 0.f;
    if (m > -INFINITY)
      for (int t = TRIAL_SUPER * c; t < t1; ++t) sm += expf(lz64[t] - m);
    lzs[c] = m > -INFINITY ? m + logf(sm) : -INFINITY;
  }
  __syncthreads();
  __shared__ int s_kept[TRIAL_WARPS];
  int tok = -1;
  for (int q0 = 0; q0 < RESIDUAL_TRIALS; q0 += TRIAL_WARPS) {  // CTA-uniform trip count
    const uint32_t st = RNG_TRIAL0 + 8u * (uint32_t)(q0 + warp);
    // y ~ p_t in three levels; first, the super-block
    float best = -INFINITY;
    int sb = 0x7fffffff;
    for (int q4 = lane; 4 * q4 < ns; q4 += 32) {
      const uint4 g4 = rng_words4(seed, (uint32_t)q4, pos, (uint32_t)req, st + RNG_SUPER_OFFSET);
      const uint32_t ws[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int S = 4 * q4 + t;
        const float l = S < ns ? lzs[S] : -INFINITY;
        if (l > -INFINITY) {
          const float G = l + rng_gumbel(ws[t]);
          if (better(G, S, best, sb)) { best = G; sb = S; }
        }
      }
    }
    block_best_reduce(best, sb);
    int y = -1;
    if (best > -INFINITY) {  // warp-uniform
      // the sampler block inside super-block sb: one per lane
      const int b = sb * TRIAL_SUPER + lane;
      const float l = (lane < TRIAL_SUPER && b < nb) ? lz64[b] : -INFINITY;
      float e2 = -INFINITY;
      int b2 = 0x7fffffff;
      if (l > -INFINITY) {
        const uint4 g4 = rng_words4(seed, (uint32_t)(b >> 2), pos, (uint32_t)req,
                                    st + RNG_BLOCK_OFFSET);
        e2 = l + rng_gumbel(uint4_get(g4, b & 3));
        b2 = b;
      }
      block_best_reduce(e2, b2);
      if (e2 > -INFINITY) {  // warp-uniform: the ids of block b2, two per lane
        const int v = b2 * GUMBEL_BLOCK + 2 * lane;
        float e3 = -INFINITY;
        int id = 0x7fffffff;
        if (v < V) {  // V is even: both ids inside
          const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(trow + v));
          const uint4 g4 = rng_words4(seed, (uint32_t)(v >> 2), pos, (uint32_t)req, st);
          const float s0 = bf16_lo(w) * inv_tau, s1 = bf16_hi(w) * inv_tau;
          if (s0 > -INFINITY) { e3 = s0 + rng_gumbel(uint4_get(g4, v & 3)); id = v; }
          if (s1 > -INFINITY) {
            const float ev = s1 + rng_gumbel(uint4_get(g4, (v & 3) + 1));
            if (better(ev, v + 1, e3, id)) { e3 = ev; id = v + 1; }
          }
        }
        block_best_reduce(e3, id);
        y = e3 > -INFINITY ? id : -1;
      }
    }
    int kept = -1;
    if (y >= 0) {  // warp-uniform: the acceptance test, p_d(y) / p_t(y) in logs
      const uint4 *w4 = reinterpret_cast<const uint4 *>(W2t + (size_t)y * r);
      float dot = 0.f;
      for (int c = lane; c < r / 8; c += 32) dot = dot8_bf16(__ldg(e4 + c), __ldg(w4 + c), dot);
      dot = warp_sum(dot);
      const float ld = (__bfloat162float(brow[y]) + dot) * inv_tau - rr.lse_d;
      const float lt = __bfloat162float(trow[y]) * inv_tau - rr.lse_t;
      const float u = rng_uniform(rng_words4(seed, 0u, pos, (uint32_t)req, st + 1).x);
      if (1.f - expf(ld - lt) - u > 0.f) kept = y;
    }
    if (lane == 0) s_kept[warp] = kept;
    __syncthreads();
    int t = -1;
#pragma unroll
    for (int w = 0; w < TRIAL_WARPS; ++w)
      if (t < 0) t = s_kept[w];  // the first kept trial in q order
    __syncthreads();  // s_kept is rewritten by the next round
    if (t >= 0) {
      tok = t;
      break;
    }
  }
  if (tok >= 0) {
    if (tid == 0) {
      bonus[req] = tok;
      rows[req].kind = KIND_TRIAL;
    }
    return;
  }
  // no trial kept its proposal: the explicit residual pass takes the row
  __shared__ int s_fs;
  if (tid == 0) {
    s_fs = atomicAdd(count_fb, 1);
    list_fb[s_fs] = req;
  }
  __syncthreads();
  uint4 *to = reinterpret_cast<uint4 *>(E_fb + (size_t)s_fs * r);
  for (int c = tid; c < r / 8; c += TRIAL_THREADS) to[c] = __ldg(e4 + c);
}

struct VerifyWs {
  SegStat *stat;
  ResampleRow *rows;
  int *done;      // [R] arrivals per request, then count and count_fb: zeroed per call
  int *count;     // rejected requests
  int *count_fb;  // of them, the rows left to the explicit residual pass
  int *list;      // [R] the rejected requests
  int *list_fb;   // [R] the explicit pass's rows
  float *lz;      // [R, V / 64 + V / 1024] log-masses of the rejected rows' target rows
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
  w.done = (int *)(base + off);
  w.count = w.done + d->R;
  w.count_fb = w.done + d->R + 1;
  off = dspark_align_up(off + sizeof(int) * ((size_t)d->R + 2), 256);
  w.list = (int *)(base + off);
  off = dspark_align_up(off + sizeof(int) * (size_t)d->R, 256);
  w.list_fb = (int *)(base + off);
  off = dspark_align_up(off + sizeof(int) * (size_t)d->R, 256);
  w.lz = (float *)(base + off);
  const size_t nb = (size_t)(d->V + GUMBEL_BLOCK - 1) / GUMBEL_BLOCK;
  off = dspark_align_up(
      off + sizeof(float) * (size_t)d->R * (nb + (nb + TRIAL_SUPER - 1) / TRIAL_SUPER), 256);
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
  // the arrival counters and the residual-row counts start at zero
  if (cudaMemsetAsync(ws.done, 0, sizeof(int) * ((size_t)R + 2), stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  VerifyArgs va{tgt, len, anchor, tokens, lse_d, logp_d, (const bf16 *)base_logits,
                (const bf16 *)W1, (const bf16 *)W2t, ws.stat, ws.done, ws.count, ws.list, ws.rows,
                accepted, bonus, R, G, V, r, inv_tau, seed};
  if (!sample) {
    if (dspark_launch_pdl(verify_rows<MODE_GREEDY>, rgrid, dim3(256), 0, stream, va) !=
        cudaSuccess)
      return DSPARK_ERR_CUDA;
    dspark_count_launches(1);
    return DSPARK_OK;
  }
  // the block scores keep one segment's log-masses in shared memory
  const size_t lz = seg_lz_bytes(V);
  if (lz > SEG_LZ_MAX) return DSPARK_ERR_TOO_LARGE;
  static DsparkPerDevice smem_attr;
  if (dspark_per_device(smem_attr, [] {
        return cudaFuncSetAttribute(verify_rows<MODE_SAMPLE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)SEG_LZ_MAX) == cudaSuccess &&
                       cudaFuncSetAttribute(resample_reduce,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)SEG_LZ_MAX) == cudaSuccess
                   ? 1
                   : -1;
      }) < 0)
    return DSPARK_ERR_CUDA;
  // each kernel's launch and set-up overlap the tail of the one before
  // (programmatic serialisation; every kernel waits before touching memory)
  if (dspark_launch_pdl(verify_rows<MODE_SAMPLE>, rgrid, dim3(256), lz, stream, va) !=
          cudaSuccess ||
      dspark_launch_pdl(residual_trials, dim3(R), dim3(TRIAL_THREADS), 0, stream, ws.rows,
                        (const int *)ws.list, (const int *)ws.count, (const bf16 *)base_logits,
                        tgt, (const bf16 *)W1, (const bf16 *)W2t, ws.lz, G, V, r, inv_tau, seed,
                        bonus, ws.list_fb, ws.count_fb, ws.E) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  // the explicit residual, for the rows no trial settled (usually none: the
  // GEMM then finds no rows and the reduction no slot)
  const int n_parts = logits_parts<MODE_RESIDUAL>(V);
  EpiLogits<MODE_RESIDUAL> epi{(const bf16 *)base_logits, tgt, ws.rows, ws.list_fb, ws.count_fb,
                               ws.part, R, V, G, 0, n_parts, inv_tau, seed};
  const int rc = gemm::launch<LogitsCfg<MODE_RESIDUAL>::EPI_WARPS, LogitsCfg<MODE_RESIDUAL>::BN>(
      ws.E, W2t, R, V, r, epi, stream, ws.count_fb, true);
  if (rc != DSPARK_OK) return rc;
  if (dspark_launch_pdl(resample_reduce, dim3(R), dim3(256), lz, stream, ws.rows,
                        (const int *)ws.list_fb, (const int *)ws.count_fb,
                        (const RowPartial *)ws.part, n_parts, (const bf16 *)base_logits, tgt,
                        (const bf16 *)ws.E, (const bf16 *)W2t, G, V, r, inv_tau, seed,
                        bonus) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  dspark_count_launches(3);  // + the GEMM, counted by launch()
  return DSPARK_OK;
}

extern "C" int dspark_verify_residual_rows(const dspark_dims *dims, const void *workspace,
                                          size_t workspace_bytes, int32_t *rejected,
                                          int32_t *explicit_rows, dspark_stream_t stream) {
  if (!dspark_dims_ok(dims) || !rejected || !explicit_rows) return DSPARK_ERR_ARG;
  const VerifyWs ws = verify_layout(dims, (char *)workspace);
  if (!workspace || workspace_bytes < ws.bytes || ((uintptr_t)workspace & 255))
    return DSPARK_ERR_WORKSPACE;
  int v[2] = {0, 0};
  if (cudaMemcpyAsync(&v[0], ws.count, sizeof(int), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaMemcpyAsync(&v[1], ws.count_fb, sizeof(int), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  *rejected = v[0];
  *explicit_rows = v[1];
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
