// logits_tile.cuh — the fused vocabulary pass behind the Markov head and the
// verification resample, as an epilogue of the tcgen05 GEMM:
//
//   bias[i, v] = E[i, :] . W2t[v, :]          (tensor cores, f32 in TMEM;
//                                              E[i] = W1[x_{k-1}] of row i)
//   l[i, v]    = l0[row_i, v] + bias[i, v]     (never written to memory)
//
// followed, per row and per PART_N-wide vocabulary slice, by the decision the
// mode asks for and the online log-sum-exp of l / tau.  Each slice leaves one
// RowPartial per row; a small reduction combines the slices.
//
// "DSpark 深度解读" §二 设计一: B(x_{k-1}, .) = W1[x_{k-1}] W2 is added to the base
// logits and x_k is sampled from the result, left to right.
#pragma once
#include "umma_gemm.cuh"

enum TileMode { MODE_GREEDY = 0, MODE_SAMPLE = 1, MODE_RESIDUAL = 2 };
enum RowKind { KIND_NONE = 0, KIND_RESIDUAL = 1, KIND_BONUS = 2, KIND_FALLBACK = 3 };
// KIND_FALLBACK: the residual max(0, p_t - p_d) of the rejected row was empty in
// floating point; the row is then sampled from p_t itself (residual stream).

// Per-request context of a verification resample.
struct __align__(16) ResampleRow {
  int32_t kind;     // RowKind
  int32_t pos;      // 1-based position j* of the rejected (or bonus) row
  int32_t prev;     // token x_{j*-1} whose W1 row conditions the Markov bias
  float lse_t;      // logsumexp(t_{j*} / tau)
  float lse_d;      // logsumexp(l_{j*} / tau)
  int32_t pad[3];
};

// Epilogue geometry of each mode: BN columns per tile, EPI_WARPS epilogue warps
// (each TMEM lane quarter is shared by EPI_WARPS / 4 warps), SLICE columns per
// thread and tile (= vocabulary entries per partial), CH columns per TMEM
// load.  Sampling runs the most warps per column: its per-entry work (Philox
// words, log-sum-exp) needs the latency hiding.
template <int MODE>
struct LogitsCfg {
  static constexpr int BN = 256;                                     // N-tile
  static constexpr int EPI_WARPS = MODE == MODE_GREEDY ? 8 : 16;
  static constexpr int SLICE = BN / (EPI_WARPS / 4);
  static constexpr int CH = MODE == MODE_GREEDY ? 32 : 16;
};
constexpr int MIN_PART_N = 64;  // the narrowest slice of any mode

template <int MODE>
static inline int logits_parts(int V) {
  return (V + LogitsCfg<MODE>::SLICE - 1) / LogitsCfg<MODE>::SLICE;
}
// Partials per row to size a workspace for every mode.
static inline size_t logits_parts_max(int V) { return (size_t)(V + MIN_PART_N - 1) / MIN_PART_N; }

// CH bf16 starting at src[n] as 16-byte words; groups past V read nothing.
template <int CH>
__device__ __forceinline__ void load_raw(const bf16 *src, int n, int V, uint4 (&w)[CH / 8]) {
#pragma unroll
  for (int q = 0; q < CH / 8; ++q)
    w[q] = (n + q * 8 + 8 <= V) ? __ldg(reinterpret_cast<const uint4 *>(src + n + q * 8))
                                : make_uint4(0, 0, 0, 0);
}
__device__ __forceinline__ void load_raw32(const bf16 *src, int n, int V, uint4 (&w)[4]) {
  load_raw<32>(src, n, V, w);
}
// Unpack to floats; entries past V become -inf.
template <int CH>
__device__ __forceinline__ void unpack(const uint4 (&w)[CH / 8], int n, int V, float (&out)[CH]) {
  if (n + CH <= V) {  // whole chunk inside the vocabulary (warp-uniform)
#pragma unroll
    for (int q = 0; q < CH / 8; ++q) {
      const uint32_t ws[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        out[q * 8 + 2 * t] = bf16_lo(ws[t]);
        out[q * 8 + 2 * t + 1] = bf16_hi(ws[t]);
      }
    }
    return;
  }
#pragma unroll
  for (int q = 0; q < CH / 8; ++q) {
    const bool ok = n + q * 8 + 8 <= V;
    const uint32_t ws[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      out[q * 8 + 2 * t] = ok ? bf16_lo(ws[t]) : -INFINITY;
      out[q * 8 + 2 * t + 1] = ok ? bf16_hi(ws[t]) : -INFINITY;
    }
  }
}
__device__ __forceinline__ void unpack32(const uint4 (&w)[4], int n, int V, float (&out)[32]) {
  unpack<32>(w, n, V, out);
}

template <int MODE>
struct EpiLogits {
  const bf16 *base;          // [R*gamma, V]
  const bf16 *target;        // [R, gamma+1, V]       (residual)
  const ResampleRow *rows;   // [R]                    (residual)
  const int *list;           // [R] request of each compacted row (residual)
  const int *count;          // number of compacted rows           (residual)
  RowPartial *part;          // [R, n_parts]
  float *gfloor;             // [R] best Gumbel score found so far on each row, shared by
                             // every CTA of the pass (set to -inf before the pass)
  int M, V, gamma, k, n_parts;
  float inv_tau;
  uint64_t seed;

  static constexpr bool kRowAffine = true;
  static constexpr bool kStreamB = false;  // W2t is re-read by the other M blocks and steps
  static constexpr int SLICE = LogitsCfg<MODE>::SLICE;
  static constexpr int CH = LogitsCfg<MODE>::CH;
  static constexpr int CHUNKS = SLICE / 32;                       // greedy: 32-column loads
  static constexpr int BUF = MODE == MODE_GREEDY ? SLICE / 8 : CH / 8;

  // Kept by each epilogue thread across the tiles it processes.
  struct State {
    int m0 = -1;               // row block the floor belongs to
    float floor = -INFINITY;   // best score known on this row (own tiles + shared floor)
    float seen = -INFINITY;    // shared floor read at the start of the current tile
    uint4 buf[BUF];            // base logits prefetched before the accumulator is ready
  };

  __device__ __forceinline__ bool draft_row(int m0, int row, const bf16 *&brow) const {
    const int i = m0 + row;
    brow = base + (size_t)(i * gamma + k - 1) * V;
    return i < M;
  }

  __device__ void prefetch(int m0, int n0, int row, int c0, int, State &st) const {
    const int i = m0 + row;
    if (MODE != MODE_GREEDY && i < M)
      st.seen = *reinterpret_cast<volatile const float *>(gfloor + i);
    if (MODE == MODE_RESIDUAL) return;
    const bf16 *brow;
    if (!draft_row(m0, row, brow)) return;
    const int n = n0 + c0;
    // greedy: the whole slice, so the epilogue never waits on HBM; sampling:
    // the first chunk, later chunks are loaded one ahead
#pragma unroll
    for (int q = 0; q < BUF; ++q)
      st.buf[q] = (n + q * 8 + 8 <= V) ? __ldg(reinterpret_cast<const uint4 *>(brow + n + q * 8))
                                       : make_uint4(0, 0, 0, 0);
  }

  __device__ void operator()(int m0, int n0, int row, uint32_t taddr, int c0, int c1,
                             State &st) const {
    constexpr float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;
    const int i = m0 + row;
    bool active = i < M;
    int pos = k;
    float lse_t = 0.f, lse_d = 0.f;
    const bf16 *trow = nullptr;
    const bf16 *brow = base;
    int req = i;  // request id: keys the random stream and the logit rows
    if (MODE == MODE_RESIDUAL) {
      active = i < *count;
      if (active) {
        req = list[i];
        const ResampleRow rr = rows[req];
        pos = rr.pos;
        lse_t = rr.lse_t;
        lse_d = rr.lse_d;
        brow = base + (size_t)(req * gamma + pos - 1) * V;
        trow = target + ((size_t)req * (gamma + 1) + pos - 1) * V;
      }
    } else {
      draft_row(m0, row, brow);
    }
    if (st.m0 != m0) { st.m0 = m0; st.floor = -INFINITY; }
    st.floor = fmaxf(st.floor, st.seen);
    const uint32_t stream = MODE == MODE_SAMPLE ? RNG_DRAFT : RNG_RESIDUAL;

    float m2 = -INFINITY, s = 0.f, best = -INFINITY, bs = 0.f;
    int idx = 0x7fffffff;

    if (MODE == MODE_GREEDY) {
#pragma unroll
      for (int cc = 0; cc < CHUNKS; ++cc) {
        const int c = c0 + cc * 32;
        uint32_t acc[32];
        tc::tmem_ld32(taddr + (uint32_t)c, acc);
        tc::tmem_wait_ld();
        const int n = n0 + c;
        if (active && n < V) {
          const uint4 w4[4] = {st.buf[cc * 4], st.buf[cc * 4 + 1], st.buf[cc * 4 + 2],
                               st.buf[cc * 4 + 3]};
          float sv[32];
          unpack32(w4, n, V, sv);
          // four interleaved argmax chains (entries j = 4 q + p), merged with
          // ties to the lower id
          float pb[4] = {best, -INFINITY, -INFINITY, -INFINITY};
          int pi[4] = {idx, 0x7fffffff, 0x7fffffff, 0x7fffffff};
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float l = sv[j] + __uint_as_float(acc[j]);
            const bool b = l > pb[j & 3];  // strict: within a chain ids increase
            pb[j & 3] = b ? l : pb[j & 3];
            pi[j & 3] = b ? n + j : pi[j & 3];
          }
#pragma unroll
          for (int p = 1; p < 4; ++p)
            if (better(pb[p], pi[p], pb[0], pi[0])) { pb[0] = pb[p]; pi[0] = pi[p]; }
          best = pb[0];
          idx = pi[0];
        }
      }
    } else {
      const PhiloxKeys keys(seed);
      const float c2 = inv_tau * LOG2E;  // scaled logits in log2 units
      constexpr int NQ = CH / 8;         // 16-byte words per chunk
      constexpr int NH = CH / 16;        // halves of 16 entries (4 Philox calls each)
      uint4 nxt[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) nxt[q] = st.buf[q];
      if (MODE == MODE_RESIDUAL && active) load_raw<CH>(brow, n0 + c0, V, nxt);
#pragma unroll 1
      for (int c = c0; c < c1; c += CH) {
        uint32_t acc[CH];
        tc::tmem_ld<CH>(taddr + (uint32_t)c, acc);
        tc::tmem_wait_ld();
        const int n = n0 + c;
        if (active && n < V) {
          uint4 cur[NQ];
#pragma unroll
          for (int q = 0; q < NQ; ++q) cur[q] = nxt[q];
          if (c + CH < c1) load_raw<CH>(brow, n + CH, V, nxt);  // prefetch the next chunk
          float sv[CH];
          unpack<CH>(cur, n, V, sv);
          const float F = fmaxf(best, st.floor);  // a score some entry of the row reaches

          if (MODE == MODE_SAMPLE) {
            // y = base + bias (unscaled); the draft distribution is softmax(y / tau)
            float y[CH];
#pragma unroll
            for (int j = 0; j < CH; ++j) y[j] = sv[j] + __uint_as_float(acc[j]);
            float mx[CH / 2];
#pragma unroll
            for (int j = 0; j < CH / 2; ++j) mx[j] = fmaxf(y[j], y[j + CH / 2]);
#pragma unroll
            for (int w = CH / 4; w >= 1; w >>= 1)
#pragma unroll
              for (int j = 0; j < w; ++j) mx[j] = fmaxf(mx[j], mx[j + w]);
            const float cmax2 = mx[0] * c2;  // c2 = log2(e) / tau > 0
            // online log-sum-exp in base 2 (four partial sums)
            if (cmax2 > m2) {
              s *= ex2_fast(m2 - cmax2);
              m2 = cmax2;
            }
            const float nm2 = -m2;
            float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < CH; ++j) ps[j & 3] += ex2_fast(fmaf(y[j], c2, nm2));
            s += (ps[0] + ps[1]) + (ps[2] + ps[3]);

            // Gumbel-max without the logarithms of entries that cannot win.
            // Entry j beats F only if g_j > F - s_j (s_j = y_j / tau).  Since
            // -log u >= 1 - u, 1 - u_j >= e^{s_j - F + 0.01} implies
            // g_j < F - s_j - 0.01.  Chunk test first (s_j <= cmax, an integer
            // threshold on w >> 9, u = ((w >> 9) + 1/2) 2^-23), then the same
            // test per entry with e^{s_j - F} = 2^{y_j c2 - m2} e^{m - F}.
            int w_thr = -1;
            if (F > -INFINITY) {
              const float t = fminf(F - cmax2 * LN2, 15.f);
              const float X = __expf(-(t - 0.01f)) * 8388608.f;
              w_thr = X >= 8388607.f ? -1 : 8388607 - (int)ceilf(X);
            }
            const float K = F > -INFINITY ? __expf(m2 * LN2 - F + 0.01f) : INFINITY;
            const bool per_entry = K < 1e30f;
            // Philox words in halves of 16 entries (one call per 4 entries).
            // The common path needs only their maximum; the per-entry test,
            // needed only when the chunk test fails, draws them again.
#pragma unroll
            for (int h = 0; h < NH; ++h) {
              uint32_t wmax = 0;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint4 w = keys(make_uint4((uint32_t)((n >> 2) + 4 * h + q), (uint32_t)pos,
                                                (uint32_t)req, stream));
                wmax = max(max(wmax, max(w.x, w.y)), max(w.z, w.w));
              }
              if ((int)(wmax >> 9) > w_thr) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const uint4 w = keys(make_uint4((uint32_t)((n >> 2) + 4 * h + q),
                                                  (uint32_t)pos, (uint32_t)req, stream));
                  const uint32_t wq[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                  for (int l = 0; l < 4; ++l) {
                    const int j = 16 * h + 4 * q + l;
                    const bool cand = !per_entry || (1.f - rng_uniform(wq[l])) <
                                                        ex2_fast(fmaf(y[j], c2, nm2)) * K;
                    if (cand) {
                      const float sn = y[j] * inv_tau;
                      const float sc = sn + rng_gumbel(wq[l]);
                      if (sc > best) { best = sc; idx = n + j; bs = sn; }
                    }
                  }
                }
              }
            }
          } else {
            // residual max(0, p_t - p_d) at the rejected position.  The score
            // log q_j + g_j <= log p_t(j) + g_j, so by the same argument an
            // entry is skipped when 1 - u_j >= p_t(j) e^{-F + 0.01}; the chunk
            // test uses the chunk's largest p_t.
            uint4 tw[NQ];
            load_raw<CH>(trow, n, V, tw);
            float tv[CH];
            unpack<CH>(tw, n, V, tv);
            float mx[CH / 2];
#pragma unroll
            for (int j = 0; j < CH / 2; ++j) mx[j] = fmaxf(tv[j], tv[j + CH / 2]);
#pragma unroll
            for (int w = CH / 4; w >= 1; w >>= 1)
#pragma unroll
              for (int j = 0; j < w; ++j) mx[j] = fmaxf(mx[j], mx[j + w]);
            int w_thr = -1;
            if (F > -INFINITY) {
              const float X = __expf(fminf(mx[0] * inv_tau - lse_t - F + 0.01f, 0.f)) * 8388608.f;
              w_thr = X >= 8388607.f ? -1 : 8388607 - (int)ceilf(X);
            }
            const float K = F > -INFINITY ? __expf(0.01f - F) : INFINITY;
            const bool per_entry = K < 1e30f;
#pragma unroll
            for (int h = 0; h < NH; ++h) {
              uint32_t ws[16];
              uint32_t wmax = 0;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint4 w = keys(make_uint4((uint32_t)((n >> 2) + 4 * h + q), (uint32_t)pos,
                                                (uint32_t)req, stream));
                ws[q * 4 + 0] = w.x; ws[q * 4 + 1] = w.y; ws[q * 4 + 2] = w.z; ws[q * 4 + 3] = w.w;
                wmax = max(max(wmax, max(w.x, w.y)), max(w.z, w.w));
              }
              if ((int)(wmax >> 9) > w_thr) {
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const int j = 16 * h + e;
                  const float pt = __expf(tv[j] * inv_tau - lse_t);
                  const bool cand = (n + j < V) &&
                                    (!per_entry || (1.f - rng_uniform(ws[e])) < pt * K);
                  if (cand) {
                    const float sl = (sv[j] + __uint_as_float(acc[j])) * inv_tau;
                    const float qv = pt - __expf(sl - lse_d);
                    if (qv > 0.f) {
                      const float sc = __logf(qv) + rng_gumbel(ws[e]);
                      if (sc > best) { best = sc; idx = n + j; }
                    }
                  }
                }
              }
            }
          }
        }
      }
    }
    if (MODE != MODE_GREEDY && active) {
      st.floor = fmaxf(st.floor, best);
      if (st.floor > st.seen) atomic_max_float(gfloor + i, st.floor);
    }
    if (active && n0 + c0 < V) {
      RowPartial p;
      p.m = MODE == MODE_SAMPLE ? m2 * LN2 : -INFINITY;
      p.sum = s;
      p.best = best;
      p.idx = idx;
      part[(size_t)i * n_parts + (n0 + c0) / SLICE] = p;
    }
  }
  __device__ void on_timeout() const { dspark_set_status(DSPARK_ERR_TIMEOUT); }
};
