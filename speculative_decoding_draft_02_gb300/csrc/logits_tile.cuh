// logits_tile.cuh — one pass over the vocabulary for a batch of rows:
//   l[i, v] = l0[row_i, v] + E[i, :] . W2t[v, :]        (Markov bias, rank r)
// fused with a per-row decision over v (argmax, Gumbel-max, or the residual
// max(0, p_t - p_d) Gumbel-max of verification) and the log-sum-exp of l / tau.
// Logits stay on chip: each tile leaves only a RowPartial per row.
//
// "DSpark 深度解读" §二 设计一: B(x_{k-1}, .) = W1[x_{k-1}] W2 added to the base
// logits; "DSpark整体架构" stage two (sample left to right).
#pragma once
#include "common.cuh"

enum TileMode { MODE_GREEDY = 0, MODE_SAMPLE = 1, MODE_RESIDUAL = 2 };
enum RowKind { KIND_NONE = 0, KIND_RESIDUAL = 1, KIND_BONUS = 2 };

// Per-row context of a verification resample (one per request).
struct __align__(16) ResampleRow {
  int32_t kind;     // RowKind
  int32_t pos;      // 1-based draft position j* of the rejected (or bonus) row
  int32_t prev;     // token x_{j*-1} whose W1 row conditions the Markov bias
  float lse_t;      // logsumexp(t_{j*} / tau)
  float lse_d;      // logsumexp(l_{j*} / tau)
  int32_t pad[3];
};

struct TileArgs {
  const bf16 *base;      // [R*gamma, V]
  const bf16 *E;         // [M, r]  gathered W1 rows, one per row i
  const bf16 *W2t;       // [V, r]
  const bf16 *target;    // [R, gamma+1, V]            (residual)
  const ResampleRow *rows;  //                          (residual)
  RowPartial *part;      // [M, n_tiles]
  int M, V, r, gamma, k; // k: 1-based draft step (draft modes)
  int n_tiles;
  float inv_tau;
  uint64_t seed;
};

// Decision score of one vocabulary entry; also returns the scaled logit.
template <int MODE>
__device__ __forceinline__ float tile_score(const TileArgs &a, float logit, int v, int req,
                                            int pos, float lse_t, float lse_d, float tv,
                                            float &s, uint4 &rw, int &rw_q) {
  if (MODE == MODE_GREEDY) {
    s = logit;
    return logit;
  }
  const int q = v >> 2;
  if (q != rw_q) {
    rw = rng_words4(a.seed, (uint32_t)q, (uint32_t)pos, (uint32_t)req,
                    MODE == MODE_SAMPLE ? RNG_DRAFT : RNG_RESIDUAL);
    rw_q = q;
  }
  const float g = rng_gumbel(uint4_get(rw, v & 3));
  s = logit * a.inv_tau;
  if (MODE == MODE_SAMPLE) return s + g;
  // residual: p_t - p_d over the row
  const float pt = __expf(tv * a.inv_tau - lse_t);
  const float pd = __expf(s - lse_d);
  const float qv = pt - pd;
  return qv > 0.f ? __logf(qv) + g : -INFINITY;
}

// v0 tile: 32 rows x 128 vocabulary entries per CTA, rank streamed in chunks of
// 32 through shared memory, 4x4 outputs per thread, then one warp per row.
constexpr int TM = 32, TN = 128, TK = 32;

template <int MODE>
__global__ void __launch_bounds__(256) logits_tile_simple(TileArgs a) {
  __shared__ float Es[TK][TM + 1];
  __shared__ float Ws[TK][TN + 1];
  __shared__ float Ls[TM][TN + 1];
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < a.r; k0 += TK) {
    for (int e = threadIdx.x; e < TM * TK; e += 256) {
      const int mm = e / TK, kk = e % TK;
      Es[kk][mm] = (m0 + mm < a.M) ? __bfloat162float(a.E[(size_t)(m0 + mm) * a.r + k0 + kk]) : 0.f;
    }
    for (int e = threadIdx.x; e < TN * TK; e += 256) {
      const int nn = e / TK, kk = e % TK;
      Ws[kk][nn] = (n0 + nn < a.V) ? __bfloat162float(a.W2t[(size_t)(n0 + nn) * a.r + k0 + kk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < TK; ++kk) {
      float e4[4], w4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) e4[i] = Es[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) w4[j] = Ws[kk][tx + 32 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(e4[i], w4[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) Ls[ty * 4 + i][tx + 32 * j] = acc[i][j];
  __syncthreads();

  // one warp per row: add base logits, score, reduce
  for (int rr = ty; rr < TM; rr += 8) {
    const int i = m0 + rr;
    if (i >= a.M) break;
    int base_row, pos = a.k, req = i;
    float lse_t = 0.f, lse_d = 0.f;
    const bf16 *trow = nullptr;
    if (MODE == MODE_RESIDUAL) {
      const ResampleRow rw = a.rows[i];
      if (rw.kind != KIND_RESIDUAL) continue;
      pos = rw.pos;
      lse_t = rw.lse_t;
      lse_d = rw.lse_d;
      base_row = i * a.gamma + pos - 1;
      trow = a.target + ((size_t)i * (a.gamma + 1) + pos - 1) * a.V;
    } else {
      base_row = i * a.gamma + a.k - 1;
    }
    const bf16 *brow = a.base + (size_t)base_row * a.V;
    float m = -INFINITY, s = 0.f, best = -INFINITY, bs = 0.f;
    int idx = 0x7fffffff;
    float fb = -INFINITY;
    int fidx = 0x7fffffff;  // residual fallback: plain target sample
    uint4 rw4 = make_uint4(0, 0, 0, 0);
    int rw_q = -1;
    for (int c = tx; c < TN; c += 32) {
      const int v = n0 + c;
      if (v >= a.V) break;
      const float logit = __bfloat162float(brow[v]) + Ls[rr][c];
      const float tv = (MODE == MODE_RESIDUAL) ? __bfloat162float(trow[v]) : 0.f;
      float sc;
      const float score = tile_score<MODE>(a, logit, v, req, pos, lse_t, lse_d, tv, sc, rw4, rw_q);
      if (better(score, v, best, idx)) { best = score; idx = v; bs = sc; }
      if (MODE == MODE_SAMPLE) lse_merge(m, s, sc, 1.f);
      if (MODE == MODE_RESIDUAL) {
        const float g = rng_gumbel(uint4_get(rw4, v & 3));
        const float f = tv * a.inv_tau + g;
        if (better(f, v, fb, fidx)) { fb = f; fidx = v; }
      }
    }
    warp_merge(m, s, best, idx, bs);
    if (MODE == MODE_RESIDUAL) {
      float d0 = 0.f, d1 = 0.f, d2 = 0.f;
      warp_merge(d0, d1, fb, fidx, d2);
    }
    if (tx == 0) {
      RowPartial p;
      p.m = m; p.sum = s; p.best = best; p.idx = idx; p.best_s = bs;
      p.pad0 = fb; p.pad1 = __int_as_float(fidx); p.pad2 = 0.f;
      a.part[(size_t)i * a.n_tiles + blockIdx.x] = p;
    }
  }
}
