// logits_tile.cuh — the fused vocabulary pass behind the Markov head and the
// verification resample, as an epilogue of the tcgen05 GEMM:
//
//   bias[i, v] = E[i, :] . W2t[v, :]          (tensor cores, f32 in TMEM;
//                                              E[i] = W1[x_{k-1}] of row i)
//   l[i, v]    = l0[row_i, v] + bias[i, v]     (never written to memory)
//
// followed, per row and per SLICE-wide vocabulary slice, by what the mode asks
// for: greedy the slice's argmax; sampling the slice's log-sum-exp of l / tau
// and its block score (the first level of the two-level Gumbel-max draw, one
// slice = one sampler block); residual the block score of max(0, p_t - p_d).
// Each slice leaves one RowPartial per row; a small reduction combines the
// slices and, when sampling, draws inside the winning block (block_logits and
// block_pick below).
//
// "DSpark 深度解读" §二 设计一: B(x_{k-1}, .) = W1[x_{k-1}] W2 is added to the base
// logits and x_k is sampled from the result, left to right.
#pragma once
#include "umma_gemm.cuh"

enum TileMode { MODE_GREEDY = 0, MODE_SAMPLE = 1, MODE_RESIDUAL = 2 };
enum RowKind { KIND_NONE = 0, KIND_RESIDUAL = 1, KIND_BONUS = 2, KIND_FALLBACK = 3,
               KIND_TRIAL = 4 };
// KIND_FALLBACK: the residual max(0, p_t - p_d) of the rejected row was empty in
// floating point; the row is then sampled from p_t itself (residual stream).
// KIND_TRIAL: a rejection trial from p_t kept its proposal (no explicit pass).

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
  int M, V, gamma, k, n_parts;
  float inv_tau;
  uint64_t seed;

  static constexpr bool kRowAffine = true;
  static constexpr bool kStreamB = false;  // W2t is re-read by the other M blocks and steps
  static constexpr int SLICE = LogitsCfg<MODE>::SLICE;
  static constexpr int CH = LogitsCfg<MODE>::CH;
  static constexpr int CHUNKS = SLICE / 32;                       // greedy: 32-column loads
  // base-logit words prefetched per thread: the whole slice (greedy, sampling)
  // or the first chunk (residual, whose rows are known only inside the tile)
  static constexpr int BUF = MODE == MODE_RESIDUAL ? CH / 8 : SLICE / 8;
  static_assert(MODE == MODE_GREEDY || SLICE == GUMBEL_BLOCK,
                "a sampling slice is exactly one sampler block");

  // Kept by each epilogue thread across the tiles it processes.  Every tile of a
  // CTA lies in one row block (kRowAffine), so the residual row a thread
  // serves is looked up once.
  struct State {
    uint4 buf[BUF];  // base logits of the tile to process next, loaded ahead
    int req;         // residual: the request of this thread's compacted row
    bool active;
  };


  // base == nullptr: no base logits (the fused single-contraction step, whose
  // A operand carries h and the GEMM adds h . W_lm itself); they read as zeros
  __device__ __forceinline__ bool draft_row(int m0, int row, const bf16 *&brow) const {
    const int i = m0 + row;
    brow = base ? base + (size_t)(i * gamma + k - 1) * V : nullptr;
    return i < M;
  }

  // First tile: the whole slice, issued before the accumulator is ready.  Later
  // tiles: each chunk's words are reloaded for the next tile as soon as the
  // current tile has taken them (load_words inside operator()), so the loads
  // have a whole tile of work to land.
  __device__ void prefetch(int m0, int n0, int row, int c0, int, State &st) const {
    if (MODE == MODE_RESIDUAL) {
      const int i = m0 + row;
      st.active = i < *count;
      st.req = st.active ? list[i] : i;
      return;
    }
    const bf16 *brow = nullptr;
    if (!draft_row(m0, row, brow)) brow = nullptr;
    load_words<BUF>(brow, n0 + c0, st.buf);
  }

  // NW 16-byte words of row `src` from column n; zeros past V or without a row.
  template <int NW>
  __device__ __forceinline__ void load_words(const bf16 *src, int n, uint4 *dst) const {
#pragma unroll
    for (int q = 0; q < NW; ++q)
      dst[q] = (src && n + q * 8 + 8 <= V)
                   ? __ldg(reinterpret_cast<const uint4 *>(src + n + q * 8))
                   : make_uint4(0, 0, 0, 0);
  }

  __device__ void operator()(int m0, int n0, int row, uint32_t taddr, int c0, int c1,
                             int next_m0, int next_n0, State &st) const {
    constexpr float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;
    const int i = m0 + row;
    bool active = i < M;
    int pos = k;
    float lse_t = 0.f, lse_d = 0.f;
    const bf16 *trow = nullptr;
    const bf16 *brow = base;
    int req = i;  // request id: keys the random stream and the logit rows
    if (MODE == MODE_RESIDUAL) {
      active = st.active;
      if (active) {
        req = st.req;
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
    // the base-logit row of this thread in the CTA's next tile (none: zeros)
    const bf16 *nrow = nullptr;
    if (MODE != MODE_RESIDUAL && base && next_m0 >= 0 && next_m0 + row < M)
      nrow = base + (size_t)((next_m0 + row) * gamma + k - 1) * V;
    const int nn = next_n0 + c0;

    float m2 = -INFINITY, s = 0.f, best = -INFINITY;
    float z[4] = {0.f, 0.f, 0.f, 0.f};  // residual mass of the block (four partial sums)
    int idx = 0x7fffffff;

    if (MODE == MODE_GREEDY) {
#pragma unroll
      for (int cc = 0; cc < CHUNKS; ++cc) {
        const int c = c0 + cc * 32;
        uint32_t acc[32];
        tc::tmem_ld32(taddr + (uint32_t)c, acc);
        tc::tmem_wait_ld();
        const int n = n0 + c;
        const uint4 w4[4] = {st.buf[cc * 4], st.buf[cc * 4 + 1], st.buf[cc * 4 + 2],
                             st.buf[cc * 4 + 3]};
        load_words<4>(nrow, nn + cc * 32, st.buf + cc * 4);
        if (active && n < V) {
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
    } else if (MODE == MODE_SAMPLE) {
      // y = base + bias (unscaled); online log-sum-exp of y / tau in base 2
      const float c2 = inv_tau * LOG2E;  // log2(e) / tau > 0
      constexpr int NQ = CH / 8;         // 16-byte words per chunk
      constexpr int NCH = SLICE / CH;
      // TMEM loads one chunk ahead: chunk cc + 1 is in flight while cc is used
      uint32_t accs[2][CH];
      tc::tmem_ld<CH>(taddr + (uint32_t)c0, accs[0]);
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int c = c0 + cc * CH;
        tc::tmem_wait_ld();
        tc::reg_fence<CH>(accs[cc & 1]);
        if (cc + 1 < NCH) tc::tmem_ld<CH>(taddr + (uint32_t)(c + CH), accs[(cc + 1) & 1]);
        const uint32_t(&acc)[CH] = accs[cc & 1];
        const int n = n0 + c;
        uint4 cur[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) cur[q] = st.buf[cc * NQ + q];
        load_words<NQ>(nrow, nn + cc * CH, st.buf + cc * NQ);
        if (active && n < V) {
          float y[CH];
          unpack<CH>(cur, n, V, y);
#pragma unroll
          for (int j = 0; j < CH; ++j) y[j] += __uint_as_float(acc[j]);
          float mx[CH / 2];
#pragma unroll
          for (int j = 0; j < CH / 2; ++j) mx[j] = fmaxf(y[j], y[j + CH / 2]);
#pragma unroll
          for (int w = CH / 4; w >= 1; w >>= 1)
#pragma unroll
            for (int j = 0; j < w; ++j) mx[j] = fmaxf(mx[j], mx[j + w]);
          const float cmax2 = mx[0] * c2;
          if (cmax2 > m2) {
            s *= ex2_fast(m2 - cmax2);
            m2 = cmax2;
          }
          const float nm2 = -m2;
          float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < CH; ++j) ps[j & 3] += ex2_fast(fmaf(y[j], c2, nm2));
          s += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        }
      }
    } else {
      // residual mass sum_v max(0, p_t(v) - p_d(v)) at the rejected row; ids
      // past V read -inf on both sides and add nothing
      const float c2 = inv_tau * LOG2E;
      constexpr int NQ = CH / 8;
      uint4 nxt[NQ], nxt_t[NQ];  // base and target words of the next chunk
      if (active) {
        load_raw<CH>(brow, n0 + c0, V, nxt);
        load_raw<CH>(trow, n0 + c0, V, nxt_t);
      }
      const float nt = -lse_t * LOG2E, nd = -lse_d * LOG2E;
#pragma unroll 1
      for (int c = c0; c < c1; c += CH) {
        uint32_t acc[CH];
        tc::tmem_ld<CH>(taddr + (uint32_t)c, acc);
        tc::tmem_wait_ld();
        const int n = n0 + c;
        if (active && n < V) {
          uint4 cur[NQ], tw[NQ];
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            cur[q] = nxt[q];
            tw[q] = nxt_t[q];
          }
          if (c + CH < c1) {  // the next chunk's words, in flight during this one
            load_raw<CH>(brow, n + CH, V, nxt);
            load_raw<CH>(trow, n + CH, V, nxt_t);
          }
          float sv[CH], tv[CH];
          unpack<CH>(cur, n, V, sv);
          unpack<CH>(tw, n, V, tv);
#pragma unroll
          for (int j = 0; j < CH; ++j) {
            const float pt = ex2_fast(fmaf(tv[j], c2, nt));
            const float pd = ex2_fast(fmaf(sv[j] + __uint_as_float(acc[j]), c2, nd));
            z[j & 3] += fmaxf(pt - pd, 0.f);
          }
        }
      }
    }
    if (MODE != MODE_GREEDY) {
      // first level of the draw: the block score of this slice
      if (active && n0 + c0 < V) {
        const int b = (n0 + c0) / GUMBEL_BLOCK;
        const uint32_t stream = (MODE == MODE_SAMPLE ? RNG_DRAFT : RNG_RESIDUAL) + RNG_BLOCK_OFFSET;
        const uint4 w = rng_words4(seed, (uint32_t)(b >> 2), (uint32_t)pos, (uint32_t)req, stream);
        const float g = rng_gumbel(uint4_get(w, b & 3));
        if (MODE == MODE_SAMPLE) {
          best = m2 * LN2 + logf(s) + g;  // s >= 1: the block's first id is inside V
        } else {
          const float zb = (z[0] + z[1]) + (z[2] + z[3]);
          best = zb > 0.f ? logf(zb) + g : -INFINITY;
          s = zb;
        }
        idx = b;
      }
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

// ---------------------------------------------------------------------------
// Second level of a draw: the ids of the winning sampler block
// ---------------------------------------------------------------------------

// out[j] = base_row[v] + E . W2t[v] for v = b * GUMBEL_BLOCK + j, and -inf past
// V: the block's logits rebuilt from the Markov bias (E = W1[x_{k-1}]), or with
// base_row == nullptr the whole logit of a fused step (E = [h; W1[x_{k-1}]]
// against rows [W_lm; W2t], r their common length).  Every
// thread of a CTA of NT threads calls it; each warp takes GUMBEL_BLOCK / (NT/32)
// ids, and a lane has the W2t words of two passes (r = 512: all of its words)
// in flight at once.  Ends with a __syncthreads().
template <int NT>
__device__ void block_logits(const bf16 *__restrict__ base_row, const bf16 *__restrict__ E,
                             const bf16 *__restrict__ W2t, int b, int V, int r,
                             float *__restrict__ out) {
  constexpr int NW = NT / 32, PER = GUMBEL_BLOCK / NW;
  static_assert(PER * NW == GUMBEL_BLOCK, "warps must split the block evenly");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int v0 = b * GUMBEL_BLOCK + warp * PER;
  const uint4 *e4 = reinterpret_cast<const uint4 *>(E);
  const int r8 = r / 8;
  float acc[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) acc[u] = 0.f;
  int c = lane;
  for (; c + 32 < r8; c += 64) {
    const uint4 a0 = e4[c], a1 = e4[c + 32];
    uint4 w0[PER], w1[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const uint4 *rowp = reinterpret_cast<const uint4 *>(W2t + (size_t)(v0 + u) * r);
      const bool ok = v0 + u < V;
      w0[u] = ok ? __ldg(rowp + c) : make_uint4(0, 0, 0, 0);
      w1[u] = ok ? __ldg(rowp + c + 32) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) acc[u] = dot8_bf16(a1, w1[u], dot8_bf16(a0, w0[u], acc[u]));
  }
  for (; c < r8; c += 32) {  // r / 8 not a multiple of 64: one pass left
    const uint4 a = e4[c];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const uint4 w = (v0 + u < V)
                          ? __ldg(reinterpret_cast<const uint4 *>(W2t + (size_t)(v0 + u) * r) + c)
                          : make_uint4(0, 0, 0, 0);
      acc[u] = dot8_bf16(a, w, acc[u]);
    }
  }
#pragma unroll
  for (int u = 0; u < PER; ++u) acc[u] = warp_sum(acc[u]);
  if (lane == 0) {
#pragma unroll
    for (int u = 0; u < PER; ++u)
      out[warp * PER + u] =
          v0 + u < V ? (base_row ? __bfloat162float(base_row[v0 + u]) : 0.f) + acc[u]
                     : -INFINITY;
  }
  __syncthreads();
}

// The Gumbels of block b's ids on `stream`: lane l < 16 holds those of ids
// b * 64 + 4 l + t (t = 0..3).  They depend on no score, so a caller can draw
// them while the scores are still being computed.
struct BlockGumbels {
  float g[4];
};
__device__ __forceinline__ BlockGumbels block_gumbels(int b, uint64_t seed, uint32_t pos,
                                                      uint32_t req, uint32_t stream) {
  const int lane = threadIdx.x & 31;
  BlockGumbels out = {{0.f, 0.f, 0.f, 0.f}};
  if (lane < GUMBEL_BLOCK / 4) {
    const int v0 = b * GUMBEL_BLOCK + 4 * lane;
    const uint4 w = rng_words4(seed, (uint32_t)(v0 >> 2), pos, req, stream);
    out.g[0] = rng_gumbel(w.x);
    out.g[1] = rng_gumbel(w.y);
    out.g[2] = rng_gumbel(w.z);
    out.g[3] = rng_gumbel(w.w);
  }
  return out;
}

// Inside block b: the id with the largest score[j] + Gumbel(id) (lowest id on
// ties) among the ids with a finite score, given the block's Gumbels.  Called
// by one whole warp; every lane gets the id (-1 when no id qualifies).  score
// is in shared memory.
__device__ __forceinline__ int block_pick(const float *score, int b, int V,
                                          const BlockGumbels &gb) {
  const int lane = threadIdx.x & 31;
  float best = -INFINITY, d0 = 0.f, d1 = 0.f, d2 = 0.f;
  int idx = 0x7fffffff;
  if (lane < GUMBEL_BLOCK / 4) {
    const int v0 = b * GUMBEL_BLOCK + 4 * lane;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float sc = score[4 * lane + t];
      if (v0 + t < V && sc > -INFINITY) {
        const float e = sc + gb.g[t];
        if (better(e, v0 + t, best, idx)) { best = e; idx = v0 + t; }
      }
    }
  }
  warp_merge(d0, d1, best, idx, d2);
  return best > -INFINITY ? idx : -1;
}

// The same draw with the Gumbels taken on `stream` here.
__device__ __forceinline__ int block_pick(const float *score, int b, int V, uint64_t seed,
                                          uint32_t pos, uint32_t req, uint32_t stream) {
  return block_pick(score, b, V, block_gumbels(b, seed, pos, req, stream));
}
