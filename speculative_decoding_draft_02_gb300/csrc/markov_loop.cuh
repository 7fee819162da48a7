// markov_loop.cuh — the whole gamma-step Markov loop (a2-a4) as one persistent,
// cooperatively launched kernel.
//
// "DSpark 深度解读" §二 设计一: x_k is drawn from l_k = l0_k + W1[x_{k-1}] W2, left
// to right, so step k + 1 needs every vocabulary entry of step k.  One CTA per
// SM stays resident for all gamma steps:
//
//   vocabulary pass of step k   the tcgen05 GEMM E_k . W2t^T (E_k = W1[x_{k-1}]),
//                               whose epilogue adds the base logits and, per
//                               64-id slice, takes the log-sum-exp and block
//                               score (sampling) or the argmax (greedy).  Each
//                               epilogue thread folds the slices it visits into
//                               one running partial per row and writes it once
//                               per step, so a row has a few hundred partials,
//                               not V / 64.
//   grid barrier
//   row phase of step k         the epilogue warps, in groups of RW warps, take
//                               one request each: combine its partials into
//                               lse_k and the winning block (or x_k), rebuild
//                               that block's 64 logits and draw x_k inside it,
//                               then write E_{k+1} = W1[x_k] and c_{k+1}.
//   grid barrier                (k < gamma)
//
// Before step 1 a prologue row phase gathers E_1 = W1[anchor] and c_1.  The
// hidden-state part of c_{k+1}, w_h . h_{k+1}, does not depend on x_k: the
// epilogue warps take it at the start of step k, while the step's first
// accumulator is computed, and the row phase only adds w_e . W1[x_k].
//
// W2t and the base logits do not depend on x_k: before the second barrier the
// producer already issues the W2t halves of the next step's first stages and
// the epilogue holds the base-logit words of its next tile, so only the E
// halves wait for the barrier.  Every wait (mbarrier or grid barrier) is
// bounded; a CTA that gives up raises a flag that makes the others give up too.
#pragma once
#include <stdio.h>
#include <stdlib.h>

#include "logits_tile.cuh"

namespace mloop {

using gemm::A_BYTES;
using gemm::BK;
using gemm::BM;

// Grid barrier words; zeroed in stream order before every launch.
struct __align__(16) LoopSync {
  unsigned int arrived;  // arrivals of all barriers so far (monotonic in a launch)
  int abort;             // a CTA gave up on a wait
  unsigned int pad[2];
};

// Tile shape of the loop's vocabulary pass.  Sampling: 192-column tiles over
// 12 epilogue warps (3 column groups of 64 = one sampler block per thread and
// tile); 14 warps per CTA leave 128 registers per thread (18 warps would leave
// 96 and spill in the tile loop), and 674 x 2 tiles over 152 SMs fill 8.87 of
// 9 waves.  Greedy: 256-column tiles over 8 warps (128 columns per thread).
template <int MODE>
struct LoopCfg {
  static constexpr int BN = MODE == MODE_GREEDY ? 256 : 192;
  static constexpr int EPI_WARPS = MODE == MODE_GREEDY ? 8 : 12;
  static constexpr int CG = EPI_WARPS / 4;  // column groups: threads per row in a tile
  static constexpr int SLICE = BN / CG;
  static constexpr int CH = MODE == MODE_GREEDY ? 32 : 16;  // columns per TMEM load
  static_assert(MODE == MODE_GREEDY || SLICE == GUMBEL_BLOCK, "a sampling slice is one block");
};

struct LoopArgs {
  const bf16 *base;   // [R*gamma, V]  base logits l0
  const bf16 *W1;     // [V, r]
  const bf16 *W2t;    // [V, r]
  const bf16 *h;      // [R*gamma, d]  backbone hidden states
  const bf16 *w_h;    // [d]  hidden half of the confidence weight
  const bf16 *w_e;    // [r]  embedding half of the confidence weight
  const int32_t *anchor;  // [R]  x_0
  float *zh;          // [R*gamma]  w_h . h, position k written during step k's tile phase
  const float *T;     // [gamma]
  bf16 *E;            // [R, r]  A operand: W1[x_{k-1}] (row i rewritten by row i's group)
  int32_t *tokens;    // [R, gamma]
  float *conf;        // [R, gamma]
  float *lse_out;     // [R, gamma] or null
  float *logp_out;    // [R, gamma] or null
  RowPartial *part;   // [R, n_slots]
  LoopSync *sync;
  int R, V, r, d, gamma, n_slots;
  float inv_tau;
  uint64_t seed;
};

template <int STAGES>
struct LoopCtl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t go;     // the grid barrier after a row phase has passed: E may be loaded
  uint64_t efull;  // resident-E form: the step's E tile has landed
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Shared scratch of one row group (NS: room for a rebuilt block's logits,
// which only sampling needs).
template <int RW, int NS>
struct RowScratch {
  float score[NS];  // the winning block's logits, then logits / tau
  float m[RW], s[RW], b[RW], dot[RW];
  int i[RW];
  int tok;
};
template <int MODE, int RW>
using Scratch = RowScratch<RW, MODE == MODE_SAMPLE ? GUMBEL_BLOCK : 1>;

// Resident-E form of the loop (EKB > 0): each CTA keeps its row block's E (up
// to EKB k blocks of 128 x 64: r <= 64 EKB, EKB = 4 or 8) in shared memory for
// the whole step, and only W2t streams through a ring of eres_stages() stages,
// as many as fit beside E and the row groups' scratch (up to six, at least
// three).  A greedy 128 x 256 tile then moves 256 KB from L2 instead of 384 KB
// (r = 512), a sampling 128 x 192 tile 192 KB instead of 320 KB.
template <int MODE, int RW, int EKB>
constexpr int eres_stages() {
  constexpr size_t fixed = 1024 + (size_t)EKB * A_BYTES + 512 +
                           sizeof(Scratch<MODE, RW>) * (LoopCfg<MODE>::EPI_WARPS / RW);
  constexpr size_t n = (gemm::SMEM_LIMIT - fixed) / gemm::Geo<LoopCfg<MODE>::BN>::B_BYTES;
  static_assert(n >= 3, "resident E leaves room for three W2t stages");
  return n > 6 ? 6 : (int)n;
}

// Bring `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// A named barrier that also returns, to every participant, the OR of `pred`
// over them: one decision that all of them act on alike.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}
constexpr int BAR_STOP = 15;  // named barrier of the stop decision (row groups use 2 ..)

// Generic-proxy stores of this thread become visible to later TMA (async proxy)
// reads of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Every CTA of the grid arrives; returns once `target` arrivals are counted.
// Called by one thread per CTA after a CTA-level barrier.  Gives up (false)
// after tc::WAIT_LIMIT_NS or when another CTA has given up.
__device__ bool grid_barrier(LoopSync *gs, unsigned int target) {
  // release: this CTA's writes (ordered before by the CTA barrier) are visible
  // to whoever acquires the count
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&gs->arrived) : "memory");
  const uint64_t t0 = tc::globaltimer();
  for (uint32_t it = 0;; ++it) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(&gs->arrived) : "memory");
    if (v >= target) return true;  // the acquire load orders what follows
    if ((it & 15) == 15) {
      if (*(volatile int *)&gs->abort) return false;
      if (tc::globaltimer() - t0 > tc::WAIT_LIMIT_NS) {
        atomicExch(&gs->abort, 1);
        return false;
      }
    }
  }
}

// Running partial of one epilogue thread: its row's slices seen so far.
struct Run {
  float m2;   // sampling: running max of the base-2 scaled logits
  float s;    // sampling: sum of 2^(scaled - m2)
  float best; // sampling: best block score; greedy: best logit
  int idx;    // sampling: its block; greedy: its id
  __device__ __forceinline__ void reset() {
    m2 = -INFINITY;
    s = 0.f;
    best = -INFINITY;
    idx = 0x7fffffff;
  }
};

// One tile of the vocabulary pass for this thread's row and column slice
// [c0, c0 + SLICE): folds the slice into `run`.  `buf` holds the slice's base
// words on entry and the next tile's (row nrow, column nn0) on exit.
template <int MODE>
__device__ __forceinline__ void tile_slice(const LoopArgs &a, int k, int i, bool active, int n0,
                                           int c0, uint32_t taddr, const bf16 *nrow, int nn0,
                                           uint4 *buf, Run &run) {
  constexpr float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;
  constexpr int SLICE = LoopCfg<MODE>::SLICE;
  constexpr int CH = LoopCfg<MODE>::CH;
  constexpr int NQ = CH / 8;
  constexpr int NCH = SLICE / CH;
  const int V = a.V;
  auto load_next = [&](int n, uint4 *dst) {
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      dst[q] = (nrow && n + q * 8 + 8 <= V)
                   ? __ldg(reinterpret_cast<const uint4 *>(nrow + n + q * 8))
                   : make_uint4(0, 0, 0, 0);
  };
  if (MODE == MODE_GREEDY) {
    float best = run.best;
    int idx = run.idx;
#pragma unroll
    for (int cc = 0; cc < NCH; ++cc) {
      const int c = c0 + cc * CH;
      uint32_t acc[CH];
      tc::tmem_ld<CH>(taddr + (uint32_t)c, acc);
      tc::tmem_wait_ld();
      const int n = n0 + c;
      uint4 cur[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) cur[q] = buf[cc * NQ + q];
      load_next(nn0 + cc * CH, buf + cc * NQ);
      if (active && n < V) {
        float sv[CH];
        unpack<CH>(cur, n, V, sv);
        // four interleaved argmax chains (ids j = 4 q + p), merged with ties to the lower id
        float pb[4] = {best, -INFINITY, -INFINITY, -INFINITY};
        int pi[4] = {idx, 0x7fffffff, 0x7fffffff, 0x7fffffff};
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          const float l = sv[j] + __uint_as_float(acc[j]);
          const bool b = l > pb[j & 3];
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
    run.best = best;
    run.idx = idx;
  } else {
    const float c2 = a.inv_tau * LOG2E;
    float m2 = -INFINITY, s = 0.f;
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
      for (int q = 0; q < NQ; ++q) cur[q] = buf[cc * NQ + q];
      load_next(nn0 + cc * CH, buf + cc * NQ);
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
    if (active && n0 + c0 < V) {
      // first level of the draw: this slice is sampler block b
      const int b = (n0 + c0) / GUMBEL_BLOCK;
      const uint4 w = rng_words4(a.seed, (uint32_t)(b >> 2), (uint32_t)k, (uint32_t)i,
                                 RNG_DRAFT + RNG_BLOCK_OFFSET);
      const float score = m2 * LN2 + logf(s) + rng_gumbel(uint4_get(w, b & 3));
      if (m2 > run.m2) {
        run.s = run.s * ex2_fast(run.m2 - m2) + s;
        run.m2 = m2;
      } else {
        run.s += s * ex2_fast(m2 - run.m2);
      }
      if (better(score, b, run.best, run.idx)) { run.best = score; run.idx = b; }
    }
  }
}

// Markov bias of sampler block b, rebuilt by the RW warps of a row group:
// out[j] = E_row . W2t[v] for v = b * 64 + j (-inf past V).  Every lane runs
// hook() once, after its first W2t words are requested, to fill their latency.
template <int RW, class Hook>
__device__ __forceinline__ void rebuild_bias(const bf16 *E_row, const bf16 *__restrict__ W2t,
                                             int b, int V, int r, float *out, int wg, int lane,
                                             Hook hook) {
  // warp wg takes ids wg, wg + RW, wg + 2 RW, ... (RW need not divide 64), four
  // at a time: each lane has their W2t words of two passes in flight
  constexpr int CHK = 4;
  const uint4 *e4 = reinterpret_cast<const uint4 *>(E_row);
  const int r8 = r / 8;
  // this lane's first two 16-byte words of E (all of them when r <= 512)
  const uint4 e0 = lane < r8 ? __ldcg(e4 + lane) : make_uint4(0, 0, 0, 0);
  const uint4 e1 = lane + 32 < r8 ? __ldcg(e4 + lane + 32) : make_uint4(0, 0, 0, 0);
#pragma unroll 1
  for (int t0 = 0; wg + RW * t0 < GUMBEL_BLOCK; t0 += CHK) {
    int ids[CHK];
#pragma unroll
    for (int u = 0; u < CHK; ++u) ids[u] = wg + RW * (t0 + u);  // 64 or more: no id
    float acc[CHK];
#pragma unroll
    for (int u = 0; u < CHK; ++u) acc[u] = 0.f;
    for (int c = lane; c < r8; c += 64) {
      const bool two = c + 32 < r8;
      const uint4 a0 = c == lane ? e0 : __ldcg(e4 + c);
      const uint4 a1 = c == lane ? e1 : (two ? __ldcg(e4 + c + 32) : make_uint4(0, 0, 0, 0));
      uint4 w0[CHK], w1[CHK];
#pragma unroll
      for (int u = 0; u < CHK; ++u) {
        const int v = b * GUMBEL_BLOCK + ids[u];
        const uint4 *rowp = reinterpret_cast<const uint4 *>(W2t + (size_t)v * r);
        const bool ok = ids[u] < GUMBEL_BLOCK && v < V;
        w0[u] = ok ? __ldg(rowp + c) : make_uint4(0, 0, 0, 0);
        w1[u] = (ok && two) ? __ldg(rowp + c + 32) : make_uint4(0, 0, 0, 0);
      }
      if (t0 == 0 && c == lane) hook();
#pragma unroll
      for (int u = 0; u < CHK; ++u) acc[u] = dot8_bf16(a1, w1[u], dot8_bf16(a0, w0[u], acc[u]));
    }
    if (t0 == 0 && lane >= r8) hook();  // lanes that had no words to load
#pragma unroll
    for (int u = 0; u < CHK; ++u) acc[u] = warp_sum(acc[u]);
    if (lane == 0) {
#pragma unroll
      for (int u = 0; u < CHK; ++u) {
        const int v = b * GUMBEL_BLOCK + ids[u];
        if (ids[u] < GUMBEL_BLOCK) out[ids[u]] = v < V ? acc[u] : -INFINITY;
      }
    }
  }
}

// This thread's part of w_h . h[i, p] (0-based position p), "DSpark 深度解读"
// §二 设计二: the hidden-state half of the confidence logit.  Its loads do not
// depend on the drafted tokens, so the row phase issues them first.
template <int RW>
__device__ __forceinline__ float hidden_dot_part(const LoopArgs &a, int i, int p, int tg) {
  constexpr int RT = 32 * RW;
  const int n8 = a.d / 8;
  const uint4 *hr = reinterpret_cast<const uint4 *>(a.h + ((size_t)i * a.gamma + p) * a.d);
  const uint4 *wh = reinterpret_cast<const uint4 *>(a.w_h);
  float z = 0.f;
#pragma unroll 1
  for (int c0 = 0; c0 < n8; c0 += 8 * RT) {  // up to eight pairs in flight
    uint4 x[8], w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = c0 + u * RT + tg;
      x[u] = c < n8 ? __ldg(hr + c) : make_uint4(0, 0, 0, 0);
      w[u] = c < n8 ? __ldg(wh + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) z = dot8_bf16(x[u], w[u], z);
  }
  return z;
}

// zh[i, p] = w_h . h[i, p] for every request, one warp per request (warp gw of
// n_warps in the grid): run by the epilogue warps at the start of a step,
// while the step's first accumulator is being computed.
__device__ __forceinline__ void hidden_dots(const LoopArgs &a, int p, int gw, int n_warps,
                                            int lane) {
  const int n8 = a.d / 8;
  const uint4 *wh = reinterpret_cast<const uint4 *>(a.w_h);
  for (int i = gw; i < a.R; i += n_warps) {
    const size_t o = (size_t)i * a.gamma + p;
    const uint4 *hr = reinterpret_cast<const uint4 *>(a.h + o * a.d);
    float z = 0.f;
#pragma unroll 1
    for (int c0 = 0; c0 < n8; c0 += 8 * 32) {
      uint4 x[8], w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * 32 + lane;
        x[u] = c < n8 ? __ldg(hr + c) : make_uint4(0, 0, 0, 0);
        w[u] = c < n8 ? __ldg(wh + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) z = dot8_bf16(x[u], w[u], z);
    }
    z = warp_sum(z);
    if (lane == 0) a.zh[o] = z;
  }
}

// For request i and 0-based position p: E[i] = W1[prev] (the A operand of
// position p + 1's pass) and c = sigmoid((w_h . h[i, p] + w_e . W1[prev]) / T[p]),
// "DSpark 深度解读" §二 设计二; zh_part is this thread's part of w_h . h[i, p].
// Called by the RT threads of a row group.
template <int RW, class Scr>
__device__ __forceinline__ void embed_conf(const LoopArgs &a, int i, int p, int prev,
                                           float zh_part, Scr &S, int wg, int lane, int tg,
                                           int group_bar) {
  constexpr int RT = 32 * RW;
  const int r = a.r;
  if (prev < 0 || prev >= a.V) {
    if (tg == 0) dspark_set_status(DSPARK_ERR_TOKEN);
    prev = 0;
  }
  const uint4 *src = reinterpret_cast<const uint4 *>(a.W1 + (size_t)prev * r);
  const uint4 *we = reinterpret_cast<const uint4 *>(a.w_e);
  uint4 *dst = reinterpret_cast<uint4 *>(a.E + (size_t)i * r);
  float ze = 0.f;
  for (int q = tg; q < r / 8; q += RT) {
    const uint4 e = __ldg(src + q);
    dst[q] = e;
    ze = dot8_bf16(e, __ldg(we + q), ze);
  }
  float zh = warp_sum(zh_part);
  ze = warp_sum(ze);
  if (RW > 1) {
    if (lane == 0) { S.m[wg] = zh; S.dot[wg] = ze; }
    named_bar(group_bar, RT);
    zh = 0.f;
    ze = 0.f;
#pragma unroll
    for (int w = 0; w < RW; ++w) { zh += S.m[w]; ze += S.dot[w]; }
  }
  if (tg == 0) a.conf[(size_t)i * a.gamma + p] = 1.f / (1.f + expf(-(zh + ze) / a.T[p]));
}

// Row phase of step k for one group of RW epilogue warps (group g of the CTA,
// `groups` groups in the grid).  See the file comment.
template <int MODE, int RW, int EPI_WARPS>
__device__ void row_phase(const LoopArgs &a, int k, Scratch<MODE, RW> &S, int g, int wg, int lane,
                          int groups) {
  constexpr int RT = 32 * RW;
  const int tg = wg * 32 + lane;
  auto group_sync = [&]() {
    if (RW == 1) __syncwarp();
    else named_bar(2 + g, RT);
  };
  const int gamma = a.gamma, V = a.V, r = a.r;
  for (int i = blockIdx.x * (EPI_WARPS / RW) + g; i < a.R; i += groups) {
    // w_h . h for c_{k+1}, taken during this step's tile phase
    const float zh_part = (k < gamma && tg == 0) ? __ldcg(a.zh + (size_t)i * gamma + k) : 0.f;
    // combine the row's partials
    float m = -INFINITY, s = 0.f, best = -INFINITY, bs = 0.f;
    int idx = 0x7fffffff;
    const RowPartial *pr = a.part + (size_t)i * a.n_slots;
    for (int t0 = 0; t0 < a.n_slots; t0 += 4 * RT) {
      RowPartial p[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = t0 + u * RT + tg;
        if (t < a.n_slots) {
          const float4 v = __ldcg(reinterpret_cast<const float4 *>(pr + t));
          p[u].m = v.x;
          p[u].sum = v.y;
          p[u].best = v.z;
          p[u].idx = __float_as_int(v.w);
        } else {
          p[u].m = -INFINITY; p[u].sum = 0.f; p[u].best = -INFINITY; p[u].idx = 0x7fffffff;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        lse_merge(m, s, p[u].m, p[u].sum);
        if (better(p[u].best, p[u].idx, best, idx)) { best = p[u].best; idx = p[u].idx; }
      }
    }
    warp_merge(m, s, best, idx, bs);
    if (RW > 1) {
      if (lane == 0) { S.m[wg] = m; S.s[wg] = s; S.b[wg] = best; S.i[wg] = idx; }
      group_sync();
      m = -INFINITY; s = 0.f; best = -INFINITY; idx = 0x7fffffff;
#pragma unroll
      for (int w = 0; w < RW; ++w) {
        lse_merge(m, s, S.m[w], S.s[w]);
        if (better(S.b[w], S.i[w], best, idx)) { best = S.b[w]; idx = S.i[w]; }
      }
    }
    const size_t o = (size_t)i * gamma + k - 1;
    int tok;
    if (MODE == MODE_SAMPLE) {
      const float lse = m + logf(s);
      int b = idx;
      if (b < 0 || b >= (V + GUMBEL_BLOCK - 1) / GUMBEL_BLOCK) {  // no finite block score
        if (tg == 0) dspark_set_status(DSPARK_ERR_TOKEN);
        b = 0;
      }
      if (tg == 0) {  // the block's W2t rows (contiguous) into L2 in one request
        const int nv = V - b * GUMBEL_BLOCK < GUMBEL_BLOCK ? V - b * GUMBEL_BLOCK : GUMBEL_BLOCK;
        bulk_prefetch_l2(a.W2t + (size_t)b * GUMBEL_BLOCK * r, (uint32_t)(nv * r) * 2u);
      }
      // warp 0 loads the block's base logits and draws its Gumbels while the
      // group's first W2t words are on their way
      const int v_lo = b * GUMBEL_BLOCK + lane, v_hi = v_lo + 32;
      float base_lo = 0.f, base_hi = 0.f;
      if (wg == 0) {
        const bf16 *base_row = a.base + o * V;
        if (v_lo < V) base_lo = __bfloat162float(__ldg(base_row + v_lo));
        if (v_hi < V) base_hi = __bfloat162float(__ldg(base_row + v_hi));
      }
      BlockGumbels gum = {{0.f, 0.f, 0.f, 0.f}};
      rebuild_bias<RW>(a.E + (size_t)i * r, a.W2t, b, V, r, S.score, wg, lane, [&]() {
        if (wg == 0) gum = block_gumbels(b, a.seed, (uint32_t)k, (uint32_t)i, RNG_DRAFT);
      });
      group_sync();
      if (wg == 0) {
        // the block's logits over tau: (Markov bias + base logit) / tau
        S.score[lane] = v_lo < V ? (S.score[lane] + base_lo) * a.inv_tau : -INFINITY;
        S.score[lane + 32] = v_hi < V ? (S.score[lane + 32] + base_hi) * a.inv_tau : -INFINITY;
        __syncwarp();
        int t = block_pick(S.score, b, V, gum);
        if (t < 0) {
          if (lane == 0) dspark_set_status(DSPARK_ERR_TOKEN);
          t = b * GUMBEL_BLOCK;
        }
        if (lane == 0) {
          a.tokens[o] = t;
          if (a.lse_out) a.lse_out[o] = lse;
          if (a.logp_out) a.logp_out[o] = S.score[t - b * GUMBEL_BLOCK] - lse;
          S.tok = t;
        }
      }
      group_sync();
      tok = S.tok;
    } else {
      tok = idx;
      if (tg == 0) {
        a.tokens[o] = tok;
        if (a.lse_out) a.lse_out[o] = 0.f;
        if (a.logp_out) a.logp_out[o] = 0.f;
      }
    }
    // E_{k+1}[i] = W1[x_k] and c_{k+1}
    if (k < gamma) {
      if (RW > 1) group_sync();  // S.m is read above by every thread of the group
      embed_conf<RW>(a, i, k, tok, zh_part, S, wg, lane, tg, 2 + g);
    }
    group_sync();  // S is reused by the group's next row
  }
}

// Registers are split over the SM's four quadrants (16384 each): 18 warps
// (sampling) leave 96 per thread, 10 warps (greedy) 168.
// Before step 1: E[i] = W1[anchor_i] and c_1 for the group's requests.
template <int RW, int EPI_WARPS, class Scr>
__device__ void prologue_rows(const LoopArgs &a, Scr &S, int g, int wg, int lane, int groups) {
  const int tg = wg * 32 + lane;
  for (int i = blockIdx.x * (EPI_WARPS / RW) + g; i < a.R; i += groups) {
    embed_conf<RW>(a, i, 0, a.anchor[i], hidden_dot_part<RW>(a, i, 0, tg), S, wg, lane, tg,
                   2 + g);
    if (RW > 1) named_bar(2 + g, 32 * RW);
    else __syncwarp();
  }
}

// Shared-memory geometry of a loop kernel: the A region (ring stages, or the
// resident E), the W2t stages, then the barriers and the row groups' scratch.
template <int MODE, int RW, int EKB>
struct LoopSmem {
  using G = gemm::Geo<LoopCfg<MODE>::BN>;
  static constexpr int NSTAGE = EKB ? eres_stages<MODE, RW, EKB>() : G::STAGES;
  static constexpr size_t A_REGION = (size_t)(EKB ? EKB : NSTAGE) * A_BYTES;
  static constexpr size_t B_REGION = (size_t)NSTAGE * G::B_BYTES;
  static constexpr size_t CTL = A_REGION + B_REGION;
  static constexpr size_t BYTES = 1024 + CTL + 512 +
                                  sizeof(Scratch<MODE, RW>) * (LoopCfg<MODE>::EPI_WARPS / RW);
};

template <int MODE, int RW, int EKB>
__global__ void __launch_bounds__(64 + 32 * LoopCfg<MODE>::EPI_WARPS, 1) markov_loop_kernel(const __grid_constant__ CUtensorMap tma_a,
                       const __grid_constant__ CUtensorMap tma_b, const __grid_constant__ LoopArgs a) {
  constexpr bool ERES = EKB > 0;  // E resident for the step
  constexpr int EPI_WARPS = LoopCfg<MODE>::EPI_WARPS;
  constexpr int EPI_THREADS = 32 * EPI_WARPS;
  constexpr int CG = EPI_WARPS / 4;  // column groups: threads per row in a tile
  constexpr int SLICE = LoopCfg<MODE>::SLICE;
  constexpr int RG = EPI_WARPS / RW;  // row groups per CTA
  using G = gemm::Geo<LoopCfg<MODE>::BN>;
  using L = LoopSmem<MODE, RW, EKB>;
  constexpr int BN = G::BN, STAGES = L::NSTAGE, B_BYTES = G::B_BYTES;
  constexpr int STAGE_BYTES = G::STAGE_BYTES;
  constexpr uint32_t TMEM_COLS = G::TMEM_COLS;
  static_assert(EPI_WARPS % RW == 0, "row groups split the epilogue warps");
  static_assert(sizeof(LoopCtl<STAGES>) <= 512, "barrier block");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sbase = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = sbase;  // ring: stage s at s * A_BYTES; resident E: k block kb at kb * A_BYTES
  uint8_t *sB = sbase + L::A_REGION;
  LoopCtl<STAGES> *ctl = reinterpret_cast<LoopCtl<STAGES> *>(sbase + L::CTL);
  using Scr = Scratch<MODE, RW>;
  Scr *scr = reinterpret_cast<Scr *>(sbase + L::CTL + 512);
  volatile int *abort = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&ctl->full[s], 1);
      tc::mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ctl->tfull[b], 1);
      tc::mbar_init(&ctl->tempty[b], EPI_WARPS);
    }
    tc::mbar_init(&ctl->go, 1);
    tc::mbar_init(&ctl->efull, 1);
    tc::mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_desc(&tma_a);
    tc::tma_prefetch_desc(&tma_b);
  }
  if (warp == 1) tc::tmem_alloc(&ctl->tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;

  const int M = a.R, N = a.V, gamma = a.gamma;
  const int num_m = (M + BM - 1) / BM, num_n = (N + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int k_iters = a.r / BK;
  const int first = blockIdx.x, stride = gridDim.x;
  auto coords = [&](int t, int &m_blk, int &n_blk) {
    m_blk = t % num_m;
    n_blk = t / num_m;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer ----
      const uint64_t pol_a = tc::policy_evict_last();    // E: re-read by every N tile
      const uint64_t pol_b = tc::policy_evict_normal();  // W2t: re-read by the other M blocks
      int stage = 0;
      uint32_t phase = 0;
      int issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = -1;
      int e_issued = -1;  // resident E: parity of the last E load armed
      constexpr uint32_t FULL_BYTES = ERES ? B_BYTES : STAGE_BYTES;
      bool ok = true;
      for (int k = 1; ok && k <= gamma; ++k) {
        bool first_tile = true;
        for (int tile = first; ok && tile < num_tiles; tile += stride) {
          int m_blk, n_blk;
          coords(tile, m_blk, n_blk);
          int kb = 0;
          if (first_tile) {
            // W2t halves of the first stages now; their E halves once the rows
            // of E_k are written (prologue or row phase of step k-1) and the
            // grid barrier has passed
            const int nd = k_iters < STAGES ? k_iters : STAGES;
            const int s0 = stage;
            for (; kb < nd; ++kb) {
              if (!tc::mbar_wait(&ctl->empty[stage], phase ^ 1, abort)) { ok = false; break; }
              tc::mbar_expect_tx(&ctl->full[stage], FULL_BYTES);
              tc::tma_load_2d(sB + stage * B_BYTES, &tma_b, kb * BK, n_blk * BN, &ctl->full[stage],
                              pol_b);
              issued[stage] = (int)phase;
              if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            // on a timeout the E halves are still issued (valid memory), so
            // every armed stage completes before the CTA exits
            if (ok && !tc::mbar_wait(&ctl->go, (uint32_t)((k - 1) & 1), abort)) ok = false;
            fence_proxy_async_global();
            if (ERES) {
              // the step's E tile, resident for all of the step's tiles (the
              // previous step's MMAs have all completed: the grid barrier
              // behind go came after every accumulator was consumed)
              if (ok) {
                tc::mbar_expect_tx(&ctl->efull, (uint32_t)(k_iters * A_BYTES));
                for (int j = 0; j < k_iters; ++j)
                  tc::tma_load_2d(sA + j * A_BYTES, &tma_a, j * BK, m_blk * BM, &ctl->efull,
                                  pol_a);
                e_issued = (k - 1) & 1;
              }
            } else {
              for (int j = 0, s = s0; j < kb; ++j) {
                tc::tma_load_2d(sA + s * A_BYTES, &tma_a, j * BK, m_blk * BM, &ctl->full[s],
                                pol_a);
                if (++s == STAGES) s = 0;
              }
            }
            if (!ok) break;
          }
          first_tile = false;
          for (; kb < k_iters; ++kb) {
            if (!tc::mbar_wait(&ctl->empty[stage], phase ^ 1, abort)) { ok = false; break; }
            tc::mbar_expect_tx(&ctl->full[stage], FULL_BYTES);
            if (!ERES)
              tc::tma_load_2d(sA + stage * A_BYTES, &tma_a, kb * BK, m_blk * BM,
                              &ctl->full[stage], pol_a);
            tc::tma_load_2d(sB + stage * B_BYTES, &tma_b, kb * BK, n_blk * BN, &ctl->full[stage],
                            pol_b);
            issued[stage] = (int)phase;
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
          }
        }
      }
      // drain: every copy this thread issued has landed before the CTA exits
      volatile int never = 0;
      for (int s = 0; s < STAGES; ++s)
        if (issued[s] >= 0) tc::mbar_wait(&ctl->full[s], (uint32_t)issued[s], &never);
      if (ERES && e_issued >= 0) tc::mbar_wait(&ctl->efull, (uint32_t)e_issued, &never);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------- MMA issuer -----
      const uint32_t idesc = tc::idesc_bf16(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int k = 1; ok && k <= gamma; ++k) {
        if (ERES) {  // the step's resident E tile
          if (!tc::mbar_wait(&ctl->efull, (uint32_t)((k - 1) & 1), abort)) { ok = false; break; }
          tc::fence_after_sync();
        }
        for (int tile = first; ok && tile < num_tiles; tile += stride) {
          if (!tc::mbar_wait(&ctl->tempty[acc], acc_phase ^ 1, abort)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
          for (int kb = 0; kb < k_iters; ++kb) {
            if (!tc::mbar_wait(&ctl->full[stage], phase, abort)) { ok = false; break; }
            tc::fence_after_sync();
            const uint64_t a_desc =
                tc::smem_desc_sw128(sA + (ERES ? kb : stage) * A_BYTES);
            const uint64_t b_desc = tc::smem_desc_sw128(sB + stage * B_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc::umma_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc,
                            (kb | kk) != 0 ? 1u : 0u);
            tc::umma_commit(&ctl->empty[stage]);
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          tc::umma_commit(&ctl->tfull[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
      }
      tc::umma_commit(&ctl->drain);
      volatile int never = 0;
      tc::mbar_wait(&ctl->drain, 0, &never);
    }
    __syncwarp();
  } else {
    // ----------------------------------------- epilogue and row phase ---
    const int ew = warp - 2;
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const int cg = ew >> 2;
    const int c0 = cg * SLICE;
    const int g = ew / RW, wg = ew % RW;
    const int groups = (int)gridDim.x * RG;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint4 buf[SLICE / 8];
    // ---- prologue: E_1 and c_1, then a grid barrier before any E_1 load
    prologue_rows<RW, EPI_WARPS>(a, scr[g], g, wg, lane, groups);
    fence_proxy_async_global();
    named_bar(1, EPI_THREADS);
    if (ew == 0 && lane == 0) {
      if (!grid_barrier(a.sync, gridDim.x)) {
        *abort = 1;
        atomicExch(&a.sync->abort, 1);
      }
      tc::mbar_arrive(&ctl->go);
    }
    for (int k = 1; k <= gamma; ++k) {
      if (first < num_tiles && k == 1) {
        // base words of the first tile of step 1 (later steps load theirs
        // during the previous step's last tile)
        int m_blk, n_blk;
        coords(first, m_blk, n_blk);
        const bf16 *brow = m_blk * BM + row < M
                               ? a.base + ((size_t)(m_blk * BM + row) * gamma + k - 1) * N
                               : nullptr;
        const int n = n_blk * BN + c0;
#pragma unroll
        for (int q = 0; q < SLICE / 8; ++q)
          buf[q] = (brow && n + q * 8 + 8 <= N)
                       ? __ldg(reinterpret_cast<const uint4 *>(brow + n + q * 8))
                       : make_uint4(0, 0, 0, 0);
      }
      // w_h . h at position k (for c_{k+1}): off the row phase's critical path
      if (k < gamma) hidden_dots(a, k, (int)blockIdx.x * EPI_WARPS + ew, (int)gridDim.x * EPI_WARPS, lane);
      Run run;
      run.reset();
      int run_n = -1;
      int ok = 1;
      for (int tile = first; tile < num_tiles; tile += stride) {
        int m_blk, n_blk;
        coords(tile, m_blk, n_blk);
        if (run_n < 0) run_n = n_blk;
        // the next tile this thread processes: later in this step, or the
        // first one of the next step (loaded before the row phase: measured
        // 294 against 303 us per 5-step sampling loop at R = 256)
        int nm = -1, nn = -1, nk = k;
        const bool more = tile + stride < num_tiles;
        if (more) coords(tile + stride, nm, nn);
        else if (k < gamma) { coords(first, nm, nn); nk = k + 1; }
        const bf16 *nrow = (nm >= 0 && nm * BM + row < M)
                               ? a.base + ((size_t)(nm * BM + row) * gamma + nk - 1) * N
                               : nullptr;
        {
          // the base slice two tiles ahead into L2: the register loads of the
          // next tile then find it there (R = 256, V = 129280: the sampling
          // pass 46.6 -> 38.7 us, greedy 43.4 -> 38.8 us per step)
          // this CTA's tile j + 2 (j = its index in the step), or the next
          // step's tile j + 2 - n when the step has only n of them
          const int n_mine = (num_tiles - 1 - first) / stride + 1;
          int j2 = (tile - first) / stride + 2, k2 = k;
          if (j2 >= n_mine) { j2 -= n_mine; k2 = k + 1; }
          const int t2 = first + j2 * stride;
          if (k2 <= gamma && t2 < num_tiles) {
            int m2, n2;
            coords(t2, m2, n2);
            const int nc = n2 * BN + c0;
            if (m2 * BM + row < M && nc < N)
              bulk_prefetch_l2(a.base + ((size_t)(m2 * BM + row) * gamma + k2 - 1) * N + nc,
                               (uint32_t)(N - nc < SLICE ? N - nc : SLICE) * 2u);
          }
        }
        if (lane == 0) ok = tc::mbar_wait(&ctl->tfull[acc], acc_phase, abort) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
        const int i = m_blk * BM + row;
        tile_slice<MODE>(a, k, i, i < M, n_blk * BN, c0, taddr, nrow, nn * BN + c0, buf, run);
        tc::fence_before_sync();
        __syncwarp();  // every lane's TMEM reads are done before the warp's single arrival
        if (lane == 0) tc::mbar_arrive(&ctl->tempty[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
        // the run of tiles on this row block ends: one partial per (row, run)
        if (!more || nm != m_blk) {
          if (i < M) {
            const float m_out = MODE == MODE_SAMPLE && run.m2 > -INFINITY
                                    ? run.m2 * 0.6931471805599453f
                                    : -INFINITY;
            *reinterpret_cast<float4 *>(a.part + (size_t)i * a.n_slots + run_n * CG + cg) =
                make_float4(m_out, run.s, run.best, __int_as_float(run.idx));
          }
          run.reset();
          run_n = -1;
        }
      }
      // ---- grid barrier: every partial of step k is written.  One thread
      // decides whether to go on and every epilogue thread gets that decision
      // (a flag raised meanwhile by another role is seen by the next wait), so
      // all of them meet the same named barriers.
      named_bar(1, EPI_THREADS);
      bool give_up = false;
      if (ew == 0 && lane == 0) {
        if (*abort || !grid_barrier(a.sync, (unsigned)(2 * k) * gridDim.x)) {
          *abort = 1;
          atomicExch(&a.sync->abort, 1);
          give_up = true;
        }
      }
      if (named_bar_or(BAR_STOP, EPI_THREADS, give_up)) break;
      row_phase<MODE, RW, EPI_WARPS>(a, k, scr[g], g, wg, lane, groups);
      if (k < gamma) {
        // ---- grid barrier: every E row of step k+1 is written; the producer may load them
        fence_proxy_async_global();
        named_bar(1, EPI_THREADS);
        if (ew == 0 && lane == 0) {
          if (!grid_barrier(a.sync, (unsigned)(2 * k + 1) * gridDim.x)) {
            *abort = 1;
            atomicExch(&a.sync->abort, 1);
          }
          tc::mbar_arrive(&ctl->go);
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort && threadIdx.x == 0) {
    atomicExch(&a.sync->abort, 1);
    dspark_set_status(DSPARK_ERR_TIMEOUT);
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int MODE, int RW, int EKB>
constexpr size_t loop_smem_bytes() {
  return LoopSmem<MODE, RW, EKB>::BYTES;
}

// Grid of the loop: at most one CTA per SM, a multiple of the M-block count
// when there are at least as many CTAs as M blocks (each CTA then stays on one
// row block and writes one partial per row and column group per step).
struct LoopGrid {
  int grid, n_slots;
};
template <int MODE>
inline LoopGrid loop_grid(int R, int V, int sms) {
  constexpr int BN = LoopCfg<MODE>::BN, CG = LoopCfg<MODE>::EPI_WARPS / 4;
  const int num_m = (R + BM - 1) / BM, num_n = (V + BN - 1) / BN;
  const int tiles = num_m * num_n;
  LoopGrid lg;
  lg.grid = tiles < sms ? tiles : sms;
  if (lg.grid >= num_m) {
    lg.grid = lg.grid / num_m * num_m;
    lg.n_slots = lg.grid / num_m * CG;
  } else {
    lg.n_slots = num_n * CG;
  }
  return lg;
}
// Partials per row the workspace must hold for any grid and mode.
inline size_t loop_slots_max(int V) {
  const size_t g = (size_t)(V + LoopCfg<MODE_GREEDY>::BN - 1) / LoopCfg<MODE_GREEDY>::BN *
                   LoopCfg<MODE_GREEDY>::CG;
  const size_t t = (size_t)(V + LoopCfg<MODE_SAMPLE>::BN - 1) / LoopCfg<MODE_SAMPLE>::BN *
                   LoopCfg<MODE_SAMPLE>::CG;
  return g > t ? g : t;
}

// EKB: 0 (E streamed with W2t) or the k blocks of E kept resident (4 or 8,
// r <= 64 EKB).
template <int MODE, int RW, int EKB = 0>
int launch_loop(const LoopArgs &args, int grid, cudaStream_t stream) {
  auto kernel = markov_loop_kernel<MODE, RW, EKB>;
  constexpr size_t smem = loop_smem_bytes<MODE, RW, EKB>();
  static_assert(smem <= gemm::SMEM_LIMIT, "shared memory of the loop kernel");
  if (EKB && args.r > EKB * BK) return DSPARK_ERR_ARG;  // E must fit its resident room
  CUtensorMap ta, tb;
  if (dspark_make_tmap_bf16(&ta, args.E, (uint64_t)args.R, (uint64_t)args.r, BM) != 0)
    return DSPARK_ERR_CUDA;
  if (dspark_make_tmap_bf16(&tb, args.W2t, (uint64_t)args.V, (uint64_t)args.r,
                            LoopCfg<MODE>::BN) != 0)
    return DSPARK_ERR_CUDA;
  static DsparkPerDevice attr;
  if (dspark_per_device(attr, [&] {
        const cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess && getenv("DSPARK_DEBUG"))
          fprintf(stderr, "dspark: markov loop smem attribute: %s\n", cudaGetErrorString(e));
        return e == cudaSuccess ? 1 : -1;
      }) < 0)
    return DSPARK_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the grid barriers need it
  at[0].val.cooperative = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(64 + 32 * LoopCfg<MODE>::EPI_WARPS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, ta, tb, args);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // not sticky: later launches must not see it
    if (getenv("DSPARK_DEBUG")) {
      int nb = -1, nb0 = -1;
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, (int)cfg.blockDim.x, smem);
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb0, kernel, (int)cfg.blockDim.x, 0);
      cudaFuncAttributes fa;
      cudaFuncGetAttributes(&fa, kernel);
      fprintf(stderr,
              "dspark: markov loop launch (grid %d, %u threads, %zu B smem, %d CTAs/SM, %d without "
              "smem; regs %d, max threads %d, static smem %zu, max dyn smem %d, local %zu): %s\n",
              grid, cfg.blockDim.x, smem, nb, nb0, fa.numRegs, fa.maxThreadsPerBlock,
              fa.sharedSizeBytes, fa.maxDynamicSharedSizeBytes, fa.localSizeBytes,
              cudaGetErrorString(e));
    }
    return DSPARK_ERR_CUDA;
  }
  dspark_count_launches(1);
  return DSPARK_OK;
}

}  // namespace mloop
