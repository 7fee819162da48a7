// markov.cu — a2-a4: the gamma-step sequential (Markov) head with the
// confidence head.
//
// "DSpark 深度解读" §二 设计一: x_k is sampled from base logits plus the low-rank
// transition bias W1[x_{k-1}] W2; §二 设计二: c_k = sigmoid(w^T [h_k; W1[x_{k-1}]])
// calibrated per position by a temperature T_k.  "DSpark整体架构": the anchor is
// the first prediction position, so x_0 = anchor.
//
// Before the loop: zh = w_h . h for every row, and step 1's gather E = W1[x_0]
// with the confidence c_1.  Per step k: one vocabulary pass (bias + base logits
// on the tensor cores, logits stay on chip; per 64-id block its log-sum-exp and
// block score), then reduce_prep (combine the blocks into lse_k and the winning
// block, draw x_k inside it, logp_k, and gather E = W1[x_k] with c_{k+1} for
// the next step).
#include <mutex>

#include "logits_tile.cuh"

DSPARK_DECLARE_STATUS(s_status_markov)

#include "markov_loop.cuh"

namespace {

// zh[m] = w_h . h[m] for every (request, position) row m; one CTA of 128
// threads per row, each thread a strided quarter of the row's 16-byte words.
// Block 0 also zeroes the loop's grid-barrier words (when given).
__global__ void __launch_bounds__(128) conf_hidden(const bf16 *__restrict__ h,
                                                   const bf16 *__restrict__ w_conf,
                                                   float *__restrict__ zh, int d,
                                                   mloop::LoopSync *sync) {
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (sync && row == 0 && tid == 0) *sync = mloop::LoopSync{0u, 0, {0u, 0u}};
  const uint4 *hr = reinterpret_cast<const uint4 *>(h + (size_t)row * d);
  const uint4 *wr = reinterpret_cast<const uint4 *>(w_conf);
  const int n8 = d / 8;
  float acc[2] = {0.f, 0.f};
  int c = tid;
  for (; c + 128 < n8; c += 256) {
    const uint4 a0 = __ldg(hr + c), a1 = __ldg(hr + c + 128);
    acc[0] = dot8_bf16(a0, __ldg(wr + c), acc[0]);
    acc[1] = dot8_bf16(a1, __ldg(wr + c + 128), acc[1]);
  }
  for (; c < n8; c += 128) acc[0] = dot8_bf16(__ldg(hr + c), __ldg(wr + c), acc[0]);
  const float t = warp_sum(acc[0] + acc[1]);
  __shared__ float part[4];
  if (lane == 0) part[warp] = t;
  __syncthreads();
  if (tid == 0) zh[row] = (part[0] + part[1]) + (part[2] + part[3]);
}

// Step k: the embedding W1[x_{k-1}] into row i of e_next (row stride e_ld: the
// Markov head's E, or the embedding columns of the RNN head's recurrent input),
// c_k = sigmoid((zh + w_e . W1[x_{k-1}]) / T_k); one warp per request.
__global__ void step_prep(const int32_t *__restrict__ anchor, const int32_t *__restrict__ tokens,
                          const bf16 *__restrict__ W1, const bf16 *__restrict__ w_e,
                          const float *__restrict__ zh, const float *__restrict__ T,
                          bf16 *__restrict__ e_next, int e_ld, float *__restrict__ conf, int R,
                          int gamma, int V, int r, int k) {
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (i >= R) return;
  int prev = (k == 1) ? anchor[i] : tokens[(size_t)i * gamma + k - 2];
  if (prev < 0 || prev >= V) {
    if (lane == 0) dspark_set_status(DSPARK_ERR_TOKEN);
    prev = 0;
  }
  const uint4 *src = reinterpret_cast<const uint4 *>(W1 + (size_t)prev * r);
  uint4 *dst = reinterpret_cast<uint4 *>(e_next + (size_t)i * e_ld);
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

// Combine the vocabulary-slice partials of request i into x_k, lse_k, logp_k,
// then (k < gamma) prepare step k+1: E[i] = W1[x_k] and the confidence c_{k+1}.
// One CTA of RP_THREADS threads per request.  Greedy: the partials carry the
// argmax.  Sampling: they carry block scores; the best block's 64 logits are
// rebuilt (base logit + W1[x_{k-1}] . W2t[v], E still holds W1[x_{k-1}] here;
// for the fused step, no base and E row [h_k; W1[x_{k-1}]] of length e_k and
// stride e_row_ld against W2t = [W_lm; W2t]), x_k is drawn among them and
// log p_d(x_k) = l_k[x_k] / tau - lse_k.
constexpr int RP_THREADS = 256;

template <int MODE>
__global__ void __launch_bounds__(RP_THREADS) reduce_prep(
    const RowPartial *__restrict__ part, int n_parts, int gamma, int V, int r, int k,
    int32_t *__restrict__ tokens, float *__restrict__ lse_out, float *__restrict__ logp_out,
    const bf16 *__restrict__ W1, const bf16 *__restrict__ w_e, const float *__restrict__ zh,
    const float *__restrict__ T, const bf16 *E, int e_row_ld, int e_k, bf16 *e_next,
    int e_ld,  // E and e_next may share a buffer
    float *__restrict__ conf, const bf16 *__restrict__ base, const bf16 *__restrict__ W2t,
    float inv_tau, uint64_t seed) {
  const int i = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();  // the vocabulary pass of step k has completed
  float m = -INFINITY, s = 0.f, best = -INFINITY, bs = 0.f;
  int idx = 0x7fffffff;
  const RowPartial *pr = part + (size_t)i * n_parts;
  for (int t0 = 0; t0 < n_parts; t0 += 8 * RP_THREADS) {  // eight loads in flight
    RowPartial p[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = t0 + u * RP_THREADS + tid;
      if (t < n_parts) p[u] = pr[t];
      else { p[u].m = -INFINITY; p[u].sum = 0.f; p[u].best = -INFINITY; p[u].idx = 0x7fffffff; }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      lse_merge(m, s, p[u].m, p[u].sum);
      if (better(p[u].best, p[u].idx, best, idx)) { best = p[u].best; idx = p[u].idx; }
    }
  }
  warp_merge(m, s, best, idx, bs);
  constexpr int NW = RP_THREADS / 32;
  __shared__ float sm[NW], ss[NW], sb[NW], sdot[NW], s_lse;
  __shared__ float s_logit[GUMBEL_BLOCK], s_score[GUMBEL_BLOCK];
  __shared__ int si[NW], s_tok;
  if (lane == 0) { sm[warp] = m; ss[warp] = s; sb[warp] = best; si[warp] = idx; }
  __syncthreads();
  if (warp == 0) {
    m = lane < NW ? sm[lane] : -INFINITY;
    s = lane < NW ? ss[lane] : 0.f;
    best = lane < NW ? sb[lane] : -INFINITY;
    idx = lane < NW ? si[lane] : 0x7fffffff;
    warp_merge(m, s, best, idx, bs);
    if (lane == 0) {
      s_lse = MODE == MODE_SAMPLE ? m + logf(s) : 0.f;
      s_tok = idx;  // greedy: the token; sampling: the winning block
    }
  }
  __syncthreads();
  const size_t o = (size_t)i * gamma + k - 1;
  if (MODE == MODE_SAMPLE) {
    int b = s_tok;
    if (b < 0 || b >= (V + GUMBEL_BLOCK - 1) / GUMBEL_BLOCK) {  // no finite block score (non-finite logits)
      if (tid == 0) dspark_set_status(DSPARK_ERR_TOKEN);
      b = 0;
    }
    block_logits<RP_THREADS>(base ? base + o * V : nullptr, E + (size_t)i * e_row_ld, W2t, b, V,
                             e_k, s_logit);
    if (warp == 0) {
      for (int j = lane; j < GUMBEL_BLOCK; j += 32) s_score[j] = s_logit[j] * inv_tau;
      __syncwarp();
      int tok = block_pick(s_score, b, V, seed, (uint32_t)k, (uint32_t)i, RNG_DRAFT);
      if (tok < 0) {
        if (lane == 0) dspark_set_status(DSPARK_ERR_TOKEN);
        tok = b * GUMBEL_BLOCK;
      }
      if (lane == 0) {
        tokens[o] = tok;
        if (lse_out) lse_out[o] = s_lse;
        if (logp_out) logp_out[o] = s_logit[tok - b * GUMBEL_BLOCK] * inv_tau - s_lse;
        s_tok = tok;
      }
    }
    __syncthreads();  // s_tok is read and E is rewritten below
  } else if (tid == 0) {
    tokens[o] = s_tok;
    if (lse_out) lse_out[o] = 0.f;
    if (logp_out) logp_out[o] = 0.f;
  }
  if (k >= gamma) return;
  int prev = s_tok;
  if (prev < 0 || prev >= V) {
    if (tid == 0) dspark_set_status(DSPARK_ERR_TOKEN);
    prev = 0;
  }
  const uint4 *src = reinterpret_cast<const uint4 *>(W1 + (size_t)prev * r);
  uint4 *dst = reinterpret_cast<uint4 *>(e_next + (size_t)i * e_ld);
  const uint4 *wr = reinterpret_cast<const uint4 *>(w_e);
  float acc = 0.f;
  for (int c = tid; c < r / 8; c += RP_THREADS) {
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
  if (lane == 0) sdot[warp] = acc;
  __syncthreads();
  if (tid == 0) {
    const size_t o = (size_t)i * gamma + k;  // position k + 1
    float zs = zh[o];
    for (int w = 0; w < NW; ++w) zs += sdot[w];
    const float z = zs;
    conf[o] = 1.f / (1.f + expf(-z / T[k]));
  }
}

// Row blocks (of 128 requests) from which the loop keeps E resident; it does at
// a single row block too (sampling, and greedy with r <= 256).
constexpr int ERES_MIN_ROW_BLOCKS = 4;

struct MarkovWs {
  float *zh;
  bf16 *E;
  RowPartial *part;
  mloop::LoopSync *sync;
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
  const size_t slots = mloop::loop_slots_max(d->V) > logits_parts_max(d->V)
                          ? mloop::loop_slots_max(d->V)
                          : logits_parts_max(d->V);
  off = dspark_align_up(off + sizeof(RowPartial) * (size_t)d->R * slots, 256);
  w.sync = (mloop::LoopSync *)(base + off);
  off = dspark_align_up(off + sizeof(mloop::LoopSync), 256);
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
  if (((uintptr_t)W2t | (uintptr_t)W1 | (uintptr_t)h | (uintptr_t)base_logits) & 15)
    return DSPARK_ERR_ARG;  // TMA and 16-byte vector loads
  MarkovWs ws = markov_layout(dims, (char *)workspace);
  if (!workspace || workspace_bytes < ws.bytes || ((uintptr_t)workspace & 255))
    return DSPARK_ERR_WORKSPACE;
  const int R = dims->R, G = dims->gamma, V = dims->V, r = dims->r, d = dims->d;
  if (cudaMemsetAsync(ws.sync, 0, sizeof(mloop::LoopSync), stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  const float inv_tau = tau > 0.f ? 1.f / tau : 1.f;
  // all gamma steps, with the confidence head, in one cooperative launch
  mloop::LoopArgs la{(const bf16 *)base_logits, (const bf16 *)W1, (const bf16 *)W2t,
                     (const bf16 *)h, (const bf16 *)w_conf, (const bf16 *)w_conf + d, anchor,
                     ws.zh, T, ws.E, tokens, conf, lse_d, logp_d, ws.part, ws.sync, R, V, r, d, G, 0,
                     inv_tau, seed};
  const int sms = dspark_sm_count();
  if (tau > 0.f) {
    constexpr int EW = mloop::LoopCfg<MODE_SAMPLE>::EPI_WARPS;
    const mloop::LoopGrid lg = mloop::loop_grid<MODE_SAMPLE>(R, V, sms);
    la.n_slots = lg.n_slots;
    const int num_m = (R + gemm::BM - 1) / gemm::BM;
    const bool eres = lg.grid >= num_m && lg.grid % num_m == 0 && r <= 8 * gemm::BK;
    if (eres && num_m >= ERES_MIN_ROW_BLOCKS && R > lg.grid * (EW / 4))
      return mloop::launch_loop<MODE_SAMPLE, 2, 8>(la, lg.grid, stream);
    // resident E at one row block as well: every CTA would otherwise re-read
    // the same E tile from L2 for each of its tiles (R = 64, V = 151936, four
    // W2t stages: 273-275 against 284-286 us for 8 steps; at two row blocks,
    // R = 256, it measured 276-279 against 274-275 us, so it stays off there).
    // With r <= 256 E takes half the room, and six W2t stages fit.
    if (eres && num_m == 1)
      return r <= 4 * gemm::BK ? mloop::launch_loop<MODE_SAMPLE, EW, 4>(la, lg.grid, stream)
                               : mloop::launch_loop<MODE_SAMPLE, EW, 8>(la, lg.grid, stream);
    // warps per request in the row phase: as many as still cover R in one pass
    if (R <= lg.grid) return mloop::launch_loop<MODE_SAMPLE, EW>(la, lg.grid, stream);
    if (R <= lg.grid * 2) return mloop::launch_loop<MODE_SAMPLE, EW / 2>(la, lg.grid, stream);
    if (R <= lg.grid * (EW / 4)) return mloop::launch_loop<MODE_SAMPLE, 4>(la, lg.grid, stream);
    return mloop::launch_loop<MODE_SAMPLE, 2>(la, lg.grid, stream);
  }
  constexpr int EW = mloop::LoopCfg<MODE_GREEDY>::EPI_WARPS;
  const mloop::LoopGrid lg = mloop::loop_grid<MODE_GREEDY>(R, V, sms);
  la.n_slots = lg.n_slots;
  // resident E for batches of several row blocks: every W2t tile then serves
  // several CTAs from L2, and the tiles' E re-reads were a third of the pass's
  // L2 traffic (each CTA stays on one row block, and E fits up to r = 512)
  // (at four row blocks or more R exceeds two requests per CTA, so the row
  // phase takes one warp per request)
  const int num_m = (R + gemm::BM - 1) / gemm::BM;
  const bool eres = lg.grid >= num_m && lg.grid % num_m == 0 && r <= 8 * gemm::BK;
  if (eres && num_m >= ERES_MIN_ROW_BLOCKS)
    return mloop::launch_loop<MODE_GREEDY, 1, 8>(la, lg.grid, stream);
  // one row block with r <= 256: E (64 KB) resident beside five W2t stages
  if (eres && num_m == 1 && r <= 4 * gemm::BK && R <= lg.grid * (EW / 4))
    return mloop::launch_loop<MODE_GREEDY, 4, 4>(la, lg.grid, stream);
  if (R <= lg.grid * (EW / 4)) return mloop::launch_loop<MODE_GREEDY, 4>(la, lg.grid, stream);
  return mloop::launch_loop<MODE_GREEDY, 1>(la, lg.grid, stream);
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

// ---------------------------------------------------------------------------
// The RNN head variant.  "DSpark整体架构" (stage two) names a second sequential
// head that keeps a block-internal recurrent state and updates it by a gated
// step over the history, the previous token's embedding and the backbone
// hidden state; the pages give no equations.  Read as:
//   pre_k = W_rec [s_{k-1}; W1[x_{k-1}]] + W_hid h_k        (2r values; s_0 = 0)
//   s_k   = (1 - g) s_{k-1} + g tanh(c),   g = sigmoid(pre_k[0:r]), c = pre_k[r:2r]
//   l_k   = l0_k + s_k W2            (the Markov head's output map, s_k in bf16)
// W_hid h_k is known for every position before the loop: one tensor-core GEMM
// per round.  Per step: the recurrent GEMM [R, 2r] x [2r, 2r] (f32 out),
// rnn_state, then the Markov head's vocabulary pass and reduce_prep with
// E = bf16(s_k); reduce_prep gathers W1[x_k] into the recurrent input U.
// ---------------------------------------------------------------------------
namespace {

// f32 accumulator rows to C [M, N] (N a multiple of 4).
struct EpiStoreF32 {
  float *C;
  int M, N;
  struct State {};
  static constexpr bool kRowAffine = false;
  static constexpr bool kStreamB = false;
  __device__ void prefetch(int, int, int, int, int, State &) const {}
  __device__ void operator()(int m0, int n0, int row, uint32_t taddr, int c0, int c1, int, int,
                             State &) const {
    const int m = m0 + row;
    float *dst = C + (size_t)m * N;
#pragma unroll 1
    for (int c = c0; c < c1; c += 32) {
      uint32_t v[32];
      tc::tmem_ld32(taddr + (uint32_t)c, v);
      tc::tmem_wait_ld();
      if (m < M) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int n = n0 + c + 4 * q;
          if (n + 4 <= N)
            *reinterpret_cast<float4 *>(dst + n) =
                make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                            __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
      }
    }
  }
  __device__ void on_timeout() const { dspark_set_status(DSPARK_ERR_TIMEOUT); }
};

// s_k for every (request, state component): the f32 state, bf16(s_k) as the
// vocabulary pass's A operand E and into the state columns of U.  W_rec U comes
// as `splits` partial sums over K (rows s * m_pad + i of Gk) and W_hid h as
// `psplits` (rows s * pm_pad + i gamma + k - 1 of P), each added in order.
__global__ void rnn_state(const float *__restrict__ Gk, const float *__restrict__ P,
                          float *__restrict__ state, bf16 *__restrict__ E, bf16 *__restrict__ U,
                          int R, int gamma, int r, int k, int splits, int m_pad, int psplits,
                          int pm_pad) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_trigger();
  pdl_wait();  // the recurrent GEMM's partials
  if (t >= R * r) return;
  const int i = t / r, c = t % r;
  float gg = 0.f, gc = 0.f, pg = 0.f, pc = 0.f;
  for (int sp = 0; sp < splits; ++sp) {
    const float *g_row = Gk + ((size_t)sp * m_pad + i) * 2 * r;
    gg += g_row[c];
    gc += g_row[r + c];
  }
  for (int sp = 0; sp < psplits; ++sp) {
    const float *p_row = P + ((size_t)sp * pm_pad + (size_t)i * gamma + k - 1) * 2 * r;
    pg += p_row[c];
    pc += p_row[r + c];
  }
  const float g = 1.f / (1.f + expf(-(gg + pg)));
  const float cand = tanhf(gc + pc);
  const float s = (1.f - g) * state[t] + g * cand;
  state[t] = s;
  const bf16 sb = __float2bfloat16_rn(s);
  E[t] = sb;
  U[(size_t)i * 2 * r + c] = sb;
}

struct RnnWs {
  MarkovWs mk;
  bf16 *U;        // [R, 2r]  [bf16(s_{k-1}) | W1[x_{k-1}]]
  float *state;   // [R, r]
  float *Gk;      // [splits * m_pad, 2r]  W_rec U of the current step, split over K
  int splits, m_pad;
  float *P;       // [psplits * pm_pad, 2r]  W_hid h of every position, split over K
  int psplits, pm_pad;
  size_t bytes;
};

// K slices for W_hid h ([R gamma, d] x [d, 2r] on 128 x 256 tiles): the divisor
// of the 64-deep k blocks, at most 16, that minimises waves x (k blocks per
// slice + 2 for the tile's hand-over) on GB300's 152 SMs.  The split only
// balances the work, so a part with another SM count still gets right results.
int rnn_hidden_splits(int M, int N, int K) {
  const int tiles = ((M + 127) / 128) * ((N + 255) / 256), kb = K / 64, sms = 152;
  int best = 1;
  long best_cost = -1;
  for (int s = 1; s <= 16; ++s) {
    if (kb % s) continue;
    const long cost = (long)((tiles * s + sms - 1) / sms) * (kb / s + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

RnnWs rnn_layout(const dspark_dims *d, char *base) {
  RnnWs w;
  w.mk = markov_layout(d, base);
  size_t off = w.mk.bytes;
  const size_t R = d->R, G = d->gamma, r = d->r;
  w.U = (bf16 *)(base + off);
  off = dspark_align_up(off + sizeof(bf16) * R * 2 * r, 256);
  w.state = (float *)(base + off);
  off = dspark_align_up(off + sizeof(float) * R * r, 256);
  w.Gk = (float *)(base + off);
  // K = 2r in 64-deep blocks, up to four splits of equal depth
  const int kb = (int)(2 * r / 64);
  w.splits = kb % 4 == 0 ? 4 : (kb % 2 == 0 ? 2 : 1);
  w.m_pad = (int)((R + 127) / 128 * 128);
  off = dspark_align_up(off + sizeof(float) * (size_t)w.splits * w.m_pad * 2 * r, 256);
  w.P = (float *)(base + off);
  w.psplits = rnn_hidden_splits((int)(R * G), (int)(2 * r), d->d);
  w.pm_pad = (int)((R * G + 127) / 128 * 128);
  off = dspark_align_up(off + sizeof(float) * (size_t)w.psplits * w.pm_pad * 2 * r, 256);
  w.bytes = off;
  return w;
}

}  // namespace

extern "C" size_t dspark_rnn_workspace_bytes(const dspark_dims *dims) {
  if (!dspark_dims_ok(dims)) return 0;
  return rnn_layout(dims, nullptr).bytes;
}

extern "C" int dspark_rnn_draft(const dspark_dims *dims, const void *base_logits, const void *h,
                                const int32_t *anchor, const void *W1, const void *W2t,
                                const void *W_rec, const void *W_hid, const void *w_conf,
                                const float *T, float tau, uint64_t seed, int32_t *tokens,
                                float *conf, float *logp_d, float *lse_d, void *workspace,
                                size_t workspace_bytes, dspark_stream_t stream) {
  if (!dspark_dims_ok(dims) || !base_logits || !h || !anchor || !W1 || !W2t || !W_rec ||
      !W_hid || !w_conf || !T || !tokens || !conf || !(tau >= 0.f))
    return DSPARK_ERR_ARG;
  if (((uintptr_t)W2t | (uintptr_t)W1 | (uintptr_t)h | (uintptr_t)base_logits |
       (uintptr_t)W_rec | (uintptr_t)W_hid) & 15)
    return DSPARK_ERR_ARG;  // TMA and 16-byte vector loads
  RnnWs ws = rnn_layout(dims, (char *)workspace);
  if (!workspace || workspace_bytes < ws.bytes || ((uintptr_t)workspace & 255))
    return DSPARK_ERR_WORKSPACE;
  const int R = dims->R, G = dims->gamma, V = dims->V, r = dims->r, d = dims->d;
  const bf16 *w_e = (const bf16 *)w_conf + d;
  const float inv_tau = tau > 0.f ? 1.f / tau : 1.f;
  conf_hidden<<<R * G, 128, 0, stream>>>((const bf16 *)h, (const bf16 *)w_conf, ws.mk.zh, d,
                                         nullptr);
  DSPARK_CHECK_LAUNCH();
  // W_hid h for all positions at once, split over K: 2r = 1024 columns and
  // R gamma = 1280 rows make only 40 tiles, each 112 k blocks deep
  int rc = gemm::launch<4, 256>(h, W_hid, R * G, 2 * r, d,
                                EpiStoreF32{ws.P, ws.psplits * ws.pm_pad, 2 * r}, stream,
                                nullptr, true, ws.psplits);
  if (rc != DSPARK_OK) return rc;
  if (cudaMemsetAsync(ws.U, 0, sizeof(bf16) * (size_t)R * 2 * r, stream) != cudaSuccess ||
      cudaMemsetAsync(ws.state, 0, sizeof(float) * (size_t)R * r, stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  step_prep<<<(R * 32 + 255) / 256, 256, 0, stream>>>(anchor, tokens, (const bf16 *)W1, w_e,
                                                     ws.mk.zh, T, ws.U + r, 2 * r, conf, R, G,
                                                     V, r, 1);
  DSPARK_CHECK_LAUNCH();
  for (int k = 1; k <= G; ++k) {
    // split over K: 16 k blocks (r = 512) on 32 tiles would leave most SMs idle
    rc = gemm::launch<4, 64>(ws.U, W_rec, R, 2 * r, 2 * r,
                             EpiStoreF32{ws.Gk, ws.splits * ws.m_pad, 2 * r}, stream, nullptr,
                             true, ws.splits);
    if (rc != DSPARK_OK) return rc;
    if (dspark_launch_pdl(rnn_state, dim3((R * r + 255) / 256), dim3(256), 0, stream,
                          (const float *)ws.Gk, (const float *)ws.P, ws.state, ws.mk.E, ws.U, R,
                          G, r, k, ws.splits, ws.m_pad, ws.psplits, ws.pm_pad) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    if (tau > 0.f) {
      const int n_parts = logits_parts<MODE_SAMPLE>(V);
      EpiLogits<MODE_SAMPLE> epi{(const bf16 *)base_logits, nullptr, nullptr, nullptr, nullptr,
                                 ws.mk.part, R, V, G, k, n_parts, inv_tau, seed};
      rc = gemm::launch<LogitsCfg<MODE_SAMPLE>::EPI_WARPS, LogitsCfg<MODE_SAMPLE>::BN>(
          ws.mk.E, W2t, R, V, r, epi, stream, nullptr, true);
      if (rc != DSPARK_OK) return rc;
      if (dspark_launch_pdl(reduce_prep<MODE_SAMPLE>, dim3(R), dim3(RP_THREADS), 0, stream,
                            ws.mk.part, n_parts, G, V, r, k, tokens, lse_d, logp_d,
                            (const bf16 *)W1, w_e, ws.mk.zh, T, (const bf16 *)ws.mk.E, r, r,
                            ws.U + r, 2 * r, conf,
                            (const bf16 *)base_logits, (const bf16 *)W2t, inv_tau,
                            seed) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    } else {
      const int n_parts = logits_parts<MODE_GREEDY>(V);
      EpiLogits<MODE_GREEDY> epi{(const bf16 *)base_logits, nullptr, nullptr, nullptr, nullptr,
                                 ws.mk.part, R, V, G, k, n_parts, 1.f, seed};
      rc = gemm::launch<LogitsCfg<MODE_GREEDY>::EPI_WARPS, LogitsCfg<MODE_GREEDY>::BN>(
          ws.mk.E, W2t, R, V, r, epi, stream, nullptr, true);
      if (rc != DSPARK_OK) return rc;
      if (dspark_launch_pdl(reduce_prep<MODE_GREEDY>, dim3(R), dim3(RP_THREADS), 0, stream,
                            ws.mk.part, n_parts, G, V, r, k, tokens, lse_d, logp_d,
                            (const bf16 *)W1, w_e, ws.mk.zh, T, (const bf16 *)ws.mk.E, r, r,
                            ws.U + r, 2 * r, conf,
                            (const bf16 *)base_logits, (const bf16 *)W2t, inv_tau,
                            seed) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    }
    DSPARK_CHECK_LAUNCH();
  }
  dspark_count_launches(2 + 2 * (uint64_t)G);  // + the GEMMs, counted by launch()
  return DSPARK_OK;
}

// ---------------------------------------------------------------------------
// Fused single-contraction step, a measured variant: per step k the logits
// come from one contraction [h_k; W1[x_{k-1}]] . [W_lm; W2]^T, so the base
// logits never reach HBM, at the price of streaming W_lm once per step instead
// of once per round ("DSpark 深度解读" §二 设计一 reads the draft logits as the
// shared LM head's plus the Markov bias; this computes the same sum in one
// GEMM).  Per step: A_k = [h_k | W1[x_{k-1}]] (a strided copy of h_k and the
// embedding gather), the tcgen05 GEMM with the draft epilogue and no base
// logits, then reduce_prep.
// ---------------------------------------------------------------------------
namespace {

struct FusedWs {
  MarkovWs mk;
  bf16 *A;  // [R, d + r]
  size_t bytes;
};

FusedWs fused_layout(const dspark_dims *d, char *base) {
  FusedWs w;
  w.mk = markov_layout(d, base);
  size_t off = w.mk.bytes;
  w.A = (bf16 *)(base + off);
  off = dspark_align_up(off + sizeof(bf16) * (size_t)d->R * (d->d + d->r), 256);
  w.bytes = off;
  return w;
}

// d and r are multiples of 64, so d + r is a whole number of 64-deep k blocks
bool fused_dims_ok(const dspark_dims *d) { return dspark_dims_ok(d); }

}  // namespace

extern "C" size_t dspark_fused_workspace_bytes(const dspark_dims *dims) {
  if (!fused_dims_ok(dims)) return 0;
  return fused_layout(dims, nullptr).bytes;
}

extern "C" int dspark_pack_fused(const dspark_dims *dims, const void *W_lm, const void *W2t,
                                 void *W_cat, dspark_stream_t stream) {
  if (!fused_dims_ok(dims) || !W_lm || !W2t || !W_cat) return DSPARK_ERR_ARG;
  const size_t V = dims->V, d = dims->d, r = dims->r, ld = (d + r) * sizeof(bf16);
  if (cudaMemcpy2DAsync(W_cat, ld, W_lm, d * sizeof(bf16), d * sizeof(bf16), V,
                        cudaMemcpyDeviceToDevice, stream) != cudaSuccess ||
      cudaMemcpy2DAsync((char *)W_cat + d * sizeof(bf16), ld, W2t, r * sizeof(bf16),
                        r * sizeof(bf16), V, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

extern "C" int dspark_fused_draft(const dspark_dims *dims, const void *h, const int32_t *anchor,
                                  const void *W_cat, const void *W1, const void *w_conf,
                                  const float *T, float tau, uint64_t seed, int32_t *tokens,
                                  float *conf, float *logp_d, float *lse_d, void *workspace,
                                  size_t workspace_bytes, dspark_stream_t stream) {
  if (!fused_dims_ok(dims) || !h || !anchor || !W_cat || !W1 || !w_conf || !T || !tokens ||
      !conf || !(tau >= 0.f))
    return DSPARK_ERR_ARG;
  if (((uintptr_t)W_cat | (uintptr_t)W1 | (uintptr_t)h) & 15)
    return DSPARK_ERR_ARG;  // TMA and 16-byte vector loads
  FusedWs ws = fused_layout(dims, (char *)workspace);
  if (!workspace || workspace_bytes < ws.bytes || ((uintptr_t)workspace & 255))
    return DSPARK_ERR_WORKSPACE;
  const int R = dims->R, G = dims->gamma, V = dims->V, r = dims->r, d = dims->d;
  const int K = d + r;
  const bf16 *w_e = (const bf16 *)w_conf + d;
  const float inv_tau = tau > 0.f ? 1.f / tau : 1.f;
  conf_hidden<<<R * G, 128, 0, stream>>>((const bf16 *)h, (const bf16 *)w_conf, ws.mk.zh, d,
                                         nullptr);
  DSPARK_CHECK_LAUNCH();
  // E_1 = W1[anchor] into the embedding columns of A, and c_1
  step_prep<<<(R * 32 + 255) / 256, 256, 0, stream>>>(anchor, tokens, (const bf16 *)W1, w_e,
                                                     ws.mk.zh, T, ws.A + d, K, conf, R, G, V,
                                                     r, 1);
  DSPARK_CHECK_LAUNCH();
  for (int k = 1; k <= G; ++k) {
    // h_k into the first d columns of A (reduce_prep of step k-1 is done with A)
    if (cudaMemcpy2DAsync(ws.A, (size_t)K * sizeof(bf16),
                          (const bf16 *)h + (size_t)(k - 1) * d, (size_t)G * d * sizeof(bf16),
                          (size_t)d * sizeof(bf16), R, cudaMemcpyDeviceToDevice,
                          stream) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    int rc;
    if (tau > 0.f) {
      const int n_parts = logits_parts<MODE_SAMPLE>(V);
      EpiLogits<MODE_SAMPLE> epi{nullptr, nullptr, nullptr, nullptr, nullptr, ws.mk.part,
                                 R, V, G, k, n_parts, inv_tau, seed};
      rc = gemm::launch<LogitsCfg<MODE_SAMPLE>::EPI_WARPS, LogitsCfg<MODE_SAMPLE>::BN>(
          ws.A, W_cat, R, V, K, epi, stream, nullptr, true);
      if (rc != DSPARK_OK) return rc;
      if (dspark_launch_pdl(reduce_prep<MODE_SAMPLE>, dim3(R), dim3(RP_THREADS), 0, stream,
                            ws.mk.part, n_parts, G, V, r, k, tokens, lse_d, logp_d,
                            (const bf16 *)W1, w_e, ws.mk.zh, T, (const bf16 *)ws.A, K, K,
                            ws.A + d, K, conf, (const bf16 *)nullptr, (const bf16 *)W_cat,
                            inv_tau, seed) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    } else {
      const int n_parts = logits_parts<MODE_GREEDY>(V);
      EpiLogits<MODE_GREEDY> epi{nullptr, nullptr, nullptr, nullptr, nullptr, ws.mk.part,
                                 R, V, G, k, n_parts, 1.f, seed};
      rc = gemm::launch<LogitsCfg<MODE_GREEDY>::EPI_WARPS, LogitsCfg<MODE_GREEDY>::BN>(
          ws.A, W_cat, R, V, K, epi, stream, nullptr, true);
      if (rc != DSPARK_OK) return rc;
      if (dspark_launch_pdl(reduce_prep<MODE_GREEDY>, dim3(R), dim3(RP_THREADS), 0, stream,
                            ws.mk.part, n_parts, G, V, r, k, tokens, lse_d, logp_d,
                            (const bf16 *)W1, w_e, ws.mk.zh, T, (const bf16 *)ws.A, K, K,
                            ws.A + d, K, conf, (const bf16 *)nullptr, (const bf16 *)W_cat,
                            inv_tau, seed) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    }
  }
  dspark_count_launches(2 + (uint64_t)G);  // + the GEMMs, counted by launch()
  return DSPARK_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the same draft loop with its scratch in one static
// device array.  For callers that have no way to allocate device memory (a
// plugin interface that passes only tensors, a serving loop that forbids
// allocations after start-up).  The array is shared by every call: overlapping
// calls race.  No field of the scratch needs to start at zero: the draft loop
// writes every word it reads.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_markov_scratch[DSPARK_STATIC_SCRATCH_BYTES];

namespace {
constexpr int MAX_DEVICES = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[MAX_DEVICES] = {};
}  // namespace

extern "C" int dspark_markov_draft_static(const dspark_dims *dims, const void *base_logits,
                                          const void *h, const int32_t *anchor, const void *W1,
                                          const void *W2t, const void *w_conf, const float *T,
                                          float tau, uint64_t seed, int32_t *tokens, float *conf,
                                          float *logp_d, float *lse_d, dspark_stream_t stream) {
  if (!dspark_dims_ok(dims)) return DSPARK_ERR_ARG;
  if (dspark_markov_workspace_bytes(dims) > DSPARK_STATIC_SCRATCH_BYTES) return DSPARK_ERR_TOO_LARGE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return DSPARK_ERR_CUDA;
  void *ptr;
  {
    // set-up once per device, with that device current: the host-side symbol is
    // only a stand-in, the kernels need the array's device address
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_markov_scratch) != cudaSuccess || !p) return DSPARK_ERR_CUDA;
      g_scratch_ptr[dev] = p;
    }
    ptr = g_scratch_ptr[dev];
  }
  return dspark_markov_draft(dims, base_logits, h, anchor, W1, W2t, w_conf, T, tau, seed, tokens,
                             conf, logp_d, lse_d, ptr, DSPARK_STATIC_SCRATCH_BYTES, stream);
}
