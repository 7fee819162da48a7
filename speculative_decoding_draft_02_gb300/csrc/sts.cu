// sts.cu — Sequential Temperature Scaling: the per-position temperatures of the
// confidence head, fitted on held-out rounds.
//
// "DSpark 深度解读" §二 设计二 (STS 校准): position 1's temperature is searched to
// minimise the expected calibration error, then position 2's with position 1
// fixed, and so on; the stage summary adds that what is calibrated is the
// cumulative prefix survival probability.  So position j picks, from a grid,
// the T of least ECE of a_j = a_{j-1} * sigmoid(z_j / T) (f32, left to right)
// against the label "drafts 1..j all accepted".  With n_bins equal-width bins,
// ECE = sum_b |sum_{n in b} (label_n - a_n)| / N, so one sum per (grid value,
// bin) is all the state a position needs.  The sums are kept in 64-bit fixed
// point (2^-32 units; each term rounds by at most 2^-33, so the ECE moves by at
// most 2^-33): integer atomics, native in shared memory and independent of the
// order in which samples arrive.
//
// Per position, three launches: sts_hist (n_grid x chunks CTAs; a CTA bins one
// chunk of samples for one grid value in shared memory and adds its sums to
// the global ones), sts_select (one CTA: the ECE of every grid value and the
// argmin) and sts_advance (a_j at the chosen temperature).
// dspark_conf_logits gives the logits z that the fit takes.
#include "common.cuh"

DSPARK_DECLARE_STATUS(s_status_sts)

namespace {

constexpr int STS_THREADS = 256;
constexpr int STS_MAX_BINS = 64;

__device__ __forceinline__ float sigmoid_over(float z, float T) {
  return 1.f / (1.f + expf(-(z / T)));
}

constexpr float FIX_ONE = 4294967296.f;  // 2^32: one unit of label - a

// D[g][b] += sum over the CTA's samples in bin b of (label - a_j(T_g)), in 2^-32 units.
__global__ void __launch_bounds__(STS_THREADS) sts_hist(
    const float *__restrict__ z, const int32_t *__restrict__ accepted,
    const float *__restrict__ a_prev, const float *__restrict__ grid, int N, int gamma, int j,
    int n_bins, int chunk, unsigned long long *__restrict__ D) {
  __shared__ unsigned long long sd[STS_MAX_BINS];
  const int g = blockIdx.x, tid = threadIdx.x;
  for (int b = tid; b < n_bins; b += STS_THREADS) sd[b] = 0ull;
  __syncthreads();
  const float T = grid[g];
  if (!(T > 0.f) && tid == 0 && blockIdx.y == 0) dspark_set_status(DSPARK_ERR_ARG);
  const int beg = blockIdx.y * chunk, end = min(N, beg + chunk);
  const float nb = (float)n_bins;
  for (int n = beg + tid; n < end; n += STS_THREADS) {
    const float c = sigmoid_over(z[(size_t)n * gamma + j], T);
    const float a = j ? __fmul_rn(a_prev[n], c) : c;
    int b = (int)__fmul_rn(a, nb);
    b = b < 0 ? 0 : (b >= n_bins ? n_bins - 1 : b);
    // label - a in fixed point: a * 2^32 is exact in f32, its rounding to an
    // integer is the only error; negative sums wrap as two's complement
    const long long qa = __float2ll_rn(__fmul_rn(a, FIX_ONE));
    const long long q = (accepted[n] >= j + 1 ? (1ll << 32) : 0ll) - qa;
    atomicAdd(&sd[b], (unsigned long long)q);
  }
  __syncthreads();
  unsigned long long *Dg = D + ((size_t)j * gridDim.x + g) * n_bins;
  for (int b = tid; b < n_bins; b += STS_THREADS)
    if (sd[b] != 0ull) atomicAdd(&Dg[b], sd[b]);
}

// ECE of every grid value at position j; the least (first on ties) is kept.
__global__ void __launch_bounds__(STS_THREADS) sts_select(const unsigned long long *__restrict__ D,
                                                          const float *__restrict__ grid,
                                                          int n_grid, int n_bins, int N, int j,
                                                          float *__restrict__ T_out,
                                                          double *__restrict__ ece_out) {
  __shared__ double sv[STS_THREADS / 32];
  __shared__ int si[STS_THREADS / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned long long *Dj = D + (size_t)j * n_grid * n_bins;
  double best = INFINITY;
  int bg = 0x7fffffff;
  for (int g = tid; g < n_grid; g += STS_THREADS) {
    double e = 0.0;
    for (int b = 0; b < n_bins; ++b) e += fabs((double)(long long)Dj[(size_t)g * n_bins + b]);
    e = e / 4294967296.0 / (double)N;
    if (e < best) { best = e; bg = g; }  // g increases per thread: first on ties
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const double e2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int g2 = __shfl_xor_sync(0xffffffffu, bg, o);
    if (e2 < best || (e2 == best && g2 < bg)) { best = e2; bg = g2; }
  }
  if (lane == 0) { sv[warp] = best; si[warp] = bg; }
  __syncthreads();
  if (warp == 0) {
    best = lane < STS_THREADS / 32 ? sv[lane] : INFINITY;
    bg = lane < STS_THREADS / 32 ? si[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const double e2 = __shfl_xor_sync(0xffffffffu, best, o);
      const int g2 = __shfl_xor_sync(0xffffffffu, bg, o);
      if (e2 < best || (e2 == best && g2 < bg)) { best = e2; bg = g2; }
    }
    if (lane == 0) {
      if (bg < 0 || bg >= n_grid) bg = 0;  // every ECE NaN: keep the first grid value
      T_out[j] = grid[bg];
      ece_out[j] = best;
    }
  }
}

// a_j = a_{j-1} * sigmoid(z_j / T_j) with the temperature just chosen.
__global__ void sts_advance(const float *__restrict__ z, const float *__restrict__ T_out,
                            float *__restrict__ a_prev, int N, int gamma, int j) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const float c = sigmoid_over(z[(size_t)n * gamma + j], T_out[j]);
  a_prev[n] = j ? __fmul_rn(a_prev[n], c) : c;
}

// z[m] = w_h . h[m] + w_e . W1[x_{j-1}] for row m = r * gamma + j - 1 (x_0 the
// anchor): the confidence logit before its temperature.  One warp per row.
__global__ void conf_logits(const bf16 *__restrict__ h, const int32_t *__restrict__ anchor,
                            const int32_t *__restrict__ tokens, const bf16 *__restrict__ W1,
                            const bf16 *__restrict__ w_conf, float *__restrict__ z, int R,
                            int gamma, int V, int r, int d) {
  const int m = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (m >= R * gamma) return;
  const int i = m / gamma, j = m % gamma;
  int prev = j == 0 ? anchor[i] : tokens[(size_t)i * gamma + j - 1];
  if (prev < 0 || prev >= V) {
    if (lane == 0) dspark_set_status(DSPARK_ERR_TOKEN);
    prev = 0;
  }
  const uint4 *hr = reinterpret_cast<const uint4 *>(h + (size_t)m * d);
  const uint4 *wh = reinterpret_cast<const uint4 *>(w_conf);
  const uint4 *er = reinterpret_cast<const uint4 *>(W1 + (size_t)prev * r);
  const uint4 *we = reinterpret_cast<const uint4 *>(w_conf + d);
  float acc = 0.f;
  for (int c = lane; c < d / 8; c += 32) acc = dot8_bf16(hr[c], wh[c], acc);
  for (int c = lane; c < r / 8; c += 32) acc = dot8_bf16(er[c], we[c], acc);
  acc = warp_sum(acc);
  if (lane == 0) z[m] = acc;
}

struct StsWs {
  float *a_prev;
  unsigned long long *D;  // fixed-point sums [gamma][n_grid][n_bins]
  size_t bytes;
};

StsWs sts_layout(int N, int gamma, int n_grid, int n_bins, char *base) {
  StsWs w;
  size_t off = 0;
  w.a_prev = (float *)(base + off);
  off = dspark_align_up(off + sizeof(float) * (size_t)N, 256);
  w.D = (unsigned long long *)(base + off);
  off = dspark_align_up(off + sizeof(unsigned long long) * (size_t)gamma * n_grid * n_bins, 256);
  w.bytes = off;
  return w;
}

bool sts_args_ok(int N, int gamma, int n_grid, int n_bins) {
  return N >= 1 && gamma >= 1 && gamma <= 32 && n_grid >= 1 && n_bins >= 1 &&
         n_bins <= STS_MAX_BINS;
}

}  // namespace

extern "C" size_t dspark_sts_workspace_bytes(int32_t N, int32_t gamma, int32_t n_grid,
                                            int32_t n_bins) {
  if (!sts_args_ok(N, gamma, n_grid, n_bins)) return 0;
  return sts_layout(N, gamma, n_grid, n_bins, nullptr).bytes;
}

extern "C" int dspark_sts_fit(const float *z, const int32_t *accepted, int32_t N, int32_t gamma,
                              const float *T_grid, int32_t n_grid, int32_t n_bins, float *T_out,
                              double *ece_out, void *workspace, size_t workspace_bytes,
                              dspark_stream_t stream) {
  if (!z || !accepted || !T_grid || !T_out || !ece_out || !sts_args_ok(N, gamma, n_grid, n_bins))
    return DSPARK_ERR_ARG;
  StsWs ws = sts_layout(N, gamma, n_grid, n_bins, (char *)workspace);
  if (!workspace || workspace_bytes < ws.bytes || ((uintptr_t)workspace & 255))
    return DSPARK_ERR_WORKSPACE;
  if (cudaMemsetAsync(ws.D, 0, sizeof(unsigned long long) * (size_t)gamma * n_grid * n_bins, stream) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  // about four CTAs per SM over the grid values and sample chunks
  const int target = 4 * dspark_sm_count();
  int chunks = (target + n_grid - 1) / n_grid;
  const int max_chunks = (N + STS_THREADS - 1) / STS_THREADS;
  chunks = chunks < 1 ? 1 : (chunks > max_chunks ? max_chunks : chunks);
  const int chunk = (N + chunks - 1) / chunks;
  for (int j = 0; j < gamma; ++j) {
    sts_hist<<<dim3(n_grid, chunks), STS_THREADS, 0, stream>>>(z, accepted, ws.a_prev, T_grid, N,
                                                              gamma, j, n_bins, chunk, ws.D);
    DSPARK_CHECK_LAUNCH();
    sts_select<<<1, STS_THREADS, 0, stream>>>(ws.D, T_grid, n_grid, n_bins, N, j, T_out,
                                              ece_out);
    DSPARK_CHECK_LAUNCH();
    sts_advance<<<(N + 255) / 256, 256, 0, stream>>>(z, T_out, ws.a_prev, N, gamma, j);
    DSPARK_CHECK_LAUNCH();
  }
  dspark_count_launches(3 * (uint64_t)gamma);
  return DSPARK_OK;
}

extern "C" int dspark_conf_logits(const dspark_dims *dims, const void *h, const int32_t *anchor,
                                  const int32_t *tokens, const void *W1, const void *w_conf,
                                  float *z, dspark_stream_t stream) {
  if (!dspark_dims_ok(dims) || !h || !anchor || !tokens || !W1 || !w_conf || !z)
    return DSPARK_ERR_ARG;
  if (((uintptr_t)h | (uintptr_t)W1 | (uintptr_t)w_conf) & 15) return DSPARK_ERR_ARG;
  const int rows = dims->R * dims->gamma;
  conf_logits<<<(rows * 32 + 255) / 256, 256, 0, stream>>>(
      (const bf16 *)h, anchor, tokens, (const bf16 *)W1, (const bf16 *)w_conf, z, dims->R,
      dims->gamma, dims->V, dims->r, dims->d);
  DSPARK_CHECK_LAUNCH();
  dspark_count_launches(1);
  return DSPARK_OK;
}

int dspark_status_sts(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, s_status_sts, sizeof(int)) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    cudaMemcpyToSymbol(s_status_sts, &zero, sizeof(int));
  }
  return v;
}
