// lm_head.cu — a1: base draft logits through the shared LM head, and the W2
// layout preparation.
//
// "DSpark 深度解读" §二 (architecture): the parallel backbone emits gamma hidden
// states; base logits come from the LM head shared with, and frozen from, the
// target.  l0[m, v] = sum_i h[m, i] W_lm[v, i], m = r*gamma + k - 1.
#include "common.cuh"

DSPARK_DECLARE_STATUS(s_status_lmhead)

int dspark_lm_head_tc(const dspark_dims *dims, const void *h, const void *W_lm,
                      void *base_logits, cudaStream_t stream);  // lm_head_tc.cu

namespace {

// Plain smem-tiled FMA GEMM C[M, N] = A[M, K] B[N, K]^T (both K-contiguous),
// f32 accumulation, bf16 output.  64x64 tile, 256 threads, 4x4 per thread.
constexpr int SBM = 64, SBN = 64, SBK = 32;

__global__ void __launch_bounds__(256) gemm_nt_simple(const bf16 *__restrict__ A,
                                                      const bf16 *__restrict__ B,
                                                      bf16 *__restrict__ C, int M, int N,
                                                      int K) {
  __shared__ float As[SBK][SBM + 1];
  __shared__ float Bs[SBK][SBN + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * SBM, n0 = blockIdx.x * SBN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < K; k0 += SBK) {
    for (int e = threadIdx.x; e < SBM * SBK; e += 256) {
      const int mm = e / SBK, kk = e % SBK;
      As[kk][mm] = (m0 + mm < M) ? __bfloat162float(A[(size_t)(m0 + mm) * K + k0 + kk]) : 0.f;
      Bs[kk][mm] = (n0 + mm < N) ? __bfloat162float(B[(size_t)(n0 + mm) * K + k0 + kk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < SBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < N) C[(size_t)m * N + n] = __float2bfloat16_rn(acc[i][j]);
    }
  }
}

// W2t[v, i] = W2[i, v] through 32x32 shared tiles.
__global__ void transpose_bf16(const bf16 *__restrict__ in, bf16 *__restrict__ out, int rows,
                               int cols) {
  __shared__ bf16 tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int rr = r0 + i, cc = c0 + threadIdx.x;
    if (rr < rows && cc < cols) tile[i][threadIdx.x] = in[(size_t)rr * cols + cc];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int cc = c0 + i, rr = r0 + threadIdx.x;
    if (rr < rows && cc < cols) out[(size_t)cc * rows + rr] = tile[threadIdx.x][i];
  }
}

}  // namespace

int dspark_lm_head_simple(const dspark_dims *dims, const void *h, const void *W_lm,
                          void *base_logits, cudaStream_t stream) {
  const int M = dims->R * dims->gamma, N = dims->V, K = dims->d;
  dim3 grid((N + SBN - 1) / SBN, (M + SBM - 1) / SBM);
  gemm_nt_simple<<<grid, 256, 0, stream>>>((const bf16 *)h, (const bf16 *)W_lm,
                                           (bf16 *)base_logits, M, N, K);
  DSPARK_CHECK_LAUNCH();
  dspark_count_launches(1);
  return DSPARK_OK;
}

extern "C" int dspark_pack_w2(const dspark_dims *dims, const void *W2, void *W2t,
                              dspark_stream_t stream) {
  if (!dspark_dims_ok(dims) || !W2 || !W2t) return DSPARK_ERR_ARG;
  dim3 grid((dims->V + 31) / 32, (dims->r + 31) / 32);
  transpose_bf16<<<grid, dim3(32, 8), 0, stream>>>((const bf16 *)W2, (bf16 *)W2t, dims->r,
                                                   dims->V);
  DSPARK_CHECK_LAUNCH();
  dspark_count_launches(1);
  return DSPARK_OK;
}

int dspark_status_lmhead(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, s_status_lmhead, sizeof(int)) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (clear) {
    const int z = 0;
    cudaMemcpyToSymbol(s_status_lmhead, &z, sizeof(int));
  }
  return v;
}
