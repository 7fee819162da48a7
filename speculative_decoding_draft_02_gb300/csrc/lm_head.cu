// lm_head.cu — a1: base draft logits through the shared LM head, on the tensor
// cores, and the one-time W2 layout preparation.
//
// "DSpark 深度解读" §二 (architecture): the parallel backbone emits gamma hidden
// states and the base logits of all positions come from one pass through the
// LM head shared with, and frozen from, the target:
//   l0[m, v] = sum_i h[m, i] W_lm[v, i],  m = r*gamma + k - 1.
// The contraction runs on the persistent tcgen05 GEMM (TMA-fed, f32
// accumulation in TMEM); the epilogue rounds each accumulator row to bf16.
#include "umma_gemm_pair.cuh"

DSPARK_DECLARE_STATUS(s_status_lmhead)

#include "umma_skinny.cuh"

namespace {

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<const uint32_t *>(&v);
}

struct EpiStoreBF16 {
  bf16 *C;
  int M, N;
  struct State {};
  static constexpr bool kRowAffine = false;
  static constexpr bool kStreamB = true;  // W_lm streams through once per launch
  __device__ void prefetch(int, int, int, int, int, State &) const {}
  __device__ void operator()(int m0, int n0, int row, uint32_t taddr, int c0, int c1, int, int,
                             State &) const {
    const int m = m0 + row;
    bf16 *dst_row = C + (size_t)m * N;
#pragma unroll 1
    for (int c = c0; c < c1; c += 32) {
      uint32_t r[32];
      tc::tmem_ld32(taddr + (uint32_t)c, r);
      tc::tmem_wait_ld();
      if (m < M) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int n = n0 + c + q * 8;
          if (n + 8 <= N) {
            uint4 v;
            v.x = pack_bf16x2(r[q * 8 + 0], r[q * 8 + 1]);
            v.y = pack_bf16x2(r[q * 8 + 2], r[q * 8 + 3]);
            v.z = pack_bf16x2(r[q * 8 + 4], r[q * 8 + 5]);
            v.w = pack_bf16x2(r[q * 8 + 6], r[q * 8 + 7]);
            *reinterpret_cast<uint4 *>(dst_row + n) = v;
          }
        }
      }
    }
  }
  __device__ void on_timeout() const { dspark_set_status(DSPARK_ERR_TIMEOUT); }
};

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

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

int dspark_make_tmap_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                          uint32_t box_rows) {
  static EncodeTiledFn encode = nullptr;
  if (!encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return -1;
    encode = (EncodeTiledFn)fn;
  }
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
                            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

int dspark_sm_count() {
  static DsparkPerDevice sms;
  const int n = dspark_per_device(sms, [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      return -1;
    return v;
  });
  return n > 0 ? n : 1;
}

int dspark_lm_head_tc(const dspark_dims *dims, const void *h, const void *W_lm,
                      void *base_logits, cudaStream_t stream) {
  EpiStoreBF16 epi;
  epi.C = (bf16 *)base_logits;
  epi.M = dims->R * dims->gamma;
  epi.N = dims->V;
  // From four row blocks (512 rows) on, CTA pairs (cta_group::2) on 256 x 256
  // tiles: a third fewer operand bytes per SM per flop.  At R*gamma = 1280, 91%
  // of the bf16 peak against 86% for the single-CTA kernel; at 512 rows
  // (V = 151936, d = 4096) 0.383 against 0.425 ms.  Below four row blocks a
  // pair would leave up to a quarter of its rows empty.
  // Up to 16 rows, the swapped product: W_lm is the 128-row operand and h the
  // 16-column one, so the ring holds twelve stages of W_lm instead of four
  // 128 x 256 tiles beside a mostly empty 128-row tile of h.  V = 151936,
  // d = 2560: 8 rows 132 against 165 us (0.87 against 0.69 of the copy
  // peak), 16 rows 133 against 154 us; at 32 rows the 32-column form took
  // 131 against 126 us, so from 17 rows on the row-tiled kernel stays.
  const int num_m = (epi.M + gemm::BM - 1) / gemm::BM;
  if (epi.M <= 16)
    return gemm::launch_skinny<16>(h, W_lm, epi.M, epi.N, dims->d, epi.C, stream);
  if (num_m >= 4) return gemm::launch_pair<4>(h, W_lm, epi.M, epi.N, dims->d, epi, stream);
  return gemm::launch<4, 256>(h, W_lm, epi.M, epi.N, dims->d, epi, stream);
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
  if (cudaMemcpyFromSymbol(&v, s_status_lmhead, sizeof(int)) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (clear) {
    const int z = 0;
    cudaMemcpyToSymbol(s_status_lmhead, &z, sizeof(int));
  }
  return v;
}
