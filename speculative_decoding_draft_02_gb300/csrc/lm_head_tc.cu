// lm_head_tc.cu — a1 on the tensor cores: l0 = h . W_lm^T through the
// persistent tcgen05 GEMM (TMA-fed, f32 accumulation in TMEM), with an
// epilogue that rounds each accumulator row to bf16 and stores it.
//
// "DSpark 深度解读" §二 (architecture): base logits of all gamma positions come
// from one pass through the LM head shared with the target.
#include "umma_gemm.cuh"

DSPARK_DECLARE_STATUS(s_status_lmhead_tc)

namespace {

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<const uint32_t *>(&v);
}

struct EpiStoreBF16 {
  bf16 *C;
  int M, N;
  __device__ void operator()(int m0, int n0, int row, uint32_t taddr) const {
    const int m = m0 + row;
    bf16 *dst_row = C + (size_t)m * N;
#pragma unroll 1
    for (int c = 0; c < gemm::BN; c += 32) {
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
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  return sms;
}

int dspark_lm_head_tc(const dspark_dims *dims, const void *h, const void *W_lm,
                      void *base_logits, cudaStream_t stream) {
  EpiStoreBF16 epi;
  epi.C = (bf16 *)base_logits;
  epi.M = dims->R * dims->gamma;
  epi.N = dims->V;
  return gemm::launch(h, W_lm, epi.M, epi.N, dims->d, epi, stream);
}

int dspark_status_lmhead_tc(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, s_status_lmhead_tc, sizeof(int)) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (clear) {
    const int z = 0;
    cudaMemcpyToSymbol(s_status_lmhead_tc, &z, sizeof(int));
  }
  return v;
}
