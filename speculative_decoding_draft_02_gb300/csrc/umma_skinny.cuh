// umma_skinny.cuh — C[M, V] = X[M, K] . W[V, K]^T for few rows (M <= NS, NS = 16
// or 32), in bf16 out, on the tcgen05 tensor cores with the operands swapped:
// W is the 128-row A operand and X the narrow B operand (N = NS columns), so
// the accumulator holds C^T, 128 vocabulary rows by N.  With M rows on the A
// side a 128-row A tile would be mostly padding, and a wide B tile of W would
// leave room for only four ring stages; here a stage is 16 KB of W and 2-4 KB
// of X, so up to twelve stages of W are in flight per SM.  This is the shape
// of the LM head for one or a few requests (R * gamma rows), where the product
// is bound by streaming W once; the LM head takes it up to 16 rows.
//
// One CTA per SM, 192 threads: warp 0 issues the TMA loads, warp 1 allocates
// TMEM and issues the MMAs, warps 2..5 (one per TMEM lane quarter) store C.
// Vocabulary tiles of 128 rows are strided over the CTAs.  Every wait is
// bounded; on timeout the CTA raises DSPARK_ERR_TIMEOUT (through the caller's
// status word), drains its own copies and MMAs, frees TMEM and exits.
#pragma once
#include "umma_gemm.cuh"

namespace gemm {

template <int NS>
struct SkinnyGeo {
  static_assert(NS == 16 || NS == 32, "N of the swapped product: 16 or 32 rows of X");
  static constexpr int B_BYTES = NS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (int)((SMEM_LIMIT - 1024 - 512) / STAGE_BYTES) > 12
                                    ? 12
                                    : (int)((SMEM_LIMIT - 1024 - 512) / STAGE_BYTES);
  static constexpr uint32_t TMEM_COLS = 2 * NS < 32 ? 32 : 2 * NS;
  static constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 512;
};

template <int NS>
__global__ void __launch_bounds__(192, 1)
    umma_skinny_kernel(const __grid_constant__ CUtensorMap tma_w,
                       const __grid_constant__ CUtensorMap tma_x, int M, int V, int K,
                       bf16 *__restrict__ C) {
  using G = SkinnyGeo<NS>;
  constexpr int STAGES = G::STAGES, B_BYTES = G::B_BYTES, STAGE_BYTES = G::STAGE_BYTES;
  constexpr uint32_t TMEM_COLS = G::TMEM_COLS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = base;                       // W tiles, 1 KB aligned (16 KB each)
  uint8_t *sB = base + STAGES * A_BYTES;    // X tiles (B_BYTES each, a multiple of 1 KB)
  SharedCtl<STAGES> *ctl = reinterpret_cast<SharedCtl<STAGES> *>(base + STAGES * STAGE_BYTES);
  volatile int *abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&ctl->full[s], 1);
      tc::mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ctl->tfull[b], 1);
      tc::mbar_init(&ctl->tempty[b], 4);  // one arrival per epilogue warp
    }
    tc::mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_desc(&tma_w);
    tc::tma_prefetch_desc(&tma_x);
  }
  if (warp == 1) tc::tmem_alloc(&ctl->tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;
  pdl_trigger();
  pdl_wait();

  const int num_tiles = (V + BM - 1) / BM;
  const int k_iters = K / BK;
  const int first = (int)blockIdx.x, stride = (int)gridDim.x;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer ----
      const uint64_t pol_w = tc::policy_evict_first();  // W streams through once
      const uint64_t pol_x = tc::policy_evict_last();   // X is re-read by every tile
      int stage = 0;
      uint32_t phase = 0;
      int issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = -1;
      bool ok = true;
      for (int tile = first; ok && tile < num_tiles; tile += stride) {
        for (int kb = 0; kb < k_iters; ++kb) {
          if (!tc::mbar_wait(&ctl->empty[stage], phase ^ 1, abort)) { ok = false; break; }
          tc::mbar_expect_tx(&ctl->full[stage], STAGE_BYTES);  // W + X (rows past the end: zeros)
          tc::tma_load_2d(sA + stage * A_BYTES, &tma_w, kb * BK, tile * BM, &ctl->full[stage],
                          pol_w);
          tc::tma_load_2d(sB + stage * B_BYTES, &tma_x, kb * BK, 0, &ctl->full[stage], pol_x);
          issued[stage] = (int)phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      volatile int never = 0;  // drain: every copy issued has landed
      for (int s = 0; s < STAGES; ++s)
        if (issued[s] >= 0) tc::mbar_wait(&ctl->full[s], (uint32_t)issued[s], &never);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------- MMA issuer -----
      const uint32_t idesc = tc::idesc_bf16(BM, NS);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = first; ok && tile < num_tiles; tile += stride) {
        if (!tc::mbar_wait(&ctl->tempty[acc], acc_phase ^ 1, abort)) break;
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * NS);
        for (int kb = 0; kb < k_iters; ++kb) {
          if (!tc::mbar_wait(&ctl->full[stage], phase, abort)) { ok = false; break; }
          tc::fence_after_sync();
          const uint64_t a_desc = tc::smem_desc_sw128(sA + stage * A_BYTES);
          const uint64_t b_desc = tc::smem_desc_sw128(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)  // +32 B per 16-element K step
            tc::umma_bf16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc,
                          (kb | k) != 0 ? 1u : 0u);
          tc::umma_commit(&ctl->empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc::umma_commit(&ctl->tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      tc::umma_commit(&ctl->drain);  // drain: all MMAs issued have finished
      volatile int never = 0;
      tc::mbar_wait(&ctl->drain, 0, &never);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------- epilogue --------
    // TMEM lane = vocabulary row of the tile, column m = row m of X
    const int quarter = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = first; tile < num_tiles; tile += stride) {
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait(&ctl->tfull[acc], acc_phase, abort) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc::fence_after_sync();
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * NS);
      uint32_t r[NS];
      if constexpr (NS == 16) {
        tc::tmem_ld16(taddr, r);
      } else {
        tc::tmem_ld32(taddr, r);
      }
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();  // every lane's TMEM reads are done before the warp's single arrival
      if (lane == 0) tc::mbar_arrive(&ctl->tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
      const int v = tile * BM + quarter * 32 + lane;
      if (v < V) {
#pragma unroll
        for (int m = 0; m < NS; ++m)  // a warp stores 32 consecutive ids of row m
          if (m < M) C[(size_t)m * V + v] = __float2bfloat16_rn(__uint_as_float(r[m]));
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (ctl->abort && threadIdx.x == 0) dspark_set_status(DSPARK_ERR_TIMEOUT);
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// C [M, V] (bf16, row-major) = X [M, K] . W [V, K]^T for 1 <= M <= 32, K a
// multiple of 64; X, W and C 16-byte aligned.
template <int NS>
int launch_skinny(const void *X, const void *W, int M, int V, int K, bf16 *C,
                  cudaStream_t stream) {
  using G = SkinnyGeo<NS>;
  if (M < 1 || M > NS || K % BK != 0) return DSPARK_ERR_ARG;
  auto kernel = umma_skinny_kernel<NS>;
  CUtensorMap tw, tx;
  if (dspark_make_tmap_bf16(&tw, W, (uint64_t)V, (uint64_t)K, BM) != 0) return DSPARK_ERR_CUDA;
  if (dspark_make_tmap_bf16(&tx, X, (uint64_t)M, (uint64_t)K, NS) != 0) return DSPARK_ERR_CUDA;
  static DsparkPerDevice attr;
  if (dspark_per_device(attr, [&] {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)G::SMEM_BYTES) == cudaSuccess
                   ? 1
                   : -1;
      }) < 0)
    return DSPARK_ERR_CUDA;
  const int tiles = (V + BM - 1) / BM;
  const int sms = dspark_sm_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles < sms ? tiles : sms);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = G::SMEM_BYTES;
  cfg.stream = stream;
  if (cudaLaunchKernelEx(&cfg, kernel, tw, tx, M, V, K, C) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  dspark_count_launches(1);
  return DSPARK_OK;
}

}  // namespace gemm
