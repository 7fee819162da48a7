// umma_gemm.cuh — persistent tcgen05 GEMM  D[M, N] = A[M, K] . B[N, K]^T with a
// pluggable epilogue that reads the f32 accumulator straight from TMEM.
//
// One CTA per SM, 64 + 32 * EPI_WARPS threads:
//   warp 0      one thread issues TMA loads of A (128 x 64) and B (256 x 64)
//               tiles into a STAGES-deep shared-memory ring;
//   warp 1      allocates TMEM (2 x 256 columns: a double-buffered 128 x 256 f32
//               accumulator) and one thread issues tcgen05.mma (M=128, N=256,
//               K=16 per instruction, 4 per 64-wide stage), committing each
//               stage back to the producer and each finished tile to the
//               epilogue;
//   warps 2..   the epilogue (EPI_WARPS = 4, 8 or 16): a thread owns one
//               accumulator row (its TMEM lane) and a contiguous slice of its
//               columns (256, 128 or 64), so a row-wise reduction over the
//               slice needs no shuffles.
// Tiles are visited m-fastest, so the CTAs working at the same time share one
// B tile (one read from HBM, the rest from L2).  Every wait is bounded; on
// timeout the CTA raises DSPARK_ERR_TIMEOUT, drains its own copies and MMAs,
// frees TMEM and exits.
#pragma once
#include "tcgen05.cuh"

namespace gemm {

constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr size_t SMEM_LIMIT = 232448;  // opt-in dynamic shared memory per CTA

// Tile geometry for an N-tile of BN columns (BN = 256 or 192): the ring holds
// as many 64-deep stages of A and B as fit, the double-buffered accumulator
// takes 2*BN TMEM columns (allocated as the next power of two).
template <int BN_>
struct Geo {
  static constexpr int BN = BN_;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (int)((SMEM_LIMIT - 1024 - 512) / STAGE_BYTES) > 6
                                    ? 6
                                    : (int)((SMEM_LIMIT - 1024 - 512) / STAGE_BYTES);
  static constexpr uint32_t TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
  static constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 512;
  static_assert(BN % 16 == 0 && BN >= 64 && BN <= 256, "UMMA N for M = 128");
};
constexpr int BN = 256;  // the default N-tile (LM head, greedy and residual passes)

template <int STAGES>
struct SharedCtl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Epi must provide
//   struct State;                         per-thread state kept across tiles
//   static constexpr bool kRowAffine;     keep each thread on one row when possible
//   static constexpr bool kStreamB;       B is read once: evict its tiles from L2 first
//   __device__ void prefetch(int m0, int n0, int row, int c0, int c1, State &) const
//       (called once, for the CTA's first tile, before its accumulator is
//        ready: start global loads)
//   __device__ void operator()(int m0, int n0, int row, uint32_t taddr, int c0, int c1,
//                              int next_m0, int next_n0, State &) const
//       (every epilogue thread, once per tile, for its row and column slice
//        [c0, c1); tcgen05.ld of each 32-column chunk must be warp-uniform;
//        next_m0 / next_n0 locate the CTA's next tile, -1 after the last, so
//        the loads for it can start while this one is processed)
//   __device__ void on_timeout() const.
template <class Epi, int EPI_WARPS, int BN_>
__global__ void __launch_bounds__(64 + 32 * EPI_WARPS, 1)
    umma_gemm_kernel(const __grid_constant__ CUtensorMap tma_a,
                     const __grid_constant__ CUtensorMap tma_b, int M, int N, int K,
                     const int *m_dev, int ksplit, Epi epi) {
  using G = Geo<BN_>;
  constexpr int BN = G::BN, STAGES = G::STAGES, B_BYTES = G::B_BYTES;
  constexpr int STAGE_BYTES = G::STAGE_BYTES;
  constexpr uint32_t TMEM_COLS = G::TMEM_COLS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = base;
  uint8_t *sB = base + STAGES * A_BYTES;
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
      tc::mbar_init(&ctl->tempty[b], EPI_WARPS);  // one arrival per epilogue warp
    }
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
  // everything above overlaps the previous kernel of the stream; A, the row
  // count, the epilogue's inputs and its outputs belong to the kernels around
  // this one
  pdl_trigger();
  pdl_wait();

  if (m_dev) {  // rows counted on the device by an earlier kernel (at most M)
    const int md = *m_dev;
    M = md < M ? (md > 0 ? md : 0) : M;
  }
  const int num_m = (M + BM - 1) / BM, num_n = (N + BN - 1) / BN;
  // split K (ksplit > 1): split s of a tile takes k blocks [s * k_iters, (s+1) *
  // k_iters) and hands its partial to the epilogue as rows s * num_m * BM + ...
  const int k_iters = K / BK / ksplit;
  // tile sequence: t -> (m block, n block), m fastest
  const int split_tiles = num_m * num_n;
  const int num_tiles = split_tiles * ksplit;
  const int first = (int)blockIdx.x;
  const int stride = (int)gridDim.x;
  auto coords = [&](int t, int &m_blk, int &n_blk) {
    const int u = t % split_tiles;
    m_blk = u % num_m;
    n_blk = u / num_m;
  };
  auto out_row0 = [&](int t, int m_blk) { return ((t / split_tiles) * num_m + m_blk) * BM; };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer ----
      const uint64_t pol_a = tc::policy_evict_last();   // A tiles are re-read
      // B: streamed once (LM head) or re-read by other M blocks and later steps
      const uint64_t pol_b =
          Epi::kStreamB ? tc::policy_evict_first() : tc::policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      int issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = -1;
      bool ok = true;
      for (int tile = first; ok && tile < num_tiles; tile += stride) {
        int m_blk, n_blk;
        coords(tile, m_blk, n_blk);
        const int kb0 = (tile / split_tiles) * k_iters;
        for (int kb = 0; kb < k_iters; ++kb) {
          if (!tc::mbar_wait(&ctl->empty[stage], phase ^ 1, abort)) { ok = false; break; }
          tc::mbar_expect_tx(&ctl->full[stage], STAGE_BYTES);  // A + B
          const int kx = (kb0 + kb) * BK;
          tc::tma_load_2d(sA + stage * A_BYTES, &tma_a, kx, m_blk * BM, &ctl->full[stage], pol_a);
          tc::tma_load_2d(sB + stage * B_BYTES, &tma_b, kx, n_blk * BN, &ctl->full[stage], pol_b);
          issued[stage] = (int)phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      // drain: every copy this thread issued has landed before the CTA exits
      volatile int never = 0;
      for (int s = 0; s < STAGES; ++s)
        if (issued[s] >= 0) tc::mbar_wait(&ctl->full[s], (uint32_t)issued[s], &never);
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
      for (int tile = first; ok && tile < num_tiles; tile += stride) {
        if (!tc::mbar_wait(&ctl->tempty[acc], acc_phase ^ 1, abort)) break;
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
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
      // drain: all MMAs issued by this thread have finished
      tc::umma_commit(&ctl->drain);
      volatile int never = 0;
      tc::mbar_wait(&ctl->drain, 0, &never);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------- epilogue --------
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    constexpr int SLICE = BN / (EPI_WARPS / 4);
    const int c0 = ((warp - 2) >> 2) * SLICE;
    int acc = 0;
    uint32_t acc_phase = 0;
    typename Epi::State st;
    if (first < num_tiles) {
      int m_blk, n_blk;
      coords(first, m_blk, n_blk);
      epi.prefetch(out_row0(first, m_blk), n_blk * BN, row, c0, c0 + SLICE, st);
    }
    for (int tile = first; tile < num_tiles; tile += stride) {
      int m_blk, n_blk;
      coords(tile, m_blk, n_blk);
      int next_m0 = -1, next_n0 = -1;
      if (tile + stride < num_tiles) {
        int nm;
        coords(tile + stride, nm, next_n0);
        next_m0 = out_row0(tile + stride, nm);
        next_n0 *= BN;
      }
      // one lane polls, then the warp proceeds together (tcgen05.ld is warp-wide)
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait(&ctl->tfull[acc], acc_phase, abort) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc::fence_after_sync();
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      epi(out_row0(tile, m_blk), n_blk * BN, row, taddr, c0, c0 + SLICE, next_m0, next_n0, st);
      tc::fence_before_sync();
      __syncwarp();  // every lane's TMEM reads are done before the warp's single arrival
      if (lane == 0) tc::mbar_arrive(&ctl->tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (ctl->abort && threadIdx.x == 0) epi.on_timeout();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// M rows of A are described to TMA; when m_dev is given the kernel processes
// only the first *m_dev of them (read on the device, so the count can come from
// an earlier kernel in the stream).
// ksplit > 1: K is split into ksplit equal parts, and the
// epilogue receives split s's partial of M block m as rows (s * num_m + m) * BM.
template <int EPI_WARPS, int BN_ = 256, class Epi>
int launch(const void *A, const void *B, int M, int N, int K, const Epi &epi,
           cudaStream_t stream, const int *m_dev = nullptr, bool pdl = false, int ksplit = 1) {
  if (ksplit < 1 || K % (BK * ksplit) != 0) return DSPARK_ERR_ARG;
  using G = Geo<BN_>;
  constexpr int BN = G::BN;
  static_assert(EPI_WARPS % 4 == 0 && EPI_WARPS >= 4 && EPI_WARPS <= 16 &&
                    BN % (EPI_WARPS / 4) == 0 && (BN / (EPI_WARPS / 4)) % 32 == 0,
                "epilogue warps: 4 per TMEM lane quarter group, slices of whole 32-column loads");
  auto kernel = umma_gemm_kernel<Epi, EPI_WARPS, BN_>;
  CUtensorMap ta, tb;
  if (dspark_make_tmap_bf16(&ta, A, (uint64_t)M, (uint64_t)K, BM) != 0) return DSPARK_ERR_CUDA;
  if (dspark_make_tmap_bf16(&tb, B, (uint64_t)N, (uint64_t)K, BN) != 0)
    return DSPARK_ERR_CUDA;
  static DsparkPerDevice attr;
  if (dspark_per_device(attr, [&] {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)G::SMEM_BYTES) == cudaSuccess
                   ? 1
                   : -1;
      }) < 0)
    return DSPARK_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[1];
  cfg.blockDim = dim3(64 + 32 * EPI_WARPS);
  cfg.dynamicSmemBytes = G::SMEM_BYTES;
  cfg.stream = stream;
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int sms = dspark_sm_count();
  const int tiles = num_m * num_n * ksplit;
  int grid = tiles < sms ? tiles : sms;
  // a multiple of the M-block count keeps every CTA (and epilogue thread) on one row block
  if (Epi::kRowAffine && grid > num_m) grid = grid / num_m * num_m;
  cfg.gridDim = dim3(grid);
  if (pdl) {  // may start while the previous kernel of the stream finishes
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
  }
  if (cudaLaunchKernelEx(&cfg, kernel, ta, tb, M, N, K, m_dev, ksplit, epi) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  dspark_count_launches(1);
  return DSPARK_OK;
}

}  // namespace gemm
