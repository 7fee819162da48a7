// umma_gemm_pair.cuh — the persistent tcgen05 GEMM on CTA pairs (.cta_group::2):
// D[M, N] = A[M, K] . B[N, K]^T with the epilogue interface of umma_gemm.cuh.
//
// A cluster of two CTAs (two SMs) computes one 256 x 256 tile at a time.  CTA
// rank q holds rows [128 q, 128 q + 128) of the tile's A and rows
// [128 q, 128 q + 128) of its B (the tile's N range split in halves), each in
// its own 7-stage ring of 32 KB stages, and receives accumulator rows
// [128 q, 128 q + 128) x all 256 columns in its own TMEM.  The rank-0 CTA
// issues tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16) for both; each MMA
// reads A from each CTA's own shared memory and B from both.  Per SM and per
// 64-deep k block that is 32 KB of operands instead of the 48 KB of the
// one-CTA kernel, for the same flops.
//
// Barriers: rank 0's producer arms rank 0's full barrier with the bytes of
// both CTAs, and both CTAs' TMA loads complete there (a copy may land before
// the barrier is armed: its phase cannot end while the arrival is pending);
// rank 0's commits arrive on both CTAs' empty and accumulator-full barriers;
// both CTAs' epilogue warps release an accumulator on rank 0's
// accumulator-empty barrier.  Every wait is bounded as in umma_gemm.cuh.
#pragma once
#include "umma_gemm.cuh"

namespace gemm {

struct PairGeo {
  static constexpr int BN = 256;         // N per pair tile
  static constexpr int BNH = BN / 2;     // B rows each CTA holds
  static constexpr int B_BYTES = BNH * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB
  // as many as fit (7 x 32 KB + 1.5 KB of 227 KB): against six, 1% faster at
  // 512, 1280 and 7168 rows of a V = 129280-151936 LM head
  static constexpr int STAGES = 7;
  static constexpr uint32_t TMEM_COLS = 512;             // 2 x 256 f32 columns
  static constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 512;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "ring fits the opt-in shared memory");
};

// After an abnormal exit of the producer loop: the TMA loads this CTA issued
// complete on the peer's barrier, which it cannot poll, so it waits a fixed,
// generous time for them to land before its shared memory may go away.
__device__ __forceinline__ void pair_settle() {
  const uint64_t t0 = tc::globaltimer();
  while (tc::globaltimer() - t0 < 2000000ull) {}  // 2 ms
}

template <class Epi, int EPI_WARPS>
__global__ void __launch_bounds__(64 + 32 * EPI_WARPS, 1)
    umma_gemm_pair_kernel(const __grid_constant__ CUtensorMap tma_a,
                          const __grid_constant__ CUtensorMap tma_b, int M, int N, int K,
                          const int *m_dev, Epi epi) {
  using G = PairGeo;
  constexpr int BN = G::BN, BNH = G::BNH, STAGES = G::STAGES, B_BYTES = G::B_BYTES;
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
  const uint32_t rank = tc::cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&ctl->full[s], 1);  // rank 0's producer (rank 0's copy is the one used)
      tc::mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ctl->tfull[b], 1);
      tc::mbar_init(&ctl->tempty[b], 2 * EPI_WARPS);  // one arrival per epilogue warp of each CTA
    }
    tc::mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_desc(&tma_a);
    tc::tma_prefetch_desc(&tma_b);
  }
  if (warp == 1) tc::tmem_alloc_pair(&ctl->tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();  // both CTAs' barriers exist before any remote arrive or multicast
  tc::fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;
  pdl_trigger();
  pdl_wait();

  if (m_dev) {
    const int md = *m_dev;
    M = md < M ? (md > 0 ? md : 0) : M;
  }
  const int num_m = (M + BM - 1) / BM, num_n = (N + BN - 1) / BN;
  const int num_mp = (num_m + 1) / 2;
  const int num_tiles = num_mp * num_n;
  const int k_iters = K / BK;
  const int first = (int)(blockIdx.x >> 1), stride = (int)(gridDim.x >> 1);
  // Tiles go M-pair-fastest within groups of gp pairs whose A rows (256 K
  // bf16 per pair) fit in 32 MiB of L2; a group visits every N tile before the
  // next starts.  Up to 32 MiB of A (every workload but the largest) this is
  // the plain M-fastest order.  At 7168 rows (A 98 MiB, two groups) it took
  // the LM head from 8.95-8.97 to 8.25-8.28 ms (same box, 100 calls each); the
  // pairs of an N tile still drift apart and re-read most B tiles from HBM
  // (26.3 against 28.1 GB per launch).
  const long a_pair = 2L * BM * K * 2;
  const int n_groups = (int)(((long)num_mp * a_pair + (32L << 20) - 1) / (32L << 20));
  const int gp = (num_mp + n_groups - 1) / n_groups;  // pairs per group
  auto coords = [&](int t, int &m_blk, int &n_blk) {
    const int g = t / (gp * num_n);
    const int u = t - g * gp * num_n;
    const int gsz = num_mp - g * gp < gp ? num_mp - g * gp : gp;  // the last group may be smaller
    m_blk = 2 * (g * gp + u % gsz) + (int)rank;
    n_blk = u / gsz;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer ----
      // B lines are read by the clusters on each M-block pair of an N tile, at
      // different times: they must survive in L2 until the last of them
      const uint64_t pol_a = tc::policy_evict_last();
      const uint64_t pol_b = tc::policy_evict_normal();
      const uint32_t full0 = tc::map_to_rank0(&ctl->full[0]);  // rank 0's full barriers
      int stage = 0;
      uint32_t phase = 0;
      int issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = -1;
      bool ok = true;
      for (int tile = first; ok && tile < num_tiles; tile += stride) {
        int m_blk, n_blk;
        coords(tile, m_blk, n_blk);
        for (int kb = 0; kb < k_iters; ++kb) {
          if (!tc::mbar_wait_spin(&ctl->empty[stage], phase ^ 1, abort)) { ok = false; break; }
          const uint32_t full = full0 + 8u * (uint32_t)stage;
          if (leader) tc::mbar_expect_tx(&ctl->full[stage], 2 * STAGE_BYTES);  // both CTAs
          tc::tma_load_2d_pair(sA + stage * A_BYTES, &tma_a, kb * BK, m_blk * BM, full, pol_a);
          tc::tma_load_2d_pair(sB + stage * B_BYTES, &tma_b, kb * BK, n_blk * BN + (int)rank * BNH,
                               full, pol_b);
          issued[stage] = (int)phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (leader) {
        // rank 0's full barriers see both CTAs' copies land
        volatile int never = 0;
        for (int s = 0; s < STAGES; ++s)
          if (issued[s] >= 0) tc::mbar_wait_spin(&ctl->full[s], (uint32_t)issued[s], &never);
      } else if (!ok) {
        pair_settle();
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------- MMA issuer -----
      const uint32_t idesc = tc::idesc_bf16(2 * BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = first; ok && tile < num_tiles; tile += stride) {
        if (!tc::mbar_wait_spin(&ctl->tempty[acc], acc_phase ^ 1, abort)) break;
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < k_iters; ++kb) {
          if (!tc::mbar_wait_spin(&ctl->full[stage], phase, abort)) { ok = false; break; }
          tc::fence_after_sync();
          const uint64_t a_desc = tc::smem_desc_sw128(sA + stage * A_BYTES);
          const uint64_t b_desc = tc::smem_desc_sw128(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc::umma_bf16_pair(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc,
                               (kb | k) != 0 ? 1u : 0u);
          tc::umma_commit_pair_mcast(&ctl->empty[stage], (uint16_t)0x3);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc::umma_commit_pair_mcast(&ctl->tfull[acc], (uint16_t)0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      tc::umma_commit_pair_mcast(&ctl->drain, (uint16_t)0x1);
      volatile int never = 0;
      tc::mbar_wait_spin(&ctl->drain, 0, &never);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------- epilogue --------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    constexpr int SLICE = BN / (EPI_WARPS / 4);
    const int c0 = ((warp - 2) >> 2) * SLICE;
    const uint32_t tempty0 = tc::map_to_rank0(&ctl->tempty[0]);
    int acc = 0;
    uint32_t acc_phase = 0;
    typename Epi::State st;
    if (first < num_tiles) {
      int m_blk, n_blk;
      coords(first, m_blk, n_blk);
      epi.prefetch(m_blk * BM, n_blk * BN, row, c0, c0 + SLICE, st);
    }
    for (int tile = first; tile < num_tiles; tile += stride) {
      int m_blk, n_blk;
      coords(tile, m_blk, n_blk);
      int next_m0 = -1, next_n0 = -1;
      if (tile + stride < num_tiles) {
        coords(tile + stride, next_m0, next_n0);
        next_m0 *= BM;
        next_n0 *= BN;
      }
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait_spin(&ctl->tfull[acc], acc_phase, abort) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc::fence_after_sync();
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      epi(m_blk * BM, n_blk * BN, row, taddr, c0, c0 + SLICE, next_m0, next_n0, st);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_cluster(tempty0 + 8u * (uint32_t)acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();  // no remote arrive, copy or commit still targets either CTA
  if (ctl->abort && threadIdx.x == 0) epi.on_timeout();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// The pair GEMM over M rows (at most *m_dev when given).  Clusters of two CTAs;
// as many clusters as fit, each walking pair tiles (M block pairs fastest).
template <int EPI_WARPS, class Epi>
int launch_pair(const void *A, const void *B, int M, int N, int K, const Epi &epi,
                cudaStream_t stream, const int *m_dev = nullptr, bool pdl = false) {
  using G = PairGeo;
  static_assert(EPI_WARPS % 4 == 0 && EPI_WARPS >= 4 && EPI_WARPS <= 16 &&
                    (G::BN / (EPI_WARPS / 4)) % 32 == 0,
                "epilogue warps: 4 per TMEM lane quarter group, slices of whole 32-column loads");
  auto kernel = umma_gemm_pair_kernel<Epi, EPI_WARPS>;
  CUtensorMap ta, tb;
  if (dspark_make_tmap_bf16(&ta, A, (uint64_t)M, (uint64_t)K, BM) != 0) return DSPARK_ERR_CUDA;
  if (dspark_make_tmap_bf16(&tb, B, (uint64_t)N, (uint64_t)K, G::BNH) != 0) return DSPARK_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 2;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(64 + 32 * EPI_WARPS);
  cfg.dynamicSmemBytes = G::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  // the shared-memory limit and the number of co-resident clusters, per device
  static DsparkPerDevice clusters;
  const int max_clusters = dspark_per_device(clusters, [&] {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)G::SMEM_BYTES) != cudaSuccess)
      return -1;
    cudaLaunchConfig_t q = cfg;
    q.gridDim = dim3(2 * (dspark_sm_count() / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &q) != cudaSuccess || n < 1) return -1;
    return n;
  });
  if (max_clusters < 1) return DSPARK_ERR_CUDA;
  const int num_m = (M + BM - 1) / BM;
  const int tiles = ((num_m + 1) / 2) * ((N + G::BN - 1) / G::BN);
  cfg.gridDim = dim3(2 * (tiles < max_clusters ? tiles : max_clusters));
  if (pdl) {
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  if (cudaLaunchKernelEx(&cfg, kernel, ta, tb, M, N, K, m_dev, epi) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  dspark_count_launches(1);
  return DSPARK_OK;
}

}  // namespace gemm
