// schedule.cu — a5-a7: the hardware-aware prefix scheduler.
//
// "DSpark 深度解读" §二 设计二 (Hardware-Aware Prefix Scheduler): prefix survival
// a_{r,j} = prod_{i<=j} c_{r,i}; all candidate extensions sorted globally by a
// descending; admitting K of them gives verify batch B = R + K and expected
// accepted tokens tau = R + S_K (S_K = sum of the admitted a), and the system
// throughput Theta = tau * SPS(B).  The theoretical greedy admission stops at
// the first K where Theta stops increasing (non-anticipating); §三 挑战2 drops
// that break and searches every budget because measured SPS(B) curves are
// stair-stepped; §三 挑战1 admits a capacity K fixed ahead of time (top-K), in
// production the capacity that the unconstrained search found two rounds
// earlier (asynchronous mode, a two-slot ring of predictions on the device).
//
// One CTA of 1024 threads: f32 survival products, a sort of composite keys
// (~bits(a) << 32 | id) so that ties go to the lower (request, position) -- a
// merge of the per-request runs (each already in order) up to 8192 keys, a
// bitonic sort above -- a fixed-point block scan of the sorted products and the
// Theta search.
#include "common.cuh"

DSPARK_DECLARE_STATUS(s_status_sched)

namespace {

constexpr int SCHED_THREADS = 1024;
constexpr int SCHED_MAX = 16384;
// Least sorted slots per scanning thread.  Each thread's Theta products form
// one dependent chain of f64 conversions and multiplies, so short chains on
// more warps win: 4 slots took the V4-shaped schedule (1280 candidates) from
// 34.3-34.6 to 29.6-30.6 us, and the 512-candidate one from 27-28 to 23 us.
constexpr int SCAN_PER = 4;

// S_K is summed in fixed point with 2^-48 units: every survival product a in
// [0, 1] rounded to the nearest unit, then exact 64-bit integer sums, so the
// order of the additions does not matter and no f64 addition (slow to issue
// and long in latency on this part) lies on a dependency chain.  Each term is
// off by at most 2^-49, so R + S_K is within gamma * 2^-49 of the exact sum
// relative to it.  R (1 + gamma) <= 2^15 keeps every sum below 2^63.
constexpr int FIX_BITS = 48;

// a (f32, 0 <= a <= 1) in 2^-48 units, rounded to nearest, with integer ops.
__device__ __forceinline__ unsigned long long to_fix(float a) {
  const uint32_t u = __float_as_uint(a);
  const int e = (int)(u >> 23) & 0xff;
  const int sh = e - (150 - FIX_BITS);  // a * 2^48 = m * 2^(e - 150 + 48)
  if (e == 0 || sh < -24) return 0ull;  // below half a unit (m < 2^24)
  const unsigned long long m = (u & 0x7fffffu) | 0x800000u;
  if (sh >= 0) return m << sh;          // a <= 1: sh <= 25
  return (m + (1ull << (-sh - 1))) >> (-sh);
}

// Theta(K) = (R + S_K) * SPS(R + K), with spsK[K] = SPS(R + K) and RS = R + S_K
// in 2^-48 units.
__device__ __forceinline__ double theta_at(long K, unsigned long long RS, const float *spsK) {
  return (double)RS * ((double)spsK[K] * 0x1p-48);
}

// A signed 64-bit key that orders doubles as `<` does (-0 equal to +0); NaN
// takes the least key, so it never wins the argmax.
__device__ __forceinline__ long long theta_key(double th) {
  const long long b = __double_as_longlong(th);
  if ((b & 0x7fffffffffffffffLL) > 0x7ff0000000000000LL) return (long long)0x8000000000000000ULL;
  if (((unsigned long long)b << 1) == 0ull) return 0;  // +0 and -0
  return b >= 0 ? b : (b ^ 0x7fffffffffffffffLL);
}

template <int E>
__global__ void __launch_bounds__(SCHED_THREADS) schedule_kernel(
    const float *__restrict__ conf, int R, int gamma, const float *__restrict__ sps, int mode,
    int k_fixed, int n_pad, int32_t *__restrict__ len, int32_t *__restrict__ K_out,
    double *__restrict__ theta_out, float *__restrict__ a_out, int32_t *__restrict__ order_out,
    int32_t *__restrict__ k_ring) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // keys [n_pad] (merge sort: and a second buffer of n_pad), then cnt [R]
  unsigned long long *keys = reinterpret_cast<unsigned long long *>(smem_raw);
  int32_t *cnt = reinterpret_cast<int32_t *>(keys + (E == 0 ? 2 * n_pad : n_pad));
  __shared__ unsigned long long warp_tot[32];
  __shared__ long long red_val[32];
  __shared__ long red_k[32];
  __shared__ long s_K;
  __shared__ double s_theta;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = R * gamma;
  pdl_trigger();
  pdl_wait();  // the confidences come from the draft

  // a5: survival products, f32 left to right; keys for the global order.  The
  // merge-sort form first brings the confidences into shared memory with one
  // coalesced pass (its second key buffer is free until the sort).
  const float *cs = conf;
  if constexpr (E == 0) {
    float *stage = reinterpret_cast<float *>(keys + n_pad);
    for (int id = tid; id < n; id += SCHED_THREADS) stage[id] = conf[id];
    __syncthreads();
    cs = stage;
  }
  for (int i = tid; i < R; i += SCHED_THREADS) {
    float a = 1.f;
    for (int j = 0; j < gamma; ++j) {
      float c = cs[(size_t)i * gamma + j];
      if (!(c >= 0.f && c <= 1.f)) {  // NaN or outside [0, 1]
        dspark_set_status(DSPARK_ERR_ARG);
        c = c > 1.f ? 1.f : 0.f;
      }
      a = (j == 0) ? c : __fmul_rn(a, c);
      const int id = i * gamma + j;
      if (a_out) a_out[id] = a;
      keys[id] = ((unsigned long long)(~__float_as_uint(a)) << 32) | (unsigned)id;
    }
    cnt[i] = 0;
  }
  for (int i = n + tid; i < n_pad; i += SCHED_THREADS) keys[i] = ~0ull;
  __syncthreads();

  const float *spsK = sps + R - 1;  // spsK[K] = SPS(R + K), K = 0..n
  if constexpr (E == 0) {
    // a6 as a merge sort.  A request's keys are already in order (a_{r,j} does
    // not increase with j and ids increase), so the R runs of gamma keys are
    // merged pairwise, log2(R) levels.  Keys are unique (the id is in the low
    // bits): a key's place in the merged run is its index in its own run plus
    // the number of smaller keys in the partner run, found by binary search.
    unsigned long long *src = keys, *dst = keys + n_pad;
    for (int L = gamma; L < n; L <<= 1) {
      for (int p = tid; p < n; p += SCHED_THREADS) {
        const int a0 = p / (2 * L) * (2 * L), b0 = a0 + L;
        const unsigned long long x = src[p];
        int lo, hi, own;
        if (p < b0) { lo = b0; hi = min(b0 + L, n); own = p - a0; }  // x in the left run
        else        { lo = a0; hi = b0;             own = p - b0; }  // x in the right run
        int l = lo, h = hi > lo ? hi : lo;  // first slot of the partner run holding a key >= x
        while (l < h) {
          const int m = (l + h) >> 1;
          if (src[m] < x) l = m + 1;
          else h = m;
        }
        dst[a0 + own + (l - lo)] = x;
      }
      __syncthreads();
      unsigned long long *t = src;
      src = dst;
      dst = t;
    }
    keys = src;  // the sorted keys; the other buffer is free again
    float *sp = reinterpret_cast<float *>(dst);
    for (int K = tid; K <= n; K += SCHED_THREADS) sp[K] = sps[R + K - 1];
    spsK = sp;
    __syncthreads();
  } else {
  // a6: bitonic sort, ascending keys = descending a, ties by ascending id.
  // Thread t holds keys [t*E, t*E + E) in registers (E = n_pad / 1024, at
  // least 1; when n_pad < 1024 the slots past n_pad hold the largest key and
  // only ever meet each other, since a stride below n_pad never crosses it).
  // Partners closer than E are in the thread, closer than 32 E in the warp
  // (shuffles); only the wider strides go through shared memory (n_pad keys).
  {
    unsigned long long k[E > 0 ? E : 1];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = tid * E + e;
      k[e] = i < n_pad ? keys[i] : ~0ull;
    }
    for (int size = 2; size <= n_pad; size <<= 1) {
      int stride = size >> 1;
      if (stride >= 32 * E) {
        __syncthreads();  // every thread is done reading keys[] before it is rewritten
#pragma unroll
        for (int e = 0; e < E; ++e)
          if (tid * E + e < n_pad) keys[tid * E + e] = k[e];
        __syncthreads();
        for (; stride >= 32 * E; stride >>= 1) {
          for (int t = tid; t < n_pad / 2; t += SCHED_THREADS) {
            const int lo = 2 * t - (t & (stride - 1));
            const int hi = lo + stride;
            const bool up = ((lo & size) == 0);
            const unsigned long long x = keys[lo], y = keys[hi];
            if ((x > y) == up) { keys[lo] = y; keys[hi] = x; }
          }
          __syncthreads();
        }
#pragma unroll
        for (int e = 0; e < E; ++e) k[e] = tid * E + e < n_pad ? keys[tid * E + e] : ~0ull;
      }
      for (; stride >= E; stride >>= 1) {  // partner in lane ^ (stride / E), same slot
        const int lo_bit = stride / E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = tid * E + e;
          const unsigned long long y = __shfl_xor_sync(0xffffffffu, k[e], lo_bit);
          const bool lower = (i & stride) == 0;  // i is the lower index of its pair
          const bool up = (i & size) == 0;
          // ascending pairs keep the smaller key at the lower index
          const bool take_min = lower == up;
          k[e] = take_min ? (y < k[e] ? y : k[e]) : (y > k[e] ? y : k[e]);
        }
      }
      // both partners in this thread: strides stride, stride / 2, ..., 1 (all
      // below E), unrolled over compile-time strides so k[] stays in registers
#pragma unroll
      for (int st = E / 2; st >= 1; st >>= 1) {
        if (st > stride) continue;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & st) != 0) continue;
          const int i = tid * E + e;
          const bool up = (i & size) == 0;
          const unsigned long long x = k[e], y = k[e + st];
          if ((x > y) == up) { k[e] = y; k[e + st] = x; }
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = tid * E + e;
      if (i < n_pad) keys[i] = k[e];
    }
    __syncthreads();
  }
  }

  // a7: S_K by a block scan in fixed point; thread t owns sorted slots
  // [t*per, (t+1)*per).  The slots go to as few warps as give each thread at
  // least SCAN_PER of them; only those warps (`scanner`, warp-uniform) scan
  // and evaluate Theta, whose f64 products are independent of one another.
  using u64 = unsigned long long;
  const int per = max((n_pad + SCHED_THREADS - 1) / SCHED_THREADS, SCAN_PER);
  const int beg = tid * per;
  const int scan_warps = ((n + per - 1) / per + 31) / 32;
  const bool scanner = warp < scan_warps;
  auto a_at = [&](int p) { return __uint_as_float(~(unsigned)(keys[p] >> 32)); };
  u64 incl = 0;
  if (scanner) {
    u64 local = 0;
    for (int p = beg; p < beg + per && p < n; ++p) local += to_fix(a_at(p));
    // inclusive scan of `local` over the warp
    incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const u64 y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
  }
  __syncthreads();
  if (warp == 0) {
    const u64 w = lane < scan_warps ? warp_tot[lane] : 0ull;
    u64 wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const u64 y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
  }
  __syncthreads();
  const u64 R_fix = (u64)R << FIX_BITS;
  u64 RS_beg = R_fix;  // R + S_{beg}

  // Theta over K = beg .. beg+per (K = 0 handled by thread 0)
  long long best = (long long)0x8000000000000000ULL;  // threads past the end never win
  long bestK = 0x7fffffffffffffffL;
  long firstDrop = 0x7fffffffffffffffL;  // smallest K with Theta(K+1) > Theta(K) false
  if (scanner) {
    u64 excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0ull;
    RS_beg = R_fix + warp_tot[warp] + excl;
    u64 RS = RS_beg;
    double prevTheta = 0.0;
    if (beg <= n) {  // sps[R + K - 1] exists for K <= n only
      prevTheta = theta_at(beg, RS, spsK);
      best = theta_key(prevTheta);
      bestK = beg;
    }
    for (int p = beg; p < beg + per && p < n; ++p) {
      RS += to_fix(a_at(p));
      const long K = p + 1;
      const double th = theta_at(K, RS, spsK);
      const long long key = theta_key(th);
      if (key > best) { best = key; bestK = K; }
      // break admits K only while Theta strictly rises (a NaN stops it)
      if (!(th > prevTheta) && firstDrop > K - 1) firstDrop = K - 1;
      prevTheta = th;
    }
  }

  long K = 0;
  if (mode == DSPARK_SCHED_UNCONSTRAINED || mode == DSPARK_SCHED_ASYNC) {
    // argmax Theta, ties to the smallest K
    if (scanner) {
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const long long b2 = __shfl_xor_sync(0xffffffffu, best, o);
        const long k2 = __shfl_xor_sync(0xffffffffu, bestK, o);
        if (b2 > best || (b2 == best && k2 < bestK)) { best = b2; bestK = k2; }
      }
    }
    if (lane == 0) { red_val[warp] = best; red_k[warp] = bestK; }
    __syncthreads();
    if (warp == 0) {
      best = lane < scan_warps ? red_val[lane] : (long long)0x8000000000000000ULL;
      bestK = lane < scan_warps ? red_k[lane] : 0x7fffffffffffffffL;
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const long long b2 = __shfl_xor_sync(0xffffffffu, best, o);
        const long k2 = __shfl_xor_sync(0xffffffffu, bestK, o);
        if (b2 > best || (b2 == best && k2 < bestK)) { best = b2; bestK = k2; }
      }
      if (lane == 0) s_K = bestK;
    }
  } else if (mode == DSPARK_SCHED_BREAK) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const long k2 = __shfl_xor_sync(0xffffffffu, firstDrop, o);
      firstDrop = k2 < firstDrop ? k2 : firstDrop;
    }
    if (lane == 0) red_k[warp] = firstDrop;
    __syncthreads();
    if (warp == 0) {
      long f = red_k[lane];
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const long k2 = __shfl_xor_sync(0xffffffffu, f, o);
        f = k2 < f ? k2 : f;
      }
      if (lane == 0) s_K = f < n ? f : n;
    }
  } else {
    if (tid == 0) s_K = k_fixed < 0 ? 0 : (k_fixed > n ? n : k_fixed);
  }
  __syncthreads();
  if (mode == DSPARK_SCHED_ASYNC) {
    // admit the capacity predicted two rounds ago; this round's optimum s_K is
    // the prediction for round t + 2 and takes its slot
    if (tid == 0) {
      const int c = k_ring[2] & 1;
      const long use = k_ring[c];
      k_ring[c] = (int32_t)s_K;
      k_ring[2] = c ^ 1;
      s_K = use < 0 ? 0 : (use > n ? n : use);
    }
    __syncthreads();
  }
  K = s_K;
  if (K < 0 || K > n) K = 0;  // unreachable for finite tables; keeps every index in range

  // per-request lengths: count admitted candidates of each request
  for (int p = tid; p < K; p += SCHED_THREADS) {
    const int id = (int)(keys[p] & 0xffffffffu);
    atomicAdd(&cnt[id / gamma], 1);
  }
  if (order_out)
    for (int p = tid; p < n; p += SCHED_THREADS) order_out[p] = (int)(keys[p] & 0xffffffffu);
  // Theta(K): the owner of slot K recomputes it from its scan segment
  if (tid == 0 && K == 0) s_theta = theta_at(0, R_fix, spsK);
  if (K > beg && K <= beg + per) {  // the owner of slot K - 1 (a scanner thread)
    u64 RS2 = RS_beg;
    for (int p = beg; p < K; ++p) RS2 += to_fix(a_at(p));
    s_theta = theta_at(K, RS2, spsK);
  }
  __syncthreads();
  for (int i = tid; i < R; i += SCHED_THREADS) len[i] = cnt[i];
  if (tid == 0) {
    *K_out = (int32_t)K;
    *theta_out = s_theta;
  }
}

}  // namespace

namespace {
int launch_schedule(const float *conf, int32_t R, int32_t gamma, const float *sps, int32_t n_sps,
                    int32_t mode, int32_t k_fixed, int32_t *len, int32_t *K_out,
                    double *theta_out, float *a_out, int32_t *order_out, int32_t *k_ring,
                    cudaStream_t stream) {
  if (!conf || !sps || !len || !K_out || !theta_out || R < 1 || gamma < 1 || gamma > 32)
    return DSPARK_ERR_ARG;
  const long n = (long)R * gamma;
  if (n > SCHED_MAX) return DSPARK_ERR_ARG;
  if ((long)n_sps < (long)R * (gamma + 1)) return DSPARK_ERR_SPS_SHORT;
  int n_pad = 2;
  while (n_pad < n) n_pad <<= 1;
  // up to 8192 candidates: merge sort (two key buffers); beyond: bitonic sort
  const bool merge = n_pad <= 8192;
  const size_t smem = sizeof(unsigned long long) * n_pad * (merge ? 2 : 1) + sizeof(int32_t) * R;
  const int smem_max = (int)(sizeof(unsigned long long) * SCHED_MAX + sizeof(int32_t) * SCHED_MAX);
  static DsparkPerDevice attr;
  if (dspark_per_device(attr, [&] {
        for (auto k : {schedule_kernel<0>, schedule_kernel<1>, schedule_kernel<2>,
                       schedule_kernel<4>, schedule_kernel<8>, schedule_kernel<16>})
          if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) !=
              cudaSuccess)
            return -1;
        return 1;
      }) < 0)
    return DSPARK_ERR_CUDA;
  // keys per thread: n_pad / 1024, at least one
  auto kernel = merge        ? schedule_kernel<0>
              : n_pad <= 1024 ? schedule_kernel<1>
              : n_pad == 2048 ? schedule_kernel<2>
              : n_pad == 4096 ? schedule_kernel<4>
              : n_pad == 8192 ? schedule_kernel<8>
                              : schedule_kernel<16>;
  // launch and set-up overlap the tail of the draft (the kernel waits for it)
  if (dspark_launch_pdl(kernel, dim3(1), dim3(SCHED_THREADS), smem, stream, conf, R, gamma, sps,
                        mode, k_fixed, n_pad, len, K_out, theta_out, a_out, order_out,
                        k_ring) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  dspark_count_launches(1);
  return DSPARK_OK;
}
}  // namespace

extern "C" int dspark_schedule(const float *conf, int32_t R, int32_t gamma, const float *sps,
                               int32_t n_sps, int32_t mode, int32_t k_fixed, int32_t *len,
                               int32_t *K_out, double *theta_out, float *a_out,
                               int32_t *order_out, dspark_stream_t stream) {
  if (mode < DSPARK_SCHED_UNCONSTRAINED || mode > DSPARK_SCHED_FIXED_K) return DSPARK_ERR_ARG;
  return launch_schedule(conf, R, gamma, sps, n_sps, mode, k_fixed, len, K_out, theta_out, a_out,
                         order_out, nullptr, stream);
}

extern "C" int dspark_schedule_async(const float *conf, int32_t R, int32_t gamma,
                                     const float *sps, int32_t n_sps, int32_t *k_ring,
                                     int32_t *len, int32_t *K_out, double *theta_out,
                                     float *a_out, int32_t *order_out, dspark_stream_t stream) {
  if (!k_ring) return DSPARK_ERR_ARG;
  return launch_schedule(conf, R, gamma, sps, n_sps, DSPARK_SCHED_ASYNC, 0, len, K_out, theta_out,
                         a_out, order_out, k_ring, stream);
}

int dspark_status_sched(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, s_status_sched, sizeof(int)) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (clear) {
    const int z = 0;
    cudaMemcpyToSymbol(s_status_sched, &z, sizeof(int));
  }
  return v;
}
