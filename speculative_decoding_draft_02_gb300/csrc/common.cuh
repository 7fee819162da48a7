// common.cuh — shared device helpers of the DSpark CUDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/dspark.h"

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// host-side plumbing shared by every translation unit (defined in abi.cu)
// ---------------------------------------------------------------------------
void dspark_count_launches(uint64_t n);
int dspark_sm_count();  // SMs of the current device (defined in lm_head.cu)

#define DSPARK_CHECK_LAUNCH()                                   \
  do {                                                          \
    cudaError_t _e = cudaGetLastError();                        \
    if (_e != cudaSuccess) return DSPARK_ERR_CUDA;              \
  } while (0)

static inline int dspark_dims_ok(const dspark_dims *d) {
  return d && d->R >= 1 && d->gamma >= 1 && d->gamma <= 32 && d->V >= 8 && d->V % 8 == 0 &&
         d->r >= 64 && d->r % 64 == 0 && d->d >= 64 && d->d % 64 == 0;
}

static inline size_t dspark_align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// One-time settings of a device (a kernel's shared-memory limit, an occupancy
// query): cudaFuncSetAttribute and the like act on the current device only, so
// a process that drives several GPUs needs them once per device.  `init` runs
// under the lock, with the device current, until it returns a value >= 0,
// which is then kept for that device; a negative value is returned and not kept.
constexpr int DSPARK_MAX_DEVICES = 64;
struct DsparkPerDevice {
  std::mutex mu;
  bool done[DSPARK_MAX_DEVICES];
  int value[DSPARK_MAX_DEVICES];
};
template <class F>
static inline int dspark_per_device(DsparkPerDevice &s, F init) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= DSPARK_MAX_DEVICES) return -1;
  std::lock_guard<std::mutex> lock(s.mu);
  if (!s.done[dev]) {
    const int v = init();
    if (v < 0) return v;
    s.value[dev] = v;
    s.done[dev] = true;
  }
  return s.value[dev];
}

// Launch with the programmatic stream-serialisation attribute (see pdl_wait).
template <class... KArgs, class... Args>
static inline cudaError_t dspark_launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                            size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// device status word: one per translation unit, read by dspark_device_status
// ---------------------------------------------------------------------------
// Each translation unit that launches kernels defines its own word with
// DSPARK_DECLARE_STATUS and exports a host reader; device code records the
// first problem it finds with dspark_set_status().
static __device__ void dspark_set_status(int code);

#define DSPARK_DECLARE_STATUS(name)                                        \
  static __device__ int name;                                              \
  static __device__ void dspark_set_status(int code) { atomicCAS(&name, 0, code); }

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): 10 rounds of
//   (c0,c1,c2,c3) <- (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0))
// with the key bumped by the Weyl constants between rounds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;  // one wide multiply: hi and lo
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c.w ^ k1, (uint32_t)p0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Philox with the ten round keys computed once (the key is the seed, fixed for
// a whole pass over the vocabulary).
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
  __device__ __forceinline__ explicit PhiloxKeys(uint64_t seed) {
    uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
#pragma unroll
    for (int i = 0; i < 10; ++i) {
      k0[i] = a;
      k1[i] = b;
      a += 0x9E3779B9u;
      b += 0xBB67AE85u;
    }
  }
  __device__ __forceinline__ uint4 operator()(uint4 c) const {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
      const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
      const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
      c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0[i], (uint32_t)p1,
                     (uint32_t)(p0 >> 32) ^ c.w ^ k1[i], (uint32_t)p0);
    }
    return c;
  }
};

// Random streams of the library's draw layout.  Every draw from a softmax is a
// two-level Gumbel-max over blocks of GUMBEL_BLOCK consecutive vocabulary ids:
// block b scores log(sum of its weights) + the Gumbel of id b in stream
// s + RNG_BLOCK_OFFSET, and inside the best block each id v scores its
// log-weight + the Gumbel of id v in stream s.  Max-stability of the Gumbel
// law makes this an exact sample (Maddison, Tarlow, Minka, "A* Sampling",
// NIPS 2014, top-down Gumbel processes).
// The residual's rejection trial q draws its proposal on stream RNG_TRIAL0 + 8q
// (ids; sampler blocks + RNG_BLOCK_OFFSET, super-blocks + RNG_SUPER_OFFSET) and
// its acceptance uniform on RNG_TRIAL0 + 8q + 1.
enum { RNG_DRAFT = 0, RNG_ACCEPT = 1, RNG_RESIDUAL = 2, RNG_BONUS = 3, RNG_BLOCK_OFFSET = 4,
       RNG_SUPER_OFFSET = 5, RNG_TRIAL0 = 16 };
constexpr int GUMBEL_BLOCK = 64;

// The four words for vocabulary slots 4*q .. 4*q+3 at (position, request, stream).
__device__ __forceinline__ uint4 rng_words4(uint64_t seed, uint32_t q, uint32_t pos,
                                            uint32_t req, uint32_t stream) {
  return philox4x32_10(make_uint4(q, pos, req, stream), (uint32_t)seed,
                       (uint32_t)(seed >> 32));
}

// u = ((w >> 9) + 1/2) * 2^-23: exact in float, strictly inside (0, 1).
__device__ __forceinline__ float rng_uniform(uint32_t w) {
  return fmaf((float)(w >> 9), 0x1p-23f, 0x1p-24f);
}

// Gumbel(0,1) from one word: -log(-log u).  The inner log needs full relative
// accuracy near u = 1 (the largest Gumbel values), the outer one does not.
__device__ __forceinline__ float rng_gumbel(uint32_t w) {
  const float e = -logf(rng_uniform(w));
  return -__logf(e);
}

__device__ __forceinline__ uint32_t uint4_get(const uint4 &v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// ---------------------------------------------------------------------------
// argmax / log-sum-exp partial state (one per row and vocabulary tile)
// ---------------------------------------------------------------------------
struct __align__(16) RowPartial {
  float m;       // max of the scaled logits s = l / tau       (sampling)
  float sum;     // sum exp(s - m)                               (sampling)
  float best;    // best decision score (logit, or s + Gumbel, or residual score)
  int32_t idx;   // vocabulary id of `best` (lowest on ties)
};

// Is (a, ia) a better decision than (b, ib)?  Larger score, ties to lower id.
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Combine an online (m, sum) log-sum-exp pair with another.
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; s = s2; return; }
  if (m2 > m) { s = s * __expf(m - m2) + s2; m = m2; }
  else        { s = s + s2 * __expf(m2 - m); }
}

// Warp-wide merge of (m, sum, best, idx, best_s); every lane gets the result.
__device__ __forceinline__ void warp_merge(float &m, float &s, float &best, int &idx,
                                           float &bs) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    const float bs2 = __shfl_xor_sync(0xffffffffu, bs, o);
    lse_merge(m, s, m2, s2);
    if (better(b2, i2, best, idx)) { best = b2; idx = i2; bs = bs2; }
  }
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialisation attribute may start while its predecessor in the stream
// still runs; pdl_wait() returns once that predecessor has completed and its
// memory is visible (immediately when there is no such predecessor), and
// pdl_trigger() lets the successor's launch begin.  Every kernel of the library
// triggers only after it is resident and never waits on its successor, so a
// chain of them cannot deadlock.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 2^x with the hardware approximation (flushes subnormal results to zero).
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// acc + the dot product of eight bf16 pairs packed in two 16-byte words
__device__ __forceinline__ float dot8_bf16(const uint4 a, const uint4 b, float acc) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    acc = fmaf(bf16_lo(av[t]), bf16_lo(bv[t]), acc);
    acc = fmaf(bf16_hi(av[t]), bf16_hi(bv[t]), acc);
  }
  return acc;
}
