// Device helpers shared by the kernels of liblayer_rnn.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace lr {

typedef __nv_bfloat16 bf16;

// device status word values (same numbers as rnn_status_t)
constexpr int kDevOk = 0;
constexpr int kDevTimeout = 6;
constexpr int kDevCheck = 8;   // a kernel's own index check failed (access skipped)

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

// element load that bypasses L1 (data written by other CTAs in this launch)
__device__ __forceinline__ float ldcg_f(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float ldcg_f(const bf16* p) {
  unsigned short u = __ldcg(reinterpret_cast<const unsigned short*>(p));
  return __uint_as_float(((unsigned)u) << 16);
}

__device__ __forceinline__ float load_any(const void* p, int64_t i, int is_bf16) {
  return is_bf16 ? ldcg_f(reinterpret_cast<const bf16*>(p) + i)
                 : ldcg_f(reinterpret_cast<const float*>(p) + i);
}

// element e of a 16-byte vector of fp32 (e < 4) or bf16 (e < 8) values
__device__ __forceinline__ float lane_f32(const uint4& v, int e) {
  const unsigned w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
  return __uint_as_float(w);
}
__device__ __forceinline__ float lane_bf16(const uint4& v, int e) {
  const int q = e >> 1;
  const unsigned w = q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
  return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
}

__device__ __forceinline__ float sigmoidf_(float a) { return 1.0f / (1.0f + expf(-a)); }

// The gate nonlinearities of the tensor-core recurrent kernels with the
// hardware exponential (ex2.approx, a few ulp) and approximate division, at a
// relative error near 1e-6 or better.  sigmoid = 1 / (1 + e^{-a}) has no
// cancellation.  tanh = 1 - 2 / (1 + e^{2a}) cancels near 0, so |a| < 1/4 takes
// the Taylor series of tanh to a^9 (x - x^3/3 + 2x^5/15 - 17x^7/315 +
// 62x^9/2835; the first omitted term, 1382x^11/155925, is below 2e-9 there).
// Large |a| saturates cleanly: e^{|a|} overflows to inf and the division
// gives 0.
__device__ __forceinline__ float sigmoid_fast(float a) {
  return __fdividef(1.0f, 1.0f + __expf(-a));
}
__device__ __forceinline__ float tanh_fast(float a) {
  const float big = 1.0f - __fdividef(2.0f, 1.0f + __expf(2.0f * a));
  const float x2 = a * a;
  float poly = fmaf(x2, 62.0f / 2835.0f, -17.0f / 315.0f);
  poly = fmaf(x2, poly, 2.0f / 15.0f);
  poly = fmaf(x2, poly, -1.0f / 3.0f);
  const float small = fmaf(a * x2, poly, a);
  return fabsf(a) < 0.25f ? small : big;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_volatile_int(const int* p) {
  return *reinterpret_cast<const volatile int*>(p);
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
  unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// 16-byte load that bypasses L1 (data written by other blocks of this launch)
__device__ __forceinline__ uint4 ldcg16(const void* p) {
  return __ldcg(reinterpret_cast<const uint4*>(p));
}

// Wait until *f >= value: spin on relaxed loads, finish with one acquire load.
// Bounded: gives up once `timeout_ns` has passed or another block has recorded
// a failure in *status (then records kDevTimeout itself and returns false).
__device__ __forceinline__ bool wait_flag(const unsigned* f, unsigned value, int* status,
                                          long long timeout_ns, int spin_ns) {
  if (ld_relaxed_gpu(f) < value) {
    const unsigned long long t0 = globaltimer_ns();
    unsigned it = 0;
    while (ld_relaxed_gpu(f) < value) {
      if (spin_ns > 0) __nanosleep(spin_ns);
      if ((++it & 31u) == 0) {
        if (ld_volatile_int(status) != kDevOk) return false;
        if ((long long)(globaltimer_ns() - t0) > timeout_ns) {
          atomicCAS(status, kDevOk, kDevTimeout);
          return false;
        }
      }
    }
  }
  (void)ld_acquire_gpu(f);
  return true;
}

// Publish `value` in this block's flag after every thread's stores of the step:
// call after __syncthreads, from one thread.  The release store is cumulative
// over the writes the barrier ordered before it, so no separate fence.
__device__ __forceinline__ void publish_flag(unsigned* f, unsigned value) {
  st_release_gpu(f, value);
}

// The lanes of a warp wait, together, for the flags of blocks lo..hi
// (inclusive; block b's flag at flags[b * stride]) to reach `value`.  Bounded
// like wait_flag; returns false (in every lane) if any wait gave up.
// - At most one flag a lane: each lane runs wait_flag (measured fastest there).
// - More: lane l polls flags lo + l + 32 j with all of its loads in flight at
//   once and re-polls only the flags not yet set, so a warp sees up to 256 set
//   flags in one round trip to L2 (one after another costs two round trips a
//   flag: the relaxed load, then the acquire load).
// - The acquire side of the writers' releases: with up to two flags a lane, an
//   acquire load of each flag; with more, one gpu-scope acquire fence after
//   the relaxed loads that saw the values.  The fence also waits for the
//   lane's own stores and loads still in flight, so a caller with a wide range
//   issues its prefetches after the wait or from other warps.
__device__ __forceinline__ bool warp_wait_flags(const unsigned* flags, int stride, int lo, int hi,
                                                unsigned value, int* status,
                                                long long timeout_ns, int spin_ns) {
  constexpr int kPer = 8;
  const int lane = threadIdx.x & 31;
  bool ok = true;
  if (hi - lo < 32) {  // at most one flag a lane
    if (lo + lane <= hi)
      ok = wait_flag(flags + (size_t)(lo + lane) * stride, value, status, timeout_ns, spin_ns);
    return __all_sync(0xffffffffu, ok);
  }
  for (int base = lo; base <= hi && ok; base += 32 * kPer) {
    unsigned pending = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (base + lane + 32 * j <= hi) pending |= 1u << j;
    unsigned long long t0 = 0;
    unsigned it = 0;
    while (pending) {
      unsigned v[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        v[j] = (pending >> j) & 1u
                   ? ld_relaxed_gpu(flags + (size_t)(base + lane + 32 * j) * stride)
                   : value;
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        if (v[j] >= value) pending &= ~(1u << j);
      if (!pending) break;
      if (it == 0) t0 = globaltimer_ns();
      if (spin_ns > 0) __nanosleep(spin_ns);
      if ((++it & 31u) == 0) {
        if (ld_volatile_int(status) != kDevOk) {
          ok = false;
        } else if ((long long)(globaltimer_ns() - t0) > timeout_ns) {
          atomicCAS(status, kDevOk, kDevTimeout);
          ok = false;
        }
        if (!ok) break;
      }
    }
  }
  if (ok) {
    if (hi - lo + 1 > 64)
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
    else
      for (int i = lo + lane; i <= hi; i += 32) (void)ld_acquire_gpu(flags + (size_t)i * stride);
  }
  return __all_sync(0xffffffffu, ok);
}

// Step barrier among the `nblocks` blocks of one direction.  Each block
// publishes `value` in its own flag (flags[b * stride]); threads
// 0..nblocks-1 of every block wait, each on one flag.  Every wait is bounded
// (see wait_flag), so the kernel can leave without touching the data of an
// unfinished step.  Needs nblocks <= blockDim.x.  All threads must call it.
__device__ __forceinline__ bool step_barrier(unsigned* flags, int stride, int nblocks, int me,
                                             unsigned value, int* status, long long timeout_ns,
                                             int spin_ns, bool skip_arrive) {
  __syncthreads();
  if (threadIdx.x == 0 && !skip_arrive) publish_flag(flags + (size_t)me * stride, value);
  int fail = 0;
  if ((int)threadIdx.x < nblocks)
    fail = wait_flag(flags + (size_t)threadIdx.x * stride, value, status, timeout_ns, spin_ns) ? 0
                                                                                             : 1;
  return __syncthreads_or(fail) == 0;
}

// sum of p[0], p[stride], ..., p[(n-1)*stride] (n <= MAX) in index order, with
// every load issued before the first addition: a loop with a runtime trip
// count would wait for each load before the next
template <int MAX>
__device__ __forceinline__ float sum_strided(const float* p, size_t stride, int n) {
  float v[MAX];
#pragma unroll
  for (int i = 0; i < MAX; ++i) v[i] = i < n ? p[(size_t)i * stride] : 0.f;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < MAX; ++i) acc += v[i];
  return acc;
}

}  // namespace lr
