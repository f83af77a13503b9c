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

__device__ __forceinline__ float sigmoidf_(float a) { return 1.0f / (1.0f + expf(-a)); }

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
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Step barrier among the `nblocks` blocks of one direction.  Each block
// publishes `value` in its own flag (release); threads 0..nblocks-1 of every
// block wait, each on one flag (acquire), until it reaches `value`.  Every wait
// is bounded: past `timeout_ns`, or once another block has recorded a failure
// in *status, the block records kDevTimeout and the call returns false, so
// the kernel can leave without touching the data of the unfinished step.
// Needs nblocks <= blockDim.x.  All threads of the block must call it.
__device__ __forceinline__ bool step_barrier(unsigned* flags, int nblocks, int me,
                                             unsigned value, int* status,
                                             long long timeout_ns, bool skip_arrive) {
  __syncthreads();
  if (threadIdx.x == 0 && !skip_arrive) {
    __threadfence();
    st_release_gpu(flags + me, value);
  }
  int fail = 0;
  if ((int)threadIdx.x < nblocks) {
    const unsigned* f = flags + threadIdx.x;
    if (ld_acquire_gpu(f) < value) {
      const unsigned long long t0 = globaltimer_ns();
      unsigned it = 0;
      while (ld_acquire_gpu(f) < value) {
        if ((++it & 31u) == 0) {
          if (ld_volatile_int(status) != kDevOk) { fail = 1; break; }
          if ((long long)(globaltimer_ns() - t0) > timeout_ns) {
            atomicCAS(status, kDevOk, kDevTimeout);
            fail = 1;
            break;
          }
        }
      }
    }
  }
  return __syncthreads_or(fail) == 0;
}

}  // namespace lr
