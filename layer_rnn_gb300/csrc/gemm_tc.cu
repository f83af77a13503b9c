// Tensor-core GEMM for the dense phases on sm_103a: tcgen05.mma with the
// accumulator in tensor memory, operands staged by TMA (cp.async.bulk.tensor,
// 128-byte swizzle) through a multi-stage shared-memory ring.
//
//   C[m][n] (+)= sum_k A[m][k] * B[n][k]   (+ a second product over K2)
//
// A and B are K-major (row-major with K contiguous).  bf16 operands run one
// kind::f16 pass.  fp32 operands run as scaled fp16 pairs, x s = hi + lo
// (hi = fp16(x s), lo = fp16(x s - hi), s a power of two per operand that maps
// its largest magnitude below 2^14): three kind::f16 passes, A_hi*B_hi +
// A_hi*B_lo + A_lo*B_hi, into one fp32 accumulator, multiplied by 1/(s_A s_B)
// in the epilogue.  About 22 significant bits per operand, as the
// error-compensated split of Ootomo & Yokota (2022) on tf32, at the f16
// tensor rate and with 16-bit operands (half the bytes per K of tf32 pairs).
//
// One CTA computes one 128 x BN output tile (or one K range of it when the
// problem is split along K; the partial tiles are then summed in a fixed order
// by splitk_reduce_kernel).  Thread 0 issues the TMA loads, thread 32 the MMAs,
// and all four warps read the accumulator out of tensor memory for the
// epilogue, which stores fp32 results written whole with TMA (32 x 32 boxes)
// and the others through a padded shared-memory tile.  The tile width and
// the K split come from a wave model (gemm_tc_shape); multi-wave fp32 GEMMs
// run two CTAs per SM.  Every mbarrier wait is bounded by %globaltimer.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "gemm.h"

namespace lr {

namespace {

constexpr int BM = 128;
constexpr int kTcThreads = 128;
constexpr int kSmemBudget = 200 * 1024;

struct TcKParams {
  int M, N;
  int nk1, nk2;         // 128-byte K blocks of product 1 and 2
  int ksplit;
  int stages;
  void* C;
  int64_t ldc;
  int out_bf16;
  int accumulate;
  const void* bias1;
  const void* bias2;
  int64_t bias2_limit;
  int bias_bf16;
  float* part;          // split-K partials [ksplit][M][N] (fp32), or null
  const unsigned* amax;  // scaled fp16 pairs: largest |A|, |B| (float bit patterns)
  const unsigned* bmax;
  // the epilogue's stores: 0 plain stores, 1 TMA stores of C (fp32, no
  // accumulate) through maps.cout [M][N], 2 TMA stores of the split-K
  // partials through maps.cout [ksplit][M][N]
  int tma_out;
  int* status;
  long long timeout_ns;
};

struct TcMaps {
  CUtensorMap a1h, a1l, b1h, b1l, a2h, a2l, b2h, b2l;
  CUtensorMap cout;  // fp32 output (tma_out != 0), box 32 x 32 (x 1), 128-byte swizzle
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// bounded wait for the phase of `parity` to complete
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* status,
                                          long long timeout_ns, volatile int* abort_flag) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  unsigned it = 0;
  while (!mbar_try(bar, parity)) {
    if ((++it & 63u) == 0) {
      if (*abort_flag) return false;
      if ((long long)(globaltimer_ns() - t0) > timeout_ns) {
        atomicCAS(status, kDevOk, kDevTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
  return true;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// shared-memory matrix descriptor: K-major tile of rows x ROWB bytes (128 or
// 64), swizzled over the row (128- or 64-byte swizzle), 8-row groups
// 8 * ROWB bytes apart (tile base 1024-byte aligned)
template <int ROWB>
__device__ __forceinline__ uint64_t sw_desc(uint32_t saddr) {
  static_assert(ROWB == 128 || ROWB == 64, "128- or 64-byte rows");
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused for this layout)
  d |= (uint64_t)((8 * ROWB) >> 4) << 32;    // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;                    // descriptor version
  d |= (uint64_t)(ROWB == 128 ? 2 : 4) << 61;  // 128- or 64-byte swizzle
  return d;
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// tile store from shared memory (the box the map names at {x, y} or
// {x, y, z}); completion tracked by the issuing thread's bulk groups
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// operand scale exponent from the largest magnitude (the split kernels use
// the same function); defined with the split kernels below
__device__ __forceinline__ int f16_scale_exp(unsigned mb);
__device__ __forceinline__ float pow2f(int e);

template <int BN, bool SPLIT>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcKParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * 8 + 1];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float s_bias[BN];  // the tile's column bias (TMA-store epilogue)
  // K bytes per tile row and stage: 64 for the fp16 pairs at BN > 128 (four
  // operand tiles a stage: 48 KB at BN = 256, so four stages fit instead of
  // two), else 128 (at BN = 128 the 64-byte rows measured slower: twice the
  // stages for the same data)
  constexpr int ROWB = (SPLIT && BN > 128) ? 64 : 128;
  // tensor-memory columns: a power of two of at least 32
  constexpr uint32_t kCols = BN <= 32 ? 32u : BN <= 64 ? 64u : BN <= 128 ? 128u : 256u;
  constexpr int kA = BM * ROWB;                    // bytes of one A tile
  constexpr int kB = BN * ROWB;                    // bytes of one B tile
  constexpr int kStage = (kA + kB) * (SPLIT ? 2 : 1);
  // kind::f16, fp32 accumulate; A and B fp16 (0, scaled pairs) or bf16 (1)
  constexpr uint32_t kIdesc = (1u << 4) | ((SPLIT ? 0u : 1u) << 7) | ((SPLIT ? 0u : 1u) << 10) |
                              ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.stages;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[8]), done = smem_u32(&bars[16]);

  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int nkt = p.nk1 + p.nk2;
  const int z = blockIdx.z;
  const int kb0 = (int)((int64_t)z * nkt / p.ksplit), kb1 = (int)((int64_t)(z + 1) * nkt / p.ksplit);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (p.tma_out) {
    for (int c = threadIdx.x; c < BN; c += kTcThreads) {
      const int n = n0 + c;
      float b = 0.f;
      if (p.tma_out == 1 && n < p.N) {
        if (p.bias1) b += load_any(p.bias1, n, p.bias_bf16);
        if (p.bias2 && n < p.bias2_limit) b += load_any(p.bias2, n, p.bias_bf16);
      }
      s_bias[c] = b;
    }
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_slot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_slot;

  if (threadIdx.x == 0) {
    // TMA producer
    for (int kb = kb0; kb < kb1; ++kb) {
      const int it = kb - kb0, s = it % S;
      const uint32_t ph = (uint32_t)((it / S) & 1);
      if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, p.status, p.timeout_ns, &abort_flag)) break;
      const uint32_t st = base + (uint32_t)(s * kStage);
      const uint32_t fb = full0 + 8 * s;
      mbar_expect_tx(fb, (uint32_t)kStage);
      const bool second = kb >= p.nk1;
      const int kx = (second ? kb - p.nk1 : kb) * (ROWB / 2);
      const CUtensorMap* ah = second ? &maps.a2h : &maps.a1h;
      const CUtensorMap* bh = second ? &maps.b2h : &maps.b1h;
      tma_load_2d(st, ah, kx, m0, fb);
      tma_load_2d(st + kA, bh, kx, n0, fb);
      if (SPLIT) {
        const CUtensorMap* al = second ? &maps.a2l : &maps.a1l;
        const CUtensorMap* bl = second ? &maps.b2l : &maps.b1l;
        tma_load_2d(st + kA + kB, al, kx, m0, fb);
        tma_load_2d(st + 2 * kA + kB, bl, kx, n0, fb);
      }
    }
  } else if (threadIdx.x == 32) {
    // MMA issuer
    for (int kb = kb0; kb < kb1; ++kb) {
      const int it = kb - kb0, s = it % S;
      const uint32_t ph = (uint32_t)((it / S) & 1);
      if (!mbar_wait(full0 + 8 * s, ph, p.status, p.timeout_ns, &abort_flag)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t st = base + (uint32_t)(s * kStage);
      const uint64_t ah = sw_desc<ROWB>(st), bh = sw_desc<ROWB>(st + kA);
#pragma unroll
      for (int kk = 0; kk < ROWB / 32; ++kk) {  // 32 bytes of K per instruction
        const uint64_t adv = (uint64_t)(kk * 2);
        const uint32_t acc0 = (it > 0 || kk > 0) ? 1u : 0u;
        if (SPLIT) {
          // hi hi + hi lo + lo hi into one accumulator (lo is not rescaled)
          const uint64_t al = sw_desc<ROWB>(st + kA + kB), bl = sw_desc<ROWB>(st + 2 * kA + kB);
          mma_f16(tmem, ah + adv, bh + adv, kIdesc, acc0);
          mma_f16(tmem, ah + adv, bl + adv, kIdesc, 1u);
          mma_f16(tmem, al + adv, bh + adv, kIdesc, 1u);
        } else {
          mma_f16(tmem, ah + adv, bh + adv, kIdesc, acc0);
        }
      }
      mma_commit(empty0 + 8 * s);  // frees the stage once these MMAs have read it
    }
    mma_commit(done);
  }
  __syncwarp();

  // epilogue: warp w owns TMEM lanes / tile rows 32w .. 32w+31
  const bool have_k = kb1 > kb0;
  bool ok = true;
  if (have_k) ok = mbar_wait(done, 0, p.status, p.timeout_ns, &abort_flag);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (ok && !abort_flag && p.tma_out) {
    // the pipeline stages are free now: warp w stages its 32 rows, 32 columns
    // at a time, in the 128-byte-swizzled layout of a 32 x 32 fp32 box (16-byte
    // piece j of row r at piece j ^ (r & 7): conflict-free vector stores), and
    // one lane stores each box with TMA (full lines; rows and columns past
    // the output are clipped by the map).  Box bases are 4 KB apart from the
    // 1024-byte-aligned ring base, as the swizzle wants.
    // the scales one at a time, as the plain epilogue applies them (their
    // product alone may leave the fp32 range where the result does not)
    float ia = 1.f, ib = 1.f;
    if (SPLIT) {
      ia = pow2f(-f16_scale_exp(*p.amax));
      ib = pow2f(-f16_scale_exp(*p.bmax));
    }
    const int row0 = m0 + warp * 32;
    // two 4 KB boxes per warp, alternating: a box is rewritten once the
    // store that read it has finished reading (at most one store pending)
    const uint32_t wbuf = base + (uint32_t)(warp * 2 * 4096);
    if (row0 < p.M) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        if (n0 + c0 >= p.N) break;
        float v[32];
        if (have_k) {
          tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        const uint32_t box = wbuf + (uint32_t)((c0 >> 5) & 1) * 4096u;
        if (c0 >= 64) {
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          __syncwarp();
        }
        const uint32_t rb = box + (uint32_t)lane * 128u;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          st_shared_v4(rb + ((uint32_t)(j ^ (lane & 7)) << 4),
                       fmaf(v[4 * j] * ia, ib, s_bias[c0 + 4 * j]),
                       fmaf(v[4 * j + 1] * ia, ib, s_bias[c0 + 4 * j + 1]),
                       fmaf(v[4 * j + 2] * ia, ib, s_bias[c0 + 4 * j + 2]),
                       fmaf(v[4 * j + 3] * ia, ib, s_bias[c0 + 4 * j + 3]));
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          if (p.tma_out == 2)
            tma_store_3d(&maps.cout, box, n0 + c0, row0, z);
          else
            tma_store_2d(&maps.cout, box, n0 + c0, row0);
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      }
      if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
      __syncwarp();
    }
  } else if (ok && !abort_flag) {
    // the pipeline stages are free now: each warp stages its 32 rows x BN
    // accumulators in shared memory (row pitch BN + 1 floats, conflict-free),
    // then writes them row by row, 32 consecutive columns per instruction
    float* tile = reinterpret_cast<float*>(smem_raw + (base - smem_u32(smem_raw))) +
                  (size_t)warp * 32 * (BN + 1);
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      float v[32];
      if (have_k) {
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) tile[lane * (BN + 1) + c0 + i] = v[i];
    }
    __syncwarp();
    const int rbase = m0 + warp * 32;
    // scaled fp16 pairs: the product carries s_A s_B (powers of two)
    float ia = 1.f, ib = 1.f;
    if (SPLIT) {
      ia = pow2f(-f16_scale_exp(*p.amax));
      ib = pow2f(-f16_scale_exp(*p.bmax));
    }
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      const int n = n0 + c0 + lane;
      if (n >= p.N) continue;
      float bias = 0.f;
      if (!p.part) {
        if (p.bias1) bias += load_any(p.bias1, n, p.bias_bf16);
        if (p.bias2 && n < p.bias2_limit) bias += load_any(p.bias2, n, p.bias_bf16);
      }
#pragma unroll 4
      for (int r = 0; r < 32; ++r) {
        const int row = rbase + r;
        if (row >= p.M) break;
        float x = tile[r * (BN + 1) + c0 + lane];
        if (SPLIT) x = x * ia * ib;
        if (p.part) {
          p.part[((int64_t)z * p.M + row) * p.N + n] = x;
          continue;
        }
        x += bias;
        if (p.out_bf16) {
          bf16* c = reinterpret_cast<bf16*>(p.C) + (int64_t)row * p.ldc + n;
          if (p.accumulate) x += __bfloat162float(*c);
          *c = __float2bfloat16_rn(x);
        } else {
          float* c = reinterpret_cast<float*>(p.C) + (int64_t)row * p.ldc + n;
          if (p.accumulate) x += *c;
          *c = x;
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 2)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols)
                 : "memory");
}

// C = sum_z part[z] (+ bias) (+ C); fixed order over z; four columns per
// thread and step (N % 4 == 0, ldc % 4 == 0, fp32 output, 16-byte aligned)
__global__ void __launch_bounds__(256) splitk_reduce_v_kernel(
    const float* __restrict__ part, int ks, int64_t M, int64_t N, float* C, int64_t ldc,
    int accumulate, const void* bias1, const void* bias2, int64_t bias2_limit, int bias_bf16) {
  const int64_t nv = N / 4, total = M * nv, plane = M * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / nv, n = (i - m * nv) * 4;
    float4 x = __ldg(reinterpret_cast<const float4*>(part + m * N + n));
    for (int zz = 1; zz < ks; ++zz) {
      const float4 y = __ldg(reinterpret_cast<const float4*>(part + (int64_t)zz * plane + m * N + n));
      x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
    }
    float b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (bias1) b[u] += load_any(bias1, n + u, bias_bf16);
      if (bias2 && n + u < bias2_limit) b[u] += load_any(bias2, n + u, bias_bf16);
    }
    x.x += b[0]; x.y += b[1]; x.z += b[2]; x.w += b[3];
    float4* c = reinterpret_cast<float4*>(C + m * ldc + n);
    if (accumulate) {
      const float4 o = *c;
      x.x += o.x; x.y += o.y; x.z += o.z; x.w += o.w;
    }
    *c = x;
  }
}

// C = sum_z part[z] (+ bias) (+ C); fixed order over z
__global__ void splitk_reduce_kernel(const float* part, int ks, int64_t M, int64_t N, void* C,
                                     int64_t ldc, int out_bf16, int accumulate, const void* bias1,
                                     const void* bias2, int64_t bias2_limit, int bias_bf16) {
  const int64_t total = M * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / N, n = i - m * N;
    float x = 0.f;
    for (int zz = 0; zz < ks; ++zz) x += part[(int64_t)zz * total + i];
    if (bias1) x += load_any(bias1, n, bias_bf16);
    if (bias2 && n < bias2_limit) x += load_any(bias2, n, bias_bf16);
    if (out_bf16) {
      bf16* c = reinterpret_cast<bf16*>(C) + m * ldc + n;
      if (accumulate) x += __bfloat162float(*c);
      *c = __float2bfloat16_rn(x);
    } else {
      float* c = reinterpret_cast<float*>(C) + m * ldc + n;
      if (accumulate) x += *c;
      *c = x;
    }
  }
}

// ---------------------------------------------------------------------------
// operand preparation: fp32 -> scaled fp16 (hi, lo) pairs, optionally
// transposed; bf16 transpose
// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// fp32 operands as scaled fp16 pairs: x * s = hi + lo + e with hi = fp16(x s),
// lo = fp16(x s - hi) (unscaled: the three products hi hi, hi lo, lo hi go to
// one accumulator), |e| <= 2^-22 |x s| for |x s| >= 2^-14; s is a power of
// two per operand that maps the operand's largest magnitude into
// [2^13, 2^14) (fp16 holds up to 65504), and the product is multiplied by
// 1 / (s_A s_B) in the epilogue (exact: powers of two).  Elements more than
// 2^27 below the largest lose relative precision; they weigh less than
// 2^-27 of it in any sum.
// ---------------------------------------------------------------------------

// largest |x| of an operand, as the bit pattern of a non-negative float
// (ordered like the values): atomicMax into *out, which starts at 0
__global__ void __launch_bounds__(256) absmax_kernel(const float* __restrict__ src, int64_t rows,
                                                     int64_t cols, int64_t lds, unsigned* out) {
  unsigned m = 0;
  const int64_t total = rows * cols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / cols, c = i - r * cols;
    m = max(m, __float_as_uint(src[r * lds + c]) & 0x7FFFFFFFu);
  }
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0 && m) atomicMax(out, m);
}

// the same for 16-byte aligned rows whose length is a multiple of 4: four
// 16-byte loads in flight per thread, one atomic per block
__global__ void __launch_bounds__(256) absmax_v_kernel(const float* __restrict__ src, int64_t rows,
                                                       int64_t cols, int64_t lds, unsigned* out) {
  __shared__ unsigned red[8];
  unsigned m = 0;
  const int64_t cv = cols / 4, total = rows * cv;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  auto amax4 = [](float4 v) {
    return max(max(__float_as_uint(v.x) & 0x7FFFFFFFu, __float_as_uint(v.y) & 0x7FFFFFFFu),
               max(__float_as_uint(v.z) & 0x7FFFFFFFu, __float_as_uint(v.w) & 0x7FFFFFFFu));
  };
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < total; i += 4 * stride) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t j = i + u * stride, r = j / cv, c = (j - r * cv) * 4;
      v[u] = __ldg(reinterpret_cast<const float4*>(src + r * lds + c));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) m = max(m, amax4(v[u]));
  }
  for (; i < total; i += stride) {
    const int64_t r = i / cv, c = (i - r * cv) * 4;
    m = max(m, amax4(__ldg(reinterpret_cast<const float4*>(src + r * lds + c))));
  }
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = max(m, red[w]);
    if (m) atomicMax(out, m);
  }
}

// exponent sh of the scale s = 2^sh for an operand whose largest magnitude
// has the bit pattern `mb`: the largest lands in [2^13, 2^14); an all-zero or
// non-finite operand gets s = 1
__device__ __forceinline__ int f16_scale_exp(unsigned mb) {
  if (mb == 0u || mb >= 0x7F800000u) return 0;
  const int E = (int)(mb >> 23) - 127;  // largest in [2^E, 2^(E+1)) (E = -127: subnormal)
  return min(max(13 - E, -126), 126);
}
__device__ __forceinline__ float pow2f(int e) {  // 2^e, -126 <= e <= 127
  return __uint_as_float((unsigned)(e + 127) << 23);
}

__device__ __forceinline__ void f16_pair(float v, float s, __half& h, __half& l) {
  const float x = v * s;  // exact: s is a power of two (no overflow: |x| < 2^14)
  h = __float2half_rn(x);
  l = __float2half_rn(x - __half2float(h));  // x - h is exact in fp32
}

// plain split, 4 columns per thread and step (16-byte aligned source rows,
// 8-byte aligned destination rows, cols % 4 == 0)
__global__ void __launch_bounds__(256) split_f16_v_kernel(const float* __restrict__ src,
                                                          int64_t rows, int64_t cols, int64_t lds,
                                                          __half* __restrict__ hi,
                                                          __half* __restrict__ lo, int64_t ldd,
                                                          const unsigned* maxbits) {
  const float s = pow2f(f16_scale_exp(*maxbits));
  const int64_t cv = cols / 4, total = rows * cv;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / cv, c = (i - r * cv) * 4;
    const float4 v = __ldg(reinterpret_cast<const float4*>(src + r * lds + c));
    __align__(8) __half h[4], l[4];
    f16_pair(v.x, s, h[0], l[0]);
    f16_pair(v.y, s, h[1], l[1]);
    f16_pair(v.z, s, h[2], l[2]);
    f16_pair(v.w, s, h[3], l[3]);
    *reinterpret_cast<uint2*>(hi + r * ldd + c) = *reinterpret_cast<const uint2*>(h);
    *reinterpret_cast<uint2*>(lo + r * ldd + c) = *reinterpret_cast<const uint2*>(l);
  }
}

// transposing split: a 64 x 64 tile through shared memory (row pitch 65
// floats), 16-byte reads; each thread writes 4 output columns (8 bytes) of a
// row (rows % 4 == 0, 16-byte aligned source rows, 8-byte aligned destination)
__global__ void __launch_bounds__(256) split_f16_tt_kernel(const float* __restrict__ src,
                                                           int64_t rows, int64_t cols,
                                                           int64_t lds, __half* __restrict__ hi,
                                                           __half* __restrict__ lo, int64_t ldd,
                                                           const unsigned* maxbits) {
  __shared__ float tile[64][65];
  const float s = pow2f(f16_scale_exp(*maxbits));
  const int64_t r0 = (int64_t)blockIdx.y * 64, c0 = (int64_t)blockIdx.x * 64;
  const int tid = threadIdx.x, q = tid & 15, sub = tid >> 4;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int row = p * 16 + sub;
    const int64_t r = r0 + row, c = c0 + 4 * q;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < rows && c < cols) v = __ldg(reinterpret_cast<const float4*>(src + r * lds + c));
    tile[row][4 * q + 0] = v.x;
    tile[row][4 * q + 1] = v.y;
    tile[row][4 * q + 2] = v.z;
    tile[row][4 * q + 3] = v.w;
  }
  __syncthreads();
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int oc = p * 16 + sub;
    const int64_t orow = c0 + oc, ocol = r0 + 4 * q;
    if (orow >= cols || ocol >= rows) continue;
    __align__(8) __half h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) f16_pair(tile[4 * q + i][oc], s, h[i], l[i]);
    *reinterpret_cast<uint2*>(hi + orow * ldd + ocol) = *reinterpret_cast<const uint2*>(h);
    *reinterpret_cast<uint2*>(lo + orow * ldd + ocol) = *reinterpret_cast<const uint2*>(l);
  }
}

// generic split (any shape and alignment), optionally transposed
__global__ void split_f16_kernel(const float* src, int64_t rows, int64_t cols, int64_t lds,
                                 __half* hi, __half* lo, int64_t ldd, int transpose,
                                 const unsigned* maxbits) {
  __shared__ float tile[32][33];
  const float s = pow2f(f16_scale_exp(*maxbits));
  const int64_t r0 = (int64_t)blockIdx.y * 32, c0 = (int64_t)blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int k = ty; k < 32; k += 8) {
    const int64_t r = r0 + k, c = c0 + tx;
    tile[k][tx] = (r < rows && c < cols) ? src[r * lds + c] : 0.f;
  }
  __syncthreads();
  for (int k = ty; k < 32; k += 8) {
    float v;
    int64_t orow, ocol;
    if (transpose) {
      v = tile[tx][k];
      orow = c0 + k;
      ocol = r0 + tx;
      if (orow >= cols || ocol >= rows) continue;
    } else {
      v = tile[k][tx];
      orow = r0 + k;
      ocol = c0 + tx;
      if (orow >= rows || ocol >= cols) continue;
    }
    __half h, l;
    f16_pair(v, s, h, l);
    hi[orow * ldd + ocol] = h;
    lo[orow * ldd + ocol] = l;
  }
}

__global__ void transpose_bf16_kernel(const bf16* src, int64_t rows, int64_t cols, int64_t lds,
                                      bf16* dst, int64_t ldd) {
  __shared__ bf16 tile[32][34];
  const int64_t r0 = (int64_t)blockIdx.y * 32, c0 = (int64_t)blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int k = ty; k < 32; k += 8) {
    const int64_t r = r0 + k, c = c0 + tx;
    tile[k][tx] = (r < rows && c < cols) ? src[r * lds + c] : __float2bfloat16_rn(0.f);
  }
  __syncthreads();
  for (int k = ty; k < 32; k += 8) {
    const int64_t orow = c0 + k, ocol = r0 + tx;
    if (orow < cols && ocol < rows) dst[orow * ldd + ocol] = tile[tx][k];
  }
}

// bf16 transpose for aligned shapes (rows % 16 == 0, cols % 8 == 0, both row
// strides multiples of 8 elements, 16-byte aligned buffers): each thread reads
// a 16-row x 8-column block as sixteen 16-byte row pieces (a warp reads 512
// contiguous bytes of a row per load), transposes it in registers with byte
// permutes and writes 8 output rows of 32 contiguous bytes (whole sectors).
// Block = 8 warps = 128 source rows x 256 source columns.
__device__ __forceinline__ uint32_t u4_word(const uint4& a, int k) {
  return k == 0 ? a.x : k == 1 ? a.y : k == 2 ? a.z : a.w;
}

__global__ void __launch_bounds__(256) transpose_bf16_v_kernel(const bf16* __restrict__ src,
                                                               int64_t rows, int64_t cols,
                                                               int64_t lds, bf16* __restrict__ dst,
                                                               int64_t ldd) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t r0 = (int64_t)blockIdx.y * 128 + w * 16;
  const int64_t c0 = ((int64_t)blockIdx.x * 32 + lane) * 8;
  if (r0 >= rows || c0 >= cols) return;
  uint4 v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    v[i] = __ldg(reinterpret_cast<const uint4*>(src + (r0 + i) * lds + c0));
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    // element j of source rows 2k and 2k+1 -> the low and high half of word k
    const unsigned sel = (j & 1) ? 0x7632u : 0x5410u;
    uint4 o0, o1;
    o0.x = __byte_perm(u4_word(v[0], j >> 1), u4_word(v[1], j >> 1), sel);
    o0.y = __byte_perm(u4_word(v[2], j >> 1), u4_word(v[3], j >> 1), sel);
    o0.z = __byte_perm(u4_word(v[4], j >> 1), u4_word(v[5], j >> 1), sel);
    o0.w = __byte_perm(u4_word(v[6], j >> 1), u4_word(v[7], j >> 1), sel);
    o1.x = __byte_perm(u4_word(v[8], j >> 1), u4_word(v[9], j >> 1), sel);
    o1.y = __byte_perm(u4_word(v[10], j >> 1), u4_word(v[11], j >> 1), sel);
    o1.z = __byte_perm(u4_word(v[12], j >> 1), u4_word(v[13], j >> 1), sel);
    o1.w = __byte_perm(u4_word(v[14], j >> 1), u4_word(v[15], j >> 1), sel);
    uint4* out = reinterpret_cast<uint4*>(dst + (c0 + j) * ldd + r0);
    out[0] = o0;
    out[1] = o1;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// K-major 16-bit operand [rows][K] with row stride ld (elements); box =
// row_bytes / 2 x box_rows, swizzled over row_bytes (128 or 64)
bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K, int64_t ld,
              int row_bytes, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !ptr || (row_bytes != 128 && row_bytes != 64)) return false;
  const int e = 2;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * e)};
  cuuint32_t box[2] = {(cuuint32_t)(row_bytes / e), (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool operand_ok(const void* p, int64_t ld, int e) {
  return p && (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld * e) % 16 == 0);
}

template <int BN, bool SPLIT>
cudaError_t launch_tc(const TcMaps& maps, const TcKParams& kp, dim3 grid, cudaStream_t st) {
  constexpr int kStage = (BM + BN) * ((SPLIT && BN > 128) ? 64 : 128) * (SPLIT ? 2 : 1);
  // at least 80 KB: never three CTAs on an SM (their accumulators would not
  // all fit in its tensor memory)
  const size_t smem = std::max<size_t>((size_t)kp.stages * kStage + 1024, 80 * 1024);
  auto fn = gemm_tc_kernel<BN, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  fn<<<grid, kTcThreads, smem, st>>>(maps, kp);
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

}  // namespace

bool tma_encode(void* map, int rank, bool bf, const void* ptr, const uint64_t* dims,
                const uint64_t* strides_bytes, const uint32_t* box) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !ptr || rank < 2 || rank > 3) return false;
  cuuint64_t d[3], sb[2];
  cuuint32_t bx[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = (cuuint64_t)dims[i];
    bx[i] = (cuuint32_t)box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) sb[i] = (cuuint64_t)strides_bytes[i];
  return enc(static_cast<CUtensorMap*>(map),
             bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
             (cuuint32_t)rank, const_cast<void*>(ptr), d, sb, bx, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tile width and K split from a wave model.  One 64-element K block of a
// 128 x BN tile costs the larger of its MMA time (three passes for scaled fp16
// pairs, at about 1/152 of the dense f16 rate per SM) and its operand feed
// (128 + BN rows of 128 bytes, twice for hi and lo, at about 64 bytes per
// clock per SM: wide tiles read each A tile once for more MMA work).  The grid
// runs in ceil(units / SMs) waves of ceil(nkt / ks) K blocks plus a fixed
// cost per tile (launch, pipeline fill, epilogue: about 10 us, fitted to the
// DS2 GEMMs); a split adds its fp32 partial sums (written and read once) at
// HBM speed.  A 160-wide tile pays where it empties the last wave: the DS2
// dX (N = 800) runs 2 waves of 47 x 5 tiles instead of 3 of 47 x 7 at 128,
// and the weight gradients one wave of 25 x 5 tiles with no split.  (224
// wide measured no faster than 256 at the same number of waves.)
namespace {
double kb_clocks(int BN, bool split16) {
  const double mma = 2.0 * BM * BN * 64.0 * (split16 ? 3.0 : 1.0) / (2.25e15 / 152.0 / 2.07e9);
  const double feed = (double)(BM + BN) * 128.0 * (split16 ? 2.0 : 1.0) / 64.0;
  return std::max(mma, feed);
}
}  // namespace

void gemm_tc_shape(int64_t M, int64_t N, int64_t K_total, bool split16, int num_sms,
                   bool allow_split, int* bn_out, int* ks_out) {
  const int64_t nkt = (K_total * 2 + 127) / 128;
  const int sms = std::max(1, num_sms);
  const double red_clk = 8.0 * (double)M * N / 6.0e12 * 2.07e9;  // per split
  int best_bn = N <= 64 ? 64 : 128, best_ks = 1;
  double best = -1;
  const double fixed_clk = 20000.0;  // per tile and wave
  for (int BN : {64, 128, 160, 192, 256}) {
    if ((BN == 64) != (N <= 64)) continue;
    if (BN > 128 && BN > (N + 31) / 32 * 32) continue;  // no tile wider than the output
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const double t_kb = kb_clocks(BN, split16);
    for (int ks = 1; ks <= 8; ++ks) {
      if (ks > 1 && (!allow_split || nkt < 8 || nkt / ks < 4)) break;
      const int64_t units = tiles * ks;
      const double waves = (double)((units + sms - 1) / sms);
      const double cost = waves * ((double)((nkt + ks - 1) / ks) * t_kb + fixed_clk) +
                          (ks > 1 ? red_clk * ks : 0.0);
      if (best < 0 || cost < best) {
        best = cost;
        best_bn = BN;
        best_ks = ks;
      }
    }
  }
  *bn_out = best_bn;
  *ks_out = best_ks;
}

bool gemm_tc_supported(const TcGemm& g) {
  const int e = 2;
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return false;
  if (!operand_ok(g.A_hi, g.lda, e) || !operand_ok(g.B_hi, g.ldb, e)) return false;
  if (g.split16 && (!operand_ok(g.A_lo, g.lda, e) || !operand_ok(g.B_lo, g.ldb, e) || !g.amax ||
                    !g.bmax))
    return false;
  if (g.K2 > 0) {
    if (!operand_ok(g.A2_hi, g.lda2, e) || !operand_ok(g.B2_hi, g.ldb2, e)) return false;
    if (g.split16 && (!operand_ok(g.A2_lo, g.lda2, e) || !operand_ok(g.B2_lo, g.ldb2, e)))
      return false;
  }
  return encode_fn() != nullptr;
}

cudaError_t gemm_tc(const TcGemm& g, cudaStream_t st) {
  const bool sp = g.split16 != 0;
  int BN = g.bn, ks_unused = 1;
  if (BN == 0) gemm_tc_shape(g.M, g.N, g.K + g.K2, sp, 148, false, &BN, &ks_unused);
  if (BN != 64 && BN != 128 && BN != 160 && BN != 192 && BN != 256) return cudaErrorInvalidValue;
  TcMaps maps;
  memset(&maps, 0, sizeof(maps));
  // every operand is 16-bit (fp16 pairs or bf16): TMA copies bytes, so one
  // 16-bit map type serves both
  const int rowb = (sp && BN > 128) ? 64 : 128;  // K bytes per tile row and stage
  bool ok = make_map(&maps.a1h, g.A_hi, g.M, g.K, g.lda, rowb, BM) &&
            make_map(&maps.b1h, g.B_hi, g.N, g.K, g.ldb, rowb, BN);
  if (sp)
    ok = ok && make_map(&maps.a1l, g.A_lo, g.M, g.K, g.lda, rowb, BM) &&
         make_map(&maps.b1l, g.B_lo, g.N, g.K, g.ldb, rowb, BN);
  if (g.K2 > 0) {
    ok = ok && make_map(&maps.a2h, g.A2_hi, g.M, g.K2, g.lda2, rowb, BM) &&
         make_map(&maps.b2h, g.B2_hi, g.N, g.K2, g.ldb2, rowb, BN);
    if (sp)
      ok = ok && make_map(&maps.a2l, g.A2_lo, g.M, g.K2, g.lda2, rowb, BM) &&
           make_map(&maps.b2l, g.B2_lo, g.N, g.K2, g.ldb2, rowb, BN);
  }
  if (!ok) return cudaErrorInvalidValue;
  const int kpe = rowb / 2;
  TcKParams kp;
  memset(&kp, 0, sizeof(kp));
  kp.M = (int)g.M;
  kp.N = (int)g.N;
  kp.nk1 = (int)((g.K + kpe - 1) / kpe);
  kp.nk2 = g.K2 > 0 ? (int)((g.K2 + kpe - 1) / kpe) : 0;
  kp.ksplit = std::max(1, g.ksplit);
  const int stage = (BM + BN) * rowb * (sp ? 2 : 1);
  kp.stages = std::max(2, std::min(8, kSmemBudget / stage));
  kp.amax = g.amax;
  kp.bmax = g.bmax;
  kp.status = g.status;
  kp.timeout_ns = g.timeout_ns;
  if (kp.ksplit > 1) {
    kp.part = g.part;
    if (!kp.part) return cudaErrorInvalidValue;
    // partials [ksplit][M][N] fp32 through a 3-D map (rows past M clipped
    // within each split)
    if (reinterpret_cast<uintptr_t>(g.part) % 16 == 0 && g.N % 4 == 0) {
      const uint64_t dims[3] = {(uint64_t)g.N, (uint64_t)g.M, (uint64_t)kp.ksplit};
      const uint64_t strides[2] = {(uint64_t)g.N * 4, (uint64_t)g.N * g.M * 4};
      const uint32_t box[3] = {32u, 32u, 1u};
      if (tma_encode(&maps.cout, 3, false, g.part, dims, strides, box)) kp.tma_out = 2;
    }
  } else {
    kp.C = g.C;
    kp.ldc = g.ldc;
    kp.out_bf16 = g.out_bf16;
    kp.accumulate = g.accumulate;
    kp.bias1 = g.bias1;
    kp.bias2 = g.bias2;
    kp.bias2_limit = g.bias2_limit;
    kp.bias_bf16 = g.bias_bf16;
    // fp32 C written whole (no accumulate): TMA stores
    if (!g.out_bf16 && !g.accumulate && reinterpret_cast<uintptr_t>(g.C) % 16 == 0 &&
        g.ldc % 4 == 0) {
      const uint64_t dims[2] = {(uint64_t)g.N, (uint64_t)g.M};
      const uint64_t strides[1] = {(uint64_t)g.ldc * 4};
      const uint32_t box[2] = {32u, 32u};
      if (tma_encode(&maps.cout, 2, false, g.C, dims, strides, box)) kp.tma_out = 1;
    }
  }
  // two CTAs per SM (a ring of at most 100 KB each: one CTA's accumulator
  // drain and stores run under the other's main loop) with the TMA-store
  // epilogue, whose staging is small
  if (kp.tma_out && g.ctas_per_sm == 2) kp.stages = std::max(2, std::min(8, (100 * 1024) / stage));
  // the TMA-store epilogue stages two 32 x 32 fp32 boxes per warp in the
  // ring, the plain one a 32 x (BN + 1) fp32 tile per warp
  if (kp.tma_out && (size_t)kp.stages * stage < (size_t)4 * 2 * 4096) kp.tma_out = 0;
  if (!kp.tma_out && (size_t)kp.stages * stage < (size_t)4 * 32 * (BN + 1) * 4)
    return cudaErrorInvalidValue;
  dim3 grid((unsigned)((g.N + BN - 1) / BN), (unsigned)((g.M + BM - 1) / BM), (unsigned)kp.ksplit);
  cudaError_t e;
  if (sp)
    e = BN == 256   ? launch_tc<256, true>(maps, kp, grid, st)
        : BN == 192 ? launch_tc<192, true>(maps, kp, grid, st)
        : BN == 160 ? launch_tc<160, true>(maps, kp, grid, st)
        : BN == 128 ? launch_tc<128, true>(maps, kp, grid, st)
                    : launch_tc<64, true>(maps, kp, grid, st);
  else
    e = BN == 256   ? launch_tc<256, false>(maps, kp, grid, st)
        : BN == 192 ? launch_tc<192, false>(maps, kp, grid, st)
        : BN == 160 ? launch_tc<160, false>(maps, kp, grid, st)
        : BN == 128 ? launch_tc<128, false>(maps, kp, grid, st)
                    : launch_tc<64, false>(maps, kp, grid, st);
  if (e != cudaSuccess || kp.ksplit == 1) return e;
  const int64_t total = g.M * g.N;
  const bool vec = !g.out_bf16 && g.N % 4 == 0 && g.ldc % 4 == 0 &&
                   reinterpret_cast<uintptr_t>(g.C) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(g.part) % 16 == 0;
  if (vec) {
    const int blocks = (int)std::min<int64_t>((total / 4 + 255) / 256, 152 * 8);
    splitk_reduce_v_kernel<<<blocks, 256, 0, st>>>(g.part, kp.ksplit, g.M, g.N,
                                                   static_cast<float*>(g.C), g.ldc, g.accumulate,
                                                   g.bias1, g.bias2, g.bias2_limit, g.bias_bf16);
  } else {
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, 4096);
    splitk_reduce_kernel<<<blocks, 256, 0, st>>>(g.part, kp.ksplit, g.M, g.N, g.C, g.ldc,
                                                 g.out_bf16, g.accumulate, g.bias1, g.bias2,
                                                 g.bias2_limit, g.bias_bf16);
  }
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

cudaError_t absmax_operand(const float* src, int64_t rows, int64_t cols, int64_t lds,
                           unsigned* mx, int num_sms, cudaStream_t st) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const bool al = cols % 4 == 0 && lds % 4 == 0 && reinterpret_cast<uintptr_t>(src) % 16 == 0;
  const int64_t work = al ? rows * (cols / 4) : rows * cols;
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((work + 1023) / 1024,
                                                                  (int64_t)std::max(1, num_sms) * 4));
  if (al)
    absmax_v_kernel<<<blocks, 256, 0, st>>>(src, rows, cols, lds, mx);
  else
    absmax_kernel<<<blocks, 256, 0, st>>>(src, rows, cols, lds, mx);
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

cudaError_t split_f16_operand(const float* src, int64_t rows, int64_t cols, int64_t lds, void* hi,
                              void* lo, int64_t ldd, bool transpose, const unsigned* mx,
                              cudaStream_t st) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  __half* h = static_cast<__half*>(hi);
  __half* l = static_cast<__half*>(lo);
  const bool al = cols % 4 == 0 && lds % 4 == 0 && ldd % 4 == 0 &&
                  reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
                  reinterpret_cast<uintptr_t>(hi) % 8 == 0 &&
                  reinterpret_cast<uintptr_t>(lo) % 8 == 0;
  if (al && transpose && rows % 4 == 0 && (rows + 63) / 64 <= 65535) {
    dim3 grid((unsigned)((cols + 63) / 64), (unsigned)((rows + 63) / 64));
    split_f16_tt_kernel<<<grid, 256, 0, st>>>(src, rows, cols, lds, h, l, ldd, mx);
    g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
  }
  if (al && !transpose) {
    const int64_t blocks = std::min<int64_t>((rows * (cols / 4) + 255) / 256, 152 * 16);
    split_f16_v_kernel<<<(unsigned)blocks, 256, 0, st>>>(src, rows, cols, lds, h, l, ldd, mx);
    g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
  }
  dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows + 31) / 32));
  split_f16_kernel<<<grid, 256, 0, st>>>(src, rows, cols, lds, h, l, ldd, transpose ? 1 : 0, mx);
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

cudaError_t transpose_bf16(const void* src, int64_t rows, int64_t cols, int64_t lds, void* dst,
                           int64_t ldd, cudaStream_t st) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const bool vec = rows % 16 == 0 && cols % 8 == 0 && lds % 8 == 0 && ldd % 8 == 0 &&
                   reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(dst) % 16 == 0 && (rows + 127) / 128 <= 65535;
  if (vec) {
    dim3 grid((unsigned)((cols / 8 + 31) / 32), (unsigned)((rows + 127) / 128));
    transpose_bf16_v_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const bf16*>(src), rows, cols,
                                                  lds, reinterpret_cast<bf16*>(dst), ldd);
    g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
  }
  dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows + 31) / 32));
  transpose_bf16_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const bf16*>(src), rows, cols, lds,
                                              reinterpret_cast<bf16*>(dst), ldd);
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

}  // namespace lr
