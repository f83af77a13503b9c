// Device helpers of the tensor-core persistent recurrent kernels: cluster
// queries and barriers, DSMEM stores, tcgen05 MMA / tensor-memory access with
// the accumulator and A operand in tensor memory, bounded mbarrier waits.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace lr {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned cl_size() {
  unsigned n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
__device__ __forceinline__ unsigned cl_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16-byte store into the same offset of cluster block `rank`'s shared memory
__device__ __forceinline__ void st_peer4(float* local_ptr, unsigned rank, float a, float b,
                                         float c, float d) {
  unsigned raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(raddr)
               : "r"(smem_addr(local_ptr)), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(raddr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// 16-byte asynchronous store into cluster block `rank`'s shared memory (same
// offset as local_ptr) that completes 16 bytes of the transaction count of
// the barrier at local_bar's offset in that block: the receiver learns of the
// data from its own barrier, the sender waits for nothing
__device__ __forceinline__ void st_async4(float* local_ptr, uint32_t local_bar, unsigned rank,
                                          float a, float b, float c, float d) {
  unsigned raddr, rbar;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(raddr)
               : "r"(smem_addr(local_ptr)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(local_bar), "r"(rank));
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          raddr),
      "f"(a), "f"(b), "f"(c), "f"(d), "r"(rbar)
      : "memory");
}

// one arrival on a barrier of this block that also expects `bytes` more
// transaction bytes in the current phase
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// plain 4-byte load from this block's shared memory (shared-window address)
__device__ __forceinline__ float ld_shared_f32(uint32_t saddr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(saddr) : "memory");
  return v;
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// B tile descriptor: K-major rows of 128 bytes, 128-byte swizzle, 8-row groups
// 1024 bytes apart (tile base 1024-byte aligned)
__device__ __forceinline__ uint64_t b_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// byte offset of the 16-byte chunk `c` (0..7) of row `n` inside one K atom
// (rows x 128 bytes, 128-byte swizzle: chunk index XOR row index within the
// 8-row group)
__device__ __forceinline__ uint32_t sw_off(int n, int c) {
  return (uint32_t)((n >> 3) * 1024 + (n & 7) * 128 + ((c ^ (n & 7)) << 4));
}

__device__ __forceinline__ void mma_a_tmem(bool bf, uint32_t d, uint32_t a, uint64_t b,
                                           uint32_t idesc, uint32_t acc) {
  if (bf)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// The MMAs of one pass over NA K atoms of 64 16-bit elements (four K steps of
// 16 each): A from tensor memory (32 columns per atom), B from the swizzled
// shared tile (atoms bstep descriptor units apart), accumulate into dcol from
// the second MMA on.  Fully unrolled: the issuing thread runs a straight line
// of MMA instructions (a loop with a runtime trip count issues them about half
// as fast).
template <int NA>
__device__ __forceinline__ void mma_pass(uint32_t dcol, uint32_t acol0, uint64_t bd0,
                                         uint64_t bstep, uint32_t idesc) {
#pragma unroll
  for (int at = 0; at < NA; ++at)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_a_tmem(true, dcol, acol0 + (uint32_t)(at * 32 + kk * 8),
                 bd0 + (uint64_t)at * bstep + (uint64_t)(kk * 2), idesc, (at | kk) ? 1u : 0u);
}

// mma_pass for a runtime atom count: straight lines up to 8 atoms, a loop
// beyond
__device__ __forceinline__ void mma_pass_n(int na, uint32_t dcol, uint32_t acol0, uint64_t bd0,
                                           uint64_t bstep, uint32_t idesc) {
  switch (na) {
    case 1: mma_pass<1>(dcol, acol0, bd0, bstep, idesc); return;
    case 2: mma_pass<2>(dcol, acol0, bd0, bstep, idesc); return;
    case 3: mma_pass<3>(dcol, acol0, bd0, bstep, idesc); return;
    case 4: mma_pass<4>(dcol, acol0, bd0, bstep, idesc); return;
    case 5: mma_pass<5>(dcol, acol0, bd0, bstep, idesc); return;
    case 6: mma_pass<6>(dcol, acol0, bd0, bstep, idesc); return;
    case 7: mma_pass<7>(dcol, acol0, bd0, bstep, idesc); return;
    case 8: mma_pass<8>(dcol, acol0, bd0, bstep, idesc); return;
    default:
      for (int at = 0; at < na; ++at)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_a_tmem(true, dcol, acol0 + (uint32_t)(at * 32 + kk * 8),
                     bd0 + (uint64_t)at * bstep + (uint64_t)(kk * 2), idesc, (at | kk) ? 1u : 0u);
  }
}

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

// 16 columns of one tensor-memory lane quarter (32x32b shape, x16)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// three 16-column loads (three accumulators at columns ta, tb, tc of the same
// lanes) in flight together, one wait; the wait is in the same statement as
// the loads, so no use of the values can be scheduled before it
__device__ __forceinline__ void tmem_ld16x3(uint32_t ta, uint32_t tb, uint32_t tc,
                                            float (&a)[16], float (&b)[16], float (&c)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%48];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%49];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%50];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=f"(a[0]), "=f"(a[1]), "=f"(a[2]), "=f"(a[3]), "=f"(a[4]), "=f"(a[5]), "=f"(a[6]), "=f"(a[7]), "=f"(a[8]), "=f"(a[9]), "=f"(a[10]), "=f"(a[11]), "=f"(a[12]), "=f"(a[13]), "=f"(a[14]), "=f"(a[15]),
        "=f"(b[0]), "=f"(b[1]), "=f"(b[2]), "=f"(b[3]), "=f"(b[4]), "=f"(b[5]), "=f"(b[6]), "=f"(b[7]), "=f"(b[8]), "=f"(b[9]), "=f"(b[10]), "=f"(b[11]), "=f"(b[12]), "=f"(b[13]), "=f"(b[14]), "=f"(b[15]),
        "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3]), "=f"(c[4]), "=f"(c[5]), "=f"(c[6]), "=f"(c[7]), "=f"(c[8]), "=f"(c[9]), "=f"(c[10]), "=f"(c[11]), "=f"(c[12]), "=f"(c[13]), "=f"(c[14]), "=f"(c[15])
      : "r"(ta), "r"(tb), "r"(tc)
      : "memory");
}

// MMA with both operands in shared memory (descriptors), accumulator in
// tensor memory
__device__ __forceinline__ void mma_a_smem(bool bf, uint32_t d, uint64_t a, uint64_t b,
                                           uint32_t idesc, uint32_t acc) {
  if (bf)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// fp16 split of two values (already scaled): hi = fp16(x) and lo =
// fp16((x - hi) * 2^11) for each, packed two to a 32-bit word (the first
// value in the low half), so x = hi + lo * 2^-11 to about 22 bits
__device__ __forceinline__ void split_f16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn((x0 - hf.x) * 2048.f, (x1 - hf.y) * 2048.f);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Poll nb (<= R) rows of tagged exchange words: row j's pair of 8-byte words
// (value in the low half, step tag in the high half) at p + (row0 + j *
// rstep) * ld, loaded 16 bytes at a time, all pending rows in flight at once;
// returns when every pair carries `tag` (lanes with active = false return at
// once).  Each 8-byte word is single-copy atomic, so a word with the right tag
// holds the right value.  Bounded like warp_wait_flags; every lane of the
// warp must call it.
template <int R>
__device__ __forceinline__ bool poll_tagged(const unsigned long long* p, int row0, int rstep,
                                            int64_t ld, int nb, bool active, unsigned tag,
                                            unsigned long long (&w0)[R],
                                            unsigned long long (&w1)[R], int* status,
                                            long long timeout_ns) {
  unsigned pending = active ? ((1u << nb) - 1u) : 0u;
  unsigned long long t0 = 0;
  unsigned it = 0;
  bool ok = true;
  while (pending) {
#pragma unroll
    for (int j = 0; j < R; ++j)
      if ((pending >> j) & 1u) {
        const unsigned long long* q = p + (int64_t)(row0 + j * rstep) * ld;
        asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];"
                     : "=l"(w0[j]), "=l"(w1[j])
                     : "l"(q)
                     : "memory");
      }
#pragma unroll
    for (int j = 0; j < R; ++j)
      if (((pending >> j) & 1u) && (unsigned)(w0[j] >> 32) == tag &&
          (unsigned)(w1[j] >> 32) == tag)
        pending &= ~(1u << j);
    if (!pending) break;
    if (it == 0) t0 = globaltimer_ns();
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
  return __all_sync(0xffffffffu, ok);
}

// As poll_tagged, four consecutive words per row (one 32-byte load, 32-byte
// aligned): word i of row j of this lane lands in w[j][i].
template <int R>
__device__ __forceinline__ bool poll_tagged4(const unsigned long long* p, int row0, int rstep,
                                             int64_t ld, int nb, bool active, unsigned tag,
                                             unsigned long long (&w)[R][4], int* status,
                                             long long timeout_ns) {
  unsigned pending = active ? ((1u << nb) - 1u) : 0u;
  unsigned long long t0 = 0;
  unsigned it = 0;
  bool ok = true;
  while (pending) {
#pragma unroll
    for (int j = 0; j < R; ++j)
      if ((pending >> j) & 1u) {
        const unsigned long long* q = p + (int64_t)(row0 + j * rstep) * ld;
        asm volatile("ld.relaxed.gpu.global.v4.b64 {%0, %1, %2, %3}, [%4];"
                     : "=l"(w[j][0]), "=l"(w[j][1]), "=l"(w[j][2]), "=l"(w[j][3])
                     : "l"(q)
                     : "memory");
      }
#pragma unroll
    for (int j = 0; j < R; ++j)
      if (((pending >> j) & 1u) && (unsigned)(w[j][0] >> 32) == tag &&
          (unsigned)(w[j][1] >> 32) == tag && (unsigned)(w[j][2] >> 32) == tag &&
          (unsigned)(w[j][3] >> 32) == tag)
        pending &= ~(1u << j);
    if (!pending) break;
    if (it == 0) t0 = globaltimer_ns();
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
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// arrive (release, CTA scope) on a barrier of this block
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// arrive (release, cluster scope) on the barrier at the same offset in block
// `rank` of this cluster: orders this thread's earlier stores, including
// distributed-shared-memory stores, before the arrival
__device__ __forceinline__ void mbar_arrive_peer(uint32_t local_bar, unsigned rank) {
  uint32_t raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(local_bar), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(raddr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// bounded wait (acquire, cluster scope) for a phase that peers complete;
// false once the limit passed or another block recorded a failure
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity,
                                                          int* status, long long timeout_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  unsigned it = 0;
  while (!mbar_try_wait_cluster(bar, parity)) {
    if ((++it & 63u) == 0) {
      if (ld_volatile_int(status) != kDevOk) return false;
      if ((long long)(globaltimer_ns() - t0) > timeout_ns) {
        atomicCAS(status, kDevOk, kDevTimeout);
        return false;
      }
    }
  }
  return true;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// bounded; false once the limit passed or another block recorded a failure
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int* status,
                                                  long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  unsigned it = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++it & 63u) == 0) {
      if (ld_volatile_int(status) != kDevOk) return false;
      if ((long long)(globaltimer_ns() - t0) > timeout_ns) {
        atomicCAS(status, kDevOk, kDevTimeout);
        return false;
      }
    }
  }
  return true;
}

}  // namespace tc
}  // namespace lr
