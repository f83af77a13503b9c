// Tensor-core recurrent backward for large batches (bf16): the batch is the
// MMA's M dimension.
//
// Per step the backward contraction is
//     dh_{t-1}[n][k] = sum_j dG_h[t][n][j] * W_hh[j][k]
// (reverse-mode through the recurrences of the "rnn training example?" thread,
// reading 13 of the design notes).  With a batch of 64..128 sequences the
// batch fills the 128 rows of a tcgen05 MMA, so here A = dG_h[t] (batch rows,
// K-major along the G*H gate rows, exactly as the workspace stores it) and
// B = W_hh^T (hidden units as the MMA's N).  Clusters of Pk blocks own row
// groups of Ur units; the blocks of a cluster split the G*H contraction:
//   * B, the block's W_hh^T slice [Ur units][Kk gate rows] in bf16, stays in
//     shared memory for the whole sequence (128-byte-swizzled K-major atoms);
//   * A, the previous step's dG_h slice [N][Kk], streams from L2 through a
//     TMA ring (cp.async.bulk.tensor.3d over [T][N][G*H]; batch rows beyond N
//     read as zeros) while one thread issues the MMAs;
//   * the accumulator D[n][u] (tensor memory, lane = batch row) is pushed, 4
//     units per 16-byte DSMEM store, to the block that owns the units'
//     pointwise step (with two partial-sum buffers as st.async stores that
//     complete the owner's barrier for the step, else plain stores and a
//     cluster barrier); the owners sum the partials in a fixed order, run the
//     gate-gradient chain and store dG (bf16), then release their step flag.
// The loads read what other blocks stored, so the writer fences its stores to
// the async proxy before its release and the reader after its acquire.  All
// waits are bounded.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "rec.h"
#include "tc_common.cuh"

#ifdef LAYER_RNN_TRACE
// per block (up to 160), per step (up to 1024), 8 time marks
__device__ unsigned long long g_mtrace[160][1024][8];
#define MTRACE(s, k)                                                                   \
  do {                                                                                 \
    if (blockIdx.x < 160 && threadIdx.x == 0 && (s) < 1024)                            \
      g_mtrace[blockIdx.x][(s)][(k)] = lr::globaltimer_ns();                           \
  } while (0)
#else
#define MTRACE(s, k) ((void)0)
#endif

namespace lr {

namespace {

using namespace tc;

constexpr int kMThreads = 256;
constexpr int kMRows = 128;     // MMA M (batch rows)
constexpr int kMChunk = 64;     // bf16 elements of K per ring stage / B atom
constexpr int kMStages = 8;      // most ring stages the kernel supports
constexpr int kRingUse = 4;      // stages the plan uses
constexpr int kMNIn = 7;        // pointwise inputs per item: dy, 4 gates, c_t, c_{t-1}
constexpr int kRegItems = 5;    // items per thread when the inputs are prefetched to registers
// threads that prefetch the pointwise inputs, into registers or shared memory
// (warps 1..7: the producer warp ends a wide flag wait with an acquire fence,
// which would also wait for its own loads and copies in flight)
constexpr int kRegThreads = kMThreads - 32;

struct MMaps {
  CUtensorMap a[2];  // dG_h of each direction: [T][N][G*H] bf16, box 64 x 128 x 1
};

__device__ __forceinline__ int owner_flag_m(int u, int Ur, int Uq, int Pk) {
  const int r = u / Ur;
  return r * Pk + (u - r * Ur) / Uq;
}

__device__ __forceinline__ void tma3(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                     uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mma_ss_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tmem_ld4m(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

struct MLayout {
  uint32_t b;         // resident B: KC atoms x (Urp rows x 128 bytes)
  uint32_t ring;      // pl.ring stages x (128 rows x 128 bytes)
  uint32_t recv;      // [rbufs][Pk][N][Uq] f32
  uint32_t outs;      // [N][Uq] f32
  uint32_t st_dc, st_carry;  // [Uq*N] f32
  uint32_t pin;       // [kMNIn][Uq*N] f32 (when pl.pin == 1)
  uint32_t total;
};

__host__ __device__ inline MLayout m_layout(const RecPlan& pl, int N) {
  MLayout L;
  uint32_t off = 0;
  L.b = off;
  off += (uint32_t)pl.KC * pl.nbp * 128u;
  L.ring = off;
  off += (uint32_t)pl.ring * kMRows * 128u;
  L.recv = off;
  off += (uint32_t)pl.rbufs * pl.cluster * N * pl.Uq * 4u;
  L.outs = off;
  off += (uint32_t)N * pl.Uq * 4u;
  L.st_dc = off;
  off += (uint32_t)pl.Uq * N * 4u;
  L.st_carry = off;
  off += (uint32_t)pl.Uq * N * 4u;
  L.pin = off;
  off += pl.pin == 1 ? (uint32_t)kMNIn * pl.Uq * N * 4u : 0u;
  L.total = (off + 1023u) & ~1023u;
  return L;
}

template <bool VL>  // VL: per-sequence lengths (p.lengths) are read
__global__ void __launch_bounds__(kMThreads, 1)
    rec_bwd_tcm(const __grid_constant__ MMaps maps, const __grid_constant__ RecParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * kMStages + 1];
  __shared__ __align__(8) uint64_t rbars[2];  // partial sums landed (two buffers)
  __shared__ uint32_t tmem_slot;
  __shared__ int s_fail, s_stop, s_issued;
  const RecPlan& pl = p.plan;
  const int P = pl.P, Pk = pl.cluster;
  const int d = blockIdx.x / P;
  const int b = blockIdx.x - d * P;
  const int r = b / Pk, q = b - r * Pk;
  const RecDirArgs& a = p.dir[d];
  const int rv = a.rev >= 0 ? a.rev : d;  // reversed time order
  const int H = p.H, N = p.N, nT = p.T, G = p.G, Ur = pl.Ur, Uq = pl.Uq;
  const int64_t GH = (int64_t)G * H;
  const int Urp = pl.nbp;
  const int u0 = r * Ur, Urc = min(Ur, H - u0);
  const int uq0 = q * Uq, Uqc = max(0, min(Uq, Urc - uq0));
  const int k0 = q * pl.Kk;
  const int Kc = (int)max((int64_t)0, min((int64_t)pl.Kk, GH - k0));
  const int nch = (Kc + kMChunk - 1) / kMChunk;
  const int S = pl.ring;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const uint32_t base_s = (smem_addr(smem_raw) + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_s - smem_addr(smem_raw));
  const MLayout Lo = m_layout(pl, N);
  float* recv0 = reinterpret_cast<float*>(base + Lo.recv);
  float* outs = reinterpret_cast<float*>(base + Lo.outs);
  float* st_dc = reinterpret_cast<float*>(base + Lo.st_dc);
  float* st_carry = reinterpret_cast<float*>(base + Lo.st_carry);
  float* pin = reinterpret_cast<float*>(base + Lo.pin);
  const uint32_t full0 = smem_addr(&bars[0]), empty0 = smem_addr(&bars[kMStages]);
  const uint32_t done = smem_addr(&bars[2 * kMStages]);
  const uint32_t ncols = (uint32_t)pl.lda;
  const uint32_t bytesA = kMRows * 128u;
  const int items = Uqc * N;
  const int icap = Uq * N;

  const bool cfg_bad = cl_size() != (unsigned)Pk || cl_rank() != (unsigned)q || N > kMRows ||
                       Urp % 16 != 0 || Urp > 256 || Urp < Ur || (uint32_t)Urp > ncols ||
                       ncols > 512u || (ncols & (ncols - 1u)) != 0 || ncols < 32u ||
                       pl.Kk % kMChunk != 0 || Uq % 4 != 0 || Uq * Pk < Ur || d >= 2 ||
                       S < 2 || S > kMStages || pl.rbufs < 1 || pl.rbufs > 2 || Pk > 8;
  if (tid == 0) {
    s_fail = ld_volatile_int(p.status) != kDevOk || cfg_bad;
    if (cfg_bad) atomicCAS(p.status, kDevOk, kDevCheck);
    s_stop = 0;
    s_issued = 0;
    for (int s = 0; s < kMStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(full0 + 8 * s) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(empty0 + 8 * s) : "memory");
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(done) : "memory");
    for (int i = 0; i < 2; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&rbars[i])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 2 && !cfg_bad) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // resident B = W_hh^T slice: element (unit u, gate row k0 + jj) at atom jj/64,
  // row u, 16-byte chunk (jj%64)/8 (swizzled), 2-byte lane jj%8; consecutive
  // threads read consecutive units of one W_hh row
  {
    const bf16* W = reinterpret_cast<const bf16*>(a.whh);
    const int total = pl.KC * kMChunk * Urp;
    for (int idx = tid; idx < total; idx += kMThreads) {
      const int jj = idx / Urp, u = idx - jj * Urp;
      const bf16 v = (!cfg_bad && u < Urc && jj < Kc) ? W[(int64_t)(k0 + jj) * H + u0 + u]
                                                      : __float2bfloat16_rn(0.f);
      const uint32_t off = (uint32_t)(jj / kMChunk) * (uint32_t)Urp * 128u +
                           sw_off(u, (jj % kMChunk) / 8) + (uint32_t)(jj % 8) * 2u;
      *reinterpret_cast<bf16*>(base + Lo.b + off) = v;
    }
  }
  for (int it = tid; it < items; it += kMThreads) {
    const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
    st_dc[it] = a.dcy ? a.dcy[(int64_t)n * H + j] : 0.f;
    st_carry[it] = 0.f;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_slot;
  unsigned* flags = p.flags + (size_t)d * P * p.flag_stride;
  bf16* dgx = reinterpret_cast<bf16*>(a.dgx);
  bf16* dgh = reinterpret_cast<bf16*>(a.dgh);
  const bf16* hseq = reinterpret_cast<const bf16*>(a.hseq);
  const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(Urp >> 3) << 17) |
                         ((uint32_t)(kMRows >> 4) << 24);
  bool failed = s_fail != 0;
  // with two partial-sum buffers the partials of step s land in buffer s & 1
  // with barrier-completing st.async stores that complete rbars[s & 1]: the
  // owner waits for the bytes, not for a cluster barrier.  Only blocks with a
  // K slice push (one with an empty slice waits on no flag and would run
  // ahead); a pusher's step-s pushes follow its own step s-1 sums and the
  // flags of step s - 1, so buffer s & 1 is free again by then.
  const bool async_rx = pl.rbufs == 2;
  const int pushers = (int)min((int64_t)Pk, (GH + max(1, pl.Kk) - 1) / max(1, pl.Kk));
  const uint32_t rx_bytes = (uint32_t)(pushers * N * ((Uqc + 3) / 4) * 16);
  const uint32_t rbar0 = smem_addr(&rbars[0]);
  // every block's barriers are initialised before any peer pushes into them
  fence_before();
  cl_sync();
  fence_after();
  uint32_t chunk_it = 0;  // ring position (chunks issued over all steps)
  uint32_t done_ph = 0;
  const int q4 = warp & 3, half = warp >> 2;
  const int nrow = q4 * 32 + lane;  // batch row of this thread's tensor-memory lane

  for (int s = 0; s <= nT; ++s) {
    const int t = rv ? s : nT - 1 - s;
    const int tp = rv ? s - 1 : nT - s;
    MTRACE(s, 0);
    const int sc = rv ? t : t + 1, sp = rv ? t + 1 : t;
    // the pointwise inputs of item it at time t: dy, the saved gates, c_t,
    // c_{t-1}
    auto fetch_inputs = [&](int it, float (&v)[kMNIn]) {
      const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
      const int64_t row = (int64_t)t * N + n;
      const int64_t dyo = row * p.lddy + (int64_t)d * H + j;
      v[0] = a.dy_bf16 ? __bfloat162float(reinterpret_cast<const bf16*>(a.dy)[dyo])
                       : reinterpret_cast<const float*>(a.dy)[dyo];
      if (p.mode == 0) {
        v[1] = a.gates[row * H + j];
      } else {
        const float* gp = a.gates + row * 4 * H + j;
#pragma unroll
        for (int g = 0; g < 4; ++g) v[1 + g] = gp[(int64_t)g * H];
        if (p.mode == 1) {
          v[5] = a.cseq[((int64_t)sc * N + n) * H + j];
          v[6] = a.cseq[((int64_t)sp * N + n) * H + j];
        }
      }
    };
    // prefetch: into registers (loads in flight during the contraction), or
    // with cp.async into shared memory
    float rin[kRegItems][kMNIn];
    if (!failed && s < nT && pl.pin == 2) {
      if (warp > 0) {
#pragma unroll
        for (int k = 0; k < kRegItems; ++k) {
          const int it = tid - 32 + k * kRegThreads;
          if (it < items) fetch_inputs(it, rin[k]);
        }
      }
    } else if (!failed && s < nT && pl.pin == 1 && warp > 0) {
      for (int it = tid - 32; it < items; it += kRegThreads) {
        const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
        const int64_t row = (int64_t)t * N + n;
        if (!a.dy_bf16)
          cp_async4(pin + it,
                    reinterpret_cast<const float*>(a.dy) + row * p.lddy + (int64_t)d * H + j);
        if (p.mode == 0) {
          cp_async4(pin + 1 * icap + it, a.gates + row * H + j);
        } else {
          const float* gp = a.gates + row * 4 * H + j;
#pragma unroll
          for (int g = 0; g < 4; ++g) cp_async4(pin + (1 + g) * icap + it, gp + (int64_t)g * H);
          if (p.mode == 1) {
            cp_async4(pin + 5 * icap + it, a.cseq + ((int64_t)sc * N + n) * H + j);
            cp_async4(pin + 6 * icap + it, a.cseq + ((int64_t)sp * N + n) * H + j);
          }
        }
      }
    }
    cp_async_commit();
    const bool have = !failed && s > 0 && Kc > 0;
    if (have) {
      if (warp == 0) {
        // wait for the owners of this block's gate rows, then stream the slice
        bool ok = true;
        for (int g = 0; g < G && ok; ++g) {
          const int lo = max(k0, g * H), hi = min(k0 + Kc, (g + 1) * H);
          if (lo < hi)
            ok = warp_wait_flags(flags, p.flag_stride, owner_flag_m(lo - g * H, Ur, Uq, Pk),
                                 owner_flag_m(hi - 1 - g * H, Ur, Uq, Pk), (unsigned)s, p.status,
                                 p.timeout_ns, p.spin_ns);
        }
        __syncwarp();
        MTRACE(s, 5);
        int c = 0;
        for (; ok && c < nch; ++c) {
          const uint32_t it = chunk_it + (uint32_t)c;
          const uint32_t st = it % (uint32_t)S, ph = (it / (uint32_t)S) & 1u;
          int okl = 1;
          if (lane == 0) {
            okl = mbar_try_wait(empty0 + 8 * st, ph ^ 1u) ? 1 : 0;
            if (!okl) {
              const unsigned long long t0 = globaltimer_ns();
              unsigned spins = 0;
              while (!(okl = mbar_try_wait(empty0 + 8 * st, ph ^ 1u) ? 1 : 0)) {
                if ((++spins & 63u) == 0 && (long long)(globaltimer_ns() - t0) > p.timeout_ns) {
                  atomicCAS(p.status, kDevOk, kDevTimeout);
                  break;
                }
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
          if (!ok) break;
          if (lane == 0) {
            if (c == 0) asm volatile("fence.proxy.async.global;" ::: "memory");
            const uint32_t fb = full0 + 8 * st;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb),
                         "r"(bytesA)
                         : "memory");
            tma3(base_s + Lo.ring + st * bytesA, &maps.a[d], k0 + c * kMChunk, 0, tp, fb);
          }
          __syncwarp();
        }
        MTRACE(s, 6);
        if (lane == 0 && c < nch) {
          s_issued = c;
          __threadfence_block();
          s_stop = 1;
          s_fail = 1;
        }
        __syncwarp();
      } else if (warp == 1 && lane == 0) {
        int c = 0;
        for (; c < nch; ++c) {
          const uint32_t it = chunk_it + (uint32_t)c;
          const uint32_t st = it % (uint32_t)S, ph = (it / (uint32_t)S) & 1u;
          bool got = mbar_try_wait(full0 + 8 * st, ph);
          if (!got) {
            const unsigned long long t0 = globaltimer_ns();
            unsigned spins = 0;
            while (!(got = mbar_try_wait(full0 + 8 * st, ph))) {
              if (ld_volatile_int(&s_stop) && c >= ld_volatile_int(&s_issued)) break;
              if ((++spins & 63u) == 0 && (long long)(globaltimer_ns() - t0) > p.timeout_ns) {
                atomicCAS(p.status, kDevOk, kDevTimeout);
                s_fail = 1;
                break;
              }
            }
          }
          if (!got) break;
          fence_after();
          const uint64_t ad = b_desc(base_s + Lo.ring + st * bytesA);
          const uint64_t bd = b_desc(base_s + Lo.b + (uint32_t)c * (uint32_t)Urp * 128u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss_bf16(tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                        (c > 0 || kk > 0) ? 1u : 0u);
          asm volatile(
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                  empty0 + 8 * st)
              : "memory");
        }
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                done)
            : "memory");
      }
      __syncwarp();
      // the commit above always arrives: every thread waits for it
      const unsigned long long t0 = globaltimer_ns();
      unsigned spins = 0;
      while (!mbar_try_wait(done, done_ph)) {
        if ((++spins & 63u) == 0 && (long long)(globaltimer_ns() - t0) > p.timeout_ns) {
          atomicCAS(p.status, kDevOk, kDevTimeout);
          s_fail = 1;
          break;
        }
      }
      done_ph ^= 1u;
      chunk_it += (uint32_t)nch;
      fence_after();
    }
    __syncthreads();
    failed = s_fail != 0;
    MTRACE(s, 1);
    // push the accumulator rows (batch n) to the owners of the units, 4 units
    // per 16-byte store (Uq is a multiple of 4)
    float* recv = recv0 + (size_t)(pl.rbufs == 2 ? (s & 1) : 0) * Pk * N * Uq;
    const uint32_t rbar = rbar0 + 8u * (uint32_t)(s & 1);
    if (async_rx && !failed && s > 0 && tid == 0) mbar_arrive_expect_tx(rbar, rx_bytes);
    if (!failed && s > 0 && (!async_rx || Kc > 0)) {
      for (int cg = half; cg < Urp / 4; cg += 2) {
        float v[4];
        tmem_ld4m(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(cg * 4), v);
        const int u = cg * 4;
        if (nrow >= N || u >= Urc) continue;
        const int owner = u / Uq, uo = u - owner * Uq;
        if (owner >= Pk) continue;
        float* dst = recv + ((size_t)q * N + nrow) * Uq + uo;
        if (async_rx)
          st_async4(dst, rbar, (unsigned)owner, have ? v[0] : 0.f, have ? v[1] : 0.f,
                    have ? v[2] : 0.f, have ? v[3] : 0.f);
        else
          st_peer4(dst, (unsigned)owner, have ? v[0] : 0.f, have ? v[1] : 0.f, have ? v[2] : 0.f,
                   have ? v[3] : 0.f);
      }
    }
    fence_before();
    if (async_rx) {
      // this step's partials: the owners' threads wait for the pushed bytes
      if (!failed && s > 0 && tid < items &&
          !mbar_wait_cluster_bounded(rbar, (uint32_t)((s - 1) >> 1) & 1u, p.status,
                                     p.timeout_ns))
        s_fail = 1;
    } else {
      cl_sync();
    }
    if (!failed && s > 0) {
      const int nsum = async_rx ? pushers : Pk;
      for (int it = tid; it < items; it += kMThreads) {
        const int uu = it % Uqc, n = it / Uqc;
        outs[n * Uq + uu] = sum_strided<8>(recv + (size_t)n * Uq + uu, (size_t)N * Uq, nsum);
      }
    }
    // one partial-sum buffer: nobody pushes the next step's partials before
    // every owner has summed this step's
    if (pl.rbufs == 1) cl_sync();
    cp_async_wait_all();
    __syncthreads();
    failed = s_fail != 0;  // a wait for the partials may have given up
    MTRACE(s, 2);
    // one item's gate-gradient chain; v = its inputs (unused at s == nT)
    auto point = [&](int it, const float (&v)[kMNIn]) {
      const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
      float dhf;
      if (s == 0)
        dhf = a.dhy ? __bfloat162float(reinterpret_cast<const bf16*>(a.dhy)[(int64_t)n * H + j])
                    : 0.f;
      else
        dhf = outs[n * Uq + uu] + st_carry[it];
      if (s == nT) {
        if (a.dh0) reinterpret_cast<bf16*>(a.dh0)[(int64_t)n * H + j] = __float2bfloat16_rn(dhf);
        if (a.dc0) a.dc0[(int64_t)n * H + j] = st_dc[it];
        return;
      }
      const int64_t row = (int64_t)t * N + n;
      bf16* gxo = dgx + row * GH + j;
      if (VL && t >= __ldg(p.lengths + n)) {
        // a step the forward skipped (past the sequence's length): no gate
        // gradients, dy unused, dh and (LSTM) dc pass straight through
        const int G = p.mode == 1 ? 4 : p.mode == 2 ? 3 : 1;
        for (int g = 0; g < G; ++g) gxo[(int64_t)g * H] = __float2bfloat16_rn(0.f);
        if (p.mode == 2) {
          bf16* gho = dgh + row * GH + j;
          for (int g = 0; g < 3; ++g) gho[(int64_t)g * H] = __float2bfloat16_rn(0.f);
        }
        st_carry[it] = dhf;
        return;
      }
      const float dh = v[0] + dhf;
      const float g0 = v[1];
      if (p.mode == 1) {  // LSTM: g0..g3 = i, f, g, o
        const float g1 = v[2], g2 = v[3], g3 = v[4], cc = v[5], cpv = v[6];
        const float tc = tanhf(cc);
        const float dc = st_dc[it] + dh * g3 * (1.f - tc * tc);
        gxo[0] = __float2bfloat16_rn(dc * g2 * g0 * (1.f - g0));
        gxo[H] = __float2bfloat16_rn(dc * cpv * g1 * (1.f - g1));
        gxo[2 * H] = __float2bfloat16_rn(dc * g0 * (1.f - g2 * g2));
        gxo[3 * H] = __float2bfloat16_rn(dh * tc * g3 * (1.f - g3));
        st_dc[it] = dc * g1;
        if (VL) st_carry[it] = 0.f;  // a pass-through ends here
      } else if (p.mode == 2) {  // GRU: g0..g3 = r, z, n, W_hn h + b_hn
        const float g1 = v[2], g2 = v[3], g3 = v[4];
        const float hp = __bfloat162float(hseq[((int64_t)sp * N + n) * H + j]);
        const float dan = dh * (1.f - g1) * (1.f - g2 * g2);
        const float daz = dh * (hp - g2) * g1 * (1.f - g1);
        const float dar = dan * g3 * g0 * (1.f - g0);
        gxo[0] = __float2bfloat16_rn(dar);
        gxo[H] = __float2bfloat16_rn(daz);
        gxo[2 * H] = __float2bfloat16_rn(dan);
        bf16* gho = dgh + row * GH + j;
        gho[0] = __float2bfloat16_rn(dar);
        gho[H] = __float2bfloat16_rn(daz);
        gho[2 * H] = __float2bfloat16_rn(dan * g0);
        st_carry[it] = dh * g1;
      } else {  // tanh RNN: g0 = h_t
        gxo[0] = __float2bfloat16_rn(dh * (1.f - g0 * g0));
        if (VL) st_carry[it] = 0.f;
      }
    };
    if (!failed) {
      if (pl.pin == 2) {
        if (warp > 0) {
#pragma unroll
          for (int k = 0; k < kRegItems; ++k) {
            const int it = tid - 32 + k * kRegThreads;
            if (it < items) point(it, rin[k]);
          }
        }
      } else {
        for (int it = tid; it < items; it += kMThreads) {
          float v[kMNIn];
          if (s < nT) {
            if (pl.pin == 1) {
#pragma unroll
              for (int k = 0; k < kMNIn; ++k) v[k] = pin[k * icap + it];
              if (a.dy_bf16) {
                const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
                v[0] = __bfloat162float(reinterpret_cast<const bf16*>(
                    a.dy)[((int64_t)t * N + n) * p.lddy + (int64_t)d * H + j]);
              }
            } else {
              fetch_inputs(it, v);
            }
          }
          point(it, v);
        }
      }
    }
    fence_before();
    __syncthreads();
    MTRACE(s, 3);
    if (!failed && tid == 0 && s < nT && !(blockIdx.x == p.fault_block && s == p.fault_step)) {
      // this block's dG stores (ordered before this thread by the barrier)
      // become visible to the other blocks' tensor loads: proxy fence, release
      asm volatile("fence.proxy.async.global;" ::: "memory");
      publish_flag(flags + (size_t)b * p.flag_stride, (unsigned)(s + 1));
    }
    MTRACE(s, 4);
  }
  cl_sync();  // no block leaves while a peer may still store into it
  fence_before();
  __syncthreads();
  if (warp == 2 && !cfg_bad)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols)
                 : "memory");
}

}  // namespace

bool rec_tcm_bwd_plan(int mode, int bf16, int D, int H, int N, int num_sms, size_t smem_limit,
                      const int* max_clusters, RecPlan* out) {
  if (!bf16 || N < 64 || N > kMRows || H % 8 != 0) return false;
  const int G = mode == 1 ? 4 : mode == 2 ? 3 : 1;
  const int GH = G * H;
  bool found = false;
  double best = 0;
  RecPlan bp;
  for (int Pk : {4, 8, 2}) {
    const int cap = max_clusters[Pk];
    const int Pr_max = std::min(cap / D, (num_sms / D) / Pk);
    if (Pr_max < 1) continue;
    const int Ur = (H + Pr_max - 1) / Pr_max;
    const int Urp = (Ur + 15) / 16 * 16;
    if (Urp > 256) continue;
    const int Pr = (H + Ur - 1) / Ur;
    const int Uq = ((Ur + Pk - 1) / Pk + 3) / 4 * 4;
    const int Kk = ((GH + Pk - 1) / Pk + kMChunk - 1) / kMChunk * kMChunk;
    int cols = 32;
    while (cols < Urp) cols *= 2;
    RecPlan pl;
    pl.direct = 0;
    pl.cluster = Pk; pl.Pr = Pr; pl.P = Pr * Pk; pl.Ur = Ur; pl.Uq = Uq;
    pl.Kk = Kk;
    pl.K = Kk;
    pl.KC = Kk / kMChunk;
    pl.nbp = Urp;
    pl.lda = cols;
    pl.Mloc = Ur; pl.Mp = kMRows; pl.nb = N;
    pl.tc = 3;
    // as many ring stages (bytes in flight on the dG_h stream) as fit, for
    // each of: prefetched pointwise inputs (in registers when they fit, else
    // in shared memory) with double-buffered partial sums, the same with one
    // partial-sum buffer, no prefetch with two, no prefetch with one
    // per-step time model (microseconds, fitted to step traces of this kernel):
    // the dG_h stream, about 2 us per 64 KB of the slice; pointwise items cost
    // 0.3 us each with prefetched inputs and 1.4 us reading them inline; a
    // single partial-sum buffer costs a second cluster barrier
    const bool regs = (Uq * N + kRegThreads - 1) / kRegThreads <= kRegItems;
    // registers whenever the items fit (measured faster than shared memory)
    const int cfgs[4][2] = {{regs ? 2 : 1, 2}, {regs ? 2 : 0, 1}, {0, 2}, {0, 1}};
    double best_cfg = 0;
    int best_ring = 0, best_pin = 1, best_rb = 2;
    for (int cfg = 0; cfg < 4; ++cfg) {
      pl.pin = cfgs[cfg][0];
      pl.rbufs = cfgs[cfg][1];
      pl.ring = 0;
      const size_t fixed = m_layout(pl, N).total + 1024;
      // four stages: a deeper ring was measured no faster (the slice is read
      // by every row group at once; the stream is bound by L2, not in-flight
      // bytes)
      const int ring = fixed < smem_limit
                           ? (int)std::min<size_t>(kRingUse, (smem_limit - fixed) / (kMRows * 128))
                           : 0;
      if (ring < 2) continue;
      const int workers = pl.pin == 2 ? kRegThreads : kMThreads;
      const double per_thread = (double)((Uq * N + workers - 1) / workers);
      const double t_stream = (double)Kk * kMRows * 2.0 / (kRingUse * kMRows * 128.0) * 2.0 *
                              (ring < kRingUse ? (double)kRingUse / ring : 1.0);
      const double t_point = per_thread * (pl.pin ? 0.3 : 1.4);
      const double t_red = 1.0 + 0.02 * Pk * Uq * N / kMThreads + (pl.rbufs == 1 ? 2.0 : 0.0);
      const double t = t_stream + t_point + t_red;
      if (best_ring == 0 || t < best_cfg) {
        best_cfg = t;
        best_ring = ring;
        best_pin = pl.pin;
        best_rb = pl.rbufs;
      }
    }
    if (best_ring < 2) continue;
    pl.ring = best_ring; pl.pin = best_pin; pl.rbufs = best_rb;
    const MLayout L = m_layout(pl, N);
    pl.smem = std::max<size_t>(L.total + 1024, 120 * 1024);
    if (pl.smem > smem_limit) continue;
    if (D * pl.P > num_sms) continue;
    const double cost = best_cfg;
    if (!found || cost < best) {
      found = true;
      best = cost;
      bp = pl;
    }
  }
  if (found) *out = bp;
  return found;
}

#ifdef LAYER_RNN_TRACE
extern "C" int rnn_debug_mtrace_copy(void* host, size_t bytes) {
  if (bytes > sizeof(g_mtrace)) bytes = sizeof(g_mtrace);
  return (int)cudaMemcpyFromSymbol(host, g_mtrace, bytes);
}
extern "C" int rnn_debug_mtrace_clear() {
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_mtrace);
  if (e == cudaSuccess) e = cudaMemset(ptr, 0, sizeof(g_mtrace));
  return (int)e;
}
#endif

cudaError_t rec_tcm_bwd_launch(const RecParams& p, cudaStream_t st) {
  const RecPlan& pl = p.plan;
  MMaps maps;
  memset(&maps, 0, sizeof(maps));
  const uint64_t GH = (uint64_t)p.G * p.H, N = (uint64_t)p.N, T = (uint64_t)p.T;
  for (int d = 0; d < p.D; ++d) {
    const uint64_t dims[3] = {GH, N, T}, strides[2] = {GH * 2, N * GH * 2};
    const uint32_t box[3] = {(uint32_t)kMChunk, (uint32_t)kMRows, 1u};
    if (!tma_encode(&maps.a[d], 3, true, p.dir[d].dgh, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  void* fn = p.lengths ? (void*)rec_bwd_tcm<true> : (void*)rec_bwd_tcm<false>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.flags, 0, sizeof(unsigned) * (size_t)p.D * pl.P * p.flag_stride, st);
  if (e != cudaSuccess) return e;
  RecParams copy = p;
  void* args[] = {&maps, &copy};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.D * pl.P);
  cfg.blockDim = dim3(kMThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace lr
