// Tensor-core path of the persistent recurrent backward kernel.
//
// Backward through time (reverse-mode through the recurrences of the
// "rnn training example?" thread, reading 13 of the design notes for the
// loss): per step
//     dh_{t-1}[n][k] = sum_j dG_h[t][n][j] * W_hh[j][k]   (+ GRU: dh_t[n][k] * z_t[n][k])
// with j over the G*H gate rows.  The contraction is K = G*H long, so the
// blocks of a cluster (up to 16, a non-portable cluster size) split it: block
// (r, q) keeps W_hh^T for the Ur units of row group r and the gate rows
// k0 .. k0+Kk-1 in tensor memory as the MMA's A operand (fp32: tf32 hi and lo
// parts, three passes; bf16: one pass, two elements per 32-bit column), stages
// the previous step's dG_h slice as the swizzled K-major B operand, and pushes
// each row of the accumulator over distributed shared memory (16-byte stores)
// to the block that owns the unit's pointwise step.  The owners sum the Pk
// partials in a fixed order, run the gate-gradient chain, store dG_x (and
// dG_h for the GRU) and release their step flag.  The pointwise inputs of the
// step (dy, the saved gates, c_t and c_{t-1}) are fetched with cp.async at
// the start of the step, so their latency hides behind the contraction.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "rec.h"
#include "tc_common.cuh"

#ifdef LAYER_RNN_TRACE
__device__ unsigned long long g_btrace[4][1024][8];
#define BTRACE(s, k)                                                                          \
  do {                                                                                        \
    const int nb_ = gridDim.x;                                                                \
    const int b_ = blockIdx.x == 0 ? 0 : blockIdx.x == nb_ / 3 ? 1 : blockIdx.x == (2 * nb_) / 3 \
                 ? 2 : blockIdx.x == nb_ - 1 ? 3 : -1;                                       \
    if (b_ >= 0 && threadIdx.x == 0 && (s) < 1024) g_btrace[b_][(s)][(k)] = lr::globaltimer_ns();\
  } while (0)
#else
#define BTRACE(s, k) ((void)0)
#endif

namespace lr {

namespace {

using namespace tc;

constexpr int kBThreads = 256;
constexpr int kBM = 128;    // MMA M: output units per row group (padded)
constexpr int kNIn = 7;     // pointwise inputs per item: dy, 4 gates, c_t, c_{t-1} / h_{t-1}

__device__ __forceinline__ int owner_flag_b(int u, int Ur, int Uq, int Pk) {
  const int r = u / Ur;
  return r * Pk + (u - r * Ur) / Uq;
}

struct BLayout {
  uint32_t b_hi, b_lo;   // staged B tiles: KC atoms x (Nm rows x 128 bytes)
  uint32_t recv;         // [2][Pk][Uq][Nm] f32
  uint32_t outs;         // [N][Uq] f32 summed partials
  uint32_t st_dc, st_carry;  // [Uq*N] f32: LSTM dc, GRU dh*z
  uint32_t pin;          // [kNIn][Uq*N] f32
  uint32_t total;
};

__host__ __device__ inline BLayout b_layout(const RecPlan& pl, int N, bool bf) {
  BLayout L;
  const uint32_t atom = (uint32_t)pl.nbp * 128u;
  const uint32_t ntile = (uint32_t)pl.KC * atom;
  uint32_t off = 0;
  L.b_hi = off;
  off += ntile;
  L.b_lo = off;
  off += bf ? 0 : ntile;
  L.recv = off;
  off += 2u * pl.cluster * pl.Uq * pl.nbp * 4u;
  L.outs = off;
  off += (uint32_t)pl.Uq * N * 4u;
  L.st_dc = off;
  off += (uint32_t)pl.Uq * N * 4u;
  L.st_carry = off;
  off += (uint32_t)pl.Uq * N * 4u;
  L.pin = off;
  off += (uint32_t)kNIn * pl.Uq * N * 4u;
  L.total = (off + 1023u) & ~1023u;
  return L;
}

template <bool BF>
__global__ void __launch_bounds__(kBThreads, 1) rec_bwd_tc(const __grid_constant__ RecParams p) {
  typedef typename std::conditional<BF, bf16, float>::type T;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int s_fail;
  const RecPlan& pl = p.plan;
  const int P = pl.P, Pk = pl.cluster;
  const int d = blockIdx.x / P;
  const int b = blockIdx.x - d * P;
  const int r = b / Pk, q = b - r * Pk;
  const RecDirArgs& a = p.dir[d];
  const int rv = a.rev >= 0 ? a.rev : d;  // reversed time order
  const int H = p.H, N = p.N, nT = p.T, G = p.G, Ur = pl.Ur, Uq = pl.Uq;
  const int64_t GH = (int64_t)G * H;
  const int Nm = pl.nbp, Kp = pl.K;
  const int u0 = r * Ur, Urc = min(Ur, H - u0);
  const int uq0 = q * Uq, Uqc = max(0, min(Uq, Urc - uq0));
  const int k0 = q * pl.Kk;
  const int Kc = (int)max((int64_t)0, min((int64_t)pl.Kk, GH - k0));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const uint32_t base_s = (smem_addr(smem_raw) + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_s - smem_addr(smem_raw));
  const BLayout Lo = b_layout(pl, N, BF);
  float* recv0 = reinterpret_cast<float*>(base + Lo.recv);
  float* outs = reinterpret_cast<float*>(base + Lo.outs);
  float* st_dc = reinterpret_cast<float*>(base + Lo.st_dc);
  float* st_carry = reinterpret_cast<float*>(base + Lo.st_carry);
  float* pin = reinterpret_cast<float*>(base + Lo.pin);
  const uint32_t atom_bytes = (uint32_t)Nm * 128u;
  const uint32_t bar = smem_addr(&mma_bar);
  const uint32_t a_col = (uint32_t)Nm;
  const uint32_t a_lo_col = (uint32_t)(Nm + Kp);
  const uint32_t ncols = (uint32_t)pl.lda;
  const int items = Uqc * N;
  const int icap = Uq * N;  // stride of one input array in pin

  const bool cfg_bad = cl_size() != (unsigned)Pk || cl_rank() != (unsigned)q ||
                       (uint32_t)(Nm + (BF ? Kp / 2 : 2 * Kp)) > ncols || ncols > 512u ||
                       (ncols & (ncols - 1u)) != 0 || ncols < 32u || Ur > kBM || N > Nm ||
                       Nm % 16 != 0 || Nm > 256 || Kp % (BF ? 64 : 32) != 0 || pl.Kk > Kp ||
                       Uq * Pk < Ur;
  if (tid == 0) {
    s_fail = ld_volatile_int(p.status) != kDevOk || cfg_bad;
    if (cfg_bad) atomicCAS(p.status, kDevOk, kDevCheck);
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && !cfg_bad) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  for (uint32_t i = tid; i < Lo.recv / 16u; i += kBThreads)
    reinterpret_cast<uint4*>(base)[i] = make_uint4(0, 0, 0, 0);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_slot;

  // A = W_hh^T slice into tensor memory: lane m = unit u0 + m, columns = gate
  // rows k0 + jj; lanes of a warp read consecutive units of one W_hh row
  if (!cfg_bad) {
    const T* W = reinterpret_cast<const T*>(a.whh);
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const bool row_ok = m < Urc;
    const int epc = BF ? 64 : 32;
    const int nchunk = Kp / epc;
    for (int ci = warp >> 2; ci < nchunk; ci += kBThreads / 128) {
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (BF) {
          const int jj = ci * 64 + 2 * i;
          const float e0 = (row_ok && jj < Kc) ? to_f(W[(int64_t)(k0 + jj) * H + u0 + m]) : 0.f;
          const float e1 =
              (row_ok && jj + 1 < Kc) ? to_f(W[(int64_t)(k0 + jj + 1) * H + u0 + m]) : 0.f;
          hi[i] = (__float_as_uint(e0) >> 16) | ((__float_as_uint(e1) >> 16) << 16);
          lo[i] = 0;
        } else {
          const int jj = ci * 32 + i;
          const float v = (row_ok && jj < Kc) ? to_f(W[(int64_t)(k0 + jj) * H + u0 + m]) : 0.f;
          const uint32_t hb = __float_as_uint(v) & 0xFFFFE000u;
          hi[i] = hb;
          lo[i] = __float_as_uint(v - __uint_as_float(hb));
        }
      }
      const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
      tmem_st32(tmem + lane_base + a_col + (uint32_t)(ci * 32), hi);
      if (!BF) tmem_st32(tmem + lane_base + a_lo_col + (uint32_t)(ci * 32), lo);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  }

  // state of the own items: item it = n * Uqc + uu (consecutive threads take
  // consecutive units: coalesced global accesses)
  for (int it = tid; it < items; it += kBThreads) {
    const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
    st_dc[it] = a.dcy ? a.dcy[(int64_t)n * H + j] : 0.f;
    st_carry[it] = 0.f;
  }
  unsigned* flags = p.flags + (size_t)d * P * p.flag_stride;
  T* dgx = reinterpret_cast<T*>(a.dgx);
  T* dgh = reinterpret_cast<T*>(a.dgh);
  const T* hseq = reinterpret_cast<const T*>(a.hseq);
  const uint32_t idesc = (1u << 4) | ((BF ? 1u : 2u) << 7) | ((BF ? 1u : 2u) << 10) |
                         ((uint32_t)(Nm >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
  const int kstep = BF ? 16 : 8;
  const int nsteps = (Kc + kstep - 1) / kstep;
  fence_before();
  __syncthreads();
  fence_after();
  bool failed = s_fail != 0;
  uint32_t phase = 0;

  for (int s = 0; s <= nT; ++s) {
    const int t = rv ? s : nT - 1 - s;   // time processed at this step (s < nT)
    const int tp = rv ? s - 1 : nT - s;  // time processed at the previous step (s > 0)
    BTRACE(s, 0);
    // pointwise inputs of time t (fp32 sources by cp.async; bf16 ones are read
    // in the pointwise loop)
    if (!failed && s < nT) {
      const int sc = rv ? t : t + 1, sp = rv ? t + 1 : t;
      for (int it = tid; it < items; it += kBThreads) {
        const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
        const int64_t row = (int64_t)t * N + n;
        if (!a.dy_bf16)
          cp_async4(pin + 0 * icap + it,
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
          } else if (!BF) {
            cp_async4(pin + 6 * icap + it,
                      reinterpret_cast<const float*>(hseq) + ((int64_t)sp * N + n) * H + j);
          }
        }
      }
    }
    cp_async_commit();
    // the previous step's dG_h slice: wait for the blocks that own its units
    if (!failed && s > 0 && Kc > 0 && warp == 0) {
      bool ok = true;
      for (int g = 0; g < G && ok; ++g) {
        const int lo = max(k0, g * H), hi = min(k0 + Kc, (g + 1) * H);
        if (lo < hi)
          ok = warp_wait_flags(flags, p.flag_stride, owner_flag_b(lo - g * H, Ur, Uq, Pk),
                               owner_flag_b(hi - 1 - g * H, Ur, Uq, Pk), (unsigned)s, p.status,
                               p.timeout_ns, p.spin_ns);
      }
      if (!ok && lane == 0) s_fail = 1;
    }
    __syncthreads();
    BTRACE(s, 1);
    failed = s_fail != 0;
    const bool have = !failed && s > 0 && Kc > 0;
    if (have) {
      constexpr int VE = 16 / (int)sizeof(T);
      const int nv = Kc / VE;
      const T* src = dgh + (int64_t)tp * N * GH + k0;
      for (int idx = tid; idx < N * nv; idx += kBThreads) {
        const int n = idx / nv, c16 = idx - n * nv;
        const uint4 v = ldcg16(src + (int64_t)n * GH + c16 * VE);
        const int atom = c16 >> 3, c = c16 & 7;
        const uint32_t off = (uint32_t)atom * atom_bytes + sw_off(n, c);
        if (BF) {
          *reinterpret_cast<uint4*>(base + Lo.b_hi + off) = v;
        } else {
          uint4 h4, l4;
          h4.x = v.x & 0xFFFFE000u; l4.x = __float_as_uint(__uint_as_float(v.x) - __uint_as_float(h4.x));
          h4.y = v.y & 0xFFFFE000u; l4.y = __float_as_uint(__uint_as_float(v.y) - __uint_as_float(h4.y));
          h4.z = v.z & 0xFFFFE000u; l4.z = __float_as_uint(__uint_as_float(v.z) - __uint_as_float(h4.z));
          h4.w = v.w & 0xFFFFE000u; l4.w = __float_as_uint(__uint_as_float(v.w) - __uint_as_float(h4.w));
          *reinterpret_cast<uint4*>(base + Lo.b_hi + off) = h4;
          *reinterpret_cast<uint4*>(base + Lo.b_lo + off) = l4;
        }
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    fence_before();
    __syncthreads();
    fence_after();
    BTRACE(s, 6);
    if (have && tid == 0) {
      for (int ks = 0; ks < nsteps; ++ks) {
        const uint32_t atom = (uint32_t)(ks >> 2), kk = (uint32_t)(ks & 3);
        const uint64_t bh = b_desc(base_s + Lo.b_hi + atom * atom_bytes) + kk * 2;
        const uint32_t acc0 = ks > 0 ? 1u : 0u;
        if (BF) {
          mma_a_tmem(true, tmem, tmem + a_col + (uint32_t)(ks * 8), bh, idesc, acc0);
        } else {
          const uint64_t bl = b_desc(base_s + Lo.b_lo + atom * atom_bytes) + kk * 2;
          mma_a_tmem(false, tmem, tmem + a_col + (uint32_t)(ks * 8), bh, idesc, acc0);
          mma_a_tmem(false, tmem, tmem + a_col + (uint32_t)(ks * 8), bl, idesc, 1u);
          mma_a_tmem(false, tmem, tmem + a_lo_col + (uint32_t)(ks * 8), bh, idesc, 1u);
        }
      }
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
          : "memory");
    }
    bool mma_ok = true;
    if (have) {
      mma_ok = mbar_wait_bounded(bar, phase, p.status, p.timeout_ns);
      phase ^= 1u;
    }
    fence_after();
    BTRACE(s, 2);
    // push each accumulator row (unit u0 + m) to the block that owns the unit
    float* recv = recv0 + (size_t)(s & 1) * Pk * Uq * Nm;
    if (!failed && s > 0) {
      const int quarter = warp & 3;
      const int m = quarter * 32 + lane;
      const bool row_ok = m < Urc;
      const int owner = row_ok ? m / Uq : 0, uo = m - owner * Uq;
      for (int c0 = (warp >> 2) * 32; c0 < Nm; c0 += (kBThreads / 128) * 32) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0, v);
        if (!row_ok || owner >= Pk) continue;
        float* dst = recv + ((size_t)q * Uq + uo) * Nm + c0;
        const bool ok = have && mma_ok;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          if (c0 + i < N)
            st_peer4(dst + i, (unsigned)owner, ok ? v[i] : 0.f, ok ? v[i + 1] : 0.f,
                     ok ? v[i + 2] : 0.f, ok ? v[i + 3] : 0.f);
      }
    }
    fence_before();
    cl_sync();
    if (!failed && s > 0) {
      // batch index fastest: consecutive threads read consecutive partials
      for (int idx = tid; idx < items; idx += kBThreads) {
        const int n = idx % N, uu = idx / N;
        float v = 0.f;
        for (int rank = 0; rank < Pk; ++rank) v += recv[((size_t)rank * Uq + uu) * Nm + n];
        outs[n * Uq + uu] = v;
      }
    }
    cp_async_wait_all();
    __syncthreads();
    BTRACE(s, 3);
    if (!failed) {
      for (int it = tid; it < items; it += kBThreads) {
        const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
        float dhf;
        if (s == 0)
          dhf = a.dhy ? to_f(reinterpret_cast<const T*>(a.dhy)[(int64_t)n * H + j]) : 0.f;
        else
          dhf = outs[n * Uq + uu] + st_carry[it];
        if (s == nT) {
          if (a.dh0) reinterpret_cast<T*>(a.dh0)[(int64_t)n * H + j] = from_f<T>(dhf);
          if (a.dc0) a.dc0[(int64_t)n * H + j] = st_dc[it];
          continue;
        }
        const int64_t row = (int64_t)t * N + n;
        const float dyv = a.dy_bf16
                              ? to_f(reinterpret_cast<const bf16*>(a.dy)[row * p.lddy + (int64_t)d * H + j])
                              : pin[it];
        const float dh = dyv + dhf;
        const float g0 = pin[1 * icap + it];
        T* gxo = dgx + row * GH + j;
        if (p.mode == 1) {  // LSTM: g0..g3 = i, f, g, o
          const float g1 = pin[2 * icap + it], g2 = pin[3 * icap + it], g3 = pin[4 * icap + it];
          const float cc = pin[5 * icap + it], cpv = pin[6 * icap + it];
          const float tc = tanhf(cc);
          const float dc = st_dc[it] + dh * g3 * (1.f - tc * tc);
          gxo[0] = from_f<T>(dc * g2 * g0 * (1.f - g0));
          gxo[H] = from_f<T>(dc * cpv * g1 * (1.f - g1));
          gxo[2 * H] = from_f<T>(dc * g0 * (1.f - g2 * g2));
          gxo[3 * H] = from_f<T>(dh * tc * g3 * (1.f - g3));
          st_dc[it] = dc * g1;
        } else if (p.mode == 2) {  // GRU: g0..g3 = r, z, n, W_hn h + b_hn
          const float g1 = pin[2 * icap + it], g2 = pin[3 * icap + it], g3 = pin[4 * icap + it];
          const int sp = rv ? t + 1 : t;
          const float hp = BF ? to_f(hseq[((int64_t)sp * N + n) * H + j]) : pin[6 * icap + it];
          const float dan = dh * (1.f - g1) * (1.f - g2 * g2);
          const float daz = dh * (hp - g2) * g1 * (1.f - g1);
          const float dar = dan * g3 * g0 * (1.f - g0);
          gxo[0] = from_f<T>(dar);
          gxo[H] = from_f<T>(daz);
          gxo[2 * H] = from_f<T>(dan);
          T* gho = dgh + row * GH + j;
          gho[0] = from_f<T>(dar);
          gho[H] = from_f<T>(daz);
          gho[2 * H] = from_f<T>(dan * g0);
          st_carry[it] = dh * g1;
        } else {  // tanh RNN: g0 = h_t
          gxo[0] = from_f<T>(dh * (1.f - g0 * g0));
        }
      }
    }
    __syncthreads();
    BTRACE(s, 4);
    if (!failed && tid == 0 && s < nT && !(blockIdx.x == p.fault_block && s == p.fault_step))
      publish_flag(flags + (size_t)b * p.flag_stride, (unsigned)(s + 1));
    BTRACE(s, 5);
  }
  cl_sync();  // no block leaves while a peer may still store into it
  fence_before();
  __syncthreads();
  if (warp == 0 && !cfg_bad)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols)
                 : "memory");
}

void* bwd_kernel(bool bf) {
  return bf ? (void*)rec_bwd_tc<true> : (void*)rec_bwd_tc<false>;
}

}  // namespace

int rec_tc_bwd_capacity(int cluster, size_t smem) {
  void* fn = bwd_kernel(false);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster * 16);
  cfg.blockDim = dim3(kBThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

bool rec_tc_bwd_plan(int mode, int bf16, int D, int H, int N, int num_sms, size_t smem_limit,
                     const int* caps, RecPlan* out) {
  const int G = mode == 1 ? 4 : mode == 2 ? 3 : 1;
  const int e = bf16 ? 2 : 4;
  if ((H * e) % 16 != 0 || N < 1 || N > 256) return false;
  const int GH = G * H;
  const int Nm = (N + 15) / 16 * 16;
  bool found = false;
  double best = 0;
  RecPlan bp;
  for (int Pk : {16, 14, 12, 8, 4}) {
    const int cap = caps[Pk];
    const int Pr_max = std::min(cap / D, (num_sms / D) / Pk);
    if (Pr_max < 1) continue;
    const int Ur = (H + Pr_max - 1) / Pr_max;
    if (Ur > kBM) continue;
    const int Pr = (H + Ur - 1) / Ur;
    const int Uq = (Ur + Pk - 1) / Pk;
    const int epc = bf16 ? 64 : 32;
    const int Kk = (((GH + Pk - 1) / Pk) + 7) / 8 * 8;
    const int Kp = (Kk + epc - 1) / epc * epc;
    const int acols = bf16 ? Kp / 2 : 2 * Kp;
    int cols = 32;
    while (cols < Nm + acols) cols *= 2;
    if (cols > 512) continue;
    RecPlan pl;
    pl.direct = 0;
    pl.cluster = Pk; pl.Pr = Pr; pl.P = Pr * Pk; pl.Ur = Ur; pl.Uq = Uq;
    pl.Kk = Kk;
    pl.K = Kp;
    pl.KC = Kp / (bf16 ? 64 : 32);
    pl.nbp = Nm;
    pl.lda = cols;
    pl.Mloc = Ur; pl.Mp = kBM; pl.nb = N;
    pl.tc = 2;
    const BLayout L = b_layout(pl, N, bf16 != 0);
    pl.smem = std::max<size_t>(L.total + 1024, 120 * 1024);
    if (pl.smem > smem_limit) continue;
    if (D * pl.P > num_sms) continue;
    // MMA issue (K slice, passes), the push of Ur rows, the owners' reduction
    // over Pk partials and their pointwise items
    const double cost = (double)Kp * (bf16 ? 1 : 3) * (Nm / 32.0) * 2.0 + (double)Ur * N / 16.0 +
                        (double)Uq * N * (Pk / 4.0 + 8.0);
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
extern "C" int rnn_debug_btrace_copy(void* host, size_t bytes) {
  if (bytes > sizeof(g_btrace)) bytes = sizeof(g_btrace);
  return (int)cudaMemcpyFromSymbol(host, g_btrace, bytes);
}
extern "C" int rnn_debug_btrace_clear() {
  static unsigned long long zeros[4][1024][8];
  return (int)cudaMemcpyToSymbol(g_btrace, zeros, sizeof(zeros));
}
#endif

cudaError_t rec_tc_bwd_launch(const RecParams& p, cudaStream_t st) {
  const RecPlan& pl = p.plan;
  void* fn = bwd_kernel(p.bf16 != 0);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  if (pl.cluster > 8) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  e = cudaMemsetAsync(p.flags, 0, sizeof(unsigned) * (size_t)p.D * pl.P * p.flag_stride, st);
  if (e != cudaSuccess) return e;
  RecParams copy = p;
  void* args[] = {&copy};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.D * pl.P);
  cfg.blockDim = dim3(kBThreads);
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
