// Tensor-core path of the persistent recurrent forward kernel.
//
// Same 2-D decomposition as the cluster path (clusters own row groups of
// hidden units, the blocks of a cluster split the contraction length K), but
// each block's per-step product
//     D[m][n] = sum_k W_hh[row m][k0 + k] * h_{t-1}[n][k0 + k]      (m < 128)
// runs on the tensor cores: the block's W_hh slice stays for the whole
// sequence in tensor memory as the MMA's A operand (fp32: tf32 hi and lo
// parts, three passes hi*hi + hi*lo + lo*hi as in the dense phases; bf16: one
// pass, two elements per 32-bit column), the step's h slice is staged into
// shared memory in the 128-byte-swizzled K-major layout the MMA reads as B,
// and the accumulator D lands in tensor memory.  D's rows are pushed over
// distributed shared memory to the blocks that own the units' pointwise math,
// as in the cluster path.  All waits are bounded; the cluster barriers are
// executed by every block on every step, work or not.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "rec.h"
#include "tc_common.cuh"

#ifdef LAYER_RNN_TRACE
__device__ unsigned long long g_ttrace[4][1024][8];
#define TTRACE(s, k)                                                                          \
  do {                                                                                        \
    const int nb_ = gridDim.x;                                                                \
    const int b_ = blockIdx.x == 0 ? 0 : blockIdx.x == nb_ / 3 ? 1 : blockIdx.x == (2 * nb_) / 3 \
                 ? 2 : blockIdx.x == nb_ - 1 ? 3 : -1;                                       \
    if (b_ >= 0 && threadIdx.x == 0 && (s) < 1024) g_ttrace[b_][(s)][(k)] = lr::globaltimer_ns();\
  } while (0)
#else
#define TTRACE(s, k) ((void)0)
#endif

namespace lr {

namespace {

using namespace tc;

constexpr int kTThreads = 256;
constexpr int kTM = 128;  // MMA M (rows of W per block, padded)

__device__ __forceinline__ int owner_of(int j, int Ur, int Uq, int Pk) {
  const int r = j / Ur;
  return r * Pk + (j - r * Ur) / Uq;
}

// shared memory layout (offsets in bytes from a 1024-aligned base)
struct TcLayout {
  uint32_t b_hi, b_lo;      // staged B tiles: n_atoms x (Nm x 128 bytes)
  uint32_t recv;            // [2][Pk][G*Uq][Nm] f32
  uint32_t outs;            // [G][N][Uq] f32 summed partials
  uint32_t hst, cst;        // [N][Uq] f32 state of the own units
  uint32_t gxs;             // [G][N][Uq] f32 next projection values
  uint32_t total;
};

__host__ __device__ inline TcLayout tc_layout(const RecPlan& pl, int G, int N, bool bf) {
  TcLayout L;
  const uint32_t atom = (uint32_t)pl.nbp * 128u;  // Nm rows x 128 bytes
  const uint32_t ntile = (uint32_t)pl.KC * atom;  // KC = K atoms per slice
  uint32_t off = 0;
  L.b_hi = off;
  off += ntile;
  L.b_lo = off;
  off += bf ? 0 : ntile;
  L.recv = off;
  off += 2u * pl.cluster * G * pl.Uq * pl.nbp * 4u;
  L.outs = off;
  off += (uint32_t)G * pl.Uq * N * 4u;
  L.hst = off;
  off += (uint32_t)pl.Uq * N * 4u;
  L.cst = off;
  off += (uint32_t)pl.Uq * N * 4u;
  L.gxs = off;
  off += (uint32_t)G * pl.Uq * N * 4u;
  L.total = (off + 1023u) & ~1023u;
  return L;
}

template <bool BF>
__global__ void __launch_bounds__(kTThreads, 1) rec_fwd_tc(const __grid_constant__ RecParams p) {
  typedef typename std::conditional<BF, bf16, float>::type T;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int s_fail;
  __shared__ float s_bhn[kTM];
  const RecPlan& pl = p.plan;
  const int P = pl.P, Pk = pl.cluster;
  const int d = blockIdx.x / P;
  const int b = blockIdx.x - d * P;
  const int r = b / Pk, q = b - r * Pk;
  const RecDirArgs& a = p.dir[d];
  const int H = p.H, N = p.N, nT = p.T, G = p.G, Ur = pl.Ur, Uq = pl.Uq;
  const int Nm = pl.nbp;                       // MMA N (columns of D)
  const int Kp = pl.K;                         // padded K slice (elements)
  const int u0 = r * Ur, Urc = min(Ur, H - u0);
  const int uq0 = q * Uq, Uqc = max(0, min(Uq, Urc - uq0));
  const int k0 = q * pl.Kk, Kc = max(0, min(pl.Kk, H - k0));
  const int Mb = G * Ur;                       // rows of the block's A (<= 128)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t GH = (int64_t)G * H;

  const uint32_t base_s = (smem_addr(smem_raw) + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_s - smem_addr(smem_raw));
  const TcLayout Lo = tc_layout(pl, G, N, BF);
  float* recv0 = reinterpret_cast<float*>(base + Lo.recv);
  float* outs = reinterpret_cast<float*>(base + Lo.outs);
  float* hst = reinterpret_cast<float*>(base + Lo.hst);
  float* cst = reinterpret_cast<float*>(base + Lo.cst);
  float* gxs = reinterpret_cast<float*>(base + Lo.gxs);
  const uint32_t atom_bytes = (uint32_t)Nm * 128u;
  const uint32_t bar = smem_addr(&mma_bar);
  // tensor memory: D at column 0 (Nm columns), A after it
  const uint32_t a_col = (uint32_t)Nm;
  const uint32_t a_lo_col = (uint32_t)(Nm + Kp);
  const uint32_t ncols = (uint32_t)pl.lda;     // allocated columns (power of two)

  // the launch formed the planned clusters, the tensor-memory columns hold D
  // and A, D's rows fit the MMA's M and N the staged tile: otherwise the block
  // touches neither tensor memory nor a peer's shared memory
  const bool cfg_bad = cl_size() != (unsigned)Pk || cl_rank() != (unsigned)q ||
                       (uint32_t)(Nm + (BF ? Kp / 2 : 2 * Kp)) > ncols || ncols > 512u ||
                       (ncols & (ncols - 1u)) != 0 || ncols < 32u || Mb > kTM || N > Nm ||
                       Nm % 16 != 0 || Nm > 256 || Kp % (BF ? 64 : 32) != 0 || pl.Kk > Kp;
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
  // zero the staged B tiles (rows >= N and columns >= Kc stay zero) and state
  for (uint32_t i = tid; i < (Lo.recv) / 16u; i += kTThreads)
    reinterpret_cast<uint4*>(base)[i] = make_uint4(0, 0, 0, 0);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_slot;

  // A (this block's W_hh slice) into tensor memory: lane m = row g*Ur + u,
  // column chunks of 32; warp w serves lanes 32*(w%4) .. +31
  if (!cfg_bad) {
    const T* W = reinterpret_cast<const T*>(a.whh);
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const int g = m / Ur, u = m - g * Ur;
    const bool row_ok = m < Mb && g < G && u < Urc;
    const T* wrow = row_ok ? W + (int64_t)(g * H + u0 + u) * H + k0 : W;
    const int epc = BF ? 64 : 32;              // elements per 32-column chunk
    const int nchunk = Kp / epc;
    for (int ci = warp >> 2; ci < nchunk; ci += kTThreads / 128) {
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (BF) {
          const int k = ci * 64 + 2 * i;
          float e0 = (row_ok && k < Kc) ? to_f(wrow[k]) : 0.f;
          float e1 = (row_ok && k + 1 < Kc) ? to_f(wrow[k + 1]) : 0.f;
          const uint32_t b0 = __float_as_uint(e0) >> 16, b1 = __float_as_uint(e1) >> 16;
          hi[i] = b0 | (b1 << 16);
          lo[i] = 0;
        } else {
          const int k = ci * 32 + i;
          const float v = (row_ok && k < Kc) ? to_f(wrow[k]) : 0.f;
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

  // state of the own units (rows uq0 .. uq0+Uqc-1 of the row group)
  const int items = Uqc * N;
  for (int it = tid; it < items; it += kTThreads) {
    const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
    const int64_t o = (int64_t)n * H + j;
    const float hv = a.h0 ? to_f(reinterpret_cast<const T*>(a.h0)[o]) : 0.f;
    const float cv = a.c0 ? a.c0[o] : 0.f;
    hst[n * Uq + uu] = hv;
    cst[n * Uq + uu] = cv;
    const int slot0 = d ? nT : 0;
    if (a.hseq) reinterpret_cast<T*>(a.hseq)[(int64_t)slot0 * N * H + o] = from_f<T>(hv);
    if (a.cseq) a.cseq[(int64_t)slot0 * N * H + o] = cv;
  }
  for (int uu = tid; uu < Uqc; uu += kTThreads)
    s_bhn[uu] = p.mode == 2 ? to_f(reinterpret_cast<const T*>(a.bhh)[2 * H + u0 + uq0 + uu]) : 0.f;
  const int flo = Kc > 0 ? owner_of(k0, Ur, Uq, Pk) : 0;
  const int fhi = Kc > 0 ? owner_of(k0 + Kc - 1, Ur, Uq, Pk) : -1;
  unsigned* flags = p.flags + (size_t)d * P * p.flag_stride;
  T* y = reinterpret_cast<T*>(a.y);
  T* hseq = reinterpret_cast<T*>(a.hseq);
  const uint32_t idesc = (1u << 4) | ((BF ? 1u : 2u) << 7) | ((BF ? 1u : 2u) << 10) |
                         ((uint32_t)(Nm >> 3) << 17) | ((uint32_t)(kTM >> 4) << 24);
  const int kstep = BF ? 16 : 8;               // K per MMA
  const int nsteps = (Kc + kstep - 1) / kstep;
  fence_before();
  __syncthreads();
  fence_after();
  bool failed = s_fail != 0;
  uint32_t phase = 0;  // parity of the next completion of the MMA barrier

  for (int s = 0; s < nT; ++s) {
    const int t = d ? nT - 1 - s : s;
    const int tp = d ? t + 1 : t - 1;
    TTRACE(s, 0);
    // this step's input projection values of the own items (consumed after the
    // contraction, so their latency hides behind it)
    for (int it = tid; it < G * items; it += kTThreads) {
      const int g = it / items, rem = it - g * items;
      const int uu = rem % Uqc, n = rem / Uqc;
      cp_async4(gxs + (g * N + n) * Uq + uu,
                a.gx + ((int64_t)t * N + n) * GH + (int64_t)g * H + u0 + uq0 + uu);
    }
    cp_async_commit();
    if (!failed && s > 0 && Kc > 0 && warp == 0) {
      if (!warp_wait_flags(flags, p.flag_stride, flo, fhi, (unsigned)s, p.status, p.timeout_ns,
                           p.spin_ns) &&
          lane == 0)
        s_fail = 1;
    }
    __syncthreads();
    TTRACE(s, 1);
    failed = s_fail != 0;
    const T* src = s == 0 ? reinterpret_cast<const T*>(a.h0)
                          : y + (int64_t)tp * N * p.ldy + (int64_t)d * H;
    const int64_t ldsrc = s == 0 ? H : p.ldy;
    const bool have = !failed && src != nullptr && Kc > 0;
    // stage B = h_{t-1}[n][k0 .. k0+Kc) into the swizzled K-major tiles
    if (have) {
      constexpr int VE = 16 / (int)sizeof(T);
      const int nv = Kc / VE;
      for (int idx = tid; idx < N * nv; idx += kTThreads) {
        const int n = idx / nv, c16 = idx - n * nv;
        const uint4 v = ldcg16(src + k0 + (int64_t)n * ldsrc + c16 * VE);
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
    TTRACE(s, 6);
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
    // wait for the products (every thread: the phase of this step)
    bool mma_ok = true;
    if (have) {
      mma_ok = mbar_wait_bounded(bar, phase, p.status, p.timeout_ns);
      phase ^= 1u;
    }
    fence_after();
    TTRACE(s, 2);
    // push D's rows (partials over this block's K slice) to the owners
    float* recv = recv0 + (size_t)(s & 1) * Pk * G * Uq * Nm;
    if (!failed) {
      const int quarter = warp & 3;
      const int m = quarter * 32 + lane;
      const int g = m / Ur, u = m - g * Ur;
      const bool row_ok = m < Mb && g < G && u < Urc;
      const int owner = row_ok ? u / Uq : 0, uo = u - owner * Uq;
      for (int c0 = (warp >> 2) * 32; c0 < Nm; c0 += (kTThreads / 128) * 32) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0, v);
        if (!row_ok || owner >= Pk) continue;
        // 16-byte pieces (row starts are 64-byte aligned, Nm % 16 == 0); columns
        // N .. Nm-1 of D are zero (the staged rows beyond N are zero) and unread
        float* dst = recv + ((size_t)q * G * Uq + g * Uq + uo) * Nm + c0;
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
    if (!failed) {
      // batch index fastest: consecutive threads read consecutive partials
      for (int idx = tid; idx < G * items; idx += kTThreads) {
        const int n = idx % N, gu = idx / N;
        const int g = gu / Uqc, uu = gu - g * Uqc;
        float v = 0.f;
        for (int rank = 0; rank < Pk; ++rank)
          v += recv[((size_t)rank * G * Uq + g * Uq + uu) * Nm + n];
        outs[(g * N + n) * Uq + uu] = v;
      }
    }
    cp_async_wait_all();
    __syncthreads();
    TTRACE(s, 3);
    if (!failed) {
      for (int it = tid; it < items; it += kTThreads) {
        const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
        const int64_t row = (int64_t)t * N + n;
        const int slot = d ? t : t + 1;
        const float* gv = gxs + n * Uq + uu;    // gate g at gv[g * N * Uq]
        const float* ov = outs + n * Uq + uu;   // likewise
        float h;
        if (p.mode == 1) {
          const float ig = sigmoidf_(gv[0] + ov[0]);
          const float fg = sigmoidf_(gv[N * Uq] + ov[N * Uq]);
          const float gg = tanhf(gv[2 * N * Uq] + ov[2 * N * Uq]);
          const float og = sigmoidf_(gv[3 * N * Uq] + ov[3 * N * Uq]);
          const float c = fg * cst[n * Uq + uu] + ig * gg;
          h = og * tanhf(c);
          cst[n * Uq + uu] = c;
          if (a.gates) {
            float* gp = a.gates + row * 4 * H + j;
            gp[0] = ig; gp[H] = fg; gp[2 * H] = gg; gp[3 * H] = og;
          }
          if (a.cseq) a.cseq[((int64_t)slot * N + n) * H + j] = c;
        } else if (p.mode == 2) {
          const float ghn = ov[2 * N * Uq] + s_bhn[uu];
          const float rg = sigmoidf_(gv[0] + ov[0]);
          const float z = sigmoidf_(gv[N * Uq] + ov[N * Uq]);
          const float nv = tanhf(gv[2 * Uq * N] + rg * ghn);
          h = (1.f - z) * nv + z * hst[n * Uq + uu];
          if (a.gates) {
            float* gp = a.gates + row * 4 * H + j;
            gp[0] = rg; gp[H] = z; gp[2 * H] = nv; gp[3 * H] = ghn;
          }
        } else {
          h = tanhf(gv[0] + ov[0]);
          if (a.gates) a.gates[row * H + j] = h;
        }
        hst[n * Uq + uu] = h;
        y[row * p.ldy + (int64_t)d * H + j] = from_f<T>(h);
        if (hseq) hseq[((int64_t)slot * N + n) * H + j] = from_f<T>(h);
      }
    }
    __syncthreads();
    TTRACE(s, 4);
    if (!failed && tid == 0 && s + 1 < nT && !(blockIdx.x == p.fault_block && s == p.fault_step))
      publish_flag(flags + (size_t)b * p.flag_stride, (unsigned)(s + 1));
    TTRACE(s, 5);
  }
  cl_sync();  // no block leaves while a peer may still store into it
  if (!failed) {
    for (int it = tid; it < items; it += kTThreads) {
      const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
      const int64_t o = (int64_t)n * H + j;
      if (a.hy) reinterpret_cast<T*>(a.hy)[o] = from_f<T>(hst[n * Uq + uu]);
      if (a.cy) a.cy[o] = cst[n * Uq + uu];
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 0 && !cfg_bad)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols)
                 : "memory");
}

}  // namespace

bool rec_tc_plan(int mode, int bf16, int D, int H, int N, int num_sms, size_t smem_limit,
                 const int* max_clusters, RecPlan* out) {
  const int G = mode == 1 ? 4 : mode == 2 ? 3 : 1;
  const int e = bf16 ? 2 : 4;
  if ((H * e) % 16 != 0 || N < 1 || N > 256) return false;
  const int Nm = (N + 15) / 16 * 16;
  const int Ur_max = kTM / G;
  bool found = false;
  double best = 0;
  RecPlan bp;
  for (int Pk : {4, 2, 8}) {
    const int cap = max_clusters[Pk];
    const int Pr_max = std::min(cap / D, (num_sms / D) / Pk);
    if (Pr_max < 1) continue;
    int Ur = (H + Pr_max - 1) / Pr_max;
    if (Ur > Ur_max) continue;
    const int Pr = (H + Ur - 1) / Ur;
    const int Uq = (Ur + Pk - 1) / Pk;
    const int epc = bf16 ? 64 : 32;                       // elements per 32 TMEM columns
    const int Kk = (((H + Pk - 1) / Pk) + 7) / 8 * 8;     // 16-byte aligned slices
    const int Kp = (Kk + epc - 1) / epc * epc;
    const int acols = bf16 ? Kp / 2 : 2 * Kp;
    int cols = 32;
    while (cols < Nm + acols) cols *= 2;
    if (cols > 512) continue;
    RecPlan pl;
    pl.direct = 0;
    pl.cluster = Pk; pl.Pr = Pr; pl.P = Pr * Pk; pl.Ur = Ur; pl.Uq = Uq;
    pl.Kk = Kk;
    pl.K = Kp;                       // padded K slice
    pl.KC = Kp / (bf16 ? 64 : 32);   // K atoms of 128 bytes
    pl.nbp = Nm;                     // MMA N
    pl.lda = cols;                   // tensor memory columns
    pl.Mloc = G * Ur; pl.Mp = kTM; pl.nb = N;
    pl.tc = 1;
    const TcLayout L = tc_layout(pl, G, N, bf16 != 0);
    // at least 120 KB so that no two blocks share an SM: each block allocates
    // all the tensor-memory columns it needs and keeps them for the sequence
    pl.smem = std::max<size_t>(L.total + 1024, 120 * 1024);
    if (pl.smem > smem_limit) continue;
    if (D * pl.P > num_sms) continue;
    // fewer units per block: less pointwise and push work; then smaller K slices
    const double cost = (double)Uq * N * (G + 2) + (double)G * Ur * N / 8.0 + Kp * 2.0;
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
extern "C" int rnn_debug_ttrace_copy(void* host, size_t bytes) {
  if (bytes > sizeof(g_ttrace)) bytes = sizeof(g_ttrace);
  return (int)cudaMemcpyFromSymbol(host, g_ttrace, bytes);
}
extern "C" int rnn_debug_ttrace_clear() {
  static unsigned long long zeros[4][1024][8];
  return (int)cudaMemcpyToSymbol(g_ttrace, zeros, sizeof(zeros));
}
#endif

cudaError_t rec_tc_launch(const RecParams& p, cudaStream_t st) {
  const RecPlan& pl = p.plan;
  void* fn = p.bf16 ? (void*)rec_fwd_tc<true> : (void*)rec_fwd_tc<false>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.flags, 0, sizeof(unsigned) * (size_t)p.D * pl.P * p.flag_stride, st);
  if (e != cudaSuccess) return e;
  RecParams copy = p;
  void* args[] = {&copy};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.D * pl.P);
  cfg.blockDim = dim3(kTThreads);
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
