// Cluster path of the persistent recurrent kernels (small batches: N <= 20).
//
// The per-step contraction of one direction is split over a 2-D grid of
// blocks: clusters own row groups (hidden units) and the blocks of a cluster
// split the contraction length K.  Block (r, q) -- cluster r, rank q -- keeps
// the slice "rows of row group r x K slice q" of W_hh (forward: the G gate rows
// of the units; backward: W_hh transposed, units x gate rows) in shared memory
// for the whole sequence, so per step it only stages its K slice of the
// previous step's broadcast vector (h_{t-1} forward, dG_h backward) instead of
// the whole vector.  The cluster's partial sums meet through distributed shared
// memory: every block stores each row's partial straight into the shared
// memory of the block that owns that unit's pointwise step; after a cluster
// barrier each block sums the partials it received in rank order
// (deterministic), applies the fused gate math, stores, and publishes its step
// flag.
//
// Every wait is bounded.  The cluster barrier itself has no time limit, so a
// block that gives up on a step flag keeps executing every cluster barrier of
// the schedule (skipping the work) instead of leaving early; blocks of a
// cluster are scheduled together, so every cluster barrier completes.
#include <algorithm>

#include "common.cuh"
#include "rec.h"

#ifdef LAYER_RNN_TRACE
__device__ unsigned long long g_ctrace[4][1024][8];
#define CTRACE(s, k)                                                                          \
  do {                                                                                        \
    const int nb_ = gridDim.x;                                                                \
    const int b_ = blockIdx.x == 0 ? 0 : blockIdx.x == nb_ / 3 ? 1 : blockIdx.x == (2 * nb_) / 3 \
                 ? 2 : blockIdx.x == nb_ - 1 ? 3 : -1;                                       \
    if (b_ >= 0 && threadIdx.x == 0 && (s) < 1024) g_ctrace[b_][(s)][(k)] = lr::globaltimer_ns();   \
  } while (0)
#else
#define CTRACE(s, k) ((void)0)
#endif

namespace lr {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxTiles = 2;  // row tiles per warp
constexpr int kNB = 20;       // batch columns of every shape (RN * LN)

struct Shape { int RM, RN, LM, LN; };
constexpr Shape kCShapes[4] = {{3, 5, 8, 4}, {3, 5, 4, 4}, {3, 5, 2, 4}, {3, 5, 1, 4}};
constexpr int kNumCShapes = 4;

__device__ __forceinline__ unsigned cluster_size() {
  unsigned n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// store a float to the same shared-memory offset in block `rank` of this cluster
__device__ __forceinline__ void st_peer_f32(float* local_ptr, unsigned rank, float v) {
  const unsigned laddr = static_cast<unsigned>(__cvta_generic_to_shared(local_ptr));
  unsigned raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(laddr), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(raddr), "f"(v) : "memory");
}

struct CSmem {
  void* A; void* B; float* red; float* part; float* recv; float* outs;
};

template <typename T>
__device__ __forceinline__ CSmem carve_c(unsigned char* smem, const RecPlan& pl, int orows) {
  CSmem c;
  T* A = reinterpret_cast<T*>(smem);
  T* B = A + (size_t)pl.Mp * pl.lda;
  c.A = A;
  c.B = B;
  c.red = reinterpret_cast<float*>(B + (size_t)kNB * pl.ldbs);
  c.part = c.red + (pl.Wk > 1 ? (size_t)pl.Wk * pl.Mp * kNB : 0);
  // partials pushed by every rank of the cluster, by step parity:
  // recv[parity][sender][orows][kNB]
  c.recv = c.part + (size_t)pl.Mp * kNB;
  c.outs = c.recv + (size_t)2 * pl.cluster * orows * kNB;
  return c;
}

// flag index (within the direction) of the block whose pointwise step owns unit j
__device__ __forceinline__ int owner_flag(int j, int Ur, int Uq, int Pk) {
  const int r = j / Ur;
  return r * Pk + (j - r * Ur) / Uq;
}

// Stage B[n][k0 .. k0+Kc) (row stride ldsrc, n < N) into Bs[n][0 .. Kc), 16-byte
// cp.async by all threads; src == nullptr leaves zeros.
template <typename T>
__device__ __forceinline__ void stage_slice(T* Bs, int ldbs, const T* src, int64_t ldsrc, int N,
                                            int Kc) {
  constexpr int VE = 16 / (int)sizeof(T);
  const int nv = Kc / VE;
  if (N > kNB || Kc > ldbs) return;  // never, by construction (checked by the plan)
  for (int idx = threadIdx.x; idx < N * nv; idx += kThreads) {
    const int n = idx / nv, c = idx - n * nv;
    cp_async16(Bs + n * ldbs + c * VE, src + n * ldsrc + c * VE);
  }
  cp_async_commit();
  cp_async_wait_all();
}

// This warp's share of the block contraction: row tiles wm, wm + Wm, ... (at
// most kMaxTiles) over K vectors [vb, ve) of the staged slice; the result goes
// (after the reduction over the LK lanes) to dst[row * kNB + n].
template <typename T, int RM, int RN, int LM, int LN>
__device__ __forceinline__ void warp_contract_store(const T* As, int lda, const T* Bs, int ldbs,
                                                    int ntiles, int wm, int Wm, int vb, int ve,
                                                    bool active, float* dst) {
  constexpr int LK = 32 / (LM * LN);
  constexpr int VK = 16 / (int)sizeof(T);
  constexpr int TR = LM * RM;
  const int lane = threadIdx.x & 31;
  const int lm = lane % LM, ln = (lane / LM) % LN, kl = lane / (LM * LN);
  float acc[kMaxTiles][RM][RN];
#pragma unroll
  for (int ti = 0; ti < kMaxTiles; ++ti)
#pragma unroll
    for (int i = 0; i < RM; ++i)
#pragma unroll
      for (int j = 0; j < RN; ++j) acc[ti][i][j] = 0.f;
  if (active) {
    const T* b0 = Bs + ln * ldbs;
#pragma unroll 2
    for (int v = vb + kl; v < ve; v += LK) {
      uint4 bv[RN];
#pragma unroll
      for (int j = 0; j < RN; ++j) bv[j] = *reinterpret_cast<const uint4*>(b0 + (LN * j) * ldbs + v * VK);
#pragma unroll
      for (int ti = 0; ti < kMaxTiles; ++ti) {
        const int tile = wm + ti * Wm;
        if (tile < ntiles) {
          const T* a0 = As + (tile * TR + lm) * lda + v * VK;
          uint4 av[RM];
#pragma unroll
          for (int i = 0; i < RM; ++i) av[i] = *reinterpret_cast<const uint4*>(a0 + (LM * i) * lda);
#pragma unroll
          for (int e = 0; e < VK; ++e) {
            float af[RM], bf[RN];
#pragma unroll
            for (int i = 0; i < RM; ++i) af[i] = sizeof(T) == 4 ? lane_f32(av[i], e) : lane_bf16(av[i], e);
#pragma unroll
            for (int j = 0; j < RN; ++j) bf[j] = sizeof(T) == 4 ? lane_f32(bv[j], e) : lane_bf16(bv[j], e);
#pragma unroll
            for (int i = 0; i < RM; ++i)
#pragma unroll
              for (int j = 0; j < RN; ++j) acc[ti][i][j] = fmaf(af[i], bf[j], acc[ti][i][j]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int ti = 0; ti < kMaxTiles; ++ti)
#pragma unroll
    for (int off = LM * LN; off < 32; off <<= 1)
#pragma unroll
      for (int i = 0; i < RM; ++i)
#pragma unroll
        for (int j = 0; j < RN; ++j) acc[ti][i][j] += __shfl_xor_sync(0xffffffffu, acc[ti][i][j], off);
  if (kl == 0) {
#pragma unroll
    for (int ti = 0; ti < kMaxTiles; ++ti) {
      const int tile = wm + ti * Wm;
      if (tile < ntiles) {
#pragma unroll
        for (int i = 0; i < RM; ++i)
#pragma unroll
          for (int j = 0; j < RN; ++j)
            dst[(tile * TR + lm + LM * i) * kNB + ln + LN * j] = active ? acc[ti][i][j] : 0.f;
      }
    }
  }
}

// The block's contraction for one step (staged slice already in Bs) ending with
// the block's partial sums in `part` (rows x kNB); block-synchronising.
template <typename T, int RM, int RN, int LM, int LN>
__device__ __forceinline__ void block_contract(const CSmem& sm, const RecPlan& pl, int Kc,
                                               bool active, float* part) {
  constexpr int VK = 16 / (int)sizeof(T);
  constexpr int TR = LM * RM;
  const int warp = threadIdx.x >> 5;
  const int wm = warp % pl.Wm, wk = warp / pl.Wm;
  const int ntiles = pl.Mp / TR;
  const int nvk = Kc / VK;
  const int vb = wk * nvk / pl.Wk, ve = (wk + 1) * nvk / pl.Wk;
  float* dst = pl.Wk > 1 ? sm.red + (size_t)wk * pl.Mp * kNB : part;
  warp_contract_store<T, RM, RN, LM, LN>(reinterpret_cast<const T*>(sm.A), pl.lda,
                                         reinterpret_cast<const T*>(sm.B), pl.ldbs, ntiles, wm,
                                         pl.Wm, vb, ve, active && ve > vb, dst);
  __syncthreads();
  if (pl.Wk > 1) {
    for (int idx = threadIdx.x; idx < pl.Mp * kNB; idx += kThreads) {
      float s = 0.f;
      for (int w = 0; w < pl.Wk; ++w) s += sm.red[(size_t)w * pl.Mp * kNB + idx];
      part[idx] = s;
    }
  }
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
template <typename T, int RM, int RN, int LM, int LN>
__global__ void __launch_bounds__(kThreads, 1)
    rec_fwd_cluster(const __grid_constant__ RecParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_fail;
  const RecPlan& pl = p.plan;
  const int P = pl.P, Pk = pl.cluster;
  const int d = blockIdx.x / P;
  const int b = blockIdx.x - d * P;
  const int r = b / Pk, q = b - r * Pk;
  const RecDirArgs& a = p.dir[d];
  const int H = p.H, N = p.N, nT = p.T, G = p.G, Ur = pl.Ur, Uq = pl.Uq;
  const int u0 = r * Ur, Urc = min(Ur, H - u0);
  const int uq0 = q * Uq, Uqc = max(0, min(Uq, Urc - uq0));
  const int k0 = q * pl.Kk, Kc = max(0, min(pl.Kk, H - k0));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const CSmem sm = carve_c<T>(smem, pl, G * Uq);
  T* As = reinterpret_cast<T*>(sm.A);
  T* Bs = reinterpret_cast<T*>(sm.B);
  const int64_t GH = (int64_t)G * H;

  if (tid == 0) {
    s_fail = ld_volatile_int(p.status) != kDevOk;
    // the launch must have formed the planned clusters, with this block at rank
    // q: otherwise no peer shared memory is touched at all
    if (cluster_size() != (unsigned)Pk || cluster_rank() != (unsigned)q || Pk > 8) {
      atomicCAS(p.status, kDevOk, kDevCheck);
      s_fail = 1;
    }
  }
  // resident slice: row g*Ur + u, column kk <- W_hh[g*H + u0 + u][k0 + kk]
  const T* W = reinterpret_cast<const T*>(a.whh);
  for (int64_t idx = tid; idx < (int64_t)pl.Mp * pl.lda; idx += kThreads) {
    const int m = (int)(idx / pl.lda), kk = (int)(idx - (int64_t)m * pl.lda);
    const int g = m / Ur, u = m - g * Ur;
    As[idx] = (g < G && u < Urc && kk < Kc) ? W[(int64_t)(g * H + u0 + u) * H + k0 + kk]
                                            : from_f<T>(0.f);
  }
  for (int idx = tid; idx < kNB * pl.ldbs; idx += kThreads) Bs[idx] = from_f<T>(0.f);

  // this thread's pointwise item: unit u0 + uq0 + uu, sequence n
  const bool item = tid < Uqc * N;
  const int uu = item ? tid % Uqc : 0, n = item ? tid / Uqc : 0, j = u0 + uq0 + uu;
  float h_own = 0.f, c_own = 0.f, bhn = 0.f;
  float gxv[4] = {0.f, 0.f, 0.f, 0.f};
  if (item) {
    const int64_t o = (int64_t)n * H + j;
    if (a.h0) h_own = to_f(reinterpret_cast<const T*>(a.h0)[o]);
    if (a.c0) c_own = a.c0[o];
    const int slot0 = d ? nT : 0;
    if (a.hseq) reinterpret_cast<T*>(a.hseq)[(int64_t)slot0 * N * H + o] = from_f<T>(h_own);
    if (a.cseq) a.cseq[(int64_t)slot0 * N * H + o] = c_own;
    if (p.mode == 2) bhn = to_f(reinterpret_cast<const T*>(a.bhh)[2 * H + j]);
    const float* gp = a.gx + ((int64_t)(d ? nT - 1 : 0) * N + n) * GH + j;
#pragma unroll
    for (int g = 0; g < 4; ++g)
      if (g < G) gxv[g] = __ldg(gp + g * H);
  }
  // producers of this block's K slice (units k0 .. k0+Kc-1)
  const int flo = Kc > 0 ? owner_flag(k0, Ur, Uq, Pk) : 0;
  const int fhi = Kc > 0 ? owner_flag(k0 + Kc - 1, Ur, Uq, Pk) : -1;
  unsigned* flags = p.flags + (size_t)d * P * p.flag_stride;
  T* y = reinterpret_cast<T*>(a.y);
  T* hseq = reinterpret_cast<T*>(a.hseq);
  __syncthreads();
  bool failed = s_fail != 0;

  for (int s = 0; s < nT; ++s) {
    const int t = d ? nT - 1 - s : s;
    const int tp = d ? t + 1 : t - 1;
    float* part = sm.part;
    CTRACE(s, 0);
    if (!failed && s > 0 && Kc > 0 && warp == 0) {
      if (!warp_wait_flags(flags, p.flag_stride, flo, fhi, (unsigned)s, p.status, p.timeout_ns,
                           p.spin_ns) &&
          lane == 0)
        s_fail = 1;
    }
    __syncthreads();
    CTRACE(s, 1);
    failed = s_fail != 0;
    const T* src = s == 0 ? reinterpret_cast<const T*>(a.h0)
                          : y + (int64_t)tp * N * p.ldy + (int64_t)d * H;
    const int64_t ldsrc = s == 0 ? H : p.ldy;
    const bool have = !failed && src != nullptr && Kc > 0;
    if (have) stage_slice<T>(Bs, pl.ldbs, src + k0, ldsrc, N, Kc);
    __syncthreads();
    CTRACE(s, 6);
    block_contract<T, RM, RN, LM, LN>(sm, pl, Kc, have, part);
    __syncthreads();
    CTRACE(s, 2);
    // push each row's partial to the rank that owns the unit's pointwise step
    float* recv = sm.recv + (size_t)(s & 1) * Pk * G * Uq * kNB;
    if (!failed) {
      for (int idx = tid; idx < G * Urc * N; idx += kThreads) {
        const int g = idx / (Urc * N), rem = idx - g * (Urc * N);
        const int u = rem / N, nn = rem - u * N;
        const int owner = u / Uq, uo = u - owner * Uq;
        if (owner >= Pk || nn >= kNB || g * Ur + u >= pl.Mp) {  // never, by construction
          atomicCAS(p.status, kDevOk, kDevCheck);
          continue;
        }
        st_peer_f32(recv + ((size_t)q * G * Uq + g * Uq + uo) * kNB + nn, (unsigned)owner,
                    part[(g * Ur + u) * kNB + nn]);
      }
    }
    cluster_sync_all();
    float* outs = sm.outs;
    if (!failed) {
      for (int idx = tid; idx < G * Uqc * N; idx += kThreads) {
        const int g = idx / (Uqc * N), rem = idx - g * (Uqc * N);
        const int u = rem / N, nn = rem - u * N;
        outs[(g * Uq + u) * kNB + nn] =
            sum_strided<8>(recv + ((size_t)g * Uq + u) * kNB + nn, (size_t)G * Uq * kNB, Pk);
      }
    }
    __syncthreads();
    CTRACE(s, 3);
    if (!failed && item) {
      const int64_t row = (int64_t)t * N + n;
      const int slot = d ? t : t + 1;
      float h;
      if (p.mode == 1) {  // LSTM, gate blocks i, f, g, o
        const float ig = sigmoidf_(gxv[0] + outs[(0 * Uq + uu) * kNB + n]);
        const float fg = sigmoidf_(gxv[1] + outs[(1 * Uq + uu) * kNB + n]);
        const float gg = tanhf(gxv[2] + outs[(2 * Uq + uu) * kNB + n]);
        const float og = sigmoidf_(gxv[3] + outs[(3 * Uq + uu) * kNB + n]);
        c_own = fg * c_own + ig * gg;
        h = og * tanhf(c_own);
        if (a.gates) {
          float* gp = a.gates + row * 4 * H + j;
          gp[0] = ig; gp[H] = fg; gp[2 * H] = gg; gp[3 * H] = og;
        }
        if (a.cseq) a.cseq[((int64_t)slot * N + n) * H + j] = c_own;
      } else if (p.mode == 2) {  // GRU, gate blocks r, z, n
        const float ghn = outs[(2 * Uq + uu) * kNB + n] + bhn;
        const float rg = sigmoidf_(gxv[0] + outs[(0 * Uq + uu) * kNB + n]);
        const float z = sigmoidf_(gxv[1] + outs[(1 * Uq + uu) * kNB + n]);
        const float nv = tanhf(gxv[2] + rg * ghn);
        h = (1.f - z) * nv + z * h_own;
        if (a.gates) {
          float* gp = a.gates + row * 4 * H + j;
          gp[0] = rg; gp[H] = z; gp[2 * H] = nv; gp[3 * H] = ghn;
        }
      } else {  // tanh RNN
        h = tanhf(gxv[0] + outs[uu * kNB + n]);
        if (a.gates) a.gates[row * H + j] = h;
      }
      h_own = h;
      y[row * p.ldy + (int64_t)d * H + j] = from_f<T>(h);
      if (hseq) hseq[((int64_t)slot * N + n) * H + j] = from_f<T>(h);
      if (s + 1 < nT) {
        const int tn = d ? t - 1 : t + 1;
        const float* gp = a.gx + ((int64_t)tn * N + n) * GH + j;
#pragma unroll
        for (int g = 0; g < 4; ++g)
          if (g < G) gxv[g] = __ldg(gp + g * H);
      }
    }
    __syncthreads();
    CTRACE(s, 4);
    if (!failed && tid == 0 && s + 1 < nT && !(blockIdx.x == p.fault_block && s == p.fault_step))
      publish_flag(flags + (size_t)b * p.flag_stride, (unsigned)(s + 1));
    CTRACE(s, 5);
  }
  cluster_sync_all();  // no block leaves while a peer may still store into it
  if (!failed && item) {
    const int64_t o = (int64_t)n * H + j;
    if (a.hy) reinterpret_cast<T*>(a.hy)[o] = from_f<T>(h_own);
    if (a.cy) a.cy[o] = c_own;
  }
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------
template <typename T, int RM, int RN, int LM, int LN>
__global__ void __launch_bounds__(kThreads, 1)
    rec_bwd_cluster(const __grid_constant__ RecParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_fail;
  const RecPlan& pl = p.plan;
  const int P = pl.P, Pk = pl.cluster;
  const int d = blockIdx.x / P;
  const int b = blockIdx.x - d * P;
  const int r = b / Pk, q = b - r * Pk;
  const RecDirArgs& a = p.dir[d];
  const int H = p.H, N = p.N, nT = p.T, G = p.G, Ur = pl.Ur, Uq = pl.Uq;
  const int64_t GH = (int64_t)G * H;
  const int u0 = r * Ur, Urc = min(Ur, H - u0);
  const int uq0 = q * Uq, Uqc = max(0, min(Uq, Urc - uq0));
  const int k0 = q * pl.Kk, Kc = (int)max((int64_t)0, min((int64_t)pl.Kk, GH - k0));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const CSmem sm = carve_c<T>(smem, pl, Uq);
  T* As = reinterpret_cast<T*>(sm.A);
  T* Bs = reinterpret_cast<T*>(sm.B);

  if (tid == 0) {
    s_fail = ld_volatile_int(p.status) != kDevOk;
    // the launch must have formed the planned clusters, with this block at rank
    // q: otherwise no peer shared memory is touched at all
    if (cluster_size() != (unsigned)Pk || cluster_rank() != (unsigned)q || Pk > 8) {
      atomicCAS(p.status, kDevOk, kDevCheck);
      s_fail = 1;
    }
  }
  // resident slice, transposed: A[u][kk] = W_hh[k0 + kk][u0 + u]; consecutive
  // threads read consecutive units of one row
  const T* W = reinterpret_cast<const T*>(a.whh);
  for (int64_t idx = tid; idx < (int64_t)pl.Mp * pl.lda; idx += kThreads) {
    const int kk = (int)(idx / pl.Mp), u = (int)(idx - (int64_t)kk * pl.Mp);
    As[(int64_t)u * pl.lda + kk] = (u < Urc && kk < Kc) ? W[(int64_t)(k0 + kk) * H + u0 + u]
                                                        : from_f<T>(0.f);
  }
  for (int idx = tid; idx < kNB * pl.ldbs; idx += kThreads) Bs[idx] = from_f<T>(0.f);

  const bool item = tid < Uqc * N;
  const int uu = item ? tid % Uqc : 0, n = item ? tid / Uqc : 0, j = u0 + uq0 + uu;
  float dc_own = 0.f, carry = 0.f;
  float dyv = 0.f, g0 = 0.f, g1 = 0.f, g2 = 0.f, g3 = 0.f, cc = 0.f, cpv = 0.f, hp = 0.f;
  const T* hseq = reinterpret_cast<const T*>(a.hseq);
  auto load_inputs = [&](int t) {
    const int64_t row = (int64_t)t * N + n;
    dyv = load_any(a.dy, row * p.lddy + (int64_t)d * H + j, a.dy_bf16);
    if (p.mode == 0) {
      g0 = __ldg(a.gates + row * H + j);
    } else {
      const float* gp = a.gates + row * 4 * H + j;
      g0 = __ldg(gp); g1 = __ldg(gp + H); g2 = __ldg(gp + 2 * H); g3 = __ldg(gp + 3 * H);
      const int sc = d ? t : t + 1, sp = d ? t + 1 : t;
      if (p.mode == 1) {
        cc = __ldg(a.cseq + ((int64_t)sc * N + n) * H + j);
        cpv = __ldg(a.cseq + ((int64_t)sp * N + n) * H + j);
      } else {
        hp = to_f(hseq[((int64_t)sp * N + n) * H + j]);
      }
    }
  };
  if (item) {
    if (a.dcy) dc_own = a.dcy[(int64_t)n * H + j];
    load_inputs(d ? 0 : nT - 1);
  }
  unsigned* flags = p.flags + (size_t)d * P * p.flag_stride;
  T* dgx = reinterpret_cast<T*>(a.dgx);
  T* dgh = reinterpret_cast<T*>(a.dgh);
  __syncthreads();
  bool failed = s_fail != 0;

  for (int s = 0; s <= nT; ++s) {
    const int t = d ? s : nT - 1 - s;    // time processed at this step (s < nT)
    const int tp = d ? s - 1 : nT - s;   // time processed at the previous step (s > 0)
    float* part = sm.part;
    CTRACE(s, 0);
    if (!failed && s > 0 && Kc > 0 && warp == 0) {
      bool ok = true;
      for (int g = 0; g < G && ok; ++g) {
        const int lo = max(k0, g * H), hi = min(k0 + Kc, (g + 1) * H);
        if (lo < hi)
          ok = warp_wait_flags(flags, p.flag_stride, owner_flag(lo - g * H, Ur, Uq, Pk),
                               owner_flag(hi - 1 - g * H, Ur, Uq, Pk), (unsigned)s, p.status,
                               p.timeout_ns, p.spin_ns);
      }
      if (!ok && lane == 0) s_fail = 1;
    }
    __syncthreads();
    CTRACE(s, 1);
    failed = s_fail != 0;
    const bool have = !failed && s > 0 && Kc > 0;
    if (have) stage_slice<T>(Bs, pl.ldbs, dgh + (int64_t)tp * N * GH + k0, GH, N, Kc);
    __syncthreads();
    CTRACE(s, 6);
    block_contract<T, RM, RN, LM, LN>(sm, pl, Kc, have, part);
    __syncthreads();
    CTRACE(s, 2);
    float* recv = sm.recv + (size_t)(s & 1) * Pk * Uq * kNB;
    if (!failed) {
      for (int idx = tid; idx < Urc * N; idx += kThreads) {
        const int u = idx / N, nn = idx - u * N;
        const int owner = u / Uq, uo = u - owner * Uq;
        if (owner >= Pk || nn >= kNB || u >= pl.Mp) {  // never, by construction
          atomicCAS(p.status, kDevOk, kDevCheck);
          continue;
        }
        st_peer_f32(recv + ((size_t)q * Uq + uo) * kNB + nn, (unsigned)owner, part[u * kNB + nn]);
      }
    }
    cluster_sync_all();
    float* outs = sm.outs;
    if (!failed) {
      for (int idx = tid; idx < Uqc * N; idx += kThreads) {
        const int u = idx / N, nn = idx - u * N;
        outs[u * kNB + nn] = sum_strided<8>(recv + (size_t)u * kNB + nn, (size_t)Uq * kNB, Pk);
      }
    }
    __syncthreads();
    CTRACE(s, 3);
    if (!failed && item) {
      float dhf;
      if (s == 0)
        dhf = a.dhy ? to_f(reinterpret_cast<const T*>(a.dhy)[(int64_t)n * H + j]) : 0.f;
      else
        dhf = outs[uu * kNB + n] + carry;
      if (s == nT) {
        if (a.dh0) reinterpret_cast<T*>(a.dh0)[(int64_t)n * H + j] = from_f<T>(dhf);
        if (a.dc0) a.dc0[(int64_t)n * H + j] = dc_own;
      } else {
        const int64_t row = (int64_t)t * N + n;
        const float dh = dyv + dhf;
        T* gxo = dgx + row * GH + j;
        if (p.mode == 1) {  // LSTM: g0..g3 = i, f, g, o; cc = c_t; cpv = c_{t-1}
          const float tc = tanhf(cc);
          const float dc = dc_own + dh * g3 * (1.f - tc * tc);
          gxo[0] = from_f<T>(dc * g2 * g0 * (1.f - g0));
          gxo[H] = from_f<T>(dc * cpv * g1 * (1.f - g1));
          gxo[2 * H] = from_f<T>(dc * g0 * (1.f - g2 * g2));
          gxo[3 * H] = from_f<T>(dh * tc * g3 * (1.f - g3));
          dc_own = dc * g1;
        } else if (p.mode == 2) {  // GRU: g0..g3 = r, z, n, W_hn h + b_hn; hp = h_{t-1}
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
          carry = dh * g1;
        } else {  // tanh RNN: g0 = h_t
          gxo[0] = from_f<T>(dh * (1.f - g0 * g0));
        }
        if (s + 1 < nT) load_inputs(d ? t + 1 : t - 1);
      }
    }
    __syncthreads();
    CTRACE(s, 4);
    if (!failed && tid == 0 && s < nT && !(blockIdx.x == p.fault_block && s == p.fault_step))
      publish_flag(flags + (size_t)b * p.flag_stride, (unsigned)(s + 1));
    CTRACE(s, 5);
  }
  cluster_sync_all();
}

template <typename T, int S>
void* cfwd() {
  return (void*)rec_fwd_cluster<T, kCShapes[S].RM, kCShapes[S].RN, kCShapes[S].LM, kCShapes[S].LN>;
}
template <typename T, int S>
void* cbwd() {
  return (void*)rec_bwd_cluster<T, kCShapes[S].RM, kCShapes[S].RN, kCShapes[S].LM, kCShapes[S].LN>;
}

void* pick_cluster_kernel(bool backward, int is_bf16, int shape) {
  static void* const table[2][2][kNumCShapes] = {
      {{cfwd<float, 0>(), cfwd<float, 1>(), cfwd<float, 2>(), cfwd<float, 3>()},
       {cfwd<bf16, 0>(), cfwd<bf16, 1>(), cfwd<bf16, 2>(), cfwd<bf16, 3>()}},
      {{cbwd<float, 0>(), cbwd<float, 1>(), cbwd<float, 2>(), cbwd<float, 3>()},
       {cbwd<bf16, 0>(), cbwd<bf16, 1>(), cbwd<bf16, 2>(), cbwd<bf16, 3>()}}};
  return table[backward ? 1 : 0][is_bf16 ? 1 : 0][shape];
}

int64_t rup(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

}  // namespace

int rec_cluster_capacity(int cluster, size_t smem) {
  void* fn = pick_cluster_kernel(false, 0, 0);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster * 64);
  cfg.blockDim = dim3(kThreads);
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

bool rec_cluster_plan(bool backward, int mode, int bf16, int D, int H, int N, int num_sms,
                      size_t smem_limit, const int* max_clusters, RecPlan* out) {
  const int G = mode == 1 ? 4 : mode == 2 ? 3 : 1;
  const int e = bf16 ? 2 : 4;
  const int VK = 16 / e;
  if (N > kNB || (H * e) % 16 != 0) return false;
  const int K = backward ? G * H : H;
  bool found = false;
  double best_cost = 0;
  RecPlan best;
  for (int Pk : {8, 4, 2}) {
    const int cap = max_clusters[Pk];
    const int Pr_max = std::min(cap / D, (num_sms / D) / Pk);
    if (Pr_max < 1) continue;
    const int Ur = (H + Pr_max - 1) / Pr_max;
    const int Pr = (H + Ur - 1) / Ur;
    const int Uq = (Ur + Pk - 1) / Pk;
    if (Uq * N > kThreads) continue;
    const int Kk = (int)rup((K + Pk - 1) / Pk, VK);
    const int Mb = backward ? Ur : G * Ur;
    for (int sh = 0; sh < kNumCShapes; ++sh) {
      const Shape S = kCShapes[sh];
      const int LK = 32 / (S.LM * S.LN);
      const int TR = S.LM * S.RM;
      const int ntiles = (Mb + TR - 1) / TR;
      for (int Wk : {1, 2, 4, 8, 16}) {
        const int Wm = kWarps / Wk;
        const int tpw = (ntiles + Wm - 1) / Wm;
        if (tpw > kMaxTiles) continue;
        const int nvk = Kk / VK;
        if (nvk < Wk * LK) continue;
        RecPlan pl;
        pl.cluster = Pk; pl.Pr = Pr; pl.P = Pr * Pk; pl.Ur = Ur; pl.Uq = Uq; pl.Kk = Kk;
        pl.Wm = Wm; pl.Wk = Wk; pl.shape = sh;
        pl.Mloc = Mb; pl.Mp = ntiles * TR; pl.K = K; pl.nb = N; pl.nbp = kNB;
        pl.tiles_m = tpw; pl.tiles_n = 1;
        const int pad = (16 * LK) / e;
        pl.lda = (int)(rup(Kk, 128 / e) + pad);
        pl.ldbs = (int)(rup(Kk, 128 / e) + pad);
        const int orows = backward ? Uq : G * Uq;
        pl.smem = (size_t)pl.Mp * pl.lda * e + (size_t)kNB * pl.ldbs * e +
                  (Wk > 1 ? (size_t)Wk * pl.Mp * kNB * 4 : 0) + (size_t)pl.Mp * kNB * 4 +
                  (size_t)2 * Pk * orows * kNB * 4 + (size_t)orows * kNB * 4 + 256;
        if (pl.smem > smem_limit) continue;
        if (D * pl.P > num_sms) continue;
        // rough cycle estimate per step: the contraction is bound by FMA issue
        // (4 warps per SM sub-partition) or by shared-memory wavefronts (one
        // 128-byte wavefront per clock per SM), then staging and reductions
        const double vec_per_warp = tpw * ((double)nvk / (Wk * LK));
        const int wf = S.RM * ((S.LM * LK * 16 + 127) / 128) + S.RN * ((S.LN * LK * 16 + 127) / 128);
        const double fma = std::max(4.0 * vec_per_warp * S.RM * S.RN * VK,
                                    (double)kWarps * vec_per_warp * wf) * 1.2;
        const double stage = (double)N * Kk * e / 64.0;
        const double lred = Wk > 1 ? (double)pl.Mp * kNB * Wk / kThreads * 8 + 60 : 0;
        const double cred = (double)Mb * N / kThreads * 10 + (double)Pk * orows * N / kThreads * 4 + 150;
        const double cost = fma + stage + lred + cred;
        if (!found || cost < best_cost) {
          found = true;
          best_cost = cost;
          best = pl;
        }
      }
    }
  }
  if (found) *out = best;
  return found;
}

cudaError_t rec_cluster_launch(bool backward, const RecParams& p, cudaStream_t st) {
  const RecPlan& pl = p.plan;
  void* fn = pick_cluster_kernel(backward, p.bf16, pl.shape);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.flags, 0, sizeof(unsigned) * (size_t)p.D * pl.P * p.flag_stride, st);
  if (e != cudaSuccess) return e;
  RecParams copy = p;
  void* args[] = {&copy};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.D * pl.P);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  // Not a cooperative launch: the plan keeps the grid within the measured
  // co-resident cluster capacity (one block per SM), and every step wait is
  // bounded, so a cluster that is not resident shows up as RNN_ERR_TIMEOUT.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  e = cudaLaunchKernelExC(&cfg, fn, args);
  return e;
}

}  // namespace lr

#ifdef LAYER_RNN_TRACE
// trace builds only: co-resident clusters of `cluster` blocks at `smem` bytes
extern "C" int rnn_debug_cluster_capacity(int cluster, long long smem) {
  return lr::rec_cluster_capacity(cluster, (size_t)smem);
}
extern "C" int rnn_debug_ctrace_copy(void* host, size_t bytes) {
  if (bytes > sizeof(g_ctrace)) bytes = sizeof(g_ctrace);
  return (int)cudaMemcpyFromSymbol(host, g_ctrace, bytes);
}
extern "C" int rnn_debug_ctrace_clear() {
  static unsigned long long zeros[4][1024][8];
  return (int)cudaMemcpyToSymbol(g_ctrace, zeros, sizeof(zeros));
}
#endif
