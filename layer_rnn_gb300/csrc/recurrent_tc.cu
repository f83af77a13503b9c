// Tensor-core path of the persistent recurrent forward kernel.
//
// Same 2-D decomposition as the cluster path (clusters own row groups of
// hidden units, the blocks of a cluster split the contraction length K), but
// each block's per-step product
//     D[m][n] = sum_k W_hh[row m][k0 + k] * h_{t-1}[n][k0 + k]      (m < 128)
// runs on the tensor cores with W_hh's slice resident in tensor memory for the
// whole sequence.
//
// fp32 operands are split into fp16 pairs, x = (hi + lo * 2^-11) / scale, with
// hi = fp16(x * scale), lo = fp16((x * scale - hi) * 2^11) and a power-of-two
// scale per block and operand (W: its slice's largest magnitude maps just
// below 2^14; h: every |h_t| is at most max(1, max |h0|) -- LSTM and tanh
// outputs lie in (-1, 1), a GRU state is a convex mix of its candidate and the
// previous state -- so one scale from h0's slice holds for the whole
// sequence).  The product keeps hi*hi + hi*lo + lo*hi, three MMA passes of 16
// K each: about 22 significant bits per operand, as three tf32 passes on
// tf32 hi / lo splits, in half the MMA instructions (an MMA's issue, not the
// tensor pipe, bounds these small N = batch products).  bf16 runs one pass.
//
// Step pipeline (one step = one time step of one direction):
//   1. staging, K atoms (128 bytes of every batch row) spread over the warps:
//      a warp waits only for the step flags of the blocks that produced its
//      atom's hidden units, loads its rows of the atom of h_{t-1} from L2,
//      splits them (fp32) and stores them in the 128-byte-swizzled K-major
//      layout the MMA reads as B;
//   2. MMA issue after one block barrier: fp32 has one issuing thread per
//      pass, each with its own accumulator in tensor memory, so the three
//      passes issue in parallel;
//   3. the accumulators' rows are combined in a fixed order and pushed over
//      distributed shared memory to the block that owns each unit's pointwise
//      step, as asynchronous stores that complete the transaction count of
//      the owner's receive barrier (one per buffer of the double-buffered
//      partials): an owner waits only for its own inputs, and no block waits
//      for a cluster barrier whose release would also drain its earlier
//      global stores;
//   4. the owner sums the partials in rank order (deterministic), runs the
//      fused gate math, and writes the exchange word of each h first (value
//      and step in one 8-byte word: the data is its own flag, the other
//      blocks poll it), then y and the workspace (gates, c, h sequence).
// The step's input projection values are fetched with cp.async once the K
// slice is staged, while the MMAs and the exchange run (the pages' ping-pong
// prefetch).  All waits are bounded.
#include <algorithm>
#include <cstdio>
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
// per-warp stamps of the step pipeline: [block][step][0..15 atom staged,
// 16..18 issuer i done]
__device__ unsigned long long g_wtrace[4][1024][32];
#define WTRACE(s, k)                                                                          \
  do {                                                                                        \
    const int nb_ = gridDim.x;                                                                \
    const int b_ = blockIdx.x == 0 ? 0 : blockIdx.x == nb_ / 3 ? 1 : blockIdx.x == (2 * nb_) / 3 \
                 ? 2 : blockIdx.x == nb_ - 1 ? 3 : -1;                                       \
    if (b_ >= 0 && (threadIdx.x & 31) == 0 && (s) < 1024) g_wtrace[b_][(s)][(k)] = lr::globaltimer_ns();\
  } while (0)
// per block and step: [0] thread 0's exchange-word store issued, [1] staging
// done (after the block barrier)
__device__ unsigned long long g_xtrace[256][512][2];
#define XTRACE(s, k)                                                                          \
  do {                                                                                        \
    if (threadIdx.x == 0 && blockIdx.x < 256 && (s) < 512)                                    \
      g_xtrace[blockIdx.x][(s)][(k)] = lr::globaltimer_ns();                                  \
  } while (0)
// a stamp of warp 0 taken only once v is computed (the shared store waits for v)
#define PTRACE(s, k, v)                                                                       \
  do {                                                                                        \
    if (warp == 0) {                                                                          \
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(smem_addr(&s_tsink)), "f"(v) : "memory");  \
      WTRACE(s, k);                                                                           \
    }                                                                                         \
  } while (0)
#else
#define TTRACE(s, k) ((void)0)
#define WTRACE(s, k) ((void)0)
#define PTRACE(s, k, v) ((void)0)
#define XTRACE(s, k) ((void)0)
#endif

namespace lr {

namespace {

using namespace tc;

constexpr int kTThreads = 256;
constexpr int kTWarps = kTThreads / 32;
constexpr int kTM = 128;        // MMA M (rows of W per block, padded)
constexpr int kMaxAtoms = 16;   // K atoms (128 bytes of K per row) of a block's slice
constexpr int kPollRows4 = 8;   // rows of 4 words a lane of the forward polls at once
constexpr int kMaxPushers = 8;  // largest cluster of the plan

// shared memory layout (offsets in bytes from a 1024-aligned base)
struct TcLayout {
  uint32_t b_hi, b_lo;      // staged B tiles: KC atoms x (Nm rows x 128 bytes)
  uint32_t recv;            // [2][Pk][G*Uq][Nm] f32 partial sums pushed by the cluster
  uint32_t hst, cst;        // [N][Uq] f32 state of the own units
  uint32_t gxs;             // [G][N][Uq] f32 this step's projection values
  uint32_t outs;            // [6][N][Uq] f32 the previous step's h, gates, c (stored late)
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
  off += 2u * pl.cluster * G * pl.Uq * (pl.nbp + 4) * 4u;
  L.hst = off;
  off += (uint32_t)pl.Uq * N * 4u;
  L.cst = off;
  off += (uint32_t)pl.Uq * N * 4u;
  L.gxs = off;
  off += (uint32_t)G * pl.Uq * N * 4u;
  L.outs = off;
  off += 6u * pl.Uq * N * 4u;
  L.total = (off + 1023u) & ~1023u;
  return L;
}

template <bool BF, bool VL>  // VL: per-sequence lengths (p.lengths) are read
__global__ void __launch_bounds__(kTThreads, 1) rec_fwd_tc(const __grid_constant__ RecParams p) {
  typedef typename std::conditional<BF, bf16, float>::type T;
  constexpr int NI = BF ? 1 : 3;   // issuing threads = accumulators (one per pass)
  constexpr int EPA = 64;            // K elements (16-bit) per 128-byte atom
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ __align__(8) uint64_t recv_bar[2];  // partial sums of steps s (s & 1) landed
  __shared__ uint32_t tmem_slot;
  __shared__ int s_fail, s_mma_bad;
  __shared__ float s_bhn[kTM];
  __shared__ float s_red[kTThreads / 32][2];
#ifdef LAYER_RNN_TRACE
  __shared__ float s_tsink;
#endif
  const RecPlan& pl = p.plan;
  const int P = pl.P, Pk = pl.cluster;
  const int d = blockIdx.x / P;
  const int b = blockIdx.x - d * P;
  const int r = b / Pk, q = b - r * Pk;
  const RecDirArgs& a = p.dir[d];
  const int rv = a.rev >= 0 ? a.rev : d;       // reversed time order
  const int H = p.H, N = p.N, nT = p.T, G = p.G, Ur = pl.Ur, Uq = pl.Uq;
  const int Nm = pl.nbp;                       // MMA N (columns of D)
  const int Kp = pl.K;                         // padded K slice (elements)
  const int u0 = r * Ur, Urc = min(Ur, H - u0);
  const int uq0 = q * Uq, Uqc = max(0, min(Uq, Urc - uq0));
  const int k0 = q * pl.Kk, Kc = max(0, min(pl.Kk, H - k0));
  const int KCu = (Kc + EPA - 1) / EPA;        // atoms this block stages and multiplies
  const int Mb = G * Ur;                       // rows of the block's A (<= 128)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t GH = (int64_t)G * H;

#ifdef LAYER_RNN_TRACE
  if (blockIdx.x == 0 && threadIdx.x == 0)
    printf("%s plan: P %d cluster %d Ur %d Uq %d Kk %d K %d KC %d Nm %d cols %d\n", "fwd", pl.P,
           pl.cluster, pl.Ur, pl.Uq, pl.Kk, pl.K, pl.KC, pl.nbp, pl.lda);
#endif
  const uint32_t base_s = (smem_addr(smem_raw) + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_s - smem_addr(smem_raw));
  const TcLayout Lo = tc_layout(pl, G, N, BF);
  float* recv0 = reinterpret_cast<float*>(base + Lo.recv);
  float* hst = reinterpret_cast<float*>(base + Lo.hst);
  float* cst = reinterpret_cast<float*>(base + Lo.cst);
  float* gxs = reinterpret_cast<float*>(base + Lo.gxs);
  float* outs = reinterpret_cast<float*>(base + Lo.outs);
  const uint32_t atom_bytes = (uint32_t)Nm * 128u;
  const uint32_t mbar = smem_addr(&mma_bar);
  const uint32_t rbar0 = smem_addr(&recv_bar[0]);
  // tensor memory: accumulator i at column i * Nm, then the A operands, two
  // 16-bit elements per column: W (bf16) or W_hi and W_lo (fp32 split)
  const uint32_t a_col = (uint32_t)(NI * Nm);
  const uint32_t a_lo_col = a_col + (uint32_t)(Kp / 2);
  const uint32_t ncols = (uint32_t)pl.lda;     // allocated columns (power of two)

  // the launch formed the planned clusters, the tensor-memory columns hold the
  // accumulators and A, D's rows fit the MMA's M and N the staged tile:
  // otherwise the block touches neither tensor memory nor a peer's memory
  const bool cfg_bad = cl_size() != (unsigned)Pk || cl_rank() != (unsigned)q ||
                       a_col + (uint32_t)(BF ? Kp / 2 : Kp) > ncols || ncols > 512u ||
                       (ncols & (ncols - 1u)) != 0 || ncols < 32u || Mb > kTM || N > Nm ||
                       Nm % 16 != 0 || Nm > 256 || Kp % EPA != 0 || pl.KC * EPA != Kp ||
                       pl.KC > kMaxAtoms || pl.Kk > Kp || Pk > kMaxPushers || a.hx == nullptr ||
                       (H & 3) != 0 || (pl.Kk & 3) != 0;
  if (tid == 0) {
    s_fail = ld_volatile_int(p.status) != kDevOk || cfg_bad;
    s_mma_bad = 0;
    if (cfg_bad) atomicCAS(p.status, kDevOk, kDevCheck);
    mbar_init(mbar, NI);
    mbar_init(rbar0, 1);
    mbar_init(rbar0 + 8u, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && !cfg_bad) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // zero the staged B tiles and the W_lo tile (rows >= N / >= Mb and columns
  // >= Kc stay zero)
  for (uint32_t i = tid; i < Lo.recv / 16u; i += kTThreads)
    reinterpret_cast<uint4*>(base)[i] = make_uint4(0, 0, 0, 0);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_slot;

  // the split's scales (fp32): largest |W| of the slice and largest |h0| of
  // the staged K slice, each mapped just below 2^14 by a power of two
  float w_scale = 1.f, h_scale = 1.f, out_scale = 1.f;
  if (!BF) {
    const T* W = reinterpret_cast<const T*>(a.whh);
    float wm = 0.f, hm = 1.f;
    if (!cfg_bad) {
      for (int idx = tid; idx < Mb * Kc; idx += kTThreads) {
        const int m = idx / Kc, k = idx - m * Kc;
        const int g = m / Ur, u = m - g * Ur;
        if (g < G && u < Urc) wm = fmaxf(wm, fabsf(to_f(W[(int64_t)(g * H + u0 + u) * H + k0 + k])));
      }
      if (a.h0)
        for (int idx = tid; idx < N * Kc; idx += kTThreads) {
          const int n = idx / Kc, k = idx - n * Kc;
          hm = fmaxf(hm, fabsf(to_f(reinterpret_cast<const T*>(a.h0)[(int64_t)n * H + k0 + k])));
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
      wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
      hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, o));
    }
    if (lane == 0) {
      s_red[warp][0] = wm;
      s_red[warp][1] = hm;
    }
    __syncthreads();
    wm = 0.f;
    hm = 1.f;
    for (int w = 0; w < kTThreads / 32; ++w) {
      wm = fmaxf(wm, s_red[w][0]);
      hm = fmaxf(hm, s_red[w][1]);
    }
    int ew = 0, eh = 0;
    if (wm > 0.f) (void)frexpf(wm, &ew);  // wm < 2^ew
    (void)frexpf(hm, &eh);
    ew = min(max(14 - ew, -100), 100);
    eh = min(max(14 - eh, -100), 100);
    w_scale = ldexpf(1.f, ew);
    h_scale = ldexpf(1.f, eh);
    out_scale = ldexpf(1.f, -(ew + eh));
  }

  // A (this block's W_hh slice) into tensor memory: lane / row m = g*Ur + u,
  // 32-column chunks of 64 K elements (two 16-bit elements per column); warp w
  // serves lanes 32*(w%4) .. +31.  fp32: W_hi at a_col, W_lo at a_lo_col.
  if (!cfg_bad) {
    const T* W = reinterpret_cast<const T*>(a.whh);
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const int g = m / Ur, u = m - g * Ur;
    const bool row_ok = m < Mb && g < G && u < Urc;
    const T* wrow = row_ok ? W + (int64_t)(g * H + u0 + u) * H + k0 : W;
    const int nchunk = pl.KC;                  // one 32-column chunk per atom
    for (int ci = warp >> 2; ci < nchunk; ci += kTThreads / 128) {
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int k = ci * 64 + 2 * i;
        const float e0 = (row_ok && k < Kc) ? to_f(wrow[k]) : 0.f;
        const float e1 = (row_ok && k + 1 < Kc) ? to_f(wrow[k + 1]) : 0.f;
        if (BF) {
          hi[i] = (__float_as_uint(e0) >> 16) | ((__float_as_uint(e1) >> 16) << 16);
          lo[i] = 0;
        } else {
          split_f16x2(e0 * w_scale, e1 * w_scale, hi[i], lo[i]);
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
    const int slot0 = rv ? nT : 0;
    if (a.hseq) reinterpret_cast<T*>(a.hseq)[(int64_t)slot0 * N * H + o] = from_f<T>(hv);
    if (a.cseq) a.cseq[(int64_t)slot0 * N * H + o] = cv;
  }
  for (int uu = tid; uu < Uqc; uu += kTThreads)
    s_bhn[uu] = p.mode == 2 ? to_f(reinterpret_cast<const T*>(a.bhh)[2 * H + u0 + uq0 + uu]) : 0.f;
  T* y = reinterpret_cast<T*>(a.y);
  T* hseq = reinterpret_cast<T*>(a.hseq);
  // kind::f16 with bf16 (1) or fp16 (0) operands, fp32 accumulate
  const uint32_t idesc = (1u << 4) | ((BF ? 1u : 0u) << 7) | ((BF ? 1u : 0u) << 10) |
                         ((uint32_t)(Nm >> 3) << 17) | ((uint32_t)(kTM >> 4) << 24);
  // bytes of partial sums pushed to this block per step: G rows per own unit,
  // N columns in 16-byte pieces, from each block of the cluster (this one
  // included) whose K slice is not empty.  A block with an empty slice pushes
  // nothing: it polls nothing either, so it runs ahead of the exchange, and
  // its zeros could land in a later step's phase.  Every pusher polls its
  // slice each step, which keeps it within one step of the blocks that read
  // its owners' units: its step-s pushes land only after every owner of its
  // cluster consumed the partials of step s - 2, the other buffer's use.
  const int pushers = min(Pk, (H + max(1, pl.Kk) - 1) / max(1, pl.Kk));
  const uint32_t rx_bytes = (uint32_t)(pushers * G * Uqc * ((N + 3) / 4) * 16);
  // every block's barriers are initialised before any peer pushes into them
  fence_before();
  cl_sync();
  fence_after();
  uint32_t mma_phase = 0;  // parity of the next completion of the MMA barrier
  // step-invariant index work, once: this thread's accumulator row (the
  // epilogue) and its first pointwise item
  int e_g, e_uo, e_owner;
  bool e_row_ok;
  {
    const int m = (warp & 3) * 32 + lane;
    e_g = m / Ur;
    const int u = m - e_g * Ur;
    e_row_ok = m < Mb && e_g < G && u < Urc;
    e_owner = e_row_ok ? u / Uq : 0;
    e_uo = u - e_owner * Uq;
  }
  const int i_uu = Uqc > 0 ? tid % Uqc : 0, i_n = Uqc > 0 ? tid / Uqc : 0;
  // the valid length of this thread's first item's sequence (read once, off
  // the steps' critical path); other items read theirs when they run
  const int i_len = (VL && tid < items) ? __ldg(p.lengths + i_n) : 0x7fffffff;
  auto seq_len = [&](int it, int n) {
    if constexpr (!VL) return 0x7fffffff;
    else return it == tid ? i_len : __ldg(p.lengths + n);
  };
  const int icap = Uq * N;  // stride of one array of the output stash
  // the outputs of step sp (y, the saved gates, c_t, the h sequence) from the
  // stash, each item by the thread that computed it: written one step late,
  // after the next step's polls and MMA issue, so that these stores do not
  // queue ahead of the poll loads
  auto flush = [&](int sp) {
    const int tq = rv ? nT - 1 - sp : sp;
    const int slot = rv ? tq : tq + 1;
    for (int it = tid; it < items; it += kTThreads) {
      const int uu = it == tid ? i_uu : it % Uqc, n = it == tid ? i_n : it / Uqc;
      const int j = u0 + uq0 + uu;
      const int64_t row = (int64_t)tq * N + n;
      const float h = outs[it];
      const T hs = from_f<T>(h);
      // past the sequence's length the output is zero (the state is kept)
      const bool act = !VL || tq < seq_len(it, n);
      y[row * p.ldy + (int64_t)d * H + j] = act ? hs : from_f<T>(0.f);
      if (a.gates) {
        if (p.mode == 0) {
          a.gates[row * H + j] = h;
        } else {
          float* gp = a.gates + row * 4 * H + j;
          gp[0] = outs[icap + it];
          gp[H] = outs[2 * icap + it];
          gp[2 * H] = outs[3 * icap + it];
          gp[3 * H] = outs[4 * icap + it];
        }
      }
      if (a.cseq) a.cseq[((int64_t)slot * N + n) * H + j] = outs[5 * icap + it];
      if (hseq) hseq[((int64_t)slot * N + n) * H + j] = hs;
    }
  };
  int pend = -1;  // the step whose outputs wait in the stash

  for (int s = 0; s < nT; ++s) {
    const int t = rv ? nT - 1 - s : s;
    const int tp = rv ? t + 1 : t - 1;
    const bool failed = s_fail != 0;  // read after the previous step's barrier
    const uint32_t rbar = rbar0 + 8u * (uint32_t)(s & 1);
    TTRACE(s, 0);
    // this step's partial sums: one arrival plus the bytes the peers push (a
    // peer's bytes may land first; the phase cannot complete before this)
    if (!failed && tid == 0) mbar_arrive_expect_tx(rbar, rx_bytes);
    const bool have = !failed && Kc > 0;
    const T* src = s == 0 ? reinterpret_cast<const T*>(a.h0)
                          : y + (int64_t)tp * N * p.ldy + (int64_t)d * H;
    const int64_t ldsrc = s == 0 ? H : p.ldy;
    // 1. staging: task (atom, row part) -> warp.  Step 0 stages h0 from
    // memory; later steps poll the tagged exchange words of h_{t-1} written by
    // the producers of the atom's units (value and step in one 8-byte word, so
    // the data is its own flag: no release fence on the writer's side, no
    // second round trip on the reader's) and stage them as B (fp16 hi / lo
    // for fp32).
    const int parts = max(1, kTWarps / max(1, KCu));
    if (have) {
      const unsigned long long* hxp = a.hx + (size_t)((s + 2) % 3) * N * H + k0;
      for (int task = warp; task < KCu * parts; task += kTWarps) {
        const int at = task % KCu, part = task / KCu;
        const int ka = at * EPA, kn = min(EPA, Kc - ka);
        const int nr = (N - part + parts - 1) / parts;  // rows part, part + parts, ...
        unsigned char* bh = base + Lo.b_hi + (uint32_t)at * atom_bytes;
        unsigned char* bl = base + Lo.b_lo + (uint32_t)at * atom_bytes;
        if (s == 0) {
          // 16-byte chunk c of row n holds K elements ka + 8c .. +7
          for (int idx = lane; idx < nr * 8; idx += 32) {
            const int n = part + (idx >> 3) * parts, c = idx & 7;
            const uint32_t off = sw_off(n, c);
            const bool in = src != nullptr && c * 8 < kn;
            const T* sp = src + k0 + ka + c * 8 + (int64_t)n * ldsrc;
            if (BF) {
              const uint4 v = in ? ldcg16(sp) : make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(bh + off) = v;
            } else {
              // K slices are multiples of 4 fp32 elements: the last chunk of a
              // slice may hold only its first half
              uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
              if (in) {
                v0 = ldcg16(sp);
                if (c * 8 + 4 < kn) v1 = ldcg16(sp + 4);
              }
              uint4 h4, l4;
              split_f16x2(__uint_as_float(v0.x) * h_scale, __uint_as_float(v0.y) * h_scale, h4.x, l4.x);
              split_f16x2(__uint_as_float(v0.z) * h_scale, __uint_as_float(v0.w) * h_scale, h4.y, l4.y);
              split_f16x2(__uint_as_float(v1.x) * h_scale, __uint_as_float(v1.y) * h_scale, h4.z, l4.z);
              split_f16x2(__uint_as_float(v1.z) * h_scale, __uint_as_float(v1.w) * h_scale, h4.w, l4.w);
              *reinterpret_cast<uint4*>(bh + off) = h4;
              *reinterpret_cast<uint4*>(bl + off) = l4;
            }
          }
        } else {
          // lane l takes the rows of half l >> 4 of the task's rows (rows
          // part + (2 i + (l >> 4)) * parts) and units 4 (l & 15) .. +3 of the
          // atom (bytes 8 (l & 1) .. +7 of 16-byte chunk (l & 15) >> 1 of the
          // swizzled row): one 32-byte load per row, two rows per warp load,
          // up to kPollRows4 rows of a lane in flight at once
          const int hsub = lane >> 4, q4 = lane & 15;
          const bool lane_in = 4 * q4 < kn;  // slices and atoms hold multiples of 4 units
          const uint32_t woff = (uint32_t)(q4 & 1) * 8u;
          const int nl = (nr - hsub + 1) / 2;  // this lane's rows
          for (int r0 = 0; r0 < (nr + 1) / 2; r0 += kPollRows4) {  // warp-uniform trip count
            const int nb = max(0, min(kPollRows4, nl - r0));
            unsigned long long w[kPollRows4][4];
            if (!poll_tagged4<kPollRows4>(hxp + ka + 4 * q4, part + (2 * r0 + hsub) * parts,
                                          2 * parts, H, nb, lane_in, (unsigned)s, w, p.status,
                                          p.timeout_ns) &&
                lane == 0)
              s_fail = 1;  // the data is not used: the status word holds the failure
            if (lane_in) {
#pragma unroll
              for (int j = 0; j < kPollRows4; ++j) {
                if (j >= nb) break;
                const int n = part + (2 * (r0 + j) + hsub) * parts;
                const uint32_t off = sw_off(n, q4 >> 1) + woff;
                const float f0 = __uint_as_float((uint32_t)w[j][0]);
                const float f1 = __uint_as_float((uint32_t)w[j][1]);
                const float f2 = __uint_as_float((uint32_t)w[j][2]);
                const float f3 = __uint_as_float((uint32_t)w[j][3]);
                if (BF) {
                  *reinterpret_cast<uint2*>(bh + off) =
                      make_uint2((__float_as_uint(f0) >> 16) | ((__float_as_uint(f1) >> 16) << 16),
                                 (__float_as_uint(f2) >> 16) | ((__float_as_uint(f3) >> 16) << 16));
                } else {
                  uint32_t h0, l0, h1, l1;
                  split_f16x2(f0 * h_scale, f1 * h_scale, h0, l0);
                  split_f16x2(f2 * h_scale, f3 * h_scale, h1, l1);
                  *reinterpret_cast<uint2*>(bh + off) = make_uint2(h0, h1);
                  *reinterpret_cast<uint2*>(bl + off) = make_uint2(l0, l1);
                }
              }
            }
          }
        }
        WTRACE(s, at);
      }
    }
    // the staged tiles to the tensor cores' (async) proxy, then one barrier: a
    // per-atom mbarrier measured slower (each wait costs about 100 ns)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    TTRACE(s, 1);
    XTRACE(s, 1);
    if (have) {
      // 2. MMA issue: issuer i is lane 0 of warp kTWarps-1-i and runs pass i
      // into accumulator i (pass 0: W_hi h_hi, 1: W_hi h_lo, 2: W_lo h_hi);
      // descriptors advance by whole atoms and 32-byte K steps inside the
      // start-address field; the padded tail of the last atom multiplies
      // zeros (B columns >= Kc are staged as zeros, W columns >= Kc are zero;
      // predicating its K steps off measured slower: the issue loop must stay
      // minimal)
      const int iss = kTWarps - 1 - warp;
      if (iss >= 0 && iss < NI) {
        if (lane == 0) {
          const uint32_t dcol = tmem + (uint32_t)(iss * Nm);
          const uint64_t bd0 = b_desc(base_s + ((!BF && iss == 1) ? Lo.b_lo : Lo.b_hi));
          const uint64_t bstep = (uint64_t)(atom_bytes >> 4);
          const uint32_t acol0 = tmem + ((!BF && iss == 2) ? a_lo_col : a_col);
          fence_after();
          // a loop over the atoms: the fully unrolled issue (mma_pass_n)
          // measured slower in this kernel (more code in the step loop)
          for (int at = 0; at + 1 < KCu; ++at) {
            const uint64_t bd = bd0 + (uint64_t)at * bstep;
            const uint32_t acol = acol0 + (uint32_t)(at * 32);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_a_tmem(true, dcol, acol + (uint32_t)(kk * 8), bd + (uint64_t)(kk * 2), idesc,
                         (at | kk) ? 1u : 0u);
          }
          {
            // the last atom: only its K steps that hold some of the slice
            const int at = KCu - 1;
            const int ksl = (Kc - at * EPA + 15) / 16;
            const uint64_t bd = bd0 + (uint64_t)at * bstep;
            const uint32_t acol = acol0 + (uint32_t)(at * 32);
            for (int kk = 0; kk < ksl; ++kk)
              mma_a_tmem(true, dcol, acol + (uint32_t)(kk * 8), bd + (uint64_t)(kk * 2), idesc,
                         (at | kk) ? 1u : 0u);
          }
          asm volatile(
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                  mbar)
              : "memory");
          WTRACE(s, 16 + iss);
        }
        __syncwarp();
      }
      TTRACE(s, 6);
    }
    // this step's input projection values, each item's G values fetched by the
    // thread that consumes them (it waits for its own copies only): issued
    // after the polls, whose loads would otherwise queue behind these reads
    // of memory, and consumed after the contraction and the exchange
    if (!failed) {
      const int64_t grow = (int64_t)t * N;
      for (int it = tid; it < items; it += kTThreads) {
        const int uu = it == tid ? i_uu : it % Uqc, n = it == tid ? i_n : it / Uqc;
        const float* src = a.gx + (grow + n) * GH + u0 + uq0 + uu;
        for (int g = 0; g < G; ++g) cp_async4(gxs + (g * N + n) * Uq + uu, src + (int64_t)g * H);
      }
    }
    cp_async_commit();
    // wait for the products (every thread, the phase of this step)
    bool mma_ok = true;
    if (have) {
      mma_ok = mbar_wait_bounded(mbar, mma_phase, p.status, p.timeout_ns);
      if (!mma_ok) s_mma_bad = 1;
      mma_phase ^= 1u;
    }
    mma_ok = __all_sync(0xffffffffu, mma_ok);
    fence_after();
    TTRACE(s, 2);
    // 3. push D's rows (partials over this block's K slice, accumulators summed
    // in a fixed order) to the owners; warps 0-3 take columns 0-15, warps 4-7
    // columns 16-31 (then 32-47 and 48-63, ...)
    const int Rs = Nm + 4;  // exchange row stride (floats): 16-byte rows, fewer bank conflicts
    float* recv = recv0 + (size_t)(s & 1) * Pk * G * Uq * Rs;
    if (!failed && Kc > 0) {
      const int quarter = warp & 3;
      const int g = e_g, uo = e_uo, owner = e_owner;
      const bool row_ok = e_row_ok;
      const bool ok = have && mma_ok;
      const uint32_t lrow = tmem + ((uint32_t)(quarter * 32) << 16);
      for (int c0 = (warp >> 2) * 16; c0 < N; c0 += (kTWarps / 4) * 16) {
        float v[NI][16];
        if (ok) {
          if constexpr (NI == 3) {
            // the three accumulators' loads in flight together, one wait
            tmem_ld16x3(lrow + (uint32_t)c0, lrow + (uint32_t)(Nm + c0),
                        lrow + (uint32_t)(2 * Nm + c0), v[0], v[1], v[2]);
            // (hi hi + (hi lo + lo hi) 2^-11) / (w_scale h_scale), powers of two
#pragma unroll
            for (int e = 0; e < 16; ++e)
              v[0][e] = fmaf(v[1][e] + v[2][e], 1.f / 2048.f, v[0][e]) * out_scale;
          } else {
            tmem_ld16(lrow + (uint32_t)c0, v[0]);
          }
          if (warp == 0 && c0 == 0) WTRACE(s, 24);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[0][e] = 0.f;
        }
        if (!row_ok || owner >= Pk) continue;
        // 16-byte pieces (rows of Nm + 4 floats, Nm % 16 == 0); columns N .. Nm-1
        // of D are zero (the staged rows beyond N are zero) and unread
        float* dst = recv + ((size_t)q * G * Uq + g * Uq + uo) * Rs + c0;
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          if (c0 + i < N)
            st_async4(dst + i, rbar, (unsigned)owner, v[0][i], v[0][i + 1], v[0][i + 2],
                      v[0][i + 3]);
      }
      if (warp == 0) WTRACE(s, 25);
    }
    // the previous step's outputs, while the partners' partials are in flight
    // (issued here, not beside the MMA issue, whose issuing lanes share their
    // schedulers with these warps)
    if (pend >= 0) flush(pend);
    pend = -1;
    // 4. the threads with pointwise items wait for this step's partials: the
    // pushes complete the owner's barrier themselves, so no cluster barrier
    // and no release of this block's earlier global stores is waited for
    bool live = !failed && mma_ok;
    if (live && tid < items) {
      live = mbar_wait_cluster_bounded(rbar, (uint32_t)(s >> 1) & 1u, p.status, p.timeout_ns);
      if (!live) s_fail = 1;
    }
    WTRACE(s, 22 + (warp & 1));
    TTRACE(s, 3);
    if (live) {
      // the partial sums of each gate (rank order, fixed; ranks with an empty K
      // slice push nothing) feed the gate math;
      // the exchange word of h_t goes out first; the workspace outputs wait in
      // the stash until the next step
      const size_t rstride = (size_t)G * Uq * Rs;
      for (int it = tid; it < items; it += kTThreads) {
        const int uu = it == tid ? i_uu : it % Uqc, n = it == tid ? i_n : it / Uqc;
        const int j = u0 + uq0 + uu;
        cp_async_wait_all();                    // this thread's projection values
        const float* gv = gxs + n * Uq + uu;    // gate g at gv[g * N * Uq]
        // all partials loaded first (independent shared loads in flight
        // together), then summed in rank order
        float ov[4], pv[4][kMaxPushers];
        {
          const uint32_t rp0 = smem_addr(recv + (size_t)uu * Rs + n);
#pragma unroll
          for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int rank = 0; rank < kMaxPushers; ++rank)
              pv[g][rank] = (g < G && rank < pushers)
                                ? ld_shared_f32(rp0 + 4u * (uint32_t)(g * Uq * Rs + rank * rstride))
                                : 0.f;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            ov[g] = 0.f;
#pragma unroll
            for (int rank = 0; rank < kMaxPushers; ++rank) ov[g] += pv[g][rank];
          }
        }
        if (it == tid) PTRACE(s, 26, ov[0] + ov[1] + ov[2] + ov[3] + gv[0]);
#ifdef LAYER_RNN_TRACE
        // the same loads once more, now with the code and data warm
        if (it == tid) {
          const uint32_t rq = smem_addr(recv + (size_t)uu * Rs + n);
          float w2 = 0.f;
#pragma unroll
          for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int rank = 0; rank < kMaxPushers; ++rank)
              w2 += (g < G && rank < pushers)
                        ? ld_shared_f32(rq + 4u * (uint32_t)(g * Uq * Rs + rank * rstride))
                        : 0.f;
          PTRACE(s, 31, w2);
        }
#endif
        float h, g0 = 0.f, g1 = 0.f, g2 = 0.f, g3 = 0.f, c = 0.f;
        if (p.mode == 1) {
          g0 = sigmoid_fast(gv[0] + ov[0]);
          g1 = sigmoid_fast(gv[N * Uq] + ov[1]);
          g2 = tanh_fast(gv[2 * N * Uq] + ov[2]);
          g3 = sigmoid_fast(gv[3 * N * Uq] + ov[3]);
          c = g1 * cst[n * Uq + uu] + g0 * g2;
          h = g3 * tanh_fast(c);
        } else if (p.mode == 2) {
          g3 = ov[2] + s_bhn[uu];  // W_hn h + b_hn
          g0 = sigmoid_fast(gv[0] + ov[0]);
          g1 = sigmoid_fast(gv[N * Uq] + ov[1]);
          g2 = tanh_fast(gv[2 * Uq * N] + g0 * g3);
          h = (1.f - g1) * g2 + g1 * hst[n * Uq + uu];
        } else {
          h = tanh_fast(gv[0] + ov[0]);
        }
        if (VL && t >= seq_len(it, n)) {
          // past the sequence's length: the state is kept (its gates are
          // still stored; the backward does not read them there)
          h = hst[n * Uq + uu];
          if (p.mode == 1) c = cst[n * Uq + uu];
        }
        const T hs = from_f<T>(h);
        if (it == tid) PTRACE(s, 27, h);
        // the exchange word of h_t: its value as stored (what y holds) and the
        // step that reads it
        if (s + 1 < nT && !(blockIdx.x == p.fault_block && s == p.fault_step))
          st_relaxed_u64(a.hx + ((size_t)(s % 3) * N + n) * H + j,
                         ((unsigned long long)(s + 1) << 32) | __float_as_uint(to_f(hs)));
        if (it == tid) PTRACE(s, 28, h);
        if (it == tid) XTRACE(s, 0);
        hst[n * Uq + uu] = h;
        if (p.mode == 1) cst[n * Uq + uu] = c;
        outs[it] = h;
        outs[icap + it] = g0;
        outs[2 * icap + it] = g1;
        outs[3 * icap + it] = g2;
        outs[4 * icap + it] = g3;
        outs[5 * icap + it] = c;
        if (it == tid) PTRACE(s, 29, h);
      }
      pend = s;
    }
    PTRACE(s, 30, 0.f);
    TTRACE(s, 4);
    TTRACE(s, 5);
    if ((!live || s_mma_bad) && tid == 0) s_fail = 1;
    __syncthreads();
  }
  if (pend >= 0) flush(pend);
  fence_before();
  cl_sync();  // no block leaves while a peer may still store into it
  if (s_fail == 0) {
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

// The forward kernel's step protocol with no work: per step, each warp polls
// the exchange words of its atoms' units, one block barrier, each block with
// a K slice pushes 16 bytes to every owner of its cluster (completing the
// owner's receive barrier), the owners' threads wait for their barrier and
// write the exchange words of their units -- the part of a step's latency
// that no arithmetic removes.  Same grid, clusters, exchange words, barriers
// and waits as rec_fwd_tc; bounded like it.
__global__ void __launch_bounds__(kTThreads, 1) rec_step_probe(const __grid_constant__ RecParams p) {
  __shared__ int s_fail;
  __shared__ __align__(8) uint64_t recv_bar[2];
  __shared__ __align__(16) float recv[2][32][4];
  const RecPlan& pl = p.plan;
  const int P = pl.P, Pk = pl.cluster;
  const int d = blockIdx.x / P;
  const int b = blockIdx.x - d * P;
  const int r = b / Pk, q = b % Pk;
  const RecDirArgs& a = p.dir[d];
  const int H = p.H, N = p.N, Ur = pl.Ur, Uq = pl.Uq;
  const int u0 = r * Ur, Urc = min(Ur, H - u0);
  const int uq0 = q * Uq, Uqc = max(0, min(Uq, Urc - uq0));
  const int Kk = max(1, pl.Kk);
  const int k0 = q * Kk, Kc = max(0, min(Kk, H - k0));
  const int EPA = 64, KCu = (Kc + EPA - 1) / EPA;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x, items = Uqc * N;
  const int pushers = min(Pk, (H + Kk - 1) / Kk);
  const uint32_t rbar0 = smem_addr(&recv_bar[0]);
  const bool cfg_bad = cl_size() != (unsigned)Pk || cl_rank() != (unsigned)q || a.hx == nullptr ||
                       Pk > 32 || (H & 3) != 0 || (Kk & 3) != 0;
  if (tid == 0) {
    s_fail = cfg_bad;
    if (cfg_bad) atomicCAS(p.status, kDevOk, kDevCheck);
    mbar_init(rbar0, 1);
    mbar_init(rbar0 + 8u, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cl_sync();
  const int parts = max(1, kTWarps / max(1, KCu));
  for (int s = 0; s < p.T; ++s) {
    const bool failed = s_fail != 0;
    const uint32_t rbar = rbar0 + 8u * (uint32_t)(s & 1);
    if (!failed && tid == 0) mbar_arrive_expect_tx(rbar, Uqc > 0 ? (uint32_t)pushers * 16u : 0u);
    if (!failed && s > 0) {
      const unsigned long long* hxp = a.hx + (size_t)((s + 2) % 3) * N * H + k0;
      for (int task = warp; task < KCu * parts; task += kTWarps) {
        const int at = task % KCu, part = task / KCu;
        const int ka = at * EPA, kn = min(EPA, Kc - ka);
        const int nr = (N - part + parts - 1) / parts;
        const int hsub = lane >> 4, q4 = lane & 15;
        const int nl = (nr - hsub + 1) / 2;
        for (int r0 = 0; r0 < (nr + 1) / 2; r0 += kPollRows4) {
          unsigned long long w[kPollRows4][4];
          if (!poll_tagged4<kPollRows4>(hxp + ka + 4 * q4, part + (2 * r0 + hsub) * parts,
                                        2 * parts, H, max(0, min(kPollRows4, nl - r0)),
                                        4 * q4 < kn, (unsigned)s, w, p.status, p.timeout_ns) &&
              lane == 0)
            s_fail = 1;
        }
      }
    }
    __syncthreads();
    // one 16-byte piece to each owner of the cluster that has units
    if (!failed && Kc > 0 && tid < Pk && min(Uq, Urc - tid * Uq) > 0)
      st_async4(&recv[s & 1][q][0], rbar, (unsigned)tid, 0.f, 0.f, 0.f, 0.f);
    bool live = !failed;
    if (live && tid < items) {
      live = mbar_wait_cluster_bounded(rbar, (uint32_t)(s >> 1) & 1u, p.status, p.timeout_ns);
      if (!live) s_fail = 1;
    }
    if (live && s + 1 < p.T)
      for (int it = tid; it < items; it += kTThreads) {
        const int uu = it % Uqc, n = it / Uqc;
        st_relaxed_u64(a.hx + ((size_t)(s % 3) * N + n) * H + u0 + uq0 + uu,
                       (unsigned long long)(s + 1) << 32);
      }
    __syncthreads();
  }
  cl_sync();
}

}  // namespace

cudaError_t rec_tc_probe_launch(const RecParams& p, cudaStream_t st) {
  const RecPlan& pl = p.plan;
  void* fn = (void*)rec_step_probe;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  for (int d = 0; d < p.D; ++d) {
    if (!p.dir[d].hx) return cudaErrorInvalidValue;
    e = cudaMemsetAsync(p.dir[d].hx, 0, rec_tc_xchg_bytes(p.N, p.H), st);
    if (e != cudaSuccess) return e;
  }
  RecParams copy = p;
  void* args[] = {&copy};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.D * pl.P);
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = pl.smem;  // the forward's size: one block per SM, as there
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

size_t rec_tc_xchg_bytes(int N, int H) { return (size_t)3 * N * H * 8; }

bool rec_tc_plan(int mode, int bf16, int D, int H, int N, int num_sms, size_t smem_limit,
                 const int* max_clusters, RecPlan* out) {
  const int G = mode == 1 ? 4 : mode == 2 ? 3 : 1;
  const int e = bf16 ? 2 : 4;
  if ((H * e) % 16 != 0 || N < 1 || N > 256) return false;
  const int Nm = (N + 15) / 16 * 16;
  const int Ur_max = kTM / G;
  const int NI = bf16 ? 1 : 3;
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
    const int epc = 64;                                   // 16-bit elements per 128-byte atom
    const int Kk = (((H + Pk - 1) / Pk) + 7) / 8 * 8;     // 16-byte aligned slices
    const int Kp = (Kk + epc - 1) / epc * epc;
    if (Kp / epc > kMaxAtoms) continue;
    const int acols = bf16 ? Kp / 2 : Kp;                 // W (bf16) / W_hi and W_lo (fp32 split)
    int cols = 32;
    while (cols < NI * Nm + acols) cols *= 2;
    if (cols > 512) continue;
    RecPlan pl;
    pl.direct = 0;
    pl.cluster = Pk; pl.Pr = Pr; pl.P = Pr * Pk; pl.Ur = Ur; pl.Uq = Uq;
    pl.Kk = Kk;
    pl.K = Kp;                       // padded K slice
    pl.KC = Kp / epc;                // K atoms of 128 bytes
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
extern "C" int rnn_debug_fwtrace_copy(void* host, size_t bytes) {
  if (bytes > sizeof(g_wtrace)) bytes = sizeof(g_wtrace);
  return (int)cudaMemcpyFromSymbol(host, g_wtrace, bytes);
}
extern "C" int rnn_debug_xtrace_copy(void* host, size_t bytes) {
  if (bytes > sizeof(g_xtrace)) bytes = sizeof(g_xtrace);
  return (int)cudaMemcpyFromSymbol(host, g_xtrace, bytes);
}
extern "C" int rnn_debug_ttrace_clear() {
  static unsigned long long zeros[4][1024][8];
  return (int)cudaMemcpyToSymbol(g_ttrace, zeros, sizeof(zeros));
}
#endif

cudaError_t rec_tc_launch(const RecParams& p, cudaStream_t st) {
  const RecPlan& pl = p.plan;
  void* fn = p.lengths ? (p.bf16 ? (void*)rec_fwd_tc<true, true> : (void*)rec_fwd_tc<false, true>)
                       : (p.bf16 ? (void*)rec_fwd_tc<true, false> : (void*)rec_fwd_tc<false, false>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  // exchange words from an earlier launch must not look current: tags start at 1
  for (int d = 0; d < p.D; ++d) {
    if (!p.dir[d].hx) return cudaErrorInvalidValue;
    e = cudaMemsetAsync(p.dir[d].hx, 0, rec_tc_xchg_bytes(p.N, p.H), st);
    if (e != cudaSuccess) return e;
  }
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
