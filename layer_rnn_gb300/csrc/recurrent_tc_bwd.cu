// Tensor-core path of the persistent recurrent backward kernel.
//
// Backward through time (reverse-mode through the recurrences of the
// "rnn training example?" thread, reading 13 of the design notes for the
// loss): per step
//     dh_{t-1}[n][k] = sum_j dG_h[t][n][j] * W_hh[j][k]   (+ GRU: dh_t[n][k] * z_t[n][k])
// with j over the G*H gate rows.  The contraction is K = G*H long, so the
// blocks of a cluster (up to 16, a non-portable cluster size) split it: block
// (r, q) keeps W_hh^T for the Ur units of row group r and the gate rows
// k0 .. k0+Kk-1 in tensor memory as the MMA's A operand and stages the
// previous step's dG_h slice as the swizzled K-major B operand.
//
// fp32 operands are split into fp16 pairs, x = (hi + lo * 2^-11) / scale
// (hi = fp16(x * scale), lo = fp16((x * scale - hi) * 2^11)), with power-of-
// two scales per block: W_hh^T's from its slice once (its largest magnitude
// just below 2^14), dG_h's per step (gradients have no fixed range): the
// slice is split as it is polled with a scale predicted from the previous
// step's slice (three binades of room for growth), and split again from its
// fp32 copy only when this step's largest magnitude would overflow that scale
// or sit more than nine binades under it.  The product keeps hi*hi + hi*lo + lo*hi:
// three passes of 16 K, each issued by its own thread into its own
// accumulator, about 22 significant bits per operand as three tf32 passes,
// in half the MMA instructions.  bf16 runs one pass.
//
// Per step: warps poll the exchange words of their K atoms -- each 8-byte word
// holds a dG_h value and the step that reads it, written by the owner of the
// gate row, so the data is its own flag -- and stage them; one block barrier;
// the MMAs; the accumulator rows go over distributed shared memory (16-byte
// asynchronous stores that complete the owner's receive barrier) to the block
// that owns each unit's pointwise step; the owners wait for their barrier,
// sum the partials in a fixed order, run the gate-gradient chain, and write
// the exchange words of dG_h; the canonical dG_h (GRU: and dG_x), which no
// block of this launch reads, waits in shared memory and is stored after the
// next step's polls.  The step's pointwise inputs (dy, the saved gates, c_t
// and c_{t-1}) are fetched with cp.async at the start of the step.
#include <algorithm>
#include <cstdio>
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
constexpr int kBWarps = kBThreads / 32;
constexpr int kBM = 128;    // MMA M: output units per row group (padded)
constexpr int kNIn = 7;     // pointwise inputs per item: dy, 4 gates, c_t, c_{t-1} / h_{t-1}
constexpr int kBMaxAtoms = 16;
constexpr int kBPollRows4 = 8;  // rows of 4 words a lane polls at once
constexpr int kBMaxPushers = 16;  // largest cluster of the plan

struct BLayout {
  uint32_t b_hi, b_lo;   // staged B tiles: KC atoms x (Nm rows x 128 bytes)
  uint32_t raw;          // fp32: the staged dG_h slice before its split, [N][Kp + 4]
  uint32_t recv;         // [2][Pk][Uq][Nm + 4] f32
  uint32_t st_dc, st_carry;  // [Uq*N] f32: LSTM dc, GRU dh*z
  uint32_t stash;        // [7][Uq*N] f32: GRU dG_x, then dG_h (stored one step late)
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
  L.raw = off;
  off += bf ? 0 : (uint32_t)N * (pl.K + 4) * 4u;
  L.recv = off;
  off += 2u * pl.cluster * pl.Uq * (pl.nbp + 4) * 4u;
  L.st_dc = off;
  off += (uint32_t)pl.Uq * N * 4u;
  L.st_carry = off;
  off += (uint32_t)pl.Uq * N * 4u;
  L.stash = off;
  off += 7u * pl.Uq * N * 4u;
  L.pin = off;
  off += (uint32_t)kNIn * pl.Uq * N * 4u;
  L.total = (off + 1023u) & ~1023u;
  return L;
}

template <bool BF, bool VL>  // VL: per-sequence lengths (p.lengths) are read
__global__ void __launch_bounds__(kBThreads, 1) rec_bwd_tc(const __grid_constant__ RecParams p) {
  typedef typename std::conditional<BF, bf16, float>::type T;
  constexpr int NI = BF ? 1 : 3;     // issuing threads = accumulators (one per pass)
  constexpr int EPA = 64;            // K elements (16-bit) per 128-byte atom
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ __align__(8) uint64_t recv_bar[2];  // partials of steps s (s & 1) landed
  __shared__ uint32_t tmem_slot;
  __shared__ int s_fail, s_mma_bad;
  __shared__ float s_red[kBWarps];
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
  const int KCu = (Kc + EPA - 1) / EPA;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

#ifdef LAYER_RNN_TRACE
  if (blockIdx.x == 0 && threadIdx.x == 0)
    printf("%s plan: P %d cluster %d Ur %d Uq %d Kk %d K %d KC %d Nm %d cols %d\n", "bwd", pl.P,
           pl.cluster, pl.Ur, pl.Uq, pl.Kk, pl.K, pl.KC, pl.nbp, pl.lda);
#endif
  const uint32_t base_s = (smem_addr(smem_raw) + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_s - smem_addr(smem_raw));
  const BLayout Lo = b_layout(pl, N, BF);
  float* raw = reinterpret_cast<float*>(base + Lo.raw);
  float* recv0 = reinterpret_cast<float*>(base + Lo.recv);
  float* st_dc = reinterpret_cast<float*>(base + Lo.st_dc);
  float* st_carry = reinterpret_cast<float*>(base + Lo.st_carry);
  float* stash = reinterpret_cast<float*>(base + Lo.stash);
  float* pin = reinterpret_cast<float*>(base + Lo.pin);
  const uint32_t atom_bytes = (uint32_t)Nm * 128u;
  const uint32_t mbar = smem_addr(&mma_bar);
  const uint32_t rbar0 = smem_addr(&recv_bar[0]);
  // tensor memory: accumulator i at column i * Nm, then the A operands, two
  // 16-bit elements per column: W^T (bf16) or its hi and lo halves (fp32)
  const uint32_t a_col = (uint32_t)(NI * Nm);
  const uint32_t a_lo_col = a_col + (uint32_t)(Kp / 2);
  const uint32_t ncols = (uint32_t)pl.lda;
  const int items = Uqc * N;
  const int icap = Uq * N;  // stride of one input array in pin
  const int Rs = Nm + 4;    // exchange row stride (floats)
  const int Ks = Kp + 4;    // raw staging row stride (floats)

  const bool cfg_bad = cl_size() != (unsigned)Pk || cl_rank() != (unsigned)q ||
                       a_col + (uint32_t)(BF ? Kp / 2 : Kp) > ncols || ncols > 512u ||
                       (ncols & (ncols - 1u)) != 0 || ncols < 32u || Ur > kBM || N > Nm ||
                       Nm % 16 != 0 || Nm > 256 || Kp % EPA != 0 || pl.KC * EPA != Kp ||
                       pl.KC > kBMaxAtoms || pl.Kk > Kp || Uq * Pk < Ur || Pk > kBMaxPushers ||
                       a.hx == nullptr || (GH & 3) != 0 || (pl.Kk & 3) != 0;
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
  // staged tiles zero: rows >= N and columns >= Kc stay zero
  for (uint32_t i = tid; i < Lo.recv / 16u; i += kBThreads)
    reinterpret_cast<uint4*>(base)[i] = make_uint4(0, 0, 0, 0);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_slot;
  const T* W = reinterpret_cast<const T*>(a.whh);

  // W^T's split scale (fp32): its slice's largest magnitude just below 2^14
  int ew = 0;
  float w_scale = 1.f;
  if (!BF) {
    float wm = 0.f;
    if (!cfg_bad)
      for (int idx = tid; idx < Kc * Urc; idx += kBThreads) {
        const int jj = idx / Urc, m = idx - jj * Urc;
        wm = fmaxf(wm, fabsf(to_f(W[(int64_t)(k0 + jj) * H + u0 + m])));
      }
    for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
    if (lane == 0) s_red[warp] = wm;
    __syncthreads();
    wm = 0.f;
    for (int w = 0; w < kBWarps; ++w) wm = fmaxf(wm, s_red[w]);
    __syncthreads();
    if (wm > 0.f) (void)frexpf(wm, &ew);
    ew = min(max(14 - ew, -100), 100);
    w_scale = ldexpf(1.f, ew);
  }

  // A = W_hh^T slice into tensor memory: lane m = unit u0 + m, columns =
  // gate-row pairs (k0 + jj, k0 + jj + 1); lanes of a warp read consecutive
  // units of one W_hh row
  if (!cfg_bad) {
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const bool row_ok = m < Urc;
    const int nchunk = pl.KC;  // 32 columns = 64 gate rows per chunk
    for (int ci = warp >> 2; ci < nchunk; ci += kBThreads / 128) {
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int jj = ci * 64 + 2 * i;
        const float e0 = (row_ok && jj < Kc) ? to_f(W[(int64_t)(k0 + jj) * H + u0 + m]) : 0.f;
        const float e1 =
            (row_ok && jj + 1 < Kc) ? to_f(W[(int64_t)(k0 + jj + 1) * H + u0 + m]) : 0.f;
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

  // state of the own items: item it = n * Uqc + uu (consecutive threads take
  // consecutive units: coalesced global accesses)
  for (int it = tid; it < items; it += kBThreads) {
    const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
    st_dc[it] = a.dcy ? a.dcy[(int64_t)n * H + j] : 0.f;
    st_carry[it] = 0.f;
  }
  T* dgx = reinterpret_cast<T*>(a.dgx);
  T* dgh = reinterpret_cast<T*>(a.dgh);
  const T* hseq = reinterpret_cast<const T*>(a.hseq);
  // kind::f16 with bf16 (1) or fp16 (0) operands, fp32 accumulate
  const uint32_t idesc = (1u << 4) | ((BF ? 1u : 0u) << 7) | ((BF ? 1u : 0u) << 10) |
                         ((uint32_t)(Nm >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
  const int parts = max(1, kBWarps / max(1, KCu));
  // bytes of partial sums pushed to this block per step (s >= 1): one row per
  // own unit, N columns in 16-byte pieces, from each block of the cluster
  // whose K slice is not empty (a block with an empty slice polls nothing and
  // would run ahead of the exchange, so it pushes nothing); every pusher
  // polls its slice each step, so its step-s pushes land only after every
  // owner of its cluster consumed the partials of step s - 2
  const int pushers = (int)min((int64_t)Pk, (GH + max(1, pl.Kk) - 1) / max(1, pl.Kk));
  const uint32_t rx_bytes = (uint32_t)(pushers * Uqc * ((N + 3) / 4) * 16);
  // every block's barriers are initialised before any peer pushes into them
  fence_before();
  cl_sync();
  fence_after();
  uint32_t mma_phase = 0;
  // the gate gradients of step sp (dG_h; GRU: also dG_x) from the stash, each
  // item by the thread that computed it: written one step late, after the
  // next step's polls, so that these stores do not queue ahead of the polls
  const int ngo = p.mode == 1 ? 4 : p.mode == 2 ? 3 : 1;
  auto flush = [&](int sp) {
    const int tq = rv ? sp : nT - 1 - sp;
    for (int it = tid; it < items; it += kBThreads) {
      const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
      const int64_t row = (int64_t)tq * N + n;
      T* gho = dgh + row * GH + j;  // dG_x itself, except for the GRU
      for (int g = 0; g < ngo; ++g) gho[(int64_t)g * H] = from_f<T>(stash[(3 + g) * icap + it]);
      if (p.mode == 2) {
        T* gxo = dgx + row * GH + j;
        gxo[0] = from_f<T>(stash[it]);
        gxo[H] = from_f<T>(stash[icap + it]);
        gxo[2 * H] = from_f<T>(stash[2 * icap + it]);
      }
    }
  };
  int pend = -1;  // the step whose gradients wait in the stash
  // the valid length of this thread's first item's sequence (read once, off
  // the steps' critical path); other items read theirs when they run
  const int i_len =
      (VL && tid < items) ? __ldg(p.lengths + tid / max(1, Uqc)) : 0x7fffffff;
  // fp32: the dG_h scale exponent predicted from the previous step's slice
  int pred_eh = 0;
  float pred_scale = 1.f;
  bool pred_ok = false;

  for (int s = 0; s <= nT; ++s) {
    const int t = rv ? s : nT - 1 - s;   // time processed at this step (s < nT)
    const bool failed = s_fail != 0;     // read after the previous step's barrier
    // the partials of step s >= 1 land in buffer and barrier s & 1 (use
    // (s - 1) >> 1 of that barrier): one arrival plus the peers' bytes
    const uint32_t rbar = rbar0 + 8u * (uint32_t)(s & 1);
    if (!failed && s > 0 && tid == 0) mbar_arrive_expect_tx(rbar, rx_bytes);
    BTRACE(s, 0);
    const bool have = !failed && s > 0 && Kc > 0;
    // 1. staging of the previous step's dG_h slice: task (atom, row part) ->
    // warp; the warp polls the exchange words of its atom (value and step in
    // one 8-byte word, written by the owners of those gate rows: the data is
    // its own flag) and stages them as B (bf16) or as raw fp32 until the
    // step's scale is known
    float lmax = 0.f;
    if (have) {
      const unsigned long long* gxp = a.hx + (size_t)((s + 2) % 3) * N * GH + k0;
      for (int task = warp; task < KCu * parts; task += kBWarps) {
        const int at = task % KCu, part = task / KCu;
        const int ka = at * EPA, kn = min(EPA, Kc - ka);
        const int nr = (N - part + parts - 1) / parts;  // rows part, part + parts, ...
        // lane l takes the rows of half l >> 4 of the task's rows (rows
        // part + (2 i + (l >> 4)) * parts) and gate rows ka + 4 (l & 15) .. +3:
        // one 32-byte load per row, two rows per warp load
        const int hsub = lane >> 4, q4 = lane & 15;
        const bool lane_in = 4 * q4 < kn;  // slices and atoms hold multiples of 4 gate rows
        const int nl = (nr - hsub + 1) / 2;  // this lane's rows
        for (int r0 = 0; r0 < (nr + 1) / 2; r0 += kBPollRows4) {  // warp-uniform trip count
          const int nb = max(0, min(kBPollRows4, nl - r0));
          unsigned long long w[kBPollRows4][4];
          if (!poll_tagged4<kBPollRows4>(gxp + ka + 4 * q4, part + (2 * r0 + hsub) * parts,
                                         2 * parts, GH, nb, lane_in, (unsigned)s, w, p.status,
                                         p.timeout_ns) &&
              lane == 0)
            s_fail = 1;  // the data is not used: the status word holds the failure
          if (!lane_in) continue;
#pragma unroll
          for (int j = 0; j < kBPollRows4; ++j) {
            if (j >= nb) break;
            const int n = part + (2 * (r0 + j) + hsub) * parts;
            const float f0 = __uint_as_float((uint32_t)w[j][0]);
            const float f1 = __uint_as_float((uint32_t)w[j][1]);
            const float f2 = __uint_as_float((uint32_t)w[j][2]);
            const float f3 = __uint_as_float((uint32_t)w[j][3]);
            if (BF) {
              *reinterpret_cast<uint2*>(base + Lo.b_hi + (uint32_t)at * atom_bytes +
                                        sw_off(n, q4 >> 1) + (uint32_t)(q4 & 1) * 8u) =
                  make_uint2((__float_as_uint(f0) >> 16) | ((__float_as_uint(f1) >> 16) << 16),
                             (__float_as_uint(f2) >> 16) | ((__float_as_uint(f3) >> 16) << 16));
            } else {
              *reinterpret_cast<float4*>(raw + n * Ks + ka + 4 * q4) = make_float4(f0, f1, f2, f3);
              lmax = fmaxf(lmax, fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3))));
              if (pred_ok) {
                // split now with the predicted scale (kept if the step's max
                // turns out to fit it)
                uint32_t h0, l0, h1, l1;
                split_f16x2(f0 * pred_scale, f1 * pred_scale, h0, l0);
                split_f16x2(f2 * pred_scale, f3 * pred_scale, h1, l1);
                const uint32_t off = (uint32_t)at * atom_bytes + sw_off(n, q4 >> 1) +
                                     (uint32_t)(q4 & 1) * 8u;
                *reinterpret_cast<uint2*>(base + Lo.b_hi + off) = make_uint2(h0, h1);
                *reinterpret_cast<uint2*>(base + Lo.b_lo + off) = make_uint2(l0, l1);
              }
            }
          }
        }
      }
    }
    float out_scale = 1.f;
    // the staged tiles (bf16, or fp32 split with the predicted scale) to the
    // tensor cores' proxy before the barrier that ends the staging
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (!BF) {
      // the step's dG_h scale (its largest magnitude just below 2^14); the
      // tiles split with the predicted scale stand when that maps the largest
      // magnitude into [2^4, 2^15) (no fp16 overflow, at most 9 binades of
      // precision headroom given up), else the slice is split again
      for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
      if (lane == 0) s_red[warp] = lmax;
      __syncthreads();
      bool keep = true;
      if (have) {
        float hm = 0.f;
        for (int w = 0; w < kBWarps; ++w) hm = fmaxf(hm, s_red[w]);
        int eh = 0;
        if (hm > 0.f) (void)frexpf(hm, &eh);
        eh = min(max(14 - eh, -100), 100);
        keep = pred_ok && pred_eh >= eh - 9 && pred_eh <= eh + 1;
        out_scale = ldexpf(1.f, -(ew + (keep ? pred_eh : eh)));
        // the next step's prediction: three binades of room for growth
        pred_eh = eh - 3;
        pred_scale = ldexpf(1.f, pred_eh);
        pred_ok = true;
        if (!keep) {
          const float h_scale = ldexpf(1.f, eh);
          for (int idx = tid; idx < N * KCu * 8; idx += kBThreads) {
            const int c = idx & 7, at = (idx >> 3) % KCu, n = (idx >> 3) / KCu;
            const float* rp = raw + n * Ks + at * EPA + c * 8;
            const float4 v0 = *reinterpret_cast<const float4*>(rp);
            const float4 v1 = *reinterpret_cast<const float4*>(rp + 4);
            uint4 h4, l4;
            split_f16x2(v0.x * h_scale, v0.y * h_scale, h4.x, l4.x);
            split_f16x2(v0.z * h_scale, v0.w * h_scale, h4.y, l4.y);
            split_f16x2(v1.x * h_scale, v1.y * h_scale, h4.z, l4.z);
            split_f16x2(v1.z * h_scale, v1.w * h_scale, h4.w, l4.w);
            const uint32_t off = (uint32_t)at * atom_bytes + sw_off(n, c);
            *reinterpret_cast<uint4*>(base + Lo.b_hi + off) = h4;
            *reinterpret_cast<uint4*>(base + Lo.b_lo + off) = l4;
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
      }
      // a block-uniform decision: the second barrier only when the slice was
      // split again
      if (have && !keep) __syncthreads();
    } else {
      __syncthreads();
    }
    BTRACE(s, 1);

    // 2. MMA issue: issuer i is lane 0 of warp kBWarps-1-i and runs pass i
    // into accumulator i (pass 0: W_hi g_hi, 1: W_hi g_lo, 2: W_lo g_hi); the
    // padded tail of the last atom multiplies zeros
    if (have) {
      const int iss = kBWarps - 1 - warp;
      if (iss >= 0 && iss < NI) {
        if (lane == 0) {
          const uint32_t dcol = tmem + (uint32_t)(iss * Nm);
          const uint64_t bd0 = b_desc(base_s + ((!BF && iss == 1) ? Lo.b_lo : Lo.b_hi));
          const uint64_t bstep = (uint64_t)(atom_bytes >> 4);
          const uint32_t acol0 = tmem + ((!BF && iss == 2) ? a_lo_col : a_col);
          fence_after();
          mma_pass_n(KCu, dcol, acol0, bd0, bstep, idesc);
          asm volatile(
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                  mbar)
              : "memory");
        }
        __syncwarp();
      }
    }
    BTRACE(s, 6);
    if (pend >= 0) flush(pend);
    pend = -1;
    // pointwise inputs of time t, issued after the polls (whose loads would
    // otherwise queue behind these reads of memory) and consumed after the
    // contraction and the exchange, each by the thread that fetched it (fp32
    // sources by cp.async; bf16 ones are read
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
    bool mma_ok = true;
    if (have) {
      mma_ok = mbar_wait_bounded(mbar, mma_phase, p.status, p.timeout_ns);
      if (!mma_ok) s_mma_bad = 1;
      mma_phase ^= 1u;
    }
    mma_ok = __all_sync(0xffffffffu, mma_ok);
    fence_after();
    BTRACE(s, 2);
    // 3. push each accumulator row (unit u0 + m) to the block that owns the
    // unit: warps 0-3 take columns 0-15, warps 4-7 columns 16-31, ...
    float* recv = recv0 + (size_t)(s & 1) * Pk * Uq * Rs;
    if (!failed && s > 0 && Kc > 0) {
      const int quarter = warp & 3;
      const int m = quarter * 32 + lane;
      const bool row_ok = m < Urc;
      const int owner = row_ok ? m / Uq : 0, uo = m - owner * Uq;
      const bool ok = have && mma_ok;
      const uint32_t lrow = tmem + ((uint32_t)(quarter * 32) << 16);
      for (int c0 = (warp >> 2) * 16; c0 < N; c0 += (kBWarps / 4) * 16) {
        float v[NI][16];
        if (ok) {
          if constexpr (NI == 3) {
            tmem_ld16x3(lrow + (uint32_t)c0, lrow + (uint32_t)(Nm + c0),
                        lrow + (uint32_t)(2 * Nm + c0), v[0], v[1], v[2]);
            // (hi hi + (hi lo + lo hi) 2^-11) / (w_scale g_scale), powers of two
#pragma unroll
            for (int e = 0; e < 16; ++e)
              v[0][e] = fmaf(v[1][e] + v[2][e], 1.f / 2048.f, v[0][e]) * out_scale;
          } else {
            tmem_ld16(lrow + (uint32_t)c0, v[0]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[0][e] = 0.f;
        }
        if (!row_ok || owner >= Pk) continue;
        float* dst = recv + ((size_t)q * Uq + uo) * Rs + c0;
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          if (c0 + i < N)
            st_async4(dst + i, rbar, (unsigned)owner, v[0][i], v[0][i + 1], v[0][i + 2],
                      v[0][i + 3]);
      }
    }
    // 4. the threads with pointwise items wait for this step's partials (the
    // pushes complete the owner's barrier: no cluster barrier)
    bool live = !failed && mma_ok;
    if (live && s > 0 && tid < items) {
      live = mbar_wait_cluster_bounded(rbar, (uint32_t)((s - 1) >> 1) & 1u, p.status,
                                       p.timeout_ns);
      if (!live) s_fail = 1;
    }
    BTRACE(s, 3);
    if (live) {
      cp_async_wait_all();  // this thread's pointwise inputs (it reads only its own)
      for (int it = tid; it < items; it += kBThreads) {
        const int uu = it % Uqc, n = it / Uqc, j = u0 + uq0 + uu;
        float dhf;
        if (s == 0) {
          dhf = a.dhy ? to_f(reinterpret_cast<const T*>(a.dhy)[(int64_t)n * H + j]) : 0.f;
        } else {
          // the partials in rank order (fixed; all loads in flight together),
          // then the GRU's direct term
          const uint32_t rp0 = smem_addr(recv + (size_t)uu * Rs + n);
          float pv[kBMaxPushers];
#pragma unroll
          for (int rank = 0; rank < kBMaxPushers; ++rank)
            pv[rank] = rank < pushers ? ld_shared_f32(rp0 + 4u * (uint32_t)(rank * Uq * Rs)) : 0.f;
          float v = 0.f;
#pragma unroll
          for (int rank = 0; rank < kBMaxPushers; ++rank) v += pv[rank];
          dhf = v + st_carry[it];
        }
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
        // the exchange words of this step's dG_h (value as stored, and the
        // step that reads it: every step below nT, the last one included,
        // has a successor that multiplies it)
        const bool xw = !(blockIdx.x == p.fault_block && s == p.fault_step);
        unsigned long long* xo = a.hx + ((size_t)(s % 3) * N + n) * GH + j;
        const unsigned long long tag = (unsigned long long)(s + 1) << 32;
        float gh[4];
        int ng = 1;
        if (VL && t >= (it == tid ? i_len : __ldg(p.lengths + n))) {
          // a step the forward skipped (past the sequence's length): no gate
          // gradients, dy unused, dh and (LSTM) dc pass straight through
          ng = ngo;
#pragma unroll
          for (int g = 0; g < 4; ++g) gh[g] = 0.f;
          if (p.mode == 2) stash[it] = stash[icap + it] = stash[2 * icap + it] = 0.f;
          st_carry[it] = dhf;
        } else if (p.mode == 1) {  // LSTM: g0..g3 = i, f, g, o
          const float g1 = pin[2 * icap + it], g2 = pin[3 * icap + it], g3 = pin[4 * icap + it];
          const float cc = pin[5 * icap + it], cpv = pin[6 * icap + it];
          const float tc = tanh_fast(cc);
          const float dc = st_dc[it] + dh * g3 * (1.f - tc * tc);
          gh[0] = dc * g2 * g0 * (1.f - g0);
          gh[1] = dc * cpv * g1 * (1.f - g1);
          gh[2] = dc * g0 * (1.f - g2 * g2);
          gh[3] = dh * tc * g3 * (1.f - g3);
          ng = 4;
          st_dc[it] = dc * g1;
          if (VL) st_carry[it] = 0.f;  // a pass-through ends here
        } else if (p.mode == 2) {  // GRU: g0..g3 = r, z, n, W_hn h + b_hn
          const float g1 = pin[2 * icap + it], g2 = pin[3 * icap + it], g3 = pin[4 * icap + it];
          const int sp = rv ? t + 1 : t;
          const float hp = BF ? to_f(hseq[((int64_t)sp * N + n) * H + j]) : pin[6 * icap + it];
          const float dan = dh * (1.f - g1) * (1.f - g2 * g2);
          const float daz = dh * (hp - g2) * g1 * (1.f - g1);
          const float dar = dan * g3 * g0 * (1.f - g0);
          gh[0] = dar;
          gh[1] = daz;
          gh[2] = dan * g0;
          ng = 3;
          stash[it] = dar;
          stash[icap + it] = daz;
          stash[2 * icap + it] = dan;
          st_carry[it] = dh * g1;
        } else {  // tanh RNN: g0 = h_t
          gh[0] = dh * (1.f - g0 * g0);
          if (VL) st_carry[it] = 0.f;
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          if (g >= ng) break;
          const T v = from_f<T>(gh[g]);
          if (xw) st_relaxed_u64(xo + (int64_t)g * H, tag | __float_as_uint(to_f(v)));
          stash[(3 + g) * icap + it] = gh[g];
        }
      }
      if (s < nT) pend = s;
    }
    BTRACE(s, 4);
    BTRACE(s, 5);
    if ((!live || s_mma_bad) && tid == 0) s_fail = 1;
    __syncthreads();
  }
  if (pend >= 0) flush(pend);
  fence_before();
  cl_sync();  // no block leaves while a peer may still store into it
  fence_before();
  __syncthreads();
  if (warp == 0 && !cfg_bad)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols)
                 : "memory");
}

void* bwd_kernel(bool bf, bool varlen) {
  return varlen ? (bf ? (void*)rec_bwd_tc<true, true> : (void*)rec_bwd_tc<false, true>)
                : (bf ? (void*)rec_bwd_tc<true, false> : (void*)rec_bwd_tc<false, false>);
}

}  // namespace

int rec_tc_bwd_capacity(int cluster, size_t smem) {
  void* fn = bwd_kernel(false, false);
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
    const int epc = 64;  // 16-bit elements per 128-byte atom
    const int Kk = (((GH + Pk - 1) / Pk) + 7) / 8 * 8;
    const int Kp = (Kk + epc - 1) / epc * epc;
    if (Kp / epc > kBMaxAtoms) continue;
    const int NI = bf16 ? 1 : 3;
    const int acols = bf16 ? Kp / 2 : Kp;
    int cols = 32;
    while (cols < NI * Nm + acols) cols *= 2;
    if (cols > 512) continue;
    RecPlan pl;
    pl.direct = 0;
    pl.cluster = Pk; pl.Pr = Pr; pl.P = Pr * Pk; pl.Ur = Ur; pl.Uq = Uq;
    pl.Kk = Kk;
    pl.K = Kp;
    pl.KC = Kp / epc;
    pl.nbp = Nm;
    pl.lda = cols;
    pl.Mloc = Ur; pl.Mp = kBM; pl.nb = N;
    pl.tc = 2;
    const BLayout L = b_layout(pl, N, bf16 != 0);
    pl.smem = std::max<size_t>(L.total + 1024, 120 * 1024);
    if (pl.smem > smem_limit) continue;
    if (D * pl.P > num_sms) continue;
    // MMA issue (K slice, passes), the staging of the K slice (its polls:
    // rows of the slice per lane), the push of Ur rows, the owners' reduction
    // over Pk partials and their pointwise items.  Without the staging term
    // the GRU took clusters of 8 (slices of 5 atoms) and staged 60 % slower
    // than with clusters of 16.
    const double cost = (double)Kp * (Nm / 32.0) * 2.0 + (double)Kp * N / 4.0 +
                        (double)Ur * N / 16.0 + (double)Uq * N * (Pk / 4.0 + 8.0);
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
  void* fn = bwd_kernel(p.bf16 != 0, p.lengths != nullptr);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  if (pl.cluster > 8) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  // exchange words from an earlier launch must not look current: tags start at 1
  for (int d = 0; d < p.D; ++d) {
    if (!p.dir[d].hx) return cudaErrorInvalidValue;
    e = cudaMemsetAsync(p.dir[d].hx, 0, rec_tc_xchg_bytes(p.N, p.G * p.H), st);
    if (e != cudaSuccess) return e;
  }
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
