// Persistent recurrent kernels: the serial time loop of one layer (both
// directions of a bidirectional layer in the same launch, on disjoint blocks).
//
// Design (the persistent-RNN idea of the TVM "Persist RNN Implementation"
// thread: recurrent weights stay on chip across time steps, one launch per
// sequence):
//   * every block owns U consecutive hidden units j0 .. j0+U-1 of one
//     direction and keeps, for the whole launch, the slice of W_hh it needs in
//     shared memory:
//       forward : the G*U gate rows of those units (rows ordered g*U + u), so
//                 all gates of a unit land in the same block and the gate
//                 nonlinearities, the cell update and the workspace stores are
//                 fused behind the contraction ("fused point-wise operations"
//                 of the cuDNN optimisation table quoted in Keras issue #3692);
//       backward: the U columns of W_hh (stored transposed), so that
//                 dh_{t-1}[j] = sum_r dG_h[r] W_hh[r][j] is local to the block;
//   * per step each block stages the previous step's broadcast vector (h_{t-1}
//     in forward, dG_h of the previous step in backward; written by all blocks)
//     from L2 into shared memory, contracts it with its resident slice on the
//     CUDA cores (fp32 FMA, register-tiled), applies the fused pointwise math
//     for its units and stores its slice of the next broadcast vector;
//   * blocks of a direction meet at a bounded step barrier (flags in global
//     memory), see common.cuh.
#include <algorithm>

#include "common.cuh"
#include "rec.h"

namespace lr {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

// register-tile shapes: RM x RN outputs per lane, lanes LM (rows) x LN (batch)
// x LK (split of K inside the warp, LK = 32 / (LM*LN))
struct Shape { int RM, RN, LM, LN; };
constexpr Shape kShapes[4] = {{3, 5, 8, 4}, {4, 4, 8, 4}, {3, 5, 2, 4}, {4, 4, 2, 4}};
constexpr int kNumShapes = 4;


// acc[i][j] += sum over this lane's 16-byte K vectors of A[lm + LM*i][k] * B[ln + LN*j][k]
template <typename T, int RM, int RN, int LM, int LN>
__device__ __forceinline__ void warp_tile_fma(float (&acc)[RM][RN], const T* As, int lda,
                                              const T* Bs, int ldb, int v_begin, int v_end,
                                              int lane) {
  constexpr int LK = 32 / (LM * LN);
  constexpr int VK = 16 / (int)sizeof(T);
  const int lm = lane % LM, ln = (lane / LM) % LN, kl = lane / (LM * LN);
  const T* a0 = As + lm * lda;
  const T* b0 = Bs + ln * ldb;
  for (int v = v_begin + kl; v < v_end; v += LK) {
    uint4 av[RM], bv[RN];
#pragma unroll
    for (int i = 0; i < RM; ++i) av[i] = *reinterpret_cast<const uint4*>(a0 + (LM * i) * lda + v * VK);
#pragma unroll
    for (int j = 0; j < RN; ++j) bv[j] = *reinterpret_cast<const uint4*>(b0 + (LN * j) * ldb + v * VK);
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
        for (int j = 0; j < RN; ++j) acc[i][j] = fmaf(af[i], bf[j], acc[i][j]);
    }
  }
}

// copy rows x cols elements (row stride lds) from global into shared (row stride
// ldd); src == nullptr writes zeros.  Uses 16-byte cp.async when `vec` says every
// row start is 16-byte aligned on both sides.
template <typename T>
__device__ __forceinline__ void stage_rows(T* dst, int ldd, const T* src, int64_t lds,
                                           int rows, int cols, bool vec) {
  const int tid = threadIdx.x;
  if (src == nullptr) {
    for (int idx = tid; idx < rows * cols; idx += kThreads) {
      const int r = idx / cols, c = idx - r * cols;
      dst[r * ldd + c] = from_f<T>(0.f);
    }
    return;
  }
  constexpr int VE = 16 / (int)sizeof(T);
  int done = 0;
  if (vec) {
    const int cv = cols / VE;
    for (int idx = tid; idx < rows * cv; idx += kThreads) {
      const int r = idx / cv, c = idx - r * cv;
      cp_async16(dst + r * ldd + c * VE, src + r * lds + c * VE);
    }
    cp_async_commit();
    done = cv * VE;
  }
  const int rest = cols - done;
  if (rest > 0) {
    for (int idx = tid; idx < rows * rest; idx += kThreads) {
      const int r = idx / rest, c = done + (idx - r * rest);
      dst[r * ldd + c] = from_f<T>(ldcg_f(src + r * lds + c));
    }
  }
  if (vec) cp_async_wait_all();
}

// Reduce the per-warp register tiles (intra-warp over the LK lanes, then over
// the WK warps of each tile in a fixed order) into outs[m * nbp + n].
template <int RM, int RN, int LM, int LN>
__device__ __forceinline__ void reduce_tiles(float (&acc)[RM][RN], float* red, float* outs,
                                             const RecPlan& pl, bool active, int warp, int lane) {
  constexpr int TE = RM * RN * LM * LN;
#pragma unroll
  for (int off = LM * LN; off < 32; off <<= 1)
#pragma unroll
    for (int i = 0; i < RM; ++i)
#pragma unroll
      for (int j = 0; j < RN; ++j) acc[i][j] += __shfl_xor_sync(0xffffffffu, acc[i][j], off);
  const int lm = lane % LM, ln = (lane / LM) % LN, kl = lane / (LM * LN);
  if (active && kl == 0) {
    float* r = red + warp * TE;
#pragma unroll
    for (int i = 0; i < RM; ++i)
#pragma unroll
      for (int j = 0; j < RN; ++j) r[(i * RN + j) * (LM * LN) + ln * LM + lm] = acc[i][j];
  }
  __syncthreads();
  const int ntile = pl.tiles_m * pl.tiles_n;
  for (int idx = threadIdx.x; idx < ntile * TE; idx += kThreads) {
    const int tl = idx / TE, e = idx - tl * TE;
    float sum = 0.f;
    for (int w = 0; w < pl.WK; ++w) sum += red[(tl * pl.WK + w) * TE + e];
    const int ij = e / (LM * LN), lp = e - ij * (LM * LN);
    const int i = ij / RN, j = ij - i * RN;
    const int m = (tl / pl.tiles_n) * (LM * RM) + (lp % LM) + LM * i;
    const int n = (tl % pl.tiles_n) * (LN * RN) + (lp / LM) + LN * j;
    outs[m * pl.nbp + n] = sum;
  }
  __syncthreads();
}

struct Smem {
  void* A; void* B; float* red; float* outs; float* st0; float* st1;
};

template <typename T, int RM, int RN, int LM, int LN>
__device__ __forceinline__ Smem carve(unsigned char* smem, const RecPlan& pl, int N) {
  Smem s;
  T* A = reinterpret_cast<T*>(smem);
  T* B = A + (size_t)pl.Mp * pl.lda;
  s.A = A;
  s.B = B;
  s.red = reinterpret_cast<float*>(B + (size_t)pl.nbp * pl.ldb);
  s.outs = s.red + kWarps * RM * RN * LM * LN;
  s.st0 = s.outs + (size_t)pl.Mp * pl.nbp;
  s.st1 = s.st0 + (size_t)pl.U * N;
  return s;
}

// One batch chunk of the per-step contraction: outs[m][n] = sum_k A[m][k] B[n][k]
// with B[n][k] = src[(n0 + n) * lds + k] (src == nullptr: zeros), k over
// [kb, ke) (the whole K by default).
template <typename T, int RM, int RN, int LM, int LN>
__device__ __forceinline__ void step_contract(const Smem& sm, const RecPlan& pl, const T* src,
                                              int64_t lds, int nbc, bool vec, int kb = 0,
                                              int ke = -1) {
  if (ke < 0) ke = pl.K;
  constexpr int VK = 16 / (int)sizeof(T);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ntile = pl.tiles_m * pl.tiles_n;
  const int tile = warp / pl.WK, wk = warp - tile * pl.WK;
  const bool active = tile < ntile;
  const int tm = active ? tile / pl.tiles_n : 0, tn = active ? tile % pl.tiles_n : 0;
  const T* As = reinterpret_cast<const T*>(sm.A);
  T* Bs = reinterpret_cast<T*>(sm.B);
  float acc[RM][RN];
#pragma unroll
  for (int i = 0; i < RM; ++i)
#pragma unroll
    for (int j = 0; j < RN; ++j) acc[i][j] = 0.f;
  for (int k0 = kb; k0 < ke; k0 += pl.KC) {
    const int kc = min(pl.KC, ke - k0);
    stage_rows<T>(Bs, pl.ldb, src ? src + k0 : nullptr, lds, nbc, kc, vec);
    __syncthreads();
    if (active) {
      const int nv = (kc + VK - 1) / VK;
      const int vb = (wk * nv) / pl.WK, ve = ((wk + 1) * nv) / pl.WK;
      warp_tile_fma<T, RM, RN, LM, LN>(acc, As + (size_t)(tm * LM * RM) * pl.lda + k0, pl.lda,
                                       Bs + (size_t)(tn * LN * RN) * pl.ldb, pl.ldb, vb, ve, lane);
    }
    __syncthreads();
  }
  reduce_tiles<RM, RN, LM, LN>(acc, sm.red, sm.outs, pl, active, warp, lane);
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
template <typename T, int RM, int RN, int LM, int LN>
__global__ void __launch_bounds__(kThreads, 1) rec_fwd_kernel(const __grid_constant__ RecParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const RecPlan& pl = p.plan;
  const int d = blockIdx.x / pl.P;
  const int blk = blockIdx.x - d * pl.P;
  const RecDirArgs& a = p.dir[d];
  const int H = p.H, N = p.N, nT = p.T, G = p.G, U = pl.U;
  const int j0 = blk * U;
  const int Uc = min(U, H - j0);
  const int tid = threadIdx.x;
  const Smem sm = carve<T, RM, RN, LM, LN>(smem, pl, N);
  T* As = reinterpret_cast<T*>(sm.A);
  float* hown = sm.st0;   // [U][N] fp32 hidden state of the own units
  float* cst = sm.st1;    // [U][N] fp32 cell state (LSTM)

  if (ld_volatile_int(p.status) != kDevOk) return;

  // resident slice: row g*U + u <- W_hh[g*H + j0 + u][:]; zero padding
  const T* W = reinterpret_cast<const T*>(a.whh);
  for (int64_t idx = tid; idx < (int64_t)pl.Mp * pl.lda; idx += kThreads) {
    const int r = (int)(idx / pl.lda), k = (int)(idx - (int64_t)r * pl.lda);
    const int g = r / U, u = r - g * U;
    As[idx] = (g < G && u < Uc && k < H) ? W[(int64_t)(g * H + j0 + u) * H + k] : from_f<T>(0.f);
  }
  T* Bs = reinterpret_cast<T*>(sm.B);
  for (int idx = tid; idx < pl.nbp * pl.ldb; idx += kThreads) Bs[idx] = from_f<T>(0.f);
  const int slot0 = d ? nT : 0;
  for (int idx = tid; idx < U * N; idx += kThreads) {
    const int u = idx / N, n = idx - u * N;
    float hv = 0.f, cv = 0.f;
    if (u < Uc) {
      const int64_t o = (int64_t)n * H + j0 + u;
      if (a.h0) hv = to_f(reinterpret_cast<const T*>(a.h0)[o]);
      if (a.c0) cv = a.c0[o];
      if (a.hseq) reinterpret_cast<T*>(a.hseq)[(int64_t)slot0 * N * H + o] = from_f<T>(hv);
      if (a.cseq) a.cseq[(int64_t)slot0 * N * H + o] = cv;
    }
    hown[idx] = hv;
    cst[idx] = cv;
  }
  __syncthreads();

  const bool vec = ((H * (int)sizeof(T)) % 16 == 0) && ((p.ldy * (int64_t)sizeof(T)) % 16 == 0);
  const T* bhh = reinterpret_cast<const T*>(a.bhh);
  T* y = reinterpret_cast<T*>(a.y);
  T* hseq = reinterpret_cast<T*>(a.hseq);
  const int64_t GH = (int64_t)G * H;
  const int* lens = p.lengths;  // variable lengths: the host also passes hseq

  for (int s = 0; s < nT; ++s) {
    const int t = d ? nT - 1 - s : s;
    const int tp = d ? t + 1 : t - 1;
    const T* src;
    int64_t lds;
    if (s == 0) {
      src = reinterpret_cast<const T*>(a.h0);
      lds = H;
    } else if (lens) {
      // y is zero past a sequence's length; the state it carries is in hseq
      // (slot of the state after time tp)
      src = hseq + (int64_t)(d ? t + 1 : t) * N * H;
      lds = H;
    } else {
      src = y + (int64_t)tp * N * p.ldy + (int64_t)d * H;
      lds = p.ldy;
    }
    const int slot = d ? t : t + 1;
    if (p.mode == 3) {
      // TensorFlow-flavour GRU ("rnn training example?", the TensorFlow GRU
      // equations: n = tanh(W_in x + b_in + W_hn (r * h) + b_hn)).  Phase 1:
      // r and z from h_{t-1}, and r * h_{t-1} of the own units into the
      // direction's exchange buffer; a barrier over the direction's blocks;
      // phase 2: W_hn (r * h_{t-1}) for the own units, the candidate and the
      // new state.  b_hn is folded into G_x (it is outside the product).
      T* rh = reinterpret_cast<T*>(a.xbuf);
      for (int n0 = 0; n0 < N; n0 += pl.nb) {
        const int nbc = min(pl.nb, N - n0);
        step_contract<T, RM, RN, LM, LN>(sm, pl, src ? src + (int64_t)n0 * lds : nullptr, lds,
                                         nbc, vec);
        const float* outs = sm.outs;
        for (int idx = tid; idx < Uc * nbc; idx += kThreads) {
          const int u = idx % Uc, nn = idx / Uc, n = n0 + nn, j = j0 + u;
          const int64_t row = (int64_t)t * N + n;
          const float* gxr = a.gx + row * GH + j;
          const float r = sigmoidf_(__ldg(gxr) + outs[(0 * U + u) * pl.nbp + nn]);
          const float z = sigmoidf_(__ldg(gxr + H) + outs[(1 * U + u) * pl.nbp + nn]);
          const T rhv = from_f<T>(r * hown[u * N + n]);
          rh[(int64_t)n * H + j] = rhv;
          cst[u * N + n] = z;  // kept for phase 2 (the GRU has no cell state)
          if (a.gates) {
            float* gp = a.gates + row * 4 * H + j;
            gp[0] = r; gp[H] = z; gp[3 * H] = to_f(rhv);
          }
        }
        __syncthreads();
      }
      if (!step_barrier(p.flags + (size_t)d * pl.P * p.flag_stride, p.flag_stride, pl.P, blk,
                        (unsigned)(2 * s + 1), p.status, p.timeout_ns, p.spin_ns, false))
        return;
      const bool vrh = (H * (int)sizeof(T)) % 16 == 0;
      for (int n0 = 0; n0 < N; n0 += pl.nb) {
        const int nbc = min(pl.nb, N - n0);
        step_contract<T, RM, RN, LM, LN>(sm, pl, rh + (int64_t)n0 * H, H, nbc, vrh);
        const float* outs = sm.outs;
        for (int idx = tid; idx < Uc * nbc; idx += kThreads) {
          const int u = idx % Uc, nn = idx / Uc, n = n0 + nn, j = j0 + u;
          const int64_t row = (int64_t)t * N + n;
          const bool act = !lens || t < __ldg(lens + n);
          const float z = cst[u * N + n];
          const float nv = tanhf(__ldg(a.gx + row * GH + 2 * H + j) + outs[(2 * U + u) * pl.nbp + nn]);
          float h = (1.f - z) * nv + z * hown[u * N + n];
          if (a.gates) a.gates[row * 4 * H + 2 * H + j] = nv;
          if (!act) h = hown[u * N + n];
          hown[u * N + n] = h;
          y[row * p.ldy + (int64_t)d * H + j] = from_f<T>(act ? h : 0.f);
          if (hseq) hseq[((int64_t)slot * N + n) * H + j] = from_f<T>(h);
        }
        __syncthreads();
      }
      if (s + 1 < nT) {
        const bool skip = (blockIdx.x == p.fault_block) && (s == p.fault_step);
        if (!step_barrier(p.flags + (size_t)d * pl.P * p.flag_stride, p.flag_stride, pl.P, blk,
                          (unsigned)(2 * s + 2), p.status, p.timeout_ns, p.spin_ns, skip))
          return;
      }
      continue;
    }
    for (int n0 = 0; n0 < N; n0 += pl.nb) {
      const int nbc = min(pl.nb, N - n0);
      step_contract<T, RM, RN, LM, LN>(sm, pl, src ? src + (int64_t)n0 * lds : nullptr, lds, nbc,
                                       vec);
      const float* outs = sm.outs;
      for (int idx = tid; idx < Uc * nbc; idx += kThreads) {
        const int u = idx % Uc, nn = idx / Uc, n = n0 + nn, j = j0 + u;
        const int64_t row = (int64_t)t * N + n;
        const float* gxr = a.gx + row * GH + j;
        // past the sequence's length the step keeps the state and outputs zero
        const bool act = !lens || t < __ldg(lens + n);
        float h;
        if (p.mode == 1) {  // LSTM, gate blocks i, f, g, o
          const float ig = sigmoidf_(__ldg(gxr) + outs[(0 * U + u) * pl.nbp + nn]);
          const float fg = sigmoidf_(__ldg(gxr + H) + outs[(1 * U + u) * pl.nbp + nn]);
          const float gg = tanhf(__ldg(gxr + 2 * H) + outs[(2 * U + u) * pl.nbp + nn]);
          const float og = sigmoidf_(__ldg(gxr + 3 * H) + outs[(3 * U + u) * pl.nbp + nn]);
          const float c = fg * cst[u * N + n] + ig * gg;
          h = og * tanhf(c);
          if (act) cst[u * N + n] = c;
          if (a.gates) {
            float* gp = a.gates + row * 4 * H + j;
            gp[0] = ig; gp[H] = fg; gp[2 * H] = gg; gp[3 * H] = og;
          }
          if (a.cseq) a.cseq[((int64_t)slot * N + n) * H + j] = cst[u * N + n];
        } else if (p.mode == 2) {  // GRU, gate blocks r, z, n
          const float ghn = outs[(2 * U + u) * pl.nbp + nn] + to_f(bhh[2 * H + j]);
          const float r = sigmoidf_(__ldg(gxr) + outs[(0 * U + u) * pl.nbp + nn]);
          const float z = sigmoidf_(__ldg(gxr + H) + outs[(1 * U + u) * pl.nbp + nn]);
          const float nv = tanhf(__ldg(gxr + 2 * H) + r * ghn);
          h = (1.f - z) * nv + z * hown[u * N + n];
          if (a.gates) {
            float* gp = a.gates + row * 4 * H + j;
            gp[0] = r; gp[H] = z; gp[2 * H] = nv; gp[3 * H] = ghn;
          }
        } else {  // tanh RNN
          h = tanhf(__ldg(gxr) + outs[u * pl.nbp + nn]);
          if (a.gates) a.gates[row * H + j] = h;
        }
        if (!act) h = hown[u * N + n];
        hown[u * N + n] = h;
        y[row * p.ldy + (int64_t)d * H + j] = from_f<T>(act ? h : 0.f);
        if (hseq) hseq[((int64_t)slot * N + n) * H + j] = from_f<T>(h);
      }
      __syncthreads();
    }
    if (s + 1 < nT) {
      const bool skip = (blockIdx.x == p.fault_block) && (s == p.fault_step);
      if (!step_barrier(p.flags + (size_t)d * pl.P * p.flag_stride, p.flag_stride, pl.P, blk,
                        (unsigned)(s + 1), p.status, p.timeout_ns, p.spin_ns, skip))
        return;
    }
  }
  for (int idx = tid; idx < Uc * N; idx += kThreads) {
    const int u = idx % Uc, n = idx / Uc;
    const int64_t o = (int64_t)n * H + j0 + u;
    if (a.hy) reinterpret_cast<T*>(a.hy)[o] = from_f<T>(hown[u * N + n]);
    if (a.cy) a.cy[o] = cst[u * N + n];
  }
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------
template <typename T, int RM, int RN, int LM, int LN>
__global__ void __launch_bounds__(kThreads, 1) rec_bwd_kernel(const __grid_constant__ RecParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const RecPlan& pl = p.plan;
  const int d = blockIdx.x / pl.P;
  const int blk = blockIdx.x - d * pl.P;
  const RecDirArgs& a = p.dir[d];
  const int H = p.H, N = p.N, nT = p.T, G = p.G, U = pl.U;
  const int j0 = blk * U;
  const int Uc = min(U, H - j0);
  const int tid = threadIdx.x;
  const Smem sm = carve<T, RM, RN, LM, LN>(smem, pl, N);
  T* As = reinterpret_cast<T*>(sm.A);
  float* dcs = sm.st0;    // [U][N] dc carried to the previous step (LSTM)
  float* carry = sm.st1;  // [U][N] dh * z carried to the previous step (GRU)

  if (ld_volatile_int(p.status) != kDevOk) return;

  const int64_t GH = (int64_t)G * H;
  // resident slice, transposed: A[u][r] = W_hh[r][j0 + u]; consecutive threads
  // read consecutive units of one row
  const T* W = reinterpret_cast<const T*>(a.whh);
  for (int64_t idx = tid; idx < (int64_t)pl.Mp * pl.lda; idx += kThreads) {
    const int r = (int)(idx / pl.Mp), u = (int)(idx - (int64_t)r * pl.Mp);
    As[(int64_t)u * pl.lda + r] = (u < Uc && r < GH) ? W[(int64_t)r * H + j0 + u] : from_f<T>(0.f);
  }
  T* Bs = reinterpret_cast<T*>(sm.B);
  for (int idx = tid; idx < pl.nbp * pl.ldb; idx += kThreads) Bs[idx] = from_f<T>(0.f);
  for (int idx = tid; idx < U * N; idx += kThreads) {
    const int u = idx / N, n = idx - u * N;
    float dc = 0.f;
    if (u < Uc && a.dcy) dc = a.dcy[(int64_t)n * H + j0 + u];
    dcs[idx] = dc;
    carry[idx] = 0.f;
  }
  __syncthreads();

  const bool vec = ((GH * (int64_t)sizeof(T)) % 16 == 0);
  T* dgx = reinterpret_cast<T*>(a.dgx);
  T* dgh = reinterpret_cast<T*>(a.dgh);
  const T* hseq = reinterpret_cast<const T*>(a.hseq);
  const int* lens = p.lengths;

  const bool tf = p.mode == 3;
  T* xb = reinterpret_cast<T*>(a.xbuf);  // TF-flavour GRU: [N][G*H] exchange rows

  for (int s = 0; s <= nT; ++s) {
    const int t = d ? s : nT - 1 - s;        // time processed at this step (s < T)
    const int tp = d ? s - 1 : nT - s;       // time processed at the previous step (s > 0)
    if (s > 0) {
      const bool skip = (blockIdx.x == p.fault_block) && (s - 1 == p.fault_step);
      if (!step_barrier(p.flags + (size_t)d * pl.P * p.flag_stride, p.flag_stride, pl.P, blk,
                        (unsigned)(tf ? 2 * s : s), p.status, p.timeout_ns, p.spin_ns, skip))
        return;
    }
    if (tf) {
      // TensorFlow-flavour GRU, reverse mode through n = tanh(a_n + W_hn (r*h)):
      //   dh_{t-1} = dh z + r * W_hn^T da_n + W_hr^T da_r + W_hz^T da_z,
      //   da_r = (W_hn^T da_n) * h_{t-1} * r (1 - r).
      // Part A: dh from the previous step's W_hr^T da_r + W_hz^T da_z (K rows
      // 0 .. 2H of the exchange rows) and the carried dh z + r * W_hn^T da_n;
      // da_n, da_z of the own units out; barrier; part B: W_hn^T da_n (K rows
      // 2H .. 3H), da_r out.
      for (int n0 = 0; n0 < N; n0 += pl.nb) {
        const int nbc = min(pl.nb, N - n0);
        if (s > 0)
          step_contract<T, RM, RN, LM, LN>(sm, pl, xb + (int64_t)n0 * GH, GH, nbc, vec, 0, 2 * H);
        const float* outs = sm.outs;
        for (int idx = tid; idx < Uc * nbc; idx += kThreads) {
          const int u = idx % Uc, nn = idx / Uc, n = n0 + nn, j = j0 + u;
          float dhf;
          if (s == 0)
            dhf = a.dhy ? to_f(reinterpret_cast<const T*>(a.dhy)[(int64_t)n * H + j]) : 0.f;
          else
            dhf = outs[u * pl.nbp + nn] + carry[u * N + n];
          if (s == nT) {
            if (a.dh0) reinterpret_cast<T*>(a.dh0)[(int64_t)n * H + j] = from_f<T>(dhf);
            continue;
          }
          const int64_t row = (int64_t)t * N + n;
          T* gxo = dgx + row * GH + j;
          if (lens && t >= __ldg(lens + n)) {
            // a step the forward skipped: no gate gradients, dh passes through
            gxo[H] = from_f<T>(0.f);
            gxo[2 * H] = from_f<T>(0.f);
            xb[(int64_t)n * GH + 2 * H + j] = from_f<T>(0.f);
            dcs[u * N + n] = 0.f;
            carry[u * N + n] = dhf;
            continue;
          }
          const float dh = load_any(a.dy, row * p.lddy + (int64_t)d * H + j, a.dy_bf16) + dhf;
          const float* gp = a.gates + row * 4 * H + j;
          const float z = gp[H], nv = gp[2 * H];
          const float hp = to_f(hseq[((int64_t)(d ? t + 1 : t) * N + n) * H + j]);
          const float dan = dh * (1.f - z) * (1.f - nv * nv);
          const float daz = dh * (hp - nv) * z * (1.f - z);
          const T dant = from_f<T>(dan);
          gxo[H] = from_f<T>(daz);
          gxo[2 * H] = dant;
          xb[(int64_t)n * GH + 2 * H + j] = dant;
          dcs[u * N + n] = daz;          // for part B (no cell state in a GRU)
          carry[u * N + n] = dh * z;     // part B adds r * W_hn^T da_n
        }
        __syncthreads();
      }
      if (s == nT) continue;
      if (!step_barrier(p.flags + (size_t)d * pl.P * p.flag_stride, p.flag_stride, pl.P, blk,
                        (unsigned)(2 * s + 1), p.status, p.timeout_ns, p.spin_ns, false))
        return;
      for (int n0 = 0; n0 < N; n0 += pl.nb) {
        const int nbc = min(pl.nb, N - n0);
        step_contract<T, RM, RN, LM, LN>(sm, pl, xb + (int64_t)n0 * GH, GH, nbc, vec, 2 * H,
                                         3 * H);
        const float* outs = sm.outs;
        for (int idx = tid; idx < Uc * nbc; idx += kThreads) {
          const int u = idx % Uc, nn = idx / Uc, n = n0 + nn, j = j0 + u;
          const int64_t row = (int64_t)t * N + n;
          T* gxo = dgx + row * GH + j;
          T* xr = xb + (int64_t)n * GH + j;
          if (lens && t >= __ldg(lens + n)) {
            gxo[0] = from_f<T>(0.f);
            xr[0] = from_f<T>(0.f);
            xr[H] = from_f<T>(0.f);
            continue;
          }
          const float drh = outs[u * pl.nbp + nn];
          const float r = a.gates[row * 4 * H + j];
          const float hp = to_f(hseq[((int64_t)(d ? t + 1 : t) * N + n) * H + j]);
          const float dar = drh * hp * r * (1.f - r);
          const T dart = from_f<T>(dar);
          gxo[0] = dart;
          xr[0] = dart;
          xr[H] = from_f<T>(dcs[u * N + n]);
          carry[u * N + n] += r * drh;
        }
        __syncthreads();
      }
      continue;
    }
    for (int n0 = 0; n0 < N; n0 += pl.nb) {
      const int nbc = min(pl.nb, N - n0);
      if (s > 0)
        step_contract<T, RM, RN, LM, LN>(sm, pl, dgh + ((int64_t)tp * N + n0) * GH, GH, nbc, vec);
      const float* outs = sm.outs;
      for (int idx = tid; idx < Uc * nbc; idx += kThreads) {
        const int u = idx % Uc, nn = idx / Uc, n = n0 + nn, j = j0 + u;
        // gradient arriving at h_t from the later steps (or from hy)
        float dhf;
        if (s == 0)
          dhf = a.dhy ? to_f(reinterpret_cast<const T*>(a.dhy)[(int64_t)n * H + j]) : 0.f;
        else
          dhf = outs[u * pl.nbp + nn] + carry[u * N + n];
        if (s == nT) {
          if (a.dh0) reinterpret_cast<T*>(a.dh0)[(int64_t)n * H + j] = from_f<T>(dhf);
          if (a.dc0) a.dc0[(int64_t)n * H + j] = dcs[u * N + n];
          continue;
        }
        const int64_t row = (int64_t)t * N + n;
        T* gxo = dgx + row * GH + j;
        if (lens && t >= __ldg(lens + n)) {
          // the forward kept the state at this step: no gate gradients, and
          // the state gradients (dh here, dc in dcs) pass straight through
          for (int g = 0; g < G; ++g) gxo[(int64_t)g * H] = from_f<T>(0.f);
          if (p.mode == 2) {
            T* gho = dgh + row * GH + j;
            for (int g = 0; g < G; ++g) gho[(int64_t)g * H] = from_f<T>(0.f);
          }
          carry[u * N + n] = dhf;
          continue;
        }
        const float dh = load_any(a.dy, row * p.lddy + (int64_t)d * H + j, a.dy_bf16) + dhf;
        if (p.mode == 1) {  // LSTM
          const float* gp = a.gates + row * 4 * H + j;
          const float ig = gp[0], fg = gp[H], gg = gp[2 * H], og = gp[3 * H];
          const int sc = d ? t : t + 1, sp = d ? t + 1 : t;
          const float c = a.cseq[((int64_t)sc * N + n) * H + j];
          const float cp = a.cseq[((int64_t)sp * N + n) * H + j];
          const float tc = tanhf(c);
          const float dout = dh * tc;
          const float dc = dcs[u * N + n] + dh * og * (1.f - tc * tc);
          gxo[0] = from_f<T>(dc * gg * ig * (1.f - ig));
          gxo[H] = from_f<T>(dc * cp * fg * (1.f - fg));
          gxo[2 * H] = from_f<T>(dc * ig * (1.f - gg * gg));
          gxo[3 * H] = from_f<T>(dout * og * (1.f - og));
          dcs[u * N + n] = dc * fg;
          if (lens) carry[u * N + n] = 0.f;
        } else if (p.mode == 2) {  // GRU
          const float* gp = a.gates + row * 4 * H + j;
          const float r = gp[0], z = gp[H], nv = gp[2 * H], ghn = gp[3 * H];
          const int sp = d ? t + 1 : t;
          const float hp = to_f(hseq[((int64_t)sp * N + n) * H + j]);
          const float dan = dh * (1.f - z) * (1.f - nv * nv);
          const float daz = dh * (hp - nv) * z * (1.f - z);
          const float dar = dan * ghn * r * (1.f - r);
          gxo[0] = from_f<T>(dar);
          gxo[H] = from_f<T>(daz);
          gxo[2 * H] = from_f<T>(dan);
          T* gho = dgh + row * GH + j;
          gho[0] = from_f<T>(dar);
          gho[H] = from_f<T>(daz);
          gho[2 * H] = from_f<T>(dan * r);
          carry[u * N + n] = dh * z;
        } else {  // tanh RNN
          const float hv = a.gates[row * H + j];
          gxo[0] = from_f<T>(dh * (1.f - hv * hv));
          if (lens) carry[u * N + n] = 0.f;
        }
      }
      __syncthreads();
    }
  }
}

// ---------------------------------------------------------------------------
// direct path (one batch chunk, N <= LN*RN, and at most one pointwise item --
// one (unit, sequence) pair -- per thread).  No block-wide staging: every warp
// owns a contiguous slice of K, waits only for the blocks that produce that
// slice of the previous step's broadcast vector, reads it straight from L2
// with 16-byte loads and contracts it with the resident rows of all tiles.
// Per-item state (h, c, dc, carry) stays in registers, and the pointwise
// inputs of the next step (G_x, or dy and the saved activations) are loaded
// into registers one step ahead, hiding their latency behind the contraction.
// ---------------------------------------------------------------------------
constexpr int kMaxTilesM = 3;

// Optional step trace (build with -DLAYER_RNN_TRACE): thread 0 of a few blocks
// stamps %globaltimer at the phase boundaries of every step, and
// rnn_debug_trace_copy() copies the stamps out.  Off in normal builds.
#ifdef LAYER_RNN_TRACE
constexpr int kTraceBlocks = 4, kTraceSteps = 1024, kTraceMarks = 8;
__device__ unsigned long long g_trace[4][1024][8];
__device__ __forceinline__ void trace_mark(int s, int k, int nblk) {
  const int b = blockIdx.x == 0 ? 0 : blockIdx.x == nblk / 3 ? 1 : blockIdx.x == (2 * nblk) / 3 ? 2
              : blockIdx.x == nblk - 1 ? 3 : -1;
  if (b >= 0 && threadIdx.x == 0 && s < kTraceSteps) g_trace[b][s][k] = globaltimer_ns();
}
#define TRACE(s, k) trace_mark((s), (k), pl.P)
#else
#define TRACE(s, k) ((void)0)
#endif

// Per-warp contraction over this warp's K vectors [vb, ve):
//   acc[tm][i][j] += sum_k A[tm*LM*RM + lm + LM*i][k] * B[ln + LN*j][k]
// A is resident in shared memory; B rows (row stride ldb elements, nrows of
// them) are streamed from L2 into the warp's own double-buffered staging area
// with 16-byte cp.async, `chv` vectors per chunk, so that a whole chunk is in
// flight at once and the next chunk loads while this one is computed.
template <typename T, int RM, int RN, int LM, int LN>
__device__ __forceinline__ void warp_direct_contract(float (&acc)[kMaxTilesM][RM][RN], int tiles_m,
                                                     const T* As, int lda, const T* B, int64_t ldb,
                                                     int nrows, int vb, int ve, int lane,
                                                     uint4* wbuf, int chv, int wstride, int nst,
                                                     int trace_s, int trace_nblk) {
  (void)trace_s;
  (void)trace_nblk;
  constexpr int LK = 32 / (LM * LN);
  constexpr int VK = 16 / (int)sizeof(T);
  constexpr int NR = LN * RN;
  const int lm = lane % LM, ln = (lane / LM) % LN, kl = lane / (LM * LN);
  const int nchunks = (ve - vb + chv - 1) / chv;
  auto issue = [&](int c) {
    const int v0 = vb + c * chv, nv = min(chv, ve - v0);
    uint4* dst = wbuf + (c % nst) * NR * wstride;
    for (int idx = lane; idx < nrows * nv; idx += 32) {
      const int r = idx / nv, q = idx - r * nv;
      cp_async16(dst + r * wstride + q, B + r * ldb + (int64_t)(v0 + q) * VK);
    }
    cp_async_commit();
  };
  issue(0);
  for (int c = 0; c < nchunks; ++c) {
    if (c + 1 < nchunks && nst > 1) {
      issue(c + 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncwarp();
#ifdef LAYER_RNN_TRACE
    if (c == 0) trace_mark(trace_s, 6, trace_nblk);
#endif
    const int v0 = vb + c * chv, nv = min(chv, ve - v0);
    const uint4* bs = wbuf + (c % nst) * NR * wstride;
    const T* arow = As + lm * lda + v0 * VK;
    for (int q = kl; q < nv; q += LK) {
      uint4 bv[RN];
#pragma unroll
      for (int j = 0; j < RN; ++j) {
        const int r = ln + LN * j;
        bv[j] = r < nrows ? bs[r * wstride + q] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int tm = 0; tm < kMaxTilesM; ++tm) {
        if (tm < tiles_m) {
          uint4 av[RM];
#pragma unroll
          for (int i = 0; i < RM; ++i)
            av[i] = *reinterpret_cast<const uint4*>(arow + (tm * LM * RM + LM * i) * lda + q * VK);
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
              for (int j = 0; j < RN; ++j) acc[tm][i][j] = fmaf(af[i], bf[j], acc[tm][i][j]);
          }
        }
      }
    }
    __syncwarp();  // the stage is refilled by a later chunk
    if (nst == 1 && c + 1 < nchunks) issue(c + 1);
  }
}

// intra-warp reduction over the LK lanes, warp partials to red[warp][tm][TE],
// block sync, fixed-order sum over the warps into outs[m * nbp + n], block sync.
// Returns false (uniformly) when some warp recorded a failed wait in *fail.
template <int RM, int RN, int LM, int LN>
__device__ __forceinline__ bool direct_reduce(float (&acc)[kMaxTilesM][RM][RN], int tiles_m,
                                              uint4* wall, int wslot, float* outs, int nbp,
                                              int lane, int warp, volatile int* fail) {
  constexpr int TE = RM * RN * LM * LN;
#pragma unroll
  for (int tm = 0; tm < kMaxTilesM; ++tm)
#pragma unroll
    for (int off = LM * LN; off < 32; off <<= 1)
#pragma unroll
      for (int i = 0; i < RM; ++i)
#pragma unroll
        for (int j = 0; j < RN; ++j) acc[tm][i][j] += __shfl_xor_sync(0xffffffffu, acc[tm][i][j], off);
  const int lm = lane % LM, ln = (lane / LM) % LN, kl = lane / (LM * LN);
  if (kl == 0) {
#pragma unroll
    for (int tm = 0; tm < kMaxTilesM; ++tm) {
      if (tm < tiles_m) {
        float* r = reinterpret_cast<float*>(wall + (size_t)warp * wslot) + tm * TE;
#pragma unroll
        for (int i = 0; i < RM; ++i)
#pragma unroll
          for (int j = 0; j < RN; ++j) r[(i * RN + j) * (LM * LN) + ln * LM + lm] = acc[tm][i][j];
      }
    }
  }
  __syncthreads();
  if (*fail) return false;
  for (int idx = threadIdx.x; idx < tiles_m * TE; idx += kThreads) {
    const int tm = idx / TE, e = idx - tm * TE;
    float sum = 0.f;
#pragma unroll 4
    for (int w = 0; w < kWarps; ++w)
      sum += reinterpret_cast<const float*>(wall + (size_t)w * wslot)[tm * TE + e];
    const int ij = e / (LM * LN), lp = e - ij * (LM * LN);
    const int i = ij / RN, j = ij - i * RN;
    const int m = tm * (LM * RM) + (lp % LM) + LM * i;
    const int n = (lp / LM) + LN * j;
    outs[m * nbp + n] = sum;
  }
  __syncthreads();
  return true;
}

template <typename T, int RM, int RN, int LM, int LN>
__global__ void __launch_bounds__(kThreads, 1)
    rec_fwd_direct(const __grid_constant__ RecParams p) {
  constexpr int VK = 16 / (int)sizeof(T);
  constexpr int TE = RM * RN * LM * LN;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_fail;
  const RecPlan& pl = p.plan;
  const int d = blockIdx.x / pl.P;
  const int blk = blockIdx.x - d * pl.P;
  const RecDirArgs& a = p.dir[d];
  const int H = p.H, N = p.N, nT = p.T, G = p.G, U = pl.U;
  const int j0 = blk * U;
  const int Uc = min(U, H - j0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  T* As = reinterpret_cast<T*>(smem);
  float* outs = reinterpret_cast<float*>(As + (size_t)pl.Mp * pl.lda);
  // per-warp slots: staging stages during the contraction, then the warp's
  // partial tiles for the cross-warp reduction
  uint4* wall = reinterpret_cast<uint4*>(outs + pl.Mp * pl.nbp);
  const int wslot = max(pl.nst * (LN * RN) * pl.ldb, (pl.tiles_m * TE * 4 + 15) / 16);
  uint4* wbuf = wall + (size_t)warp * wslot;

  if (ld_volatile_int(p.status) != kDevOk) return;
  if (tid == 0) s_fail = 0;
  const T* W = reinterpret_cast<const T*>(a.whh);
  for (int64_t idx = tid; idx < (int64_t)pl.Mp * pl.lda; idx += kThreads) {
    const int r = (int)(idx / pl.lda), k = (int)(idx - (int64_t)r * pl.lda);
    const int g = r / U, u = r - g * U;
    As[idx] = (g < G && u < Uc && k < H) ? W[(int64_t)(g * H + j0 + u) * H + k] : from_f<T>(0.f);
  }

  // the (unit, sequence) item of this thread
  const bool item = tid < Uc * N;
  const int u = item ? tid % Uc : 0, n = item ? tid / Uc : 0, j = j0 + u;
  const int64_t GH = (int64_t)G * H;
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
  // this warp's slice of K (16-byte vectors) and the blocks that produce it
  const int nvec = H / VK;
  const int vb = warp * nvec / kWarps, ve = (warp + 1) * nvec / kWarps;
  const int plo = (vb * VK) / U, phi = ve > vb ? (ve * VK - 1) / U : -1;
  unsigned* flags = p.flags + (size_t)d * pl.P * p.flag_stride;
  T* y = reinterpret_cast<T*>(a.y);
  T* hseq = reinterpret_cast<T*>(a.hseq);
  __syncthreads();

  for (int s = 0; s < nT; ++s) {
    TRACE(s, 0);
    const int t = d ? nT - 1 - s : s;
    const int tp = d ? t + 1 : t - 1;
    float acc[kMaxTilesM][RM][RN];
#pragma unroll
    for (int tm = 0; tm < kMaxTilesM; ++tm)
#pragma unroll
      for (int i = 0; i < RM; ++i)
#pragma unroll
        for (int jj = 0; jj < RN; ++jj) acc[tm][i][jj] = 0.f;
    const T* B = nullptr;
    int64_t ldb = 0;
    if (s == 0) {
      B = reinterpret_cast<const T*>(a.h0);
      ldb = H;
    } else {
      B = y + (int64_t)tp * N * p.ldy + (int64_t)d * H;
      ldb = p.ldy;
    }
    if (B != nullptr && ve > vb) {
      bool ok = true;
      if (s > 0)
        ok = warp_wait_flags(flags, p.flag_stride, plo, phi, (unsigned)s, p.status, p.timeout_ns,
                             p.spin_ns);
      TRACE(s, 1);
      if (ok)
        warp_direct_contract<T, RM, RN, LM, LN>(acc, pl.tiles_m, As, pl.lda, B, ldb, N, vb, ve,
                                                lane, wbuf, pl.KC, pl.ldb, pl.nst, s, pl.P);
      else if (lane == 0)
        s_fail = 1;
      TRACE(s, 2);
    }
    if (!direct_reduce<RM, RN, LM, LN>(acc, pl.tiles_m, wall, wslot, outs, pl.nbp, lane, warp,
                                       &s_fail))
      return;
    TRACE(s, 3);
    if (item) {
      const int64_t row = (int64_t)t * N + n;
      const int slot = d ? t : t + 1;
      float h;
      if (p.mode == 1) {  // LSTM, gate blocks i, f, g, o
        const float ig = sigmoidf_(gxv[0] + outs[(0 * U + u) * pl.nbp + n]);
        const float fg = sigmoidf_(gxv[1] + outs[(1 * U + u) * pl.nbp + n]);
        const float gg = tanhf(gxv[2] + outs[(2 * U + u) * pl.nbp + n]);
        const float og = sigmoidf_(gxv[3] + outs[(3 * U + u) * pl.nbp + n]);
        c_own = fg * c_own + ig * gg;
        h = og * tanhf(c_own);
        if (a.gates) {
          float* gp = a.gates + row * 4 * H + j;
          gp[0] = ig; gp[H] = fg; gp[2 * H] = gg; gp[3 * H] = og;
        }
        if (a.cseq) a.cseq[((int64_t)slot * N + n) * H + j] = c_own;
      } else if (p.mode == 2) {  // GRU, gate blocks r, z, n
        const float ghn = outs[(2 * U + u) * pl.nbp + n] + bhn;
        const float r = sigmoidf_(gxv[0] + outs[(0 * U + u) * pl.nbp + n]);
        const float z = sigmoidf_(gxv[1] + outs[(1 * U + u) * pl.nbp + n]);
        const float nv = tanhf(gxv[2] + r * ghn);
        h = (1.f - z) * nv + z * h_own;
        if (a.gates) {
          float* gp = a.gates + row * 4 * H + j;
          gp[0] = r; gp[H] = z; gp[2 * H] = nv; gp[3 * H] = ghn;
        }
      } else {  // tanh RNN
        h = tanhf(gxv[0] + outs[u * pl.nbp + n]);
        if (a.gates) a.gates[row * H + j] = h;
      }
      h_own = h;
      y[row * p.ldy + (int64_t)d * H + j] = from_f<T>(h);
      if (hseq) hseq[((int64_t)slot * N + n) * H + j] = from_f<T>(h);
      if (s + 1 < nT) {  // next step's input projection, one step ahead
        const int tn = d ? t - 1 : t + 1;
        const float* gp = a.gx + ((int64_t)tn * N + n) * GH + j;
#pragma unroll
        for (int g = 0; g < 4; ++g)
          if (g < G) gxv[g] = __ldg(gp + g * H);
      }
    }
    if (s + 1 < nT) {
      __syncthreads();
      TRACE(s, 4);
      if (tid == 0 && !(blockIdx.x == p.fault_block && s == p.fault_step))
        publish_flag(flags + (size_t)blk * p.flag_stride, (unsigned)(s + 1));
      TRACE(s, 5);
    }
  }
  if (item) {
    const int64_t o = (int64_t)n * H + j;
    if (a.hy) reinterpret_cast<T*>(a.hy)[o] = from_f<T>(h_own);
    if (a.cy) a.cy[o] = c_own;
  }
}

template <typename T, int RM, int RN, int LM, int LN>
__global__ void __launch_bounds__(kThreads, 1)
    rec_bwd_direct(const __grid_constant__ RecParams p) {
  constexpr int VK = 16 / (int)sizeof(T);
  constexpr int TE = RM * RN * LM * LN;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_fail;
  const RecPlan& pl = p.plan;
  const int d = blockIdx.x / pl.P;
  const int blk = blockIdx.x - d * pl.P;
  const RecDirArgs& a = p.dir[d];
  const int H = p.H, N = p.N, nT = p.T, G = p.G, U = pl.U;
  const int j0 = blk * U;
  const int Uc = min(U, H - j0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t GH = (int64_t)G * H;
  T* As = reinterpret_cast<T*>(smem);
  float* outs = reinterpret_cast<float*>(As + (size_t)pl.Mp * pl.lda);
  // per-warp slots: staging stages during the contraction, then the warp's
  // partial tiles for the cross-warp reduction
  uint4* wall = reinterpret_cast<uint4*>(outs + pl.Mp * pl.nbp);
  const int wslot = max(pl.nst * (LN * RN) * pl.ldb, (pl.tiles_m * TE * 4 + 15) / 16);
  uint4* wbuf = wall + (size_t)warp * wslot;

  if (ld_volatile_int(p.status) != kDevOk) return;
  if (tid == 0) s_fail = 0;
  // resident slice, transposed: A[u][r] = W_hh[r][j0 + u]
  const T* W = reinterpret_cast<const T*>(a.whh);
  for (int64_t idx = tid; idx < (int64_t)pl.Mp * pl.lda; idx += kThreads) {
    const int r = (int)(idx / pl.Mp), u = (int)(idx - (int64_t)r * pl.Mp);
    As[(int64_t)u * pl.lda + r] = (u < Uc && r < GH) ? W[(int64_t)r * H + j0 + u] : from_f<T>(0.f);
  }

  const bool item = tid < Uc * N;
  const int u = item ? tid % Uc : 0, n = item ? tid / Uc : 0, j = j0 + u;
  float dc_own = 0.f, carry = 0.f;
  // inputs of the coming step's pointwise math, loaded one step ahead
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
  // this warp's slice of K = G*H and the blocks that produce it
  const int nvec = (int)(GH / VK);
  const int vb = warp * nvec / kWarps, ve = (warp + 1) * nvec / kWarps;
  unsigned* flags = p.flags + (size_t)d * pl.P * p.flag_stride;
  T* dgx = reinterpret_cast<T*>(a.dgx);
  T* dgh = reinterpret_cast<T*>(a.dgh);
  __syncthreads();

  for (int s = 0; s <= nT; ++s) {
    TRACE(s, 0);
    const int t = d ? s : nT - 1 - s;    // time processed at this step (s < nT)
    const int tp = d ? s - 1 : nT - s;   // time processed at the previous step (s > 0)
    if (s > 0) {
      float acc[kMaxTilesM][RM][RN];
#pragma unroll
      for (int tm = 0; tm < kMaxTilesM; ++tm)
#pragma unroll
        for (int i = 0; i < RM; ++i)
#pragma unroll
          for (int jj = 0; jj < RN; ++jj) acc[tm][i][jj] = 0.f;
      if (ve > vb) {
        bool ok = true;
        for (int g = 0; g < G && ok; ++g) {
          const int lo = max(vb * VK, g * H), hi = min(ve * VK, (g + 1) * H);
          if (lo < hi)
            ok = warp_wait_flags(flags, p.flag_stride, (lo - g * H) / U, (hi - 1 - g * H) / U,
                                 (unsigned)s, p.status, p.timeout_ns, p.spin_ns);
        }
        TRACE(s, 1);
        if (ok)
          warp_direct_contract<T, RM, RN, LM, LN>(acc, pl.tiles_m, As, pl.lda,
                                                  dgh + (int64_t)tp * N * GH, GH, N, vb, ve, lane,
                                                  wbuf, pl.KC, pl.ldb, pl.nst, s, pl.P);
        else if (lane == 0)
          s_fail = 1;
      }
      TRACE(s, 2);
      if (!direct_reduce<RM, RN, LM, LN>(acc, pl.tiles_m, wall, wslot, outs, pl.nbp, lane, warp,
                                         &s_fail))
        return;
      TRACE(s, 3);
    }
    if (item) {
      float dhf;
      if (s == 0)
        dhf = a.dhy ? to_f(reinterpret_cast<const T*>(a.dhy)[(int64_t)n * H + j]) : 0.f;
      else
        dhf = outs[u * pl.nbp + n] + carry;
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
    if (s < nT) {
      __syncthreads();
      TRACE(s, 4);
      if (tid == 0 && !(blockIdx.x == p.fault_block && s == p.fault_step))
        publish_flag(flags + (size_t)blk * p.flag_stride, (unsigned)(s + 1));
      TRACE(s, 5);
    }
  }
}

template <typename T, int S>
void* fwd_fn() {
  return (void*)rec_fwd_kernel<T, kShapes[S].RM, kShapes[S].RN, kShapes[S].LM, kShapes[S].LN>;
}
template <typename T, int S>
void* bwd_fn() {
  return (void*)rec_bwd_kernel<T, kShapes[S].RM, kShapes[S].RN, kShapes[S].LM, kShapes[S].LN>;
}
template <typename T, int S>
void* fwd_direct_fn() {
  return (void*)rec_fwd_direct<T, kShapes[S].RM, kShapes[S].RN, kShapes[S].LM, kShapes[S].LN>;
}
template <typename T, int S>
void* bwd_direct_fn() {
  return (void*)rec_bwd_direct<T, kShapes[S].RM, kShapes[S].RN, kShapes[S].LM, kShapes[S].LN>;
}

void* pick_kernel(bool backward, bool direct, int is_bf16, int shape) {
  static void* const table[2][2][2][kNumShapes] = {
      {{{fwd_fn<float, 0>(), fwd_fn<float, 1>(), fwd_fn<float, 2>(), fwd_fn<float, 3>()},
        {fwd_fn<bf16, 0>(), fwd_fn<bf16, 1>(), fwd_fn<bf16, 2>(), fwd_fn<bf16, 3>()}},
       {{bwd_fn<float, 0>(), bwd_fn<float, 1>(), bwd_fn<float, 2>(), bwd_fn<float, 3>()},
        {bwd_fn<bf16, 0>(), bwd_fn<bf16, 1>(), bwd_fn<bf16, 2>(), bwd_fn<bf16, 3>()}}},
      {{{fwd_direct_fn<float, 0>(), fwd_direct_fn<float, 1>(), fwd_direct_fn<float, 2>(),
         fwd_direct_fn<float, 3>()},
        {fwd_direct_fn<bf16, 0>(), fwd_direct_fn<bf16, 1>(), fwd_direct_fn<bf16, 2>(),
         fwd_direct_fn<bf16, 3>()}},
       {{bwd_direct_fn<float, 0>(), bwd_direct_fn<float, 1>(), bwd_direct_fn<float, 2>(),
         bwd_direct_fn<float, 3>()},
        {bwd_direct_fn<bf16, 0>(), bwd_direct_fn<bf16, 1>(), bwd_direct_fn<bf16, 2>(),
         bwd_direct_fn<bf16, 3>()}}}};
  return table[direct ? 1 : 0][backward ? 1 : 0][is_bf16 ? 1 : 0][shape];
}

cudaError_t launch(bool backward, const RecParams& p, cudaStream_t st) {
  const RecPlan& pl = p.plan;
  void* fn = pick_kernel(backward, pl.direct != 0, p.bf16, pl.shape);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.flags, 0, sizeof(unsigned) * (size_t)p.D * pl.P * p.flag_stride, st);
  if (e != cudaSuccess) return e;
  RecParams copy = p;
  void* args[] = {&copy};
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaLaunchCooperativeKernel(fn, dim3(p.D * pl.P), dim3(kThreads), args, pl.smem, st);
}

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// direct-path plan, or false when the problem does not qualify
bool make_direct_plan(bool backward, int G, int e, int D, int H, int N, int P, int U,
                      size_t smem_limit, RecPlan* out) {
  const int VK = 16 / e;
  const int Mloc = backward ? U : G * U;
  const int K = backward ? G * H : H;
  if (K % VK != 0 || (H * e) % 16 != 0) return false;
  if ((int64_t)U * N > kThreads) return false;
  bool found = false;
  double best_cost = 0;
  RecPlan best;
  for (int sh = 0; sh < kNumShapes; ++sh) {
    const Shape S = kShapes[sh];
    const int LK = 32 / (S.LM * S.LN);
    const int tmr = S.LM * S.RM, tnc = S.LN * S.RN;
    if (N > tnc) continue;
    const int tiles_m = (Mloc + tmr - 1) / tmr;
    if (tiles_m > kMaxTilesM) continue;
    const int nvec = K / VK;
    if (nvec < kWarps * LK / 2) continue;  // too little K to spread over the warps
    RecPlan pl;
    pl.direct = 1;
    pl.shape = sh; pl.P = P; pl.U = U; pl.Mloc = Mloc; pl.Mp = tiles_m * tmr;
    pl.K = K; pl.nb = N; pl.nbp = tnc;
    pl.tiles_m = tiles_m; pl.tiles_n = 1; pl.WK = kWarps;
    const int pad = (16 * LK) / e;
    pl.lda = (int)(round_up(K, 128 / e) + pad);
    const size_t fixed = (size_t)pl.Mp * pl.lda * e + (size_t)pl.Mp * pl.nbp * 4 + 256;
    if (fixed >= smem_limit) continue;
    // per-warp slots of nst stages x tnc rows x stride vectors of 16 B; the row
    // stride puts the rows a warp reads together on distinct bank groups, and a
    // slot also holds the warp's partial tiles after the contraction
    const int slice = (nvec + kWarps - 1) / kWarps;
    // row strides that keep the rows one warp-wide load touches on distinct
    // bank groups: 4 rows x 16 B (LK = 1) need stride % 4 != 0; 4 rows x 64 B
    // (LK = 4) need stride % 8 == 4
    auto stride_of = [&](int c) {
      int st = std::max(c, 1);
      while (LK == 1 ? (st % 4 == 0) : (st % 8 != 4)) ++st;
      return st;
    };
    const int part_vecs = (tiles_m * S.RM * S.RN * S.LM * S.LN * 4 + 15) / 16;
    auto slot_vecs = [&](int c, int st) {
      return std::max(st * tnc * stride_of(c), part_vecs);
    };
    auto bytes_of = [&](int c, int st) { return fixed + (size_t)kWarps * slot_vecs(c, st) * 16; };
    int chv = slice, nst = 1;
    if (bytes_of(chv, 1) > smem_limit) {
      nst = 2;
      while (chv > 1 && bytes_of(chv, 2) > smem_limit) --chv;
    }
    if (bytes_of(chv, nst) > smem_limit) continue;
    if (chv < LK && chv < slice) continue;
    pl.KC = chv;
    pl.nst = nst;
    pl.ldb = stride_of(chv);
    pl.smem = bytes_of(chv, nst);
    const int nchunk = (slice + chv - 1) / chv;
    const double cost = (double)tiles_m * S.RM * S.RN * ((double)K / (kWarps * LK)) *
                        ((double)N / tnc > 0.5 ? 1.0 : 1.25) * (1.0 + 0.15 * nchunk);
    if (!found || cost < best_cost) {
      found = true;
      best_cost = cost;
      best = pl;
    }
  }
  if (found) *out = best;
  return found;
}

}  // namespace

#ifdef LAYER_RNN_TRACE
extern "C" int rnn_debug_trace_copy(void* host, size_t bytes) {
  if (bytes > sizeof(g_trace)) bytes = sizeof(g_trace);
  return (int)cudaMemcpyFromSymbol(host, g_trace, bytes);
}
#endif

bool rec_make_plan(bool backward, int mode, int bf16, int D, int H, int N, int num_sms,
                   size_t smem_limit, RecPlan* out, bool allow_direct) {
  const int G = mode == 1 ? 4 : mode == 2 ? 3 : 1;
  const int e = bf16 ? 2 : 4;
  const int VK = 16 / e;
  int P = num_sms / D;
  if (P < 1) P = 1;
  if (P > kThreads) P = kThreads;
  if (P > H) P = H;
  const int U = (H + P - 1) / P;
  P = (H + U - 1) / U;
  if (allow_direct && make_direct_plan(backward, G, e, D, H, N, P, U, smem_limit, out)) return true;
  const int Mloc = backward ? U : G * U;
  const int K = backward ? G * H : H;
  bool found = false;
  double best_cost = 0;
  RecPlan best;
  for (int sh = 0; sh < kNumShapes; ++sh) {
    const Shape S = kShapes[sh];
    const int LK = 32 / (S.LM * S.LN);
    const int tmr = S.LM * S.RM, tnc = S.LN * S.RN;
    const int tiles_m = (Mloc + tmr - 1) / tmr;
    if (tiles_m > kWarps) continue;
    const int max_tn = kWarps / tiles_m;
    const int nchunks = (N + max_tn * tnc - 1) / (max_tn * tnc);
    const int nb = (N + nchunks - 1) / nchunks;
    const int tiles_n = (nb + tnc - 1) / tnc;
    const int WK = kWarps / (tiles_m * tiles_n);
    RecPlan pl;
    pl.shape = sh; pl.P = P; pl.U = U; pl.Mloc = Mloc; pl.Mp = tiles_m * tmr;
    pl.K = K; pl.nb = nb; pl.nbp = tiles_n * tnc;
    pl.tiles_m = tiles_m; pl.tiles_n = tiles_n; pl.WK = WK;
    const int pad = (16 * LK) / e;          // bank offset between consecutive rows
    const int row_align = 128 / e;
    pl.lda = (int)(round_up(round_up(K, VK), row_align) + pad);
    const size_t fixed = (size_t)pl.Mp * pl.lda * e + (size_t)kWarps * S.RM * S.RN * 32 * 4 +
                         (size_t)pl.Mp * pl.nbp * 4 + (size_t)2 * U * N * 4 + 256;
    if (fixed >= smem_limit) continue;
    const size_t room = smem_limit - fixed;
    // largest K chunk (multiple of row_align, or all of K) whose staging fits
    int KC = (int)round_up(K, VK);
    auto bytes_for = [&](int kc) { return (size_t)pl.nbp * (round_up(kc, row_align) + pad) * e; };
    if (bytes_for(KC) > room) {
      KC = (int)(room / ((size_t)pl.nbp * e)) - pad;
      KC = KC / row_align * row_align;
      while (KC > 0 && bytes_for(KC) > room) KC -= row_align;
    }
    if (KC < row_align && KC < K) continue;
    pl.KC = KC;
    pl.ldb = (int)(round_up(KC, row_align) + pad);
    pl.smem = fixed + bytes_for(KC);
    const double cost = (double)nchunks * S.RM * S.RN * ((double)K / (WK * LK)) *
                        (1.0 + 0.02 * ((K + KC - 1) / KC));
    if (!found || cost < best_cost) {
      found = true;
      best_cost = cost;
      best = pl;
    }
  }
  if (found) *out = best;
  return found;
}

cudaError_t rec_forward(const RecParams& p, cudaStream_t st) { return launch(false, p, st); }
cudaError_t rec_backward(const RecParams& p, cudaStream_t st) { return launch(true, p, st); }

}  // namespace lr
