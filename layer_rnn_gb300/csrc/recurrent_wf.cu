// Layer wavefront for unidirectional bf16 stacks: the forward of all L layers
// in one persistent launch.
//
// The "Four layers" rung of the cuDNN optimisation table quoted in the Keras
// issue "Exposing Cudnn v5 RNN models (in tensorflow) from within keras" runs
// layer l+1's step t while layer l runs step t+1.  Here every layer owns Pr
// blocks for the whole launch; block (l, r) owns hidden units
// u0 .. u0+Ur-1 of layer l and, for each time step, contracts
//
//     a[m][n] = sum_k Wp[m][k] * [x_t | h_{t-1}][n][k],   K = I_l + H,
//
// i.e. the input projection of the step (x_t = the input for l = 0, layer
// l-1's h_t above) and the recurrent product in one tensor-core accumulation
// (tcgen05.mma kind::f16, fp32 accumulator in tensor memory), then applies the
// fused gate math of its units.  A layer's step t needs only layer l-1's step
// t and its own step t-1, so the layers proceed as a wavefront: the sequence
// takes T + L - 1 step latencies instead of L * T.
//
// The weights of all layers do not fit on chip at the sizes this serves (4
// layers x [W_ih | W_hh] bf16 = 56 MB at H = I = 1024), so both operands are
// streamed every step from L2 (the packed weights stay L2-resident: at most a
// few tens of MB) through a multi-stage TMA ring (cp.async.bulk.tensor,
// 128-byte swizzle): warp 0 issues the loads, one thread of warp 1 the MMAs,
// and all eight warps read the accumulator back for the pointwise math.
//
// Packed weights (built per call by wf_pack_kernel, the "matrix
// pre-transposition" rung of the same table): the rows of block r are the
// R * Ur rows of its units, unit-major (row u*R + g), each row [W_ih row | pad
// to 64 | W_hh row | pad to 64].  LSTM rows g = i, f, g, o; GRU rows r, z,
// n_x (W_in, x part only) and n_h (W_hn, h part only), because the GRU of the
// "rnn training example?" thread multiplies r into (W_hn h + b_hn) alone; tanh
// RNN one row per unit.  Biases are folded per packed row (b_ih + b_hh; GRU:
// b_in on n_x, b_hn on n_h).  With four rows per unit in adjacent tensor-memory
// lanes, a unit's gates meet in four lanes of one warp and are exchanged with
// shuffles: no shared-memory staging of the accumulator.
//
// Synchronisation: one flag per block (128 bytes apart) counts the hseq slots
// the block has written (slot 0 = h0, slot t+1 = h_t).  Step t of layer l
// waits for its own layer's flags >= t+1 and layer l-1's flags >= t+2, then
// its loads (async proxy) read what other blocks stored (generic proxy): the
// writer fences its stores to the async proxy before its release, the reader
// after its acquire.  Every wait is bounded; the launch is cooperative, so all
// blocks are co-resident.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "wf.h"

#ifdef LAYER_RNN_TRACE
__device__ unsigned long long g_wtrace[4][1024][8];
#define WTRACE(s, k)                                                                    \
  do {                                                                                  \
    const int b_ = (blockIdx.x % p.plan.Pr == 0) ? (int)(blockIdx.x / p.plan.Pr) : -1; \
    if (b_ >= 0 && b_ < 4 && threadIdx.x == 0 && (s) < 1024)                            \
      g_wtrace[b_][(s)][(k)] = lr::globaltimer_ns();                                    \
  } while (0)
#else
#define WTRACE(s, k) ((void)0)
#endif

namespace lr {

namespace {

constexpr int kWThreads = 256;
constexpr int kRows = 128;       // MMA M
constexpr int kChunk = 64;       // bf16 elements of K per ring stage (128 bytes)
constexpr int kMaxStages = 8;
constexpr int kMaxNm = 128;      // batch columns per block
constexpr int kStateSlots = kMaxNm / 8;  // fp32 state items per thread (4-column groups / 2)

struct WfMaps {
  CUtensorMap a[kWfMaxLayers];   // packed weights [rows][kp], box 64 x 128
  CUtensorMap bx[kWfMaxLayers];  // x part source [slots][N][K_x], box 64 x Nm x 1
  CUtensorMap bh[kWfMaxLayers];  // own hseq [T+1][N][H], box 64 x Nm x 1
};

__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mb_try(uint32_t bar, uint32_t parity) {
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

// bounded by time only: used where the awaited arrival is certain to come
// (already issued copies / MMAs), so the block never leaves with work in flight
__device__ __forceinline__ bool mb_wait_time(uint32_t bar, uint32_t parity, int* status,
                                             long long timeout_ns) {
  if (mb_try(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  unsigned it = 0;
  while (!mb_try(bar, parity)) {
    if ((++it & 63u) == 0 && (long long)(globaltimer_ns() - t0) > timeout_ns) {
      atomicCAS(status, kDevOk, kDevTimeout);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// K-major tile of rows x 128 bytes, 128-byte swizzle, 8-row groups 1024 bytes
// apart (tile base 1024-byte aligned)
__device__ __forceinline__ uint64_t sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

// element i (0..3, may differ per lane) of (a, b, c, d) with predicated
// selects, never a branch: lanes of a warp take different i here
__device__ __forceinline__ float sel_if(unsigned cond, float if_set, float if_clear) {
  float r;
  asm("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %3, 0;\n\tselp.f32 %0, %1, %2, p;\n\t}"
      : "=f"(r)
      : "f"(if_set), "f"(if_clear), "r"(cond));
  return r;
}
__device__ __forceinline__ float pick4(float a, float b, float c, float d, int i) {
  const unsigned b0 = (unsigned)i & 1u, b1 = (unsigned)i & 2u;
  return sel_if(b1, sel_if(b0, d, c), sel_if(b0, b, a));
}

__device__ __forceinline__ void store_bf16(void* base, int64_t i, float v) {
  reinterpret_cast<bf16*>(base)[i] = __float2bfloat16_rn(v);
}

// Gate nonlinearities on the bf16 path: the hardware tanh (tanh.approx.f32,
// relative error about 2^-11, below the bf16 resolution of the stored h) and
// the identity sigmoid(x) = (1 + tanh(x / 2)) / 2.
__device__ __forceinline__ float tanh_hw(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigm_hw(float x) { return fmaf(0.5f, tanh_hw(0.5f * x), 0.5f); }

// EXT: per-sequence lengths and / or inter-layer dropout are in use (a
// separate instance, so the plain path carries none of their code)
template <bool EXT>
__global__ void __launch_bounds__(kWThreads, 1)
    rec_wf_kernel(const __grid_constant__ WfMaps maps, const __grid_constant__ WfParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxStages + 1];
  __shared__ uint32_t tmem_slot;
  __shared__ int s_fail;    // a wait of this block gave up, or the status was set
  __shared__ int s_stop;    // the load issuer stopped inside the current step
  __shared__ int s_issued;  // ... after issuing this many chunks of it

  const WfPlan& pl = p.plan;
  const int l = blockIdx.x / pl.Pr, r = blockIdx.x - l * pl.Pr;
  const WfLayer& a = p.layer[l];
  const int H = p.H, N = p.N, nT = p.T, Ur = pl.Ur, R = pl.R, Nm = pl.Nm, S = pl.stages;
  const int u0 = r * Ur, Urc = min(Ur, H - u0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nch = a.nch, nchx = a.nchx;
  const uint32_t base = (su32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bytesA = kRows * 128u, bytesB = (uint32_t)Nm * 128u, stage = bytesA + bytesB;
  const uint32_t full0 = su32(&bars[0]), empty0 = su32(&bars[kMaxStages]);
  const uint32_t done = su32(&bars[2 * kMaxStages]);
  const uint32_t ncols = (uint32_t)pl.tmem_cols;

  // the plan fits the kernel's fixed limits; otherwise touch nothing
  const bool cfg_bad = l >= p.L || l >= kWfMaxLayers || Nm < 16 || Nm > kMaxNm || Nm % 16 != 0 ||
                       N > Nm || R * Ur > kRows || (R != 1 && R != 4) || S < 2 ||
                       S > kMaxStages || (uint32_t)Nm > ncols || ncols > 512u ||
                       (ncols & (ncols - 1u)) != 0 || ncols < 32u || nchx < 1 || nchx >= nch;
  if (tid == 0) {
    s_fail = cfg_bad || ld_volatile_int(p.status) != kDevOk;
    if (cfg_bad) atomicCAS(p.status, kDevOk, kDevCheck);
    s_stop = 0;
    s_issued = 0;
    for (int s = 0; s < kMaxStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(full0 + 8 * s) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(empty0 + 8 * s) : "memory");
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(done) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 2 && !cfg_bad) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(&tmem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_slot;
  bool failed = s_fail != 0;

  // epilogue ownership: warp w reads tensor-memory lanes 32*(w%4) .. +31
  // (packed rows), columns in 16-wide chunks ci = w/4, w/4 + 2, ...
  const int q = warp & 3, half = warp >> 2;
  const int m = q * 32 + lane;
  const int u = R == 4 ? m >> 2 : m;
  const int g = R == 4 ? (lane & 3) : 0;
  const bool unit_ok = u < Urc;
  const int j = u0 + u;
  const int nci = Nm / 16;
  float bias[4] = {0.f, 0.f, 0.f, 0.f};
  if (unit_ok) {
    const float* bp = a.bias + (int64_t)r * R * Ur;
    if (R == 4) {
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) bias[gg] = bp[u * 4 + gg];
    } else {
      bias[0] = bp[u];
    }
  }
  // fp32 state of this thread's (unit, batch) items: LSTM c, GRU h
  // kept in shared memory (slot i of thread tid at st_s[i * kWThreads + tid]):
  // the epilogue below is a loop, not unrolled, to stay small in the
  // instruction cache
  float* st_s = reinterpret_cast<float*>(smem_raw + (base - su32(smem_raw)) + S * stage);
  for (int i = 0; i < kStateSlots; ++i) st_s[i * kWThreads + tid] = 0.f;
  // slot 0 of hseq (and cseq) and the initial state
  const bf16* h0 = reinterpret_cast<const bf16*>(a.h0);
  if (R == 4) {
    // the epilogue's item mapping: column n = 4*cg + g, cg = half, half + 2, ...
    for (int cg = half; cg < Nm / 4; cg += 2) {
      const int n = cg * 4 + g;
      if (failed || !unit_ok || n >= N) continue;
      const int64_t o = (int64_t)n * H + j;
      const float hv = h0 ? __bfloat162float(h0[o]) : 0.f;
      const float cv = a.c0 ? a.c0[o] : 0.f;
      st_s[(cg >> 1) * kWThreads + tid] = p.mode == 1 ? cv : hv;
      store_bf16(a.hseq, o, hv);
      if (a.cseq) a.cseq[o] = cv;
    }
  } else {
    for (int ci = half; ci < nci; ci += 2)
      for (int i = 0; i < 16; ++i) {
        const int n = ci * 16 + i;
        if (failed || !unit_ok || n >= N) continue;
        const int64_t o = (int64_t)n * H + j;
        store_bf16(a.hseq, o, h0 ? __bfloat162float(h0[o]) : 0.f);
      }
  }
  __syncthreads();
  unsigned* flags = p.flags;
  const int fstride = p.flag_stride;
  if (tid == 0 && !failed) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    publish_flag(flags + (size_t)blockIdx.x * fstride, 1u);
  }

  const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(Nm >> 3) << 17) |
                         ((uint32_t)(kRows >> 4) << 24);
  const unsigned* own_flags = flags + (size_t)l * pl.Pr * fstride;
  const unsigned* prev_flags = flags + (size_t)(l > 0 ? l - 1 : 0) * pl.Pr * fstride;
  const int arow = r * R * Ur;   // first packed row of this block
  const int64_t GsH = (int64_t)p.Gs * H;
  // the x part's time coordinate: row t of x, or of the layer below's
  // dropped output; else slot t + 1 of the layer below's hidden states
  const bool x_row0 = l == 0 || (EXT && p.layer[l - 1].drop_mask != nullptr);
  const float dscale = a.drop_scale;
  // sequence n's step t: inside its length?
  auto active = [&](int t, int n) {
    if constexpr (!EXT) return true;
    else return p.lengths == nullptr || t < __ldg(p.lengths + n);
  };
  // the value of y for output h at element e: zero past the length, the
  // dropped value where dropout applies
  auto y_value = [&](float h, bool act, int64_t e) {
    if constexpr (!EXT) return h;
    else {
      if (!act) return 0.f;
      if (a.drop_mask == nullptr) return h;
      return __ldg(a.drop_mask + e) != 0 ? __bfloat162float(__float2bfloat16_rn(h)) * dscale : 0.f;
    }
  };

  for (int t = 0; t < nT && !failed; ++t) {
    WTRACE(t, 0);
    if (warp == 0) {
      // ---- loads: x part (ready early: the layer below runs ahead), then h part
      bool ok = true;
      if (l > 0)
        ok = warp_wait_flags(prev_flags, fstride, 0, pl.Pr - 1, (unsigned)(t + 2), p.status,
                             p.timeout_ns, 0);
      __syncwarp();  // the lanes' acquires order lane 0's loads below
      int c = 0;
      for (; ok && c < nch; ++c) {
        if (c == nchx) {
          ok = warp_wait_flags(own_flags, fstride, 0, pl.Pr - 1, (unsigned)(t + 1), p.status,
                               p.timeout_ns, 0);
          __syncwarp();
          if (!ok) break;
        }
        const uint32_t it = (uint32_t)t * (uint32_t)nch + (uint32_t)c;
        const uint32_t s = it % (uint32_t)S, ph = (it / (uint32_t)S) & 1u;
        int okl = 1;
        if (lane == 0) okl = mb_wait_time(empty0 + 8 * s, ph ^ 1u, p.status, p.timeout_ns);
        ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
        if (!ok) break;
        if (lane == 0) {
          if (c == 0 || c == nchx) asm volatile("fence.proxy.async.global;" ::: "memory");
          const uint32_t dst = base + s * stage;
          const uint32_t fb = full0 + 8 * s;
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb),
                       "r"(stage)
                       : "memory");
          tma_2d(dst, &maps.a[l], c * kChunk, arow, fb);
          if (c < nchx)
            tma_3d(dst + bytesA, &maps.bx[l], c * kChunk, 0, x_row0 ? t : t + 1, fb);
          else
            tma_3d(dst + bytesA, &maps.bh[l], (c - nchx) * kChunk, 0, t, fb);
        }
        __syncwarp();
      }
      if (lane == 0 && c < nch) {
        s_issued = c;
        __threadfence_block();
        s_stop = 1;
        s_fail = 1;
      }
      __syncwarp();
    } else if (warp == 1 && lane == 0) {
      // ---- MMAs: exactly the chunks the load issuer issued
      int c = 0;
      for (; c < nch; ++c) {
        const uint32_t it = (uint32_t)t * (uint32_t)nch + (uint32_t)c;
        const uint32_t s = it % (uint32_t)S, ph = (it / (uint32_t)S) & 1u;
        bool got = mb_try(full0 + 8 * s, ph);
        if (!got) {
          const unsigned long long t0 = globaltimer_ns();
          unsigned spins = 0;
          while (!(got = mb_try(full0 + 8 * s, ph))) {
            if (ld_volatile_int(&s_stop) && c >= ld_volatile_int(&s_issued)) break;
            if ((++spins & 63u) == 0 && (long long)(globaltimer_ns() - t0) > p.timeout_ns) {
              atomicCAS(p.status, kDevOk, kDevTimeout);
              s_fail = 1;
              break;
            }
          }
        }
        if (!got) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t st = base + s * stage;
        const uint64_t ad = sw128(st), bd = sw128(st + bytesA);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                   (c > 0 || kk > 0) ? 1u : 0u);
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                empty0 + 8 * s)
            : "memory");
      }
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(done)
          : "memory");
    }
    __syncwarp();
    WTRACE(t, 1);
    // ---- accumulator complete (the commit above always arrives)
    const bool dok = mb_wait_time(done, (uint32_t)(t & 1), p.status, p.timeout_ns);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (!dok) s_fail = 1;
    __syncthreads();
    failed = s_fail != 0;
    WTRACE(t, 2);
    if (!failed) {
      const bool last = t == nT - 1;
      const int64_t row0 = (int64_t)t * N;
      bf16* hs = reinterpret_cast<bf16*>(a.hseq) + (int64_t)(t + 1) * N * H;
      if (R == 4) {
        // 4-column groups, alternating between the two warp halves.  Lanes
        // 4u .. 4u+3 hold gates 0..3 of unit u for the group's 4 columns; lane
        // 4u+g collects all gates of column 4*cg+g with three shuffles.  The
        // loop body stays small (it runs from the instruction cache).
#pragma unroll 2
        for (int cg = half; cg < Nm / 4; cg += 2) {
          float v[4];
          tmem_ld4(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(cg * 4), v);
          float got[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float send = pick4(v[0], v[1], v[2], v[3], (g - k) & 3);
            got[k] = __shfl_sync(0xffffffffu, send, (lane & ~3) | ((g + k) & 3));
          }
          // got[k] is gate (g + k) & 3; gate i is got[(i - g) & 3]
          const float a0 = pick4(got[0], got[1], got[2], got[3], (0 - g) & 3) + bias[0];
          const float a1 = pick4(got[0], got[1], got[2], got[3], (1 - g) & 3) + bias[1];
          const float a2 = pick4(got[0], got[1], got[2], got[3], (2 - g) & 3) + bias[2];
          const float a3 = pick4(got[0], got[1], got[2], got[3], (3 - g) & 3) + bias[3];
          const int n = cg * 4 + g;
          float& stv = st_s[(cg >> 1) * kWThreads + tid];
          float o0, o1, o2, o3, h, sn;
          if (p.mode == 1) {  // LSTM: i, f, g, o
            o0 = sigm_hw(a0);
            o1 = sigm_hw(a1);
            o2 = tanh_hw(a2);
            o3 = sigm_hw(a3);
            sn = fmaf(o1, stv, o0 * o2);
            h = o3 * tanh_hw(sn);
          } else {  // GRU: r, z, W_in x + b_in, W_hn h + b_hn
            o0 = sigm_hw(a0);
            o1 = sigm_hw(a1);
            o2 = tanh_hw(fmaf(o0, a3, a2));
            o3 = a3;
            h = fmaf(o1, stv - o2, o2);  // (1 - z) n + z h
            sn = h;
          }
          const bool in = unit_ok && n < N;
          const bool act = !in || active(t, n);
          if (act) {
            stv = sn;
          } else {
            // past the sequence's length: the state is kept (the LSTM's
            // h_{t-1} as stored in slot t by this thread, the GRU's state)
            h = p.mode == 1 ? __bfloat162float(reinterpret_cast<const bf16*>(a.hseq)
                                                   [(int64_t)t * N * H + (int64_t)n * H + j])
                            : stv;
          }
          if (!in) continue;
          const int64_t row = row0 + n;
          const int64_t o = (int64_t)n * H + j;
          if (a.gates) {
            float* gp = a.gates + row * GsH + j;
            gp[0] = o0; gp[H] = o1; gp[2 * H] = o2; gp[3 * H] = o3;
          }
          hs[o] = __float2bfloat16_rn(h);
          if (a.y) store_bf16(a.y, row * H + j, y_value(h, act, row * H + j));
          if (p.mode == 1 && a.cseq) a.cseq[(int64_t)(t + 1) * N * H + o] = stv;
          if (last) {
            if (a.hy) store_bf16(a.hy, o, h);
            if (a.cy) a.cy[o] = stv;
          }
        }
      } else {
#pragma unroll 2
        for (int cg = half; cg < Nm / 4; cg += 2) {
          float v[4];
          tmem_ld4(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(cg * 4), v);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int n = cg * 4 + i;
            if (!unit_ok || n >= N) continue;
            const int64_t row = row0 + n;
            const float hn = tanh_hw(v[i] + bias[0]);
            const int64_t o = (int64_t)n * H + j;
            const bool act = active(t, n);
            // past the sequence's length: h_{t-1} as stored in slot t
            const float h = act ? hn
                                : __bfloat162float(reinterpret_cast<const bf16*>(a.hseq)
                                                       [(int64_t)t * N * H + o]);
            hs[o] = __float2bfloat16_rn(h);
            if (a.y) store_bf16(a.y, row * H + j, y_value(h, act, row * H + j));
            if (a.gates) a.gates[row * GsH + j] = hn;
            if (last && a.hy) store_bf16(a.hy, o, h);
          }
        }
      }
    }
    WTRACE(t, 5);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    WTRACE(t, 3);
    failed = s_fail != 0;
    if (!failed && tid == 0 && !((int)blockIdx.x == p.fault_block && t == p.fault_step)) {
      // the block's stores (ordered before this thread by the barrier) become
      // visible to the other blocks' tensor loads: proxy fence, then release
      asm volatile("fence.proxy.async.global;" ::: "memory");
      publish_flag(flags + (size_t)blockIdx.x * fstride, (unsigned)(t + 2));
    }
    WTRACE(t, 4);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 2 && !cfg_bad)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols)
                 : "memory");
}

// packed row (r, m): unit u = m / R, gate row g = m % R of block r (rows
// r*R*Ur .. r*R*Ur + R*Ur - 1); 16-byte vectors (I_l and H multiples of 8)
__global__ void wf_pack_kernel(const bf16* wih, const bf16* whh, const bf16* bih, const bf16* bhh,
                               int mode, int64_t I, int64_t H, int64_t Kxp, int64_t kp, int Pr,
                               int Ur, int R, bf16* wp, float* bp) {
  const int64_t vpr = kp / 8;
  const int64_t rows = (int64_t)Pr * R * Ur;
  const int64_t total = rows * vpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / vpr, k = (i - row * vpr) * 8;
    const int64_t r = row / (R * Ur), mm = row - r * R * Ur;
    const int64_t uu = mm / R, g = mm - uu * R, jj = r * Ur + uu;
    uint4 v = make_uint4(0, 0, 0, 0);
    float b = 0.f;
    if (jj < H) {
      int64_t src = g;            // source gate block of W_ih / W_hh
      bool use_x = true, use_h = true;
      if (mode == 2 && g == 2) use_h = false;
      if (mode == 2 && g == 3) {
        src = 2;
        use_x = false;
      }
      if (k < Kxp) {
        if (use_x && k < I) v = *reinterpret_cast<const uint4*>(wih + (src * H + jj) * I + k);
      } else {
        const int64_t kh = k - Kxp;
        if (use_h && kh < H) v = *reinterpret_cast<const uint4*>(whh + (src * H + jj) * H + kh);
      }
      if (k == 0) {
        const float bi = __bfloat162float(bih[src * H + jj]);
        const float bh = __bfloat162float(bhh[src * H + jj]);
        b = (mode == 2 && g == 2) ? bi : (mode == 2 && g == 3) ? bh : bi + bh;
      }
    }
    *reinterpret_cast<uint4*>(wp + row * kp + k) = v;
    if (k == 0) bp[row] = b;
  }
}

}  // namespace

int64_t wf_kp(int64_t I_l, int64_t H) {
  return (I_l + kChunk - 1) / kChunk * kChunk + (H + kChunk - 1) / kChunk * kChunk;
}

bool wf_plan(int mode, int bf16, int L, int D, int64_t I, int64_t H, int64_t N, int num_sms,
             size_t smem_optin, WfPlan* out) {
  if (!bf16 || D != 1 || L < 2 || L > kWfMaxLayers) return false;
  if (N < 1 || N > kMaxNm || H % 8 != 0 || I % 8 != 0 || H < 8) return false;
  const int R = mode == 0 ? 1 : 4;
  const int per_layer = num_sms / L;
  if (per_layer < 1) return false;
  const int Ur = (int)((H + per_layer - 1) / per_layer);
  if (Ur * R > kRows) return false;
  WfPlan pl;
  pl.R = R;
  pl.Ur = Ur;
  pl.Pr = (int)((H + Ur - 1) / Ur);
  pl.Nm = (int)((N + 15) / 16 * 16);
  int cols = 32;
  while (cols < pl.Nm) cols *= 2;
  pl.tmem_cols = cols;
  const size_t stage = (size_t)kRows * 128 + (size_t)pl.Nm * 128;
  const size_t state_bytes = (size_t)kStateSlots * kWThreads * 4;
  const size_t budget = std::min<size_t>(smem_optin, 227 * 1024) - 1024 - 1024 - state_bytes;
  pl.stages = (int)std::min<size_t>(kMaxStages, budget / stage);
  if (pl.stages < 2) return false;
  pl.smem = pl.stages * stage + 1024 + state_bytes;
  // more than half of the shared memory: one block per SM, so each block's
  // tensor-memory allocation never waits for another's
  pl.smem = std::max<size_t>(pl.smem, 120 * 1024);
  if (pl.smem > smem_optin) return false;
  if ((int64_t)pl.Pr * L > num_sms) return false;
  *out = pl;
  return true;
}

int64_t wf_pack_bytes_bound(int mode, int L, int64_t I, int64_t H) {
  const int64_t R = mode == 0 ? 1 : 4;
  const int64_t rows = R * H + kRows;  // Pr * Ur < H + Ur, R * Ur <= 128
  int64_t total = 0;
  for (int l = 0; l < L; ++l) {
    const int64_t I_l = l == 0 ? I : H;
    total += (rows * wf_kp(I_l, H) * 2 + 255) / 256 * 256 + (rows * 4 + 255) / 256 * 256;
  }
  return total;
}

cudaError_t wf_pack(const WfPlan& pl, int mode, int64_t I_l, int64_t H, const void* wih,
                    const void* whh, const void* bih, const void* bhh, void* wp, float* bias,
                    cudaStream_t st) {
  const int64_t kp = wf_kp(I_l, H);
  const int64_t Kxp = (I_l + kChunk - 1) / kChunk * kChunk;
  const int64_t total = (int64_t)pl.Pr * pl.R * pl.Ur * (kp / 8);
  const int blocks = (int)std::min<int64_t>((total + 255) / 256, 16384);
  wf_pack_kernel<<<blocks, 256, 0, st>>>(
      reinterpret_cast<const bf16*>(wih), reinterpret_cast<const bf16*>(whh),
      reinterpret_cast<const bf16*>(bih), reinterpret_cast<const bf16*>(bhh), mode, I_l, H, Kxp,
      kp, pl.Pr, pl.Ur, pl.R, reinterpret_cast<bf16*>(wp), bias);
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

#ifdef LAYER_RNN_TRACE
extern "C" int rnn_debug_wtrace_copy(void* host, size_t bytes) {
  if (bytes > sizeof(g_wtrace)) bytes = sizeof(g_wtrace);
  return (int)cudaMemcpyFromSymbol(host, g_wtrace, bytes);
}
extern "C" int rnn_debug_wtrace_clear() {
  static unsigned long long zeros[4][1024][8];
  return (int)cudaMemcpyToSymbol(g_wtrace, zeros, sizeof(zeros));
}
#endif

cudaError_t wf_launch(const WfParams& p, cudaStream_t st) {
  const WfPlan& pl = p.plan;
  if (p.L < 2 || p.L > kWfMaxLayers) return cudaErrorInvalidValue;
  WfMaps maps;
  memset(&maps, 0, sizeof(maps));
  const uint64_t N = (uint64_t)p.N, H = (uint64_t)p.H, T = (uint64_t)p.T;
  for (int l = 0; l < p.L; ++l) {
    const WfLayer& a = p.layer[l];
    const uint64_t rows = (uint64_t)pl.Pr * pl.R * pl.Ur;
    const uint64_t da[2] = {(uint64_t)a.kp, rows}, sa[1] = {(uint64_t)a.kp * 2};
    const uint32_t ba[2] = {(uint32_t)kChunk, (uint32_t)kRows};
    if (!tma_encode(&maps.a[l], 2, true, a.wp, da, sa, ba)) return cudaErrorInvalidValue;
    const uint32_t bb[3] = {(uint32_t)kChunk, (uint32_t)pl.Nm, 1u};
    const uint64_t dh[3] = {H, N, T + 1}, sh[2] = {H * 2, N * H * 2};
    if (!tma_encode(&maps.bh[l], 3, true, a.hseq, dh, sh, bb)) return cudaErrorInvalidValue;
    if (l == 0) {
      const uint64_t I = (uint64_t)p.I;
      const uint64_t dx[3] = {I, N, T}, sx[2] = {I * 2, N * I * 2};
      if (!tma_encode(&maps.bx[0], 3, true, p.x, dx, sx, bb)) return cudaErrorInvalidValue;
    } else if (p.layer[l - 1].drop_mask) {
      // the layer below's dropped output, [T][N][H]
      if (!p.layer[l - 1].y) return cudaErrorInvalidValue;
      const uint64_t dy[3] = {H, N, T};
      if (!tma_encode(&maps.bx[l], 3, true, p.layer[l - 1].y, dy, sh, bb))
        return cudaErrorInvalidValue;
    } else {
      if (!tma_encode(&maps.bx[l], 3, true, p.layer[l - 1].hseq, dh, sh, bb))
        return cudaErrorInvalidValue;
    }
  }
  bool ext = p.lengths != nullptr;
  for (int l = 0; l < p.L; ++l) ext = ext || p.layer[l].drop_mask != nullptr;
  void* fn = ext ? (void*)rec_wf_kernel<true> : (void*)rec_wf_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.flags, 0, sizeof(unsigned) * (size_t)p.L * pl.Pr * p.flag_stride, st);
  if (e != cudaSuccess) return e;
  WfParams copy = p;
  void* args[] = {&maps, &copy};
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaLaunchCooperativeKernel(fn, dim3(p.L * pl.Pr), dim3(kWThreads), args, pl.smem, st);
}

}  // namespace lr
