// CUDA-core GEMM for the dense phases (input projection, dX, dW) with arbitrary
// operand strides, fp32 accumulation, fused bias and optional second product.
// 128x128 block tile, K step 16, 256 threads, 8x8 outputs per thread, operands
// converted to fp32 in shared memory, register-prefetched double buffering.
#include <algorithm>

#include "common.cuh"
#include "gemm.h"

namespace lr {

namespace {

constexpr int BM = 128, BN = 128, BK = 16, NT = 256;
constexpr int PADS = 4;

struct Seg {
  const void* A; int64_t sam, sak;
  const void* B; int64_t sbk, sbn;
  int64_t K;
};

struct KParams {
  int64_t M, N;
  Seg seg[2];
  int nseg;
  void* C; int64_t ldc;
  const void* bias1; const void* bias2; int64_t bias2_limit;
  int bias_bf16;
  int accumulate;
};

template <typename TI>
__device__ __forceinline__ float ld_in(const TI* p) { return to_f(p[0]); }

// A_KM: A has unit stride along k (else along m); B_KM: B has unit stride along k
// (else along n).  The thread-to-element map puts consecutive threads on the
// unit-stride dimension so that loads coalesce.
template <typename TI, bool A_KM, bool B_KM>
__device__ __forceinline__ void load_tile(float (&ra)[8], float (&rb)[8], const Seg& s,
                                          int64_t m0, int64_t n0, int64_t k0, int64_t M,
                                          int64_t N) {
  const TI* A = reinterpret_cast<const TI*>(s.A);
  const TI* B = reinterpret_cast<const TI*>(s.B);
  const int tid = threadIdx.x;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int idx = tid + NT * r;
    int mm, kk;
    if (A_KM) { mm = idx / BK; kk = idx % BK; } else { mm = idx % BM; kk = idx / BM; }
    const int64_t m = m0 + mm, k = k0 + kk;
    ra[r] = (m < M && k < s.K) ? ld_in(A + m * s.sam + k * s.sak) : 0.f;
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int idx = tid + NT * r;
    int nn, kk;
    if (B_KM) { nn = idx / BK; kk = idx % BK; } else { nn = idx % BN; kk = idx / BN; }
    const int64_t n = n0 + nn, k = k0 + kk;
    rb[r] = (n < N && k < s.K) ? ld_in(B + k * s.sbk + n * s.sbn) : 0.f;
  }
}

template <bool A_KM, bool B_KM>
__device__ __forceinline__ void store_tile(const float (&ra)[8], const float (&rb)[8],
                                           float (*As)[BM + PADS], float (*Bs)[BN + PADS]) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int idx = tid + NT * r;
    int mm, kk;
    if (A_KM) { mm = idx / BK; kk = idx % BK; } else { mm = idx % BM; kk = idx / BM; }
    As[kk][mm] = ra[r];
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int idx = tid + NT * r;
    int nn, kk;
    if (B_KM) { nn = idx / BK; kk = idx % BK; } else { nn = idx % BN; kk = idx / BN; }
    Bs[kk][nn] = rb[r];
  }
}

template <typename TI, typename TO, bool A_KM, bool B_KM>
__global__ void __launch_bounds__(NT) gemm_kernel(const __grid_constant__ KParams p) {
  __shared__ __align__(16) float As[2][BK][BM + PADS];
  __shared__ __align__(16) float Bs[2][BK][BN + PADS];
  const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  // flattened list of K tiles over the segments
  int64_t nk0 = (p.seg[0].K + BK - 1) / BK;
  int64_t nk1 = p.nseg > 1 ? (p.seg[1].K + BK - 1) / BK : 0;
  const int64_t nk = nk0 + nk1;
  float ra[8], rb[8];
  if (nk > 0) {
    const Seg& s = nk0 > 0 ? p.seg[0] : p.seg[1];
    load_tile<TI, A_KM, B_KM>(ra, rb, s, m0, n0, 0, p.M, p.N);
    store_tile<A_KM, B_KM>(ra, rb, As[0], Bs[0]);
  }
  __syncthreads();
  for (int64_t kt = 0; kt < nk; ++kt) {
    const int buf = (int)(kt & 1);
    if (kt + 1 < nk) {
      const int64_t nt = kt + 1;
      if (nt < nk0) load_tile<TI, A_KM, B_KM>(ra, rb, p.seg[0], m0, n0, nt * BK, p.M, p.N);
      else load_tile<TI, A_KM, B_KM>(ra, rb, p.seg[1], m0, n0, (nt - nk0) * BK, p.M, p.N);
    }
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (kt + 1 < nk) store_tile<A_KM, B_KM>(ra, rb, As[buf ^ 1], Bs[buf ^ 1]);
    __syncthreads();
  }

  TO* C = reinterpret_cast<TO*>(p.C);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
    if (n >= p.N) continue;
    float bias = 0.f;
    if (p.bias1) bias += load_any(p.bias1, n, p.bias_bf16);
    if (p.bias2 && n < p.bias2_limit) bias += load_any(p.bias2, n, p.bias_bf16);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
      if (m >= p.M) continue;
      float v = acc[i][j] + bias;
      TO* c = C + m * p.ldc + n;
      if (p.accumulate) v += to_f(*c);
      *c = from_f<TO>(v);
    }
  }
}

template <typename TI, typename TO>
cudaError_t launch_typed(const KParams& kp, bool a_km, bool b_km, cudaStream_t st) {
  dim3 grid((unsigned)((kp.N + BN - 1) / BN), (unsigned)((kp.M + BM - 1) / BM));
  if (a_km && b_km) gemm_kernel<TI, TO, true, true><<<grid, NT, 0, st>>>(kp);
  else if (a_km) gemm_kernel<TI, TO, true, false><<<grid, NT, 0, st>>>(kp);
  else if (b_km) gemm_kernel<TI, TO, false, true><<<grid, NT, 0, st>>>(kp);
  else gemm_kernel<TI, TO, false, false><<<grid, NT, 0, st>>>(kp);
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

// column sums, fixed summation order: block = 32 columns x 32 row lanes
__global__ void __launch_bounds__(1024) colsum_kernel(void* dst, int dst_bf16, const void* src,
                                                      int src_bf16, int64_t rows, int64_t cols,
                                                      int64_t ld) {
  __shared__ float part[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 32 + tx;
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  if (c < cols) {
    int64_t r = ty;
    for (; r + 96 < rows; r += 128) {
#pragma unroll
      for (int q = 0; q < 4; ++q) s[q] += load_any(src, (r + 32 * q) * ld + c, src_bf16);
    }
    for (; r < rows; r += 32) s[0] += load_any(src, r * ld + c, src_bf16);
  }
  part[ty][tx] = (s[0] + s[1]) + (s[2] + s[3]);
  __syncthreads();
  if (ty == 0 && c < cols) {
    float t = 0.f;
    for (int q = 0; q < 32; ++q) t += part[q][tx];
    if (dst_bf16) reinterpret_cast<bf16*>(dst)[c] = __float2bfloat16_rn(t);
    else reinterpret_cast<float*>(dst)[c] = t;
  }
}

// Column sums in two passes: pass 1 gives every block a 16-byte column
// vector per thread and a chunk of rows (coalesced: a warp reads 512
// consecutive bytes of a row, four rows in flight), writing fp32 partials
// [chunk][cols]; pass 2 adds the chunks in a fixed order.  Deterministic.
template <typename T>
__global__ void __launch_bounds__(256) colsum_part_kernel(const T* src, int64_t rows, int64_t cols,
                                                          int64_t ld, int64_t rows_per_chunk,
                                                          float* part) {
  constexpr int VE = 16 / (int)sizeof(T);
  const int64_t cv = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * VE;  // first column
  if (cv >= cols) return;
  const int64_t r0 = (int64_t)blockIdx.y * rows_per_chunk;
  const int64_t r1 = min(rows, r0 + rows_per_chunk);
  float acc[VE];
#pragma unroll
  for (int e = 0; e < VE; ++e) acc[e] = 0.f;
  int64_t r = r0;
  for (; r + 3 < r1; r += 4) {
    uint4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = __ldg(reinterpret_cast<const uint4*>(src + (r + q) * ld + cv));
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int e = 0; e < VE; ++e) acc[e] += sizeof(T) == 4 ? lane_f32(v[q], e) : lane_bf16(v[q], e);
  }
  for (; r < r1; ++r) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + r * ld + cv));
#pragma unroll
    for (int e = 0; e < VE; ++e) acc[e] += sizeof(T) == 4 ? lane_f32(v, e) : lane_bf16(v, e);
  }
  float* out = part + (int64_t)blockIdx.y * cols + cv;
#pragma unroll
  for (int e = 0; e < VE; ++e)
    if (cv + e < cols) out[e] = acc[e];
}

// pass 2: a block per 32 columns; warp w adds the chunks w, w + 8, ... of
// its lane's column (four loads in flight), then the eight warp sums are added
// in warp order: a fixed order, so the result is deterministic
__global__ void __launch_bounds__(256) colsum_final_kernel(const float* __restrict__ part,
                                                           int64_t chunks, int64_t cols, void* dst,
                                                           int dst_bf16) {
  __shared__ float red[8][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 32 + lane;
  float t = 0.f;
  if (c < cols) {
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    int64_t k = w;
    for (; k + 24 < chunks; k += 32) {
#pragma unroll
      for (int q = 0; q < 4; ++q) a[q] += __ldg(part + (k + 8 * q) * cols + c);
    }
    for (; k < chunks; k += 8) a[0] += __ldg(part + k * cols + c);
    t = (a[0] + a[1]) + (a[2] + a[3]);
  }
  red[w][lane] = t;
  __syncthreads();
  if (w == 0 && c < cols) {
    float u = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) u += red[q][lane];
    if (dst_bf16) reinterpret_cast<bf16*>(dst)[c] = __float2bfloat16_rn(u);
    else reinterpret_cast<float*>(dst)[c] = u;
  }
}

}  // namespace

std::atomic<int64_t> g_kernel_launches{0};

cudaError_t gemm_simt(const GemmArgs& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  KParams kp{};
  kp.M = g.M; kp.N = g.N;
  kp.seg[0] = Seg{g.A, g.sam, g.sak, g.B, g.sbk, g.sbn, g.K};
  kp.nseg = 1;
  if (g.K2 > 0 && g.A2 && g.B2) {
    kp.seg[1] = Seg{g.A2, g.sam2, g.sak2, g.B2, g.sbk2, g.sbn2, g.K2};
    kp.nseg = 2;
  }
  kp.C = g.C; kp.ldc = g.ldc;
  kp.bias1 = g.bias1; kp.bias2 = g.bias2; kp.bias2_limit = g.bias2_limit;
  kp.bias_bf16 = g.bias_bf16; kp.accumulate = g.accumulate;
  const bool a_km = g.sak == 1, b_km = g.sbk == 1;
  if (g.in_bf16) {
    return g.out_bf16 ? launch_typed<bf16, bf16>(kp, a_km, b_km, st)
                      : launch_typed<bf16, float>(kp, a_km, b_km, st);
  }
  return g.out_bf16 ? launch_typed<float, bf16>(kp, a_km, b_km, st)
                    : launch_typed<float, float>(kp, a_km, b_km, st);
}

cudaError_t colsum(void* dst, int dst_bf16, const void* src, int src_bf16, int64_t rows,
                   int64_t cols, int64_t ld, float* scratch, int64_t scratch_bytes,
                   int num_sms, cudaStream_t st) {
  if (cols <= 0) return cudaSuccess;
  const int e = src_bf16 ? 2 : 4;
  const int VE = 16 / e;
  const bool vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (ld * e) % 16 == 0 &&
                   cols % VE == 0;
  if (vec && scratch && rows > 0) {
    const int64_t vecs = cols / VE;
    const int64_t bx = (vecs + 255) / 256;
    // about four waves of blocks, at least 16 rows per chunk
    int64_t chunks = std::max<int64_t>(1, ((int64_t)num_sms * 4 + bx - 1) / bx);
    chunks = std::min<int64_t>(chunks, (rows + 15) / 16);
    while (chunks > 1 && chunks * cols * 4 > scratch_bytes) chunks /= 2;
    const int64_t rpc = (rows + chunks - 1) / chunks;
    chunks = (rows + rpc - 1) / rpc;
    dim3 grid((unsigned)bx, (unsigned)chunks);
    if (src_bf16)
      colsum_part_kernel<bf16><<<grid, 256, 0, st>>>(reinterpret_cast<const bf16*>(src), rows,
                                                     cols, ld, rpc, scratch);
    else
      colsum_part_kernel<float><<<grid, 256, 0, st>>>(reinterpret_cast<const float*>(src), rows,
                                                      cols, ld, rpc, scratch);
    colsum_final_kernel<<<(unsigned)((cols + 31) / 32), 256, 0, st>>>(scratch, chunks, cols, dst,
                                                                      dst_bf16);
    g_kernel_launches.fetch_add(2, std::memory_order_relaxed);
    return cudaGetLastError();
  }
  colsum_kernel<<<(unsigned)((cols + 31) / 32), 1024, 0, st>>>(dst, dst_bf16, src, src_bf16, rows,
                                                              cols, ld);
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

// Inter-layer dropout with given masks: buf[i] *= mask[i] * scale, in place
// (fp32 or bf16 elements; mask bytes are 0 or 1).  A select, not a product
// with the mask, so a dropped element is exactly zero whatever its value.
__global__ void dropout_kernel(void* buf, int bf16, const uint8_t* __restrict__ mask, int64_t n,
                               float scale) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool keep = __ldg(mask + i) != 0;
    if (bf16) {
      __nv_bfloat16* b = static_cast<__nv_bfloat16*>(buf);
      b[i] = __float2bfloat16_rn(keep ? __bfloat162float(b[i]) * scale : 0.f);
    } else {
      float* f = static_cast<float*>(buf);
      f[i] = keep ? f[i] * scale : 0.f;
    }
  }
}

__global__ void to_bf16_kernel(const float* src, int64_t rows, int64_t cols, int64_t lds,
                               bf16* dst) {
  const int64_t n = rows * cols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / cols, c = i - r * cols;
    dst[i] = __float2bfloat16_rn(src[r * lds + c]);
  }
}

cudaError_t to_bf16(const float* src, int64_t rows, int64_t cols, int64_t lds, void* dst,
                    int num_sms, cudaStream_t st) {
  const int64_t n = rows * cols;
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)std::max(1, num_sms) * 8);
  to_bf16_kernel<<<(unsigned)blocks, 256, 0, st>>>(src, rows, cols, lds,
                                                   reinterpret_cast<bf16*>(dst));
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

cudaError_t dropout_apply(void* buf, int bf16, const uint8_t* mask, int64_t n, float scale,
                          int num_sms, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)std::max(1, num_sms) * 8);
  dropout_kernel<<<(unsigned)blocks, 256, 0, st>>>(buf, bf16, mask, n, scale);
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

}  // namespace lr
