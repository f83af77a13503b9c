// Host-side declarations of the dense phases (gemm_simt.cu, gemm_tc.cu).
#pragma once

#include "host_common.h"

namespace lr {

// ---------------------------------------------------------------------------
// dense phases: C[M, N] (+)= A[M, K] B[K, N] (+ A2 B2) + bias
// ---------------------------------------------------------------------------
struct GemmArgs {
  int64_t M = 0, N = 0, K = 0;
  const void* A = nullptr; int64_t sam = 0, sak = 0;   // A(m, k) = A[m*sam + k*sak]
  const void* B = nullptr; int64_t sbk = 0, sbn = 0;   // B(k, n) = B[k*sbk + n*sbn]
  // optional second product over K2 accumulated into the same result
  int64_t K2 = 0;
  const void* A2 = nullptr; int64_t sam2 = 0, sak2 = 0;
  const void* B2 = nullptr; int64_t sbk2 = 0, sbn2 = 0;
  void* C = nullptr; int64_t ldc = 0;                  // C(m, n) = C[m*ldc + n]
  const void* bias1 = nullptr;                         // + bias1[n]
  const void* bias2 = nullptr; int64_t bias2_limit = 0;  // + bias2[n] for n < limit
  int in_bf16 = 0;    // A, B (and A2, B2) element type
  int out_bf16 = 0;   // C element type
  int bias_bf16 = 0;  // bias element type
  int accumulate = 0; // C += result instead of C = result
  int no_split = 0;   // never split K (the result must not depend on scratch room)
};

cudaError_t gemm_simt(const GemmArgs& g, cudaStream_t st);

// tensor-core GEMM: C[M][N] (+)= sum_k A[m][k] B[n][k] (+ second product),
// A / B K-major (row stride lda / ldb elements, 16-bit); split16 = 1: fp32
// operands given as scaled fp16 (hi, lo) pairs (three passes; amax / bmax: the
// largest |A| over both products, the largest |B|, as float bit patterns),
// split16 = 0: bf16 operands (one pass)
struct TcGemm {
  int64_t M = 0, N = 0, K = 0, K2 = 0;
  int split16 = 1;
  const unsigned* amax = nullptr; const unsigned* bmax = nullptr;
  const void* A_hi = nullptr; const void* A_lo = nullptr; int64_t lda = 0;
  const void* B_hi = nullptr; const void* B_lo = nullptr; int64_t ldb = 0;
  const void* A2_hi = nullptr; const void* A2_lo = nullptr; int64_t lda2 = 0;
  const void* B2_hi = nullptr; const void* B2_lo = nullptr; int64_t ldb2 = 0;
  void* C = nullptr; int64_t ldc = 0; int out_bf16 = 0; int accumulate = 0;
  const void* bias1 = nullptr; const void* bias2 = nullptr; int64_t bias2_limit = 0;
  int bias_bf16 = 0;
  int bn = 0;  // output tile width (64, 128, 160, 192, 256; 0: chosen by the wave model)
  int ctas_per_sm = 1;  // 2: a smaller ring, two CTAs per SM (fp32 C or partials only)
  int ksplit = 1; float* part = nullptr;  // split-K partials [ksplit][M][N]
  int* status = nullptr; long long timeout_ns = 2000000000LL;
};
bool gemm_tc_supported(const TcGemm& g);
cudaError_t gemm_tc(const TcGemm& g, cudaStream_t st);
// tile width and K split for an M x N output with K_total contraction length
// (allow_split = false: one split)
void gemm_tc_shape(int64_t M, int64_t N, int64_t K_total, bool split16, int num_sms,
                   bool allow_split, int* bn, int* ksplit);
// largest |x| of fp32 [rows][cols] (row stride lds) into *mx (atomicMax of the
// float bit pattern: the caller zeroes *mx first; several operands may share it)
cudaError_t absmax_operand(const float* src, int64_t rows, int64_t cols, int64_t lds,
                           unsigned* mx, int num_sms, cudaStream_t st);
// fp32 [rows][cols] (row stride lds) -> scaled fp16 pairs hi / lo, [rows][cols]
// or transposed [cols][rows], row stride ldd, with the scale of the largest
// magnitude *mx (written by absmax_operand before)
cudaError_t split_f16_operand(const float* src, int64_t rows, int64_t cols, int64_t lds, void* hi,
                              void* lo, int64_t ldd, bool transpose, const unsigned* mx,
                              cudaStream_t st);
cudaError_t transpose_bf16(const void* src, int64_t rows, int64_t cols, int64_t lds, void* dst,
                           int64_t ldd, cudaStream_t st);

// column sums: dst[c] = sum_r src[r*ld + c], r < rows (fp32 accumulate, fixed
// order); with `scratch` (fp32 partials) in two coalesced passes
cudaError_t colsum(void* dst, int dst_bf16, const void* src, int src_bf16,
                   int64_t rows, int64_t cols, int64_t ld, float* scratch,
                   int64_t scratch_bytes, int num_sms, cudaStream_t st);
// dst [rows][cols] bf16 (round to nearest even) <- src [rows][cols] fp32 with
// row stride lds
cudaError_t to_bf16(const float* src, int64_t rows, int64_t cols, int64_t lds, void* dst,
                    int num_sms, cudaStream_t st);
// buf[i] = mask[i] ? buf[i] * scale : 0 for i < n (inter-layer dropout)
cudaError_t dropout_apply(void* buf, int bf16, const uint8_t* mask, int64_t n, float scale,
                          int num_sms, cudaStream_t st);

}  // namespace lr
