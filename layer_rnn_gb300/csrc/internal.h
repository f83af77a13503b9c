// Host-side declarations shared by the translation units of liblayer_rnn.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace lr {

// kernels launched by this library (all handles, all threads); the phase
// timing of a handle reports its share per phase
extern std::atomic<int64_t> g_kernel_launches;

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
// A / B K-major (row stride lda / ldb elements); tf32 = 1: fp32 operands given
// as hi / lo splits (three passes), tf32 = 0: bf16 operands (one pass)
struct TcGemm {
  int64_t M = 0, N = 0, K = 0, K2 = 0;
  int tf32 = 1;
  const void* A_hi = nullptr; const void* A_lo = nullptr; int64_t lda = 0;
  const void* B_hi = nullptr; const void* B_lo = nullptr; int64_t ldb = 0;
  const void* A2_hi = nullptr; const void* A2_lo = nullptr; int64_t lda2 = 0;
  const void* B2_hi = nullptr; const void* B2_lo = nullptr; int64_t ldb2 = 0;
  void* C = nullptr; int64_t ldc = 0; int out_bf16 = 0; int accumulate = 0;
  const void* bias1 = nullptr; const void* bias2 = nullptr; int64_t bias2_limit = 0;
  int bias_bf16 = 0;
  int ksplit = 1; float* part = nullptr;  // split-K partials [ksplit][M][N]
  int* status = nullptr; long long timeout_ns = 2000000000LL;
};
bool gemm_tc_supported(const TcGemm& g);
cudaError_t gemm_tc(const TcGemm& g, cudaStream_t st);
// K splits worth using for an M x N output with K_total contraction length
int gemm_tc_splitk(int64_t M, int64_t N, int64_t K_total, bool tf32, int num_sms);
// fp32 [rows][cols] (row stride lds) -> hi / lo (lo may be null), [rows][cols]
// or transposed [cols][rows], row stride ldd
cudaError_t split_operand(const float* src, int64_t rows, int64_t cols, int64_t lds, float* hi,
                          float* lo, int64_t ldd, bool transpose, cudaStream_t st);
cudaError_t transpose_bf16(const void* src, int64_t rows, int64_t cols, int64_t lds, void* dst,
                           int64_t ldd, cudaStream_t st);

// column sums: dst[c] = sum_r src[r*ld + c], r < rows (fp32 accumulate, fixed
// order); with `scratch` (fp32 partials) in two coalesced passes
cudaError_t colsum(void* dst, int dst_bf16, const void* src, int src_bf16,
                   int64_t rows, int64_t cols, int64_t ld, float* scratch,
                   int64_t scratch_bytes, int num_sms, cudaStream_t st);
// buf[i] = mask[i] ? buf[i] * scale : 0 for i < n (inter-layer dropout)
cudaError_t dropout_apply(void* buf, int bf16, const uint8_t* mask, int64_t n, float scale,
                          int num_sms, cudaStream_t st);

// ---------------------------------------------------------------------------
// persistent recurrent kernels
// ---------------------------------------------------------------------------
struct RecDirArgs {
  // forward
  const float* gx = nullptr;     // [T][N][G*H] input projection + folded biases
  const void* whh = nullptr;     // canonical W_hh [G*H][H]
  const void* bhh = nullptr;     // canonical b_hh [G*H] (GRU: its n block is used)
  const void* h0 = nullptr;      // [N][H] or null (zeros)
  const float* c0 = nullptr;     // [N][H] or null (zeros)
  void* y = nullptr;             // layer output, row (t*N+n)*ldy, column d*H + j
  void* hseq = nullptr;          // [T+1][N][H] or null
  float* gates = nullptr;        // [T][N][Gs*H] or null
  float* cseq = nullptr;         // [T+1][N][H] or null
  void* hy = nullptr;            // [N][H] or null
  float* cy = nullptr;           // [N][H] or null
  // backward
  const void* dy = nullptr;      // row (t*N+n)*lddy, column d*H + j
  int dy_bf16 = 0;
  const void* dhy = nullptr;     // [N][H] or null
  const float* dcy = nullptr;    // [N][H] or null
  void* dgx = nullptr;           // [T][N][G*H] (compute type)
  void* dgh = nullptr;           // [T][N][G*H] (compute type), == dgx unless GRU
  void* dh0 = nullptr;           // [N][H] or null
  float* dc0 = nullptr;          // [N][H] or null
  // time order of this direction's arrays: 1 = reversed (a bidirectional
  // layer's second direction), 0 = forward, -1 = taken from the block's
  // direction index (both directions in one launch)
  int rev = -1;
};

struct RecPlan {
  int direct = 0;       // 1: per-warp dataflow path (one batch chunk)
  int tc = 0;           // 1: tensor-core forward (recurrent_tc.cu), 2: backward
                        // (recurrent_tc_bwd.cu), 3: batch-as-M backward (recurrent_tc_bwdm.cu)
  int shape = 0;        // register-tile shape id (see recurrent.cu)
  int P = 0;            // blocks per direction
  int U = 0;            // hidden units per block (last block may have fewer)
  int Mloc = 0, Mp = 0; // rows of the resident operand, padded to the tile
  int K = 0, lda = 0;   // contraction length, smem row stride (elements)
  int nb = 0, nbp = 0;  // batch chunk and its padded size
  int KC = 0, ldb = 0;  // K chunk of the staged operand and its smem row stride
                        // (direct path: in 16-byte vectors, per warp)
  int tiles_m = 0, tiles_n = 0, WK = 0;
  int nst = 1;          // direct path: staging stages per warp (1 or 2)
  // cluster path (cluster > 0): blocks of a cluster split K; block (r, q) of a
  // direction is cluster r, rank q
  int cluster = 0;      // blocks per cluster (K split); 0 = path not used
  int Pr = 0;           // clusters (row groups) per direction
  int Ur = 0, Uq = 0;   // units per row group; units per block in the pointwise
  int Kk = 0;           // K elements per cluster rank (multiple of 16 bytes)
  int Wm = 0, Wk = 0;   // warps along rows x along K inside a block
  int ldbs = 0;         // shared-memory row stride of the staged K slice (elements)
  // batch-as-M backward: TMA ring stages, pointwise inputs prefetched into
  // shared memory (1) or read in the pointwise step (0), partial-sum buffers
  int ring = 0, pin = 1, rbufs = 2;
  size_t smem = 0;
};

struct RecParams {
  int mode = 0, T = 0, N = 0, H = 0, G = 0, Gs = 0, D = 1;
  int bf16 = 0;
  int64_t ldy = 0, lddy = 0;
  RecPlan plan;
  unsigned* flags = nullptr;   // step flags of block b of direction d at
                               // flags[(d * P + b) * flag_stride], zeroed before the launch
  int flag_stride = 32;        // one flag per 128-byte line
  int spin_ns = 0;             // back-off between polls of a flag (0 = none)
  int* status = nullptr;
  long long timeout_ns = 0;
  int fault_block = -1, fault_step = -1;
  // valid length of each sequence ([N] int32, device), or null: every sequence
  // runs all T steps.  A step t >= lengths[n] keeps sequence n's state and
  // outputs zero (values outside 0..T act as 0 or T).  Only the staged
  // CUDA-core kernels (rec_make_plan with allow_direct = false) read it.
  const int* lengths = nullptr;
  RecDirArgs dir[2];
};

// Choose the tiling for the forward (backward = false) or backward kernel.
// Returns false when no supported tiling fits in shared memory.
// allow_direct = false: the staged kernel only (the one that reads lengths).
bool rec_make_plan(bool backward, int mode, int bf16, int D, int H, int N, int num_sms,
                   size_t smem_limit, RecPlan* out, bool allow_direct = true);

// Cluster path: plan (false if the problem does not qualify) and launch.
// max_clusters[c] = co-resident clusters of c blocks (c = 1, 2, 4, 8; 0 = unknown).
bool rec_cluster_plan(bool backward, int mode, int bf16, int D, int H, int N, int num_sms,
                      size_t smem_limit, const int* max_clusters, RecPlan* out);
cudaError_t rec_cluster_launch(bool backward, const RecParams& p, cudaStream_t st);
// Tensor-core forward path: plan (false if the problem does not qualify) and launch.
bool rec_tc_plan(int mode, int bf16, int D, int H, int N, int num_sms, size_t smem_limit,
                 const int* max_clusters, RecPlan* out);
cudaError_t rec_tc_launch(const RecParams& p, cudaStream_t st);
// co-resident clusters of `cluster` blocks of the cluster kernels with `smem` bytes
int rec_cluster_capacity(int cluster, size_t smem);
// Tensor-core backward path (recurrent_tc_bwd.cu): plan (false if the problem
// does not qualify; caps[c] = co-resident clusters of c blocks, c <= 16) and
// launch; capacity of its kernel for clusters of up to 16 blocks.
bool rec_tc_bwd_plan(int mode, int bf16, int D, int H, int N, int num_sms, size_t smem_limit,
                     const int* caps, RecPlan* out);
cudaError_t rec_tc_bwd_launch(const RecParams& p, cudaStream_t st);
int rec_tc_bwd_capacity(int cluster, size_t smem);
// Tensor-core backward with the batch as the MMA's M (recurrent_tc_bwdm.cu;
// bf16, batch 64..128): plan (false if the problem does not qualify) and launch.
bool rec_tcm_bwd_plan(int mode, int bf16, int D, int H, int N, int num_sms, size_t smem_limit,
                      const int* max_clusters, RecPlan* out);
cudaError_t rec_tcm_bwd_launch(const RecParams& p, cudaStream_t st);

// ---------------------------------------------------------------------------
// layer wavefront (unidirectional bf16 stacks): one persistent launch runs all
// layers; layer l step t overlaps layer l-1 step t+1 and later.  Per step each
// block contracts [x_t | h_{t-1}] (K = I_l + H) with its packed weight rows on
// the tensor cores, streaming both operands from L2 through a TMA ring.
// ---------------------------------------------------------------------------
constexpr int kWfMaxLayers = 8;

struct WfPlan {
  int Pr = 0;          // blocks (row groups) per layer
  int Ur = 0;          // hidden units per block
  int R = 0;           // packed rows per unit (4: LSTM i,f,g,o / GRU r,z,n_x,n_h; 1: tanh)
  int Nm = 0;          // MMA N (batch padded to 16)
  int stages = 0;      // TMA ring stages
  int tmem_cols = 0;
  size_t smem = 0;
};

struct WfLayer {
  const void* wp = nullptr;     // packed weights [Pr*R*Ur][kp] bf16 (x part, then h part)
  const float* bias = nullptr;  // packed per-row bias [Pr*R*Ur] fp32
  int64_t kp = 0;               // packed row length (elements)
  int nchx = 0, nch = 0;        // 64-element K chunks of the x part / in all
  const void* h0 = nullptr;     // [N][H] or null (zeros)
  const float* c0 = nullptr;    // [N][H] or null
  void* hseq = nullptr;         // [T+1][N][H] bf16, slot 0 = h0 (always written)
  void* y = nullptr;            // [T][N][H] layer output or null
  float* gates = nullptr;       // [T][N][Gs*H] or null
  float* cseq = nullptr;        // [T+1][N][H] or null
  void* hy = nullptr;           // [N][H] or null
  float* cy = nullptr;          // [N][H] or null
};

struct WfParams {
  int mode = 0, T = 0, N = 0, H = 0, I = 0, L = 0, Gs = 1;
  WfPlan plan;
  const void* x = nullptr;      // [T][N][I] bf16 (layer 0 input)
  unsigned* flags = nullptr;    // flag of block b at flags[b * flag_stride], zeroed at launch
  int flag_stride = 32;
  int* status = nullptr;
  long long timeout_ns = 0;
  int fault_block = -1, fault_step = -1;
  WfLayer layer[kWfMaxLayers];
};

// false when the problem does not qualify (then the layers run one by one)
bool wf_plan(int mode, int bf16, int L, int D, int64_t I, int64_t H, int64_t N, int num_sms,
             size_t smem_optin, WfPlan* out);
// upper bound of the packed weight and bias bytes of all layers, any device
int64_t wf_pack_bytes_bound(int mode, int L, int64_t I, int64_t H);
// packed K length of layer l (x part padded to 64, h part padded to 64)
int64_t wf_kp(int64_t I_l, int64_t H);
// pack layer l's canonical W_ih, W_hh, b_ih, b_hh into the plan's row order
cudaError_t wf_pack(const WfPlan& pl, int mode, int64_t I_l, int64_t H, const void* wih,
                    const void* whh, const void* bih, const void* bhh, void* wp, float* bias,
                    cudaStream_t st);
cudaError_t wf_launch(const WfParams& p, cudaStream_t st);
// encode a tiled TMA map (bf16 / fp32, rank 2 or 3, 128-byte swizzle)
bool tma_encode(void* map, int rank, bool bf, const void* ptr, const uint64_t* dims,
                const uint64_t* strides_bytes, const uint32_t* box);

// Launch (cooperative, so the whole grid is co-resident).  Zeroes the flags
// on the stream first.
cudaError_t rec_forward(const RecParams& p, cudaStream_t st);
cudaError_t rec_backward(const RecParams& p, cudaStream_t st);

}  // namespace lr
