// Host-side declarations of the persistent recurrent kernels (recurrent*.cu).
#pragma once

#include "host_common.h"

namespace lr {

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
  // tensor-core kernels: exchange words of the step outputs the other blocks
  // read, value bits | step << 32 -- forward h [3][N][H]
  // (rec_tc_xchg_bytes(N, H) bytes), backward dG_h [3][N][G*H]
  // (rec_tc_xchg_bytes(N, G*H) bytes)
  unsigned long long* hx = nullptr;
  // staged kernels, TensorFlow-flavour GRU (mode 3): the direction's exchange
  // rows of the second contraction of each step -- forward r * h_{t-1} [N][H],
  // backward [N][G*H] (da_r, da_z, da_n) -- in the storage type
  void* xbuf = nullptr;
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
  int mode = 0, T = 0, N = 0, H = 0, G = 0, Gs = 0, D = 1;  // mode: rnn_mode_t
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
  // outputs zero (values outside 0..T act as 0 or T).  The tensor-core
  // kernels (forward, backward, batch-as-M backward) and the staged CUDA-core
  // kernels (rec_make_plan with allow_direct = false) read it; the direct and
  // cluster kernels do not.
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
// bytes of one direction's exchange words of a tensor-core recurrent kernel
// whose step output is [N][width] (forward width = H, backward G*H)
size_t rec_tc_xchg_bytes(int N, int width);
// The tensor-core forward's step protocol with no work (flag waits, cluster
// barrier, flag release), p.T steps, same plan and grid as rec_tc_launch.
cudaError_t rec_tc_probe_launch(const RecParams& p, cudaStream_t st);
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

// Launch (cooperative, so the whole grid is co-resident).  Zeroes the flags
// on the stream first.
cudaError_t rec_forward(const RecParams& p, cudaStream_t st);
cudaError_t rec_backward(const RecParams& p, cudaStream_t st);

}  // namespace lr
