/*
 * layer_rnn.h -- C ABI of liblayer_rnn.so, a fused multi-layer RNN operator
 * (tanh RNN, LSTM, GRU; stacked, optionally bidirectional) for one GB300 GPU.
 *
 * The operator follows the shape the pages give a fused RNN:
 *   - one operator for a whole multi-layer (optionally bidirectional) RNN
 *     ("Fused RNN operator for CPU", MXNet design page: Problem Statement and
 *     Operator Registration; the "CudnnLSTM(num_layers, num_units,
 *     input_size)" call quoted in Keras issue #3692);
 *   - a training forward that fills a workspace which the backward pass then
 *     reads ("rnn training example?", oneDNN issue #218: the six workspace
 *     steps -- create forward_training, query the workspace size, allocate it,
 *     pass it as an output of forward and as an input of backward);
 *   - PyTorch's tensor names and shapes (same issue: w_ih, w_hh, b_ih, b_hh
 *     and their gradients as separate tensors; hx / cx / hy / cy of shape
 *     (num_layers * num_directions, batch, hidden); input in TNC order).
 *
 * Recurrences (a = pre-activation, * = elementwise):
 *   tanh RNN: h' = tanh(W_ih x + b_ih + W_hh h + b_hh)
 *   LSTM    : gate blocks i, f, g, o;  c' = f*c + i*g;  h' = o*tanh(c')
 *   GRU     : gate blocks r, z, n (the PyTorch / cuDNN flavour of the oneDNN
 *             issue, "PyTorch equations"): n = tanh(W_in x + b_in +
 *             r*(W_hn h + b_hn)),  h' = (1-z)*n + z*h.
 * Direction 1 of a bidirectional layer walks t = T-1 .. 0 and writes its
 * output at the original time index; a layer's output is [fwd || bwd] along
 * features and feeds the next layer.
 *
 * Conventions for every call below
 *   - All tensors and the workspace are caller-owned DEVICE memory, dense,
 *     row-major, 16-byte aligned (the workspace 256-byte aligned); otherwise
 *     RNN_ERR_MISALIGNED.  Pointers of different arguments must not overlap,
 *     except that the weight buffer W may be shared by several calls.
 *   - x [T, N, I]; y, dy [T, N, D*H]; h0, hy, dh0, dhy, c0, cy, dc0, dcy
 *     [L*D, N, H] with index layer*D + direction.
 *   - Element types: RNN_F32 -> every tensor float32.  RNN_BF16 -> x, y, dy,
 *     dx, W, dW, h0, hy, dhy, dh0 are bfloat16; c0, cy, dcy, dc0 (cell
 *     state) are float32.  Accumulation and the cell state are float32
 *     internally in both.
 *   - Compute calls are asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and return after enqueueing.  Argument errors
 *     are returned before anything is enqueued.  A device-side failure (a
 *     step barrier that ran past its time limit) is recorded in a status word
 *     that rnn_check_status() returns; with RNN_FLAG_SYNC_CHECK every compute
 *     call synchronises and returns it itself.
 *   - One handle serves one stream at a time (it owns the step-barrier
 *     counters its kernels use).  No call allocates device memory except
 *     rnn_forward_inference (first call per (T, N) growth, see there),
 *     rnn_measure_step_protocol (a temporary buffer) and the first compute
 *     call of a handle (its 64 KB of step flags); rnn_forward_inference_static
 *     never allocates.
 */
#ifndef LAYER_RNN_H
#define LAYER_RNN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct rnn_handle* rnn_t;

/* RNN_GRU_TF: the GRU flavour with the reset gate applied before the
 * recurrent product of the candidate (TensorFlow's equations quoted in "rnn
 * training example?", oneDNN issue #218; oneDNN's linear_before_reset = 0):
 *   n = tanh(W_in x + b_in + W_hn (r*h) + b_hn), r, z and h' as RNN_GRU.
 * Same weight layout as RNN_GRU (gate blocks r, z, n).  Each step needs r
 * before the candidate's product, so it runs on the CUDA-core recurrent
 * kernels with two barriers per step (the dense phases still use the tensor
 * cores); the workspace's fourth gate slot keeps r*h for dW_hn. */
typedef enum { RNN_TANH = 0, RNN_LSTM = 1, RNN_GRU = 2, RNN_GRU_TF = 3 } rnn_mode_t;
typedef enum { RNN_F32 = 0, RNN_BF16 = 1 } rnn_dtype_t;

typedef enum {
  RNN_OK = 0,
  RNN_ERR_INVALID_ARG = 1,        /* bad mode/dtype/size, NULL required pointer  */
  RNN_ERR_UNSUPPORTED = 2,        /* valid but beyond what the kernels support   */
  RNN_ERR_WORKSPACE_TOO_SMALL = 3,
  RNN_ERR_MISALIGNED = 4,
  RNN_ERR_CUDA = 5,               /* a CUDA runtime call failed                  */
  RNN_ERR_TIMEOUT = 6,            /* a step barrier gave up waiting (device)     */
  RNN_ERR_NO_RESIDENCY = 7,       /* the persistent grid cannot be co-resident   */
  RNN_ERR_DEVICE_CHECK = 8        /* a kernel's own index check failed; the
                                     access was skipped (device)                */
} rnn_status_t;

/* flags for rnn_create */
#define RNN_FLAG_SYNC_CHECK 0x1u  /* each compute call synchronises `stream` and
                                     returns the device status word            */
#define RNN_FLAG_SIMT_GEMM  0x2u  /* dense phases on the CUDA-core GEMM instead
                                     of the tensor-core GEMM                    */
#define RNN_FLAG_SIMT_RECURRENT 0x4u  /* recurrent forward and backward on the
                                         CUDA-core kernels instead of the
                                         tensor-core ones                        */
#define RNN_FLAG_NO_WAVEFRONT 0x8u    /* unidirectional stacks run layer after
                                         layer instead of as one layer wavefront */

/* regions for rnn_workspace_layout */
typedef enum {
  RNN_WS_GATES = 0,   /* per (l,d): [T, N, G'*H] f32 saved activations; G' = 4 for
                         LSTM (i,f,g,o), GRU (r,z,n, W_hn h + b_hn) and TF-flavour
                         GRU (r,z,n, r*h), 1 for tanh RNN (h); time-indexed         */
  RNN_WS_CSEQ = 1,    /* per (l,d): [T+1, N, H] f32 cell states (LSTM only); slot
                         0 (dir 0) or T (dir 1) holds c0, slot t+1 / t holds c_t    */
  RNN_WS_HSEQ = 2,    /* per (l,d): [T+1, N, H] hidden states, same slots as CSEQ,
                         element type of h                                          */
  RNN_WS_YLAYER = 3,  /* per l < L-1: [T, N, D*H] layer output (next layer's input) */
  RNN_WS_DGX = 4,     /* per (l,d): [T, N, G*H] gate-gradients w.r.t. W_ih x + b_ih
                         (f32, or bf16 for RNN_BF16)                                */
  RNN_WS_DGH = 5,     /* per (l,d): [T, N, G*H] gate-gradients w.r.t. W_hh h + b_hh
                         (GRU only; equals DGX for LSTM / tanh RNN)                 */
  RNN_WS_GX = 6,      /* [D, T, N, G*H] f32 input projection scratch                */
  RNN_WS_DY = 7,      /* [2, T, N, D*H] f32 gradient ping-pong between layers       */
  RNN_WS_GEMM = 8,    /* tensor-core GEMM operand copies (K-major, fp32 hi/lo split)
                         and split-K partial sums; scratch between calls            */
  RNN_WS_NUM_REGIONS = 9
} rnn_ws_region_t;

/* phases for rnn_get_phase_times */
typedef enum {
  RNN_PHASE_INPUT_GEMM = 0,   /* G_x = X W_ih^T + b over all T (per layer)           */
  RNN_PHASE_REC_FWD = 1,      /* persistent recurrent forward (per layer)            */
  RNN_PHASE_REC_BWD = 2,      /* persistent recurrent backward (per layer)           */
  RNN_PHASE_DX_GEMM = 3,      /* dX = dG_x W_ih (per layer)                          */
  RNN_PHASE_DW_GEMM = 4,      /* dW_ih, dW_hh and db (per layer and direction)       */
  RNN_PHASE_NUM = 5
} rnn_phase_t;

/* Create a handle.  mode: rnn_mode_t; num_layers >= 1; bidirectional 0/1;
 * input_size, hidden_size >= 1; dtype: rnn_dtype_t; flags: RNN_FLAG_*.
 * Host only (no CUDA call).  *out is owned by the caller until rnn_destroy. */
rnn_status_t rnn_create(rnn_t* out, int mode, int num_layers, int bidirectional,
                        int64_t input_size, int64_t hidden_size, int dtype,
                        uint32_t flags);

/* Release the handle and the device memory it owns.  NULL is accepted.
 * Waits for nothing: the caller must have finished using it on the device. */
rnn_status_t rnn_destroy(rnn_t h);

/* Number of elements (of the handle's element type) of the canonical weight
 * buffer W / dW.  Host only. */
rnn_status_t rnn_weight_count(rnn_t h, int64_t* n_elems);

/* Canonical weight buffer layout.  For each (layer, dir) in order
 * layer*D + dir: W_ih [G*H, I_l] (which=0), W_hh [G*H, H] (1), b_ih [G*H] (2),
 * b_hh [G*H] (3), row-major and back to back; I_l = input_size for layer 0 and
 * D*H above.  Gate blocks along the G*H rows: LSTM i,f,g,o; GRU r,z,n; tanh
 * RNN one block -- the PyTorch order.  Returns the element offset and the
 * shape (cols = 1 for biases).  Host only. */
rnn_status_t rnn_weight_layout(rnn_t h, int layer, int dir, int which,
                               int64_t* offset, int64_t* rows, int64_t* cols);

/* Bytes of the training workspace for sequence length T and batch N
 * (forward_training writes it; backward_data and backward_weights read it,
 * backward_data also writes the gate-gradient regions; RNN_WS_GEMM is scratch
 * of every call).  Host only. */
rnn_status_t rnn_workspace_size(rnn_t h, int64_t T, int64_t N, int64_t* bytes);

/* Byte offset and size of one workspace region (rnn_ws_region_t) for
 * (layer, dir); per-layer regions ignore dir, global ones ignore both.
 * A region that does not exist for the mode reports bytes = 0.  Host only. */
rnn_status_t rnn_workspace_layout(rnn_t h, int64_t T, int64_t N, int region,
                                  int layer, int dir, int64_t* offset, int64_t* bytes);

/* Training forward: y = the top layer's output, hy / cy = final states, and
 * the workspace filled for the backward calls.  h0 / c0 NULL = zeros;
 * hy / cy NULL = not written; c0 / cy ignored unless LSTM. */
rnn_status_t rnn_forward_training(rnn_t h, void* stream, int64_t T, int64_t N,
                                  const void* x, const void* h0, const void* c0,
                                  const void* W, void* y, void* hy, void* cy,
                                  void* workspace, int64_t ws_bytes);

/* Inference forward: as rnn_forward_training without a workspace.  The
 * handle keeps device scratch for the input projection and the intermediate
 * layer outputs, allocated (cudaMalloc) when a call needs more than it has;
 * make one call per shape before capturing a CUDA graph. */
rnn_status_t rnn_forward_inference(rnn_t h, void* stream, int64_t T, int64_t N,
                                   const void* x, const void* h0, const void* c0,
                                   const void* W, void* y, void* hy, void* cy);

/* Inference forward that allocates nothing.  The pages have no counterpart of
 * this call: it exists for callers that cannot allocate device memory (a
 * memory pool that owns the device, an allocator that must not be re-entered,
 * a fixed memory budget), since rnn_forward_inference allocates its scratch on
 * first use.  Arguments, results and errors are those of
 * rnn_forward_inference.  All scratch -- step flags and status word, the input
 * projection, two intermediate layer outputs -- lives in one static device
 * array of 32 MiB per device, held by every GPU that loads the library until
 * the process exits.  A call needs 65536 + A(D*T*N*G*H*4) + D*A(24*N*H)
 * bytes, plus 2*A(T*N*D*H*elem) when num_layers > 1 (A = round up to 256,
 * elem = 4 for RNN_F32, 2 for RNN_BF16); larger problems return
 * RNN_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress); make
 * that first call before any stream capture.  Every call on a device shares
 * the array and leaves its contents behind: calls that overlap on the GPU
 * (other streams, other handles) race and must be serialised by the caller.
 * The array has its own status word.  Each call clears it first; a barrier
 * timeout of the call is returned by the call itself when the handle has
 * RNN_FLAG_SYNC_CHECK, else by the next rnn_check_status on that device
 * (which reads and clears it too) before the next static call.  A handle
 * already bound to another device returns RNN_ERR_INVALID_ARG. */
rnn_status_t rnn_forward_inference_static(rnn_t h, void* stream, int64_t T, int64_t N,
                                          const void* x, const void* h0, const void* c0,
                                          const void* W, void* y, void* hy, void* cy);

/* Backward through time for the data: dx (and dh0, dc0) of the loss
 * sum(y*dy) + sum(hy*dhy) + sum(cy*dcy).  Needs the workspace of the
 * matching rnn_forward_training (same T, N, W), writes its DGX / DGH / DY
 * regions.  dhy / dcy NULL = zeros; dh0 / dc0 NULL = not written. */
rnn_status_t rnn_backward_data(rnn_t h, void* stream, int64_t T, int64_t N,
                               const void* W, const void* dy, const void* dhy,
                               const void* dcy, void* dx, void* dh0, void* dc0,
                               void* workspace, int64_t ws_bytes);

/* Weight gradients dW (canonical layout, overwritten -- not accumulated):
 * dW_ih = sum_t dG_x[t]^T x_t, dW_hh = sum_t dG_h[t]^T h_{t-1}, db_ih =
 * sum dG_x, db_hh = sum dG_h.  Must follow rnn_backward_data on the same
 * workspace.  x is the forward input.  h0 and y may be NULL: the workspace
 * already holds the hidden-state sequences.  The call reads the workspace and
 * overwrites only its RNN_WS_GEMM region (scratch of every call). */
rnn_status_t rnn_backward_weights(rnn_t h, void* stream, int64_t T, int64_t N,
                                  const void* x, const void* h0, const void* y,
                                  const void* workspace, int64_t ws_bytes, void* dW);

/* Variable-length (padded) batches.  The same calls with one more argument,
 * lengths: device memory, N int32 values, the valid length of each sequence
 * of the padded [T, N, ...] batch (the PyTorch packed-sequence layout after
 * unpacking to TNC, which "rnn training example?" (oneDNN issue #218) raises
 * as the way such batches arrive).  Semantics, per sequence n and direction:
 * a step t >= lengths[n] leaves the state unchanged and writes zero output,
 * so y is zero past the length, hy / cy are the state after the last valid
 * step, and the reverse direction starts from h0 at step lengths[n] - 1.
 * rnn_backward_data_varlen is the derivative of that: dy past a sequence's
 * length is ignored, and its gate gradients are zero.  rnn_backward_weights
 * needs no lengths (the zero gate gradients drop the padded steps); the padded
 * entries of x must be finite, because dW_ih multiplies them by zero.
 * Values outside 0..T act as 0 or T.  The lengths buffer is read by the
 * enqueued kernels: keep it unchanged until they have run.  The recurrent
 * phases run on the layer wavefront and the tensor-core kernels where those
 * fit (rnn_get_paths_varlen names the choice), else on the staged CUDA-core
 * kernels; the dense phases use the tensor cores as without lengths.
 * Errors: as the calls without lengths, and RNN_ERR_INVALID_ARG for a NULL
 * lengths, RNN_ERR_MISALIGNED for one not 4-byte aligned. */
rnn_status_t rnn_forward_training_varlen(rnn_t h, void* stream, int64_t T, int64_t N,
                                         const int32_t* lengths, const void* x,
                                         const void* h0, const void* c0, const void* W,
                                         void* y, void* hy, void* cy, void* workspace,
                                         int64_t ws_bytes);
rnn_status_t rnn_forward_inference_varlen(rnn_t h, void* stream, int64_t T, int64_t N,
                                          const int32_t* lengths, const void* x,
                                          const void* h0, const void* c0, const void* W,
                                          void* y, void* hy, void* cy);
rnn_status_t rnn_backward_data_varlen(rnn_t h, void* stream, int64_t T, int64_t N,
                                      const int32_t* lengths, const void* W, const void* dy,
                                      const void* dhy, const void* dcy, void* dx, void* dh0,
                                      void* dc0, void* workspace, int64_t ws_bytes);

/* Inter-layer dropout in training, as cuDNN has it (the ask of "rnn training
 * example?", oneDNN issue #218).  The same calls with the dropout
 * probability p in [0, 1) and masks: device memory, (L-1) x [T, N, D*H]
 * bytes, each 0 (dropped) or 1, one block per layer boundary (the caller
 * draws them).  The output of layer l < L-1 becomes layer l+1's input
 * multiplied by mask_l / (1 - p); y, hy and cy are not dropped.
 * rnn_backward_data_dropout must get the same p and masks.
 * rnn_backward_weights needs neither, because the workspace keeps the dropped
 * inputs.  Inference does not drop.  For L = 1, masks may be NULL.  The
 * forward takes the same recurrent kernels as rnn_forward_training (the layer
 * wavefront applies the masks as each layer writes its output).  The masks
 * buffer is read by the enqueued kernels: keep it unchanged until they have
 * run.
 * Errors: as the calls without dropout, and RNN_ERR_INVALID_ARG for p outside
 * [0, 1) or NULL masks with L > 1. */
rnn_status_t rnn_forward_training_dropout(rnn_t h, void* stream, int64_t T, int64_t N,
                                          float dropout, const uint8_t* masks, const void* x,
                                          const void* h0, const void* c0, const void* W,
                                          void* y, void* hy, void* cy, void* workspace,
                                          int64_t ws_bytes);
rnn_status_t rnn_backward_data_dropout(rnn_t h, void* stream, int64_t T, int64_t N,
                                       float dropout, const uint8_t* masks, const void* W,
                                       const void* dy, const void* dhy, const void* dcy,
                                       void* dx, void* dh0, void* dc0, void* workspace,
                                       int64_t ws_bytes);

/* Synchronise `stream`, then return and clear the device status word
 * (RNN_OK, RNN_ERR_TIMEOUT or RNN_ERR_DEVICE_CHECK): the handle's own, and,
 * once rnn_forward_inference_static has run on the current device, that
 * call's (synchronise the stream it ran on first). */
rnn_status_t rnn_check_status(rnn_t h, void* stream);

/* Test hook for failure detection.  timeout_ns > 0 sets the step-barrier
 * time limit (default 2 s).  fault_block >= 0 makes that block of the next
 * persistent launches skip its barrier arrival at step fault_step, so every
 * waiting block runs into the time limit, records RNN_ERR_TIMEOUT and
 * returns (no trap, no unbounded wait).  fault_block = -1 disables. */
rnn_status_t rnn_set_debug(rnn_t h, int fault_block, int fault_step, int64_t timeout_ns);

/* Per-phase timing with CUDA events recorded on the launching stream.
 * enable = 1 starts recording (and zeroes the totals), 0 stops. */
rnn_status_t rnn_enable_phase_timing(rnn_t h, int enable);

/* Synchronise the events recorded so far and return, per rnn_phase_t, the
 * summed milliseconds between the events bracketing the phase and the number
 * of kernels the library launched inside it (arrays of RNN_PHASE_NUM). */
rnn_status_t rnn_get_phase_times(rnn_t h, double* ms, int64_t* launches);

/* Kernels the recurrent phases of a call with batch N run on this device
 * (the choice depends on the sizes, the flags and the device).  Sets up the
 * handle's device state like a compute call; enqueues nothing.
 *   *fwd: RNN_PATH_* of the recurrent forward; *bwd: of the backward. */
typedef enum {
  RNN_PATH_STAGED = 0,     /* CUDA-core, per-block slice in shared memory      */
  RNN_PATH_DIRECT = 1,     /* CUDA-core, per-warp dataflow                     */
  RNN_PATH_CLUSTER = 2,    /* CUDA-core, cluster K split over DSMEM            */
  RNN_PATH_TENSOR = 3,     /* tcgen05, slice in tensor memory, cluster K split */
  RNN_PATH_WAVEFRONT = 4   /* tcgen05 layer wavefront, all layers in one launch */
} rnn_path_t;
rnn_status_t rnn_get_paths(rnn_t h, int64_t N, int* fwd, int* bwd);
/* The same for the *_varlen calls (per-sequence lengths): the layer
 * wavefront and the tensor-core kernels read the lengths where they fit,
 * else the staged CUDA-core kernels run the recurrent phases. */
rnn_status_t rnn_get_paths_varlen(rnn_t h, int64_t N, int* fwd, int* bwd);

/* The step protocol of the tensor-core recurrent forward, timed alone.  The
 * pages have no counterpart of this call: it measures the part of a
 * recurrent step's latency that no arithmetic removes, the term a latency
 * bound of the recurrence adds to the time of streaming W_hh and of the MMA.
 * It runs `steps` (2 .. 2^20) empty steps of the forward kernel's protocol for
 * batch N with one direction -- the same grid and clusters, each block
 * writing the exchange words of its units and polling those of its K slice,
 * one block barrier, one push per owner that completes the owner's receive
 * barrier and the owners' wait for it, with no MMA and no gate math -- once to warm
 * up and once between two CUDA events on `stream`, synchronises `stream`, and
 * returns the average microseconds per step.  It allocates (cudaMalloc) and
 * frees a temporary exchange buffer of 24*N*H bytes and uses the handle's
 * status word.  RNN_ERR_UNSUPPORTED when the forward of batch N does not run
 * on the tensor-core recurrent kernel; a wait that runs out of time returns
 * RNN_ERR_TIMEOUT. */
rnn_status_t rnn_measure_step_protocol(rnn_t h, void* stream, int64_t N, int64_t steps,
                                       double* us_per_step);

/* Test hooks for the packed operand forms.  The pages have no counterpart:
 * the forms are this library's own (the "matrix pre-transposition" of the
 * cuDNN table in Keras issue #3692 names the idea, not a layout).  Each runs
 * the library's packing kernel asynchronously on `stream` into caller
 * buffers, so a test can check that the packing loses and invents nothing.
 *
 * rnn_debug_split_f16: the scaled fp16 pairs of the dense phases' fp32
 * operands.  src [rows][cols] (row stride lds floats) -> hi, lo (fp16)
 * [rows][cols] (transpose = 0) or [cols][rows] (transpose = 1), row stride
 * ldd elements; *maxbits (a 4-byte device word) receives the largest |value|
 * as its float bit pattern.  With s = 2^(13 - E), E the binary exponent of
 * that largest magnitude (s = 1 when it is 0 or not finite; 13 - E clamped
 * to [-126, 126]): hi = fp16(value * s) and lo = fp16(value * s - hi), both
 * rounded to nearest even, so hi + lo equals value * s within 2^-22 of it
 * (down to the fp16 subnormal range).
 *
 * rnn_debug_transpose_bf16: the K-major bf16 operand copy of the dense
 * phases.  src [rows][cols] (row stride lds elements) -> dst [cols][rows]
 * (row stride ldd elements), bit for bit.
 *
 * rnn_debug_wf_pack: the layer wavefront's packed rows of one layer (bf16
 * handles of a unidirectional stack with 2..8 layers only, as the wavefront;
 * RNN_ERR_UNSUPPORTED otherwise) for batch N, from the canonical buffer W.
 * layout[0..4] receives Pr (blocks of the layer), Ur (units per block), R
 * (packed rows per unit: 4 for LSTM i, f, g, o and GRU r, z, n_x, n_h; 1 for
 * tanh), kp (packed row length, elements) and Kxp (the x part's padded
 * length).  Row (r*Ur + u)*R + g of wp [Pr*Ur*R][kp] bf16 is, for unit
 * j = r*Ur + u < H: [W_ih row of gate g of unit j | zeros to Kxp | W_hh row |
 * zeros to kp], with the GRU's n_x row taking only W_in and its n_h row only
 * W_hn (n_h is W_hn's row in the h part, zeros in the x part); bias[row] (fp32)
 * = b_ih + b_hh of that row (GRU: b_in on n_x, b_hn on n_h).  Rows of units
 * j >= H are zero.  wp_bytes / bias_bytes are the buffers' sizes:
 * RNN_ERR_WORKSPACE_TOO_SMALL when they are short. */
rnn_status_t rnn_debug_split_f16(const float* src, int64_t rows, int64_t cols, int64_t lds,
                                 void* hi, void* lo, int64_t ldd, int transpose, unsigned* maxbits,
                                 void* stream);
rnn_status_t rnn_debug_transpose_bf16(const void* src, int64_t rows, int64_t cols, int64_t lds,
                                      void* dst, int64_t ldd, void* stream);
rnn_status_t rnn_debug_wf_pack(rnn_t h, void* stream, int64_t N, int layer, const void* W,
                               void* wp, int64_t wp_bytes, float* bias, int64_t bias_bytes,
                               int64_t* layout);

/* Test hook for the dense phases' launch shape (host only; no device is
 * touched).  For C[M][N] over a contraction of K_total on num_sms SMs, with
 * scaled fp16 pairs (split16 = 1, fp32 operands) or bf16 (0), K splits
 * allowed or not (allow_split), *bn receives the output tile width (64, 128,
 * 160, 192 or 256 columns; tiles are 128 rows) and *ksplit the number of K splits
 * that the library's wave model picks: per tile and 64-element K block the
 * larger of the MMA time and the operand feed, times ceil(tiles * ksplit /
 * num_sms) waves, plus a fixed cost per tile and wave and the split's partial
 * sums.  A GEMM of more than one wave whose fp32 result is written whole is
 * then re-planned for 2 * num_sms (two CTAs per SM); this hook gives the
 * plan for the num_sms it is asked about.
 * Errors: RNN_ERR_INVALID_ARG for M, N or K_total < 1, num_sms < 1 or a
 * NULL output. */
rnn_status_t rnn_debug_gemm_shape(int64_t M, int64_t N, int64_t K_total, int split16, int num_sms,
                                  int allow_split, int* bn, int* ksplit);

/* Static description of the status code. */
const char* rnn_status_string(rnn_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* LAYER_RNN_H */
