// Host-side declarations of the layer wavefront (recurrent_wf.cu).
#pragma once

#include "host_common.h"

namespace lr {

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
  // inter-layer dropout (training, every layer but the last): y holds this
  // layer's output dropped, bf16(bf16(h) * drop_scale) where the mask byte
  // [T][N][H] is nonzero, else 0, and the layer above reads its input from y
  const uint8_t* drop_mask = nullptr;
  float drop_scale = 1.f;
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
  // valid length of each sequence ([N] int32, device) or null: a step
  // t >= lengths[n] keeps sequence n's state and writes zero to y
  const int* lengths = nullptr;
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

}  // namespace lr
