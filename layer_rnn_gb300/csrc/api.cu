// C ABI of liblayer_rnn.so: handle, argument checks, weight and workspace
// layouts, and the order of the phases of each call.  See include/layer_rnn.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/layer_rnn.h"
#include "internal.h"

using namespace lr;

struct PhaseMark {
  int phase;
  int64_t kernels;
  cudaEvent_t start, stop;
};

struct rnn_handle {
  int mode = 0, L = 1, D = 1, dtype = 0, G = 1, Gs = 1;
  int64_t I = 0, H = 0;
  uint32_t flags = 0;
  // device state, set up by the first compute call
  int device = -1;
  int num_sms = 0;
  size_t smem_optin = 0;
  int max_clusters[9] = {0};   // co-resident clusters of 1..8 blocks (cluster kernels)
  int bwd_caps[17] = {0};      // co-resident clusters of up to 16 blocks (tensor-core backward)
  size_t cluster_smem = 0;     // largest dynamic shared memory at which clusters fit
  unsigned* d_sync = nullptr;  // step flags (one per 128-byte line), status word at the end
  int* d_status = nullptr;
  void* scratch = nullptr;     // inference scratch
  size_t scratch_bytes = 0;
  // debug / failure-detection hook
  long long timeout_ns = 2000000000LL;
  int fault_block = -1, fault_step = -1;
  // phase timing
  bool timing = false;
  std::vector<PhaseMark> marks;
  double ms[RNN_PHASE_NUM] = {0};
  int64_t launches[RNN_PHASE_NUM] = {0};
};

namespace {

constexpr size_t kSyncBytes = 65536;  // step flags (128 B apart) and, at the end, the status word

int64_t esize(const rnn_handle* h) { return h->dtype == RNN_BF16 ? 2 : 4; }
int64_t layer_in(const rnn_handle* h, int l) { return l == 0 ? h->I : h->D * h->H; }

// ----------------------------------------------------------------------------
// canonical weight layout
// ----------------------------------------------------------------------------
int64_t weight_block(const rnn_handle* h, int l) {
  const int64_t GH = h->G * h->H;
  return GH * layer_in(h, l) + GH * h->H + 2 * GH;
}

int64_t weight_count(const rnn_handle* h) {
  int64_t n = 0;
  for (int l = 0; l < h->L; ++l) n += h->D * weight_block(h, l);
  return n;
}

// element offset of tensor `which` of (l, d)
int64_t weight_offset(const rnn_handle* h, int l, int d, int which) {
  int64_t off = 0;
  for (int k = 0; k < l; ++k) off += h->D * weight_block(h, k);
  off += d * weight_block(h, l);
  const int64_t GH = h->G * h->H;
  const int64_t sizes[4] = {GH * layer_in(h, l), GH * h->H, GH, GH};
  for (int w = 0; w < which; ++w) off += sizes[w];
  return off;
}

// ----------------------------------------------------------------------------
// workspace layout
// ----------------------------------------------------------------------------
struct Region {
  int64_t off = 0, bytes = 0;
};

struct WsLayout {
  std::vector<Region> r;  // indexed [region][l][d]
  int L = 0, D = 0;
  int64_t total = 0;
  Region& at(int region, int l, int d) { return r[((size_t)region * L + l) * D + d]; }
};

int64_t align256(int64_t v) { return (v + 255) / 256 * 256; }

// ----------------------------------------------------------------------------
// tensor-core GEMM operands: every operand is presented K-major with 16-bit
// elements; fp32 operands as scaled fp16 (hi, lo) pairs; copies live in a
// scratch region
// ----------------------------------------------------------------------------
constexpr int kMaxKsplit = 8;

int64_t kpad(int64_t K) { return (K + 7) / 8 * 8; }  // 16-byte rows

// bytes of one operand copy: rows x K (hi and lo for fp32)
int64_t opnd_bytes(int64_t rows, int64_t K, bool f32) {
  return align256(rows * kpad(K) * 2) * (f32 ? 2 : 1);
}

// whether a call may take the layer-wavefront path (host-side conditions; the
// device-dependent plan can still decline)
bool wf_candidate(const rnn_handle* h, int64_t N) {
  return h->dtype == RNN_BF16 && h->mode != RNN_GRU_TF && h->D == 1 && h->L >= 2 &&
         h->L <= kWfMaxLayers && N <= 128 &&
         h->H % 8 == 0 && h->I % 8 == 0 &&
         !(h->flags & (RNN_FLAG_NO_WAVEFRONT | RNN_FLAG_SIMT_RECURRENT));
}

// scratch of the wavefront path: packed weights and biases, plus (inference)
// the per-layer hidden-state sequences the layers read from one another
int64_t wf_scratch_bytes(const rnn_handle* h, int64_t T, int64_t N, bool training) {
  if (!wf_candidate(h, N)) return 0;
  int64_t b = wf_pack_bytes_bound(h->mode, h->L, h->I, h->H);
  if (!training) b += h->L * align256((T + 1) * N * h->H * 2);
  return b + 4096;
}

// exchange words of the tensor-core recurrent forward (every direction), taken
// from the front of a call's scratch
int64_t xchg_bytes(const rnn_handle* h, int64_t N) {
  return h->D * align256((int64_t)rec_tc_xchg_bytes((int)N, (int)(h->G * h->H)));
}

// scratch the GEMM phases of one call need (maximum over the phases)
int64_t gemm_scratch_bytes(const rnn_handle* h, int64_t T, int64_t N, bool training) {
  const bool tf = h->dtype != RNN_BF16;
  const int64_t GH = h->G * h->H, TN = T * N, D = h->D;
  int64_t need = 0;
  for (int l = 0; l < h->L; ++l) {
    const int64_t I_l = l == 0 ? h->I : D * h->H;
    // input projection: X [TN][I_l] and W_ih [GH][I_l], both K-major already
    if (tf) need = std::max(need, opnd_bytes(TN, I_l, tf) + opnd_bytes(GH, I_l, tf));
    if (!training) continue;
    // dX: dG [TN][GH] per direction, W_ih transposed [I_l][GH] per direction
    need = std::max(need, D * ((tf ? opnd_bytes(TN, GH, tf) : 0) + opnd_bytes(I_l, GH, tf)) +
                              align256((int64_t)kMaxKsplit * TN * I_l * 4));
    // dW_ih, dW_hh: dG^T [GH][TN] (two for GRU), X^T [I_l][TN], h_prev^T [H][TN]
    const int64_t dgt = opnd_bytes(GH, TN, tf) * (h->mode == RNN_GRU ? 2 : 1);
    need = std::max(need, dgt + opnd_bytes(std::max(I_l, h->H), TN, tf) +
                              align256((int64_t)kMaxKsplit * GH * std::max(I_l, h->H) * 4));
  }
  // the TensorFlow-flavour GRU's bf16 copy of r * h_{t-1} for dW_hn
  const int64_t rh_copy = (training && h->mode == RNN_GRU_TF && !tf) ? align256(TN * h->H * 2) : 0;
  return std::max(need, wf_scratch_bytes(h, T, N, training)) + 4096 + xchg_bytes(h, N) + rh_copy;
}

struct Scratch {
  char* base = nullptr;
  int64_t cap = 0, off = 0;
  void* take(int64_t bytes) {
    const int64_t o = align256(off);
    if (!base || o + bytes > cap) return nullptr;
    off = o + bytes;
    return base + o;
  }
};

// Largest magnitude of an fp32 GEMM operand given by strides (element (r, k)
// at p[r * sr + k * sk], K-major or stored transposed) into *mx (atomicMax: a
// word zeroed before, possibly shared with another operand).
bool operand_absmax(const void* p, int64_t rows, int64_t K, int64_t sr, int64_t sk, unsigned* mx,
                    int num_sms, cudaStream_t st) {
  const float* f = static_cast<const float*>(p);
  const cudaError_t e = sk == 1 ? absmax_operand(f, rows, K, sr, mx, num_sms, st)
                                : absmax_operand(f, K, rows, sk, mx, num_sms, st);
  return e == cudaSuccess;
}

// One GEMM operand given by strides as a K-major TcGemm operand; copies into
// `sc` when needed (fp32: scaled fp16 pairs with the scale of *mx).  false:
// cannot.
bool prep_operand(const void* p, int64_t rows, int64_t K, int64_t sr, int64_t sk, bool tf,
                  Scratch* sc, const void** hi, const void** lo, int64_t* ld, const unsigned* mx,
                  cudaStream_t st) {
  const int64_t kp = kpad(K);
  if (tf) {
    void* h = sc->take(align256(rows * kp * 2));
    void* l = sc->take(align256(rows * kp * 2));
    if (!h || !l || !mx) return false;
    const bool kmaj = sk == 1;
    const float* f = static_cast<const float*>(p);
    cudaError_t e = kmaj ? split_f16_operand(f, rows, K, sr, h, l, kp, false, mx, st)
                         : split_f16_operand(f, K, rows, sk, h, l, kp, true, mx, st);
    if (e != cudaSuccess) return false;
    *hi = h;
    *lo = l;
    *ld = kp;
    return true;
  }
  if (sk == 1 && (reinterpret_cast<uintptr_t>(p) % 16 == 0) && (sr * 2) % 16 == 0) {
    *hi = p;
    *lo = nullptr;
    *ld = sr;
    return true;
  }
  if (sr != 1) return false;
  void* t = sc->take(align256(rows * kp * 2));
  if (!t) return false;
  if (transpose_bf16(p, K, rows, sk, t, kp, st) != cudaSuccess) return false;
  *hi = t;
  *lo = nullptr;
  *ld = kp;
  return true;
}

// A dense phase: tensor-core GEMM when the operands can be presented to it
// (alignment, scratch room), otherwise the CUDA-core GEMM.
// A GEMM operand already presented K-major (and split for fp32) in scratch,
// reused by the GEMMs that share it (dW_ih and dW_hh both read dG_x^T unless
// the mode is GRU)
struct PreparedA {
  bool valid = false;
  const void* src = nullptr;
  int64_t M = 0, K = 0, sam = 0, sak = 0;
  const void* hi = nullptr;
  const void* lo = nullptr;
  int64_t ld = 0;
  const unsigned* mx = nullptr;  // fp32: its largest magnitude
};

// a zeroed word for an operand's largest magnitude, from the scratch
unsigned* take_max_word(Scratch* sc, cudaStream_t st) {
  unsigned* mx = static_cast<unsigned*>(sc->take(256));
  if (mx && cudaMemsetAsync(mx, 0, 8, st) != cudaSuccess) return nullptr;
  return mx;
}

// A prepared for reuse by several GEMMs (fp32: split with its own scale)
bool prepare_a(const rnn_handle* h, PreparedA* pa, bool tf, Scratch* sc, cudaStream_t st) {
  if (tf) {
    unsigned* mx = take_max_word(sc, st);
    if (!mx || !operand_absmax(pa->src, pa->M, pa->K, pa->sam, pa->sak, mx, h->num_sms, st))
      return false;
    pa->mx = mx;
  }
  return prep_operand(pa->src, pa->M, pa->K, pa->sam, pa->sak, tf, sc, &pa->hi, &pa->lo, &pa->ld,
                      pa->mx, st);
}

// Below this many multiply-adds a dense phase runs on the CUDA cores: the
// tensor-core path's operand preparation (max and split kernels, fp32) costs
// more launches than the product is worth (a 5-step, batch-2 LSTM ran about
// 20 % slower end to end with it)
constexpr int64_t kTinyGemmMacs = int64_t(1) << 20;

rnn_status_t run_gemm(const rnn_handle* h, const GemmArgs& g, Scratch sc, cudaStream_t st,
                      const PreparedA* pa = nullptr) {
  const bool tiny = g.M * g.N * (g.K + g.K2) < kTinyGemmMacs;
  if (!(h->flags & RNN_FLAG_SIMT_GEMM) && !tiny) {
    const bool tf = !g.in_bf16;
    TcGemm t;
    t.M = g.M; t.N = g.N; t.K = g.K; t.split16 = tf ? 1 : 0;
    const bool reuse = pa && pa->valid && pa->src == g.A && pa->M == g.M && pa->K == g.K &&
                       pa->sam == g.sam && pa->sak == g.sak && g.K2 == 0;
    if (reuse) {
      t.A_hi = pa->hi;
      t.A_lo = pa->lo;
      t.lda = pa->ld;
    }
    bool ok = true;
    unsigned* mx = nullptr;  // fp32: [0] largest |A| (and |A2|), [1] largest |B| (and |B2|)
    if (tf) {
      mx = take_max_word(&sc, st);
      ok = mx != nullptr;
      if (ok && !reuse) ok = operand_absmax(g.A, g.M, g.K, g.sam, g.sak, mx, h->num_sms, st);
      if (ok) ok = operand_absmax(g.B, g.N, g.K, g.sbn, g.sbk, mx + 1, h->num_sms, st);
      if (ok && g.K2 > 0)
        ok = operand_absmax(g.A2, g.M, g.K2, g.sam2, g.sak2, mx, h->num_sms, st) &&
             operand_absmax(g.B2, g.N, g.K2, g.sbn2, g.sbk2, mx + 1, h->num_sms, st);
      t.amax = reuse ? pa->mx : mx;
      t.bmax = mx ? mx + 1 : nullptr;
    }
    ok = ok &&
         (reuse ||
          prep_operand(g.A, g.M, g.K, g.sam, g.sak, tf, &sc, &t.A_hi, &t.A_lo, &t.lda, mx, st)) &&
         prep_operand(g.B, g.N, g.K, g.sbn, g.sbk, tf, &sc, &t.B_hi, &t.B_lo, &t.ldb,
                      mx ? mx + 1 : nullptr, st);
    if (ok && g.K2 > 0) {
      t.K2 = g.K2;
      ok = prep_operand(g.A2, g.M, g.K2, g.sam2, g.sak2, tf, &sc, &t.A2_hi, &t.A2_lo, &t.lda2, mx,
                        st) &&
           prep_operand(g.B2, g.N, g.K2, g.sbn2, g.sbk2, tf, &sc, &t.B2_hi, &t.B2_lo, &t.ldb2,
                        mx ? mx + 1 : nullptr, st);
    }
    if (ok) {
      t.C = g.C; t.ldc = g.ldc; t.out_bf16 = g.out_bf16; t.accumulate = g.accumulate;
      t.bias1 = g.bias1; t.bias2 = g.bias2; t.bias2_limit = g.bias2_limit;
      t.bias_bf16 = g.bias_bf16;
      t.status = h->d_status;
      t.timeout_ns = h->timeout_ns;
      int ks = 1;
      gemm_tc_shape(g.M, g.N, g.K + g.K2, tf, h->num_sms, !g.no_split, &t.bn, &ks);
      // more than one wave with an fp32 result written whole: two CTAs per SM
      // (measured at the DS2 shapes: input projection 0.128 -> 0.118 ms, dX
      // 0.153 -> 0.138 ms; the one-wave weight gradients were slower so)
      const int64_t units = ((g.M + 127) / 128) * ((g.N + t.bn - 1) / t.bn) * ks;
      if (tf && !g.out_bf16 && !g.accumulate && units > h->num_sms) {
        t.ctas_per_sm = 2;
        gemm_tc_shape(g.M, g.N, g.K + g.K2, tf, 2 * h->num_sms, !g.no_split, &t.bn, &ks);
      }
      if (ks > 1) {
        t.part = static_cast<float*>(sc.take(ks * g.M * g.N * 4));
        if (t.part) t.ksplit = ks;
      }
      if (gemm_tc_supported(t)) return gemm_tc(t, st) == cudaSuccess ? RNN_OK : RNN_ERR_CUDA;
    }
  }
  return gemm_simt(g, st) == cudaSuccess ? RNN_OK : RNN_ERR_CUDA;
}

WsLayout ws_layout(const rnn_handle* h, int64_t T, int64_t N) {
  WsLayout w;
  w.L = h->L;
  w.D = h->D;
  w.r.assign((size_t)RNN_WS_NUM_REGIONS * h->L * h->D, Region());
  const int64_t e = esize(h), H = h->H, G = h->G, D = h->D;
  int64_t off = 0;
  auto put = [&](int region, int l, int d, int64_t bytes) {
    Region& R = w.at(region, l, d);
    R.off = bytes > 0 ? off : 0;
    R.bytes = bytes;
    off += align256(bytes);
  };
  for (int l = 0; l < h->L; ++l)
    for (int d = 0; d < h->D; ++d) {
      put(RNN_WS_GATES, l, d, T * N * h->Gs * H * 4);
      put(RNN_WS_CSEQ, l, d, h->mode == RNN_LSTM ? (T + 1) * N * H * 4 : 0);
      put(RNN_WS_HSEQ, l, d, (T + 1) * N * H * e);
      put(RNN_WS_DGX, l, d, T * N * G * H * e);
      put(RNN_WS_DGH, l, d, h->mode == RNN_GRU ? T * N * G * H * e : 0);
    }
  for (int l = 0; l < h->L; ++l) put(RNN_WS_YLAYER, l, 0, l < h->L - 1 ? T * N * D * H * e : 0);
  put(RNN_WS_GX, 0, 0, D * T * N * G * H * 4);
  put(RNN_WS_DY, 0, 0, h->L > 1 ? 2 * T * N * D * H * 4 : 0);
  put(RNN_WS_GEMM, 0, 0, gemm_scratch_bytes(h, T, N, true));
  w.total = off;
  return w;
}

// ----------------------------------------------------------------------------
// checks and device set-up
// ----------------------------------------------------------------------------
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

rnn_status_t check_sizes(const rnn_handle* h, int64_t T, int64_t N) {
  if (!h) return RNN_ERR_INVALID_ARG;
  if (T < 1 || N < 1) return RNN_ERR_INVALID_ARG;
  if (T > (1 << 24) || N > (1 << 20)) return RNN_ERR_UNSUPPORTED;
  // 32-bit index products inside the kernels
  if (T * N * std::max<int64_t>(h->G * h->H * 4, std::max(h->I, h->D * h->H)) > (int64_t(1) << 31))
    return RNN_ERR_UNSUPPORTED;
  return RNN_OK;
}

// Clusters need a little shared memory of each SM for themselves: find the
// largest per-block size at which a cluster of 2 still fits, and the number of
// co-resident clusters of 2, 4 and 8 blocks at that size.  No allocation.
void query_clusters(int optin, size_t* cluster_smem, int* max_clusters) {
  *cluster_smem = 0;
  for (int c = 0; c < 9; ++c) max_clusters[c] = 0;
  for (size_t sm : {(size_t)optin, (size_t)optin - 1024, (size_t)optin - 4096,
                    (size_t)optin - 16384, (size_t)200 * 1024}) {
    if (rec_cluster_capacity(2, sm) > 0) {
      *cluster_smem = sm;
      break;
    }
  }
  if (*cluster_smem)
    for (int c : {2, 4, 8}) max_clusters[c] = rec_cluster_capacity(c, *cluster_smem);
}

rnn_status_t device_setup(rnn_handle* h) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RNN_ERR_CUDA;
  if (h->device == dev && h->d_sync) return RNN_OK;
  if (h->device >= 0 && h->device != dev) return RNN_ERR_INVALID_ARG;  // one device per handle
  int sms = 0, optin = 0, coop = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
    return RNN_ERR_CUDA;
  if (!coop) return RNN_ERR_UNSUPPORTED;
  void* p = nullptr;
  if (cudaMalloc(&p, kSyncBytes) != cudaSuccess) return RNN_ERR_CUDA;
  if (cudaMemset(p, 0, kSyncBytes) != cudaSuccess) {
    cudaFree(p);
    return RNN_ERR_CUDA;
  }
  h->d_sync = static_cast<unsigned*>(p);
  h->d_status = reinterpret_cast<int*>(static_cast<char*>(p) + kSyncBytes - 64);
  h->device = dev;
  h->num_sms = sms;
  h->smem_optin = (size_t)optin;
  query_clusters(optin, &h->cluster_smem, h->max_clusters);
  for (int c : {4, 8, 12, 14, 16}) h->bwd_caps[c] = rec_tc_bwd_capacity(c, 120 * 1024);
  return RNN_OK;
}

rnn_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return RNN_OK;
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();
    return RNN_ERR_NO_RESIDENCY;
  }
  return RNN_ERR_CUDA;
}

// read a device status word and clear it when it holds a failure
rnn_status_t take_status_word(int* word) {
  int v = 0;
  if (cudaMemcpy(&v, word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return RNN_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return RNN_ERR_CUDA;
  }
  return (rnn_status_t)v;
}

rnn_status_t read_status(rnn_handle* h, cudaStream_t st) {
  if (cudaStreamSynchronize(st) != cudaSuccess) return RNN_ERR_CUDA;
  if (!h->d_status) return RNN_OK;
  return take_status_word(h->d_status);
}

rnn_status_t finish(rnn_handle* h, cudaStream_t st, rnn_status_t s) {
  if (s != RNN_OK) return s;
  if (h->flags & RNN_FLAG_SYNC_CHECK) return read_status(h, st);
  return RNN_OK;
}

// phase timing helpers
struct PhaseScope {
  rnn_handle* h;
  cudaStream_t st;
  PhaseMark m;
  bool on;
  PhaseScope(rnn_handle* hh, cudaStream_t s, int phase) : h(hh), st(s), on(hh->timing) {
    if (!on) return;
    m.phase = phase;
    m.kernels = g_kernel_launches.load();
    cudaEventCreate(&m.start);
    cudaEventCreate(&m.stop);
    cudaEventRecord(m.start, st);
  }
  ~PhaseScope() {
    if (!on) return;
    cudaEventRecord(m.stop, st);
    m.kernels = g_kernel_launches.load() - m.kernels;
    h->marks.push_back(m);
  }
};

// Kernel choice for D directions in one launch (D = 1 also for one direction
// of a bidirectional layer run on its own).
rnn_status_t plan_rec(rnn_handle* h, bool backward, int64_t N, RecPlan* pl, int D,
                      bool varlen = false) {
  const bool bf = h->dtype == RNN_BF16;
  // per-sequence lengths: the tensor-core kernels (the forward, both backward
  // kernels) and the staged CUDA-core kernels read them
  if (varlen && h->mode != RNN_GRU_TF && !(h->flags & RNN_FLAG_SIMT_RECURRENT)) {
    if (!backward && rec_tc_plan(h->mode, bf, D, (int)h->H, (int)N, h->num_sms, h->cluster_smem,
                                 h->max_clusters, pl))
      return RNN_OK;
    if (backward &&
        rec_tcm_bwd_plan(h->mode, bf, D, (int)h->H, (int)N, h->num_sms, h->cluster_smem,
                         h->max_clusters, pl) &&
        (size_t)pl->P * D * 128 <= kSyncBytes - 64)
      return RNN_OK;
    if (backward &&
        rec_tc_bwd_plan(h->mode, bf, D, (int)h->H, (int)N, h->num_sms, h->smem_optin,
                        h->bwd_caps, pl) &&
        (size_t)pl->P * D * 128 <= kSyncBytes - 64)
      return RNN_OK;
  }
  if (varlen || h->mode == RNN_GRU_TF) {
    // the TensorFlow-flavour GRU's two dependent contractions per step, and
    // lengths where no tensor-core plan fits: the staged CUDA-core kernels
    // (the TensorFlow-flavour GRU has the GRU's sizes: three gate blocks)
    if (!rec_make_plan(backward, h->mode == RNN_GRU_TF ? RNN_GRU : h->mode, bf, D, (int)h->H,
                       (int)N, h->num_sms, h->smem_optin, pl, false))
      return RNN_ERR_UNSUPPORTED;
    if (pl->P * D > h->num_sms) return RNN_ERR_NO_RESIDENCY;
    if ((size_t)pl->P * D * 128 > kSyncBytes - 64) return RNN_ERR_UNSUPPORTED;
    return RNN_OK;
  }
  if (!backward && !(h->flags & RNN_FLAG_SIMT_RECURRENT) &&
      rec_tc_plan(h->mode, bf, D, (int)h->H, (int)N, h->num_sms, h->cluster_smem,
                  h->max_clusters, pl))
    return RNN_OK;
  if (backward && !(h->flags & RNN_FLAG_SIMT_RECURRENT) &&
      rec_tcm_bwd_plan(h->mode, bf, D, (int)h->H, (int)N, h->num_sms, h->cluster_smem,
                       h->max_clusters, pl) &&
      (size_t)pl->P * D * 128 <= kSyncBytes - 64)
    return RNN_OK;
  if (backward && !(h->flags & RNN_FLAG_SIMT_RECURRENT) &&
      rec_tc_bwd_plan(h->mode, bf, D, (int)h->H, (int)N, h->num_sms, h->smem_optin,
                      h->bwd_caps, pl) &&
      (size_t)pl->P * D * 128 <= kSyncBytes - 64)
    return RNN_OK;
  if (!rec_cluster_plan(backward, h->mode, bf, D, (int)h->H, (int)N, h->num_sms,
                        h->cluster_smem, h->max_clusters, pl) &&
      !rec_make_plan(backward, h->mode, bf, D, (int)h->H, (int)N, h->num_sms, h->smem_optin,
                     pl))
    return RNN_ERR_UNSUPPORTED;
  if (pl->P * D > h->num_sms) return RNN_ERR_NO_RESIDENCY;
  if ((size_t)pl->P * D * 128 > kSyncBytes - 64) return RNN_ERR_UNSUPPORTED;
  return RNN_OK;
}

rnn_status_t plan_rec(rnn_handle* h, bool backward, int64_t N, RecPlan* pl) {
  return plan_rec(h, backward, N, pl, h->D);
}

// Backward of a bidirectional LSTM layer: when both directions together only
// fit a CUDA-core kernel, the two directions run one after the other, each on
// the tensor-core plan for one direction (5-layer bidirectional LSTM: 24 us
// per step for the pair against 2 x 7 us).  GRU and tanh-RNN layers measured
// no better this way.
bool bwd_directions_in_turn(rnn_handle* h, int64_t N, const RecPlan& both, RecPlan* one,
                            bool varlen) {
  if (h->D != 2 || both.tc || h->mode != RNN_LSTM || (h->flags & RNN_FLAG_SIMT_RECURRENT))
    return false;
  return plan_rec(h, true, N, one, 1, varlen) == RNN_OK && one->tc;
}

// Forward of a bidirectional layer: when both directions together only fit a
// CUDA-core kernel, the two directions run one after the other, each on the
// tensor-core plan for one direction (5-layer bidirectional LSTM at H = 800:
// 2 x 3.6 us per step against 13.2 us for the pair on the cluster kernel).
bool fwd_directions_in_turn(rnn_handle* h, int64_t N, const RecPlan& both, RecPlan* one,
                            bool varlen) {
  if (h->D != 2 || both.tc || h->mode == RNN_GRU_TF || (h->flags & RNN_FLAG_SIMT_RECURRENT))
    return false;
  return plan_rec(h, false, N, one, 1, varlen) == RNN_OK && one->tc;
}

void fill_rec_common(rnn_handle* h, int64_t T, int64_t N, RecParams* rp) {
  rp->mode = h->mode;
  rp->T = (int)T;
  rp->N = (int)N;
  rp->H = (int)h->H;
  rp->G = h->G;
  rp->Gs = h->Gs;
  rp->D = h->D;
  rp->bf16 = h->dtype == RNN_BF16;
  rp->flags = h->d_sync;
  rp->status = h->d_status;
  rp->timeout_ns = h->timeout_ns;
  rp->fault_block = h->fault_block;
  rp->fault_step = h->fault_step;
#ifdef LAYER_RNN_TRACE
  if (const char* v = getenv("LAYER_RNN_FLAG_STRIDE")) rp->flag_stride = atoi(v);
  if (const char* v = getenv("LAYER_RNN_SPIN_NS")) rp->spin_ns = atoi(v);
#endif
}

template <typename P>
const P* cp(const void* base, int64_t byte_off) {
  return reinterpret_cast<const P*>(static_cast<const char*>(base) + byte_off);
}
template <typename P>
P* mp(void* base, int64_t byte_off) {
  return reinterpret_cast<P*>(static_cast<char*>(base) + byte_off);
}

// G_x[d] = in W_ih[l,d]^T + b_ih + b_hh (GRU: b_hn stays in the recurrence)
rnn_status_t input_projection(rnn_handle* h, cudaStream_t st, int l, int64_t T, int64_t N,
                              const void* in, const void* W, float* gx, Scratch sc) {
  const int64_t e = esize(h), GH = h->G * h->H, I_l = layer_in(h, l);
  for (int d = 0; d < h->D; ++d) {
    GemmArgs g;
    g.M = T * N; g.N = GH; g.K = I_l;
    g.A = in; g.sam = I_l; g.sak = 1;
    g.B = cp<char>(W, weight_offset(h, l, d, 0) * e); g.sbk = 1; g.sbn = I_l;
    g.C = gx + (int64_t)d * T * N * GH; g.ldc = GH;
    g.bias1 = cp<char>(W, weight_offset(h, l, d, 2) * e);
    g.bias2 = cp<char>(W, weight_offset(h, l, d, 3) * e);
    // GRU: b_hn stays inside r * (W_hn h + b_hn); the TensorFlow flavour's
    // b_hn is outside its product and folds like the others
    g.bias2_limit = h->mode == RNN_GRU ? 2 * h->H : GH;
    g.in_bf16 = g.bias_bf16 = h->dtype == RNN_BF16;
    g.out_bf16 = 0;
    // training and inference (different scratch room) must produce the same
    // G_x bit for bit: one fixed summation order, no K split
    g.no_split = 1;
    rnn_status_t s = run_gemm(h, g, sc, st);
    if (s != RNN_OK) return s;
  }
  return RNN_OK;
}

// Layer wavefront (unidirectional bf16 stacks): all layers in one persistent
// launch.  *used = false (and nothing enqueued) when the problem or the scratch
// does not qualify; the layers then run one after another.
rnn_status_t forward_wavefront(rnn_handle* h, cudaStream_t st, int64_t T, int64_t N,
                               const void* x, const void* h0, const void* c0, const void* W,
                               void* y, void* hy, void* cy, char* ws, bool training, Scratch sc,
                               bool* used, const int* lengths = nullptr,
                               const uint8_t* drop_masks = nullptr, float drop_p = 0.f) {
  *used = false;
  if (!wf_candidate(h, N)) return RNN_OK;
  if (drop_masks && !training) return RNN_OK;
  WfPlan pl;
  if (!wf_plan(h->mode, 1, h->L, h->D, h->I, h->H, N, h->num_sms, h->smem_optin, &pl))
    return RNN_OK;
  if ((size_t)h->L * pl.Pr * 128 > kSyncBytes - 64) return RNN_OK;
  const int64_t H = h->H, NH = N * H, e = 2;
  WfParams p;
  p.mode = h->mode;
  p.T = (int)T;
  p.N = (int)N;
  p.H = (int)H;
  p.I = (int)h->I;
  p.L = h->L;
  p.Gs = h->Gs;
  p.plan = pl;
  p.x = x;
  p.flags = h->d_sync;
  p.status = h->d_status;
  p.timeout_ns = h->timeout_ns;
  p.fault_block = h->fault_block;
  p.fault_step = h->fault_step;
  p.lengths = lengths;
  WsLayout lay;
  if (training) lay = ws_layout(h, T, N);
  const int64_t rows = (int64_t)pl.Pr * pl.R * pl.Ur;
  for (int l = 0; l < h->L; ++l) {
    WfLayer& a = p.layer[l];
    const int64_t I_l = layer_in(h, l);
    a.kp = wf_kp(I_l, H);
    a.nchx = (int)((I_l + 63) / 64);
    a.nch = (int)(a.kp / 64);
    a.wp = sc.take(align256(rows * a.kp * 2));
    a.bias = static_cast<float*>(sc.take(align256(rows * 4)));
    if (!a.wp || !a.bias) return RNN_OK;
    if (training) {
      a.hseq = mp<char>(ws, lay.at(RNN_WS_HSEQ, l, 0).off);
      a.gates = mp<float>(ws, lay.at(RNN_WS_GATES, l, 0).off);
      a.cseq = h->mode == RNN_LSTM ? mp<float>(ws, lay.at(RNN_WS_CSEQ, l, 0).off) : nullptr;
      a.y = l == h->L - 1 ? y : mp<char>(ws, lay.at(RNN_WS_YLAYER, l, 0).off);
    } else {
      a.hseq = sc.take(align256((T + 1) * NH * e));
      if (!a.hseq) return RNN_OK;
      a.y = l == h->L - 1 ? y : nullptr;
    }
    a.h0 = h0 ? cp<char>(h0, l * NH * e) : nullptr;
    a.c0 = (c0 && h->mode == RNN_LSTM) ? cp<float>(c0, l * NH * 4) : nullptr;
    a.hy = hy ? mp<char>(hy, l * NH * e) : nullptr;
    a.cy = (cy && h->mode == RNN_LSTM) ? mp<float>(cy, l * NH * 4) : nullptr;
    if (drop_masks && l < h->L - 1) {
      // this layer's output reaches the next layer dropped
      a.drop_mask = drop_masks + (int64_t)l * T * NH;
      a.drop_scale = 1.f / (1.f - drop_p);
    }
  }
  *used = true;
  {
    PhaseScope ps(h, st, RNN_PHASE_INPUT_GEMM);
    for (int l = 0; l < h->L; ++l) {
      WfLayer& a = p.layer[l];
      const cudaError_t ce =
          wf_pack(pl, h->mode, layer_in(h, l), H, cp<char>(W, weight_offset(h, l, 0, 0) * e),
                  cp<char>(W, weight_offset(h, l, 0, 1) * e),
                  cp<char>(W, weight_offset(h, l, 0, 2) * e),
                  cp<char>(W, weight_offset(h, l, 0, 3) * e), const_cast<void*>(a.wp),
                  const_cast<float*>(a.bias), st);
      if (ce != cudaSuccess) return RNN_ERR_CUDA;
    }
  }
  PhaseScope ps(h, st, RNN_PHASE_REC_FWD);
  return cuda_status(wf_launch(p, st));
}

// lengths: per-sequence valid lengths (device [N] int32) or null.  With
// lengths, inference needs hseq_scratch: D * (T+1) * N * H elements for the
// carried states.
rnn_status_t forward_impl(rnn_handle* h, cudaStream_t st, int64_t T, int64_t N, const void* x,
                          const void* h0, const void* c0, const void* W, void* y, void* hy,
                          void* cy, char* ws, bool training, Scratch sc,
                          const int* lengths = nullptr, char* hseq_scratch = nullptr,
                          const uint8_t* drop_masks = nullptr, float drop_p = 0.f) {
  const int64_t e = esize(h), H = h->H, NH = N * H;
  WsLayout lay = ws_layout(h, T, N);
  float* gx;
  void* ybuf[2] = {nullptr, nullptr};
  if (training) {
    gx = mp<float>(ws, lay.at(RNN_WS_GX, 0, 0).off);
  } else {
    gx = static_cast<float*>(h->scratch);
    const int64_t gx_bytes = align256(h->D * T * N * h->G * H * 4);
    const int64_t yb = align256(T * N * h->D * H * e);
    ybuf[0] = mp<char>(h->scratch, gx_bytes);
    ybuf[1] = mp<char>(h->scratch, gx_bytes + yb);
  }
  bool wf_used = false;
  rnn_status_t s = RNN_OK;
  {  // the wavefront chains the layers inside one launch
    s = forward_wavefront(h, st, T, N, x, h0, c0, W, y, hy, cy, ws, training, sc, &wf_used,
                          lengths, drop_masks, drop_p);
    if (wf_used || s != RNN_OK) return s;
  }
  RecPlan plan, plan_one;
  s = plan_rec(h, false, N, &plan, h->D, lengths != nullptr);
  if (s != RNN_OK) return s;
  const bool in_turn = fwd_directions_in_turn(h, N, plan, &plan_one, lengths != nullptr);
  unsigned long long* hx[2] = {nullptr, nullptr};
  if (plan.tc || in_turn) {
    for (int d = 0; d < h->D; ++d) {
      hx[d] = static_cast<unsigned long long*>(sc.take(rec_tc_xchg_bytes((int)N, (int)H)));
      if (!hx[d]) return RNN_ERR_WORKSPACE_TOO_SMALL;
    }
  }
  void* xrows[2] = {nullptr, nullptr};
  if (h->mode == RNN_GRU_TF) {
    for (int d = 0; d < h->D; ++d) {
      xrows[d] = sc.take(N * H * e);
      if (!xrows[d]) return RNN_ERR_WORKSPACE_TOO_SMALL;
    }
  }
  const void* in = x;
  for (int l = 0; l < h->L; ++l) {
    void* out;
    if (l == h->L - 1) out = y;
    else if (training) out = mp<char>(ws, lay.at(RNN_WS_YLAYER, l, 0).off);
    else out = ybuf[l & 1];
    {
      PhaseScope ps(h, st, RNN_PHASE_INPUT_GEMM);
      s = input_projection(h, st, l, T, N, in, W, gx, sc);
      if (s != RNN_OK) return s;
    }
    RecParams rp;
    fill_rec_common(h, T, N, &rp);
    rp.plan = plan;
    rp.ldy = h->D * H;
    rp.lengths = lengths;
    for (int d = 0; d < h->D; ++d) {
      RecDirArgs& a = rp.dir[d];
      const int k = l * h->D + d;
      a.gx = gx + (int64_t)d * T * N * h->G * H;
      a.whh = cp<char>(W, weight_offset(h, l, d, 1) * e);
      a.bhh = cp<char>(W, weight_offset(h, l, d, 3) * e);
      a.h0 = h0 ? cp<char>(h0, k * NH * e) : nullptr;
      a.c0 = (c0 && h->mode == RNN_LSTM) ? cp<float>(c0, k * NH * 4) : nullptr;
      a.y = out;
      a.hx = hx[d];
      a.xbuf = xrows[d];
      a.hy = hy ? mp<char>(hy, k * NH * e) : nullptr;
      a.cy = (cy && h->mode == RNN_LSTM) ? mp<float>(cy, k * NH * 4) : nullptr;
      if (training) {
        a.hseq = mp<char>(ws, lay.at(RNN_WS_HSEQ, l, d).off);
        a.gates = mp<float>(ws, lay.at(RNN_WS_GATES, l, d).off);
        a.cseq = h->mode == RNN_LSTM ? mp<float>(ws, lay.at(RNN_WS_CSEQ, l, d).off) : nullptr;
      } else if (lengths && !plan.tc && !in_turn) {
        // the staged kernels read the carried states back from here
        a.hseq = hseq_scratch + (int64_t)d * (T + 1) * NH * e;
      }
    }
    {
      PhaseScope ps(h, st, RNN_PHASE_REC_FWD);
      if (in_turn) {
        // one launch per direction; the second runs its time order reversed
        // and writes its half of y
        for (int d = 0; d < 2 && s == RNN_OK; ++d) {
          RecParams r1 = rp;
          r1.plan = plan_one;
          r1.D = 1;
          r1.dir[0] = rp.dir[d];
          r1.dir[0].rev = d;
          r1.dir[0].y = static_cast<char*>(out) + (int64_t)d * H * e;
          s = cuda_status(rec_tc_launch(r1, st));
        }
      } else {
        s = cuda_status(rp.plan.tc        ? rec_tc_launch(rp, st)
                        : rp.plan.cluster ? rec_cluster_launch(false, rp, st)
                                          : rec_forward(rp, st));
      }
      if (s != RNN_OK) return s;
    }
    if (drop_masks && l < h->L - 1) {
      // the next layer reads this layer's output dropped (in place: the
      // recurrent kernels keep their own copy of the states)
      const int64_t n = T * N * h->D * H;
      s = cuda_status(dropout_apply(out, h->dtype == RNN_BF16, drop_masks + (int64_t)l * n, n,
                                    1.f / (1.f - drop_p), h->num_sms, st));
      if (s != RNN_OK) return s;
    }
    in = out;
  }
  return RNN_OK;
}


}  // namespace

// ============================================================================
// exported
// ============================================================================
extern "C" {

rnn_status_t rnn_create(rnn_t* out, int mode, int num_layers, int bidirectional,
                        int64_t input_size, int64_t hidden_size, int dtype, uint32_t flags) {
  if (!out) return RNN_ERR_INVALID_ARG;
  *out = nullptr;
  if (mode < RNN_TANH || mode > RNN_GRU_TF) return RNN_ERR_INVALID_ARG;
  if (num_layers < 1 || (bidirectional != 0 && bidirectional != 1)) return RNN_ERR_INVALID_ARG;
  if (input_size < 1 || hidden_size < 1) return RNN_ERR_INVALID_ARG;
  if (dtype != RNN_F32 && dtype != RNN_BF16) return RNN_ERR_INVALID_ARG;
  if ((flags & ~(RNN_FLAG_SYNC_CHECK | RNN_FLAG_SIMT_GEMM | RNN_FLAG_SIMT_RECURRENT |
                 RNN_FLAG_NO_WAVEFRONT)) != 0)
    return RNN_ERR_INVALID_ARG;
  if (hidden_size > 65536 || input_size > (int64_t(1) << 24) || num_layers > 1024)
    return RNN_ERR_UNSUPPORTED;
  rnn_handle* h = new (std::nothrow) rnn_handle();
  if (!h) return RNN_ERR_INVALID_ARG;
  h->mode = mode;
  h->L = num_layers;
  h->D = bidirectional ? 2 : 1;
  h->I = input_size;
  h->H = hidden_size;
  h->dtype = dtype;
  h->flags = flags;
  h->G = mode == RNN_LSTM ? 4 : (mode == RNN_GRU || mode == RNN_GRU_TF) ? 3 : 1;
  h->Gs = mode == RNN_TANH ? 1 : 4;
  *out = h;
  return RNN_OK;
}

rnn_status_t rnn_destroy(rnn_t h) {
  if (!h) return RNN_OK;
  for (auto& m : h->marks) {
    cudaEventDestroy(m.start);
    cudaEventDestroy(m.stop);
  }
  if (h->d_sync) cudaFree(h->d_sync);
  if (h->scratch) cudaFree(h->scratch);
  delete h;
  return RNN_OK;
}

rnn_status_t rnn_weight_count(rnn_t h, int64_t* n) {
  if (!h || !n) return RNN_ERR_INVALID_ARG;
  *n = weight_count(h);
  return RNN_OK;
}

rnn_status_t rnn_weight_layout(rnn_t h, int layer, int dir, int which, int64_t* offset,
                               int64_t* rows, int64_t* cols) {
  if (!h || !offset || !rows || !cols) return RNN_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->L || dir < 0 || dir >= h->D || which < 0 || which > 3)
    return RNN_ERR_INVALID_ARG;
  *offset = weight_offset(h, layer, dir, which);
  *rows = h->G * h->H;
  *cols = which == 0 ? layer_in(h, layer) : which == 1 ? h->H : 1;
  return RNN_OK;
}

rnn_status_t rnn_workspace_size(rnn_t h, int64_t T, int64_t N, int64_t* bytes) {
  if (!bytes) return RNN_ERR_INVALID_ARG;
  rnn_status_t s = check_sizes(h, T, N);
  if (s != RNN_OK) return s;
  *bytes = ws_layout(h, T, N).total;
  return RNN_OK;
}

rnn_status_t rnn_workspace_layout(rnn_t h, int64_t T, int64_t N, int region, int layer, int dir,
                                  int64_t* offset, int64_t* bytes) {
  if (!offset || !bytes) return RNN_ERR_INVALID_ARG;
  rnn_status_t s = check_sizes(h, T, N);
  if (s != RNN_OK) return s;
  if (region < 0 || region >= RNN_WS_NUM_REGIONS) return RNN_ERR_INVALID_ARG;
  const bool per_layer = region == RNN_WS_YLAYER;
  const bool global = region == RNN_WS_GX || region == RNN_WS_DY || region == RNN_WS_GEMM;
  if (global) layer = 0;
  if (global || per_layer) dir = 0;
  if (layer < 0 || layer >= h->L || dir < 0 || dir >= h->D) return RNN_ERR_INVALID_ARG;
  WsLayout w = ws_layout(h, T, N);
  *offset = w.at(region, layer, dir).off;
  *bytes = w.at(region, layer, dir).bytes;
  return RNN_OK;
}

static rnn_status_t forward_training_impl(rnn_t h, void* stream, int64_t T, int64_t N,
                                          const int32_t* lengths, const void* x, const void* h0,
                                          const void* c0, const void* W, void* y, void* hy,
                                          void* cy, void* workspace, int64_t ws_bytes,
                                          const uint8_t* drop_masks = nullptr,
                                          float drop_p = 0.f) {
  rnn_status_t s = check_sizes(h, T, N);
  if (s != RNN_OK) return s;
  if (!x || !W || !y || !workspace) return RNN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(W, 16) || !aligned(y, 16) || !aligned(h0, 16) ||
      !aligned(c0, 16) || !aligned(hy, 16) || !aligned(cy, 16) || !aligned(workspace, 256))
    return RNN_ERR_MISALIGNED;
  if (ws_bytes < ws_layout(h, T, N).total) return RNN_ERR_WORKSPACE_TOO_SMALL;
  s = device_setup(h);
  if (s != RNN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Scratch sc;
  {
    const Region& R = ws_layout(h, T, N).at(RNN_WS_GEMM, 0, 0);
    sc.base = static_cast<char*>(workspace) + R.off;
    sc.cap = R.bytes;
  }
  s = forward_impl(h, st, T, N, x, h0, c0, W, y, hy, cy, static_cast<char*>(workspace), true, sc,
                   lengths, nullptr, drop_masks, drop_p);
  return finish(h, st, s);
}

rnn_status_t rnn_forward_training(rnn_t h, void* stream, int64_t T, int64_t N, const void* x,
                                  const void* h0, const void* c0, const void* W, void* y,
                                  void* hy, void* cy, void* workspace, int64_t ws_bytes) {
  return forward_training_impl(h, stream, T, N, nullptr, x, h0, c0, W, y, hy, cy, workspace,
                               ws_bytes);
}

rnn_status_t rnn_forward_training_dropout(rnn_t h, void* stream, int64_t T, int64_t N,
                                          float dropout, const uint8_t* masks, const void* x,
                                          const void* h0, const void* c0, const void* W, void* y,
                                          void* hy, void* cy, void* workspace,
                                          int64_t ws_bytes) {
  if (!h || !(dropout >= 0.f && dropout < 1.f) || (h->L > 1 && !masks))
    return RNN_ERR_INVALID_ARG;
  return forward_training_impl(h, stream, T, N, nullptr, x, h0, c0, W, y, hy, cy, workspace,
                               ws_bytes, h->L > 1 ? masks : nullptr, dropout);
}

rnn_status_t rnn_forward_training_varlen(rnn_t h, void* stream, int64_t T, int64_t N,
                                         const int32_t* lengths, const void* x, const void* h0,
                                         const void* c0, const void* W, void* y, void* hy,
                                         void* cy, void* workspace, int64_t ws_bytes) {
  if (!lengths) return RNN_ERR_INVALID_ARG;
  if (!aligned(lengths, 4)) return RNN_ERR_MISALIGNED;
  return forward_training_impl(h, stream, T, N, lengths, x, h0, c0, W, y, hy, cy, workspace,
                               ws_bytes);
}

static rnn_status_t forward_inference_impl(rnn_t h, void* stream, int64_t T, int64_t N,
                                           const int32_t* lengths, const void* x,
                                           const void* h0, const void* c0, const void* W,
                                           void* y, void* hy, void* cy) {
  rnn_status_t s = check_sizes(h, T, N);
  if (s != RNN_OK) return s;
  if (!x || !W || !y) return RNN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(W, 16) || !aligned(y, 16) || !aligned(h0, 16) ||
      !aligned(c0, 16) || !aligned(hy, 16) || !aligned(cy, 16))
    return RNN_ERR_MISALIGNED;
  s = device_setup(h);
  if (s != RNN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t hseq_off = align256(h->D * T * N * h->G * h->H * 4) +
                           2 * align256(T * N * h->D * h->H * esize(h));
  // with lengths: the carried states of every step, D x (T+1) x N x H
  const int64_t base_bytes =
      hseq_off + (lengths ? align256(h->D * (T + 1) * N * h->H * esize(h)) : 0);
  const size_t need = (size_t)(base_bytes + gemm_scratch_bytes(h, T, N, false));
  if (need > h->scratch_bytes) {
    // the old scratch may still be in use by earlier work on the stream
    if (h->scratch) {
      if (cudaStreamSynchronize(st) != cudaSuccess) return RNN_ERR_CUDA;
      cudaFree(h->scratch);
      h->scratch = nullptr;
      h->scratch_bytes = 0;
    }
    if (cudaMalloc(&h->scratch, need) != cudaSuccess) {
      h->scratch = nullptr;
      return RNN_ERR_CUDA;
    }
    h->scratch_bytes = need;
  }
  Scratch sc;
  sc.base = static_cast<char*>(h->scratch) + base_bytes;
  sc.cap = (int64_t)h->scratch_bytes - base_bytes;
  s = forward_impl(h, st, T, N, x, h0, c0, W, y, hy, cy, nullptr, false, sc, lengths,
                   static_cast<char*>(h->scratch) + hseq_off);
  return finish(h, st, s);
}

rnn_status_t rnn_forward_inference(rnn_t h, void* stream, int64_t T, int64_t N, const void* x,
                                   const void* h0, const void* c0, const void* W, void* y,
                                   void* hy, void* cy) {
  return forward_inference_impl(h, stream, T, N, nullptr, x, h0, c0, W, y, hy, cy);
}

rnn_status_t rnn_forward_inference_varlen(rnn_t h, void* stream, int64_t T, int64_t N,
                                          const int32_t* lengths, const void* x, const void* h0,
                                          const void* c0, const void* W, void* y, void* hy,
                                          void* cy) {
  if (!lengths) return RNN_ERR_INVALID_ARG;
  if (!aligned(lengths, 4)) return RNN_ERR_MISALIGNED;
  return forward_inference_impl(h, stream, T, N, lengths, x, h0, c0, W, y, hy, cy);
}

static rnn_status_t backward_data_impl(rnn_t h, void* stream, int64_t T, int64_t N,
                                       const int32_t* lengths, const void* W, const void* dy,
                                       const void* dhy, const void* dcy, void* dx, void* dh0,
                                       void* dc0, void* workspace, int64_t ws_bytes,
                                       const uint8_t* drop_masks = nullptr,
                                       float drop_p = 0.f) {
  rnn_status_t s = check_sizes(h, T, N);
  if (s != RNN_OK) return s;
  if (!W || !dy || !dx || !workspace) return RNN_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(dy, 16) || !aligned(dx, 16) || !aligned(dhy, 16) ||
      !aligned(dcy, 16) || !aligned(dh0, 16) || !aligned(dc0, 16) || !aligned(workspace, 256))
    return RNN_ERR_MISALIGNED;
  WsLayout lay = ws_layout(h, T, N);
  if (ws_bytes < lay.total) return RNN_ERR_WORKSPACE_TOO_SMALL;
  s = device_setup(h);
  if (s != RNN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int64_t e = esize(h), H = h->H, NH = N * H, GH = h->G * H;
  const bool bf = h->dtype == RNN_BF16;
  RecPlan plan, plan_one;
  s = plan_rec(h, true, N, &plan, h->D, lengths != nullptr);
  const bool in_turn =
      s == RNN_OK && bwd_directions_in_turn(h, N, plan, &plan_one, lengths != nullptr);
  if (s != RNN_OK) return finish(h, st, s);
  Scratch sc;
  sc.base = ws + lay.at(RNN_WS_GEMM, 0, 0).off;
  sc.cap = lay.at(RNN_WS_GEMM, 0, 0).bytes;
  // exchange words of the tensor-core backward, from the front of the scratch
  unsigned long long* gxw[2] = {nullptr, nullptr};
  if (plan.tc == 2 || (in_turn && plan_one.tc == 2)) {
    for (int d = 0; d < h->D; ++d) {
      gxw[d] = static_cast<unsigned long long*>(sc.take(rec_tc_xchg_bytes((int)N, (int)GH)));
      if (!gxw[d]) return finish(h, st, RNN_ERR_WORKSPACE_TOO_SMALL);
    }
  }
  void* xrows[2] = {nullptr, nullptr};
  if (h->mode == RNN_GRU_TF) {
    for (int d = 0; d < h->D; ++d) {
      xrows[d] = sc.take(N * GH * e);
      if (!xrows[d]) return finish(h, st, RNN_ERR_WORKSPACE_TOO_SMALL);
    }
  }
  const void* dcur = dy;
  int dcur_bf16 = bf;
  for (int l = h->L - 1; l >= 0; --l) {
    RecParams rp;
    fill_rec_common(h, T, N, &rp);
    rp.plan = plan;
    rp.ldy = h->D * H;
    rp.lddy = h->D * H;
    rp.lengths = lengths;
    for (int d = 0; d < h->D; ++d) {
      RecDirArgs& a = rp.dir[d];
      const int k = l * h->D + d;
      a.whh = cp<char>(W, weight_offset(h, l, d, 1) * e);
      a.gates = mp<float>(ws, lay.at(RNN_WS_GATES, l, d).off);
      a.cseq = h->mode == RNN_LSTM ? mp<float>(ws, lay.at(RNN_WS_CSEQ, l, d).off) : nullptr;
      a.hseq = mp<char>(ws, lay.at(RNN_WS_HSEQ, l, d).off);
      a.dy = dcur;
      a.dy_bf16 = dcur_bf16;
      a.dhy = dhy ? cp<char>(dhy, k * NH * e) : nullptr;
      a.dcy = (dcy && h->mode == RNN_LSTM) ? cp<float>(dcy, k * NH * 4) : nullptr;
      a.dgx = mp<char>(ws, lay.at(RNN_WS_DGX, l, d).off);
      a.dgh = h->mode == RNN_GRU ? mp<char>(ws, lay.at(RNN_WS_DGH, l, d).off) : a.dgx;
      a.dh0 = dh0 ? mp<char>(dh0, k * NH * e) : nullptr;
      a.dc0 = (dc0 && h->mode == RNN_LSTM) ? mp<float>(dc0, k * NH * 4) : nullptr;
      a.hx = gxw[d];
      a.xbuf = xrows[d];
    }
    {
      PhaseScope ps(h, st, RNN_PHASE_REC_BWD);
      if (in_turn) {
        // one launch per direction; the second runs its time order reversed
        // and reads its half of dy
        for (int d = 0; d < 2 && s == RNN_OK; ++d) {
          RecParams r1 = rp;
          r1.plan = plan_one;
          r1.D = 1;
          r1.dir[0] = rp.dir[d];
          r1.dir[0].rev = d;
          r1.dir[0].dy = static_cast<const char*>(rp.dir[d].dy) +
                         (int64_t)d * H * (rp.dir[d].dy_bf16 ? 2 : 4);
          s = cuda_status(plan_one.tc == 3 ? rec_tcm_bwd_launch(r1, st)
                                           : rec_tc_bwd_launch(r1, st));
        }
      } else {
        s = cuda_status(rp.plan.tc == 3   ? rec_tcm_bwd_launch(rp, st)
                        : rp.plan.tc      ? rec_tc_bwd_launch(rp, st)
                        : rp.plan.cluster ? rec_cluster_launch(true, rp, st)
                                          : rec_backward(rp, st));
      }
      if (s != RNN_OK) return finish(h, st, s);
    }
    // dX = sum_d dG_x[d] W_ih[l,d]; for l > 0 it is dy of the layer below
    const int64_t I_l = layer_in(h, l);
    void* target;
    int target_bf16;
    if (l == 0) {
      target = dx;
      target_bf16 = bf;
    } else {
      target = mp<char>(ws, lay.at(RNN_WS_DY, 0, 0).off + (int64_t)((l - 1) & 1) * T * N * h->D * H * 4);
      target_bf16 = 0;
    }
    GemmArgs g;
    g.M = T * N; g.N = I_l; g.K = GH;
    g.A = rp.dir[0].dgx; g.sam = GH; g.sak = 1;
    g.B = cp<char>(W, weight_offset(h, l, 0, 0) * e); g.sbk = I_l; g.sbn = 1;
    if (h->D == 2) {
      g.K2 = GH;
      g.A2 = rp.dir[1].dgx; g.sam2 = GH; g.sak2 = 1;
      g.B2 = cp<char>(W, weight_offset(h, l, 1, 0) * e); g.sbk2 = I_l; g.sbn2 = 1;
    }
    g.C = target; g.ldc = I_l;
    g.in_bf16 = bf;
    g.out_bf16 = target_bf16;
    {
      PhaseScope ps(h, st, RNN_PHASE_DX_GEMM);
      s = run_gemm(h, g, sc, st);
      if (s != RNN_OK) return s;
    }
    if (drop_masks && l > 0) {
      // the layer below's output reached this layer dropped
      const int64_t n = T * N * h->D * H;
      s = cuda_status(dropout_apply(target, 0, drop_masks + (int64_t)(l - 1) * n, n,
                                    1.f / (1.f - drop_p), h->num_sms, st));
      if (s != RNN_OK) return finish(h, st, s);
    }
    dcur = target;
    dcur_bf16 = target_bf16;
  }
  return finish(h, st, RNN_OK);
}

rnn_status_t rnn_backward_data(rnn_t h, void* stream, int64_t T, int64_t N, const void* W,
                               const void* dy, const void* dhy, const void* dcy, void* dx,
                               void* dh0, void* dc0, void* workspace, int64_t ws_bytes) {
  return backward_data_impl(h, stream, T, N, nullptr, W, dy, dhy, dcy, dx, dh0, dc0, workspace,
                            ws_bytes);
}

rnn_status_t rnn_backward_data_dropout(rnn_t h, void* stream, int64_t T, int64_t N,
                                       float dropout, const uint8_t* masks, const void* W,
                                       const void* dy, const void* dhy, const void* dcy,
                                       void* dx, void* dh0, void* dc0, void* workspace,
                                       int64_t ws_bytes) {
  if (!h || !(dropout >= 0.f && dropout < 1.f) || (h->L > 1 && !masks))
    return RNN_ERR_INVALID_ARG;
  return backward_data_impl(h, stream, T, N, nullptr, W, dy, dhy, dcy, dx, dh0, dc0, workspace,
                            ws_bytes, h->L > 1 ? masks : nullptr, dropout);
}

rnn_status_t rnn_backward_data_varlen(rnn_t h, void* stream, int64_t T, int64_t N,
                                      const int32_t* lengths, const void* W, const void* dy,
                                      const void* dhy, const void* dcy, void* dx, void* dh0,
                                      void* dc0, void* workspace, int64_t ws_bytes) {
  if (!lengths) return RNN_ERR_INVALID_ARG;
  if (!aligned(lengths, 4)) return RNN_ERR_MISALIGNED;
  return backward_data_impl(h, stream, T, N, lengths, W, dy, dhy, dcy, dx, dh0, dc0, workspace,
                            ws_bytes);
}

namespace {
// The B operand r * h_{t-1} of the TensorFlow-flavour GRU's dW_hn: rows x cols
// fp32 with row stride lds in the workspace; bf16 handles contract in bf16,
// so those get a bf16 copy from the scratch.
rnn_status_t rh_operand(const rnn_handle* h, const void* rh, int64_t rows, int64_t cols,
                        int64_t lds, GemmArgs* g, Scratch* sc, cudaStream_t st) {
  if (h->dtype != RNN_BF16) {
    g->B = rh; g->sbk = lds; g->sbn = 1;
    return RNN_OK;
  }
  void* dst = sc->take(rows * cols * 2);
  if (!dst) return RNN_ERR_WORKSPACE_TOO_SMALL;
  if (to_bf16(static_cast<const float*>(rh), rows, cols, lds, dst, h->num_sms, st) != cudaSuccess)
    return RNN_ERR_CUDA;
  g->B = dst; g->sbk = cols; g->sbn = 1;
  return RNN_OK;
}
}  // namespace

rnn_status_t rnn_backward_weights(rnn_t h, void* stream, int64_t T, int64_t N, const void* x,
                                  const void* h0, const void* y, const void* workspace,
                                  int64_t ws_bytes, void* dW) {
  (void)h0;
  (void)y;
  rnn_status_t s = check_sizes(h, T, N);
  if (s != RNN_OK) return s;
  if (!x || !workspace || !dW) return RNN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(dW, 16) || !aligned(workspace, 256)) return RNN_ERR_MISALIGNED;
  WsLayout lay = ws_layout(h, T, N);
  if (ws_bytes < lay.total) return RNN_ERR_WORKSPACE_TOO_SMALL;
  s = device_setup(h);
  if (s != RNN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const char* ws = static_cast<const char*>(workspace);
  const int64_t e = esize(h), H = h->H, GH = h->G * H;
  const bool bf = h->dtype == RNN_BF16;
  // the GEMM scratch region is the one part of the workspace this call writes
  Scratch sc;
  sc.base = const_cast<char*>(ws) + lay.at(RNN_WS_GEMM, 0, 0).off;
  sc.cap = lay.at(RNN_WS_GEMM, 0, 0).bytes;
  PhaseScope ps(h, st, RNN_PHASE_DW_GEMM);
  for (int l = 0; l < h->L; ++l) {
    const int64_t I_l = layer_in(h, l);
    const void* in = l == 0 ? x : static_cast<const void*>(ws + lay.at(RNN_WS_YLAYER, l - 1, 0).off);
    for (int d = 0; d < h->D; ++d) {
      const void* dgx = ws + lay.at(RNN_WS_DGX, l, d).off;
      const void* dgh = h->mode == RNN_GRU ? ws + lay.at(RNN_WS_DGH, l, d).off : dgx;
      const char* hseq = ws + lay.at(RNN_WS_HSEQ, l, d).off;
      const void* hprev = hseq + (d == 1 ? N * H * e : 0);
      // dG_x^T, presented once for both weight GEMMs when dG_h is dG_x
      Scratch scl = sc;
      PreparedA pa;
      if (!(h->flags & RNN_FLAG_SIMT_GEMM) && dgh == dgx &&
          GH * std::min<int64_t>(I_l, H) * T * N >= kTinyGemmMacs) {
        pa.src = dgx; pa.M = GH; pa.K = T * N; pa.sam = 1; pa.sak = GH;
        pa.valid = prepare_a(h, &pa, !bf, &scl, st);
        if (!pa.valid) scl = sc;
      }
      GemmArgs g;
      g.M = GH; g.N = I_l; g.K = T * N;
      g.A = dgx; g.sam = 1; g.sak = GH;
      g.B = in; g.sbk = I_l; g.sbn = 1;
      g.C = mp<char>(dW, weight_offset(h, l, d, 0) * e); g.ldc = I_l;
      g.in_bf16 = bf; g.out_bf16 = bf;
      s = run_gemm(h, g, scl, st, &pa);
      if (s != RNN_OK) return s;
      GemmArgs g2;
      g2.M = GH; g2.N = H; g2.K = T * N;
      g2.A = dgh; g2.sam = 1; g2.sak = GH;
      g2.B = hprev; g2.sbk = H; g2.sbn = 1;
      g2.C = mp<char>(dW, weight_offset(h, l, d, 1) * e); g2.ldc = H;
      g2.in_bf16 = bf; g2.out_bf16 = bf;
      if (h->mode == RNN_GRU_TF) {
        // the TensorFlow-flavour GRU's W_hn multiplies r * h_{t-1}: its rows
        // of dW_hh contract da_n with that product (saved in the fourth gate
        // slot of the workspace, fp32), the r and z rows with h_{t-1}
        g2.M = 2 * H;
        s = run_gemm(h, g2, scl, st);
        if (s != RNN_OK) return s;
        const void* rh = ws + lay.at(RNN_WS_GATES, l, d).off + 3 * H * 4;
        GemmArgs g3;
        g3.M = H; g3.N = H; g3.K = T * N;
        g3.A = static_cast<const char*>(dgh) + 2 * H * e; g3.sam = 1; g3.sak = GH;
        g3.in_bf16 = bf; g3.out_bf16 = bf;
        g3.C = mp<char>(dW, (weight_offset(h, l, d, 1) + 2 * H * H) * e); g3.ldc = H;
        s = rh_operand(h, rh, T * N, H, 4 * H, &g3, &scl, st);
        if (s != RNN_OK) return s;
        s = run_gemm(h, g3, scl, st);
      } else {
        s = run_gemm(h, g2, scl, st, &pa);
      }
      if (s != RNN_OK) return s;
      // db_ih = sum of dG_x over (t, n); db_hh likewise over dG_h, which is
      // dG_x itself except for the GRU: then one sum serves both
      Scratch cs = sc;
      const int64_t cs_bytes = std::min<int64_t>(cs.cap - align256(cs.off), (int64_t)64 << 20);
      float* part = cs_bytes > 0 ? static_cast<float*>(cs.take(cs_bytes)) : nullptr;
      char* db_ih = mp<char>(dW, weight_offset(h, l, d, 2) * e);
      char* db_hh = mp<char>(dW, weight_offset(h, l, d, 3) * e);
      if (colsum(db_ih, bf, dgx, bf, T * N, GH, GH, part, part ? cs_bytes : 0, h->num_sms, st) !=
          cudaSuccess)
        return RNN_ERR_CUDA;
      const cudaError_t ce =
          dgh == dgx ? cudaMemcpyAsync(db_hh, db_ih, GH * e, cudaMemcpyDeviceToDevice, st)
                     : colsum(db_hh, bf, dgh, bf, T * N, GH, GH, part, part ? cs_bytes : 0,
                              h->num_sms, st);
      if (ce != cudaSuccess) return RNN_ERR_CUDA;
    }
  }
  return finish(h, st, RNN_OK);
}

namespace {
int* static_status_word(int dev);
}

rnn_status_t rnn_check_status(rnn_t h, void* stream) {
  if (!h) return RNN_ERR_INVALID_ARG;
  rnn_status_t s = read_status(h, static_cast<cudaStream_t>(stream));
  // the status word of rnn_forward_inference_static's array on this device,
  // when a static call has run here
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RNN_ERR_CUDA;
  if (int* w = static_status_word(dev)) {
    const rnn_status_t s2 = take_status_word(w);
    if (s == RNN_OK) s = s2;
  }
  return s;
}

rnn_status_t rnn_set_debug(rnn_t h, int fault_block, int fault_step, int64_t timeout_ns) {
  if (!h) return RNN_ERR_INVALID_ARG;
  if (timeout_ns > 0) h->timeout_ns = timeout_ns;
  h->fault_block = fault_block;
  h->fault_step = fault_step;
  return RNN_OK;
}

rnn_status_t rnn_enable_phase_timing(rnn_t h, int enable) {
  if (!h) return RNN_ERR_INVALID_ARG;
  for (auto& m : h->marks) {
    cudaEventDestroy(m.start);
    cudaEventDestroy(m.stop);
  }
  h->marks.clear();
  for (int i = 0; i < RNN_PHASE_NUM; ++i) {
    h->ms[i] = 0;
    h->launches[i] = 0;
  }
  h->timing = enable != 0;
  return RNN_OK;
}

rnn_status_t rnn_get_phase_times(rnn_t h, double* ms, int64_t* launches) {
  if (!h || !ms || !launches) return RNN_ERR_INVALID_ARG;
  for (auto& m : h->marks) {
    if (cudaEventSynchronize(m.stop) != cudaSuccess) return RNN_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, m.start, m.stop) != cudaSuccess) return RNN_ERR_CUDA;
    h->ms[m.phase] += t;
    h->launches[m.phase] += m.kernels;
    cudaEventDestroy(m.start);
    cudaEventDestroy(m.stop);
  }
  h->marks.clear();
  for (int i = 0; i < RNN_PHASE_NUM; ++i) {
    ms[i] = h->ms[i];
    launches[i] = h->launches[i];
  }
  return RNN_OK;
}

static rnn_status_t get_paths(rnn_t h, int64_t N, int* fwd, int* bwd, bool varlen) {
  if (!h || !fwd || !bwd || N < 1) return RNN_ERR_INVALID_ARG;
  rnn_status_t s = device_setup(h);
  if (s != RNN_OK) return s;
  auto kind = [](const RecPlan& pl) {
    return pl.tc ? RNN_PATH_TENSOR : pl.cluster ? RNN_PATH_CLUSTER
                                   : pl.direct  ? RNN_PATH_DIRECT
                                                : RNN_PATH_STAGED;
  };
  WfPlan wp;
  RecPlan pl;
  if (wf_candidate(h, N) &&
      wf_plan(h->mode, 1, h->L, h->D, h->I, h->H, N, h->num_sms, h->smem_optin, &wp) &&
      (size_t)h->L * wp.Pr * 128 <= kSyncBytes - 64) {
    *fwd = RNN_PATH_WAVEFRONT;
  } else {
    s = plan_rec(h, false, N, &pl, h->D, varlen);
    if (s != RNN_OK) return s;
    RecPlan one;
    *fwd = fwd_directions_in_turn(h, N, pl, &one, varlen) ? kind(one) : kind(pl);
  }
  s = plan_rec(h, true, N, &pl, h->D, varlen);
  if (s != RNN_OK) return s;
  RecPlan one;
  *bwd = bwd_directions_in_turn(h, N, pl, &one, varlen) ? kind(one) : kind(pl);
  return RNN_OK;
}

rnn_status_t rnn_get_paths(rnn_t h, int64_t N, int* fwd, int* bwd) {
  return get_paths(h, N, fwd, bwd, false);
}

rnn_status_t rnn_get_paths_varlen(rnn_t h, int64_t N, int* fwd, int* bwd) {
  return get_paths(h, N, fwd, bwd, true);
}

// ----------------------------------------------------------------------------
// test hooks: the packed operand forms, produced by the library's own kernels
// ----------------------------------------------------------------------------
rnn_status_t rnn_debug_gemm_shape(int64_t M, int64_t N, int64_t K_total, int split16, int num_sms,
                                  int allow_split, int* bn, int* ksplit) {
  if (M < 1 || N < 1 || K_total < 1 || num_sms < 1 || !bn || !ksplit) return RNN_ERR_INVALID_ARG;
  gemm_tc_shape(M, N, K_total, split16 != 0, num_sms, allow_split != 0, bn, ksplit);
  return RNN_OK;
}

rnn_status_t rnn_debug_split_f16(const float* src, int64_t rows, int64_t cols, int64_t lds,
                                 void* hi, void* lo, int64_t ldd, int transpose, unsigned* maxbits,
                                 void* stream) {
  if (!src || !hi || !lo || !maxbits || rows < 1 || cols < 1 || lds < cols ||
      ldd < (transpose ? rows : cols))
    return RNN_ERR_INVALID_ARG;
  if (!aligned(src, 16) || !aligned(hi, 16) || !aligned(lo, 16) || !aligned(maxbits, 4))
    return RNN_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 1;
  if (cudaGetDevice(&dev) == cudaSuccess)
    (void)cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e = cudaMemsetAsync(maxbits, 0, 4, st);
  if (e == cudaSuccess) e = absmax_operand(src, rows, cols, lds, maxbits, sms, st);
  if (e == cudaSuccess)
    e = split_f16_operand(src, rows, cols, lds, hi, lo, ldd, transpose != 0, maxbits, st);
  return cuda_status(e);
}

rnn_status_t rnn_debug_transpose_bf16(const void* src, int64_t rows, int64_t cols, int64_t lds,
                                      void* dst, int64_t ldd, void* stream) {
  if (!src || !dst || rows < 1 || cols < 1 || lds < cols || ldd < rows)
    return RNN_ERR_INVALID_ARG;
  if (!aligned(src, 16) || !aligned(dst, 16)) return RNN_ERR_MISALIGNED;
  return cuda_status(
      transpose_bf16(src, rows, cols, lds, dst, ldd, static_cast<cudaStream_t>(stream)));
}

rnn_status_t rnn_debug_wf_pack(rnn_t h, void* stream, int64_t N, int layer, const void* W,
                               void* wp, int64_t wp_bytes, float* bias, int64_t bias_bytes,
                               int64_t* layout) {
  if (!h || !W || !wp || !bias || !layout || N < 1 || layer < 0 || layer >= h->L)
    return RNN_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(wp, 16) || !aligned(bias, 16)) return RNN_ERR_MISALIGNED;
  rnn_status_t s = device_setup(h);
  if (s != RNN_OK) return s;
  WfPlan pl;
  if (!wf_candidate(h, N) ||
      !wf_plan(h->mode, 1, h->L, h->D, h->I, h->H, N, h->num_sms, h->smem_optin, &pl))
    return RNN_ERR_UNSUPPORTED;
  const int64_t I_l = layer_in(h, layer), H = h->H;
  const int64_t kp = wf_kp(I_l, H);
  const int64_t rows = (int64_t)pl.Pr * pl.R * pl.Ur;
  if (wp_bytes < rows * kp * 2 || bias_bytes < rows * 4) return RNN_ERR_WORKSPACE_TOO_SMALL;
  const int64_t e = 2;
  const cudaError_t ce =
      wf_pack(pl, h->mode, I_l, H, cp<char>(W, weight_offset(h, layer, 0, 0) * e),
              cp<char>(W, weight_offset(h, layer, 0, 1) * e),
              cp<char>(W, weight_offset(h, layer, 0, 2) * e),
              cp<char>(W, weight_offset(h, layer, 0, 3) * e), wp, bias,
              static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) return RNN_ERR_CUDA;
  layout[0] = pl.Pr;
  layout[1] = pl.Ur;
  layout[2] = pl.R;
  layout[3] = kp;
  layout[4] = (I_l + 63) / 64 * 64;
  return RNN_OK;
}

rnn_status_t rnn_measure_step_protocol(rnn_t h, void* stream, int64_t N, int64_t steps,
                                       double* us_per_step) {
  if (!h || !us_per_step || N < 1 || steps < 2 || steps > (1 << 20)) return RNN_ERR_INVALID_ARG;
  rnn_status_t s = device_setup(h);
  if (s != RNN_OK) return s;
  RecPlan pl;
  s = plan_rec(h, false, N, &pl, 1);
  if (s != RNN_OK) return s;
  if (pl.tc != 1) return RNN_ERR_UNSUPPORTED;
  RecParams rp;
  fill_rec_common(h, steps, N, &rp);
  rp.D = 1;
  rp.plan = pl;
  rp.fault_block = -1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* xbuf = nullptr;
  if (cudaMalloc(&xbuf, rec_tc_xchg_bytes((int)N, (int)h->H)) != cudaSuccess) return RNN_ERR_CUDA;
  rp.dir[0].hx = static_cast<unsigned long long*>(xbuf);
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) {
    cudaFree(xbuf);
    return RNN_ERR_CUDA;
  }
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    cudaFree(xbuf);
    return RNN_ERR_CUDA;
  }
  s = RNN_OK;
  // the flag memset of the launch sits outside the events: one warm-up launch,
  // then a timed one
  for (int rep = 0; rep < 2 && s == RNN_OK; ++rep) {
    if (rep == 1 && cudaEventRecord(e0, st) != cudaSuccess) s = RNN_ERR_CUDA;
    if (s == RNN_OK) s = cuda_status(rec_tc_probe_launch(rp, st));
    if (rep == 1 && s == RNN_OK && cudaEventRecord(e1, st) != cudaSuccess) s = RNN_ERR_CUDA;
  }
  float ms = 0.f;
  if (s == RNN_OK && (cudaEventSynchronize(e1) != cudaSuccess ||
                      cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess))
    s = RNN_ERR_CUDA;
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (s == RNN_OK) s = read_status(h, st);
  if (cudaStreamSynchronize(st) != cudaSuccess && s == RNN_OK) s = RNN_ERR_CUDA;
  cudaFree(xbuf);
  if (s == RNN_OK) *us_per_step = (double)ms * 1e3 / (double)steps;
  return s;
}

const char* rnn_status_string(rnn_status_t s) {
  switch (s) {
    case RNN_OK: return "ok";
    case RNN_ERR_INVALID_ARG: return "invalid argument";
    case RNN_ERR_UNSUPPORTED: return "unsupported configuration";
    case RNN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case RNN_ERR_MISALIGNED: return "misaligned pointer";
    case RNN_ERR_CUDA: return "CUDA runtime error";
    case RNN_ERR_TIMEOUT: return "step barrier timed out";
    case RNN_ERR_NO_RESIDENCY: return "persistent grid cannot be co-resident";
    case RNN_ERR_DEVICE_CHECK: return "a kernel's index check failed (access skipped)";
  }
  return "unknown status";
}

}  // extern "C"

// ============================================================================
// Inference forward without any device allocation
//
// For callers that cannot allocate device memory themselves or let a library
// do it: code running while a memory pool owns the whole device, allocators
// that must not be re-entered, or processes with a fixed memory budget set at
// start-up.  rnn_forward_inference keeps its scratch in handle-owned memory
// that it allocates on first use (and the handle allocates 64 KB of barrier
// flags on its first compute call); this entry point instead places all of its
// scratch -- the step flags and status word, the input projection and the two
// intermediate layer outputs -- in one file-scope device array, so the call
// performs no cudaMalloc or cudaFree at all.
// ============================================================================
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB per device

// Every GPU that loads this library holds this array until the process exits.
// All calls of rnn_forward_inference_static on a device share it.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {nullptr};

// Device address of the array for the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device with that device current and cached.
rnn_status_t static_scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return RNN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return RNN_ERR_CUDA;
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return RNN_OK;
}

// the array's status word on device `dev`, or null before the first static
// call there
int* static_status_word(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) return nullptr;
  return reinterpret_cast<int*>(static_cast<char*>(g_static_addr[dev]) + kSyncBytes - 64);
}

}  // namespace

extern "C" rnn_status_t rnn_forward_inference_static(rnn_t h, void* stream, int64_t T, int64_t N,
                                                     const void* x, const void* h0,
                                                     const void* c0, const void* W, void* y,
                                                     void* hy, void* cy) {
  rnn_status_t s = check_sizes(h, T, N);
  if (s != RNN_OK) return s;
  if (!x || !W || !y) return RNN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(W, 16) || !aligned(y, 16) || !aligned(h0, 16) ||
      !aligned(c0, 16) || !aligned(hy, 16) || !aligned(cy, 16))
    return RNN_ERR_MISALIGNED;
  // scratch: [flags + status | input projection | two intermediate outputs]
  const int64_t gx_bytes = align256(h->D * T * N * h->G * h->H * 4);
  const int64_t yb = align256(T * N * h->D * h->H * esize(h));
  const int64_t need = (int64_t)kSyncBytes + gx_bytes + (h->L > 1 ? 2 * yb : 0);
  if (need + xchg_bytes(h, N) > (int64_t)kStaticScratchBytes) return RNN_ERR_WORKSPACE_TOO_SMALL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RNN_ERR_CUDA;
  if (h->device >= 0 && h->device != dev) return RNN_ERR_INVALID_ARG;  // one device per handle
  void* base = nullptr;
  s = static_scratch_address(dev, &base);
  if (s != RNN_OK) return s;
  int sms = 0, optin = 0, coop = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
    return RNN_ERR_CUDA;
  if (!coop) return RNN_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the status word keeps the previous call's value: clear it (flags are
  // cleared before every persistent launch)
  if (cudaMemsetAsync(base, 0, kSyncBytes, st) != cudaSuccess) return RNN_ERR_CUDA;
  // a view of the handle whose device state points into the static array
  rnn_handle v;
  v.mode = h->mode; v.L = h->L; v.D = h->D; v.dtype = h->dtype; v.G = h->G; v.Gs = h->Gs;
  v.I = h->I; v.H = h->H; v.flags = h->flags;
  v.device = dev;
  v.num_sms = sms;
  v.smem_optin = (size_t)optin;
  query_clusters(optin, &v.cluster_smem, v.max_clusters);
  v.d_sync = static_cast<unsigned*>(base);
  v.d_status = reinterpret_cast<int*>(static_cast<char*>(base) + kSyncBytes - 64);
  v.scratch = static_cast<char*>(base) + kSyncBytes;
  v.scratch_bytes = kStaticScratchBytes - kSyncBytes;
  v.timeout_ns = h->timeout_ns;
  v.fault_block = h->fault_block;
  v.fault_step = h->fault_step;
  v.timing = false;
  // what the array has left after the projection and layer outputs serves the
  // tensor-core GEMM's operand copies; without room the GEMM runs on CUDA cores
  Scratch sc;
  sc.base = static_cast<char*>(base) + need;
  sc.cap = (int64_t)kStaticScratchBytes - need;
  s = forward_impl(&v, st, T, N, x, h0, c0, W, y, hy, cy, nullptr, false, sc);
  s = finish(&v, st, s);
  v.d_sync = nullptr;  // not owned: keep the view's destructor path inert
  v.scratch = nullptr;
  return s;
}
