"""ctypes binding of liblayer_rnn.so (include/layer_rnn.h).

Functions keep the C names and arguments; pointers are passed as integers
(device addresses, e.g. ``tensor.data_ptr()``) and streams as integers
(``torch.cuda.current_stream().cuda_stream``).  Non-zero status codes raise
``RnnError``.  ``Rnn`` is a small convenience wrapper around one handle that
takes torch tensors; it only marshals arguments -- every step of the operator
runs in the library's kernels.  Nothing here computes on the CPU, and loading
fails loudly when the library has not been built.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblayer_rnn.so")

RNN_TANH, RNN_LSTM, RNN_GRU, RNN_GRU_TF = 0, 1, 2, 3
RNN_F32, RNN_BF16 = 0, 1
RNN_FLAG_SYNC_CHECK, RNN_FLAG_SIMT_GEMM, RNN_FLAG_SIMT_RECURRENT = 0x1, 0x2, 0x4
RNN_FLAG_NO_WAVEFRONT = 0x8
(RNN_WS_GATES, RNN_WS_CSEQ, RNN_WS_HSEQ, RNN_WS_YLAYER, RNN_WS_DGX, RNN_WS_DGH,
 RNN_WS_GX, RNN_WS_DY, RNN_WS_GEMM) = range(9)
PHASES = ("input_gemm", "rec_fwd", "rec_bwd", "dx_gemm", "dw_gemm")
STATUS = {0: "RNN_OK", 1: "RNN_ERR_INVALID_ARG", 2: "RNN_ERR_UNSUPPORTED",
          3: "RNN_ERR_WORKSPACE_TOO_SMALL", 4: "RNN_ERR_MISALIGNED", 5: "RNN_ERR_CUDA",
          6: "RNN_ERR_TIMEOUT", 7: "RNN_ERR_NO_RESIDENCY", 8: "RNN_ERR_DEVICE_CHECK"}
MODES = {"rnn_tanh": RNN_TANH, "lstm": RNN_LSTM, "gru": RNN_GRU, "gru_tf": RNN_GRU_TF}
DTYPES = {"f32": RNN_F32, "bf16": RNN_BF16}

# exported symbol -> (restype, argtypes)
_i64, _i32, _u32, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_void_p
_pi64 = ctypes.POINTER(ctypes.c_int64)
SIGNATURES = {
    "rnn_create": (_i32, [ctypes.POINTER(_vp), _i32, _i32, _i32, _i64, _i64, _i32, _u32]),
    "rnn_destroy": (_i32, [_vp]),
    "rnn_weight_count": (_i32, [_vp, _pi64]),
    "rnn_weight_layout": (_i32, [_vp, _i32, _i32, _i32, _pi64, _pi64, _pi64]),
    "rnn_workspace_size": (_i32, [_vp, _i64, _i64, _pi64]),
    "rnn_workspace_layout": (_i32, [_vp, _i64, _i64, _i32, _i32, _i32, _pi64, _pi64]),
    "rnn_forward_training": (_i32, [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                    _vp, _i64]),
    "rnn_forward_inference": (_i32, [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "rnn_forward_inference_static": (_i32, [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp,
                                            _vp]),
    "rnn_backward_data": (_i32, [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                 _i64]),
    "rnn_backward_weights": (_i32, [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _i64, _vp]),
    "rnn_forward_training_dropout": (_i32, [_vp, _vp, _i64, _i64, ctypes.c_float, _vp, _vp, _vp,
                                            _vp, _vp, _vp, _vp, _vp, _vp, _i64]),
    "rnn_backward_data_dropout": (_i32, [_vp, _vp, _i64, _i64, ctypes.c_float, _vp, _vp, _vp, _vp,
                                         _vp, _vp, _vp, _vp, _vp, _i64]),
    "rnn_forward_training_varlen": (_i32, [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp,
                                           _vp, _vp, _vp, _i64]),
    "rnn_forward_inference_varlen": (_i32, [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp,
                                            _vp, _vp]),
    "rnn_backward_data_varlen": (_i32, [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                        _vp, _vp, _i64]),
    "rnn_check_status": (_i32, [_vp, _vp]),
    "rnn_set_debug": (_i32, [_vp, _i32, _i32, _i64]),
    "rnn_enable_phase_timing": (_i32, [_vp, _i32]),
    "rnn_get_phase_times": (_i32, [_vp, ctypes.POINTER(ctypes.c_double), _pi64]),
    "rnn_get_paths": (_i32, [_vp, ctypes.c_int64, ctypes.POINTER(ctypes.c_int),
                             ctypes.POINTER(ctypes.c_int)]),
    "rnn_get_paths_varlen": (_i32, [_vp, ctypes.c_int64, ctypes.POINTER(ctypes.c_int),
                                    ctypes.POINTER(ctypes.c_int)]),
    "rnn_measure_step_protocol": (_i32, [_vp, _vp, _i64, _i64, ctypes.POINTER(ctypes.c_double)]),
    "rnn_debug_split_f16": (_i32, [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _i32, _vp, _vp]),
    "rnn_debug_gemm_shape": (_i32, [_i64, _i64, _i64, _i32, _i32, _i32,
                                    ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "rnn_debug_transpose_bf16": (_i32, [_vp, _i64, _i64, _i64, _vp, _i64, _vp]),
    "rnn_debug_wf_pack": (_i32, [_vp, _vp, _i64, _i32, _vp, _vp, _i64, _vp, _i64, _pi64]),
    "rnn_status_string": (ctypes.c_char_p, [_i32]),
}


class RnnError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__("%s returned %s" % (fn, STATUS.get(code, code)))


_lib = None


def lib():
    """Load the library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("liblayer_rnn.so is not built; run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _call(name, *args):
    code = getattr(lib(), name)(*args)
    if code != 0:
        raise RnnError(name, code)


def _p(t):
    """Device pointer of a tensor (or None)."""
    return None if t is None else t.data_ptr()


def rnn_create(mode, num_layers, bidirectional, input_size, hidden_size, dtype, flags=0):
    h = _vp()
    _call("rnn_create", ctypes.byref(h), mode, num_layers, int(bidirectional), input_size,
          hidden_size, dtype, flags)
    return h


def rnn_destroy(h):
    _call("rnn_destroy", h)


def rnn_weight_count(h):
    n = ctypes.c_int64()
    _call("rnn_weight_count", h, ctypes.byref(n))
    return n.value


def rnn_weight_layout(h, layer, direction, which):
    o, r, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _call("rnn_weight_layout", h, layer, direction, which, ctypes.byref(o), ctypes.byref(r),
          ctypes.byref(c))
    return o.value, r.value, c.value


def rnn_workspace_size(h, T, N):
    b = ctypes.c_int64()
    _call("rnn_workspace_size", h, T, N, ctypes.byref(b))
    return b.value


def rnn_workspace_layout(h, T, N, region, layer=0, direction=0):
    o, b = ctypes.c_int64(), ctypes.c_int64()
    _call("rnn_workspace_layout", h, T, N, region, layer, direction, ctypes.byref(o),
          ctypes.byref(b))
    return o.value, b.value


def rnn_forward_training(h, stream, T, N, x, h0, c0, W, y, hy, cy, ws, ws_bytes):
    _call("rnn_forward_training", h, stream, T, N, x, h0, c0, W, y, hy, cy, ws, ws_bytes)


def rnn_forward_inference(h, stream, T, N, x, h0, c0, W, y, hy, cy):
    _call("rnn_forward_inference", h, stream, T, N, x, h0, c0, W, y, hy, cy)


def rnn_forward_inference_static(h, stream, T, N, x, h0, c0, W, y, hy, cy):
    _call("rnn_forward_inference_static", h, stream, T, N, x, h0, c0, W, y, hy, cy)


def rnn_backward_data(h, stream, T, N, W, dy, dhy, dcy, dx, dh0, dc0, ws, ws_bytes):
    _call("rnn_backward_data", h, stream, T, N, W, dy, dhy, dcy, dx, dh0, dc0, ws, ws_bytes)


def rnn_forward_training_dropout(h, stream, T, N, p, masks, x, h0, c0, W, y, hy, cy, ws,
                                 ws_bytes):
    _call("rnn_forward_training_dropout", h, stream, T, N, p, masks, x, h0, c0, W, y, hy, cy, ws,
          ws_bytes)


def rnn_backward_data_dropout(h, stream, T, N, p, masks, W, dy, dhy, dcy, dx, dh0, dc0, ws,
                              ws_bytes):
    _call("rnn_backward_data_dropout", h, stream, T, N, p, masks, W, dy, dhy, dcy, dx, dh0, dc0,
          ws, ws_bytes)


def rnn_forward_training_varlen(h, stream, T, N, lengths, x, h0, c0, W, y, hy, cy, ws,
                                ws_bytes):
    _call("rnn_forward_training_varlen", h, stream, T, N, lengths, x, h0, c0, W, y, hy, cy, ws,
          ws_bytes)


def rnn_forward_inference_varlen(h, stream, T, N, lengths, x, h0, c0, W, y, hy, cy):
    _call("rnn_forward_inference_varlen", h, stream, T, N, lengths, x, h0, c0, W, y, hy, cy)


def rnn_backward_data_varlen(h, stream, T, N, lengths, W, dy, dhy, dcy, dx, dh0, dc0, ws,
                             ws_bytes):
    _call("rnn_backward_data_varlen", h, stream, T, N, lengths, W, dy, dhy, dcy, dx, dh0, dc0, ws,
          ws_bytes)


def rnn_backward_weights(h, stream, T, N, x, h0, y, ws, ws_bytes, dW):
    _call("rnn_backward_weights", h, stream, T, N, x, h0, y, ws, ws_bytes, dW)


def rnn_measure_step_protocol(h, stream, N, steps):
    """Microseconds per empty step of the tensor-core forward's protocol."""
    us = ctypes.c_double()
    _call("rnn_measure_step_protocol", h, stream, N, steps, ctypes.byref(us))
    return us.value


def rnn_debug_split_f16(src, rows, cols, lds, hi, lo, ldd, transpose, maxbits, stream):
    _call("rnn_debug_split_f16", src, rows, cols, lds, hi, lo, ldd, int(transpose), maxbits,
          stream)


def rnn_debug_transpose_bf16(src, rows, cols, lds, dst, ldd, stream):
    _call("rnn_debug_transpose_bf16", src, rows, cols, lds, dst, ldd, stream)


def rnn_debug_wf_pack(h, stream, N, layer, W, wp, wp_bytes, bias, bias_bytes):
    """Returns (Pr, Ur, R, kp, Kxp)."""
    lay = (ctypes.c_int64 * 5)()
    _call("rnn_debug_wf_pack", h, stream, N, layer, W, wp, wp_bytes, bias, bias_bytes, lay)
    return tuple(lay)


def rnn_check_status(h, stream):
    return getattr(lib(), "rnn_check_status")(h, stream)


def rnn_set_debug(h, fault_block, fault_step, timeout_ns):
    _call("rnn_set_debug", h, fault_block, fault_step, timeout_ns)


def rnn_enable_phase_timing(h, enable):
    _call("rnn_enable_phase_timing", h, int(enable))


def rnn_get_phase_times(h):
    ms = (ctypes.c_double * len(PHASES))()
    n = (ctypes.c_int64 * len(PHASES))()
    _call("rnn_get_phase_times", h, ms, n)
    return {p: (ms[i], n[i]) for i, p in enumerate(PHASES)}


PATHS = {0: "staged", 1: "direct", 2: "cluster", 3: "tensor", 4: "wavefront"}


def rnn_get_paths(h, N):
    """(forward, backward) recurrent kernel paths of a call with batch N."""
    f, b = ctypes.c_int(), ctypes.c_int()
    _call("rnn_get_paths", h, N, ctypes.byref(f), ctypes.byref(b))
    return PATHS[f.value], PATHS[b.value]


def rnn_debug_gemm_shape(M, N, K_total, split16, num_sms, allow_split=True):
    """(tile width, K splits) the dense phases' wave model picks (host only)."""
    bn, ks = ctypes.c_int(), ctypes.c_int()
    _call("rnn_debug_gemm_shape", M, N, K_total, int(split16), num_sms, int(allow_split),
          ctypes.byref(bn), ctypes.byref(ks))
    return bn.value, ks.value


def rnn_get_paths_varlen(h, N):
    """(forward, backward) recurrent kernel paths of the *_varlen calls."""
    f, b = ctypes.c_int(), ctypes.c_int()
    _call("rnn_get_paths_varlen", h, N, ctypes.byref(f), ctypes.byref(b))
    return PATHS[f.value], PATHS[b.value]


def rnn_status_string(code):
    return lib().rnn_status_string(code).decode()


class Rnn:
    """One handle plus torch-tensor marshalling (device memory and streams only)."""

    def __init__(self, mode, num_layers, bidirectional, input_size, hidden_size, dtype="f32",
                 flags=0):
        import torch  # memory and streams only
        self.torch = torch
        self.mode = mode
        self.L = num_layers
        self.D = 2 if bidirectional else 1
        self.I = input_size
        self.H = hidden_size
        self.dtype = dtype
        self.tdtype = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.h = rnn_create(MODES[mode], num_layers, bidirectional, input_size, hidden_size,
                            DTYPES[dtype], flags)

    def close(self):
        if self.h is not None:
            rnn_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _stream(stream):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        return s.cuda_stream

    def weight_count(self):
        return rnn_weight_count(self.h)

    def workspace_bytes(self, T, N):
        return rnn_workspace_size(self.h, T, N)

    def alloc_workspace(self, T, N, device="cuda"):
        return self.torch.empty(self.workspace_bytes(T, N), dtype=self.torch.uint8, device=device)

    def forward_training(self, x, h0, c0, W, y, hy, cy, ws, stream=None):
        T, N = x.shape[0], x.shape[1]
        rnn_forward_training(self.h, self._stream(stream), T, N, _p(x), _p(h0), _p(c0), _p(W),
                             _p(y), _p(hy), _p(cy), _p(ws), ws.numel())

    def forward_inference(self, x, h0, c0, W, y, hy, cy, stream=None):
        T, N = x.shape[0], x.shape[1]
        rnn_forward_inference(self.h, self._stream(stream), T, N, _p(x), _p(h0), _p(c0), _p(W),
                              _p(y), _p(hy), _p(cy))

    def backward_data(self, W, dy, dhy, dcy, dx, dh0, dc0, ws, stream=None):
        T, N = dy.shape[0], dy.shape[1]
        rnn_backward_data(self.h, self._stream(stream), T, N, _p(W), _p(dy), _p(dhy), _p(dcy),
                          _p(dx), _p(dh0), _p(dc0), _p(ws), ws.numel())

    # inter-layer dropout: masks is a device uint8 tensor [L-1, T, N, D*H] of 0/1
    def forward_training_dropout(self, p, masks, x, h0, c0, W, y, hy, cy, ws, stream=None):
        T, N = x.shape[0], x.shape[1]
        rnn_forward_training_dropout(self.h, self._stream(stream), T, N, p, _p(masks), _p(x),
                                     _p(h0), _p(c0), _p(W), _p(y), _p(hy), _p(cy), _p(ws),
                                     ws.numel())

    def backward_data_dropout(self, p, masks, W, dy, dhy, dcy, dx, dh0, dc0, ws, stream=None):
        T, N = dy.shape[0], dy.shape[1]
        rnn_backward_data_dropout(self.h, self._stream(stream), T, N, p, _p(masks), _p(W),
                                  _p(dy), _p(dhy), _p(dcy), _p(dx), _p(dh0), _p(dc0), _p(ws),
                                  ws.numel())

    # variable-length batches: lengths is a device int32 tensor [N]
    def forward_training_varlen(self, lengths, x, h0, c0, W, y, hy, cy, ws, stream=None):
        T, N = x.shape[0], x.shape[1]
        rnn_forward_training_varlen(self.h, self._stream(stream), T, N, _p(lengths), _p(x),
                                    _p(h0), _p(c0), _p(W), _p(y), _p(hy), _p(cy), _p(ws),
                                    ws.numel())

    def forward_inference_varlen(self, lengths, x, h0, c0, W, y, hy, cy, stream=None):
        T, N = x.shape[0], x.shape[1]
        rnn_forward_inference_varlen(self.h, self._stream(stream), T, N, _p(lengths), _p(x),
                                     _p(h0), _p(c0), _p(W), _p(y), _p(hy), _p(cy))

    def backward_data_varlen(self, lengths, W, dy, dhy, dcy, dx, dh0, dc0, ws, stream=None):
        T, N = dy.shape[0], dy.shape[1]
        rnn_backward_data_varlen(self.h, self._stream(stream), T, N, _p(lengths), _p(W), _p(dy),
                                 _p(dhy), _p(dcy), _p(dx), _p(dh0), _p(dc0), _p(ws), ws.numel())

    def backward_weights(self, x, h0, y, ws, dW, stream=None):
        T, N = x.shape[0], x.shape[1]
        rnn_backward_weights(self.h, self._stream(stream), T, N, _p(x), _p(h0), _p(y), _p(ws),
                             ws.numel(), _p(dW))

    def check_status(self, stream=None):
        return rnn_check_status(self.h, self._stream(stream))
