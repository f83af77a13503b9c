"""Float64 CPU oracle for the fused multi-layer RNN operator.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library never
calls it, and it shares no code with the CUDA library: it computes every step
from the equations with plain NumPy float64 arithmetic, one time step at a time.

What it computes (sources, by page title and section):

* GRU -- the PyTorch / cuDNN flavour.  "rnn training example?" (oneDNN issue
  #218): the PyTorch GRU cell code in mingfeima's comment (gi = linear(x, w_ih,
  b_ih), gh = linear(h, w_hh, b_hh), chunk into r, z, n) and the "PyTorch
  equations" block of mratsim's comment:
      r  = sigmoid(W_ir x + b_ir + W_hr h + b_hr)
      z  = sigmoid(W_iz x + b_iz + W_hz h + b_hz)
      n  = tanh(W_in x + b_in + r * (W_hn h + b_hn))
      h' = (1 - z) * n + z * h
  The same comment states that the cuDNN equations are the same recurrence
  (its "bRu" bias is read as the update gate's recurrent bias).
* GRU, TensorFlow flavour (mode "gru_tf"; not the path's GRU, the groundwork
  for a flag that selects it).  The same comment of "rnn training example?"
  writes the TensorFlow equations, where the reset gate scales h before the
  recurrent matmul of the candidate:
      n  = tanh(W_in x + b_in + W_hn (r * h) + b_hn)
  with r, z and h' as above.  Same weight layout as "gru".
* LSTM -- the pages name LSTM (MXNet "Fused RNN operator for CPU" design page,
  section Performance / LSTM; Keras issue #3692 "CudnnLSTM") but never write its
  equations.  Reading taken: the standard LSTM with two biases (the two-bias
  PyTorch naming of the oneDNN issue) and gate blocks in the order i, f, g, o:
      a = W_ih x + b_ih + W_hh h + b_hh,  i = sigmoid(a_i), f = sigmoid(a_f),
      g = tanh(a_g), o = sigmoid(a_o),  c' = f * c + i * g,  h' = o * tanh(c').
* Vanilla RNN ("vRNN" on the MXNet design page) -- reading taken:
      h' = tanh(W_ih x + b_ih + W_hh h + b_hh).
* Stacking and bidirection (MXNet design page, "5-layers (vRNN/LSTM/GRU) with
  bi-direction"): direction 1 walks t = T-1 .. 0 over the same input and writes
  its output at the original time index; a layer's output is the concatenation
  [forward || backward] along features and is the next layer's input.
* Tensor shapes follow the PyTorch shapes quoted in the oneDNN issue: input in
  TNC order [T, N, I]; hx / cx / hy / cy of shape (num_layers * num_directions,
  batch, hidden), index ``layer * D + direction``.
* Variable-length batches (optional ``lengths``).  "rnn training example?"
  (oneDNN issue #218) names PyTorch's packed sequences as the form variable
  lengths arrive in, and the unpacking to TNC as the integration cost.
  Reading taken: PyTorch's packed-sequence semantics on the padded TNC batch.
  A step t >= len_n of sequence n leaves its state unchanged and writes zero
  output, so hy is the state after the last valid step, and the reverse
  direction starts from h0 at step len_n - 1.
* Inter-layer dropout (optional ``dropout`` and ``masks``).  "rnn training
  example?" (oneDNN issue #218) asks for dropout as cuDNN has it, without
  spelling it out.  Reading taken: cuDNN's / PyTorch's training dropout
  between layers.  The output of every layer but the last is multiplied by a
  0/1 mask and by 1 / (1 - dropout) before it becomes the next layer's input;
  y, hy and cy are not dropped.  The masks are the method's random draws and
  are passed in.
* Backward ("reuse forward intermediate results during backward", MXNet design
  page, Operator Registration): reverse-mode differentiation of the scalar loss
      loss = sum(y * dy) + sum(hy * dhy) + sum(cy * dcy)
  through the same graph, written out by hand per gate below.

The canonical flat weight buffer (``flatten_weights`` / ``unflatten_weights``)
holds, for each (layer, direction) in order ``layer * D + direction``:
W_ih [G*H, I_l], W_hh [G*H, H], b_ih [G*H], b_hh [G*H], row-major, back to back,
with G = 4 (LSTM, gate blocks i, f, g, o), 3 (GRU, r, z, n), 1 (tanh RNN), and
I_l = input_size for layer 0 and D*H above it.
"""

import numpy as np

MODES = ("rnn_tanh", "lstm", "gru", "gru_tf")
GATES = {"rnn_tanh": 1, "lstm": 4, "gru": 3, "gru_tf": 3}


def sigmoid(a):
    """Logistic function, evaluated without overflow for large |a|."""
    a = np.asarray(a, dtype=np.float64)
    out = np.empty_like(a)
    pos = a >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-a[pos]))
    e = np.exp(a[~pos])
    out[~pos] = e / (1.0 + e)
    return out


# ----------------------------------------------------------------------------
# canonical weight buffer
# ----------------------------------------------------------------------------

def layer_input_size(layer, input_size, hidden_size, bidirectional):
    return input_size if layer == 0 else (2 if bidirectional else 1) * hidden_size


def weight_shapes(mode, num_layers, bidirectional, input_size, hidden_size):
    """[(layer, dir, name, shape)] in canonical buffer order."""
    G = GATES[mode]
    D = 2 if bidirectional else 1
    H = hidden_size
    out = []
    for l in range(num_layers):
        I_l = layer_input_size(l, input_size, H, bidirectional)
        for d in range(D):
            out.append((l, d, "W_ih", (G * H, I_l)))
            out.append((l, d, "W_hh", (G * H, H)))
            out.append((l, d, "b_ih", (G * H,)))
            out.append((l, d, "b_hh", (G * H,)))
    return out


def unflatten_weights(flat, mode, num_layers, bidirectional, input_size, hidden_size):
    """Flat canonical buffer -> list (index l*D+d) of dicts of float64 arrays."""
    flat = np.asarray(flat, dtype=np.float64).ravel()
    D = 2 if bidirectional else 1
    params = [dict() for _ in range(num_layers * D)]
    pos = 0
    for l, d, name, shape in weight_shapes(mode, num_layers, bidirectional,
                                           input_size, hidden_size):
        n = int(np.prod(shape))
        params[l * D + d][name] = flat[pos:pos + n].reshape(shape).copy()
        pos += n
    if pos != flat.size:
        raise ValueError("flat weight buffer has %d elements, layout needs %d"
                         % (flat.size, pos))
    return params


def flatten_weights(params, mode, num_layers, bidirectional, input_size, hidden_size):
    """Inverse of ``unflatten_weights``."""
    D = 2 if bidirectional else 1
    chunks = []
    for l, d, name, shape in weight_shapes(mode, num_layers, bidirectional,
                                           input_size, hidden_size):
        a = np.asarray(params[l * D + d][name], dtype=np.float64)
        if a.shape != shape:
            raise ValueError("%s of (%d,%d) has shape %s, expected %s"
                             % (name, l, d, a.shape, shape))
        chunks.append(a.ravel())
    return np.concatenate(chunks)


# ----------------------------------------------------------------------------
# one direction of one layer
# ----------------------------------------------------------------------------

def _direction_forward(mode, x, h0, c0, p, reverse, lengths=None):
    """Run one direction over the whole sequence.

    x: [T, N, I_l]; h0, c0: [N, H].  Returns (out [T, N, H], h_T, c_T, tape);
    ``tape`` keeps, per processed step, the values the backward pass reuses.

    lengths: None, or the valid length of each sequence [N].  Step t of a
    sequence with t >= its length leaves the state unchanged and outputs zero,
    so the forward direction ends on the state of the last valid step and the
    reverse direction starts from h0 at the last valid step.
    """
    T = x.shape[0]
    valid = None if lengths is None else np.arange(T)[:, None] < np.asarray(lengths)[None, :]
    W_ih, W_hh, b_ih, b_hh = p["W_ih"], p["W_hh"], p["b_ih"], p["b_hh"]
    H = W_hh.shape[1]
    out = np.zeros((T, x.shape[1], H))
    h = h0.copy()
    c = c0.copy() if mode == "lstm" else None
    tape = []
    steps = range(T - 1, -1, -1) if reverse else range(T)
    for t in steps:
        h_prev, c_prev = h, c
        if mode == "rnn_tanh":
            h = np.tanh(x[t] @ W_ih.T + b_ih + h_prev @ W_hh.T + b_hh)
            tape.append(dict(t=t, h_prev=h_prev, h=h))
        elif mode == "lstm":
            a = x[t] @ W_ih.T + b_ih + h_prev @ W_hh.T + b_hh
            a_i, a_f, a_g, a_o = np.split(a, 4, axis=1)
            i, f, g, o = sigmoid(a_i), sigmoid(a_f), np.tanh(a_g), sigmoid(a_o)
            c = f * c_prev + i * g
            h = o * np.tanh(c)
            tape.append(dict(t=t, h_prev=h_prev, c_prev=c_prev, i=i, f=f, g=g,
                             o=o, c=c))
        elif mode == "gru":
            gi = x[t] @ W_ih.T + b_ih          # input part, blocks r, z, n
            gh = h_prev @ W_hh.T + b_hh        # recurrent part, blocks r, z, n
            i_r, i_z, i_n = np.split(gi, 3, axis=1)
            h_r, h_z, h_n = np.split(gh, 3, axis=1)
            r = sigmoid(i_r + h_r)
            z = sigmoid(i_z + h_z)
            n = np.tanh(i_n + r * h_n)
            h = (1.0 - z) * n + z * h_prev
            tape.append(dict(t=t, h_prev=h_prev, r=r, z=z, n=n, h_n=h_n))
        elif mode == "gru_tf":
            H = W_hh.shape[1]
            i_r, i_z, i_n = np.split(x[t] @ W_ih.T + b_ih, 3, axis=1)
            r = sigmoid(i_r + h_prev @ W_hh[:H].T + b_hh[:H])
            z = sigmoid(i_z + h_prev @ W_hh[H:2 * H].T + b_hh[H:2 * H])
            rh = r * h_prev                    # the reset gate acts before the matmul
            n = np.tanh(i_n + rh @ W_hh[2 * H:].T + b_hh[2 * H:])
            h = (1.0 - z) * n + z * h_prev
            tape.append(dict(t=t, h_prev=h_prev, r=r, z=z, n=n, rh=rh))
        else:
            raise ValueError("unknown mode %r" % mode)
        if valid is None:
            out[t] = h
        else:
            m = valid[t][:, None]
            tape[-1]["m"] = m
            out[t] = np.where(m, h, 0.0)
            h = np.where(m, h, h_prev)
            if c is not None:
                c = np.where(m, c, c_prev)
    return out, h, c, tape


def _direction_backward(mode, x, p, tape, dout, dh_last, dc_last):
    """Reverse-mode pass through one direction.

    dout: [T, N, H] gradient of the loss w.r.t. this direction's outputs;
    dh_last / dc_last: gradient w.r.t. the final state (hy / cy).
    Returns dx [T, N, I_l], dh0, dc0 and the parameter gradients.
    """
    W_ih, W_hh = p["W_ih"], p["W_hh"]
    grads = {k: np.zeros_like(v) for k, v in p.items()}
    dx = np.zeros_like(x)
    dh_next = dh_last.copy()
    dc_next = dc_last.copy() if mode == "lstm" else None
    for rec in reversed(tape):
        t = rec["t"]
        h_prev = rec["h_prev"]
        m = rec.get("m")
        if m is None:
            dh = dout[t] + dh_next
        else:
            # a step past the sequence's length passed h (and c) through and
            # output zero: its incoming state gradient goes straight back
            dh = np.where(m, dout[t] + dh_next, 0.0)
            carry_h = np.where(m, 0.0, dh_next)
            if mode == "lstm":
                carry_c = np.where(m, 0.0, dc_next)
                dc_next = np.where(m, dc_next, 0.0)
        if mode == "rnn_tanh":
            da = dh * (1.0 - rec["h"] ** 2)
            dgx = dgh = da
            dh_next = da @ W_hh
        elif mode == "lstm":
            i, f, g, o, c, c_prev = (rec[k] for k in ("i", "f", "g", "o", "c", "c_prev"))
            tc = np.tanh(c)
            do = dh * tc
            dc = dc_next + dh * o * (1.0 - tc ** 2)
            di = dc * g
            dg = dc * i
            df = dc * c_prev
            da = np.concatenate([di * i * (1.0 - i), df * f * (1.0 - f),
                                 dg * (1.0 - g ** 2), do * o * (1.0 - o)], axis=1)
            dc_next = dc * f
            dgx = dgh = da
            dh_next = da @ W_hh
        elif mode == "gru":
            r, z, n, h_n = rec["r"], rec["z"], rec["n"], rec["h_n"]
            dn = dh * (1.0 - z)
            dz = dh * (h_prev - n)
            da_n = dn * (1.0 - n ** 2)
            dr = da_n * h_n
            da_z = dz * z * (1.0 - z)
            da_r = dr * r * (1.0 - r)
            dgx = np.concatenate([da_r, da_z, da_n], axis=1)
            dgh = np.concatenate([da_r, da_z, da_n * r], axis=1)
            dh_next = dh * z + dgh @ W_hh
        elif mode == "gru_tf":
            H = W_hh.shape[1]
            r, z, n, rh = rec["r"], rec["z"], rec["n"], rec["rh"]
            dn = dh * (1.0 - z)
            dz = dh * (h_prev - n)
            da_n = dn * (1.0 - n ** 2)
            d_rh = da_n @ W_hh[2 * H:]         # gradient of the loss w.r.t. r * h
            da_r = d_rh * h_prev * r * (1.0 - r)
            da_z = dz * z * (1.0 - z)
            dgx = dgh = np.concatenate([da_r, da_z, da_n], axis=1)
            dh_next = dh * z + da_r @ W_hh[:H] + da_z @ W_hh[H:2 * H] + d_rh * r
            # the candidate's recurrent weights multiply r * h, not h
            whh_in = np.concatenate([np.repeat(h_prev[None], 2, 0), rh[None]], 0)
        else:
            raise ValueError("unknown mode %r" % mode)
        if m is not None:
            dh_next = dh_next + carry_h
            if mode == "lstm":
                dc_next = dc_next + carry_c
        dx[t] = dgx @ W_ih
        grads["W_ih"] += dgx.T @ x[t]
        if mode == "gru_tf":
            for g in range(3):
                blk = slice(g * H, (g + 1) * H)
                grads["W_hh"][blk] += dgh[:, blk].T @ whh_in[g]
        else:
            grads["W_hh"] += dgh.T @ h_prev
        grads["b_ih"] += dgx.sum(axis=0)
        grads["b_hh"] += dgh.sum(axis=0)
    return dx, dh_next, dc_next, grads


# ----------------------------------------------------------------------------
# whole stack
# ----------------------------------------------------------------------------

def forward(mode, x, h0, c0, params, num_layers, bidirectional, lengths=None, dropout=0.0,
            masks=None):
    """Training forward of the stack.

    x: [T, N, I]; h0, c0: [L*D, N, H] (c0 ignored unless LSTM; None = zeros);
    params: list (index l*D+d) of dicts W_ih, W_hh, b_ih, b_hh.
    lengths: None (every sequence has length T) or the valid length of each
    sequence, [N] integers in 0..T, for padded variable-length batches (the
    PyTorch packed-sequence semantics: y is zero past a sequence's length, hy
    is the state after its last valid step in each direction).
    dropout, masks: inter-layer dropout probability in [0, 1) and the L-1
    masks [T, N, D*H] (0/1) drawn for it; masks None means no dropout.
    Returns (y [T, N, D*H], hy [L*D, N, H], cy [L*D, N, H] or None, cache).
    """
    x = np.asarray(x, dtype=np.float64)
    D = 2 if bidirectional else 1
    H = params[0]["W_hh"].shape[1]
    T, N = x.shape[0], x.shape[1]
    if lengths is not None:
        lengths = np.asarray(lengths)
        if lengths.shape != (N,) or lengths.min(initial=0) < 0 or lengths.max(initial=0) > T:
            raise ValueError("lengths must be [N] integers in 0..T")
    if masks is not None:
        masks = [np.asarray(m, dtype=np.float64) for m in masks]
        if not 0.0 <= dropout < 1.0 or len(masks) != num_layers - 1 or any(
                m.shape != (T, N, D * H) or not np.isin(m, (0.0, 1.0)).all() for m in masks):
            raise ValueError("masks must be L-1 arrays [T, N, D*H] of 0/1, dropout in [0, 1)")
    if h0 is None:
        h0 = np.zeros((num_layers * D, N, H))
    if c0 is None:
        c0 = np.zeros((num_layers * D, N, H))
    h0 = np.asarray(h0, dtype=np.float64)
    c0 = np.asarray(c0, dtype=np.float64)
    hy = np.zeros((num_layers * D, N, H))
    cy = np.zeros((num_layers * D, N, H)) if mode == "lstm" else None
    layer_in = x
    cache = dict(mode=mode, L=num_layers, D=D, inputs=[], tapes=[], masks=masks,
                 keep=1.0 / (1.0 - dropout))
    for l in range(num_layers):
        outs = []
        cache["inputs"].append(layer_in)
        for d in range(D):
            k = l * D + d
            out, hT, cT, tape = _direction_forward(mode, layer_in, h0[k], c0[k],
                                                   params[k], reverse=(d == 1),
                                                   lengths=lengths)
            outs.append(out)
            hy[k] = hT
            if cy is not None:
                cy[k] = cT
            cache["tapes"].append(tape)
        layer_in = np.concatenate(outs, axis=2)
        if masks is not None and l < num_layers - 1:
            layer_in = layer_in * masks[l] * cache["keep"]
    return layer_in, hy, cy, cache


def backward(params, cache, dy, dhy=None, dcy=None):
    """Backward of ``forward`` for loss = sum(y*dy) + sum(hy*dhy) + sum(cy*dcy).

    Returns (dx [T, N, I], dh0 [L*D, N, H], dc0 or None, dparams) where dparams
    has the structure of ``params``.
    """
    mode, L, D = cache["mode"], cache["L"], cache["D"]
    dy = np.asarray(dy, dtype=np.float64)
    H = params[0]["W_hh"].shape[1]
    N = dy.shape[1]
    if dhy is None:
        dhy = np.zeros((L * D, N, H))
    if dcy is None:
        dcy = np.zeros((L * D, N, H))
    dhy = np.asarray(dhy, dtype=np.float64)
    dcy = np.asarray(dcy, dtype=np.float64)
    dh0 = np.zeros((L * D, N, H))
    dc0 = np.zeros((L * D, N, H)) if mode == "lstm" else None
    dparams = [None] * (L * D)
    d_out = dy
    for l in range(L - 1, -1, -1):
        layer_in = cache["inputs"][l]
        d_in = np.zeros_like(layer_in)
        for d in range(D):
            k = l * D + d
            dx_d, dh_first, dc_first, g = _direction_backward(
                mode, layer_in, params[k], cache["tapes"][k],
                d_out[:, :, d * H:(d + 1) * H], dhy[k], dcy[k])
            d_in += dx_d
            dh0[k] = dh_first
            if dc0 is not None:
                dc0[k] = dc_first
            dparams[k] = g
        d_out = d_in
        if cache.get("masks") is not None and l > 0:
            d_out = d_out * cache["masks"][l - 1] * cache["keep"]
    return d_out, dh0, dc0, dparams


def loss(y, hy, cy, dy, dhy=None, dcy=None):
    """The scalar whose gradient ``backward`` returns."""
    s = float(np.sum(y * dy))
    if dhy is not None:
        s += float(np.sum(hy * dhy))
    if cy is not None and dcy is not None:
        s += float(np.sum(cy * dcy))
    return s


def run_flat(mode, num_layers, bidirectional, input_size, hidden_size,
             x, h0, c0, w_flat, dy, dhy, dcy, lengths=None, dropout=0.0, masks=None):
    """Forward + backward on the canonical flat weight buffer.

    Returns a dict of float64 arrays: y, hy, cy, dx, dh0, dc0, dW (flat).
    ``lengths``, ``dropout``, ``masks``: as for ``forward``.
    """
    params = unflatten_weights(w_flat, mode, num_layers, bidirectional,
                               input_size, hidden_size)
    y, hy, cy, cache = forward(mode, x, h0, c0, params, num_layers, bidirectional,
                               lengths, dropout, masks)
    dx, dh0, dc0, dparams = backward(params, cache, dy, dhy,
                                     dcy if mode == "lstm" else None)
    dW = flatten_weights(dparams, mode, num_layers, bidirectional,
                         input_size, hidden_size)
    return dict(y=y, hy=hy, cy=cy, dx=dx, dh0=dh0, dc0=dc0, dW=dW)
