"""A naive unrolled-graph recomputation of the RNN stack, for pinning the oracle.

Every multiply, add and nonlinearity of every time step is its own node in a
scalar reverse-mode autodiff graph (no matrices, no hand-written backward).  The
cell equations are taken in the forms the pages print:

* GRU: the PyTorch code in "rnn training example?" (oneDNN issue #218,
  mingfeima's comment): resetgate = sigmoid(i_r + h_r), inputgate =
  sigmoid(i_i + h_i), newgate = tanh(i_n + resetgate * h_n),
  hy = newgate + inputgate * (hidden - newgate) -- deliberately the other
  algebraic form of the update than the oracle's (1 - z) * n + z * h.
* LSTM: standard gates i, f, g, o (the pages name LSTM without equations).
* tanh RNN: h' = tanh(W_ih x + b_ih + W_hh h + b_hh).

It is only practical for tiny sizes.
"""

import math


class V:
    """Scalar node: value plus (parent, local derivative) edges."""
    __slots__ = ("val", "edges", "grad")

    def __init__(self, val, edges=()):
        self.val = float(val)
        self.edges = edges
        self.grad = 0.0

    def __add__(self, o):
        o = o if isinstance(o, V) else V(o)
        return V(self.val + o.val, ((self, 1.0), (o, 1.0)))

    __radd__ = __add__

    def __sub__(self, o):
        o = o if isinstance(o, V) else V(o)
        return V(self.val - o.val, ((self, 1.0), (o, -1.0)))

    def __rsub__(self, o):
        o = o if isinstance(o, V) else V(o)
        return o - self

    def __mul__(self, o):
        o = o if isinstance(o, V) else V(o)
        return V(self.val * o.val, ((self, o.val), (o, self.val)))

    __rmul__ = __mul__


def vsigmoid(a):
    s = 1.0 / (1.0 + math.exp(-a.val))
    return V(s, ((a, s * (1.0 - s)),))


def vtanh(a):
    t = math.tanh(a.val)
    return V(t, ((a, 1.0 - t * t),))


def backprop(root):
    order, seen = [], set()
    stack = [(root, False)]
    while stack:
        node, done = stack.pop()
        if done:
            order.append(node)
            continue
        if id(node) in seen:
            continue
        seen.add(id(node))
        stack.append((node, True))
        for p, _ in node.edges:
            if id(p) not in seen:
                stack.append((p, False))
    root.grad = 1.0
    for node in reversed(order):
        for p, d in node.edges:
            p.grad += d * node.grad


def _leaf(a):
    """Nested lists of V leaves mirroring a numpy array."""
    if hasattr(a, "ndim") and a.ndim > 0:
        return [_leaf(e) for e in a]
    return V(float(a))


def _grad(v):
    if isinstance(v, list):
        return [_grad(e) for e in v]
    return v.grad


def _val(v):
    if isinstance(v, list):
        return [_val(e) for e in v]
    return v.val


def _dot(row, vec):
    acc = V(0.0)
    for w, v in zip(row, vec):
        acc = acc + w * v
    return acc


def run(mode, L, bidir, x, h0, c0, params, dy, dhy, dcy):
    """Forward + backward through the unrolled scalar graph.

    Arguments are numpy float64 arrays (params: list of dicts by l*D+d).
    Returns dict of nested lists: y, hy, cy, dx, dh0, dc0, dparams.
    """
    D = 2 if bidir else 1
    T, N = x.shape[0], x.shape[1]
    H = params[0]["W_hh"].shape[1]
    X = _leaf(x)
    H0 = _leaf(h0)
    C0 = _leaf(c0) if c0 is not None else None
    P = [{k: _leaf(v) for k, v in p.items()} for p in params]
    layer_in = X
    hy = [None] * (L * D)
    cy = [None] * (L * D)
    for l in range(L):
        outs = []
        for d in range(D):
            k = l * D + d
            p = P[k]
            out = [[None] * N for _ in range(T)]
            h = [list(H0[k][n]) for n in range(N)]
            c = [list(C0[k][n]) for n in range(N)] if mode == "lstm" else None
            steps = range(T - 1, -1, -1) if d == 1 else range(T)
            for t in steps:
                new_h, new_c = [], []
                for n in range(N):
                    xin = layer_in[t][n]
                    hn = h[n]

                    def gi(row):
                        return _dot(p["W_ih"][row], xin) + p["b_ih"][row]

                    def gh(row):
                        return _dot(p["W_hh"][row], hn) + p["b_hh"][row]

                    hv, cv = [], []
                    if mode == "gru_tf":
                        # TensorFlow flavour: every unit's reset gate first,
                        # then the candidate's recurrent product over r * h
                        rs = [vsigmoid(gi(j) + gh(j)) for j in range(H)]
                        rh = [rs[k] * hn[k] for k in range(H)]
                    for j in range(H):
                        if mode == "rnn_tanh":
                            hv.append(vtanh(gi(j) + gh(j)))
                        elif mode == "lstm":
                            ig = vsigmoid(gi(j) + gh(j))
                            fg = vsigmoid(gi(H + j) + gh(H + j))
                            gg = vtanh(gi(2 * H + j) + gh(2 * H + j))
                            og = vsigmoid(gi(3 * H + j) + gh(3 * H + j))
                            cj = fg * c[n][j] + ig * gg
                            cv.append(cj)
                            hv.append(og * vtanh(cj))
                        elif mode == "gru_tf":
                            inputgate = vsigmoid(gi(H + j) + gh(H + j))
                            newgate = vtanh(gi(2 * H + j) + _dot(p["W_hh"][2 * H + j], rh) +
                                            p["b_hh"][2 * H + j])
                            hv.append(newgate + inputgate * (hn[j] - newgate))
                        else:
                            resetgate = vsigmoid(gi(j) + gh(j))
                            inputgate = vsigmoid(gi(H + j) + gh(H + j))
                            newgate = vtanh(gi(2 * H + j) + resetgate * gh(2 * H + j))
                            hv.append(newgate + inputgate * (hn[j] - newgate))
                    new_h.append(hv)
                    new_c.append(cv)
                h = new_h
                if mode == "lstm":
                    c = new_c
                for n in range(N):
                    out[t][n] = h[n]
            outs.append(out)
            hy[k] = h
            cy[k] = c
        layer_in = [[sum((outs[d][t][n] for d in range(D)), [])
                     for n in range(N)] for t in range(T)]
    y = layer_in
    loss = V(0.0)
    for t in range(T):
        for n in range(N):
            for j in range(D * H):
                loss = loss + y[t][n][j] * float(dy[t][n][j])
    for k in range(L * D):
        for n in range(N):
            for j in range(H):
                loss = loss + hy[k][n][j] * float(dhy[k][n][j])
                if mode == "lstm":
                    loss = loss + cy[k][n][j] * float(dcy[k][n][j])
    backprop(loss)
    return dict(y=_val(y), hy=_val(hy), cy=_val(cy) if mode == "lstm" else None,
                dx=_grad(X), dh0=_grad(H0), dc0=_grad(C0) if C0 is not None else None,
                dparams=[{k: _grad(v) for k, v in p.items()} for p in P])
