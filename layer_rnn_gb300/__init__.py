"""GB300-native fused multi-layer RNN operator (LSTM, GRU, tanh RNN).

The compute path lives in ``liblayer_rnn.so`` (hand-written CUDA for sm_103a
behind a C ABI, declared in ``include/layer_rnn.h``).  ``layer_rnn_gb300.binding``
loads it with ctypes; importing this package does not load the library, so the
seeded workload generator (``layer_rnn_gb300.workloads``) is usable without a
GPU.
"""

__all__ = ["binding", "workloads"]
