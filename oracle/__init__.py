"""Float64 CPU oracle (test infrastructure only; see ``rnn_oracle``)."""
from .rnn_oracle import (MODES, GATES, sigmoid, forward, backward, loss, run_flat,
                         unflatten_weights, flatten_weights, weight_shapes,
                         layer_input_size)

__all__ = ["MODES", "GATES", "sigmoid", "forward", "backward", "loss", "run_flat",
           "unflatten_weights", "flatten_weights", "weight_shapes",
           "layer_input_size"]
