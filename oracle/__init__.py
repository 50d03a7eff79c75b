"""CPU float64 oracle for exact attention.  Test infrastructure only: the
product path (the CUDA library and its Python binding) never imports it."""

from .attention import (  # noqa: F401
    backward,
    backward_heads,
    forward,
    forward_heads,
    probabilities,
    scores,
)
