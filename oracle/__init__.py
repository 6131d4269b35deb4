"""fp64 CPU oracle for exact attention -- test infrastructure, not part of the product path.

Only the tests, the smoke check and the bench's CPU-baseline leg import this
package.  See ``oracle/attention.py`` for what it computes and what pins it.
"""
from .attention import (  # noqa: F401
    attention_backward,
    attention_forward,
    forward_rows,
    head_backward_rows,
    head_backward_rowwise,
    probabilities,
    scores,
)
