"""fp64 CPU oracle for exact attention.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg may
import or run anything in this package. The CUDA library never calls it and it
never calls the CUDA library: the two share no code, headers, helpers or
constants. Inputs reach both sides from ``exact_attention_gb300.synth``, which
only draws and rounds random numbers.

What it computes is the plain definition, written out in float64 with numpy:
the full score matrix, a max-subtracted softmax, and the textbook chain rule
for the gradients. See ``oracle.attention`` for the functions and the passage
each one follows.

``oracle.fp8`` writes out the FP8 forward's steps (Hadamard-times-sign
transform, E4M3 block quantisation) in float64 for the FP8 path's tests.

Parity pins (``tests/test_oracle.py``, ``tests/test_oracle_fp8.py``): high-precision
brute force on tiny inputs (forward values and mpmath derivatives of the backward),
closed forms, invariants and finite differences; for the FP8 steps a brute-force
E4M3 rounding, PyTorch's float8 conversion, the transform's orthogonality and the
FP8 error against exact attention. No function here is "parity unpinned".
"""
from .attention import (  # noqa: F401
    scores,
    probabilities,
    split_bounds,
    forward,
    backward,
    delta,
    decode,
    decode_partials,
    decode_combine,
)
