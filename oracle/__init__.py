"""CPU float64 oracle for sink-aware attention (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA library.
"""
from .sinkattn_ref import WINDOW_INF, decode_forward, forward, forward_backward, unmasked_pairs, visible  # noqa: F401
