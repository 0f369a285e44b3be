"""CPU float64 oracle for varlen GQA attention (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline leg import this
package; the library never does.
"""
from .attention import (backward, forward, probabilities, segments, unmasked_pairs, visible_mask,  # noqa: F401
                        visible_ranges)
