"""CPU float64 oracles (test infrastructure only): varlen GQA attention
(attention.py), and the Gated DeltaNet and Kimi Delta recurrences over packed
documents (gated_delta.py, kimi_delta.py).

Only tests, the smoke check and the benchmark's CPU-baseline leg import this
package; the library never does.
"""
from .attention import (backward, forward, probabilities, segments, unmasked_pairs, visible_mask,  # noqa: F401
                        visible_ranges)
