"""CPU oracle for the attention forward and backward: test infrastructure, never
the product path.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  It depends on numpy alone and
shares no code with the CUDA library.
"""

from .exact import (attention, attention_backward, attention_backward_plane, attention_plane,
                    attention_rows, online_tiled, softmax_probs)

__all__ = ["attention", "attention_backward", "attention_backward_plane", "attention_plane",
           "attention_rows", "online_tiled", "softmax_probs"]
