"""GB300-native EAGLE-3 draft-and-verify round.

The compute path is ``libeagle3.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/eagle3.h``).  ``eagle3`` is its thin ctypes
binding; ``synth`` holds the seeded synthetic-input generators.  Importing the
package does not load the library: ``from eagle_speculative_decoding_round_gb300
import eagle3`` does, and fails loudly if it has not been built.
"""
__all__ = ["eagle3", "synth", "build"]
