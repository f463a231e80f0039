"""GB300-native self-speculative block decoding.

The decode round of a shared AR / block-diffusion decoder (GravityOCR,
"Diffusion Drafts, AR Verifies", §3.2): one draft forward of the boundary
token plus B [M] tokens, one causal verify forward, and an on-device
accept / commit / roll-back step, all in hand-written sm_103a CUDA behind the
C ABI declared in include/gocr.h.

Importing the package loads nothing; `gocr.load()` opens the shared library
and fails loudly when it has not been built.
"""
from . import synth  # noqa: F401

__all__ = ["synth"]
