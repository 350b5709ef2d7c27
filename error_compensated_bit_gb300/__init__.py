"""GB300-native (sm_103a) 1-bit Adam / APMSqueeze compression-stage optimizer step.

``ob``         the binding of the C ABI (include/ob.h) to the CUDA library
``optimizer``  OneBitAdam, a user-facing object holding the state in device memory
``synth``      seeded synthetic workloads (inputs only)
"""
from . import ob  # noqa: F401

__all__ = ["ob"]
