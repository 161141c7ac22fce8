"""GB300-native generalised gated delta-rule recurrence (GDN, KLA, PGDN, Diagonal KDN).

The compute lives in ``libdr.so`` (CUDA for sm_103a behind the C ABI of
include/dr.h).  ``dr`` is its ctypes binding, ``runner`` allocates outputs and
calls it, ``workloads`` draws the seeded synthetic inputs, ``build`` compiles
the library.  Importing ``dr`` (or ``runner``) requires the built library.
"""

__all__ = ["workloads", "build"]
