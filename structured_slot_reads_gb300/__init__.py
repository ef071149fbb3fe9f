"""GB300-native structured slot reads: the DiffusionGemma denoise step on sm_103a.

The compute lives in ``libdg.so`` (hand-written CUDA for sm_103a behind a C
ABI declared in ``include/dg.h``).  ``structured_slot_reads_gb300.dg`` is the
thin ctypes binding with the same call names; ``configs`` holds workload
shapes and ``inputs`` the seeded synthetic input generators.  Importing the
package does not load the library; ``dg`` does, and raises if it is missing.
"""
__all__ = ["configs", "inputs", "dg"]
