"""GB300-native (sm_103a) speculative-decoding verify step.

The compute path is the C-ABI library ``libspecverify.so`` built from
``csrc/`` (see ``include/spec_verify.h``); ``binding`` is its thin ctypes
binding and ``workloads`` the seeded synthetic input generator.  Submodules
are imported lazily so that the generator can be used without the library.
"""

__all__ = ["binding", "workloads", "build"]
