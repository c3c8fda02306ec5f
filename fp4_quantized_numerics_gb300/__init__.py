"""GB300-native UFP4 hot path: fused RHT + 4-bit block quantization and
block-scaled FP4 GEMMs, behind the libufp4 C ABI (include/ufp4.h).

Submodules:
  ufp4    -- thin ctypes binding of libufp4 (argument marshalling only);
  inputs  -- seeded synthetic workloads (no quantization arithmetic);
  build   -- compiles libufp4.so for sm_103a with nvcc.
"""
