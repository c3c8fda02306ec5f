"""Build tests/probe/libufp4_probe.so: libufp4 with csrc/quantize.cu and
csrc/gemm.cu recompiled under -DUFP4_PROBE, which adds the capture hooks of
probe_hooks.inc and the entry points of probe_entry.inc and probe_gemm.inc.

Test infrastructure only.  The probe library exports libufp4's whole C ABI
(the same kernels, plus hooks that record the values each quantization path
hands to its block scale, and a switch that makes a GEMM's wait run out) and
three probe calls, ufp4probe_capture, ufp4probe_div_qmax and
ufp4probe_gemm_waits.  Nothing in the library or the benchmark loads it.
"""
import os

from fp4_quantized_numerics_gb300 import build as libbuild

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libufp4_probe.so")


def build_probe() -> str:
    return libbuild.build_variant(LIB, os.path.join(HERE, "_build"), ["-DUFP4_PROBE"],
                                  {"quantize.cu", "gemm.cu"}, HERE)


if __name__ == "__main__":
    print(build_probe())
