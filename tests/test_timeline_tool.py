"""The timeline tool's stamps still apply to the decode kernel's source (no
GPU, no compile: the anchors are checked as text)."""
from paged_gqa_decode_03_gb300 import timeline


def test_instrumentation_applies():
    cuh, tu = timeline.instrumented_sources()
    assert cuh.count("TL(") == len(timeline._PATCHES) + cuh.count("#define TL(")
    assert '#include "pgd_kernels_tl.cuh"' in tu and "tl_get" in tu


def test_varlen_instrumentation_applies():
    src = timeline.instrumented_varlen_source()
    assert src.count("TL(") == len(timeline._VPATCHES) + src.count("#define TL(")
    assert "tl_clear" in src
