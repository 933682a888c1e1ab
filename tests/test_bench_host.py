"""Host logic of bench.py that needs no GPU: the code-only source hash that
keys the recorded DRAM traffic (comments and layout do not change it, code
does, string literals are kept) and the traffic lookup."""
import argparse
import os
import shutil

import bench


def test_code_only_drops_comments_keeps_literals():
    src = ('int a = 1; // trailing\n/* block\n comment */ const char *s = "x // y /* z */";\n'
           "char q = '\"'; char e = '\\\\'; int b = a / 2;  // end")
    out = bench._code_only(src)
    assert "trailing" not in out and "block" not in out and "end" not in out
    assert '"x // y /* z */"' in out
    assert "'\"'" in out and "'\\\\'" in out
    assert "int b = a / 2;" in out


def test_code_only_ignores_layout_not_code():
    a = "int  f(int x)\n{\n    return x + 1; // one\n}\n"
    b = "/* the same function */ int f(int x) { return x + 1; }"
    c = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_source_hash_follows_code_not_comments(tmp_path):
    csrc = os.path.join(bench.ROOT, "paged_gqa_decode_03_gb300", "csrc")
    dst = tmp_path / "paged_gqa_decode_03_gb300" / "csrc"
    shutil.copytree(csrc, dst, ignore=shutil.ignore_patterns("*.o", "*.so"))
    root = bench.ROOT
    try:
        bench.ROOT = str(tmp_path)
        h0 = bench.kernel_source_hash(bench.DECODE_HASH_EXCLUDE)
        v0 = bench.kernel_source_hash(bench.VARLEN_HASH_EXCLUDE)
        f = dst / "pgd_varlen.cu"
        f.write_text(f.read_text() + "\n// a comment only\n")
        assert bench.kernel_source_hash(bench.VARLEN_HASH_EXCLUDE) == v0
        f.write_text(f.read_text() + "\nnamespace pgd { constexpr int kUnused = 1; }\n")
        assert bench.kernel_source_hash(bench.VARLEN_HASH_EXCLUDE) != v0
        # the decode kernels' hash leaves pgd_varlen.cu out
        assert bench.kernel_source_hash(bench.DECODE_HASH_EXCLUDE) == h0
    finally:
        bench.ROOT = root


def test_traffic_recorded_for_the_current_sources():
    """When bench.TRAFFIC holds figures for the current kernel code, they
    cover every fp16 and quantised decode workload and the three varlen
    ones (after a code change the bench reports traffic null until they are
    taken again)."""
    import pytest
    hd = bench.kernel_source_hash(bench.DECODE_HASH_EXCLUDE)
    hv = bench.kernel_source_hash(bench.VARLEN_HASH_EXCLUDE)
    if hd not in bench.TRAFFIC or hv not in bench.TRAFFIC:
        pytest.skip("no DRAM traffic recorded for the current kernel code yet")
    d = bench.TRAFFIC[hd]
    for key in [("long_context", 512), ("long_context", 256), ("ragged_tails", 256),
                ("serving_mix", 512), ("batch_decode", 512), ("batch_decode_q8", 512),
                ("long_context_q8", 512), ("ragged_tails_q8", 256), ("serving_mix_q8", 512)]:
        assert d[key] > 0
        plain = argparse.Namespace(layout="head_major", append=False)
        assert bench.traffic_for(key[0].replace("_q8", ""), key[1], key[0].endswith("_q8"),
                                 plain) == d[key]
    # other layouts and the fused append run other instantiations: no figure
    for other in (argparse.Namespace(layout="token_major", append=False),
                  argparse.Namespace(layout="head_major", append=True)):
        assert bench.traffic_for("batch_decode", 512, False, other) is None
    v = bench.TRAFFIC[hv]
    assert set(v) == {("chunked_prefill", 8320), ("prefill", 2048), ("spec_verify", 4096)}
