"""bench.py's use of the committed ncu traffic (profiles/traffic.json), on the
CPU: a kernel's DRAM bytes are reported only while the source they were taken
on is unchanged, where "source" is the kernel's file and the headers of its
own that it includes, comments and whitespace aside."""
import importlib.util
import os
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture()
def bench_in(tmp_path):
    """bench.py loaded against a copy of the kernel sources and profiles."""
    csrc = os.path.join("gqa_attention_preallocated_qa_gb300", "csrc")
    shutil.copytree(os.path.join(ROOT, csrc), tmp_path / csrc)
    shutil.copytree(os.path.join(ROOT, "profiles"), tmp_path / "profiles")
    spec = importlib.util.spec_from_file_location("bench_copy", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.ROOT = str(tmp_path)
    return mod, tmp_path / csrc


def edit(path, old, new):
    text = path.read_text()
    assert old in text
    path.write_text(text.replace(old, new, 1))


def test_comments_do_not_change_the_digest_code_does(bench_in):
    bench, csrc = bench_in
    # the committed profiles, read against the copied sources
    fresh = {k: bench.traffic_for(k, 0) is not None for k in ("k2_prefill", "k3_decode")}
    before = {k: bench.kernel_source_digest(k) for k in ("k1_norm", "k2_prefill", "k3_decode")}
    # a comment and whitespace in the prefill items header: no change anywhere
    edit(csrc / "k2_items.h", "namespace qa {", "namespace qa {\n// a note\n\n")
    assert {k: bench.kernel_source_digest(k) for k in before} == before
    # code in that header: the prefill kernel's digest changes, the others' do not
    edit(csrc / "k2_items.h", "it.jmask = it.qmin / 128;", "it.jmask = it.qmin / 64;")
    after = {k: bench.kernel_source_digest(k) for k in before}
    assert after["k2_prefill"] != before["k2_prefill"]
    assert after["k1_norm"] == before["k1_norm"] and after["k3_decode"] == before["k3_decode"]
    assert bench.traffic_for("k2_prefill", 0) is None
    assert (bench.traffic_for("k3_decode", 0) is not None) == fresh["k3_decode"]
    # a shared device header changes every kernel's digest
    edit(csrc / "qa_device.cuh", "namespace qa {", "namespace qa {\nconstexpr int kUnused = 1;")
    assert all(bench.kernel_source_digest(k) != after[k] for k in after)
