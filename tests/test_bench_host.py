"""Host-side pieces of bench.py, without a GPU: the per-workload L2 rule, the
algorithmic record bytes it is based on, the lookup of ncu traffic in the
committed profile summaries (keyed by the sha256 of the kernel sources), and
the operation count of the tridiagonal build."""
import types

import pytest

import bench
import workloads as W

F32_RECORD = (9 * 128 + 8 * 64) * 4          # fp32 record at r = 8, B = 64: 6656 bytes
I4_RECORD = 1456                             # quantised record at r = 8, B = 64


def _torch_with_l2(l2_bytes):
    props = types.SimpleNamespace(L2_cache_size=l2_bytes)
    cuda = types.SimpleNamespace(get_device_properties=lambda i: props)
    return types.SimpleNamespace(cuda=cuda)


def test_record_stream_bytes_counts_candidates_only():
    # 1M tokens, one sequence: 16384 pages, of which 16382 candidates, 8 KV heads
    w = W.get("1m")
    assert bench.record_stream_bytes(w, F32_RECORD) == 16382 * 8 * F32_RECORD
    # a partial tail page is neither summarised nor a candidate
    t = W.get("tiny").with_(seq_lens=(64 * 10 + 5,), batch=1)
    assert bench.record_stream_bytes(t, 100) == (10 - 1) * t.n_kv_heads * 100
    # two pages or fewer: no candidates; 131 tokens (pages 0, 1 complete, page
    # 2 partial and forced): page 1 only
    s = W.get("tiny").with_(seq_lens=(0, 64, 64 + 3, 64 * 2), batch=4)
    assert bench.record_stream_bytes(s, 100) == 0
    s = W.get("tiny").with_(seq_lens=(64 * 2 + 3,), batch=1)
    assert bench.record_stream_bytes(s, 100) == 1 * s.n_kv_heads * 100


@pytest.mark.parametrize("name,rec,flush", [
    ("1m", F32_RECORD, False), ("long128k", F32_RECORD, False),
    ("llama32k", F32_RECORD, True), ("qwen16k", F32_RECORD, True), ("tiny", F32_RECORD, True),
    ("1m", I4_RECORD, True), ("long128k", I4_RECORD, True),
])
def test_l2_rule(name, rec, flush):
    """No flush exactly when a step streams at least twice the L2 (129 MiB
    here) of records."""
    got, note = bench.l2_policy(_torch_with_l2(129 * 2 ** 20), W.get(name), rec)
    assert got is flush, (name, rec, note)
    assert (note == bench.FLUSH_NOTE) is flush


def test_profile_traffic_follows_the_source_digest(tmp_path, monkeypatch):
    src = tmp_path / "kern.cu"
    src.write_text("// kernel v1\n")
    other = tmp_path / "common.cuh"
    other.write_text("// helpers\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.source_digest(["kern.cu", "common.cuh"])
    (tmp_path / "profiles" / "select_demo.md").write_text(
        "# demo\n\n- source: kern.cu, common.cuh\n"
        f"- source_sha256: {digest}\n- dram_bytes_per_launch: 123456\n")
    traffic, path = bench.profile_traffic("select", "demo")
    assert traffic == 123456.0 and path.endswith("select_demo.md")
    # a changed kernel source voids the committed counters
    src.write_text("// kernel v2\n")
    assert bench.profile_traffic("select", "demo")[0] is None
    # no summary for a workload: no traffic
    assert bench.profile_traffic("select", "none") == (None, None)


def test_committed_select_profiles_parse():
    """Every committed select summary names existing source files and carries
    a digest and a DRAM figure (whether the digest still matches the sources
    is the bench's business: it reports null traffic when it does not)."""
    import os
    for name in ("1m", "long128k", "llama32k", "llama32k_i4"):
        path = os.path.join(bench.ROOT, "profiles", f"select_{name}.md")
        fields = {}
        for line in open(path):
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip()
        files = [x.strip() for x in fields["source"].split(",")]
        assert all(os.path.exists(os.path.join(bench.ROOT, f)) for f in files), name
        assert len(fields["source_sha256"]) == 64
        assert float(fields["dram_bytes_per_launch"]) > float(fields["algorithmic_bytes_per_launch"]) * 0.99


def test_tridiagonal_flop_count_scales_with_page_heads():
    one = bench.trd_flop_count(1, 64)
    assert one > 2 * 64 * 64 * 128                 # at least the Gram product
    assert bench.trd_flop_count(1000, 64) == pytest.approx(1000 * one)
    assert bench.trd_flop_count(1, 64, r=16) > one
