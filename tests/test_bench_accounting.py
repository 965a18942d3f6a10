"""bench.py's byte accounting and its use of the committed ncu summaries,
checked on the CPU.

- The Qwen3-8B layer's K/V bytes per decode step are the pages' figure:
  16 sequences x 4,164 tokens x 4 KiB per token (K + V, Hkv 8, D 128, bf16).
- The algorithmic bytes of one decode launch add the query, the fp32 output,
  the table entries the lengths need and the lengths themselves.
- `roofline.traffic` is read from a profile only while the profile's source
  hash matches the kernel sources it names."""
import os

import numpy as np
import pytest

import bench
import workloads


def test_qwen3_kv_bytes_are_the_pages_figure():
    lens = np.full(16, 4164, np.int32)
    assert bench.kv_bytes(lens, 8, 128, 2) == 16 * 4164 * 4096 == 272_891_904


def test_decode_algorithmic_bytes_add_query_output_table_and_lengths():
    lens = np.full(16, 4164, np.int32)
    kv = 272_891_904
    query = 16 * 32 * 128 * 2
    out = 16 * 32 * 128 * 4
    table = 16 * 261 * 4          # cdiv(4164, 16) = 261 blocks per sequence
    assert bench.decode_alg_bytes(lens, 32, 8, 128, 16, 2) == kv + query + out + table + 16 * 4
    # a contiguous cache reads no table
    assert bench.decode_alg_bytes(lens, 32, 8, 128, None, 2) == kv + query + out + 16 * 4
    # ragged lengths: only valid tokens and the blocks they need count
    ragged = np.array([0, 1, 16, 17], np.int32)
    assert bench.decode_alg_bytes(ragged, 4, 2, 64, 16, 2) == (
        34 * 2 * 64 * 2 * 2 + 4 * 4 * 64 * 2 + 4 * 4 * 64 * 4 + (0 + 1 + 1 + 2) * 4 + 4 * 4)
    assert bench.tables_bytes(ragged, 16) == 4 * 4


def _fake_tree(tmp_path, source_text, sha_in_profile, traffic=123456):
    csrc = tmp_path / "paged_kv_cache_121_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.DECODE_SOURCES:
        (csrc / f).write_text(source_text + f)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "pa_decode_qwen3.md").write_text(
        "# summary\n\nkernel_source_sha: %s\ntraffic_bytes_per_launch: %d\n" % (sha_in_profile, traffic))


def test_traffic_is_reported_only_for_the_profiled_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _fake_tree(tmp_path, "kernel v1 ", "0" * 16)
    sha = bench.decode_source_sha()
    assert len(sha) == 16
    # a stale hash: no traffic
    assert bench.profiled_traffic("qwen3") is None
    # the hash of the current sources: the stored traffic
    text = (tmp_path / "profiles" / "pa_decode_qwen3.md").read_text().replace("0" * 16, sha)
    (tmp_path / "profiles" / "pa_decode_qwen3.md").write_text(text)
    assert bench.profiled_traffic("qwen3") == 123456
    # any edit of a source invalidates it again
    f = tmp_path / "paged_kv_cache_121_gb300" / "csrc" / bench.DECODE_SOURCES[0]
    f.write_text(f.read_text() + "\n")
    assert bench.profiled_traffic("qwen3") is None
    # no profile for a workload: no traffic
    assert bench.profiled_traffic("long") is None


def test_committed_profiles_name_a_hash_and_a_traffic():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for name in ("pa_decode_qwen3.md", "pa_decode_gqa.md"):
        text = open(os.path.join(root, "profiles", name)).read()
        assert "kernel_source_sha:" in text and "traffic_bytes_per_launch:" in text


def test_every_ncu_command_in_the_profiles_leaves_the_clocks_alone():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pdir = os.path.join(root, "profiles")
    commands = 0
    for name in sorted(os.listdir(pdir)):
        for line in open(os.path.join(pdir, name)):
            if "ncu --" in line:
                commands += 1
                assert "--clock-control none" in line, (name, line)
    assert commands >= 4


@pytest.mark.parametrize("bs", [1, 4, 16, 128])
def test_qwen3_pool_holds_the_batch_at_every_block_size(bs):
    # the sweep keeps the pool at 613,568 tokens; 16 sequences of 4,164 tokens must fit, twice over
    need = 2 * 16 * workloads.cdiv(4164, bs)
    assert workloads.QWEN3_POOL_BLOCKS * 16 // bs >= need
