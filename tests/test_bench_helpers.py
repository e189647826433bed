"""Host helpers of bench.py (no GPU): where roofline.traffic comes from, and
how many threads the CPU oracle gets.

The traffic figure is read from the ncu summary of the benchmark's workload,
and only when that summary was taken on the kernel source being built.  Any
plan or size override gives None, because the summaries are of the default
plan at full size.  Checked on a temporary tree, so that editing the kernel
does not fail this test before the profiles are taken again.
"""
import hashlib
import os
import pytest

import bench


def _tree(tmp_path, src=b"kernel v1", recorded=None, bytes_line=True):
    csrc = tmp_path / "shared_prefix_kv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "decode.cu").write_bytes(src)
    (tmp_path / "profiles").mkdir()
    sha = hashlib.sha256(recorded if recorded is not None else src).hexdigest()
    text = f"# summary\n\nsource_sha256: {sha}\n\n"
    if bytes_line:
        text += "dram_bytes_per_launch: 123456789\n"
    (tmp_path / "profiles" / "psattn_fused_decode_skewed.md").write_text(text)
    return tmp_path


def _rec(workload="skewed", groups=None, no_fold=False, chunk_form="ragged"):
    """bench._traffic_record as main() calls it for these arguments"""
    return bench._traffic_record(workload, groups is None and not no_fold
                                 and chunk_form == "ragged")


def test_traffic_from_matching_summary(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(_tree(tmp_path)))
    traffic, source = _rec()
    assert traffic == 123456789
    assert source.startswith(os.path.join("profiles", "psattn_fused_decode_skewed.md"))


@pytest.mark.parametrize("override", [dict(groups=8), dict(no_fold=True),
                                      dict(chunk_form="levels"), dict(workload="tiny_fp32")])
def test_traffic_none_for_overrides_or_missing_summary(tmp_path, monkeypatch, override):
    monkeypatch.setattr(bench, "ROOT", str(_tree(tmp_path)))
    traffic, source = _rec(**override)
    assert traffic is None and source.startswith("none")


def test_traffic_none_for_stale_or_incomplete_summary(tmp_path, monkeypatch):
    root = _tree(tmp_path, src=b"kernel v2", recorded=b"kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert _rec()[0] is None
    other = tmp_path / "other"
    other.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(_tree(other, bytes_line=False)))
    assert _rec()[0] is None


def test_oracle_threads():
    assert bench._oracle_threads(1) == 0  # a single process: the OpenMP default
    n = bench._oracle_threads(2)         # under torchrun: every core of this process
    assert n >= 1 and n <= (os.cpu_count() or n)
