"""Host-side logic of bench.py (no GPU): the DRAM-traffic figure of the
roofline object comes from the committed ncu summary only while the GEMV
kernel sources are the ones it was taken on."""
import os

import pytest

import bench

# packed codes + scales + zeros + x + y of one 15360 x 3840 (or 3840 x 15360)
# INT4 group-128 GEMV launch
ALGORITHMIC_BYTES = 15360 * 3840 // 2 + 2 * 2 * 15360 * 30 + 2 * 3840 + 2 * 15360


def test_read_traffic_follows_the_digest(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "gemv_int4_decode_mlp_pair.md").write_text(
        "# summary\n\n- kernel_sources_sha256_16: `abcdef0123456789`\n- dram_bytes_per_launch: `31404800`\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_traffic("abcdef0123456789") == 31404800.0
    assert bench.read_traffic("0000000000000000") is None   # other kernel sources: no figure
    os.remove(prof / "gemv_int4_decode_mlp_pair.md")
    assert bench.read_traffic("abcdef0123456789") is None   # no summary at all


def test_committed_traffic_is_close_to_the_algorithmic_bytes():
    assert ALGORITHMIC_BYTES == 31372800
    v = bench.read_traffic(bench.kernel_sources_digest())
    if v is None:
        pytest.skip("the committed ncu summary was taken on other GEMV kernel sources")
    # every weight byte read once from DRAM; the output stays in L2
    assert abs(v - ALGORITHMIC_BYTES) / ALGORITHMIC_BYTES < 0.01
