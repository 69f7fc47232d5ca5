"""The bench line's DRAM traffic comes from one ncu capture of the split-decode
kernel: the figure in bench.py and the committed capture summary must name
the same source hash and the same bytes, and the figure must disappear once
the kernel source no longer has that hash (CPU only)."""
import re
from pathlib import Path

import bench

ROOT = Path(__file__).resolve().parent.parent


def test_traffic_matches_the_capture_summary():
    summary = (ROOT / "profiles" / "decode_split_qwen3_b64.md").read_text()
    sha = re.search(r"sha256 prefix ([0-9a-f]{16})", summary).group(1)
    traffic = int(re.search(r"\| traffic_bytes_per_launch \| (\d+) \|", summary).group(1))
    assert bench.DECODE_TRAFFIC == {sha: traffic}


def test_traffic_is_dropped_for_a_changed_kernel(monkeypatch):
    real = Path.read_bytes

    def changed(self):
        data = real(self)
        return data + b"\n// changed\n" if self.name == "decode.cu" else data

    monkeypatch.setattr(Path, "read_bytes", changed)
    assert bench.decode_traffic() is None
