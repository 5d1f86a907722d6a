"""The committed profile summaries: short text files, each naming the command
that made it, every ncu command with the clocks left alone; and the hot
kernel's summary carries the traffic and source hash the benchmark reads."""
import os
import re

from conftest import ROOT

PROFILES = os.path.join(ROOT, "profiles")


def _summaries():
    return sorted(os.path.join(PROFILES, f) for f in os.listdir(PROFILES))


def test_profiles_are_short_text():
    files = _summaries()
    assert files
    for path in files:
        assert path.endswith((".md", ".txt")), path
        assert os.path.getsize(path) < 16 * 1024, path
        with open(path, encoding="utf-8") as f:
            f.read()  # text, not a report


def test_every_ncu_command_leaves_clocks_alone():
    for path in _summaries():
        text = open(path, encoding="utf-8").read()
        # a command may continue over lines ending in a backslash
        commands = re.findall(r"^\s*(ncu\s+--(?:[^\n]*\\\n)*[^\n]*)", text, flags=re.M)
        assert commands, f"{path} names no ncu command"
        for cmd in commands:
            assert "--clock-control none" in cmd, (path, cmd)


def test_hot_kernel_summary_fields():
    text = open(os.path.join(PROFILES, "eval_reg_1f1b_P8_M64_n65536.md"), encoding="utf-8").read()
    traffic = re.search(r"^- traffic_bytes_per_launch: (\d+)$", text, flags=re.M)
    sha = re.search(r"^- kernel_source_sha256: ([0-9a-f]{64})$", text, flags=re.M)
    assert traffic and sha
    # within a few percent of the algorithmic bytes of one launch
    assert abs(int(traffic.group(1)) / 273_743_904 - 1) < 0.05
