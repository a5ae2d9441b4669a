"""The committed ncu summaries are well-formed evidence: each names the full
command that produced it (ncu with --clock-control none, committed files
only), and the kernel summaries carry the source digest and DRAM bytes the
benchmark's traffic figures are read from."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def test_every_kernel_summary_has_command_digest_and_traffic():
    files = sorted(glob.glob(os.path.join(PROFILES, "*.txt")))
    assert len(files) >= 10
    for path in files:
        text = open(path).read()
        cmd = re.search(r"^command: (.+)$", text, flags=re.M)
        assert cmd, path
        assert cmd.group(1).startswith("ncu ") and "--clock-control none" in cmd.group(1), path
        assert "_work" not in cmd.group(1) and "gpurun" not in cmd.group(1), path
        assert re.search(r"^source_sha256_16: [0-9a-f]{16}$", text, flags=re.M), path
        dram = re.search(r"^dram_bytes_per_launch: (\d+)$", text, flags=re.M)
        assert dram and int(dram.group(1)) > 0, path
        assert re.search(r"^gpu__time_duration.sum: [0-9.]+ (us|ms|ns)", text, flags=re.M), path


def test_every_launch_list_names_its_command():
    files = sorted(glob.glob(os.path.join(PROFILES, "launches_*.md")))
    assert len(files) == 4
    for path in files:
        text = open(path).read()
        assert "ncu --metrics gpu__time_duration.sum --clock-control none" in text, path
        assert "| kernel | launches |" in text and "_work" not in text, path


def test_profiles_hold_text_only():
    for path in glob.glob(os.path.join(PROFILES, "*")):
        assert path.endswith((".txt", ".md")), path
        assert os.path.getsize(path) < 16 * 1024, path
