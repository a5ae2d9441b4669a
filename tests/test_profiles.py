"""The committed ncu summaries are well-formed evidence: each names the full
command that produced it (ncu with --clock-control none, committed files
only), and the kernel summaries carry the source digest and DRAM bytes the
benchmark's traffic figures are read from."""
import glob
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _tracked_files():
    """Files under version control, or None where there is no git metadata."""
    try:
        out = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True, timeout=60)
    except (OSError, subprocess.SubprocessError):
        return None
    return set(out.stdout.split()) if out.returncode == 0 else None


def _assert_runs_committed_files_only(cmd: str, path: str):
    """A profile command names no absolute path and no wrapper: every script
    it runs is a file of the repository (tracked, where git metadata exists)."""
    tracked = _tracked_files()
    for tok in cmd.split():
        assert not tok.startswith(("/", "~")), (path, tok)
        if tok.endswith(".py"):
            assert os.path.isfile(os.path.join(ROOT, tok)), (path, tok)
            if tracked is not None:
                assert tok in tracked, (path, tok)


def test_every_kernel_summary_has_command_digest_and_traffic():
    files = sorted(glob.glob(os.path.join(PROFILES, "*.txt")))
    assert len(files) >= 10
    for path in files:
        text = open(path).read()
        cmd = re.search(r"^command: (.+)$", text, flags=re.M)
        assert cmd, path
        assert cmd.group(1).startswith("ncu ") and "--clock-control none" in cmd.group(1), path
        _assert_runs_committed_files_only(cmd.group(1), path)
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
        assert "| kernel | launches |" in text, path
        cmd = re.search(r"^\s*`?(ncu --metrics[^`\n]+)`?$", text, flags=re.M)
        assert cmd, path
        _assert_runs_committed_files_only(cmd.group(1), path)


def test_profiles_hold_text_only():
    for path in glob.glob(os.path.join(PROFILES, "*")):
        assert path.endswith((".txt", ".md")), path
        assert os.path.getsize(path) < 16 * 1024, path
