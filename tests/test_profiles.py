"""The ncu summaries under profiles/: each gives the command that made it,
running committed files only, and names kernels that exist in the sources."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "bwd_maxpool3d_fwd_gb300", "csrc")


def _sources():
    return "".join(open(os.path.join(CSRC, f)).read() for f in os.listdir(CSRC))


def test_every_summary_has_a_committed_command():
    for name in sorted(os.listdir(PROFILES)):
        text = open(os.path.join(PROFILES, name)).read()
        assert "ncu " in text, f"{name}: no ncu command"
        assert "--clock-control none" in text, f"{name}: ncu without --clock-control none"
        assert "_work" not in text, f"{name}: command runs a scratch file"
        for script in re.findall(r"python ([\w./]+\.py)", text):
            assert os.path.exists(os.path.join(ROOT, script)), f"{name}: {script} is not in the tree"


def test_summaries_name_existing_kernels():
    src = _sources()
    for name in sorted(os.listdir(PROFILES)):
        text = open(os.path.join(PROFILES, name)).read()
        for kernel in set(re.findall(r"\b(k_[a-z0-9_]+)<", text)):
            assert re.search(rf"\b{kernel}\(", src), f"{name}: {kernel} not in the sources"


def _ncu_commands(text):
    """Every ncu command line in a summary, with continuation lines joined
    (commands in a .txt record sit behind '#')."""
    lines = [ln.lstrip("#").strip() for ln in text.splitlines()]
    joined, cur = [], ""
    for ln in lines:
        if ln.endswith("\\"):
            cur += ln[:-1] + " "
            continue
        joined.append(cur + ln)
        cur = ""
    return [c for c in joined if c.startswith("ncu ")]


def test_captures_are_small_and_single_kernel():
    # a capture that collects more than the launch duration names one kernel
    # (no alternation), one to three launches, and a small case: a subset of
    # planes, or one of the workloads of a few hundred MB
    small_workloads = {"0", "1", "2", "4"}
    for name in sorted(os.listdir(PROFILES)):
        for cmd in _ncu_commands(open(os.path.join(PROFILES, name)).read()):
            metrics = re.search(r"--metrics (\S+)", cmd)
            if metrics and metrics.group(1) == "gpu__time_duration.sum" and "--set" not in cmd:
                continue
            k = re.search(r"-k regex:(\S+)", cmd)
            assert k and "|" not in k.group(1), f"{name}: capture without a single kernel: {cmd}"
            c = re.search(r"-c (\d+)", cmd)
            assert c and 1 <= int(c.group(1)) <= 3, f"{name}: capture of more than three launches: {cmd}"
            w = re.search(r"--workload (\S+)", cmd)
            assert "--planes" in cmd or (w and w.group(1) in small_workloads), (
                f"{name}: capture on a full-size large workload: {cmd}")
