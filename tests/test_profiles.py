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
