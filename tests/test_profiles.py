"""The committed ncu summaries: each names the command that made it, an ncu
run with --clock-control none over committed files only (bench.py), and is a
short text file."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_every_profile_gives_its_ncu_command():
    files = sorted(glob.glob(os.path.join(ROOT, "profiles", "*")))
    assert files
    for f in files:
        assert f.endswith((".md", ".txt")), f
        assert os.path.getsize(f) < 16 * 1024, f
        text = open(f).read()
        cmds = re.findall(r"^ncu [^\n]*(?:\n    [^\n]*)*", text, flags=re.M)
        assert cmds, f
        for c in cmds:
            assert "--clock-control none" in c, (f, c)
            assert "python bench.py" in c, (f, c)
