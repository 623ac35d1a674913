"""The measurement records under profiles/ are text summaries whose commands
run committed files only: every `python -m <module>` names a module of this
repository, every `python <script>.py` a committed script, and no record names
a scratch path or keeps a raw report."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*")))


def test_profiles_are_text_summaries():
    assert PROFILES
    for p in PROFILES:
        assert p.endswith((".md", ".txt")), f"{p}: profiles hold text summaries only"
        assert os.path.getsize(p) < 64 * 1024, f"{p}: a summary, not a raw report"


def test_profile_commands_run_committed_files():
    mod_re = re.compile(r"python3? -m ([A-Za-z_][\w.]*)")
    script_re = re.compile(r"python3? ([\w/]+\.py)")
    for p in PROFILES:
        text = open(p).read()
        assert "_work" not in text, f"{p} names a scratch path"
        for mod in mod_re.findall(text):
            if mod in ("pytest",):
                continue
            path = os.path.join(ROOT, *mod.split("."))
            assert os.path.exists(path + ".py") or os.path.isdir(path), f"{p}: module {mod} is not in the repository"
        for script in script_re.findall(text):
            assert os.path.exists(os.path.join(ROOT, script)), f"{p}: script {script} is not in the repository"
