"""Repository rules that a later change could break without noticing:
profile summaries give the command that made them and use committed files
only, and no committed code reaches into the untracked working directory."""
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _tracked():
    out = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True)
    if out.returncode != 0:  # not a git checkout: list the files on disk
        files = []
        for d, _, names in os.walk(ROOT):
            if "/." in d or "_work" in d or "gpurun_out" in d:
                continue
            files += [os.path.relpath(os.path.join(d, n), ROOT) for n in names]
        return files
    return out.stdout.split()


def test_profile_summaries_give_their_command():
    prof = os.path.join(ROOT, "profiles")
    for name in sorted(os.listdir(prof)):
        if not name.endswith(".md") or name == "README.md":
            continue
        text = open(os.path.join(prof, name)).read()
        assert re.search(r"(python[3]? (-m |-c |bench\.py)|ncu |nvcc )", text), name
        assert "_work/" not in text, name


def test_no_committed_code_uses_the_working_directory():
    offenders = []
    for rel in _tracked():
        if not rel.endswith((".py", ".cu", ".cuh", ".h", ".c", ".sh")):
            continue
        if rel == os.path.join("tests", "test_repo_rules.py"):
            continue
        with open(os.path.join(ROOT, rel), errors="replace") as f:
            if "_work/" in f.read():
                offenders.append(rel)
    assert not offenders, offenders
