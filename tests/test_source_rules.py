"""Committed code stands on its own: no source file, comment or docstring
points at the build's planning documents, its tooling or this machine's
paths, and the oracle is reached only from the test infrastructure (tests/,
the smoke entry point and the benchmark's CPU legs), never from the product
package."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CODE = re.compile(r"\.(py|cu|cuh|h|c|sh)$")


def committed_code():
    try:
        out = subprocess.run(["git", "-C", ROOT, "ls-files"], capture_output=True, text=True, check=True).stdout
    except (OSError, subprocess.CalledProcessError):
        pytest.skip("not a git checkout")
    return [f for f in out.splitlines() if CODE.search(f) and os.path.exists(os.path.join(ROOT, f))]


# words that name the build's own documents, tooling or machine, assembled so
# that this file does not name them itself
FORBIDDEN = [re.compile(p) for p in (
    r"PAPER" + r"\.md", r"BASELINE" + r"\.(json|md)", r"north" + r"_star", r"\b" + "SUR" + r"VEY\b",
    r"DESIGN" + r"\.md", r"\b" + "VER" + r"DICT\b", r"\b" + "ADV" + r"ICE\b", r"(?i)gpu" + r"run\b",
    r"config" + r"s\[\d\]", "/" + "root/",
)]


def test_no_source_names_the_build_documents_or_machine():
    bad = []
    for f in committed_code():
        text = open(os.path.join(ROOT, f), encoding="utf-8", errors="replace").read()
        for pat in FORBIDDEN:
            for m in pat.finditer(text):
                line = text.count("\n", 0, m.start()) + 1
                bad.append(f"{f}:{line}: {m.group(0)}")
    assert not bad, "\n".join(bad)


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "numerically_stable_online_gb300")
    imp = re.compile(r"^\s*(from\s+oracle\b|import\s+oracle\b)|oracle/|liboracle", re.M)
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for name in files:
            if CODE.search(name):
                text = open(os.path.join(dirpath, name), encoding="utf-8").read()
                assert not imp.search(text), os.path.join(dirpath, name)


def test_oracle_imports_nothing_of_the_product():
    odir = os.path.join(ROOT, "oracle")
    for name in os.listdir(odir):
        if CODE.search(name):
            text = open(os.path.join(odir, name), encoding="utf-8").read()
            assert "import numerically_stable_online_gb300" not in text
            assert "from numerically_stable_online_gb300" not in text
            assert "smx.h" not in text and "csrc" not in text, name
