"""The product path stands alone: the package never reaches the oracle, and without its
compiled library it refuses to run instead of computing anything another way.  No GPU."""
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
PKG = os.path.join(ROOT, "weight_only_bit_int4_gb300")


def _sources():
    for dirpath, dirnames, filenames in os.walk(PKG):
        dirnames[:] = [d for d in dirnames if d not in ("_build", "__pycache__")]
        for f in filenames:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp", ".c")):
                yield os.path.join(dirpath, f)


def test_package_never_loads_the_oracle():
    pattern = re.compile(r"^\s*(import\s+oracle\b|from\s+oracle\b)|liboracle|q4_oracle\.c|#include\s+\"[^\"]*oracle",
                         re.M)
    hits = [p for p in _sources() if pattern.search(open(p).read())]
    assert hits == [], hits


def test_binding_raises_without_the_library(tmp_path):
    # a copy of the package's Python files only: no libq4mm.so beside them
    dst = tmp_path / "weight_only_bit_int4_gb300"
    dst.mkdir()
    for f in os.listdir(PKG):
        if f.endswith(".py"):
            shutil.copy(os.path.join(PKG, f), dst / f)
    code = ("import weight_only_bit_int4_gb300 as q\n"
            "try:\n"
            "    q.lib()\n"
            "except RuntimeError as e:\n"
            "    print('raised:', e)\n"
            "else:\n"
            "    print('loaded')\n")
    env = dict(os.environ, PYTHONPATH=str(tmp_path))
    r = subprocess.run([sys.executable, "-c", code], cwd=str(tmp_path), env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "raised:" in r.stdout and "libq4mm.so not found" in r.stdout, r.stdout
