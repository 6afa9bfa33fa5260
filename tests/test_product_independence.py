"""The product path (the package and its C ABI) does not use the oracle: no
source file of the package imports or includes it, and importing the package
and loading the library leaves the oracle modules unimported."""
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "structured_state_space_gb300")


USE = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#\s*include\s*[<\"][^>\"]*oracle)|__import__\(\s*['\"]oracle"
                 r"|importlib\.import_module\(\s*['\"]oracle", re.M)


def test_package_sources_do_not_use_the_oracle():
    hits = []
    files = [os.path.join(ROOT, "include", "s4.h")]
    for d, _, names in os.walk(PKG):
        if "_build" in d or "__pycache__" in d:
            continue
        files += [os.path.join(d, f) for f in names if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp"))]
    for path in files:
        with open(path, encoding="utf-8") as fh:
            if USE.search(fh.read()):
                hits.append(os.path.relpath(path, ROOT))
    assert not hits, hits


def test_import_and_load_do_not_import_the_oracle():
    code = ("import sys; import structured_state_space_gb300 as s4; s4.load(); "
            "from structured_state_space_gb300 import workloads, multi; "
            "print(sorted(m for m in sys.modules if m.split('.')[0] == 'oracle'))")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == "[]", r.stdout


def test_missing_library_fails_loudly():
    # no fallback: without the built library every entry point is unavailable
    code = ("import structured_state_space_gb300 as s4\n"
            "try:\n    s4.load('/nonexistent/libs4.so')\nexcept RuntimeError as e:\n    print('raised', 'not built' in str(e))\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == "raised True", r.stdout
