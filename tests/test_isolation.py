"""The product path and the oracle share nothing, and the product never
falls back to anything when its CUDA library is missing (no GPU needed)."""
import os
import subprocess
import sys

from conftest import ROOT

PRODUCT = [os.path.join(ROOT, "movement_primitives_gb300"), os.path.join(ROOT, "include")]
ORACLE = os.path.join(ROOT, "oracle")


def _sources(roots):
    for root in roots:
        for dirpath, _dirs, files in os.walk(root):
            if "_build" in dirpath or "__pycache__" in dirpath:
                continue
            for f in files:
                if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp", ".c")):
                    yield os.path.join(dirpath, f)


def _links(path, names):
    """Import or include lines of `path` that reach any of `names`."""
    out = []
    for line in open(path):
        t = line.strip()
        if t.startswith(("import ", "from ", "#include")) and any(n in t for n in names):
            out.append(t)
    return out


def test_sources_do_not_import_or_include_each_other():
    for path in _sources(PRODUCT):
        assert not _links(path, ["oracle", "copy_oracle"]), path
        assert "oracle" not in open(path).read(), path  # not even named in the product
    for path in _sources([ORACLE]):
        assert not _links(path, ["movement_primitives_gb300", "layout_copy", "lc_internal", "liblayoutcopy"]), path


def test_importing_the_product_loads_no_oracle_module():
    code = ("import sys, movement_primitives_gb300 as M; "
            "bad = [m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')]; "
            "assert not bad, bad")
    subprocess.run([sys.executable, "-c", code], cwd=ROOT, check=True)


def test_missing_library_fails_loudly():
    code = ("import movement_primitives_gb300 as M\n"
            "try:\n"
            "    M.plan(dict(shape=(4,), stride=(1,)), dict(shape=(4,), stride=(1,)), 4)\n"
            "except RuntimeError as e:\n"
            "    assert 'no fallback' in str(e), e\n"
            "else:\n"
            "    raise SystemExit('planned without the library')\n")
    env = dict(os.environ, LC_LIBRARY_PATH=os.path.join(ROOT, "no_such_dir", "liblayoutcopy.so"))
    subprocess.run([sys.executable, "-c", code], cwd=ROOT, check=True, env=env)
