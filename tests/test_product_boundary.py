"""The product path stands alone: the package neither imports nor reaches the
oracle, and without its CUDA library it fails at once instead of computing
anything on the CPU (CPU only)."""
import ast
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "decode_kv_cache_gb300")


def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module:
            names.add(node.module.split(".")[0])
    return names


def test_package_sources_do_not_import_the_oracle():
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            path = os.path.join(dirpath, f)
            if f.endswith(".py"):
                assert not ({"oracle", "tests", "synth"} & _imports(path)), path
            if f.endswith((".cu", ".cuh", ".h", ".py")):
                assert "oracle" not in open(path).read().lower(), path


def test_importing_the_binding_loads_no_oracle():
    code = ("import sys; from decode_kv_cache_gb300 import longflow; "
            "print(sorted(m for m in sys.modules if m.split('.')[0] in ('oracle', 'synth')))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         check=True).stdout.strip()
    assert out == "[]"


def test_missing_library_fails_loudly():
    code = ("from decode_kv_cache_gb300 import longflow as lf\n"
            "try:\n"
            "    lf.lf_abi_version()\n"
            "except RuntimeError as e:\n"
            "    print('raised:', e)\n")
    env = dict(os.environ, LONGFLOW_LIB=os.path.join(ROOT, "no-such-dir", "liblongflow.so"))
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         env=env, check=True).stdout
    assert out.startswith("raised:") and "not found" in out
