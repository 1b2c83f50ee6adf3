"""The product path and the oracle share no code (static check, CPU only).

The package linear_attention_chunked_gb300 (binding, build, input generators) must never import
the oracle, and the oracle must never import the package; the CUDA sources never name the
oracle's C file.  Only tests/, __graft_entry__.smoke() and bench.py's CPU legs load the oracle."""
import ast
import glob
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "linear_attention_chunked_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    out = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            out.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            out.add(node.module.split(".")[0])
    return out


def test_package_never_imports_the_oracle():
    files = glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True)
    assert files
    for f in files:
        assert "oracle" not in _imports(f), f
        assert "harness" not in _imports(f), f


def test_oracle_never_imports_the_package():
    for f in glob.glob(os.path.join(ORACLE, "*.py")):
        assert "linear_attention_chunked_gb300" not in _imports(f), f
    src = open(os.path.join(ORACLE, "kda_oracle.c")).read()
    assert "kda_internal" not in src and "kda_tc" not in src and "kda_mma" not in src


def test_cuda_sources_never_name_the_oracle():
    for f in glob.glob(os.path.join(PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*")):
        assert "kda_oracle" not in open(f).read(), f
