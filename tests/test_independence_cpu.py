"""The CUDA path and the oracle share nothing, checked statically on the CPU.

The library's binding and build script never import the oracle. The seeded
input generators (`kvc_synth`, the one module both sides use) import neither
side. The oracle imports neither the binding nor the generators. The CUDA
sources and the C header never mention it. The scripts that may run it
(`bench.py`'s CPU legs, `__graft_entry__.smoke()`) import it only inside
those functions.
"""

import ast
import glob
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "sliding_window_attention_kvc_gb300"


def _imports(path):
    """(top-level module name, enclosing function name or None) per import."""
    with open(path) as f:
        tree = ast.parse(f.read(), path)
    found = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            inner = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            if isinstance(child, ast.Import):
                found.extend((a.name.split(".")[0], fn) for a in child.names)
            elif isinstance(child, ast.ImportFrom) and child.level == 0 and child.module:
                found.append((child.module.split(".")[0], fn))
            visit(child, inner)

    visit(tree, None)
    return found


def _py(*parts):
    return sorted(glob.glob(os.path.join(ROOT, *parts, "*.py")))


def test_binding_and_generators_never_import_the_oracle():
    for path in _py(PKG) + _py("kvc_synth"):
        mods = {m for m, _ in _imports(path)}
        assert "oracle" not in mods, path
        if "kvc_synth" in path:
            assert PKG not in mods and "bench" not in mods, path


def test_oracle_imports_neither_the_binding_nor_the_generators():
    files = _py("oracle")
    assert len(files) >= 8
    for path in files:
        mods = {m for m, _ in _imports(path)}
        assert not mods & {PKG, "kvc_synth", "bench", "tests", "torch", "ctypes"}, (path, mods)


def test_cuda_sources_and_header_never_mention_the_oracle():
    files = glob.glob(os.path.join(ROOT, PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*"))
    assert len(files) >= 10
    for path in files:
        with open(path) as f:
            assert "oracle" not in f.read().lower(), path


def test_scripts_import_the_oracle_only_in_their_cpu_legs():
    allowed = {"bench.py": {"oracle_sample"}, "__graft_entry__.py": {"smoke"}}
    for name, fns in allowed.items():
        uses = [fn for m, fn in _imports(os.path.join(ROOT, name)) if m in ("oracle", "tests")]
        assert uses, name
        assert set(uses) <= fns, (name, uses)


def test_generators_hold_none_of_the_methods_arithmetic():
    """kvc_synth draws seeded values and positions only: no rotation,
    exponential, square root, quantisation or contraction appears in it."""
    import re
    banned = re.compile(r"\b(exp2?|cos|sin|sqrt|softmax|rint|clip|clamp|einsum|matmul|rotate|quantize\w*)\s*\("
                        r"|\b127\b|[\w\)\]]\s*@\s*[\w\(]")
    for path in _py("kvc_synth"):
        with open(path) as f:
            for n, line in enumerate(f, 1):
                code = line.split("#", 1)[0]
                if code.strip().startswith(("\"", "'")) or not code.strip():
                    continue
                assert not banned.search(code), f"{os.path.basename(path)}:{n}: {line.strip()}"
