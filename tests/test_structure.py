"""Where the oracle may be used, checked on the source: the oracle imports nothing
of the library (and the library nothing of the oracle), the seeded input module
holds no attention arithmetic and imports neither, and outside tests/ only the
benchmark's CPU legs and the smoke check import the oracle, each inside its own
function.  The C sources never reach the oracle either."""
import ast
import glob
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _imports(path):
    """(module name, enclosing top-level function or None) for every import."""
    tree = ast.parse(open(path).read(), filename=path)
    found = []

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            f = func
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) and func is None:
                f = child.name
            if isinstance(child, ast.Import):
                found.extend((a.name, f) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                # a relative import stays inside its own package
                found.append(("." + (child.module or "") if child.level else child.module, f))
            visit(child, f)

    visit(tree, None)
    return found


def _top(name):
    return name.split(".")[0]


def test_oracle_imports_nothing_of_the_library():
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        mods = {_top(m) for m, _ in _imports(path)}
        assert "context_ra_forward_gb300" not in mods, path
        assert mods <= {"__future__", "numpy", "math", ""}, (path, mods)


def test_library_imports_nothing_of_the_oracle():
    for path in glob.glob(os.path.join(ROOT, "context_ra_forward_gb300", "*.py")):
        mods = {_top(m) for m, _ in _imports(path)}
        assert "oracle" not in mods, path
    for path in glob.glob(os.path.join(ROOT, "context_ra_forward_gb300", "csrc", "*")) + \
            glob.glob(os.path.join(ROOT, "include", "*")):
        assert "oracle" not in open(path, errors="replace").read(), path


def test_input_module_is_arithmetic_free():
    path = os.path.join(ROOT, "context_ra_forward_gb300", "inputs.py")
    mods = {_top(m) for m, _ in _imports(path)}
    assert mods <= {"__future__", "dataclasses", "torch", "math", "numpy"}, mods
    text = open(path).read()
    for word in ("softmax", "exp(", "logsumexp", "matmul", "einsum", " @ "):
        assert word not in text, word


def test_oracle_users_outside_tests():
    allowed = {"bench.py": {"oracle_sample", "run_reference"}, "__graft_entry__.py": {"smoke"}}
    for path in glob.glob(os.path.join(ROOT, "*.py")):
        name = os.path.basename(path)
        users = {f for m, f in _imports(path) if _top(m) == "oracle"}
        assert users <= allowed.get(name, set()), (name, users)
        assert None not in users, name  # never at module level
