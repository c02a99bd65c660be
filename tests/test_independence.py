"""The oracle and the CUDA path stay independent (static checks, CPU only).

- No module of the package (the binding, the orchestrator, the input
  generators, the build script) imports the oracle, and no CUDA source or
  header includes anything from it.
- The oracle imports neither the package nor the benchmark.
- The benchmark imports the oracle only inside the function that times it
  (the CPU-baseline leg and the reference arm), and `__graft_entry__` only
  inside smoke(); build() never touches it.
- The seeded input generators hold none of the method's arithmetic (no
  top-k, counting, softmax or matrix products)."""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "moe_expert_routing_02_b300")


def _imports(path):
    """(module name, enclosing function or None) for every import in a file."""
    tree = ast.parse(open(path).read(), path)
    out = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)):
                visit(child, child.name)
            elif isinstance(child, ast.Import):
                out.extend((a.name, fn) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                if child.level:   # relative import inside a package
                    out.append(("." * child.level + (child.module or ""), fn))
                else:
                    out.append((child.module or "", fn))
            else:
                visit(child, fn)
    visit(tree, None)
    return out


def _top(name):
    return name.split(".")[0]


def test_package_never_imports_the_oracle():
    for path in glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True):
        for mod, _ in _imports(path):
            assert _top(mod) != "oracle", (path, mod)
    for path in glob.glob(os.path.join(PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*")):
        for inc in re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', open(path).read()):
            assert "oracle" not in inc, (path, inc)


def test_oracle_imports_neither_the_package_nor_the_bench():
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        for mod, _ in _imports(path):
            assert _top(mod) not in ("moe_expert_routing_02_b300", "bench", "__graft_entry__", "tests"), (path, mod)


def test_bench_and_entry_touch_the_oracle_only_where_allowed():
    bench = [fn for mod, fn in _imports(os.path.join(ROOT, "bench.py")) if _top(mod) == "oracle"]
    assert bench and set(bench) == {"oracle_layer_sample"}
    # that function is reached only from the CPU-baseline leg and the reference arm
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    callers = set()
    for fn in [n for n in ast.walk(tree) if isinstance(n, ast.FunctionDef)]:
        for node in ast.walk(fn):
            if isinstance(node, ast.Call) and getattr(node.func, "id", None) == "oracle_layer_sample":
                callers.add(fn.name)
    assert callers <= {"run_cpu_baseline", "run_reference"}, callers
    entry = [fn for mod, fn in _imports(os.path.join(ROOT, "__graft_entry__.py")) if _top(mod) == "oracle"]
    assert entry and set(entry) == {"smoke"}


def test_input_generators_hold_none_of_the_method():
    src = open(os.path.join(PKG, "workloads.py")).read()
    code = "\n".join(line.split("#")[0] for line in src.splitlines())
    code = re.sub(r'"""[\s\S]*?"""', "", code)          # docstrings may name the stages
    for word in ("argsort", "argpartition", "topk", "bincount", "softmax", "matmul", "einsum", "lexsort", " @ "):
        assert word not in code, word
