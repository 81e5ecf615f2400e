"""The oracle and the CUDA path stay apart (static checks, no GPU).

The package never imports the oracle and the oracle never imports the
package; the only module both sides use is the seeded input generator,
which holds no attention arithmetic. In bench.py the oracle runs only in the
CPU-baseline legs (each guarded by --no-cpu-baseline) and in the reference
arm.
"""

import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "io_aware_exact_tiled_gb300")
ORACLE = os.path.join(ROOT, "oracle")

# bench.py functions that time the oracle: the contract line's CPU baseline,
# the reference arm and the table's CPU baseline
BENCH_ORACLE_FUNCTIONS = {"oracle_sample", "oracle_rows", "table_cpu_baseline"}


def imports(tree):
    """(module name, node) of every import in a syntax tree."""
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name, node
        elif isinstance(node, ast.ImportFrom):
            yield ("." * node.level) + (node.module or ""), node


def py_files(folder):
    for dirpath, _, files in os.walk(folder):
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(dirpath, f)


def parse(path):
    with open(path, encoding="utf-8") as fh:
        return ast.parse(fh.read(), path)


def test_package_never_imports_the_oracle():
    for path in py_files(PKG):
        for name, _ in imports(parse(path)):
            assert name.split(".")[0] != "oracle", (path, name)


def test_oracle_imports_only_numpy_and_itself():
    for path in py_files(ORACLE):
        for name, _ in imports(parse(path)):
            assert name.startswith(".") or name.split(".")[0] in ("__future__", "numpy"), (path, name)


def test_cuda_sources_name_no_oracle_file():
    csrc = os.path.join(PKG, "csrc")
    for f in os.listdir(csrc):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            for line in fh:
                if line.lstrip().startswith("#include"):
                    assert "oracle" not in line, (f, line)


def _bench_tree():
    tree = parse(os.path.join(ROOT, "bench.py"))
    parents = {}
    for node in ast.walk(tree):
        for child in ast.iter_child_nodes(node):
            parents[child] = node
    return tree, parents


def _context(node, parents):
    """(enclosing function names, innermost first; whether an enclosing `if`
    tests --no-cpu-baseline)."""
    chain, n = [], node
    while n in parents:
        n = parents[n]
        chain.append(n)
    funcs = [c.name for c in chain if isinstance(c, ast.FunctionDef)]
    guarded = any(isinstance(c, ast.If) and "no_cpu_baseline" in ast.unparse(c.test) for c in chain)
    return funcs, guarded


def test_bench_runs_the_oracle_only_in_its_baseline_legs():
    tree, parents = _bench_tree()
    found = 0
    for name, node in imports(tree):
        if name.split(".")[0] != "oracle":
            continue
        found += 1
        funcs, guarded = _context(node, parents)
        assert funcs, f"module-level oracle import at line {node.lineno}"
        assert guarded or funcs[-1] in BENCH_ORACLE_FUNCTIONS, \
            f"oracle imported outside a CPU-baseline leg at line {node.lineno} (in {funcs})"
    assert found > 0
    # and the functions that time it are called only from guarded legs or the reference arm
    calls = 0
    for node in ast.walk(tree):
        if isinstance(node, ast.Call) and isinstance(node.func, ast.Name) and node.func.id in BENCH_ORACLE_FUNCTIONS:
            calls += 1
            funcs, guarded = _context(node, parents)
            assert guarded or funcs[-1] == "run_reference", (node.func.id, node.lineno, funcs)
    assert calls >= 3
