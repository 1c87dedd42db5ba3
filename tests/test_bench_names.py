"""bench.py's GPU paths do not run in the CPU suite; a static check that every name a
function of bench.py reads is bound somewhere it can see (its own assignments and
parameters, enclosing functions, module globals or builtins) catches a misspelt or
missing variable in those paths before a GPU run does."""
import ast
import builtins
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bound_in(node):
    names = set()
    for x in ast.walk(node):
        if isinstance(x, ast.Name) and isinstance(x.ctx, (ast.Store, ast.Del)):
            names.add(x.id)
        elif isinstance(x, (ast.FunctionDef, ast.AsyncFunctionDef, ast.ClassDef)):
            names.add(x.name)
        if isinstance(x, (ast.FunctionDef, ast.AsyncFunctionDef, ast.Lambda)):
            a = x.args
            for arg in a.posonlyargs + a.args + a.kwonlyargs:
                names.add(arg.arg)
            if a.vararg:
                names.add(a.vararg.arg)
            if a.kwarg:
                names.add(a.kwarg.arg)
        elif isinstance(x, (ast.Import, ast.ImportFrom)):
            for al in x.names:
                names.add((al.asname or al.name).split(".")[0])
        elif isinstance(x, ast.ExceptHandler) and x.name:
            names.add(x.name)
        elif isinstance(x, (ast.Global, ast.Nonlocal)):
            names.update(x.names)
    return names


def test_bench_functions_read_only_bound_names():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    module = set(dir(builtins)) | {"__file__", "__name__"}
    for n in tree.body:
        if isinstance(n, (ast.FunctionDef, ast.ClassDef)):
            module.add(n.name)
        elif isinstance(n, (ast.Import, ast.ImportFrom)):
            for al in n.names:
                module.add((al.asname or al.name).split(".")[0])
        elif isinstance(n, (ast.Assign, ast.AnnAssign, ast.AugAssign)):
            targets = n.targets if isinstance(n, ast.Assign) else [n.target]
            for t in targets:
                for x in ast.walk(t):
                    if isinstance(x, ast.Name):
                        module.add(x.id)
        elif isinstance(n, (ast.If, ast.Try, ast.With)):
            module |= _bound_in(n)
    unbound = []
    # each top-level function with everything nested in it (a closure reads its enclosing
    # function's names)
    for n in tree.body:
        if not isinstance(n, (ast.FunctionDef, ast.AsyncFunctionDef)):
            continue
        seen = _bound_in(n) | module
        for x in ast.walk(n):
            if isinstance(x, ast.Name) and isinstance(x.ctx, ast.Load) and x.id not in seen:
                unbound.append((n.name, x.id, x.lineno))
    assert not unbound, unbound
