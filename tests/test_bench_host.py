"""Host-side checks of bench.py that need no GPU: every function or class
it calls by bare name resolves in the module (a missing helper would
otherwise show only where a GPU runs the bench), and the algorithmic-byte
model of the headline workload matches its definition."""
import ast
import builtins
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_every_called_name_resolves():
    import bench

    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    local = set()
    for node in ast.walk(tree):
        if isinstance(node, (ast.FunctionDef, ast.Lambda)):
            if isinstance(node, ast.FunctionDef):
                local.add(node.name)
            a = node.args
            local |= {x.arg for x in a.args + a.kwonlyargs + a.posonlyargs}
        elif isinstance(node, ast.Name) and isinstance(node.ctx, ast.Store):
            local.add(node.id)
    missing = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Call) and isinstance(node.func, ast.Name):
            n = node.func.id
            if not (hasattr(bench, n) or hasattr(builtins, n) or n in local):
                missing.add(n)
    assert not missing, sorted(missing)


def test_headline_algorithmic_bytes():
    import bench

    # logits read once + packed mask + one int64 token per row
    assert bench.algorithmic_bytes(256, 128256, 4, mask=True) == \
        256 * 128256 * 4 + 256 * 4008 * 4 + 256 * 8
    assert bench.algorithmic_bytes(256, 128256, 4, mask=False) == 256 * 128256 * 4 + 256 * 8
