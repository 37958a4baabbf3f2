"""The product path never reaches the CPU oracle and has no CPU fallback.

* No source of the package (Python, CUDA, headers) imports or names the
  oracle module; importing the package loads no oracle module.
* bench.py uses the oracle only in its timing of the oracle itself (the CPU
  baseline and the reference arm) and in the parity statistics taken from
  that timed oracle pass, never in the GPU arm's timed work.
* With the CUDA library missing, loading it and every call raise.
"""
import ast
import glob
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fp8_compression_tensor_gb300")


def test_package_sources_do_not_use_the_oracle():
    files = glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True)
    files += glob.glob(os.path.join(PKG, "csrc", "*"))
    files += glob.glob(os.path.join(ROOT, "include", "*.h"))
    assert files
    for f in files:
        text = open(f, encoding="utf-8", errors="replace").read()
        assert "oracle" not in text, f
        assert "taco_oracle" not in text, f


def test_importing_the_package_loads_no_oracle():
    code = ("import sys; sys.path.insert(0, %r); import fp8_compression_tensor_gb300 as t; "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "False"


def test_bench_uses_the_oracle_only_to_time_it():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    owners = []
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, (ast.Import, ast.ImportFrom)):
                    names = [a.name for a in node.names] if isinstance(node, ast.Import) else [node.module or ""]
                    if any(n == "oracle" or n.startswith("oracle.") for n in names):
                        owners.append(fn.name)
    top = [n for n in tree.body if isinstance(n, (ast.Import, ast.ImportFrom))]
    for node in top:
        names = [a.name for a in node.names] if isinstance(node, ast.Import) else [node.module or ""]
        assert not any(n == "oracle" or n.startswith("oracle.") for n in names), "module-level oracle import"
    assert sorted(owners) == ["oracle_build_info", "oracle_op_times"], owners
    # parity_against_oracle reads the tests' parity helpers (which load the
    # oracle): it counts as oracle use too.
    timing = {"oracle_op_times", "sample_rows_for", "oracle_build_info", "parity_against_oracle"}
    callers = {fn.name for fn in ast.walk(tree) if isinstance(fn, ast.FunctionDef)
               for node in ast.walk(fn) if isinstance(node, ast.Call)
               and getattr(node.func, "id", None) in timing}
    assert callers <= {"sample_rows_for", "run_reference", "run_taco"}, callers
    # In the GPU arm, only the cpu_baseline block (skipped by --no-cpu-baseline) times the oracle.
    run_taco = next(fn for fn in ast.walk(tree) if isinstance(fn, ast.FunctionDef) and fn.name == "run_taco")
    parents = {}
    for node in ast.walk(run_taco):
        for child in ast.iter_child_nodes(node):
            parents[child] = node
    calls = [node for node in ast.walk(run_taco) if isinstance(node, ast.Call)
             and getattr(node.func, "id", None) in timing]
    assert calls
    for call in calls:
        node, guarded = call, False
        while node in parents:
            node = parents[node]
            if isinstance(node, ast.If) and "no_cpu_baseline" in ast.unparse(node.test):
                guarded = True
        assert guarded, ast.unparse(call)


def test_missing_library_raises():
    code = ("import sys; sys.path.insert(0, %r)\n"
            "import fp8_compression_tensor_gb300 as t\n"
            "for f in (lambda: t.load_library(), lambda: t.compressed_bytes(4, 128, 128)):\n"
            "    try:\n"
            "        f()\n"
            "    except RuntimeError as e:\n"
            "        assert 'missing' in str(e)\n"
            "    else:\n"
            "        raise SystemExit('no error')\n"
            "print('raised')\n" % ROOT)
    env = dict(os.environ, TACO_GB300_LIBRARY=os.path.join(ROOT, "no_such_dir", "libtaco_gb300.so"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "raised"
