"""The product path has no CPU fallback and never touches the oracle: without
libzq.so every call raises, the package's sources neither import nor include
anything of oracle/, the library exports none of the oracle's symbols, and
bench.py reaches the oracle only in its CPU-baseline and reference legs."""
import ast
import ctypes
import os

import pytest

import blockwise_quantized_zero_gb300 as zq

PKG = os.path.dirname(os.path.abspath(zq.__file__))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(zq, "_lib", None)
    monkeypatch.setattr(zq, "LIB_PATH", str(tmp_path / "libzq.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        zq.lib()
    for call in (lambda: zq.codes_bytes(zq.INT8, 1024), lambda: zq.num_blocks(1024, 128),
                 lambda: zq.aquavit_schedule(0, 10), lambda: zq.gemm_plan(128, 1024, 1024),
                 lambda: zq.interleaved_bytes(zq.INT4, 1024, 128)):
        with pytest.raises(RuntimeError, match="is missing"):
            call()


def test_package_sources_do_not_use_the_oracle():
    for root, _, files in os.walk(PKG):
        for name in files:
            path = os.path.join(root, name)
            if name.endswith(".py"):
                with open(path) as f:
                    tree = ast.parse(f.read(), path)
                for node in ast.walk(tree):
                    if isinstance(node, ast.Import):
                        mods = [a.name for a in node.names]
                    elif isinstance(node, ast.ImportFrom):
                        mods = [node.module or ""]
                    else:
                        continue
                    assert not any(m.split(".")[0] == "oracle" for m in mods), (path, mods)
            elif name.endswith((".cu", ".cuh", ".h", ".cpp", ".c")):
                with open(path) as f:
                    for line in f:
                        if line.lstrip().startswith("#include"):
                            assert "oracle" not in line, (path, line)


def test_library_exports_no_oracle_symbol():
    if not os.path.exists(zq.LIB_PATH):
        pytest.skip("libzq.so is not built")
    L = ctypes.CDLL(zq.LIB_PATH)
    for sym in ("orc_quantize", "orc_dequantize", "orc_reduce", "orc_fp8_accumulate",
                "orc_gemm_dequant"):
        with pytest.raises(AttributeError):
            getattr(L, sym)


def _bench_oracle_uses():
    """(enclosing function, called name, line) for every import of the oracle
    and every call that leads to it in bench.py."""
    with open(os.path.join(os.path.dirname(PKG), "bench.py")) as f:
        tree = ast.parse(f.read())
    leads = {"oracle_sample", "_oracle_sample", "time_cpu_baseline", "time_cpu_all_cores",
             "reference_sample", "run_reference"}
    out = []

    class V(ast.NodeVisitor):
        def __init__(self):
            self.stack = ["<module>"]

        def visit_FunctionDef(self, node):
            self.stack.append(node.name)
            self.generic_visit(node)
            self.stack.pop()

        def visit_Import(self, node):
            if any(a.name.split(".")[0] == "oracle" for a in node.names):
                out.append((self.stack[-1], "import oracle", node.lineno))

        def visit_ImportFrom(self, node):
            if (node.module or "").split(".")[0] == "oracle":
                out.append((self.stack[-1], "import oracle", node.lineno))

        def visit_Call(self, node):
            f = node.func
            name = f.attr if isinstance(f, ast.Attribute) else getattr(f, "id", None)
            if name in leads:
                out.append((self.stack[-1], name, node.lineno))
            self.generic_visit(node)

    V().visit(tree)
    return out, tree


def test_bench_reaches_the_oracle_only_in_its_cpu_legs():
    """bench.py imports the oracle only in the workloads' oracle_sample
    methods, which only the CPU-baseline and reference legs reach; the GPU
    run calls those legs after its last timed region."""
    uses, tree = _bench_oracle_uses()
    allowed = {"import oracle": {"oracle_sample"},
               "oracle_sample": {"_oracle_sample", "reference_sample", "run_reference"},
               "_oracle_sample": {"time_cpu_baseline", "_oracle_core_worker"},
               "reference_sample": {"run_reference"},
               "run_reference": {"main"},
               "time_cpu_baseline": {"run_gpu"},
               "time_cpu_all_cores": {"run_gpu"}}
    assert uses
    for fn, what, _ in uses:
        assert fn in allowed[what], (fn, what)
    run_gpu = next(n for n in ast.walk(tree) if isinstance(n, ast.FunctionDef) and n.name == "run_gpu")
    timed = [n.lineno for n in ast.walk(run_gpu) if isinstance(n, ast.Call)
             and getattr(n.func, "id", getattr(n.func, "attr", None)) in
             ("time_steps", "e2e_step", "run_extra_config")]
    cpu = [ln for fn, what, ln in uses if fn == "run_gpu"]
    assert timed and cpu and min(cpu) > max(timed)
