"""The product path has no CPU fallback and never touches the oracle: without
libzq.so every call raises, the package's sources neither import nor include
anything of oracle/, and the library exports none of the oracle's symbols."""
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
