"""The C-ABI library builds, loads, exports every symbol include/ep.h declares,
and validates arguments on the host (no GPU needed)."""
import json
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep.h")


@pytest.fixture(scope="module")
def built_lib():
    from transformer_epilogue_gb300 import build
    path = build.build()
    assert os.path.exists(path)
    return path


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(ep_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_four_ops():
    names = declared_functions()
    for op in ("ep_skip_layer_norm", "ep_bias_softmax", "ep_bias_add", "ep_quick_gelu",
               "ep_bias_softmax_workspace_size", "ep_last_error", "ep_kernel_launch_count"):
        assert op in names


def test_library_exports_every_declared_symbol(built_lib):
    out = subprocess.run(["nm", "-D", "--defined-only", built_lib], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(\S+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    # and ctypes resolves each of them
    import ctypes
    lib = ctypes.CDLL(built_lib)
    for n in declared_functions():
        getattr(lib, n)


def test_binding_signatures_cover_the_header():
    from transformer_epilogue_gb300 import _binding
    assert set(declared_functions()) <= set(_binding._SIGNATURES)


def test_binding_argument_counts_match_the_prototypes():
    # a ctypes binding whose argument list drifts from the C prototype passes
    # garbage silently; compare every declared function's parameter count
    from transformer_epilogue_gb300 import _binding
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    protos = dict(re.findall(r"(ep_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S))
    assert set(protos) == set(declared_functions())
    for name, params in protos.items():
        params = params.strip()
        n = 0 if params in ("", "void") else len(params.split(","))
        assert len(_binding._SIGNATURES[name][1]) == n, name


def test_host_validation_contracts(built_lib):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "abi_host_cases.py")], env=env,
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert p.returncode == 0, p.stdout[-4000:] + p.stderr[-4000:]
    res = json.loads(p.stdout.strip().splitlines()[-1])
    assert res["cases"] >= 60 and not res["failures"]


def test_missing_library_fails_loudly(tmp_path):
    from transformer_epilogue_gb300 import _binding
    with pytest.raises(ImportError):
        _load_fresh(_binding, str(tmp_path / "nope.so"))


def _load_fresh(binding, path):
    saved = binding._lib
    binding._lib = None
    try:
        return binding.load_library(path)
    finally:
        binding._lib = saved
