"""The C-ABI library builds, loads and exports every entry point that
include/lookahead.h declares (no GPU needed: nothing is called)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"LA_API[^;(]*?\b(la_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol():
    from helpers import build_lib
    path = build_lib()
    lib = ctypes.CDLL(path)
    declared = _declared()
    assert len(declared) >= 18
    for name in sorted(declared):
        assert hasattr(lib, name), name


def test_binding_covers_every_symbol():
    import lossless_lookahead_decoding_gb300 as LA
    assert set(LA.EXPORTS) == _declared()
    for name in LA.EXPORTS:
        assert callable(getattr(LA, name))


def test_product_path_does_not_reference_oracle():
    pkg = os.path.join(ROOT, "lossless_lookahead_decoding_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in src and "from oracle" not in src and "liboracle" not in src, fn
