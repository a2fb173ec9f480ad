"""The C-ABI library builds for sm_103a, loads, and exports every entry point include/mk.h declares
(no compute calls: this runs without a GPU)."""
import ctypes
import os
import re

from quantized_gemv_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mk.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(B.build())
    names = declared_functions()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header():
    from quantized_gemv_gb300 import mk
    assert sorted(mk.EXPORTS) == declared_functions()


def test_oracle_library_builds():
    from oracle import build as OB
    assert os.path.exists(OB.build())
