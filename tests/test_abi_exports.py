"""The C-ABI library builds, loads without a GPU and exports every function
that include/*.h declares (no compute call is made)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M):
            if m.group(1) not in ("if", "sizeof"):
                names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib_path():
    from speculative_decoding_verify_split_gb300.build import build_library
    return build_library()


def test_header_declares_the_binding_names():
    import speculative_decoding_verify_split_gb300 as va
    assert _declared() == set(va.EXPORTS)


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in sorted(_declared()):
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert _declared() <= exported
    assert not any(s.startswith("cuda") for s in exported), "CUDA runtime symbols leak out"


def test_status_strings(lib_path):
    import speculative_decoding_verify_split_gb300 as va
    lib = va.library()
    for code, name in va.STATUS_NAMES.items():
        assert lib.verify_attn_status_string(code).decode().startswith(name)
    assert b"unknown" in lib.verify_attn_status_string(99)
