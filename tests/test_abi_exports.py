"""The C-ABI library loads on the host and exports every symbol include/eri.h declares.

No GPU is needed: only host-side entry points are called (status strings,
class statistics and the argument checks that run before any CUDA call).
"""

import ctypes
import os
import re

import pytest

import electron_repulsion_integrals_gb300 as eri

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(eri.LIB_PATH):
        from electron_repulsion_integrals_gb300 import build
        build.build()
    return eri.lib()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(eri_\w+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["eri_plan_create", "eri_plan_destroy", "eri_compute_class", "eri_build_J", "eri_schwarz",
                 "eri_status_string", "eri_class_info", "eri_compute_class_noalloc"]:
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported by liberi.so"


def test_status_strings(lib):
    for code in range(-8, 1):
        s = lib.eri_status_string(code)
        assert s and s != b"unknown status"


def test_class_info_host_only(lib):
    st = eri.eri_class_info((2, 2, 2, 2))
    assert st["vrr_flops"] > 0 and st["hrr_flops"] > 0
    with pytest.raises(eri.EriError):
        eri.eri_class_info((2, 3, 0, 0))  # not canonical


def test_argument_errors_before_cuda(lib):
    out = ctypes.c_void_p()
    assert lib.eri_plan_create(None, 0, None, None, ctypes.byref(out)) == -1
    assert lib.eri_plan_destroy(None) == 0
    assert lib.eri_compute_class(None, 1, 1, 1, 1, None, 0, None, 0, None) == -1
    assert lib.eri_compute_class_noalloc(None, 1, 1, 1, 1, None, 0, None, 0, None) == -1
    assert lib.eri_build_J(None, None, None, None) == -1


def test_variant_library_links_completely():
    """A library built over another class list (build.build_variant) resolves
    every symbol of the runtime, derivative entry point included."""
    import subprocess
    from electron_repulsion_integrals_gb300.build import build_variant
    path = build_variant("abi_check", [((1, 0, 0, 0), {"tier": "staged"})])
    r = subprocess.run(["nm", "-D", "--undefined-only", path], capture_output=True, text=True)
    assert r.returncode == 0
    assert not [ln for ln in r.stdout.splitlines() if " eri_" in ln], r.stdout
