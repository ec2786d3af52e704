"""The C-ABI library loads and exports every function include/bre.h declares (no GPU calls)."""
import ctypes
import os
import re

import pytest

from bit_routed_expert_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "bre.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ \*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if not n.startswith("typedef")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine", "engram_gather_decode"):
        assert n in names


def test_library_exports_every_declared_symbol():
    path = build.build()
    L = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(L, n), f"{n} declared in bre.h but not exported"
    # the binding knows every exported entry point
    assert set(declared_functions()) <= set(_lib.SIGNATURES)


def test_host_side_argument_checks_need_no_gpu():
    L = _lib.load()
    assert L.moe_route(None, None, None, 1, 32, 8, 2, None, None, None, 0, None) == _lib.BRE_ERR_ARG
    assert L.moe_permute(None, 1, 1, 1, None, None, None, None, None, None, None) == _lib.BRE_ERR_ARG
    assert L.bre_dequant(9, ctypes.c_void_p(16), 1, ctypes.c_void_p(16), None) == _lib.BRE_ERR_UNSUPPORTED
    assert L.moe_route_workspace(8, 384) >= 8 * 384 * 4
    assert L.moe_expert_ffn_workspace(0, 6, 384, 4096, 2048, 2048) == 0
    assert L.bre_status_string(2) == b"unsupported shape or format"
