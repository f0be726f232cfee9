"""The C ABI without a GPU: the library loads, exports every declared entry
point, sizes workspaces and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import fp4_mixture_experts_gb300 as moe
from fp4_mixture_experts_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(moe.lib_path()):
        build_mod.build()
    return moe.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "moe_fp4.h")).read()
    return sorted(set(re.findall(r"^(?:size_t|int|const char\*)\s+(moe_fp4_\w+)\s*\(", text, re.M)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(moe.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_workspace_sizes(lib):
    assert moe.workspace_bytes(32, 4096, 2048, 256, 8) > 0
    assert moe.host_workspace_bytes(32, 4096, 2048, 256, 8) > moe.workspace_bytes(32, 4096, 2048, 256, 8)
    # grows with T
    assert moe.workspace_bytes(64, 4096, 2048, 256, 8) > moe.workspace_bytes(32, 4096, 2048, 256, 8)
    for bad in [(0, 256, 128, 8, 2), (16, 100, 128, 8, 2), (16, 256, 96, 8, 2), (16, 256, 128, 8, 9),
                (16, 256, 128, 2000, 2), (16, 256, 128, 8, 0), (16, 256, 128, 64, 33)]:
        assert moe.workspace_bytes(*bad) == 0, bad


def test_status_strings(lib):
    for s in (0, -1, -2, -3, -4, -5, 7):
        assert isinstance(moe.status_string(s), str) and moe.status_string(s)



def test_bad_arguments_are_rejected_on_the_host(lib):
    P = ctypes.c_void_p
    d = moe.Dims(16, 256, 128, 8, 2)
    fake = 0x100000  # never dereferenced: every call below fails its host-side checks
    args = [P(fake)] * 7
    none = [None] * 5
    # null out
    rc = lib.moe_fp4_forward(ctypes.byref(d), *args[:6], None, *none, 0, P(fake), 1 << 30, None)
    assert rc == -1
    # unknown flags
    rc = lib.moe_fp4_forward(ctypes.byref(d), *args, *none, 0x80, P(fake), 1 << 30, None)
    assert rc == -1
    rc = lib.moe_fp4_forward(ctypes.byref(d), *args, *none, 0x20, P(fake), 1 << 30, None)
    assert rc == -1
    # the slot-order combine flag is a known flag: the call gets as far as the workspace check
    rc = lib.moe_fp4_forward(ctypes.byref(d), *args, *none, moe.FLAG_DETERMINISTIC, P(fake), 64, None)
    assert rc == -3
    # both path flags
    rc = lib.moe_fp4_forward(ctypes.byref(d), *args, *none, 0x3, P(fake), 1 << 30, None)
    assert rc == -1
    # unsupported sizes
    bad = moe.Dims(16, 100, 128, 8, 2)
    rc = lib.moe_fp4_forward(ctypes.byref(bad), *args, *none, 0, P(fake), 1 << 30, None)
    assert rc == -2
    # misaligned x
    rc = lib.moe_fp4_forward(ctypes.byref(d), P(fake + 2), *args[1:], *none, 0, P(fake), 1 << 30, None)
    assert rc == -1
    # misaligned workspace
    rc = lib.moe_fp4_forward(ctypes.byref(d), *args, *none, 0, P(fake + 16), 1 << 30, None)
    assert rc == -1
    # workspace too small
    rc = lib.moe_fp4_forward(ctypes.byref(d), *args, *none, 0, P(fake), 64, None)
    assert rc == -3
    # the GEMV path needs d and I multiples of 1024
    rc = lib.moe_fp4_forward(ctypes.byref(d), *args, *none, 0x1, P(fake), 1 << 30, None)
    assert rc == -2
    # route: null outputs
    rc = lib.moe_fp4_route(ctypes.byref(d), P(fake), None, P(fake), P(fake), P(fake), P(fake), 1 << 30, None)
    assert rc == -1
    rc = lib.moe_fp4_check(None, None)
    assert rc == -1


def test_mxfp8_quantize_rejects_bad_arguments_on_the_host(lib):
    P = ctypes.c_void_p
    fake = 0x100000  # never dereferenced: every call below fails its host-side checks
    q = lib.moe_fp4_mxfp8_quantize
    assert q(None, 4, 64, P(fake), P(fake), None) == -1           # null x
    assert q(P(fake), 4, 64, None, P(fake), None) == -1           # null codes
    assert q(P(fake), 4, 64, P(fake), None, None) == -1           # null scales
    assert q(P(fake), -1, 64, P(fake), P(fake), None) == -1       # negative rows
    assert q(P(fake), 4, 48, P(fake), P(fake), None) == -1        # K not a multiple of 32
    assert q(P(fake), 4, 0, P(fake), P(fake), None) == -1         # K = 0
    assert q(P(fake + 8), 4, 64, P(fake), P(fake), None) == -1    # misaligned x
    assert q(P(fake), 4, 64, P(fake + 4), P(fake), None) == -1    # misaligned codes
    assert q(P(fake), 0, 64, P(fake), P(fake), None) == 0         # no rows: nothing enqueued
    assert q(None, 0, 64, None, None, None) == 0                  # no rows: pointers not looked at
    assert q(None, 0, 48, None, None, None) == -1                 # ... but K is still checked


def test_the_header_and_library_work_from_plain_c(lib):
    """A C99 program compiled against include/moe_fp4.h and linked with the library."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(moe.lib_path())
    os.makedirs(os.path.join(libdir, "_build"), exist_ok=True)
    exe = os.path.join(libdir, "_build", "abi_from_c")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c", "abi_from_c.c"), "-L", libdir, "-lmoe_fp4",
                        "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr


def test_fault_injection_setting_is_checked_on_the_host(lib):
    assert lib.moe_fp4_set_fault_injection(9, 1000) == -1
    assert lib.moe_fp4_set_fault_injection(-1, 1000) == -1
    assert lib.moe_fp4_set_fault_injection(1, 0) == -1
    assert lib.moe_fp4_set_fault_injection(0, 0) == 0


def test_forward_mx_rejects_bad_arguments_on_the_host(lib):
    P = ctypes.c_void_p
    fake = 0x100000  # never dereferenced: every call below fails its host-side checks
    d = moe.Dims(16, 256, 128, 8, 2)
    f = lib.moe_fp4_forward_mx
    ws = moe.mx_workspace_bytes(16, 256, 128, 8, 2)
    assert ws > moe.workspace_bytes(16, 256, 128, 8, 2)  # the MXFP8 operand regions
    assert moe.mx_workspace_bytes(16, 100, 128, 8, 2) == 0
    w = [P(fake)] * 7                                     # x, logits, w13, w13 scales, w2, w2 scales, out
    opt = [None] * 5                                      # h, h codes, h scales, x codes, x scales
    # null out
    assert f(ctypes.byref(d), *w[:6], None, *opt, P(fake), ws, None, None) == -1
    # w13 / w2 must be 32-byte aligned (4-bit tensor maps)
    assert f(ctypes.byref(d), P(fake), P(fake), P(fake + 16), *w[3:], *opt, P(fake), ws, None, None) == -1
    assert f(ctypes.byref(d), *w[:4], P(fake + 16), *w[5:], *opt, P(fake), ws, None, None) == -1
    # misaligned optional code outputs
    assert f(ctypes.byref(d), *w, None, P(fake + 8), None, None, None, P(fake), ws, None, None) == -1
    assert f(ctypes.byref(d), *w, None, None, None, P(fake + 8), None, P(fake), ws, None, None) == -1
    # unsupported sizes, workspace too small, misaligned workspace
    bad = moe.Dims(16, 100, 128, 8, 2)
    assert f(ctypes.byref(bad), *w, *opt, P(fake), ws, None, None) == -2
    assert f(ctypes.byref(d), *w, *opt, P(fake), ws - 256, None, None) == -3
    assert f(ctypes.byref(d), *w, *opt, P(fake + 16), ws, None, None) == -1
