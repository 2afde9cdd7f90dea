"""The C-ABI library loads, exports every symbol include/*.h declares, and its
host-only entry points behave (no GPU needed: nothing here launches work)."""
import ctypes
import glob
import os
import re

import pytest

from combine_get_dispatch_histograms_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"\b(ep_[a-z0-9_]+)\s*\(", src):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 20
    for n in sorted(names):
        assert hasattr(lib, n), n
    # and the binding declares exactly the header's functions
    assert names == set(_lib.SIGNATURES), names ^ set(_lib.SIGNATURES)


def test_status_names_and_version(lib):
    assert lib.ep_status_name(0) == b"EP_OK"
    assert lib.ep_status_name(-4) == b"EP_ERR_TIMEOUT"
    assert b"sm_103a" in lib.ep_version()


def test_size_hint_matches_oracle(lib, orc):
    for cap, H, R, E in ((128, 7168, 16, 256), (256, 4096, 32, 256), (6, 128, 4, 8), (1, 256, 1, 1)):
        assert lib.ep_ll_message_bytes(H) == orc.ll_message_bytes(H)
        assert lib.ep_ll_size_hint(cap, H, R, E) == orc.ll_size_hint(cap, H, R, E)
    assert lib.ep_ll_size_hint(0, 128, 1, 1) == 0


@pytest.mark.parametrize("cfg", [
    (0, 8, 2, 4, 128, 2, 1),      # no ranks
    (3, 8, 2, 4, 128, 2, 1),      # E % R
    (4, 8, 0, 4, 128, 2, 1),      # K = 0
    (4, 8, 33, 4, 128, 2, 1),     # K > 32
    (4, 8, 2, -1, 128, 2, 1),     # T < 0
    (4, 8, 2, 4, 100, 2, 1),      # H % 8
    (4, 8, 2, 4, 128, 0, 1),      # C = 0
    (4, 8, 2, 4, 128, 2, 3),      # R % N
    (65, 65, 2, 4, 128, 2, 1),    # R > 64
])
def test_config_validation_before_any_cuda_call(lib, cfg):
    c = _lib.EpConfig(*cfg)
    out = ctypes.c_void_p()
    rc = lib.ep_ctx_create(ctypes.byref(c), ctypes.byref(out))
    assert rc == -1 and not out
    assert lib.ep_last_error()


def test_ll_config_validation(lib):
    out = ctypes.c_void_p()
    c = _lib.EpConfig(4, 8, 2, 4, 100, 1, 1)  # H not a multiple of 128
    assert lib.ep_ll_buffer_create(ctypes.byref(c), 4, ctypes.byref(out)) == -1
    c = _lib.EpConfig(4, 8, 2, 4, 128, 1, 1)
    assert lib.ep_ll_buffer_create(ctypes.byref(c), 0, ctypes.byref(out)) == -1


def test_null_context_rejected(lib):
    assert lib.ep_get_dispatch_layout(None, None, None, None, None, None, None, None) == -1
    assert lib.ep_ctx_check(None, None) == -1
    assert lib.ep_ll_send(None, None, None, 0, 0, None, None) == -1


def test_plain_c_caller(tmp_path):
    """include/ep.h compiles as C and a C program links and calls the library."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    lib_path = _lib.load()._name
    exe = tmp_path / "abi_host"
    src = os.path.join(ROOT, "tests", "c", "abi_host.c")
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src,
                        lib_path, f"-Wl,-rpath,{os.path.dirname(lib_path)}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and "c abi ok" in r.stdout, r.stdout + r.stderr
