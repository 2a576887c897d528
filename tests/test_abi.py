"""The C ABI on the CPU: the library loads, exports every declared entry
point, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

import gated_delta_rule_causal_gb300 as la

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    la.build()
    return la.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "la.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("la_create", "la_forward", "la_decode_step", "la_destroy", "la_last_error", "la_status"):
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in la.h but not exported"


def test_version(lib):
    assert la.la_version() == 100


def test_null_handle_is_rejected(lib):
    assert la.la_forward(None, None, None, None, None, None, None, None, None, None, 2, 8, 0, None) == la.LA_ERR_INVALID_ARG
    assert la.la_decode_step(None, None, None, None, None, None, None, None, None, None, 2, None) == la.LA_ERR_INVALID_ARG
    assert la.la_status(None, None) == la.LA_ERR_INVALID_ARG
    assert la.lib().la_backward(None, None, None, None, None, None, None, None, None, None, None, 0, 8,
                                None) == la.LA_ERR_INVALID_ARG
    assert la.lib().la_backward_gated(None, None, None, None, None, None, None, None, None, None, None, None,
                                      None, None, None, 2, 8, None) == la.LA_ERR_INVALID_ARG
    la.la_destroy(None)                     # allowed
    assert la.la_last_error(None) == "null handle"
    assert la.la_last_launches(None) == 0


@pytest.mark.parametrize("cfg,code", [
    ((0, 1, 64, 64, 0), la.LA_ERR_INVALID_ARG),     # B < 1
    ((1, 0, 64, 64, 0), la.LA_ERR_INVALID_ARG),     # H < 1
    ((1, 1, 48, 64, 0), la.LA_ERR_UNSUPPORTED),     # d_k not in {16,32,64,128}
    ((1, 1, 64, 256, 0), la.LA_ERR_UNSUPPORTED),    # d_v too large
    ((1, 1, 64, 64, 7), la.LA_ERR_INVALID_ARG),     # bad io enum
])
def test_create_validates_before_cuda(lib, cfg, code):
    rc, h = la.la_create(*cfg)
    assert rc == code and not h.value


def test_create_without_gpu_reports_cuda(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, h = la.la_create(1, 1, 64, 64)
    assert rc == la.LA_ERR_CUDA and not h.value


def test_create_null_config(lib):
    out = ctypes.c_void_p()
    assert lib.la_create(None, ctypes.byref(out)) == la.LA_ERR_INVALID_ARG


def test_header_is_plain_c(tmp_path):
    # The boundary is a C ABI: la.h compiles as C99 (pedantic, warnings as
    # errors), with every declared entry point referenced from C.
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = tmp_path / "use_la.c"
    src.write_text('#include "la.h"\ntypedef void (*any_fn)(void);\n' +
                   "".join(f"any_fn ref_{n}(void) {{ return (any_fn)&{n}; }}\n" for n in names))
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                        "-I", inc, "-c", str(src), "-o", str(tmp_path / "use_la.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
