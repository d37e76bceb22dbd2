"""Host-only checks of the C ABI: the library loads and exports every symbol
that include/gptq_q4.h declares; calls that fail argument checks before any
CUDA call report the right status.  No kernel is launched."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gptq_q4.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gptq_q4_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib_path():
    import __graft_entry__
    b = __graft_entry__._cuda_build_module()
    if not os.path.exists(b.LIB):
        b.build()
    return b.LIB


def test_header_declares_the_contract():
    names = declared_functions()
    for must in ("gptq_q4_make", "gptq_q4_matmul", "gptq_q4_dequant", "gptq_q4_free"):
        assert must in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (gptq_q4_[a-z0-9_]+)", out))
    assert set(declared_functions()) <= exported


def test_binding_names_match_header(lib_path):
    import gptq_bit_weight_gb300 as q4
    assert sorted(q4.EXPORTED) == declared_functions()
    for name in declared_functions():
        assert callable(getattr(q4, name))


def test_null_handle_is_invalid_argument(lib_path):
    import gptq_bit_weight_gb300 as q4
    lib = q4._lib
    assert lib.gptq_q4_set_path(None, 0) == q4.GPTQ_Q4_INVALID_ARGUMENT
    assert "NULL" in q4.gptq_q4_last_error()
    assert lib.gptq_q4_set_prefill_min_m(None, 4) == q4.GPTQ_Q4_INVALID_ARGUMENT
    assert lib.gptq_q4_set_format(None, q4.GPTQ_Q4_FORMAT_GPTQ_V2) == q4.GPTQ_Q4_INVALID_ARGUMENT
    assert lib.gptq_q4_debug_wait_probe(None, 1000, None) == q4.GPTQ_Q4_INVALID_ARGUMENT
    assert lib.gptq_q4_info(None, None, None, None, None, None, None) == q4.GPTQ_Q4_INVALID_ARGUMENT
    assert lib.gptq_q4_set_act_dtype(None, q4.GPTQ_Q4_DTYPE_BF16) == q4.GPTQ_Q4_INVALID_ARGUMENT
    assert q4.gptq_q4_last_status() == q4.GPTQ_Q4_INVALID_ARGUMENT
    q4.gptq_q4_free(None)


def test_make_argument_errors_need_no_device(lib_path):
    """Checks that come before any device call: NULL tensors, bad sizes."""
    import gptq_bit_weight_gb300 as q4
    lib = q4._lib
    for make in (lib.gptq_q4_make, lib.gptq_q4_make8):
        assert not make(None, None, None, None, 256, 256, 128)
        assert q4.gptq_q4_last_status() == q4.GPTQ_Q4_INVALID_ARGUMENT
        assert "NULL" in q4.gptq_q4_last_error()
        p = ctypes.c_void_p(16)                      # never dereferenced: the sizes are checked first
        assert not make(p, p, p, None, 256, 250, 128)
        assert q4.gptq_q4_last_status() == q4.GPTQ_Q4_INVALID_ARGUMENT
        assert not make(p, p, p, None, 256, 256, 100)   # groupsize must divide K
        assert q4.gptq_q4_last_status() == q4.GPTQ_Q4_INVALID_ARGUMENT
    assert not lib.gptq_q4_make8(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), None, 96, 256, 32)
    assert q4.gptq_q4_last_status() == q4.GPTQ_Q4_UNSUPPORTED    # K % 64


def test_missing_library_fails_loudly(tmp_path):
    """Importing the binding without the built library raises ImportError."""
    pkg = os.path.join(ROOT, "gptq_bit_weight_gb300", "__init__.py")
    dst = tmp_path / "gptq_bit_weight_gb300"
    dst.mkdir()
    (dst / "__init__.py").write_text(open(pkg).read())
    code = "import sys; sys.path.insert(0, %r)\ntry:\n import gptq_bit_weight_gb300\nexcept ImportError as e:\n print('IMPORTERROR', e)\n" % str(tmp_path)
    r = subprocess.run(["python", "-c", code], capture_output=True, text=True)
    assert "IMPORTERROR" in r.stdout
