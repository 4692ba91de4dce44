"""The C-ABI library builds, loads, and exports every entry point that
include/ua.h declares; descriptor validation needs no GPU.  CPU only (no
compute call is made here)."""
import ctypes
import os
import re

import pytest

import paged_varlen_flash_gb300 as ua
from paged_varlen_flash_gb300 import build as ua_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(ua_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    ua_build.build()
    return ua.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ua_problem_create", "ua_forward", "ua_destroy", "ua_check_device_error",
                     "ua_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_status_strings(lib):
    assert ua.ua_status_string(0) == "ok"
    assert "invalid" in ua.ua_status_string(1)
    assert "unsupported" in ua.ua_status_string(2)


def _desc(**over):
    base = dict(num_q_heads=8, num_kv_heads=2, head_size=128, block_size=16, num_blocks=64,
                max_num_seqs=4, max_blocks_per_seq=8, max_total_q=64, dtype=0,
                flags=ua.UA_FLAG_CAUSAL, scale=0.125, softcap=0.0, window=0)
    base.update(over)
    return ua.binding.ProblemDesc(**base)


@pytest.mark.parametrize("over,status", [
    (dict(num_kv_heads=3), 1),                      # H_q % H_k != 0
    (dict(num_q_heads=0), 1),
    (dict(num_blocks=0), 1),
    (dict(scale=0.0), 1),
    (dict(flags=ua.UA_FLAG_WINDOW, window=4), 1),   # window without causal
    (dict(flags=ua.UA_FLAG_CAUSAL | ua.UA_FLAG_WINDOW, window=0), 1),
    (dict(flags=ua.UA_FLAG_CAUSAL | ua.UA_FLAG_SOFTCAP, softcap=0.0), 1),
    (dict(flags=1 << 9), 1),                        # unknown flag
    (dict(head_size=96), 2),
    (dict(block_size=8), 2),
    (dict(dtype=1), 2),
    (dict(split_partials=2), 1),                    # unknown partials type
])
def test_descriptor_validation_before_any_device_work(lib, over, status):
    h = ctypes.c_void_p()
    st = lib.ua_problem_create(ctypes.byref(_desc(**over)), ctypes.byref(h))
    assert st == status
    assert not h.value


def test_null_arguments_are_rejected(lib):
    assert lib.ua_problem_create(None, None) == 1
    assert lib.ua_forward(None, None, None, None, None, None, None, 0, 0, 0, 0, 0, None,
                          None, None, None) == 1
    code = ctypes.c_int32(0)
    assert lib.ua_check_device_error(None, None, ctypes.byref(code)) == 1
    lib.ua_destroy(None)  # no-op


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from paged_varlen_flash_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "_LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.load_library()


def test_qq_bias_setter_checks_its_arguments_on_the_host(lib):
    # No problem handle: rejected before anything else is looked at.
    assert lib.ua_set_qq_bias(None, None, 0, 0) == 1
    assert ua.UA_FLAG_QQ_BIAS == 1 << 5


def test_noalloc_rejects_the_qq_bias_flag_before_any_device_work(lib):
    d = _desc(flags=ua.UA_FLAG_CAUSAL | ua.UA_FLAG_QQ_BIAS)
    st = ua.ua_forward_noalloc(d, None, None, None, None, None, None, 1, 1, 1, 1,
                               ua.UA_FLAG_CAUSAL | ua.UA_FLAG_QQ_BIAS, None, None, None,
                               stream=0)
    assert st == 2


def test_topk_entry_checks_its_handle_on_the_host(lib):
    # No problem handle: rejected before any pointer is looked at.
    assert ua.ua_forward_topk(None, None, None, None, None, None, None, 1, 1, 1, 1, None, None,
                              16, ua.UA_FLAG_CAUSAL, None, None, None, stream=0) == 1
