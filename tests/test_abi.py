"""The C-ABI libraries load and export every symbol their headers declare
(no compute calls: this runs without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

from cached_masked_decoding_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIBDIR = os.path.join(ROOT, "cached_masked_decoding_gb300", "_lib")


def declared(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^[A-Za-z_][A-Za-z0-9_ \*]*?\b(dllm_[a-z0-9_]+)\s*\(", text, flags=re.M))


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(os.path.join(LIBDIR, "libdllm.so")) or \
            not os.path.exists(os.path.join(LIBDIR, "libdllm_synth.so")):
        from cached_masked_decoding_gb300 import build
        build.build()


def test_header_declares_the_boundary():
    names = declared("dllm.h")
    for must in ("dllm_load", "dllm_prefill_refresh", "dllm_denoise_step", "dllm_generate", "dllm_run",
                 "dllm_op_gemm", "dllm_op_attention", "dllm_op_select_commit"):
        assert must in names
    assert set(binding.SIGNATURES) == names


@pytest.mark.parametrize("lib,header", [("libdllm.so", "dllm.h"), ("libdllm_synth.so", "dllm_synth.h")])
def test_library_exports_every_declared_symbol(lib, header):
    path = os.path.join(LIBDIR, lib)
    handle = ctypes.CDLL(path)
    for name in declared(header):
        assert hasattr(handle, name), f"{lib} does not export {name}"
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (dllm_[a-z0-9_]+)$", out, flags=re.M))
    assert declared(header) <= exported


def test_host_side_errors_without_gpu_work():
    L = binding.lib()
    assert L.dllm_version() >= 100
    assert L.dllm_status_string(binding.EINVAL) == b"invalid argument"
    # argument validation happens before any device call
    h = ctypes.c_void_p()
    bad = binding.Config(2, 100, 4, 64, 688, 1024, 1e4, 1e-5)   # d not a multiple of 128
    assert L.dllm_model_create(ctypes.byref(bad), ctypes.byref(h)) == binding.EINVAL
    assert b"unsupported config" in L.dllm_last_error()
    assert L.dllm_model_create(None, ctypes.byref(h)) == binding.EINVAL
    assert L.dllm_load(b"/nonexistent/weights.bin", ctypes.byref(h)) == binding.EIO
    assert L.dllm_prefill_refresh(None) == binding.EINVAL
    assert L.dllm_denoise_step(None, 0, 0.9, 2, None) == -binding.EINVAL
    # state switches on a NULL state
    for fn in (L.dllm_state_set_run_ahead, L.dllm_state_set_fused_refresh):
        assert fn(None, 1) == binding.EINVAL
    # the single-kernel attention entries reject bad shapes and unaligned pointers before any launch
    for fn in (L.dllm_op_attention, L.dllm_op_attention_tc, L.dllm_op_attention_noalloc):
        assert fn(None, None, None, None, 1, 1, 128, 1, 1, None) == binding.EINVAL
        assert fn(16, 16, 16, 16, 1, 1, 96, 1, 1, None) == binding.EINVAL      # hd not 64 or 128
        assert fn(16, 16, 16, 16, 1, 1, 128, 0, 1, None) == binding.EINVAL     # no query rows
    assert L.dllm_op_attention_tc(18, 16, 16, 16, 1, 1, 128, 1, 1, None) == binding.EINVAL   # q not 16-byte aligned
    assert L.dllm_op_attention_tc_ex(16, 16, 16, 16, 1, 1, 128, 1, 1, 9, None) == binding.EINVAL   # over 8 splits
    assert L.dllm_op_attention_tc_ex(16, 16, 16, 16, 1, 1, 128, 1, 1, -1, None) == binding.EINVAL
    assert b"bad attention arguments" in L.dllm_last_error()


def test_fault_injection_io(monkeypatch, tmp_path):
    L = binding.lib()
    p = tmp_path / "w.bin"
    p.write_bytes(b"DLLMW001" + b"\0" * 8)
    monkeypatch.setenv("DLLM_FAULT", "io")
    h = ctypes.c_void_p()
    assert L.dllm_load(str(p).encode(), ctypes.byref(h)) == binding.EIO
    assert b"DLLM_FAULT=io" in L.dllm_last_error()
    monkeypatch.delenv("DLLM_FAULT")
    # a truncated header is an I/O error, not a crash
    assert L.dllm_load(str(p).encode(), ctypes.byref(h)) == binding.EIO
