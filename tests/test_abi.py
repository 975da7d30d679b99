"""The C-ABI library builds, loads and exports every function include/pkv.h declares.

No GPU: only calls that the library rejects (or finishes) during host-side
validation, before any CUDA call, are made here.
"""
import ctypes
import subprocess

import pytest

import paged_kv_cache_165_gb300 as pkv
from paged_kv_cache_165_gb300 import _binding, _build


@pytest.fixture(scope="module")
def L():
    _build.build()
    return pkv.lib()


def test_header_declares_the_boundary():
    names = set(pkv.header_functions())
    for fn in ["pkv_kv_append", "pkv_kv_block_copy", "pkv_paged_decode_attention",
               "pkv_prefill_attention", "pkv_decode_workspace_bytes", "pkv_decode_kernel_launches",
               "pkv_paged_attention", "pkv_paged_attention_workspace_bytes",
               "pkv_paged_attention_kernel_launches", "pkv_kv_append_fp8",
               "pkv_paged_decode_attention_fp8", "pkv_decode_step", "pkv_decode_step_kernel_launches",
               "pkv_decode_step_fp8", "pkv_decode_step_fp8_kernel_launches", "pkv_get_device_error",
               "pkv_paged_decode_attention_noalloc", "pkv_selftest_bounded_wait",
               "pkv_status_string", "pkv_last_error", "pkv_version"]:
        assert fn in names


def test_library_exports_every_declared_function(L):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [fn for fn in pkv.header_functions() if fn not in exported]
    assert not missing, missing
    for fn in pkv.header_functions():
        assert hasattr(L, fn)


def test_status_strings_and_version(L):
    assert L.pkv_status_string(0) == b"ok"
    assert L.pkv_status_string(1) == b"invalid argument"
    assert L.pkv_status_string(3).startswith(b"workspace")
    assert L.pkv_version() >= 10000


def _null():
    return ctypes.c_void_p(0)


def test_host_validation_rejects_bad_arguments_before_any_launch(L):
    n = _null()
    # kv_append: T < 0, null pointers, unknown element type
    assert L.pkv_kv_append(n, n, n, n, 1, n, -1, 8, 128, 16, 4, n) == _binding.PKV_ERR_INVALID_ARG
    assert L.pkv_kv_append(n, n, n, n, 1, n, 3, 8, 128, 16, 4, n) == _binding.PKV_ERR_INVALID_ARG
    assert b"null" in L.pkv_last_error()
    assert L.pkv_kv_append(n, n, n, n, 7, n, 3, 8, 128, 16, 4, n) == _binding.PKV_ERR_UNSUPPORTED
    # T == 0 is a no-op that succeeds without touching the device
    assert L.pkv_kv_append(n, n, n, n, 1, n, 0, 8, 128, 16, 4, n) == _binding.PKV_OK
    # block copy with n == 0 is a no-op; negative n rejected
    assert L.pkv_kv_block_copy(n, n, 1, n, 0, 8, 128, 16, 4, n) == _binding.PKV_OK
    assert L.pkv_kv_block_copy(n, n, 1, n, -1, 8, 128, 16, 4, n) == _binding.PKV_ERR_INVALID_ARG
    # decode: Hq % Hkv != 0, d > 256, B == 0 (no-op), null pointers
    args = lambda B, Hq, Hkv, d: (n, n, n, n, n, 1, n, n, B, Hq, Hkv, d, 16, 8, 64, 0.1, 0, n, 0, n)
    assert L.pkv_paged_decode_attention(*args(2, 6, 4, 128)) == _binding.PKV_ERR_INVALID_ARG
    assert b"Hq % Hkv" in L.pkv_last_error()
    assert L.pkv_paged_decode_attention(*args(2, 8, 4, 512)) == _binding.PKV_ERR_INVALID_ARG
    assert L.pkv_paged_decode_attention(*args(0, 8, 4, 128)) == _binding.PKV_OK
    assert L.pkv_paged_decode_attention(*args(2, 8, 4, 128)) == _binding.PKV_ERR_INVALID_ARG
    # prefill: bad head ratio; cache write without caches
    pre = lambda Hq, Hkv, slot: (n, n, n, n, n, 1, n, 2, 10, 8, Hq, Hkv, 64, 0.1, n, n, slot, 16, 4, n)
    assert L.pkv_prefill_attention(*pre(6, 4, n)) == _binding.PKV_ERR_INVALID_ARG
    assert L.pkv_prefill_attention(*pre(8, 2, ctypes.c_void_p(16))) == _binding.PKV_ERR_INVALID_ARG
    # device error query needs a host pointer
    assert L.pkv_get_device_error(None, n) == _binding.PKV_ERR_INVALID_ARG


def test_decode_kernel_launches_rejects_what_decode_rejects(L):
    # invalid sizes and element types answer -1 before the device is queried; B == 0 is 0
    assert L.pkv_decode_kernel_launches(4, 10, 3, 128, 16, 8, 64, 1, 0) == -1   # Hq % Hkv
    assert L.pkv_decode_kernel_launches(4, 8, 8, 128, 16, 8, 0, 1, 0) == -1    # NB < 1
    assert L.pkv_decode_kernel_launches(4, 8, 8, 128, 16, 8, 64, 7, 0) == -1   # element type
    assert L.pkv_decode_kernel_launches(4, 8, 8, 128, 16, 8, 64, 1, -1) == -1  # num_splits
    assert L.pkv_decode_kernel_launches(0, 8, 8, 128, 16, 8, 64, 1, 0) == 0


def test_decode_step_rejects_bad_arguments_before_any_launch(L):
    P = ctypes.c_void_p
    args = dict(B=2, Hq=8, Hkv=2, d=64, bs=16, MBS=4, NB=8)
    def call(**kw):
        a = {**args, **kw}
        nz = P(16)   # never dereferenced: validation fails first
        return L.pkv_decode_step(nz, None, nz, nz, nz, nz, nz, nz, 1, nz, nz, a["B"], a["Hq"], a["Hkv"],
                                 a["d"], a["bs"], a["MBS"], a["NB"], 0.1, 0, None, 0, None)
    assert call(Hq=10, Hkv=3) == 1        # Hq % Hkv
    assert call(NB=0) == 1
    assert call(B=0) == 0                 # nothing to do
    assert L.pkv_decode_step(P(16), None, P(16), None, P(16), P(16), P(16), P(16), 1, P(16), P(16),
                             2, 8, 2, 64, 16, 4, 8, 0.1, 0, None, 0, None) == 1   # null k_new
    assert L.pkv_decode_step_kernel_launches(2, 10, 3, 64, 16, 4, 8, 1, 0) == -1


def test_decode_step_fp8_rejects_bad_arguments_before_any_launch(L):
    P = ctypes.c_void_p
    nz = P(16)   # never dereferenced: validation fails first
    def call(new_dt=1, B=2, Hq=8, Hkv=2, NB=8, k_new=nz):
        return L.pkv_decode_step_fp8(nz, None, nz, k_new, nz, new_dt, nz, nz, nz, nz, nz, nz, nz, B, Hq, Hkv,
                                     128, 16, 4, NB, 0.1, 0, None, 0, None)
    assert call(new_dt=2) == 2            # FP8 new rows: unsupported
    assert call(Hq=10, Hkv=3) == 1        # Hq % Hkv
    assert call(NB=0) == 1
    assert call(k_new=None) == 1          # null pointer
    assert call(B=0) == 0                 # nothing to do
    assert L.pkv_decode_step_fp8_kernel_launches(2, 8, 2, 128, 16, 4, 8, 2, 0) == -1


def test_selftest_bounded_wait_rejects_limits_and_grids_out_of_range(L):
    n = _null()
    for limit, blocks in [(0, 1), (2_000_000_000, 1), (1_000_000, 0), (1_000_000, 1025)]:
        assert L.pkv_selftest_bounded_wait(limit, blocks, 1, n, n) == _binding.PKV_ERR_INVALID_ARG
        assert b"selftest_bounded_wait" in L.pkv_last_error()
