"""The C ABI library builds for sm_103a, loads without a GPU, exports every
symbol include/pfkv.h declares, and rejects bad arguments on the host before
touching CUDA (CPU only: no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "pfkv.h")).read()
    return sorted(set(re.findall(r"PFKV_API\s+[\w\s\*]+?(pfkv_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import paged_fp8_kv_02_gb300 as pf
    from paged_fp8_kv_02_gb300 import _build
    _build.build_pfkv()
    return pf.load(build_if_missing=False)


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("pfkv_kv_append_fp8", "pfkv_paged_decode_attn", "pfkv_paged_decode_workspace_size",
              "pfkv_mla_decode_attn", "pfkv_mla_decode_workspace_size", "pfkv_validate_tables",
              "pfkv_last_error", "pfkv_kv_append_bf16", "pfkv_workspace_status", "pfkv_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_only_declared_symbols_are_exported():
    import subprocess
    from paged_fp8_kv_02_gb300 import _build
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln and ln.split()[-1].startswith("pfkv_")}
    assert exported == set(_declared())


def test_workspace_sizes_are_host_computable(lib):
    n2 = lib.pfkv_paged_decode_workspace_size(32, 48, 48, 128, 0, 0)
    n5 = lib.pfkv_paged_decode_workspace_size(8, 64, 8, 128, 4096, 1376)
    assert n2 > 0 and n5 > n2
    assert lib.pfkv_paged_decode_workspace_size(4, 6, 4, 128, 0, 0) == 0  # Hq % Hkv != 0
    assert lib.pfkv_mla_decode_workspace_size(64, 128, 512, 2048) >= 256


def test_host_validation_rejects_bad_arguments_without_cuda(lib):
    i64 = ctypes.c_int64
    # negative token count
    rc = lib.pfkv_kv_append_fp8(None, None, None, None, None, -1, 1, 128, 16, i64(1), 1.0, 1.0, None)
    assert rc == -1 and "bad sizes" in lib.pfkv_last_error().decode()
    # zero tokens is a no-op
    assert lib.pfkv_kv_append_fp8(None, None, None, None, None, 0, 1, 128, 16, i64(1), 1.0, 1.0, None) == 0
    # unsupported head_dim for decode
    rc = lib.pfkv_paged_decode_attn(None, None, None, None, 0, None, 4, None, 1, 8, 2, 64, 16, i64(8),
                                    1.0, 1.0, 0.1, 0, None, 0, None, None)
    assert rc == -2
    # group size 32 unsupported
    rc = lib.pfkv_paged_decode_attn(None, None, None, None, 0, None, 4, None, 1, 32, 1, 128, 16, i64(8),
                                    1.0, 1.0, 0.1, 0, None, 0, None, None)
    assert rc == -2
    # page size 8 unsupported
    rc = lib.pfkv_paged_decode_attn(None, None, None, None, 0, None, 4, None, 1, 8, 2, 128, 8, i64(8),
                                    1.0, 1.0, 0.1, 0, None, 0, None, None)
    assert rc == -2
    # batch 0 is a no-op
    rc = lib.pfkv_paged_decode_attn(None, None, None, None, 0, None, 4, None, 0, 8, 2, 128, 16, i64(8),
                                    1.0, 1.0, 0.1, 0, None, 0, None, None)
    assert rc == 0
    # null pointers with work to do
    rc = lib.pfkv_paged_decode_attn(None, None, None, None, 0, None, 4, None, 1, 8, 2, 128, 16, i64(8),
                                    1.0, 1.0, 0.1, 0, None, 0, None, None)
    assert rc == -1
    # MLA: only 512 + 64
    rc = lib.pfkv_mla_decode_attn(None, None, None, None, 4, None, None, 0, 1, 128, 256, 64, 64, i64(4),
                                  1.0, 0.1, None, 0, None, None)
    assert rc == -2
    rc = lib.pfkv_validate_tables(None, 4, None, 1, 16, i64(4), None, 0, None, 0, None, None)
    assert rc == -1
    assert lib.pfkv_version().decode().startswith("pfkv")
