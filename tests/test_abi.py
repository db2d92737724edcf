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


def _fake(addr=0x10000):
    """A device-looking address that the host checks never dereference."""
    return ctypes.c_void_p(addr)


def _err(lib):
    return lib.pfkv_last_error().decode()


def test_prefill_host_validation_without_cuda(lib):
    i64 = ctypes.c_int64
    ptrs = [_fake()] * 5  # out, q, k_cache, v_cache, block_tables

    def call(*, B=2, Hq=16, Hkv=2, D=128, P=16, pages=64, maxp=8, mq=4, mctx=100, ks=1.0, vs=1.0,
             sm=0.088, split=0, ctx=_fake(), qs=_fake(), ws=_fake(), wsb=1 << 20, out=None, lse=None):
        p = list(ptrs)
        if out is not None:
            p[0] = out
        return lib.pfkv_paged_prefill_attn(*p, maxp, ctx, qs, B, Hq, Hkv, D, P, i64(pages), mq, mctx, ks,
                                           vs, sm, split, ws, wsb, lse, None)

    assert call(B=-1) == -1 and "bad sizes" in _err(lib)
    assert call(Hkv=3) == -1                      # 16 % 3 != 0
    assert call(Hq=96, Hkv=1) == -2               # G = 96 does not divide 128
    assert call(D=64) == -2
    assert call(P=8) == -2
    assert call(split=32) == -1                   # not a multiple of 64
    assert call(sm=0.0) == -1 and call(ks=float("inf")) == -1
    assert call(pages=1 << 28) == -2              # 2^31 token rows or more
    assert call(B=0) == 0                         # nothing to do
    assert call(ctx=None) == -1 and "null pointer" in _err(lib)
    assert call(out=_fake(0x10008)) == -1 and "misaligned" in _err(lib)
    assert call(ws=_fake(0x10080)) == -1           # workspace not 256-byte aligned
    # 4 queries x G 8 = 32 rows: the tile space is split evenly over the SMs,
    # so the workspace holds request offsets and partial states whatever the split
    need = lib.pfkv_paged_prefill_workspace_size(2, 16, 2, 128, 4, 100, 64)
    assert need > 256 and need == lib.pfkv_paged_prefill_workspace_size(2, 16, 2, 128, 4, 100, 0)
    assert call(split=64, wsb=need - 1) == -5 and "too small" in _err(lib)
    assert call(wsb=need - 1) == -5
    # 16 queries x G 8 = 128 rows, one pass: the status word only; chunks add partial states
    assert lib.pfkv_paged_prefill_workspace_size(2, 16, 2, 128, 16, 100, 0) == 256
    assert lib.pfkv_paged_prefill_workspace_size(2, 16, 2, 128, 16, 100, 64) > 256
    assert lib.pfkv_paged_prefill_workspace_size(2, 16, 3, 128, 4, 100, 0) == 0


def test_scaled_decode_host_validation_without_cuda(lib):
    i64 = ctypes.c_int64

    def call(gran=0, kscl=_fake(), vscl=_fake(), B=2, Hq=16, Hkv=2, D=128, P=16, split=0, ws=_fake(), wsb=1 << 24):
        return lib.pfkv_paged_decode_attn_scaled(_fake(), _fake(), _fake(), _fake(), gran, kscl, vscl, _fake(), 8,
                                                 _fake(), B, Hq, Hkv, D, P, i64(64), 0.088, split, ws, wsb, None,
                                                 None)

    assert call(gran=7) == -1 and "granularity" in _err(lib)
    assert call(kscl=None) == -1 and "null scale" in _err(lib)
    assert call(vscl=_fake(0x10004)) == -1 and "16-byte" in _err(lib)
    assert call(Hq=64, Hkv=2) == -2               # group size 32
    assert call(split=8) == -1
    assert call(B=0) == 0
    assert call(wsb=64) == -5


def test_scaled_append_host_validation_without_cuda(lib):
    i64 = ctypes.c_int64

    def call(gran=2, T=4, H=2, D=128, kscl=_fake(), vscl=_fake(), v=True, slots=_fake()):
        vn, vc = (_fake(), _fake()) if v else (None, None)
        return lib.pfkv_kv_append_fp8_scaled(_fake(), vn, _fake(), vc, slots, T, H, D, 16, i64(8), gran, kscl,
                                             vscl if v else None, None)

    assert call(gran=3) == -1 and "granularity" in _err(lib)
    assert call(kscl=None) == -1 and "null scale" in _err(lib)
    assert call(vscl=_fake(0x10002)) == -1 and "4-byte" in _err(lib)
    assert call(D=576) == -2                      # per-token scales need head_dim <= 512
    assert call(D=24) == -2                       # not a multiple of 16
    assert call(T=0) == 0
    assert call(slots=_fake(0x10004)) == -1       # slot mapping must be 8-byte aligned


def test_page_tag_check_host_validation_without_cuda(lib):
    i64 = ctypes.c_int64

    def call(B=3, maxp=4, P=16, pages=64, bt=_fake(), tt=_fake(), ctx=_fake(), pt=_fake(), st=_fake()):
        return lib.pfkv_verify_page_tags(bt, tt, maxp, ctx, B, P, pt, i64(pages), st, None)

    assert call(B=-1) == -1 and call(P=0) == -1 and call(pages=0) == -1
    assert call(B=0) == 0
    assert call(pt=None) == -1 and "null pointer" in _err(lib)
    assert call(st=_fake(0x10002)) == -1 and "misaligned" in _err(lib)


def test_mla_and_table_validation_reject_misaligned_arrays_without_cuda(lib):
    i64 = ctypes.c_int64

    def mla(bt=_fake(), ctx=_fake(), topk=None, k=0, lse=None):
        return lib.pfkv_mla_decode_attn(_fake(), _fake(), _fake(), bt, 4, ctx, topk, k, 2, 128, 512, 64, 64,
                                        i64(16), 0.05, 0.07, _fake(), 256, lse, None)

    assert mla(bt=_fake(0x10002)) == -1 and "misaligned" in _err(lib)
    assert mla(ctx=_fake(0x10001)) == -1
    assert mla(topk=_fake(0x10006), k=8) == -1
    assert mla(lse=_fake(0x10003)) == -1

    def val(err=_fake(), bt=_fake(), slots=None, n=0):
        return lib.pfkv_validate_tables(bt, 4, _fake(), 2, 16, i64(8), None, 0, slots, n, err, None)

    assert val(err=_fake(0x10002)) == -1 and "misaligned" in _err(lib)
    assert val(bt=_fake(0x10001)) == -1
    assert val(slots=_fake(0x10004), n=3) == -1   # int64 slots need 8 bytes
    assert val(slots=None, n=3) == -1 and "null slot" in _err(lib)


def test_noalloc_decode_rejects_on_the_host_without_cuda(lib):
    i64 = ctypes.c_int64

    def call(B=8, Hq=64, Hkv=8, split=0, chunks=0):
        return lib.pfkv_paged_decode_attn_noalloc(_fake(), _fake(), _fake(), _fake(), 0, _fake(), 64, _fake(), B, Hq,
                                                  Hkv, 128, 16, i64(4096), 1.0, 1.0, 0.088, split, i64(chunks),
                                                  None, None, None)

    assert call(Hkv=3) == -1 and "head counts" in _err(lib)
    # 8 requests x 1M tokens cut into 4096-token chunks: 2048 chunks x 8 KV heads of partial states
    need = lib.pfkv_paged_decode_workspace_size(8, 64, 8, 128, 4096, 2048)
    assert need > 64 << 20
    assert call(split=4096, chunks=2048) == -5 and "64 MiB" in _err(lib)


@pytest.mark.parametrize("compiler,std,lang", [("gcc", "-std=c99", "c"), ("g++", "-std=c++11", "c++")])
def test_header_compiles_as_plain_c_and_cpp(tmp_path, compiler, std, lang):
    """The boundary header needs no CUDA or torch headers and no extensions."""
    import shutil
    import subprocess
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not installed")
    src = tmp_path / "use_header.c"
    src.write_text('#include "pfkv.h"\nint main(void) { return pfkv_version() == 0; }\n')
    r = subprocess.run([compiler, std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only", "-x", lang,
                        "-I", os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
