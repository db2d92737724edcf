"""The oracle's e4m3 encoder against the GPU's hardware conversion
(cvt.rn.satfinite.e4m3x2.f32) on every one of the 2^32 fp32 bit patterns.

Workers AI post, §1 "KV キャッシュの量子化": keys and values are stored as
e4m3 codes; the oracle encodes by exact comparison with the decoded grid
(nearest value, ties to the even mantissa, finite overflow clamped to +-448),
which is what the conversion instruction defines.  Codes must be equal bit
for bit for every non-NaN input (signed zeros and fp32 subnormals included);
a NaN input must give a NaN code (0x7F or 0xFF).  The hardware side is a
test-only kernel (tests/cuda/e4m3_cvt.cu), compiled here; the product's
append, which converts fp32(bf16) / scale with the same instruction, is
checked separately over every bf16 input and 519 scales."""
import concurrent.futures as cf
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CHUNK = 1 << 26


def _build(tmp_path):
    from paged_fp8_kv_02_gb300 import _build as b
    lib = str(tmp_path / "libe4m3cvt.so")
    subprocess.run([b._nvcc(), *b.ARCH, "-O2", "-shared", "-Xcompiler", "-fPIC", "-o", lib,
                    os.path.join(HERE, "cuda", "e4m3_cvt.cu")], check=True, capture_output=True)
    L = ctypes.CDLL(lib)
    L.e4m3_cvt_range.restype = ctypes.c_int
    L.e4m3_cvt_range.argtypes = [ctypes.c_uint32, ctypes.c_void_p, ctypes.c_uint32]
    return L


def _oracle_codes(x, pool, parts):
    out = np.empty(x.shape[0], np.uint8)
    step = x.shape[0] // parts

    def run(k):
        sl = slice(k * step, (k + 1) * step)
        oracle.lib().orc_e4m3_encode_array(x[sl].ctypes.data, out[sl].ctypes.data, step)

    list(pool.map(run, range(parts)))
    return out


def test_oracle_encoder_equals_hardware_on_every_fp32(tmp_path):
    import torch
    L = _build(tmp_path)
    dev = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    parts = max(1, min(32, os.cpu_count() or 1))
    assert CHUNK % parts == 0
    nan_codes = np.array([0x7F, 0xFF], np.uint8)
    with cf.ThreadPoolExecutor(parts) as pool:
        for start in range(0, 1 << 32, CHUNK):
            assert L.e4m3_cvt_range(start, dev.data_ptr(), CHUNK) == 0
            torch.cuda.synchronize()
            hw = dev.cpu().numpy()
            bits = np.arange(start, start + CHUNK, dtype=np.uint32)
            ref = _oracle_codes(bits.view(np.float32), pool, parts)
            nan = ((bits & 0x7F800000) == 0x7F800000) & ((bits & 0x007FFFFF) != 0)
            bad = np.flatnonzero((hw != ref) & ~nan)
            assert bad.size == 0, (f"{bad.size} codes differ from 0x{start:08x}; first input 0x{int(bits[bad[0]]):08x}: "
                                   f"hardware 0x{int(hw[bad[0]]):02x}, oracle 0x{int(ref[bad[0]]):02x}")
            if nan.any():
                assert np.isin(hw[nan], nan_codes).all() and np.isin(ref[nan], nan_codes).all()
