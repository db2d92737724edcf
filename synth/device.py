"""Device-side generation of the synthetic workloads (bit-identical to the host
generator in ``synth.gen``) and set-up of resident caches.

Input generation only.  Writing the generated rows into the paged cache is
done by the append function the caller passes in (the product's
``kv_append_fp8`` / ``kv_append_bf16``), so this module holds none of the
method's arithmetic and imports nothing from the product.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from . import gen
from .workloads import MlaWorkload, PagedWorkload, amax_from_bits, scale_from_amax

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB):
            raise OSError(f"libsynth not built: {_LIB} (run __graft_entry__.build())")
        L = ctypes.CDLL(_LIB)
        L.synth_normal_bf16.restype = ctypes.c_int
        L.synth_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                        ctypes.c_void_p, ctypes.c_void_p]
        _lib = L
    return _lib


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def fill_normal_bf16(out, key: int, base: int, amax_word=None):
    """Fill a contiguous CUDA tensor of 2-byte elements with the counter-based
    normals for counters base .. base + numel - 1 (bf16 bits)."""
    rc = _load().synth_normal_bf16(ctypes.c_void_p(out.data_ptr()), key, base, out.numel(),
                                   None if amax_word is None else ctypes.c_void_p(amax_word.data_ptr()),
                                   _stream())
    if rc != 0:
        raise RuntimeError(f"synth_normal_bf16 failed ({rc})")


def reduce_amax_bits(key: int, base: int, n: int, amax_word):
    rc = _load().synth_normal_bf16(None, key, base, n, ctypes.c_void_p(amax_word.data_ptr()), _stream())
    if rc != 0:
        raise RuntimeError(f"synth_normal_bf16 failed ({rc})")


def device_amax_paged(w: PagedWorkload, which: str) -> float:
    import torch
    key = w.key_k if which == "k" else w.key_v
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    for b in range(w.B):
        t0 = w.shared_tokens if 0 < b < w.shared_requests else 0
        for a, z, base in w.kv_runs(b, t0, int(w.context_lens[b])):
            reduce_amax_bits(key, base, (z - a) * w.Hkv * w.D, word)
    return amax_from_bits(int(word.item()))


def device_amax_mla(m: MlaWorkload) -> float:
    import torch
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    for b in range(m.B):
        reduce_amax_bits(m.key_c, m.ckv_run_base(b, 0), int(m.context_lens[b]) * m.Dqk, word)
    return amax_from_bits(int(word.item()))


@dataclass
class PagedDeviceState:
    k_cache: object
    v_cache: object
    block_tables: object
    context_lens: object
    q: object
    k_new: object
    v_new: object
    step_slots: object


def setup_paged(w: PagedWorkload, append, bf16_cache: bool = False, chunk_tokens: int = 1 << 16,
                scales_on_device: bool = True) -> PagedDeviceState:
    """Resident caches holding every prefill token of `w`, plus the step's
    inputs (q, new K/V rows, their slots) on the device.  `append(k, v, kc, vc,
    slots)` writes rows into the caches (the product's append call)."""
    import torch
    dev = "cuda"
    if not bf16_cache and (w.k_scale is None or w.v_scale is None):
        if scales_on_device:
            w.k_scale = scale_from_amax(device_amax_paged(w, "k"))
            w.v_scale = scale_from_amax(device_amax_paged(w, "v"))
        else:
            w.set_scales_host()
    dt = torch.bfloat16 if bf16_cache else torch.uint8
    shape = (w.num_pages, w.Hkv, w.P, w.D)
    kc = torch.zeros(shape, dtype=dt, device=dev)
    vc = torch.zeros(shape, dtype=dt, device=dev)
    for b in range(w.B):
        t0, t1 = w.prefill_range(b)
        for c0 in range(t0, t1, chunk_tokens):
            c1 = min(t1, c0 + chunk_tokens)
            n = c1 - c0
            kb = torch.empty((n, w.Hkv, w.D), dtype=torch.bfloat16, device=dev)
            vb = torch.empty_like(kb)
            off = 0
            for a, z, base in w.kv_runs(b, c0, c1):
                cnt = (z - a) * w.Hkv * w.D
                fill_normal_bf16(kb.view(-1)[off:off + cnt], w.key_k, base)
                fill_normal_bf16(vb.view(-1)[off:off + cnt], w.key_v, base)
                off += cnt
            slots = torch.from_numpy(w.slots(b, c0, c1)).to(dev)
            append(kb, vb, kc, vc, slots)
    q = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    fill_normal_bf16(q, w.key_q, 0)
    k_new = torch.from_numpy(w.step_kv_bits("k").view(np.int16)).to(dev).view(torch.bfloat16)
    v_new = torch.from_numpy(w.step_kv_bits("v").view(np.int16)).to(dev).view(torch.bfloat16)
    return PagedDeviceState(
        k_cache=kc, v_cache=vc,
        block_tables=torch.from_numpy(w.block_tables).to(dev),
        context_lens=torch.from_numpy(w.context_lens).to(dev),
        q=q, k_new=k_new.contiguous(), v_new=v_new.contiguous(),
        step_slots=torch.from_numpy(w.step_slots()).to(dev))


@dataclass
class MlaDeviceState:
    ckv_cache: object
    block_tables: object
    context_lens: object
    q: object
    topk: object
    c_new: object
    step_slots: object


def setup_mla(m: MlaWorkload, append, chunk_tokens: int = 1 << 16, scales_on_device: bool = True):
    """`append(c, cache4d, slots)` writes latent rows [n][1][Dqk] into the cache
    viewed as [pages][1][P][Dqk]."""
    import torch
    dev = "cuda"
    if m.ckv_scale is None:
        m.ckv_scale = scale_from_amax(device_amax_mla(m)) if scales_on_device else m.set_scales_host().ckv_scale
    cache = torch.zeros((m.num_pages, m.P, m.Dqk), dtype=torch.uint8, device=dev)
    c4 = cache.view(m.num_pages, 1, m.P, m.Dqk)
    for b in range(m.B):
        t0, t1 = m.prefill_range(b)
        for c0 in range(t0, t1, chunk_tokens):
            c1 = min(t1, c0 + chunk_tokens)
            cb = torch.empty((c1 - c0, 1, m.Dqk), dtype=torch.bfloat16, device=dev)
            fill_normal_bf16(cb, m.key_c, m.ckv_run_base(b, c0))
            append(cb, c4, torch.from_numpy(m.slots(b, c0, c1)).to(dev))
    q = torch.empty((m.B, m.H, m.Dqk), dtype=torch.bfloat16, device=dev)
    fill_normal_bf16(q, m.key_q, 0)
    c_new = torch.from_numpy(m.step_ckv_bits().view(np.int16)).to(dev).view(torch.bfloat16).contiguous()
    return MlaDeviceState(
        ckv_cache=cache, block_tables=torch.from_numpy(m.block_tables).to(dev),
        context_lens=torch.from_numpy(m.context_lens).to(dev), q=q,
        topk=None if m.topk is None else torch.from_numpy(m.topk).to(dev),
        c_new=c_new, step_slots=torch.from_numpy(m.step_slots()).to(dev))
