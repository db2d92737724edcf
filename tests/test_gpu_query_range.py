"""Queries far from unit magnitude, on every attention kernel, against the oracle.

Every kernel takes its score products in a narrow format (two e4m3 parts, or
f16) after multiplying the query rows by a power of two, and multiplies the
raw scores by its inverse.  These cases check that any finite bf16 query stays
within the tolerance:

- mixed: heads of one work unit whose magnitudes differ by up to 2^130 (down
  to bf16 subnormals), plus an all-zero head;
- large: every query times 2^17, beyond f16's largest value;
- tiny: every query times 2^-124, so small that 448 / max|q| overflows fp32
  and the power of two has to be clamped.

In the last two the softmax scale is divided by the same power of two, so
the logits stay of order one and the comparison is not a bare argmax."""
import numpy as np
import pytest

import oracle
import synth
from synth import gen

import test_gpu_mla_and_validate as tmla
import test_gpu_paged_decode as tdec
import test_gpu_prefill as tpre
import test_gpu_scales as tscl
from gpu_helpers import assert_within_tolerance, oracle_caches, pf

pytestmark = pytest.mark.gpu

MIXED_EXP = (0, -3, -9, -20, -60, -130)
REGIMES = ["mixed", "large", "tiny"]
SHIFT = {"large": 17, "tiny": -124}


def _query_bits(bits, regime):
    """bf16 query bits [rows][heads][d] rescaled by powers of two: exact,
    except where values fall into bf16's subnormal range, where they round
    like any bf16 input would.  In the mixed regime the G heads of a work
    unit (G >= 6) see all six exponents."""
    x = gen.bf16_bits_to_f32(bits).astype(np.float64)
    if regime == "mixed":
        r, h = np.indices(x.shape[:2])
        e = np.take(MIXED_EXP, (r + h) % len(MIXED_EXP))
        x = np.ldexp(x, e[:, :, None])
        x[0, 1 % x.shape[1]] = 0.0
    else:
        x = np.ldexp(x, SHIFT[regime])
    return gen.f32_to_bf16_bits(x.astype(np.float32))


def _rescale(w, regime, attr):
    """Replace the workload's query generator `attr` by the rescaled rows and
    divide its softmax scale by the regime's power of two (exact in fp32)."""
    orig = getattr(w, attr)
    cache = {}

    def bits(*args):
        key = repr(args)
        if key not in cache:
            cache[key] = _query_bits(orig(*args), regime)
        return cache[key]

    setattr(w, attr, bits)
    w.softmax_scale = float(np.float32(np.ldexp(w.softmax_scale, -SHIFT.get(regime, 0))))
    assert np.isfinite(np.float32(w.softmax_scale))
    return w


def _dev_bits(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)


# ---------------------------------------------------------------- decode, host scales
DECODE_CASES = [
    dict(Hq=16, Hkv=2, lens=(40, 300, 17, 129)),   # G = 8: one head tile
    dict(Hq=32, Hkv=2, lens=(64, 200, 3, 77)),     # G = 16: two head tiles
    dict(Hq=4, Hkv=4, lens=(1, 50, 17, 300)),      # MHA
]


@pytest.mark.parametrize("regime", REGIMES)
@pytest.mark.parametrize("case,bf16", [(i, False) for i in range(len(DECODE_CASES))] + [(0, True)])
def test_decode_query_range(regime, case, bf16):
    p = pf()
    c = dict(DECODE_CASES[case])
    lens = c.pop("lens")
    w = synth.PagedWorkload("qrange", B=len(lens), D=128, P=16, context_lens=np.array(lens), seed=41, **c)
    st = tdec._setup(p, w, bf16)
    _rescale(w, regime, "q_bits")
    q = w.q_bits()
    st.q.copy_(_dev_bits(q))
    out, lse, status = tdec._run(p, w, st)
    assert status == 0
    kc, vc = oracle_caches(w, bf16=bf16)
    ks, vs = (1.0, 1.0) if bf16 else (w.k_scale, w.v_scale)
    ref, ref_lse = oracle.paged_decode(q, kc, vc, w.block_tables, w.context_lens, w.P, ks, vs,
                                       w.softmax_scale, w.Hkv)
    assert_within_tolerance(out, ref, f"{regime} case {case} bf16 {bf16}")
    np.testing.assert_allclose(lse, ref_lse, rtol=2e-5, atol=2e-4)


# ---------------------------------------------------------------- decode, device scales
@pytest.mark.parametrize("regime", REGIMES)
@pytest.mark.parametrize("gran", tscl.GRANS)
def test_scaled_decode_query_range(regime, gran):
    p = pf()
    lens = (5, 40, 300)
    w = synth.PagedWorkload("qrange", B=len(lens), Hq=16, Hkv=2, D=128, P=16, context_lens=np.array(lens),
                            seed=43)
    _rescale(w, regime, "q_bits")
    okc, ovc, oks, ovs = tscl.oracle_fill_scaled(w, gran, zero_rows=True)
    out, lse, status = tscl._decode(p, w, tscl._dev(okc), tscl._dev(ovc), gran, tscl._dev(oks),
                                    tscl._dev(ovs))
    assert status == 0
    ref, ref_lse = oracle.paged_decode_scaled(w.q_bits(), okc, ovc, gran, oks, ovs, w.block_tables,
                                              w.context_lens, w.P, w.softmax_scale, w.Hkv)
    assert_within_tolerance(out, ref, f"{regime} gran {gran}")
    np.testing.assert_allclose(lse, ref_lse, rtol=2e-5, atol=2e-4)


# ---------------------------------------------------------------- several queries per request
PREFILL_CASES = [
    dict(Hq=16, Hkv=2, n_new=2, lens=(40, 300, 17, 129)),    # <= 64 rows per block: wide tiles
    dict(Hq=8, Hkv=1, n_new=12, lens=(40, 300, 17, 129)),    # 96 rows: one block per CTA
    dict(Hq=8, Hkv=1, n_new=40, lens=(60, 300, 45, 129)),    # 320 rows: two blocks per CTA
]


@pytest.mark.parametrize("regime", REGIMES)
@pytest.mark.parametrize("case", range(len(PREFILL_CASES)))
def test_prefill_query_range(regime, case):
    c = dict(PREFILL_CASES[case])
    w = tpre._w("qrange", c["Hq"], c["Hkv"], c["lens"], c["n_new"], seed=47)
    _rescale(w, regime, "q_new_bits")
    tpre._check_small(w)


# ---------------------------------------------------------------- MLA
@pytest.mark.parametrize("regime", REGIMES)
def test_mla_query_range(regime):
    """Also, in the mixed regime, rows whose two halves (the columns the two
    CTAs of a request contract, each under its own power of two) differ by
    2^12 in either direction; the larger half keeps its magnitude, so the
    logits stay of order one."""
    p = pf()
    m = synth.MlaWorkload("qrange", B=2, H=128, context_lens=np.array([300, 129]), topk_n=64, P=64, seed=53)
    st = tmla._setup_mla(p, m)
    q = _query_bits(m.q_bits(), regime)
    if regime == "mixed":
        x = gen.bf16_bits_to_f32(q).astype(np.float64)
        x[:, 0::4, 256:] *= 2.0 ** -12
        x[:, 2::4, :256] *= 2.0 ** -12
        q = gen.f32_to_bf16_bits(x.astype(np.float32))
    m.softmax_scale = float(np.float32(np.ldexp(m.softmax_scale, -SHIFT.get(regime, 0))))
    st.q.copy_(_dev_bits(q))
    out, lse, status = tmla._run_mla(p, m, st)
    assert status == 0
    c = tmla._oracle_cache(m)
    ref, ref_lse = oracle.mla_decode(q, c, m.block_tables, m.context_lens, m.topk, m.P, m.Dv, m.ckv_scale,
                                     m.softmax_scale)
    assert_within_tolerance(out, ref, f"mla {regime}")
    np.testing.assert_allclose(lse, ref_lse, rtol=2e-5, atol=2e-4)
