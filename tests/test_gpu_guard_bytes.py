"""Every kernel that writes device memory writes only its own outputs, and all
of them: each output (and, for the append, each cache) sits inside a buffer
whose surrounding guard bytes must come back unchanged, and no output element
may be left holding the guard pattern.  The element values themselves are
compared with the oracle by the other GPU tests."""
import numpy as np
import pytest

import oracle
import synth

import test_gpu_mla_and_validate as tmla
import test_gpu_paged_decode as tdec
import test_gpu_prefill as tpre
import test_gpu_scales as tscl
from guard_helpers import Guarded
from gpu_helpers import pf
from oracle_helpers import oracle_fill_paged

pytestmark = pytest.mark.gpu


def _sync():
    import torch
    torch.cuda.synchronize()


def _outputs(rows, Hq, D):
    import torch
    return Guarded((rows, Hq, D), torch.bfloat16, "cuda"), Guarded((rows, Hq), torch.float32, "cuda")


def _check_outputs(out, lse, what):
    out.check(f"{what} out")
    lse.check(f"{what} lse")
    assert out.unwritten() == 0, f"{what}: output elements left unwritten"
    assert lse.unwritten() == 0, f"{what}: lse elements left unwritten"


DECODE_CASES = [
    dict(Hq=4, Hkv=4, lens=(1, 15, 17, 300)),                  # MHA, ragged tails
    dict(Hq=16, Hkv=2, P=64, lens=(64, 65, 700, 129)),         # G = 8, page 64
    dict(Hq=32, Hkv=2, lens=(40, 500, 3, 77)),                 # G = 16
    dict(Hq=8, Hkv=8, lens=(0, 50, 0, 7)),                     # empty contexts
]


# the bf16 cache on the configuration its oracle tests also run (MHA, page 16)
@pytest.mark.parametrize("case,bf16", [(i, False) for i in range(len(DECODE_CASES))] + [(0, True)])
@pytest.mark.parametrize("split", [0, 16])
def test_decode_writes_only_its_outputs(case, split, bf16):
    p = pf()
    c = dict(DECODE_CASES[case])
    lens = c.pop("lens")
    w = synth.PagedWorkload("guard", B=len(lens), D=128, P=c.pop("P", 16), context_lens=np.array(lens),
                            seed=61, n_new=1 if min(lens) > 0 else 0, **c)
    st = tdec._setup(p, w, bf16)
    out, lse = _outputs(w.B, w.Hq, w.D)
    maxc = int(sum((int(L) + split - 1) // split for L in w.context_lens)) if split else 0
    ks, vs = (1.0, 1.0) if bf16 else (w.k_scale, w.v_scale)
    ws = p.paged_decode_attn(out.t, st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens, ks, vs,
                             w.softmax_scale, kv_split_tokens=split, lse_out=lse.t, max_total_chunks=maxc)
    _sync()
    assert p.workspace_status(ws) == 0
    _check_outputs(out, lse, f"decode case {case} split {split} bf16 {bf16}")


@pytest.mark.parametrize("gran", tscl.GRANS)
def test_scaled_decode_writes_only_its_outputs(gran):
    p = pf()
    lens = (5, 40, 300, 17)
    w = synth.PagedWorkload("guard", B=len(lens), Hq=16, Hkv=2, D=128, P=16, context_lens=np.array(lens),
                            seed=62)
    okc, ovc, oks, ovs = tscl.oracle_fill_scaled(w, gran, zero_rows=True)
    out, lse = _outputs(w.B, w.Hq, w.D)
    ws = p.paged_decode_attn_scaled(out.t, tscl._dev_bits(w.q_bits()), tscl._dev(okc), tscl._dev(ovc), gran,
                                    tscl._dev(oks), tscl._dev(ovs), tscl._dev(w.block_tables),
                                    tscl._dev(w.context_lens), w.softmax_scale, kv_split_tokens=16,
                                    lse_out=lse.t,
                                    max_total_chunks=int(sum((int(L) + 15) // 16 for L in lens)))
    _sync()
    assert p.workspace_status(ws) == 0
    _check_outputs(out, lse, f"scaled decode gran {gran}")


@pytest.mark.parametrize("gran", [None] + tscl.GRANS)
def test_append_writes_only_the_cache(gran):
    """Skipped slots (negative, or past the pool) write nothing either."""
    import torch
    p = pf()
    w = synth.PagedWorkload("guard", B=3, Hq=4, Hkv=2, D=128, P=16, context_lens=np.array([1, 31, 70]), seed=63)
    w.set_scales_host()
    shape = (w.num_pages, w.Hkv, w.P, w.D)
    kc, vc = Guarded(shape, torch.uint8, "cuda"), Guarded(shape, torch.uint8, "cuda")
    kc.t.zero_()
    vc.t.zero_()
    if gran == oracle.SCALE_TOKEN:
        ks, vs = Guarded(shape[:3], torch.float32, "cuda"), Guarded(shape[:3], torch.float32, "cuda")
    elif gran is not None:
        n = 1 if gran == oracle.SCALE_TENSOR else w.Hkv
        ks, vs = Guarded((n,), torch.float32, "cuda"), Guarded((n,), torch.float32, "cuda")
        ks.t.fill_(w.k_scale)
        vs.t.fill_(w.v_scale)
    for b in range(w.B):
        L = int(w.context_lens[b])
        kb = tscl._dev_bits(w.kv_bits("k", b, 0, L))
        vb = tscl._dev_bits(w.kv_bits("v", b, 0, L))
        slots = w.slots(b, 0, L).copy()
        if L > 2:
            slots[0] = -1                          # skipped
            slots[1] = w.num_pages * w.P + 3       # past the pool: skipped
        sl = tscl._dev(slots)
        if gran is None:
            p.kv_append_fp8(kb, vb, kc.t, vc.t, sl, w.k_scale, w.v_scale)
        else:
            p.kv_append_fp8_scaled(kb, vb, kc.t, vc.t, sl, gran, ks.t, vs.t)
    _sync()
    kc.check("k cache")
    vc.check("v cache")
    if gran is not None:
        ks.check("k scales")
        vs.check("v scales")


PREFILL_CASES = [
    dict(Hq=16, Hkv=2, n_new=2, lens=(40, 300, 17, 129), split=0),     # wide tiles
    dict(Hq=16, Hkv=2, n_new=2, lens=(40, 300, 17, 129), split=64),
    dict(Hq=8, Hkv=1, n_new=12, lens=(40, 300, 17, 129), split=0),     # one block per CTA
    dict(Hq=8, Hkv=1, n_new=40, lens=(60, 300, 45, 129), split=0),     # two blocks per CTA
    dict(Hq=4, Hkv=4, n_new=200, lens=(200, 250, 333), split=128),     # two blocks, MHA, chunks
]


@pytest.mark.parametrize("case", range(len(PREFILL_CASES)))
def test_prefill_writes_only_its_outputs(case):
    p = pf()
    c = PREFILL_CASES[case]
    w = tpre._w("guard", c["Hq"], c["Hkv"], c["lens"], c["n_new"], seed=67)
    w.set_scales_host()
    kc, vc = oracle_fill_paged(w)
    qs = w.q_start()
    q = tpre._dev_bits(w.q_new_bits())
    out, lse = _outputs(q.shape[0], w.Hq, w.D)
    ws = p.paged_prefill_attn(out.t, q, tpre._dev(kc), tpre._dev(vc), tpre._dev(w.block_tables),
                              tpre._dev(w.context_lens), tpre._dev(qs), int(np.diff(qs).max()),
                              int(w.context_lens.max()), w.k_scale, w.v_scale, w.softmax_scale,
                              kv_split_tokens=c["split"], lse_out=lse.t)
    _sync()
    assert p.workspace_status(ws) == 0
    _check_outputs(out, lse, f"prefill case {case}")


@pytest.mark.parametrize("case", [
    dict(H=128, lens=(300, 129, 70), topk=64),
    dict(H=128, lens=(64, 1000, 17), topk=0),
])
def test_mla_writes_only_its_outputs(case):
    p = pf()
    m = synth.MlaWorkload("guard", B=len(case["lens"]), H=case["H"], context_lens=np.array(case["lens"]),
                          topk_n=case["topk"], P=64, seed=71)
    st = tmla._setup_mla(p, m)
    out, lse = _outputs(m.B, m.H, m.Dv)
    ws = p.mla_decode_attn(out.t, st.q, st.ckv_cache, st.block_tables, st.context_lens,
                           st.topk if case["topk"] else None, m.ckv_scale, m.softmax_scale, lse_out=lse.t)
    _sync()
    assert p.workspace_status(ws) == 0
    _check_outputs(out, lse, f"mla {case}")
