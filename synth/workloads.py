"""Synthetic workloads of the pages' shapes (seeded, deterministic).

Five named workloads (``workload(name)``), plus free construction of smaller
cases for parity tests.  Each workload yields host arrays (block tables, context
lengths, slot mappings, top-k lists) and a recipe for its bf16 tensors: element
``(b, t, h, d)`` of the K, V or latent tensor takes counter index
``((b << 21) + t) * H * D + h * D + d`` in that tensor's stream, so any token
range of one request is one contiguous run of counters (filled on the device
by ``synth.device`` or regenerated on the host by ``synth.gen``).  Tokens of a
shared prefix take the index of request 0, so every sharer sees identical data.

Context length convention: ``context_lens[b]`` counts every token attended,
including the ``n_new`` tokens appended in the same step.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import gen

TOKEN_SHIFT = 21  # tokens per request < 2^21

# the five workloads of the pages' shapes, by name
TINY_GQA = "tiny_gqa_b4"
MHA_B32 = "mha_b32_h48_l8192_p16"
GQA_PREFIX = "gqa_prefix_b64_h64kv8_p16"
MLA_TOPK = "mla_topk2048_b64_h128_l65536_p64"
LONG_SPLITKV = "long_splitkv_b8_h64kv8_p64"
WORKLOADS = (TINY_GQA, MHA_B32, GQA_PREFIX, MLA_TOPK, LONG_SPLITKV)

E4M3_MAX = np.float32(448.0)


def scale_from_amax(amax: float) -> float:
    """Per-tensor fp32 scale = amax / 448 (computed in fp32)."""
    return float(np.float32(amax) / E4M3_MAX)


def amax_from_bits(bits: int) -> float:
    return float(gen.bf16_bits_to_f32(np.array([bits & 0x7FFF], np.uint16))[0])


@dataclass
class PagedWorkload:
    """GQA/MHA decode over a paged KV cache."""

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    P: int
    context_lens: np.ndarray
    n_new: int = 1
    num_pages: int | None = None
    shared_requests: int = 0
    shared_tokens: int = 0
    seed: int = 0
    kv_split_tokens: int = 0
    max_pages_per_seq: int | None = None
    k_scale: float | None = None
    v_scale: float | None = None
    block_tables: np.ndarray = field(init=False)

    def __post_init__(self):
        self.context_lens = np.asarray(self.context_lens, dtype=np.int32)
        assert self.context_lens.shape == (self.B,)
        assert self.Hq % self.Hkv == 0
        assert self.shared_tokens % self.P == 0
        L = self.context_lens.astype(np.int64)
        self.pages_per_req = (L + self.P - 1) // self.P
        if self.shared_requests > 1:
            assert np.all(L[: self.shared_requests] > self.shared_tokens)
        shared_pages = self.shared_tokens // self.P
        needed = int(self.pages_per_req.sum()) - max(self.shared_requests - 1, 0) * shared_pages
        if self.num_pages is None:
            self.num_pages = needed
        assert self.num_pages >= needed, "page pool too small"
        maxp = self.max_pages_per_seq or int(self.pages_per_req.max(initial=1))
        self.max_pages_per_seq = maxp
        perm = gen.permutation(gen.make_key(self.seed, gen.TENSOR_PERM), self.num_pages)
        bt = np.full((self.B, maxp), -1, dtype=np.int32)
        nxt = 0
        for b in range(self.B):
            for lp in range(int(self.pages_per_req[b])):
                if 0 < b < self.shared_requests and lp < shared_pages:
                    bt[b, lp] = bt[0, lp]
                else:
                    bt[b, lp] = perm[nxt]
                    nxt += 1
        self.block_tables = bt
        self.softmax_scale = float(np.float32(1.0 / math.sqrt(self.D)))
        self.key_q = gen.make_key(self.seed, gen.TENSOR_Q)
        self.key_k = gen.make_key(self.seed, gen.TENSOR_K)
        self.key_v = gen.make_key(self.seed, gen.TENSOR_V)

    # ---------------------------------------------------------------- shapes
    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def unique_tokens(self) -> int:
        """Tokens whose K/V the step must read, shared prefix counted once."""
        extra = max(self.shared_requests - 1, 0) * self.shared_tokens
        return int(self.context_lens.astype(np.int64).sum()) - extra

    def src_request(self, b: int, t: np.ndarray) -> np.ndarray:
        t = np.asarray(t, dtype=np.int64)
        if 0 < b < self.shared_requests:
            return np.where(t < self.shared_tokens, 0, b)
        return np.full(t.shape, b, dtype=np.int64)

    def kv_index(self, b: int, t0: int, t1: int) -> np.ndarray:
        """Counter indices [t1-t0][Hkv][D] for tokens t0..t1-1 of request b."""
        t = np.arange(t0, t1, dtype=np.int64)
        be = self.src_request(b, t)
        tok = (be << TOKEN_SHIFT) + t
        hd = np.arange(self.Hkv * self.D, dtype=np.int64)
        return (tok[:, None] * (self.Hkv * self.D) + hd[None, :]).reshape(t1 - t0, self.Hkv, self.D)

    def kv_runs(self, b: int, t0: int, t1: int):
        """Split [t0, t1) of request b into runs with contiguous counters:
        yields (t_start, t_end, counter_base)."""
        cuts = [t0, t1]
        if 0 < b < self.shared_requests and t0 < self.shared_tokens < t1:
            cuts = [t0, self.shared_tokens, t1]
        for a, z in zip(cuts[:-1], cuts[1:]):
            be = int(self.src_request(b, np.array([a]))[0])
            yield a, z, ((be << TOKEN_SHIFT) + a) * self.Hkv * self.D

    def kv_bits(self, which: str, b: int, t0: int, t1: int) -> np.ndarray:
        key = self.key_k if which == "k" else self.key_v
        parts = [gen.normal_bf16_range(key, base, (z - a) * self.Hkv * self.D) for a, z, base in self.kv_runs(b, t0, t1)]
        flat = np.concatenate(parts) if parts else np.zeros(0, np.uint16)
        return flat.reshape(t1 - t0, self.Hkv, self.D)

    def kv_head_bits(self, which: str, b: int, kvh: int, t0: int, t1: int) -> np.ndarray:
        """[t1-t0][D] bf16 bits of one KV head (cheaper than kv_bits for long runs)."""
        key = self.key_k if which == "k" else self.key_v
        parts = [gen.normal_bf16_rows(key, base + kvh * self.D, z - a, self.D, self.Hkv * self.D)
                 for a, z, base in self.kv_runs(b, t0, t1)]
        return np.concatenate(parts) if parts else np.zeros((0, self.D), np.uint16)

    def spread_exponents(self, which: str, b: int, t0: int, t1: int, spread: int) -> np.ndarray:
        """int [t1-t0][Hkv]: a power-of-two exponent per (token, KV head), uniform
        in [-spread, spread], plus one per head in the same range."""
        key = gen.make_key(self.seed, gen.TENSOR_SPREAD) ^ (0 if which == "k" else 0x5bd1e995)
        t = np.arange(t0, t1, dtype=np.int64)
        tok = (self.src_request(b, t) << TOKEN_SHIFT) + t
        h = np.arange(self.Hkv, dtype=np.int64)
        e_tok = gen.uniform_int(key, (tok[:, None] * self.Hkv + h[None, :]).astype(np.uint64),
                                -spread, spread)
        e_head = gen.uniform_int(key ^ 0x27d4eb2f165667c5, h.astype(np.uint64) + (1 << 62),
                                 -spread, spread)
        return e_tok + e_head[None, :]

    def kv_spread_bits(self, which: str, b: int, t0: int, t1: int, spread: int = 6) -> np.ndarray:
        """kv_bits with every (token, KV head) row multiplied by 2^e
        (spread_exponents): magnitudes that differ between tokens and between
        heads, the case that finer scale granularity serves.  A power of two
        times a bf16 value is again an exact bf16 value."""
        x = gen.bf16_bits_to_f32(self.kv_bits(which, b, t0, t1))
        e = self.spread_exponents(which, b, t0, t1, spread)
        return gen.f32_to_bf16_bits(np.ldexp(x, e[:, :, None]).astype(np.float32))

    def q_bits(self) -> np.ndarray:
        n = self.B * self.Hq * self.D
        return gen.normal_bf16_range(self.key_q, 0, n).reshape(self.B, self.Hq, self.D)

    def q_new_bits(self, q_lens=None) -> np.ndarray:
        """[sum q_lens][Hq][D] bf16 bits: one query row per new token, request
        b's rows at positions L_b - q_lens[b] .. L_b - 1 (q_lens defaults to
        n_new for every request).  Row (b, position t) draws counters from its
        own run, so any subset of positions regenerates the same values."""
        q_lens = np.full(self.B, self.n_new) if q_lens is None else np.asarray(q_lens)
        rows = []
        for b in range(self.B):
            L = int(self.context_lens[b])
            for t in range(L - int(q_lens[b]), L):
                base = ((1 << 40) + (b << TOKEN_SHIFT) + t) * self.Hq * self.D
                rows.append(gen.normal_bf16_range(self.key_q, base, self.Hq * self.D))
        if not rows:
            return np.zeros((0, self.Hq, self.D), np.uint16)
        return np.stack(rows).reshape(-1, self.Hq, self.D)

    def q_start(self, q_lens=None) -> np.ndarray:
        q_lens = np.full(self.B, self.n_new) if q_lens is None else np.asarray(q_lens)
        return np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)

    # ----------------------------------------------------------------- slots
    def slots(self, b: int, t0: int, t1: int) -> np.ndarray:
        t = np.arange(t0, t1, dtype=np.int64)
        pages = self.block_tables[b, t // self.P].astype(np.int64)
        return pages * self.P + (t % self.P)

    def prefill_range(self, b: int):
        """Tokens written before the step (the shared prefix by request 0 only)."""
        t0 = self.shared_tokens if 0 < b < self.shared_requests else 0
        return t0, int(self.context_lens[b]) - self.n_new

    def new_range(self, b: int):
        L = int(self.context_lens[b])
        return L - self.n_new, L

    def step_slots(self) -> np.ndarray:
        return np.concatenate([self.slots(b, *self.new_range(b)) for b in range(self.B)])

    def step_kv_bits(self, which: str) -> np.ndarray:
        return np.concatenate([self.kv_bits(which, b, *self.new_range(b)) for b in range(self.B)])

    # ---------------------------------------------------------------- scales
    def host_amax(self, which: str) -> float:
        """max |x| over the whole bf16 tensor of the layer (every attended token)."""
        key = self.key_k if which == "k" else self.key_v
        m = 0
        for b in range(self.B):
            t0 = self.shared_tokens if 0 < b < self.shared_requests else 0
            for a, z, base in self.kv_runs(b, t0, int(self.context_lens[b])):
                bits = gen.normal_bf16_range(key, base, (z - a) * self.Hkv * self.D) & np.uint16(0x7FFF)
                if bits.size:
                    m = max(m, int(bits.max()))
        return amax_from_bits(m)

    def set_scales_host(self):
        self.k_scale = scale_from_amax(self.host_amax("k"))
        self.v_scale = scale_from_amax(self.host_amax("v"))
        return self

    # ----------------------------------------------------------------- bytes
    def kv_bytes(self, elem_bytes: int = 1) -> int:
        """Unique K+V bytes the step reads: 2 x KV heads x head_dim x tokens x bytes."""
        return 2 * self.Hkv * self.D * self.unique_tokens * elem_bytes

    def algorithmic_bytes(self, elem_bytes: int = 1) -> dict:
        q = self.B * self.Hq * self.D * 2
        o = self.B * self.Hq * self.D * 2
        tables = int(self.pages_per_req.sum()) * 4 + self.B * 4
        n_new = self.B * self.n_new
        append = n_new * self.Hkv * self.D * 2 * 2 + n_new * self.Hkv * self.D * 2 * elem_bytes + n_new * 8
        return {"kv": self.kv_bytes(elem_bytes), "q": q, "o": o, "tables": tables, "append": append,
                "total": self.kv_bytes(elem_bytes) + q + o + tables + append}


@dataclass
class MlaWorkload:
    """MLA absorbed-latent decode over one shared e4m3 latent per token."""

    name: str
    B: int
    H: int
    context_lens: np.ndarray
    topk_n: int = 0  # 0: attend every token
    d_latent: int = 512
    d_rope: int = 64
    P: int = 64
    n_new: int = 1
    num_pages: int | None = None
    seed: int = 0
    max_pages_per_seq: int | None = None
    ckv_scale: float | None = None
    softmax_scale: float = float(np.float32(1.0 / math.sqrt(192.0)))

    def __post_init__(self):
        self.context_lens = np.asarray(self.context_lens, dtype=np.int32)
        L = self.context_lens.astype(np.int64)
        self.pages_per_req = (L + self.P - 1) // self.P
        needed = int(self.pages_per_req.sum())
        if self.num_pages is None:
            self.num_pages = needed
        assert self.num_pages >= needed
        maxp = self.max_pages_per_seq or int(self.pages_per_req.max(initial=1))
        self.max_pages_per_seq = maxp
        perm = gen.permutation(gen.make_key(self.seed, gen.TENSOR_PERM), self.num_pages)
        bt = np.full((self.B, maxp), -1, dtype=np.int32)
        nxt = 0
        for b in range(self.B):
            n = int(self.pages_per_req[b])
            bt[b, :n] = perm[nxt:nxt + n]
            nxt += n
        self.block_tables = bt
        self.key_q = gen.make_key(self.seed, gen.TENSOR_QMLA)
        self.key_c = gen.make_key(self.seed, gen.TENSOR_CKV)
        if self.topk_n > 0:
            kt = gen.make_key(self.seed, gen.TENSOR_TOPK)
            self.topk = np.stack([gen.sample_sorted_unique(kt, b, int(self.context_lens[b]), self.topk_n)
                                  for b in range(self.B)]).astype(np.int32)
        else:
            self.topk = None

    @property
    def Dqk(self) -> int:
        return self.d_latent + self.d_rope

    @property
    def Dv(self) -> int:
        return self.d_latent

    def ckv_run_base(self, b: int, t0: int) -> int:
        return ((b << TOKEN_SHIFT) + t0) * self.Dqk

    def ckv_bits(self, b: int, t0: int, t1: int) -> np.ndarray:
        return gen.normal_bf16_range(self.key_c, self.ckv_run_base(b, t0), (t1 - t0) * self.Dqk).reshape(
            t1 - t0, 1, self.Dqk)

    def ckv_rows_bits(self, b: int, tokens: np.ndarray) -> np.ndarray:
        t = np.asarray(tokens, dtype=np.int64)
        idx = ((b << TOKEN_SHIFT) + t)[:, None] * self.Dqk + np.arange(self.Dqk)[None, :]
        return gen.normal_bf16(self.key_c, idx.reshape(-1).astype(np.uint64)).reshape(len(t), self.Dqk)

    def q_bits(self) -> np.ndarray:
        return gen.normal_bf16_range(self.key_q, 0, self.B * self.H * self.Dqk).reshape(self.B, self.H, self.Dqk)

    def slots(self, b: int, t0: int, t1: int) -> np.ndarray:
        t = np.arange(t0, t1, dtype=np.int64)
        return self.block_tables[b, t // self.P].astype(np.int64) * self.P + (t % self.P)

    def prefill_range(self, b: int):
        return 0, int(self.context_lens[b]) - self.n_new

    def new_range(self, b: int):
        L = int(self.context_lens[b])
        return L - self.n_new, L

    def step_slots(self) -> np.ndarray:
        return np.concatenate([self.slots(b, *self.new_range(b)) for b in range(self.B)])

    def step_ckv_bits(self) -> np.ndarray:
        return np.concatenate([self.ckv_bits(b, *self.new_range(b)) for b in range(self.B)])

    def host_amax(self) -> float:
        m = 0
        for b in range(self.B):
            bits = self.ckv_bits(b, 0, int(self.context_lens[b])) & np.uint16(0x7FFF)
            m = max(m, int(bits.max()))
        return amax_from_bits(m)

    def set_scales_host(self):
        self.ckv_scale = scale_from_amax(self.host_amax())
        return self

    def attended_tokens(self) -> int:
        if self.topk is None:
            return int(self.context_lens.astype(np.int64).sum())
        return int((self.topk >= 0).sum())

    def algorithmic_bytes(self) -> dict:
        rows = self.attended_tokens() * self.Dqk
        q = self.B * self.H * self.Dqk * 2
        o = self.B * self.H * self.Dv * 2
        topk = 0 if self.topk is None else self.topk.size * 4
        tables = self.B * self.max_pages_per_seq * 4 + self.B * 4
        append = self.B * self.n_new * (self.Dqk * 2 + self.Dqk + 8)
        return {"kv": rows, "q": q, "o": o, "topk": topk, "tables": tables, "append": append,
                "total": rows + q + o + topk + tables + append}

    def flops(self) -> int:
        return 2 * self.H * self.attended_tokens() * (self.Dqk + self.Dv)


# ------------------------------------------------------------------ workloads
def _lognormal_lens(seed: int, B: int, median: float, sigma: float, lo: int, hi: int) -> np.ndarray:
    z = gen.normal_f32(gen.make_key(seed, gen.TENSOR_CTX), np.arange(B, dtype=np.uint64)).astype(np.float64)
    L = np.rint(np.exp(math.log(median) + sigma * z)).astype(np.int64)
    return np.clip(L, lo, hi)


def workload(name: str, seed: int = 0):
    """One of the five workloads of the pages' shapes (WORKLOADS):
    tiny GQA (4 requests, 8/2 heads, contexts 16-300, a 128-page pool);
    MHA (32 requests x 48 heads x 8192 tokens, page 16);
    GQA with a shared prefix (64 requests, 64/8 heads, lognormal contexts, 16
    of them sharing 2048 prefix tokens); MLA (64 requests x 128 heads, latent
    576, top-k 2048 of 65536, page 64); long split-KV (8 requests of 256K-1M
    tokens, 64/8 heads, page 64, 8 new tokens each, 4096-token chunks)."""
    if name == TINY_GQA:
        L = gen.uniform_int(gen.make_key(seed, gen.TENSOR_CTX), np.arange(4, dtype=np.uint64), 16, 300)
        return PagedWorkload(name, B=4, Hq=8, Hkv=2, D=128, P=16, context_lens=L, n_new=1,
                             num_pages=128, seed=seed)
    if name == MHA_B32:
        return PagedWorkload(name, B=32, Hq=48, Hkv=48, D=128, P=16,
                             context_lens=np.full(32, 8192), n_new=1, seed=seed)
    if name == GQA_PREFIX:
        L = _lognormal_lens(seed, 64, 4096.0, 0.8, 256, 32768)
        L[:16] = np.maximum(L[:16], 2048 + 16)
        return PagedWorkload(name, B=64, Hq=64, Hkv=8, D=128, P=16, context_lens=L, n_new=1,
                             shared_requests=16, shared_tokens=2048, seed=seed)
    if name == MLA_TOPK:
        return MlaWorkload(name, B=64, H=128, context_lens=np.full(64, 65536), topk_n=2048,
                           P=64, n_new=1, seed=seed)
    if name == LONG_SPLITKV:
        L = np.array([262144, 393216, 524288, 655360, 786432, 917504, 1048576, 1048576])
        return PagedWorkload(name, B=8, Hq=64, Hkv=8, D=128, P=64, context_lens=L, n_new=8,
                             seed=seed, kv_split_tokens=4096)
    raise ValueError(f"unknown workload {name!r}; choose from {WORKLOADS}")
