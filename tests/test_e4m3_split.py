"""The few-row multi-query kernel feeds its score products e4m3 K rows and Q
split into two e4m3 parts (x = q s with s a power of two taking the row's
largest |q| into (224, 448]; part 1 = e4m3(x), part 2 = e4m3(x - part 1)).
Checked here over every positive bf16 value with torch's round-to-nearest
e4m3 cast: the split is exact above 0.25, and below it the error is at most
half e4m3's subnormal step (2^-10)."""
import numpy as np
import torch


def _split(x):
    p1 = x.to(torch.float8_e4m3fn).to(torch.float32)
    p2 = (x - p1).to(torch.float8_e4m3fn).to(torch.float32)
    return p1, p2


def test_two_e4m3_parts_reproduce_every_bf16_value():
    bits = np.arange(1, 0x7F80, dtype=np.int32).astype(np.int16)  # every finite positive bf16
    x = torch.from_numpy(bits).view(torch.bfloat16).to(torch.float32)
    x = x[x <= 448.0]
    p1, p2 = _split(x)
    err = (p1 + p2 - x).abs()
    big = x > 0.25
    assert int(big.sum()) == 1376  # 128 per binade over (0.25, 448]
    assert torch.equal(p1[big] + p2[big], x[big])
    assert float(err.max()) <= 2.0 ** -10
    # the sign is symmetric
    n1, n2 = _split(-x)
    assert torch.equal(n1, -p1) and torch.equal(n2, -p2)


def test_power_of_two_scale_keeps_bf16_values_exact():
    # the row scale is 2^floor(log2(448 / max|q|)): scaled values stay bf16-exact and
    # the largest lands in (224, 448]
    rng = np.random.default_rng(3)
    q = torch.from_numpy(rng.standard_normal((64, 128)).astype(np.float32)).to(torch.bfloat16).to(torch.float32)
    amax = q.abs().amax(dim=1)
    s = torch.exp2(torch.floor(torch.log2(448.0 / amax)))
    x = q * s[:, None]
    assert torch.equal(x.to(torch.bfloat16).to(torch.float32), x)
    top = x.abs().amax(dim=1)
    assert bool(((top > 224) & (top <= 448)).all())
    p1, p2 = _split(x)
    assert float((p1 + p2 - x).abs().max()) <= 2.0 ** -10
