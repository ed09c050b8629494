"""Pins of the oracle's quantised-KV functions (CPU only): E4M3 codes from
the format's definition and torch's float8_e4m3fn conversion, the row
quantiser, the append into quantised caches, and attention over quantised
rows against float64 attention over the dequantised rows.

Format read from "FlashMLA на Huawei Ascend" ("Ограничение по
деквантованию": the decode kernel reads FP8 KV and dequantises it to bf16;
"Оптимизация раскладки KV-кэша при decoding": a token's values and its scale
are stored side by side).  Scale granularity and encoding are not on the
page; the reading pinned here: one fp32 scale per row (absmax / 448) after
the row's E4M3 codes, rows padded to D + 16 bytes.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

FINITE = [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_e4m3_values_from_the_format():
    """1 sign, 4 exponent bits (bias 7), 3 mantissa bits; subnormals f * 2^-9;
    S.1111.111 is NaN; largest finite 448."""
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0x77: 240.0, 0xB8: -1.0,
             0xFE: -448.0}
    vals = oracle.e4m3_values(np.array(list(table), np.uint8))
    assert np.array_equal(vals, np.array(list(table.values())))
    nan = oracle.e4m3_values(np.array([0x7F, 0xFF], np.uint8))
    assert np.all(np.isnan(nan))
    neg0 = oracle.e4m3_values(np.array([0x80], np.uint8))
    assert neg0[0] == 0.0 and math.copysign(1.0, neg0[0]) < 0


def test_e4m3_values_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_values(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_e4m3_codes_round_trip_ties_and_saturation():
    codes = np.array(FINITE, np.uint8)
    vals = oracle.e4m3_values(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_codes(vals), codes)
    # midpoints between neighbouring positive codes go to the even code
    for c in range(0, 0x7E):
        lo, hi = oracle.e4m3_values(np.array([c, c + 1], np.uint8))
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        got = oracle.e4m3_codes(np.array([mid, -mid, np.nextafter(mid, np.float32(np.inf)),
                                          np.nextafter(mid, np.float32(0))], np.float32))
        assert list(got) == [even, even | 0x80, c + 1, c], (c, mid)
    big = np.array([448, 455, 463.9, 464, 470, 1e6, np.inf, -500, -np.inf], np.float32)
    assert list(oracle.e4m3_codes(big)) == [0x7E] * 7 + [0xFE] * 2
    assert oracle.e4m3_codes(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


def test_e4m3_codes_match_torch_rounding():
    g = torch.Generator().manual_seed(5)
    x = torch.cat([torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 140.0)])
    x = x.clamp(-460, 460)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_codes(x.numpy()), ref)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_rows(dtype):
    g = W.generator(21)
    x = W.randn(g, (3, 5, 64), dtype) * torch.tensor([1e-3, 1.0, 50.0]).view(3, 1, 1).to(dtype)
    x[1, 2] = 0
    rows = oracle.quantize_rows(x)
    assert rows.shape == (3, 5, 80) and rows.dtype == np.uint8
    xf = x.float().numpy()
    amax = np.abs(xf).max(-1)
    scale = rows[..., 64:68].copy().view("<f4")[..., 0]
    assert np.array_equal(scale, (amax / np.float32(448)).astype(np.float32))
    assert np.all(rows[..., 68:] == 0)
    assert np.all(rows[1, 2] == 0)
    # codes: torch's E4M3 conversion of the fp32 quotient v / scale
    nz = scale > 0
    q = torch.from_numpy(xf[nz] / scale[nz][:, None])
    assert np.array_equal(rows[..., :64][nz], q.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    # the absmax element lands on +-448 and the error is within half a step
    deq = oracle.dequantize_rows(rows)
    err = np.abs(deq - xf)
    step = np.maximum(2.0 ** np.floor(np.log2(np.maximum(np.abs(xf) / np.maximum(scale, 1e-45)[..., None], 2.0 ** -6))) / 8, 2.0 ** -9)
    assert np.all(err <= 0.5 * step * scale[..., None] * (1 + 1e-6) + 1e-30)


def test_append_fp8_writes_quantised_rows_only():
    g = W.generator(22)
    B, Hkv, C, D = 2, 3, 10, 64
    kc = np.random.default_rng(1).integers(0, 255, (B, Hkv, C, D + 16), dtype=np.uint8)
    vc = kc.copy()
    k0, v0 = kc.copy(), vc.copy()
    kn = W.randn(g, (B, Hkv, D), torch.bfloat16)
    vn = W.randn(g, (B, Hkv, D), torch.bfloat16)
    mask = np.zeros((B, C), np.uint8)
    assert oracle.append_fp8(kc, vc, kn, vn, torch.tensor([4, 9], dtype=torch.int32), mask) == 0
    qk, qv = oracle.quantize_rows(kn), oracle.quantize_rows(vn)
    for b, p in ((0, 4), (1, 9)):
        assert np.array_equal(kc[b, :, p], qk[b]) and np.array_equal(vc[b, :, p], qv[b])
        assert mask[b, p] == 1 and mask[b].sum() == 1
    keep = np.ones((B, Hkv, C), bool)
    keep[0, :, 4] = keep[1, :, 9] = False
    assert np.array_equal(kc[keep], k0[keep]) and np.array_equal(vc[keep], v0[keep])
    err = oracle.append_fp8(kc, vc, kn, vn, torch.tensor([10, -1], dtype=torch.int32), mask)
    assert err == oracle.ERR_POS


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 64), (4, 4, 128)])
def test_attention_over_quantised_rows(Hq, Hkv, D):
    """Equals float64 softmax attention (torch) over the dequantised rows;
    for rows whose values are already E4M3 multiples of a power-of-two scale,
    equals attention over the unquantised cache."""
    g = W.generator(23 + D)
    B, C = 2, 45
    q = W.randn(g, (B, Hq, D), torch.bfloat16)
    k = W.randn(g, (B, Hkv, C, D), torch.bfloat16)
    v = W.randn(g, (B, Hkv, C, D), torch.bfloat16)
    mask = W.prefix_mask([45, 17], C)
    mask[0, 3] = 0
    kr, vr = oracle.quantize_rows(k), oracle.quantize_rows(v)
    out, lse = oracle.attend_masked_fp8(q, kr, vr, mask, 0.125)
    kd = torch.from_numpy(oracle.dequantize_rows(kr)).repeat_interleave(Hq // Hkv, 1)
    vd = torch.from_numpy(oracle.dequantize_rows(vr)).repeat_interleave(Hq // Hkv, 1)
    s = torch.einsum("bhd,bhtd->bht", q.double(), kd) * 0.125
    s = s.masked_fill((mask == 0).view(B, 1, C), float("-inf"))
    ref = torch.einsum("bht,bhtd->bhd", torch.softmax(s, -1), vd)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=1e-12, atol=1e-12)
    # exactly representable rows: codes times 2^-5 with the row's max code 448
    codes = torch.randint(0, 0x7E, (B, Hkv, C, D), generator=g).to(torch.uint8)
    codes = codes | (torch.randint(0, 2, codes.shape, generator=g).to(torch.uint8) << 7)
    codes[..., 0] = 0x7E
    exact = (torch.from_numpy(oracle.e4m3_values(codes.numpy())) * 2.0 ** -5).float()
    er = oracle.quantize_rows(exact)
    assert np.array_equal(er[..., :D], codes.numpy())
    o1, l1 = oracle.attend_masked_fp8(q, er, er, mask, 0.125)
    o2, l2 = oracle.attend_masked(q.float(), exact, exact, mask, 0.125)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)
