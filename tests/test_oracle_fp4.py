"""Pins of the oracle's FP4 KV functions (CPU only): E2M1 codes against the
format's value table and a brute-force nearest search, the row quantiser
and its nibble order, the append into FP4 caches, and attention over FP4
rows against float64 attention over the dequantised rows.

Format read from "FlashMLA на Huawei Ascend" ("Ограничение по
деквантованию": decoding reads the KV cache in FP8 or FP4 and dequantises it
for the matrix unit; "Оптимизация раскладки KV-кэша при decoding": a token's
values and its scale side by side).  Code layout and scale are not on the
page; the reading pinned here: OCP E2M1 codes, two per byte with element 2j
in the low nibble of byte j, then the row's fp32 scale (absmax / 6), rows
padded to D/2 + 16 bytes.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

# OCP E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit): the eight
# magnitudes of codes 0..7, the same negated for codes 8..15.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_values_from_the_format():
    vals = oracle.e2m1_values(np.arange(16, dtype=np.uint8))
    assert np.array_equal(vals[:8], E2M1_MAGNITUDES)
    assert np.array_equal(vals[8:], [-m for m in E2M1_MAGNITUDES])
    assert math.copysign(1.0, vals[8]) < 0  # code 8 is -0


def _nearest_even(x):
    """Brute force: the E2M1 code nearest to x, ties to the even code (the
    one whose mantissa bit is 0), magnitudes past 6 saturating, NaN -> +6."""
    out = []
    for v in np.asarray(x, np.float64):
        if math.isnan(v):
            out.append(7)
            continue
        a = min(abs(v), 6.0)
        d = [abs(a - m) for m in E2M1_MAGNITUDES]
        best = min(d)
        cands = [i for i in range(8) if d[i] == best]
        i = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        out.append(i | (8 if math.copysign(1.0, v) < 0 else 0))
    return np.array(out, np.uint8)


def test_e2m1_codes_round_trip_ties_and_saturation():
    vals = oracle.e2m1_values(np.arange(16, dtype=np.uint8)).astype(np.float32)
    assert np.array_equal(oracle.e2m1_codes(vals), np.arange(16, dtype=np.uint8))
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    assert oracle.e2m1_codes(mids).tolist() == [0, 2, 2, 4, 4, 6, 6]  # each tie to the even code
    assert oracle.e2m1_codes(-mids).tolist() == [8, 10, 10, 12, 12, 14, 14]
    big = np.array([6.0, 6.5, 100.0, np.inf, -7.0, -np.inf, np.nan], np.float32)
    assert oracle.e2m1_codes(big).tolist() == [7, 7, 7, 7, 15, 15, 7]


def test_e2m1_codes_match_a_brute_force_search():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(-8, 8, 50000), rng.standard_normal(50000) * 2,
                        np.array(E2M1_MAGNITUDES) + 1e-7, np.array(E2M1_MAGNITUDES) - 1e-7,
                        [-0.0, 0.0, 1e-30, -1e-30]]).astype(np.float32)
    assert np.array_equal(oracle.e2m1_codes(x), _nearest_even(x))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_rows_fp4(dtype):
    g = W.generator(31)
    x = W.randn(g, (3, 5, 64), dtype) * torch.tensor([1e-3, 1.0, 50.0]).view(3, 1, 1).to(dtype)
    x[1, 2] = 0
    rows = oracle.quantize_rows_fp4(x)
    assert rows.shape == (3, 5, 48) and rows.dtype == np.uint8
    xf = x.float().numpy()
    amax = np.abs(xf).max(-1)
    scale = rows[..., 32:36].copy().view("<f4")[..., 0]
    assert np.array_equal(scale, (amax / np.float32(6)).astype(np.float32))
    assert np.all(rows[..., 36:] == 0)
    assert np.all(rows[1, 2] == 0)
    # codes: element 2j in the low nibble of byte j, each the nearest code of
    # the fp32 quotient v / scale
    nz = scale > 0
    quot = (xf[nz] / scale[nz][:, None]).astype(np.float32)
    codes = _nearest_even(quot.reshape(-1)).reshape(quot.shape)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(rows[..., :32][nz], packed)
    # the absmax element lands on +-6; the error is within half a spacing
    deq = oracle.dequantize_rows_fp4(rows)
    assert np.all(np.abs(deq).max(-1)[nz] == pytest.approx(6 * scale[nz], rel=1e-7))
    err = np.abs(deq - xf)
    assert np.all(err <= 1.0 * scale[..., None] * (1 + 1e-6) + 1e-30)  # spacing <= 2 near 6


def test_nibble_order():
    x = torch.zeros(1, 8)
    x[0, 0] = 6.0   # code 7 in the low nibble of byte 0
    x[0, 3] = -3.0  # code 13 in the high nibble of byte 1
    rows = oracle.quantize_rows_fp4(x)
    assert rows[0, 0] == 0x07 and rows[0, 1] == 0xD0 and rows[0, 2] == 0 and rows[0, 3] == 0


def test_append_fp4_writes_quantised_rows_only():
    g = W.generator(32)
    B, Hkv, C, D = 2, 3, 10, 64
    kc = np.random.default_rng(1).integers(0, 255, (B, Hkv, C, D // 2 + 16), dtype=np.uint8)
    vc = kc.copy()
    k0, v0 = kc.copy(), vc.copy()
    kn = W.randn(g, (B, Hkv, D), torch.bfloat16)
    vn = W.randn(g, (B, Hkv, D), torch.bfloat16)
    mask = np.zeros((B, C), np.uint8)
    assert oracle.append_fp4(kc, vc, kn, vn, torch.tensor([4, 9], dtype=torch.int32), mask) == 0
    qk, qv = oracle.quantize_rows_fp4(kn), oracle.quantize_rows_fp4(vn)
    for b, p in ((0, 4), (1, 9)):
        assert np.array_equal(kc[b, :, p], qk[b]) and np.array_equal(vc[b, :, p], qv[b])
        assert mask[b, p] == 1 and mask[b].sum() == 1
    keep = np.ones((B, Hkv, C), bool)
    keep[0, :, 4] = keep[1, :, 9] = False
    assert np.array_equal(kc[keep], k0[keep]) and np.array_equal(vc[keep], v0[keep])
    assert oracle.append_fp4(kc, vc, kn, vn, torch.tensor([10, -1], dtype=torch.int32),
                             mask) == oracle.ERR_POS


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 64), (4, 4, 128)])
def test_attention_over_fp4_rows(Hq, Hkv, D):
    """Equals float64 softmax attention (torch) over the dequantised rows;
    for rows whose values are E2M1 values times the row's scale, equals
    attention over the unquantised cache."""
    g = W.generator(33 + D)
    B, C = 2, 45
    q = W.randn(g, (B, Hq, D), torch.bfloat16)
    k = W.randn(g, (B, Hkv, C, D), torch.bfloat16)
    v = W.randn(g, (B, Hkv, C, D), torch.bfloat16)
    mask = W.prefix_mask([45, 17], C)
    mask[0, 3] = 0
    kr, vr = oracle.quantize_rows_fp4(k), oracle.quantize_rows_fp4(v)
    out, lse = oracle.attend_masked_fp4(q, kr, vr, mask, 0.125)
    kd = torch.from_numpy(oracle.dequantize_rows_fp4(kr)).repeat_interleave(Hq // Hkv, 1)
    vd = torch.from_numpy(oracle.dequantize_rows_fp4(vr)).repeat_interleave(Hq // Hkv, 1)
    s = torch.einsum("bhd,bhtd->bht", q.double(), kd) * 0.125
    s = s.masked_fill((mask == 0).view(B, 1, C), float("-inf"))
    ref = torch.einsum("bht,bhtd->bhd", torch.softmax(s, -1), vd)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=1e-12, atol=1e-12)
    # exactly representable rows: E2M1 values times 2^-3, each row's max code 6
    codes = torch.randint(0, 16, (B, Hkv, C, D), generator=g).to(torch.uint8)
    codes[..., 0] = 7
    exact = (torch.from_numpy(oracle.e2m1_values(codes.numpy())) * 2.0 ** -3).float()
    er = oracle.quantize_rows_fp4(exact)
    deq = oracle.dequantize_rows_fp4(er)
    assert np.array_equal(deq, exact.double().numpy())
    o1, l1 = oracle.attend_masked_fp4(q, er, er, mask, 0.125)
    o2, l2 = oracle.attend_masked(q.float(), exact, exact, mask, 0.125)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)
