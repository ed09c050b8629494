"""GPU parity of the FP4 KV path (kvd_append_fp4, kvd_attend_masked_fp4)
against the fp64 oracle, through the C ABI.  Quantisation is integer work
(E2M1 codes, nibble order and scale bytes): bit-exact.  Attention: the bf16
tolerance."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity_util import assert_attention_close, assert_lse_close, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvd():
    from decode_attention_kv_gb300 import kvd as _kvd
    _kvd.load()
    return _kvd


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [64, 128])
def test_append_fp4_bit_exact(kvd, dtype, D):
    """New rows spanning 1e-6 .. 1e4 in magnitude, a zero row, every E2M1
    rounding boundary hit exactly (ties go to the even code) with both signs
    and -0; caches pre-filled with random bytes; positions incl. the last
    slot."""
    g = W.generator(900 + D)
    B, Hkv, C = 5, 3, 40
    RB = D // 2 + 16
    kc = torch.randint(0, 256, (B, Hkv, C, RB), generator=g, dtype=torch.uint8)
    vc = torch.randint(0, 256, (B, Hkv, C, RB), generator=g, dtype=torch.uint8)
    mag = torch.tensor([1e-6, 1e-2, 1.0, 30.0, 1e4]).view(B, 1, 1)
    kn = (W.randn(g, (B, Hkv, D), torch.float32) * mag).to(dtype)
    vn = (W.randn(g, (B, Hkv, D), torch.float32) * mag).to(dtype)
    kn[2, 1] = 0
    # amax 6 -> scale 1: x / scale is x itself; the midpoints between
    # neighbouring magnitudes, just either side of two of them, and -0
    ties = [6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -2.5, -5, -0.0, 0.2500001,
            1.7499999, 4.9999]
    vn[3, 0, :len(ties)] = torch.tensor(ties, dtype=torch.float32).to(dtype)
    vn[3, 0, len(ties):] = 0.1
    pos = torch.tensor([0, 7, 39, 12, 3], dtype=torch.int32)
    mask = torch.zeros(B, C, dtype=torch.uint8)
    kh, vh, mh = kc.numpy().copy(), vc.numpy().copy(), mask.numpy().copy()
    assert oracle.append_fp4(kh, vh, kn, vn, pos, mh) == 0
    kd, vd, md = kc.cuda(), vc.cuda(), mask.cuda()
    status = kvd.status_tensor()
    kvd.append_fp4(kd, vd, kn.cuda(), vn.cuda(), pos.cuda(), md, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(host(kd).numpy(), kh)
    assert np.array_equal(host(vd).numpy(), vh)
    assert np.array_equal(host(md).numpy(), mh)
    # the tie row's codes, read back: the even neighbour on every midpoint
    row = host(vd)[3, 0, 12].numpy()
    codes = [(row[d // 2] >> (4 * (d % 2))) & 0xF for d in range(len(ties))]
    assert codes[:8] == [0x7, 0x0, 0x2, 0x2, 0x4, 0x4, 0x6, 0x6]
    assert codes[8:13] == [0x8, 0xA, 0xC, 0xE, 0x8]
    # a position outside [0, C) writes nothing for its entry and is reported
    before = host(kd).clone()
    kvd.append_fp4(kd, vd, kn.cuda(), vn.cuda(),
                   torch.tensor([40, -1, 5, 5, 5], dtype=torch.int32, device="cuda"), None, status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    after = host(kd)
    assert torch.equal(after[:2], before[:2])


CASES = [
    # B, Hq, Hkv, C, D, lengths, num_splits
    (2, 32, 8, 3000, 128, [3000, 1001], 0),     # 4 heads per kv head
    (3, 8, 8, 700, 128, [700, 65, 1], 0),       # one head per kv head
    (2, 16, 8, 900, 64, [900, 300], 3),         # two, head_dim 64
    (1, 16, 2, 2100, 128, [2099], 0),           # eight
    (2, 48, 3, 640, 64, [640, 129], 0),         # sixteen: two head groups
    (1, 4, 4, 4096, 128, [4096], 1),            # one split
    (2, 32, 8, 9000, 64, [9000, 4097], 0),      # split kernel + combine, head_dim 64
]


@pytest.mark.parametrize("B,Hq,Hkv,C,D,lengths,num_splits", CASES)
def test_attend_fp4_parity(kvd, B, Hq, Hkv, C, D, lengths, num_splits):
    g = W.generator(1600 + C + Hq)
    q = W.randn(g, (B, Hq, D), torch.bfloat16)
    k = W.fp4_rows(g, (B, Hkv, C), D)
    v = W.fp4_rows(g, (B, Hkv, C), D)
    mask = W.prefix_mask(lengths, C)
    scale = 1.0 / math.sqrt(D)
    status = kvd.status_tensor()
    lse = torch.empty(B, Hq, device="cuda")
    out = kvd.attend_masked_fp4(q.cuda(), k.cuda(), v.cuda(), mask.cuda(), scale, lse=lse,
                                num_splits=num_splits, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse = oracle.attend_masked_fp4(q, k, v, mask, scale)
    assert_attention_close(out, ref, torch.bfloat16, "fp4")
    assert_lse_close(lse, ref_lse, "fp4 lse")


def test_fp4_plan_matches_fp8_plan(kvd):
    """The two row formats share the planner: same splits, launches and
    workspace for the same sizes (only the one-launch path's shared memory
    differs, and both fit it here)."""
    for args in ((16, 32, 8, 8192, 128), (1, 32, 32, 1152, 128), (4, 8, 8, 700, 64)):
        a, b = kvd.attend_masked_fp4_plan(*args), kvd.attend_masked_fp8_plan(*args)
        assert (a.splits, a.launches) == (b.splits, b.launches)
        assert kvd.attend_masked_fp4_workspace_bytes(*args) == \
            kvd.attend_masked_fp8_workspace_bytes(*args)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 8)])
def test_fp4_bad_scales_and_codes_in_padding_are_ignored(kvd, Hq, Hkv):
    """NaN / inf scales and arbitrary codes in mask = 0 rows leave the result
    bit-identical to zero padding; sparse masks leave whole tiles out."""
    B, C, D = 2, 500, 128
    g = W.generator(1700 + Hq)
    q = W.randn(g, (B, Hq, D), torch.bfloat16)
    k = W.fp4_rows(g, (B, Hkv, C), D)
    v = W.fp4_rows(g, (B, Hkv, C), D)
    mask = W.prefix_mask([480, 37], C)
    mask[0, 5] = 0
    mask[0, 100:260] = 0
    pad = (mask == 0).view(B, 1, C).expand(B, Hkv, C)
    k0, v0 = k.clone(), v.clone()
    k0[pad] = 0
    v0[pad] = 0
    k1, v1 = k.clone(), v.clone()
    k1[pad] = 0x77
    v1[pad] = 0xFF
    nan = torch.tensor([float("nan")], dtype=torch.float32).view(torch.uint8)
    inf = torch.tensor([float("inf")], dtype=torch.float32).view(torch.uint8)
    k1[..., D // 2:D // 2 + 4][pad] = nan
    v1[..., D // 2:D // 2 + 4][pad] = inf
    outs = []
    for kk, vv in ((k0, v0), (k1, v1)):
        lse = torch.empty(B, Hq, device="cuda")
        o = kvd.attend_masked_fp4(q.cuda(), kk.cuda(), vv.cuda(), mask.cuda(), 0.09, lse=lse)
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    ref, ref_lse = oracle.attend_masked_fp4(q, k0, v0, mask, 0.09)
    assert_attention_close(outs[1][0], ref, torch.bfloat16, "fp4 padding")
    assert_lse_close(outs[1][1], ref_lse)


def test_fp4_decode_steps_end_to_end(kvd):
    """Three decode steps: append_fp4 of bf16 rows then attention, GPU vs
    oracle on its own copy of the caches (bytes equal after every step)."""
    g = W.generator(1800)
    B, Hq, Hkv, C, D = 2, 16, 4, 300, 128
    k = torch.zeros(B, Hkv, C, D // 2 + 16, dtype=torch.uint8)
    v = torch.zeros_like(k)
    prompt = W.randn(g, (2, B, Hkv, 100, D), torch.bfloat16)
    k[:, :, :100] = torch.from_numpy(oracle.quantize_rows_fp4(prompt[0]))
    v[:, :, :100] = torch.from_numpy(oracle.quantize_rows_fp4(prompt[1]))
    mask = W.prefix_mask([100, 100], C)
    kh, vh, mh = k.numpy().copy(), v.numpy().copy(), mask.numpy().copy()
    kd, vd, md = k.cuda(), v.cuda(), mask.cuda()
    status = kvd.status_tensor()
    for step in range(3):
        q = W.randn(g, (B, Hq, D), torch.bfloat16)
        kn = W.randn(g, (B, Hkv, D), torch.bfloat16)
        vn = W.randn(g, (B, Hkv, D), torch.bfloat16)
        pos = torch.tensor([100 + step, 100 + step], dtype=torch.int32)
        assert oracle.append_fp4(kh, vh, kn, vn, pos, mh) == 0
        kvd.append_fp4(kd, vd, kn.cuda(), vn.cuda(), pos.cuda(), md, status)
        out = kvd.attend_masked_fp4(q.cuda(), kd, vd, md, 1 / math.sqrt(D), dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(host(kd).numpy(), kh) and np.array_equal(host(vd).numpy(), vh)
        ref, _ = oracle.attend_masked_fp4(q, torch.from_numpy(kh), torch.from_numpy(vh),
                                          torch.from_numpy(mh), 1 / math.sqrt(D))
        assert_attention_close(out, ref, torch.bfloat16, f"fp4 step {step}")


def test_gqa_fp4_full_size(kvd):
    """The benchmark's FP4 batched-GQA configuration (16 x 32/8 heads,
    capacity 8192, lengths 512..8192): append + attend, the caches byte for
    byte and every entry and head of the output compared."""
    lay = W.gqa_fp4(device="cuda", layers=1).layers[0]
    kh, vh, mh = host(lay.k_cache).numpy().copy(), host(lay.v_cache).numpy().copy(), \
        host(lay.mask).numpy().copy()
    status = kvd.status_tensor()
    kvd.append_fp4(lay.k_cache, lay.v_cache, lay.k_new, lay.v_new, lay.pos, lay.mask, status)
    lse = torch.empty(16, 32, device="cuda")
    out = kvd.attend_masked_fp4(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.scale, lse=lse,
                                dev_status=status)
    assert oracle.append_fp4(kh, vh, host(lay.k_new), host(lay.v_new), host(lay.pos), mh) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(host(lay.k_cache).numpy(), kh)
    assert np.array_equal(host(lay.v_cache).numpy(), vh)
    assert np.array_equal(host(lay.mask).numpy(), mh)
    ref, rl = oracle.attend_masked_fp4(host(lay.q), kh, vh, mh, lay.scale)
    assert_attention_close(out, ref, torch.bfloat16, "gqa_fp4, all entries")
    assert_lse_close(lse, rl, "gqa_fp4 lse")
