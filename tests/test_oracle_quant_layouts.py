"""Pins of the oracle's quantised rows in the paged layout and through index
lists (CPU only).  The row format is the static buffer's (E4M3 or E2M1 codes,
then an fp32 scale in a 16-byte field; "FlashMLA на Huawei Ascend",
"Оптимизация раскладки KV-кэша при decoding" places a token's values and
scale side by side, on paged KV blocks), so each layout is pinned against
the static-buffer functions over the same rows laid out another way, and
against float64 softmax over the dequantised rows written out here."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

FMTS = {"fp8": (W.fp8_rows, oracle.attend_masked_fp8, oracle.dequantize_rows, 1),
        "fp4": (W.fp4_rows, oracle.attend_masked_fp4, oracle.dequantize_rows_fp4, 2)}


def _rows(fmt, g, shape, D):
    return FMTS[fmt][0](g, shape, D).numpy()


def _paged_from_static(static, lengths, BS, NB, g):
    """Lay the rows of a static buffer [B, Hkv, C, RB] out as a paged cache
    [NB, BS, Hkv, RB] behind permuted block tables; unused blocks hold other
    random bytes."""
    B, Hkv, C, RB = static.shape
    cols = (C + BS - 1) // BS
    bt = W.permuted_block_tables(g, B, cols, NB)
    paged = np.random.default_rng(5).integers(0, 256, (NB, BS, Hkv, RB), dtype=np.uint8)
    for b in range(B):
        for t in range(int(lengths[b])):
            paged[int(bt[b, t // BS]), t % BS] = static[b, :, t]
    return paged, bt


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
def test_paged_quant_attention_is_the_static_attention_of_the_same_rows(fmt):
    g = W.generator(41)
    B, Hq, Hkv, C, D, BS, NB = 3, 8, 2, 200, 64, 16, 64
    lengths = [200, 1, 77]
    q = W.randn(g, (B, Hq, D), torch.bfloat16)
    k = _rows(fmt, g, (B, Hkv, C), D)
    v = _rows(fmt, g, (B, Hkv, C), D)
    kp, bt = _paged_from_static(k, lengths, BS, NB, g)
    vp = np.ascontiguousarray(kp.copy())
    for b in range(B):
        for t in range(lengths[b]):
            vp[int(bt[b, t // BS]), t % BS] = v[b, :, t]
    sl = W.cumsum_lengths(lengths)
    out, lse = oracle.attend_paged_quant(q, kp, vp, bt, sl, None, 0.125, fmt)
    ref, ref_lse = FMTS[fmt][1](q, k, v, W.prefix_mask(lengths, C), 0.125)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13, atol=1e-13)
    # and against float64 softmax over the dequantised rows
    deq = FMTS[fmt][2]
    for b in range(B):
        kd = torch.from_numpy(deq(k[b, :, :lengths[b]]))
        vd = torch.from_numpy(deq(v[b, :, :lengths[b]]))
        for h in range(Hq):
            s = kd[h // (Hq // Hkv)] @ q[b, h].double() * 0.125
            np.testing.assert_allclose(out[b, h], (torch.softmax(s, 0) @ vd[h // (Hq // Hkv)]).numpy(),
                                       rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
def test_paged_quant_attention_with_offsets_and_errors(fmt):
    """seq_offset selects the first table column; an empty sequence gives
    zeros and -inf; an invalid table is refused (no result defined)."""
    g = W.generator(43)
    Hq, Hkv, D, BS, NB = 4, 4, 64, 8, 32
    q = W.randn(g, (2, Hq, D), torch.bfloat16)
    kp = _rows(fmt, g, (NB, BS, Hkv), D)
    vp = _rows(fmt, g, (NB, BS, Hkv), D)
    bt = torch.tensor([[5, 9, 2, 7], [11, 3, 4, 1]], dtype=torch.int32)
    sl = W.cumsum_lengths([10, 0])
    off = torch.tensor([8, 0], dtype=torch.int32)
    out, lse = oracle.attend_paged_quant(q, kp, vp, bt, sl, off, 0.2, fmt)
    # sequence 0 reads columns 1.. (blocks 9 and 2): 8 + 2 rows
    rows_k = np.concatenate([kp[9], kp[2][:2]]).transpose(1, 0, 2)[None]
    rows_v = np.concatenate([vp[9], vp[2][:2]]).transpose(1, 0, 2)[None]
    ref, ref_lse = FMTS[fmt][1](q[:1], np.ascontiguousarray(rows_k), np.ascontiguousarray(rows_v),
                                np.ones((1, 10), np.uint8), 0.2)
    assert np.array_equal(out[:1], ref) and np.array_equal(lse[:1], ref_lse)
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    bad = bt.clone()
    bad[0, 1] = NB
    with pytest.raises(ValueError):
        oracle.attend_paged_quant(q, kp, vp, bad, sl, off, 0.2, fmt)


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
def test_paged_quant_append_writes_the_quantised_row_where_the_gather_reads(fmt):
    g = W.generator(47)
    Q, Hkv, D, BS, NB, cols = 3, 2, 128, 16, 40, 4
    kp = _rows(fmt, g, (NB, BS, Hkv), D)
    vp = _rows(fmt, g, (NB, BS, Hkv), D)
    bt = W.permuted_block_tables(g, Q, cols, NB)
    kn = W.randn(g, (Q, Hkv, D), torch.bfloat16)
    vn = W.randn(g, (Q, Hkv, D), torch.bfloat16)
    pos = torch.tensor([0, 17, 63], dtype=torch.int32)
    k0, v0 = kp.copy(), vp.copy()
    assert oracle.append_paged_quant(kp, vp, bt, None, kn, vn, pos, fmt) == 0
    quant = oracle.quantize_rows if fmt == "fp8" else oracle.quantize_rows_fp4
    changed = np.zeros(kp.shape[:2], bool)
    for s in range(Q):
        t = int(pos[s])
        blk, slot = int(bt[s, t // BS]), t % BS
        assert np.array_equal(kp[blk, slot], quant(kn[s]))
        assert np.array_equal(vp[blk, slot], quant(vn[s]))
        changed[blk, slot] = True
    assert np.array_equal(kp[~changed], k0[~changed]) and np.array_equal(vp[~changed], v0[~changed])
    # the same bytes as the static buffer's quantising append
    sk = np.zeros((Q, Hkv, 64, kp.shape[-1]), np.uint8)
    sv = sk.copy()
    append = oracle.append_fp8 if fmt == "fp8" else oracle.append_fp4
    assert append(sk, sv, kn, vn, pos, None) == 0
    for s in range(Q):
        t = int(pos[s])
        assert np.array_equal(sk[s, :, t], kp[int(bt[s, t // BS]), t % BS])
    bad = torch.tensor([0, -1, 64], dtype=torch.int32)  # -1: position; 64: beyond the columns
    assert oracle.append_paged_quant(kp, vp, bt, None, kn, vn, bad, fmt) == oracle.ERR_POS | oracle.ERR_COLS


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
def test_indexed_quant_attention(fmt):
    """The listed rows as softmax terms: the prefix list equals the static
    attention with the prefix mask; a permuted list the same up to the
    summation order; a repeated entry counts twice; entries outside [-1, C)
    are reported and skipped; a list of -1 gives zeros and -inf."""
    g = W.generator(53)
    B, Hq, Hkv, C, D = 2, 8, 2, 96, 128
    q = W.randn(g, (B, Hq, D), torch.bfloat16)
    k = _rows(fmt, g, (B, Hkv, C), D)
    v = _rows(fmt, g, (B, Hkv, C), D)
    attend = FMTS[fmt][1]
    L = [96, 40]
    idx = torch.full((B, 100), -1, dtype=torch.int32)
    for b in range(B):
        idx[b, :L[b]] = torch.arange(L[b], dtype=torch.int32)
    out, lse, err = oracle.attend_indexed_quant(q, k, v, idx, 0.1, fmt)
    ref, ref_lse = attend(q, k, v, W.prefix_mask(L, C), 0.1)
    assert err == 0 and np.array_equal(out, ref) and np.array_equal(lse, ref_lse)
    perm = idx[:, torch.randperm(100, generator=g)]
    po, pl, _ = oracle.attend_indexed_quant(q, k, v, perm, 0.1, fmt)
    np.testing.assert_allclose(po, out, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(pl, lse, rtol=1e-13, atol=1e-13)
    rep = torch.tensor([[3, 3, -1], [7, 5, 5]], dtype=torch.int32)
    ro, rl, _ = oracle.attend_indexed_quant(q, k, v, rep, 0.1, fmt)
    # three-slot buffers holding the listed rows: 3, 3 (and a masked slot); 7, 5, 5
    k3 = np.ascontiguousarray(np.stack([k[0][:, [3, 3, 0]], k[1][:, [7, 5, 5]]]))
    v3 = np.ascontiguousarray(np.stack([v[0][:, [3, 3, 0]], v[1][:, [7, 5, 5]]]))
    m3 = np.array([[1, 1, 0], [1, 1, 1]], np.uint8)
    eo, el = attend(q, k3, v3, m3, 0.1)
    assert k3.shape == (B, Hkv, 3, k.shape[-1])
    assert np.array_equal(ro, eo) and np.array_equal(rl, el)
    bad = torch.tensor([[3, C, -1], [-2, 5, 5]], dtype=torch.int32)
    bo, bl, berr = oracle.attend_indexed_quant(q, k, v, bad, 0.1, fmt)
    assert berr == oracle.ERR_POS
    m3b = np.array([[1, 0, 0], [0, 1, 1]], np.uint8)
    eo, el = attend(q, k3, v3, m3b, 0.1)
    assert np.array_equal(bo[1], eo[1])
    none, nl, _ = oracle.attend_indexed_quant(q, k, v, torch.full((B, 4), -1, dtype=torch.int32), 0.1, fmt)
    assert np.all(none == 0) and np.all(np.isneginf(nl))
