"""GPU parity of quantised K/V rows (E4M3 and E2M1 codes with a per-row fp32
scale; "FlashMLA на Huawei Ascend", "Оптимизация раскладки KV-кэша при
decoding": a token's values and scale side by side, on paged KV blocks) in
the paged layout and through index lists, against the fp64 oracle: the
quantising paged append byte for byte, paged and index-list attention to
the bf16 bar, and the device status bits of bad tables, positions and
entries."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity_util import assert_attention_close, assert_lse_close, host

pytestmark = pytest.mark.gpu

ROWS = {"fp8": W.fp8_rows, "fp4": W.fp4_rows}


@pytest.fixture(scope="module")
def kvd():
    from decode_attention_kv_gb300 import kvd as _kvd
    _kvd.load()
    return _kvd


def _poison(rows, fmt, sel):
    """NaN codes (E4M3) / arbitrary codes (E2M1) and a NaN scale in the rows
    picked by `sel` (rows that no valid token reads)."""
    D = rows.shape[-1] - 16 if fmt == "fp8" else 2 * (rows.shape[-1] - 16)
    cb = D if fmt == "fp8" else D // 2
    rows[sel, ..., :cb] = 0x7F
    nan = torch.tensor([float("nan")], dtype=torch.float32).view(torch.uint8)
    rows[sel, ..., cb:cb + 4] = nan


PCASES = [
    # Q, Hq, Hkv, BS, cols, D, lengths, offsets, num_splits
    (5, 32, 8, 128, 8, 128, [1, 100, 1000, 129, 0], None, 0),   # tensor-core G = 4, ragged
    (3, 16, 16, 16, 20, 64, [320, 17, 200], None, 0),           # one head per kv head, 16-row tiles
    (2, 8, 4, 64, 6, 128, [250, 64], [64, 128], 0),             # G = 2, offsets select columns
    (2, 32, 2, 32, 8, 128, [200, 33], None, 3),                 # two head groups, explicit splits
    (4, 8, 1, 128, 4, 64, [512, 300, 1, 129], None, 0),         # G = 8
]


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
@pytest.mark.parametrize("Q,Hq,Hkv,BS,cols,D,lengths,offsets,num_splits", PCASES)
def test_paged_quant_attention_parity(kvd, fmt, Q, Hq, Hkv, BS, cols, D, lengths, offsets,
                                      num_splits):
    g = W.generator(800 + BS + cols + D + Hq)
    NB = Q * cols + 7
    q = W.randn(g, (Q, Hq, D), torch.bfloat16)
    kc = ROWS[fmt](g, (NB, BS, Hkv), D)
    vc = ROWS[fmt](g, (NB, BS, Hkv), D)
    bt = W.permuted_block_tables(g, Q, cols, NB)
    sl = W.cumsum_lengths(lengths)
    off = None if offsets is None else torch.tensor(offsets, dtype=torch.int32)
    # rows no sequence reads hold NaN codes and scales
    used = torch.zeros(NB, BS, dtype=torch.bool)
    for s in range(Q):
        c0 = 0 if off is None else int(off[s]) // BS
        for t in range(lengths[s]):
            used[int(bt[s, c0 + t // BS]), t % BS] = True
    _poison(kc, fmt, ~used)
    _poison(vc, fmt, ~used)
    scale = 1.0 / math.sqrt(D)
    status = kvd.status_tensor()
    lse = torch.empty(Q, Hq, device="cuda")
    out = kvd.attend_paged_quant(fmt, q.cuda(), kc.cuda(), vc.cuda(), bt.cuda(), sl.cuda(),
                                 None if off is None else off.cuda(), scale, lse=lse,
                                 num_splits=num_splits, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse = oracle.attend_paged_quant(q, kc, vc, bt, sl, off, scale, fmt)
    assert_attention_close(out, ref, torch.bfloat16, f"paged {fmt}")
    assert_lse_close(lse, ref_lse, f"paged {fmt} lse")
    plan = kvd.attend_paged_quant_plan(fmt, Q, Hq, Hkv, BS, cols, D, num_splits)
    assert plan.splits >= 1


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
def test_paged_quant_attention_device_errors(kvd, fmt):
    """A block id outside [0, NB) drops that block's tokens and sets
    KVD_DEV_BLOCK_RANGE; a sequence whose blocks run past the table is empty
    (KVD_DEV_TABLE_COLS); the other sequences are unaffected."""
    g = W.generator(851)
    Q, Hq, Hkv, BS, cols, D, NB = 3, 8, 2, 32, 4, 128, 20
    q = W.randn(g, (Q, Hq, D), torch.bfloat16)
    kc = ROWS[fmt](g, (NB, BS, Hkv), D)
    vc = ROWS[fmt](g, (NB, BS, Hkv), D)
    bt = W.permuted_block_tables(g, Q, cols, NB)
    lengths = [100, 128, 40]
    good = bt.clone()
    bad = bt.clone()
    bad[0, 1] = NB + 3
    sl = W.cumsum_lengths(lengths)
    off = torch.tensor([0, 32, 0], dtype=torch.int32)  # sequence 1: 4 blocks from column 1
    status = kvd.status_tensor()
    out = kvd.attend_paged_quant(fmt, q.cuda(), kc.cuda(), vc.cuda(), bad.cuda(), sl.cuda(),
                                 off.cuda(), dev_status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & kvd.DEV_BLOCK_RANGE and st & kvd.DEV_TABLE_COLS
    assert torch.all(out[1] == 0)
    # sequence 0 without its second block: the tokens of blocks 0, 2, 3 only
    keep = [t for t in range(100) if t // BS != 1]
    rows = lambda c: np.ascontiguousarray(  # noqa: E731
        np.stack([c[int(good[0, t // BS]), t % BS] for t in keep]).transpose(1, 0, 2)[None])
    attend = oracle.attend_masked_fp8 if fmt == "fp8" else oracle.attend_masked_fp4
    ref0, _ = attend(q[:1], rows(kc.numpy()), rows(vc.numpy()), np.ones((1, len(keep)), np.uint8),
                     1.0 / math.sqrt(D))
    assert_attention_close(out[:1], ref0, torch.bfloat16, f"paged {fmt}, dropped block")
    ref2, _ = oracle.attend_paged_quant(q[2:], kc, vc, good[2:], W.cumsum_lengths([40]), None,
                                        1.0 / math.sqrt(D), fmt)
    assert_attention_close(out[2:], ref2, torch.bfloat16, f"paged {fmt}, other sequence")


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_append_paged_quant_bit_exact(kvd, fmt, dt):
    g = W.generator(870)
    Q, Hkv, BS, cols, D, NB = 4, 8, 16, 8, 128, 48
    kc = ROWS[fmt](g, (NB, BS, Hkv), D)
    vc = ROWS[fmt](g, (NB, BS, Hkv), D)
    bt = W.permuted_block_tables(g, Q, cols, NB)
    kn = W.randn(g, (Q, Hkv, D), dt, scale=3.0)
    vn = W.randn(g, (Q, Hkv, D), dt)
    kn[1, 2] = 0  # an all-zero row: scale 0, zero codes
    pos = torch.tensor([0, 15, 16, 127], dtype=torch.int32)
    off = torch.tensor([0, 0, 16, 0], dtype=torch.int32)
    kh, vh = kc.numpy().copy(), vc.numpy().copy()
    assert oracle.append_paged_quant(kh, vh, bt, off, kn, vn, pos, fmt) == 0
    kd, vd = kc.cuda(), vc.cuda()
    status = kvd.status_tensor()
    append = kvd.append_paged_fp8 if fmt == "fp8" else kvd.append_paged_fp4
    append(kd, vd, bt.cuda(), off.cuda(), kn.cuda(), vn.cuda(), pos.cuda(), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(host(kd).numpy(), kh) and np.array_equal(host(vd).numpy(), vh)
    # refused sequences write nothing: a negative position, a column past the
    # table, an offset that is not a multiple of BS, a block outside [0, NB)
    bad_bt = bt.clone()
    bad_bt[3, 0] = -5
    bad_pos = torch.tensor([-1, 8 * BS, 3, 2], dtype=torch.int32)
    bad_off = torch.tensor([0, 0, 5, 0], dtype=torch.int32)
    append(kd, vd, bad_bt.cuda(), bad_off.cuda(), kn.cuda(), vn.cuda(), bad_pos.cuda(), status)
    torch.cuda.synchronize()
    assert int(status.item()) == (kvd.DEV_POS_RANGE | kvd.DEV_TABLE_COLS | kvd.DEV_SEQ_OFFSET |
                                  kvd.DEV_BLOCK_RANGE)
    assert np.array_equal(host(kd).numpy(), kh) and np.array_equal(host(vd).numpy(), vh)


ICASES = [
    # B, Hq, Hkv, C, D, lengths, topk, num_splits
    (3, 32, 8, 3000, 128, [3000, 500, 1], 700, 0),    # tensor-core G = 4, -1 padding
    (2, 8, 8, 1000, 64, [1000, 130], 300, 0),         # one head per kv head
    (2, 16, 2, 2048, 128, [2048, 2048], 1024, 0),     # G = 8
    (1, 32, 2, 600, 128, [600], 257, 2),              # two head groups, explicit splits
]


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
@pytest.mark.parametrize("B,Hq,Hkv,C,D,lengths,topk,num_splits", ICASES)
def test_indexed_quant_attention_parity(kvd, fmt, B, Hq, Hkv, C, D, lengths, topk, num_splits):
    g = W.generator(900 + C + topk + Hq)
    q = W.randn(g, (B, Hq, D), torch.bfloat16)
    k = ROWS[fmt](g, (B, Hkv, C), D)
    v = ROWS[fmt](g, (B, Hkv, C), D)
    idx = W.index_lists(lengths, topk, seed=topk)
    listed = torch.zeros(B, C, dtype=torch.bool)
    for b in range(B):
        ok = idx[b][idx[b] >= 0].long()
        listed[b, ok] = True
    for t in (k, v):
        t4 = t.view(B * Hkv, C, -1)
        _poison(t4, fmt, (~listed).repeat_interleave(Hkv, 0))
    scale = 1.0 / math.sqrt(D)
    status = kvd.status_tensor()
    lse = torch.empty(B, Hq, device="cuda")
    out = kvd.attend_indexed_quant(fmt, q.cuda(), k.cuda(), v.cuda(), idx.cuda(), scale, lse=lse,
                                   num_splits=num_splits, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse, err = oracle.attend_indexed_quant(q, k, v, idx, scale, fmt)
    assert err == 0
    assert_attention_close(out, ref, torch.bfloat16, f"indexed {fmt}")
    assert_lse_close(lse, ref_lse, f"indexed {fmt} lse")


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
def test_indexed_quant_bad_entries(kvd, fmt):
    """Entries outside [-1, C) are skipped and reported; repeated entries
    count once per entry; a list of -1 gives zeros and -inf."""
    g = W.generator(950)
    B, Hq, Hkv, C, D = 3, 16, 4, 500, 128
    q = W.randn(g, (B, Hq, D), torch.bfloat16)
    k = ROWS[fmt](g, (B, Hkv, C), D)
    v = ROWS[fmt](g, (B, Hkv, C), D)
    idx = torch.tensor([[3, 3, 499, C, -1, 7] * 20, [-2, 0, 1, 2, 3, 4] * 20, [-1] * 120],
                       dtype=torch.int32)
    status = kvd.status_tensor()
    lse = torch.empty(B, Hq, device="cuda")
    out = kvd.attend_indexed_quant(fmt, q.cuda(), k.cuda(), v.cuda(), idx.cuda(), lse=lse,
                                   dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kvd.DEV_POS_RANGE
    ref, ref_lse, err = oracle.attend_indexed_quant(q, k, v, idx, 1.0 / math.sqrt(D), fmt)
    assert err == oracle.ERR_POS
    assert torch.all(out[2] == 0) and torch.all(torch.isneginf(lse[2]))
    assert_attention_close(out, ref, torch.bfloat16, f"indexed {fmt}, bad entries")
    assert_lse_close(lse, ref_lse, f"indexed {fmt}, bad entries lse")


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
def test_named_bindings_match_the_format_argument(kvd, fmt):
    """kvd.attend_paged_fp8 / _fp4 and kvd.attend_indexed_fp8 / _fp4 (the C
    entry points' names) give the same bytes as the format-argument forms."""
    g = W.generator(990)
    Q, Hq, Hkv, BS, cols, D, NB = 2, 8, 2, 32, 4, 128, 12
    q = W.randn(g, (Q, Hq, D), torch.bfloat16).cuda()
    kc = ROWS[fmt](g, (NB, BS, Hkv), D).cuda()
    vc = ROWS[fmt](g, (NB, BS, Hkv), D).cuda()
    bt = W.permuted_block_tables(g, Q, cols, NB).cuda()
    sl = W.cumsum_lengths([100, 37]).cuda()
    a = getattr(kvd, f"attend_paged_{fmt}")(q, kc, vc, bt, sl)
    b = kvd.attend_paged_quant(fmt, q, kc, vc, bt, sl)
    plan = getattr(kvd, f"attend_paged_{fmt}_plan")(Q, Hq, Hkv, BS, cols, D)
    assert plan.splits == kvd.attend_paged_quant_plan(fmt, Q, Hq, Hkv, BS, cols, D).splits
    k = ROWS[fmt](g, (Q, Hkv, 300), D).cuda()
    v = ROWS[fmt](g, (Q, Hkv, 300), D).cuda()
    idx = W.index_lists([300, 90], 128, seed=3).cuda()
    c = getattr(kvd, f"attend_indexed_{fmt}")(q, k, v, idx)
    d = kvd.attend_indexed_quant(fmt, q, k, v, idx)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(c.view(torch.int16), d.view(torch.int16))
    assert getattr(kvd, f"attend_indexed_{fmt}_workspace_bytes")(Q, Hq, Hkv, 128, D) == \
        kvd.attend_indexed_quant_workspace_bytes(fmt, Q, Hq, Hkv, 128, D)
