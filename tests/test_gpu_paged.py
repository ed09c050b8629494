"""GPU parity of the paged path (gather_pa_kv_cache and paged split-KV
attention with in-kernel block-table indirection) against the fp64 oracle,
through the C ABI."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity_util import assert_attention_close, assert_lse_close, host

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def kvd():
    from decode_attention_kv_gb300 import kvd as _kvd
    _kvd.load()
    return _kvd


def _layout(seed, Q, BS, cols, NB, lengths, offsets_blocks=None):
    g = W.generator(seed)
    bt = W.permuted_block_tables(g, Q, cols, NB)
    sl = W.cumsum_lengths(lengths)
    off = torch.zeros(Q, dtype=torch.int32) if offsets_blocks is None else \
        torch.tensor(offsets_blocks, dtype=torch.int32) * BS
    return bt, sl, off


def _bytes(t):
    return host(t).contiguous().view(torch.uint8).numpy()


GATHER_CASES = [
    # NB, BS, Hk, Dk, Hv, Dv, dtype, lengths, cols, offsets (in blocks)
    (40, 16, 2, 128, 2, 128, torch.bfloat16, [0, 1, 15, 16, 17, 70], 6, [0, 1, 0, 2, 0, 1]),
    (64, 128, 8, 128, 8, 128, torch.bfloat16, [300, 1, 256, 129], 4, None),
    (30, 4, 1, 6, 3, 2, torch.bfloat16, [9, 2, 12], 5, [1, 0, 0]),
    (20, 32, 4, 64, 4, 64, torch.float32, [40, 64, 5], 3, None),
]


@pytest.mark.parametrize("NB,BS,Hk,Dk,Hv,Dv,dtype,lengths,cols,offs", GATHER_CASES)
def test_gather_bit_exact(kvd, NB, BS, Hk, Dk, Hv, Dv, dtype, lengths, cols, offs):
    g = W.generator(NB * BS + Dk)
    kc = W.randn(g, (NB, BS, Hk, Dk), dtype)
    vc = W.randn(g, (NB, BS, Hv, Dv), dtype)
    Q = len(lengths)
    bt, sl, off = _layout(1, Q, BS, cols, NB, lengths, offs)
    status = kvd.status_tensor()
    ko, vo = kvd.gather_paged(kc.cuda(), vc.cuda(), bt.cuda(), sl.cuda(), off.cuda(),
                              total_tokens=int(sl[-1]), dev_status=status)
    rk, rv, err = oracle.gather_paged(kc.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy(),
                                      vc.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy(),
                                      bt, sl, off)
    torch.cuda.synchronize()
    assert err == 0 and int(status.item()) == 0
    assert np.array_equal(_bytes(ko), rk.view(np.uint8).reshape(_bytes(ko).shape))
    assert np.array_equal(_bytes(vo), rv.view(np.uint8).reshape(_bytes(vo).shape))


def _split_lengths(rng, Q, T, cap):
    while True:
        cuts = np.sort(rng.integers(0, T + 1, size=Q - 1))
        lens = np.diff(np.concatenate([[0], cuts, [T]]))
        if lens.max() <= cap:
            return lens


def test_gather_page_printed_shapes(kvd):
    """Section 8.1 sweep shapes and the section 8.2 hand-picked shapes of the
    gather page, byte-equal to the oracle (the page compares with torch.equal).
    The sweep cache is [5513, 128, 1, 512] / [5513, 128, 1, 64]."""
    spec = json.load(open(os.path.join(GOLDEN, "gather_pa_kv_cache_shapes.json")))
    rng = np.random.default_rng(5)
    cases = [(spec["sweep"]["key_cache"], spec["sweep"]["value_cache"], c["Q"], c["T"],
              spec["sweep"]["block_table_cols"]) for c in spec["sweep"]["cases"]]
    cases += [(m["key_cache"], m["value_cache"], 2, m["T"], 4) for m in spec["manual"]]
    caches = {}
    for kshape, vshape, Q, T, cols in cases:
        key = (tuple(kshape), tuple(vshape))
        if key not in caches:
            g = W.generator(len(caches) + 50, "cuda")
            caches[key] = (W.randn(g, kshape, torch.bfloat16, "cuda"),
                           W.randn(g, vshape, torch.bfloat16, "cuda"))
        kc, vc = caches[key]
        NB, BS = kshape[0], kshape[1]
        lens = _split_lengths(rng, Q, T, BS * cols)
        sl = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
        bt = torch.tensor(rng.permutation(NB)[: Q * cols].reshape(Q, cols), dtype=torch.int32)
        ko, vo = kvd.gather_paged(kc, vc, bt.cuda(), sl.cuda(), None, total_tokens=T)
        # oracle on the referenced blocks only (host copies of those blocks)
        used = sorted(set(bt.reshape(-1).tolist()))
        remap = {b: i for i, b in enumerate(used)}
        bt_c = torch.tensor([[remap[int(x)] for x in row] for row in bt], dtype=torch.int32)
        idx = torch.tensor(used, device="cuda")
        kh = host(kc.index_select(0, idx)).view(torch.int16).numpy()
        vh = host(vc.index_select(0, idx)).view(torch.int16).numpy()
        rk, rv, err = oracle.gather_paged(kh, vh, bt_c, sl, None)
        assert err == 0
        assert np.array_equal(host(ko).view(torch.int16).numpy(), rk)
        assert np.array_equal(host(vo).view(torch.int16).numpy(), rv)


def test_gather_device_errors(kvd):
    NB, BS, H, D = 8, 16, 1, 64
    g = W.generator(3)
    kc = W.randn(g, (NB, BS, H, D)).cuda()
    vc = W.randn(g, (NB, BS, H, D)).cuda()
    bt = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32)
    sl = torch.tensor([0, 20, 30], dtype=torch.int32)

    def run(bt_, sl_, off_, T):
        st = kvd.status_tensor()
        ko = torch.zeros(T, H, D, dtype=torch.bfloat16, device="cuda")
        vo = torch.zeros(T, H, D, dtype=torch.bfloat16, device="cuda")
        kvd.gather_paged(kc, vc, bt_.cuda(), sl_.cuda(), None if off_ is None else off_.cuda(),
                         ko, vo, total_tokens=T, dev_status=st)
        torch.cuda.synchronize()
        kh = host(kc).view(torch.int16).numpy()
        vh = host(vc).view(torch.int16).numpy()
        rk, _, err = oracle.gather_paged(kh, vh, bt_, sl_, off_, total_tokens=T)
        assert np.array_equal(host(ko).view(torch.int16).numpy(), rk)
        return int(st.item()), err

    assert run(bt, sl, None, 30) == (0, 0)
    bad = bt.clone()
    bad[0, 1] = NB
    assert run(bad, sl, None, 30) == (kvd.DEV_BLOCK_RANGE, oracle.ERR_BLOCK)
    assert run(bt, sl, torch.tensor([8, 0], dtype=torch.int32), 30) == \
        (kvd.DEV_SEQ_OFFSET, oracle.ERR_OFFSET)
    assert run(bt, sl, torch.tensor([16, 0], dtype=torch.int32), 30) == \
        (kvd.DEV_TABLE_COLS, oracle.ERR_COLS)
    assert run(bt, torch.tensor([0, 20, 10], dtype=torch.int32), None, 20) == \
        (kvd.DEV_SEQLENS, oracle.ERR_SEQLENS)


PAGED_CASES = [
    # dtype, NB, BS, Hkv, Hq, D, lengths, cols, offsets, num_splits
    (torch.bfloat16, 64, 128, 8, 32, 128, [1, 300, 0, 1024, 129, 777], 8, None, 0),
    (torch.bfloat16, 100, 16, 2, 8, 128, [0, 5, 16, 17, 200, 63], 16, [0, 1, 2, 0, 1, 3], 3),
    (torch.bfloat16, 40, 48, 4, 4, 64, [47, 48, 49, 300], 7, None, 0),
    (torch.float32, 30, 32, 2, 6, 64, [33, 1, 95], 4, [1, 0, 0], 0),
    (torch.bfloat16, 50, 64, 1, 16, 128, [640, 3], 12, None, 2),
]


@pytest.mark.parametrize("dtype,NB,BS,Hkv,Hq,D,lengths,cols,offs,num_splits", PAGED_CASES)
def test_paged_attention_parity(kvd, dtype, NB, BS, Hkv, Hq, D, lengths, cols, offs, num_splits):
    g = W.generator(NB + BS + Hq)
    kc = W.randn(g, (NB, BS, Hkv, D), dtype)
    vc = W.randn(g, (NB, BS, Hkv, D), dtype)
    Q = len(lengths)
    q = W.randn(g, (Q, Hq, D), dtype)
    bt, sl, off = _layout(2, Q, BS, cols, NB, lengths, offs)
    scale = 1.0 / math.sqrt(D)
    lse = torch.empty(Q, Hq, device="cuda")
    status = kvd.status_tensor()
    out = kvd.attend_paged(q.cuda(), kc.cuda(), vc.cuda(), bt.cuda(), sl.cuda(), off.cuda(),
                           scale, lse=lse, num_splits=num_splits, dev_status=status)
    ref, ref_lse = oracle.attend_paged(q, kc, vc, bt, sl, off, scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_attention_close(out, ref, dtype, "paged")
    assert_lse_close(lse, ref_lse, "paged lse")


def test_paged_device_errors(kvd):
    """Bad offsets / decreasing cumsum empty their sequence (out 0, lse -inf);
    an out-of-range block id drops that block's tokens."""
    NB, BS, Hkv, Hq, D = 16, 16, 2, 4, 128
    g = W.generator(4)
    kc = W.randn(g, (NB, BS, Hkv, D))
    vc = W.randn(g, (NB, BS, Hkv, D))
    q = W.randn(g, (3, Hq, D))
    bt = torch.tensor([[0, 1, 2], [3, 4, 5], [6, 7, 8]], dtype=torch.int32)
    sl = torch.tensor([0, 40, 70, 80], dtype=torch.int32)

    def run(bt_, sl_, off_):
        st = kvd.status_tensor()
        lse = torch.empty(3, Hq, device="cuda")
        out = kvd.attend_paged(q.cuda(), kc.cuda(), vc.cuda(), bt_.cuda(), sl_.cuda(),
                               None if off_ is None else off_.cuda(), 0.1, lse=lse, dev_status=st)
        torch.cuda.synchronize()
        return host(out), host(lse), int(st.item())

    out, lse, st = run(bt, sl, torch.tensor([0, 5, 0], dtype=torch.int32))
    assert st == kvd.DEV_SEQ_OFFSET
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    ref, _ = oracle.attend_paged(q[[0, 2]], kc, vc, bt[[0, 2]],
                                 torch.tensor([0, 40, 50], dtype=torch.int32), None, 0.1)
    assert_attention_close(out[[0, 2]], ref, torch.bfloat16, "other sequences")

    out, lse, st = run(bt, torch.tensor([0, 40, 30, 40], dtype=torch.int32), None)
    assert st == kvd.DEV_SEQLENS and torch.all(out[1] == 0)

    bad = bt.clone()
    bad[0, 1] = -3
    out, lse, st = run(bad, sl, None)
    assert st == kvd.DEV_BLOCK_RANGE
    # sequence 0 keeps tokens 0..15 and 32..39 (block 1 dropped)
    keep = list(range(16)) + list(range(32, 40))
    phys = [int(bt[0, t // BS]) for t in keep]
    kk = torch.stack([kc[p, t % BS] for p, t in zip(phys, keep)]).permute(1, 0, 2)[None].contiguous()
    vv = torch.stack([vc[p, t % BS] for p, t in zip(phys, keep)]).permute(1, 0, 2)[None].contiguous()
    ref, _ = oracle.attend_masked(q[:1], kk, vv, torch.ones(1, len(keep), dtype=torch.uint8), 0.1)
    assert_attention_close(out[:1], ref, torch.bfloat16, "dropped block")

    out, lse, st = run(bt, sl, torch.tensor([0, 0, 48], dtype=torch.int32))
    assert st == kvd.DEV_TABLE_COLS and torch.all(out[2] == 0)


APPEND_CASES = [
    # dtype, NB, BS, Hkv, D, lengths (tokens before the step), cols, offsets (blocks)
    (torch.bfloat16, 160, 128, 8, 128, [0, 127, 128, 1000, 4095], 32, None),
    (torch.bfloat16, 50, 16, 2, 64, [5, 16, 31, 0], 6, [0, 1, 2, 4]),
    (torch.float32, 48, 1, 3, 64, [0, 7, 12], 15, [2, 0, 1]),
]


@pytest.mark.parametrize("dtype,NB,BS,Hkv,D,lengths,cols,offs", APPEND_CASES)
def test_append_paged_then_attend(kvd, dtype, NB, BS, Hkv, D, lengths, cols, offs):
    """One paged decode step: every sequence appends its new token at its
    current length (byte-exact against the oracle's append over the whole
    caches), then paged attention runs over the one-token-longer sequences
    (against the oracle's attention)."""
    g = W.generator(8800 + NB + BS)
    kc = W.randn(g, (NB, BS, Hkv, D), dtype)
    vc = W.randn(g, (NB, BS, Hkv, D), dtype)
    Q, Hq = len(lengths), 4 * Hkv
    kn = W.randn(g, (Q, Hkv, D), dtype)
    vn = W.randn(g, (Q, Hkv, D), dtype)
    q = W.randn(g, (Q, Hq, D), dtype)
    bt, _, off = _layout(7, Q, BS, cols, NB, lengths, offs)
    pos = torch.tensor(lengths, dtype=torch.int32)
    kd, vd = kc.cuda(), vc.cuda()
    status = kvd.status_tensor()
    kvd.append_paged(kd, vd, bt.cuda(), off.cuda(), kn.cuda(), vn.cuda(), pos.cuda(), status)
    kh = _bytes(kc).reshape(NB, BS, Hkv, -1).copy()
    vh = _bytes(vc).reshape(NB, BS, Hkv, -1).copy()
    assert oracle.append_paged(kh, vh, bt, off, _bytes(kn).reshape(Q, Hkv, -1),
                               _bytes(vn).reshape(Q, Hkv, -1), pos) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(_bytes(kd).reshape(kh.shape), kh), "append (K) not bit-exact"
    assert np.array_equal(_bytes(vd).reshape(vh.shape), vh), "append (V) not bit-exact"
    sl = W.cumsum_lengths([L + 1 for L in lengths])
    lse = torch.empty(Q, Hq, device="cuda")
    out = kvd.attend_paged(q.cuda(), kd, vd, bt.cuda(), sl.cuda(), off.cuda(), 1.0 / math.sqrt(D),
                           lse=lse, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse = oracle.attend_paged(q, host(kd), host(vd), bt, sl, off, 1.0 / math.sqrt(D))
    assert_attention_close(out, ref, dtype, "append then attend")
    assert_lse_close(lse, ref_lse, "append then attend lse")


def test_append_paged_device_errors(kvd):
    """Each failing sequence writes nothing and sets its bit; the others are
    appended (byte-exact against the oracle)."""
    NB, BS, Hkv, D, cols = 16, 4, 2, 64, 3
    g = W.generator(8900)
    kc = W.randn(g, (NB, BS, Hkv, D))
    vc = W.randn(g, (NB, BS, Hkv, D))
    kn = W.randn(g, (5, Hkv, D))
    vn = W.randn(g, (5, Hkv, D))
    bt = torch.arange(15, dtype=torch.int32).reshape(5, 3)
    bt[3, 0] = 99  # a block id out of range
    off = torch.tensor([0, 4, 3, 0, 0], dtype=torch.int32)  # q2: not a multiple of BS
    pos = torch.tensor([-1, 0, 0, 2, 12], dtype=torch.int32)  # q0 negative, q4 past the table
    kd, vd = kc.cuda(), vc.cuda()
    status = kvd.status_tensor()
    kvd.append_paged(kd, vd, bt.cuda(), off.cuda(), kn.cuda(), vn.cuda(), pos.cuda(), status)
    torch.cuda.synchronize()
    kh = _bytes(kc).reshape(NB, BS, Hkv, -1).copy()
    vh = _bytes(vc).reshape(NB, BS, Hkv, -1).copy()
    err = oracle.append_paged(kh, vh, bt, off, _bytes(kn).reshape(5, Hkv, -1),
                              _bytes(vn).reshape(5, Hkv, -1), pos)
    assert err == oracle.ERR_POS | oracle.ERR_OFFSET | oracle.ERR_BLOCK | oracle.ERR_COLS
    assert int(status.item()) == (kvd.DEV_POS_RANGE | kvd.DEV_SEQ_OFFSET |
                                  kvd.DEV_BLOCK_RANGE | kvd.DEV_TABLE_COLS)
    assert np.array_equal(_bytes(kd).reshape(kh.shape), kh)
    assert np.array_equal(_bytes(vd).reshape(vh.shape), vh)
