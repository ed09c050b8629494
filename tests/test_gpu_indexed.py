"""GPU parity of kvd_attend_indexed (decode attention over a list of cache
slots per batch entry: the top-k index lists of sparse attention) against
the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity_util import assert_attention_close, assert_lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvd():
    from decode_attention_kv_gb300 import kvd as _kvd
    _kvd.load()
    return _kvd


def _lists(g, B, C, topk, frac_unused=0.0, dup=False):
    rows = []
    for _ in range(B):
        r = torch.randperm(C, generator=g)[:topk].to(torch.int32)
        if dup:
            r[1::7] = r[0::7][: r[1::7].numel()]
        if frac_unused:
            drop = torch.rand(topk, generator=g) < frac_unused
            r[drop] = -1
        rows.append(r)
    return torch.stack(rows)


CASES = [
    # dtype, B, Hq, Hkv, C, D, topk, num_splits, unused fraction, duplicates
    (torch.bfloat16, 3, 8, 2, 3000, 128, 300, 0, 0.0, False),   # tensor-core gather, ragged tail
    (torch.bfloat16, 2, 32, 8, 8192, 128, 2048, 0, 0.1, True),  # top-2048 of 8192
    (torch.bfloat16, 2, 16, 16, 1000, 128, 129, 0, 0.0, False),  # CUDA-core gather (MHA)
    (torch.bfloat16, 2, 8, 4, 500, 64, 64, 1, 0.3, False),       # one split, head_dim 64
    (torch.float32, 2, 8, 8, 700, 64, 200, 0, 0.0, True),        # fp32
    (torch.float32, 1, 16, 2, 400, 128, 96, 3, 0.0, False),      # fp32, groups of 8
]


@pytest.mark.parametrize("dtype,B,Hq,Hkv,C,D,topk,ns,unused,dup", CASES)
def test_indexed_parity(kvd, dtype, B, Hq, Hkv, C, D, topk, ns, unused, dup):
    g = W.generator(500 + topk, "cpu")
    q = W.randn(g, (B, Hq, D), dtype)
    k = W.randn(g, (B, Hkv, C, D), dtype)
    v = W.randn(g, (B, Hkv, C, D), dtype)
    idx = _lists(g, B, C, topk, unused, dup)
    scale = 1.0 / math.sqrt(D)
    status = kvd.status_tensor()
    lse = torch.empty(B, Hq, device="cuda")
    out = kvd.attend_indexed(q.cuda(), k.cuda(), v.cuda(), idx.cuda(), scale, lse=lse,
                             num_splits=ns, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse, err = oracle.attend_indexed(q, k, v, idx, scale)
    assert err == 0
    assert_attention_close(out, ref, dtype, f"indexed {dtype} {Hq}/{Hkv} topk={topk}")
    assert_lse_close(lse, ref_lse, "indexed")


def test_indexed_bad_entries_and_empty_lists(kvd):
    """Entries outside [-1, C) are reported and dropped; an all -1 list gives
    zeros and lse -inf; garbage (inf, NaN) in unlisted slots is never read."""
    g = W.generator(77, "cpu")
    B, Hq, Hkv, C, D, topk = 3, 8, 2, 256, 128, 70
    q = W.randn(g, (B, Hq, D), torch.bfloat16)
    k = W.randn(g, (B, Hkv, C, D), torch.bfloat16)
    v = W.randn(g, (B, Hkv, C, D), torch.bfloat16)
    idx = _lists(g, B, 200, topk)  # slots < 200 listed
    k[:, :, 200:] = float("nan")
    v[:, :, 200:] = float("inf")
    idx[2] = -1
    bad = idx.clone()
    bad[0, 5] = C        # out of range
    bad[1, 9] = -7       # out of range
    status = kvd.status_tensor()
    lse = torch.empty(B, Hq, device="cuda")
    out = kvd.attend_indexed(q.cuda(), k.cuda(), v.cuda(), bad.cuda(), 0.1, lse=lse,
                             dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1  # KVD_DEV_POS_RANGE
    ref, ref_lse, err = oracle.attend_indexed(q, k, v, bad, 0.1)
    assert err == oracle.ERR_POS
    assert_attention_close(out, ref, torch.bfloat16, "bad entries")
    assert_lse_close(lse, ref_lse, "bad entries")
    assert torch.all(out[2] == 0) and torch.all(torch.isneginf(lse[2]))


def test_indexed_full_size(kvd):
    """The benchmark's configuration: the batched-GQA caches (16 x 32/8 heads,
    capacity 8192, lengths 512..8192) with 2048 listed slots per entry (fewer
    for a shorter prefix, -1 after them); every entry and head compared."""
    lay = W.gqa(device="cuda", layers=1).layers[0]
    L = [int(x) for x in lay.lengths]
    idx = W.index_lists(L, 2048)
    status = kvd.status_tensor("cuda")
    lse = torch.empty(16, 32, device="cuda")
    out = kvd.attend_indexed(lay.q, lay.k_cache, lay.v_cache, idx.cuda(), lay.scale, lse=lse,
                             dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse, err = oracle.attend_indexed(lay.q.cpu(), lay.k_cache.cpu(), lay.v_cache.cpu(),
                                              idx, lay.scale)
    assert err == 0
    assert_attention_close(out, ref, torch.bfloat16, "indexed, all entries")
    assert_lse_close(lse, ref_lse, "indexed lse")
