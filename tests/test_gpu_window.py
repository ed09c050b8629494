"""GPU parity of sliding-window decode attention (cuTile on NPU, Part 1: the
sliding-window tile variant) against the fp64 oracle, both ways a caller can
express a window: as a mask pattern through kvd_attend_masked (the kernel
reads only the tiles the window touches and skips the splits outside it),
and through the window entries, whose splits cover each row's window only."""
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


CASES = [
    # dtype, B, Hq, Hkv, C, D, lengths, window, num_splits
    (torch.bfloat16, 2, 32, 8, 3000, 128, [3000, 1777], 1000, 0),    # tensor-core consumers
    (torch.bfloat16, 2, 32, 8, 3000, 128, [3000, 1777], 1, 0),       # one row per sequence
    (torch.bfloat16, 1, 4, 4, 4096, 128, [4096], 65, 0),             # window across a tile edge
    (torch.bfloat16, 2, 16, 2, 5000, 128, [4999, 300], 4096, 0),     # window longer than a sequence
    (torch.bfloat16, 2, 8, 8, 2100, 64, [2100, 1000], 63, 0),        # CUDA-core consumers
    (torch.float32, 2, 4, 1, 700, 64, [700, 129], 100, 3),
]


@pytest.mark.parametrize("dtype,B,Hq,Hkv,C,D,lengths,window,num_splits", CASES)
def test_window_parity(kvd, dtype, B, Hq, Hkv, C, D, lengths, window, num_splits):
    g = W.generator(300 + window + C)
    q = W.randn(g, (B, Hq, D), dtype)
    k = W.randn(g, (B, Hkv, C, D), dtype)
    v = W.randn(g, (B, Hkv, C, D), dtype)
    mask = W.window_mask(lengths, C, window)
    scale = 1.0 / math.sqrt(D)
    status = kvd.status_tensor("cuda")
    lse = torch.empty(B, Hq, device="cuda")
    out = kvd.attend_masked(q.cuda(), k.cuda(), v.cuda(), mask.cuda(), scale, lse=lse,
                            num_splits=num_splits, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse = oracle.attend_masked(q, k, v, mask, scale)
    assert_attention_close(out, ref, dtype, f"window {window}")
    assert_lse_close(lse, ref_lse, f"window {window} lse")


# ------------------------------------------------ the sliding-window entries
# kvd_attend_window lays its splits over each row's window only; the mask
# still selects inside it.

ECASES = [
    # dtype, B, Hq, Hkv, C, D, lasts, W, num_splits, holes
    (torch.bfloat16, 3, 32, 8, 8192, 128, [8191, 100, 5000], 4096, 0, True),  # tensor-core, clipped at 0
    (torch.bfloat16, 2, 32, 8, 3000, 128, [2999, 1777], 1, 0, False),         # one slot
    (torch.bfloat16, 1, 32, 32, 32768, 128, [32767], 4096, 0, False),         # CUDA-core, many rows' tails
    (torch.bfloat16, 2, 8, 4, 5000, 64, [4321, 63], 65, 0, True),             # g = 2, ragged edges
    (torch.bfloat16, 2, 16, 2, 5000, 128, [4999, 300], 4096, 3, False),       # explicit split count
    (torch.bfloat16, 2, 32, 2, 2048, 128, [2047, 1000], 700, 0, True),        # two head groups per kv head
    (torch.bfloat16, 1, 4, 4, 256, 128, [255], 10000, 0, False),              # window beyond the buffer
    (torch.float32, 2, 4, 1, 700, 64, [699, 129], 100, 0, True),
    (torch.float32, 3, 8, 8, 1000, 128, [999, 31, 500], 33, 0, True),         # f32 32-slot tiles
]


def _window_inputs(dtype, B, Hq, Hkv, C, D, lasts, holes, seed):
    g = W.generator(seed)
    q = W.randn(g, (B, Hq, D), dtype)
    k = W.randn(g, (B, Hkv, C, D), dtype)
    v = W.randn(g, (B, Hkv, C, D), dtype)
    if holes:
        mask = (torch.rand(B, C, generator=g) < 0.75).to(torch.uint8)
    else:
        mask = torch.ones(B, C, dtype=torch.uint8)
    last = torch.tensor(lasts, dtype=torch.int32)
    return q, k, v, mask, last


@pytest.mark.parametrize("dtype,B,Hq,Hkv,C,D,lasts,Wn,num_splits,holes", ECASES)
def test_window_entry_parity(kvd, dtype, B, Hq, Hkv, C, D, lasts, Wn, num_splits, holes):
    q, k, v, mask, last = _window_inputs(dtype, B, Hq, Hkv, C, D, lasts, holes, 500 + Wn + C)
    scale = 1.0 / math.sqrt(D)
    status = kvd.status_tensor("cuda")
    lse = torch.empty(B, Hq, device="cuda")
    out = kvd.attend_window(q.cuda(), k.cuda(), v.cuda(), mask.cuda(), last.cuda(), Wn, scale,
                            lse=lse, num_splits=num_splits, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse, err = oracle.attend_window(q, k, v, mask, last, Wn, scale)
    assert err == 0
    assert_attention_close(out, ref, dtype, f"window entry {Wn}")
    assert_lse_close(lse, ref_lse, f"window entry {Wn} lse")
    plan = kvd.attend_window_plan(B, Hq, Hkv, C, D, Wn, dtype, num_splits)
    assert plan.splits >= 1 and plan.launches == (2 if plan.splits > 1 else 1)


FCASES = [
    # dtype, B, Hq, Hkv, C, D, first positions, W
    (torch.bfloat16, 2, 32, 8, 4096, 128, [4000, 70], 1024),   # tensor-core consumers
    (torch.bfloat16, 1, 16, 16, 9000, 128, [8990], 3000),      # CUDA-core, split kernel
    (torch.bfloat16, 2, 32, 2, 2048, 128, [2040, 5], 300),     # append kernel first
    (torch.float32, 2, 4, 2, 1500, 64, [1490, 64], 64),
]


@pytest.mark.parametrize("dtype,B,Hq,Hkv,C,D,pos0,Wn", FCASES)
def test_append_attend_window_steps(kvd, dtype, B, Hq, Hkv, C, D, pos0, Wn):
    """Three decode steps of kvd_append_attend_window: caches and mask
    byte-exact against the oracle's append, the attention against its window
    ending at the appended slot."""
    g = W.generator(700 + Wn)
    k = W.randn(g, (B, Hkv, C, D), dtype)
    v = W.randn(g, (B, Hkv, C, D), dtype)
    mask = W.prefix_mask(pos0, C)
    kd, vd, md = k.cuda(), v.cuda(), mask.cuda()
    kh, vh, mh = k.numpy().copy() if dtype == torch.float32 else k.view(torch.int16).numpy().copy(), \
        v.numpy().copy() if dtype == torch.float32 else v.view(torch.int16).numpy().copy(), \
        mask.numpy().copy()
    status = kvd.status_tensor("cuda")
    for step in range(3):
        q = W.randn(g, (B, Hq, D), dtype)
        kn = W.randn(g, (B, Hkv, D), dtype)
        vn = W.randn(g, (B, Hkv, D), dtype)
        pos = torch.tensor([p + step for p in pos0], dtype=torch.int32)
        lse = torch.empty(B, Hq, device="cuda")
        out = kvd.append_attend_window(q.cuda(), kd, vd, md, kn.cuda(), vn.cuda(), pos.cuda(), Wn,
                                       lse=lse, dev_status=status)
        knh = kn.numpy() if dtype == torch.float32 else kn.view(torch.int16).numpy()
        vnh = vn.numpy() if dtype == torch.float32 else vn.view(torch.int16).numpy()
        assert oracle.append(kh, vh, knh, vnh, pos.numpy(), mh) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        kb = kd.cpu() if dtype == torch.float32 else kd.cpu().view(torch.int16)
        vb = vd.cpu() if dtype == torch.float32 else vd.cpu().view(torch.int16)
        assert np.array_equal(kb.numpy(), kh) and np.array_equal(vb.numpy(), vh)
        assert np.array_equal(md.cpu().numpy(), mh)
        kr = torch.from_numpy(kh) if dtype == torch.float32 else torch.from_numpy(kh).view(dtype)
        vr = torch.from_numpy(vh) if dtype == torch.float32 else torch.from_numpy(vh).view(dtype)
        ref, ref_lse, err = oracle.attend_window(q, kr, vr, torch.from_numpy(mh), pos, Wn,
                                                 1.0 / math.sqrt(D))
        assert err == 0
        assert_attention_close(out, ref, dtype, f"window step {step}")
        assert_lse_close(lse, ref_lse, f"window step {step} lse")


def test_window_entry_newest_slot_out_of_range(kvd):
    """A newest slot outside [0, C) empties its row (zeros, lse = -inf) and
    sets KVD_DEV_POS_RANGE; the other rows are unaffected."""
    dtype, B, Hq, Hkv, C, D = torch.bfloat16, 3, 8, 2, 2048, 128
    q, k, v, mask, _ = _window_inputs(dtype, B, Hq, Hkv, C, D, [0, 0, 0], True, 901)
    last = torch.tensor([-1, 1500, C], dtype=torch.int32)
    status = kvd.status_tensor("cuda")
    lse = torch.empty(B, Hq, device="cuda")
    out = kvd.attend_window(q.cuda(), k.cuda(), v.cuda(), mask.cuda(), last.cuda(), 512, lse=lse,
                            dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kvd.DEV_POS_RANGE
    ref, ref_lse, err = oracle.attend_window(q, k, v, mask, last, 512, 1.0 / math.sqrt(D))
    assert err == 1
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert torch.all(torch.isneginf(lse[0])) and torch.all(torch.isneginf(lse[2]))
    assert_attention_close(out, ref, dtype, "window, bad newest slots")
    assert_lse_close(lse, ref_lse, "window, bad newest slots lse")
