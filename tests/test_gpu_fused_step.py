"""GPU parity of kvd_append_attend_masked (the append fused into the masked
attention launch) against the fp64 oracle's append followed by its masked
attention: caches and mask byte-exact, output within the tolerance."""
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


def _bits(t):
    t = host(t)
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.numpy()


CASES = [
    # dtype, B, Hq, Hkv, C, D, first positions, num_splits
    (torch.bfloat16, 1, 32, 32, 1152, 128, [1024], 0),        # the static-buffer default, one CTA per unit
    (torch.bfloat16, 2, 32, 8, 1152, 128, [5, 640], 0),       # tensor-core consumers, small launch
    (torch.bfloat16, 3, 32, 8, 8192, 128, [8191, 4096, 63], 0),  # many units per CTA
    (torch.bfloat16, 2, 8, 4, 700, 64, [0, 31], 0),           # two heads per kv head, first tiles
    (torch.float32, 2, 4, 4, 300, 128, [64, 299], 0),
    (torch.bfloat16, 2, 48, 3, 520, 64, [100, 519], 0),       # two head groups: append kernel first
    # The persistent split kernel with CUDA-core consumers and the append in
    # its scheduler warps (launches too large for the one-CTA-per-split path):
    # one query head per kv head, splits of 256 slots (a tail of 64-slot
    # splits from 6144 on); positions cross a split edge (254 -> 256) and
    # fill the last split (8189 -> 8191).
    (torch.bfloat16, 2, 32, 32, 8192, 128, [254, 8189], 0),
    (torch.bfloat16, 2, 16, 8, 4096, 128, [1023, 4093], 0),   # two query heads per kv head
    (torch.float32, 2, 4, 4, 4096, 128, [511, 4094], 0),      # fp32 rows
    (torch.bfloat16, 1, 8, 8, 2048, 64, [700], 5),            # an explicit split count, D 64
    (torch.bfloat16, 2, 32, 8, 4096, 128, [2047, 3000], 7),   # explicit splits, tensor cores
    (torch.float32, 1, 4, 2, 1000, 64, [333], 1),             # one split: rows written directly
]


@pytest.mark.parametrize("dtype,B,Hq,Hkv,C,D,pos0,num_splits", CASES)
def test_fused_step_parity(kvd, dtype, B, Hq, Hkv, C, D, pos0, num_splits):
    g = W.generator(1100 + C + Hq)
    k = W.randn(g, (B, Hkv, C, D), dtype)
    v = W.randn(g, (B, Hkv, C, D), dtype)
    mask = W.prefix_mask(pos0, C)  # rows before the first step's slot
    kd, vd, md = k.cuda(), v.cuda(), mask.cuda()
    kh, vh, mh = _bits(k).copy(), _bits(v).copy(), mask.numpy().copy()
    status = kvd.status_tensor()
    scale = 1.0 / math.sqrt(D)
    for step in range(3):
        q = W.randn(g, (B, Hq, D), dtype)
        kn = W.randn(g, (B, Hkv, D), dtype)
        vn = W.randn(g, (B, Hkv, D), dtype)
        pos = torch.tensor([min(p + step, C - 1) for p in pos0], dtype=torch.int32)
        lse = torch.empty(B, Hq, device="cuda")
        out = kvd.append_attend_masked(q.cuda(), kd, vd, md, kn.cuda(), vn.cuda(), pos.cuda(),
                                       scale, lse=lse, num_splits=num_splits,
                                       dev_status=status)
        assert oracle.append(kh, vh, kn, vn, pos, mh) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(_bits(kd), kh) and np.array_equal(_bits(vd), vh), f"step {step}"
        assert np.array_equal(host(md).numpy(), mh)
        kt = torch.from_numpy(kh).view(torch.bfloat16) if dtype == torch.bfloat16 else torch.from_numpy(kh)
        vt = torch.from_numpy(vh).view(torch.bfloat16) if dtype == torch.bfloat16 else torch.from_numpy(vh)
        ref, ref_lse = oracle.attend_masked(q, kt, vt, torch.from_numpy(mh), scale)
        assert_attention_close(out, ref, dtype, f"fused step {step}")
        assert_lse_close(lse, ref_lse)


def test_fused_step_position_out_of_range(kvd):
    """pos outside [0, C) writes nothing for its entry (reported), the other
    entries are appended, and attention runs over the mask as it is."""
    B, Hq, Hkv, C, D = 2, 16, 4, 500, 128
    g = W.generator(1200)
    k = W.randn(g, (B, Hkv, C, D))
    v = W.randn(g, (B, Hkv, C, D))
    q = W.randn(g, (B, Hq, D))
    kn = W.randn(g, (B, Hkv, D))
    vn = W.randn(g, (B, Hkv, D))
    mask = W.prefix_mask([200, 300], C)
    pos = torch.tensor([200, 500], dtype=torch.int32)
    kd, vd, md = k.cuda(), v.cuda(), mask.cuda()
    kh, vh, mh = _bits(k).copy(), _bits(v).copy(), mask.numpy().copy()
    status = kvd.status_tensor()
    out = kvd.append_attend_masked(q.cuda(), kd, vd, md, kn.cuda(), vn.cuda(), pos.cuda(), 0.1,
                                   dev_status=status)
    assert oracle.append(kh, vh, kn, vn, pos, mh) == oracle.ERR_POS
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert np.array_equal(_bits(kd), kh) and np.array_equal(host(md).numpy(), mh)
    ref, _ = oracle.attend_masked(q, torch.from_numpy(kh).view(torch.bfloat16),
                                  torch.from_numpy(vh).view(torch.bfloat16), torch.from_numpy(mh), 0.1)
    assert_attention_close(out, ref, torch.bfloat16, "pos out of range")
