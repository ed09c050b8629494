"""GPU parity of sliding-window decode attention (cuTile on NPU, Part 1: the
sliding-window tile variant) against the fp64 oracle.  A window is a mask
pattern: the static-buffer kernel reads only the tiles the window touches
and skips the splits outside it."""
import math

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
