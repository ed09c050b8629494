"""kvd_attend_masked_noalloc, the entry point for callers that cannot
allocate device memory (a host runtime that owns all device memory and gives
the library only its inputs and outputs, an enqueue step that must not
allocate, a loop that cannot take cudaMalloc's implicit synchronisation).

It is called here through the C ABI and must give the same output as
kvd_attend_masked with a caller workspace, within the bf16 attention
tolerance (max |diff| <= 1e-2, relative L2 <= 5e-3), on two calls in a row
whose shapes differ, so that whatever the first call left in the shared
built-in scratch cannot leak into the second; the same calls are also held
against the fp64 oracle.  Sizes whose scratch exceeds the built-in array are
refused.  This file is collected last on purpose.
"""
import ctypes
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


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(kvd, q, k, v, mask, out, lse, num_splits, status):
    B, Hq, D = q.shape
    _, Hkv, C, _ = k.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return kvd.load().kvd_attend_masked_noalloc(_p(q), _p(k), _p(v), _p(mask), _p(out), _p(lse),
                                                B, Hq, Hkv, C, D, 1.0 / math.sqrt(D), kvd.BF16,
                                                num_splits, _p(status), stream)


CALLS = [
    # B, Hq, Hkv, C, D, lengths, num_splits
    (3, 8, 2, 2000, 128, [2000, 1111, 7], 5),
    (2, 32, 8, 700, 64, [0, 650], 3),   # row 0 empty: its splits all have lse = -inf
]


def test_noalloc_matches_the_workspace_entry_point_twice(kvd):
    status = kvd.status_tensor()
    for n, (B, Hq, Hkv, C, D, lengths, ns) in enumerate(CALLS):
        g = W.generator(900 + n, "cuda")
        q = W.randn(g, (B, Hq, D), device="cuda")
        k = W.randn(g, (B, Hkv, C, D), device="cuda")
        v = W.randn(g, (B, Hkv, C, D), device="cuda")
        mask = W.prefix_mask(lengths, C, "cuda")
        assert kvd.attend_masked_workspace_bytes(B, Hq, Hkv, C, D, num_splits=ns) > 0
        ref_lse = torch.empty(B, Hq, device="cuda")
        ref = kvd.attend_masked(q, k, v, mask, 1.0 / math.sqrt(D), lse=ref_lse, num_splits=ns,
                                dev_status=status)
        out = torch.full_like(q, float("nan"))
        lse = torch.empty(B, Hq, device="cuda")
        assert _call_noalloc(kvd, q, k, v, mask, out, lse, ns, status) == kvd.OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_attention_close(out, ref.double().cpu().numpy(), torch.bfloat16, f"call {n}")
        r, o = ref_lse.cpu().numpy(), lse.cpu().numpy()
        assert np.array_equal(np.isneginf(r), np.isneginf(o))
        assert np.allclose(o[np.isfinite(r)], r[np.isfinite(r)], rtol=0, atol=1e-4)
        oref, olse = oracle.attend_masked(q.cpu(), k.cpu(), v.cpu(), mask.cpu(), 1.0 / math.sqrt(D))
        assert_attention_close(out, oref, torch.bfloat16, f"call {n} against the oracle")
        assert_lse_close(lse, olse, f"call {n} lse against the oracle")


def test_noalloc_refuses_sizes_beyond_its_scratch(kvd):
    B, Hq, Hkv, C, D, ns = 16, 32, 8, 8192, 128, 128
    need = kvd.attend_masked_workspace_bytes(B, Hq, Hkv, C, D, num_splits=ns)
    assert need > 8 * 2**20
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(B, Hkv, C, D, dtype=torch.bfloat16, device="cuda")
    mask = torch.ones(B, C, dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(q)
    assert _call_noalloc(kvd, q, k, k, mask, out, None, ns, None) == kvd.ERR_WORKSPACE
    msg = kvd.load().kvd_last_error().decode()
    assert "scratch" in msg and str(need) in msg
    torch.cuda.synchronize()
    assert torch.all(out == 0)
