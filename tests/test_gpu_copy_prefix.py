"""GPU parity of kvd_copy_prefix (copy_kvcache: prefill present[0:N] ->
generate past[0:N] for every layer in one launch) against the oracle, byte
for byte, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvd():
    from decode_attention_kv_gb300 import kvd as _kvd
    _kvd.load()
    return _kvd


def _caches(g, L, B, H, C, D, dtype):
    return [W.randn(g, (B, H, C, D), dtype, "cuda") for _ in range(L)]


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float32, 64), (torch.bfloat16, 8)])
@pytest.mark.parametrize("with_mask", [True, False])
def test_copy_prefix_matches_the_oracle(kvd, dtype, D, with_mask):
    g = W.generator(31, "cuda")
    L, B, H, Cs, Cd = 3, 3, 2, 40, 48
    ks, vs = _caches(g, L, B, H, Cs, D, dtype), _caches(g, L, B, H, Cs, D, dtype)
    kd, vd = _caches(g, L, B, H, Cd, D, dtype), _caches(g, L, B, H, Cd, D, dtype)
    masks = [torch.full((B, Cd), 9, dtype=torch.uint8, device="cuda") for _ in range(L)] \
        if with_mask else None
    n = torch.tensor([0, 40, 17], dtype=torch.int32, device="cuda")
    exp_k = [t.cpu().view(torch.uint8).numpy().copy() for t in kd]
    exp_v = [t.cpu().view(torch.uint8).numpy().copy() for t in vd]
    exp_m = [m.cpu().numpy().copy() for m in masks] if with_mask else [None] * L
    for l in range(L):
        src_k = ks[l].cpu().view(torch.uint8).numpy()
        src_v = vs[l].cpu().view(torch.uint8).numpy()
        # bytes view: D * elem bytes per row
        assert oracle.copy_prefix(src_k, src_v, exp_k[l], exp_v[l], n.cpu(), exp_m[l]) == 0
    status = kvd.status_tensor()
    keep = kvd.copy_prefix(ks, vs, kd, vd, n, masks, status)
    torch.cuda.synchronize()
    del keep
    assert int(status.item()) == 0
    for l in range(L):
        assert np.array_equal(kd[l].cpu().view(torch.uint8).numpy(), exp_k[l])
        assert np.array_equal(vd[l].cpu().view(torch.uint8).numpy(), exp_v[l])
        if with_mask:
            assert np.array_equal(masks[l].cpu().numpy(), exp_m[l])


def test_copy_prefix_out_of_range_and_bad_pointers(kvd):
    g = W.generator(32, "cuda")
    L, B, H, Cs, Cd, D = 2, 2, 1, 8, 6, 64
    ks, vs = _caches(g, L, B, H, Cs, D, torch.float32), _caches(g, L, B, H, Cs, D, torch.float32)
    kd, vd = _caches(g, L, B, H, Cd, D, torch.float32), _caches(g, L, B, H, Cd, D, torch.float32)
    before = [t.clone() for t in kd]
    n = torch.tensor([7, 3], dtype=torch.int32, device="cuda")  # 7 > min(8, 6)
    status = kvd.status_tensor()
    keep = kvd.copy_prefix(ks, vs, kd, vd, n, None, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1  # KVD_DEV_POS_RANGE
    for l in range(L):
        assert torch.equal(kd[l][0], before[l][0])            # entry 0 untouched
        assert torch.equal(kd[l][1, :, :3], ks[l][1, :, :3])  # entry 1 copied
        assert torch.equal(kd[l][1, :, 3:], before[l][1, :, 3:])
    # a misaligned destination pointer in the array: that layer is skipped
    lib = kvd.load()
    arrays = [kvd.pointer_array(x, "cuda") for x in (ks, vs, kd, vd)]
    arrays[2][1] += 4
    before = kd[1].clone()
    status.zero_()
    n_ok = torch.tensor([2, 3], dtype=torch.int32, device="cuda")
    import ctypes
    st = lib.kvd_copy_prefix(*(ctypes.c_void_p(a.data_ptr()) for a in arrays), None,
                             ctypes.c_void_p(n_ok.data_ptr()), L, B, H, Cs, Cd, D, kvd.F32,
                             ctypes.c_void_p(status.data_ptr()), None)
    torch.cuda.synchronize()
    assert st == kvd.OK
    assert int(status.item()) & 64  # KVD_DEV_POINTER
    assert torch.equal(kd[1], before)
    assert torch.equal(kd[0][0, :, :2], ks[0][0, :, :2])
