"""GPU parity of the static-buffer path (append + masked split-KV attention +
combine) against the fp64 oracle, through the C ABI."""
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


def _run_masked(kvd, q, k, v, mask, scale, num_splits=0):
    dev = "cuda"
    qd, kd, vd, md = (t.to(dev).contiguous() for t in (q, k, v, mask))
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    status = kvd.status_tensor(dev)
    out = kvd.attend_masked(qd, kd, vd, md, scale, lse=lse, num_splits=num_splits,
                            dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, lse


def test_tiny_workload_fp32(kvd):
    """4-token prompt, appends at 4, 5, 6 with +-1e3 garbage in the padding
    (fp32, head_dim 64, capacity 32): append bit-exact, attention within the
    fp32 tolerance after every step."""
    k, v, mask, steps, scale = W.tiny()
    kd, vd, md = k.cuda(), v.cuda(), mask.cuda()
    kh, vh, mh = k.numpy().copy(), v.numpy().copy(), mask.numpy().copy()
    status = kvd.status_tensor()
    for st in steps:
        kvd.append(kd, vd, st["k_new"].cuda(), st["v_new"].cuda(), st["pos"].cuda(), md, status)
        assert oracle.append(kh, vh, st["k_new"], st["v_new"], st["pos"], mh) == 0
        torch.cuda.synchronize()
        assert np.array_equal(host(kd).numpy(), kh) and np.array_equal(host(vd).numpy(), vh)
        assert np.array_equal(host(md).numpy(), mh)
        lse = torch.empty(1, 4, device="cuda")
        out = kvd.attend_masked(st["q"].cuda(), kd, vd, md, scale, lse=lse, dev_status=status)
        ref, ref_lse = oracle.attend_masked(st["q"], torch.from_numpy(kh), torch.from_numpy(vh),
                                            torch.from_numpy(mh), scale)
        assert_attention_close(out, ref, torch.float32, f"tiny step pos={int(st['pos'])}")
        assert_lse_close(lse, ref_lse)
    assert int(status.item()) == 0


CASES = [
    # dtype, B, Hq, Hkv, C, D, lengths, num_splits
    (torch.bfloat16, 3, 8, 2, 1000, 128, [1000, 517, 1], 0),
    (torch.bfloat16, 2, 32, 8, 2048, 128, [2048, 777], 3),
    (torch.bfloat16, 2, 4, 4, 300, 64, [300, 33], 0),
    (torch.bfloat16, 1, 6, 2, 4100, 128, [4099], 0),
    (torch.float32, 2, 4, 1, 200, 64, [200, 65], 2),
    (torch.float32, 2, 8, 8, 96, 128, [96, 40], 0),
    (torch.bfloat16, 1, 16, 1, 640, 128, [639], 5),
    (torch.bfloat16, 2, 48, 3, 512, 64, [512, 100], 0),
]


@pytest.mark.parametrize("dtype,B,Hq,Hkv,C,D,lengths,num_splits", CASES)
def test_masked_parity(kvd, dtype, B, Hq, Hkv, C, D, lengths, num_splits):
    """Several tiles, ragged tails, several splits, group sizes 1..16."""
    g = W.generator(100 + C + Hq)
    q = W.randn(g, (B, Hq, D), dtype)
    k = W.randn(g, (B, Hkv, C, D), dtype)
    v = W.randn(g, (B, Hkv, C, D), dtype)
    mask = W.prefix_mask(lengths, C)
    scale = 1.0 / math.sqrt(D)
    out, lse = _run_masked(kvd, q, k, v, mask, scale, num_splits)
    ref, ref_lse = oracle.attend_masked(q, k, v, mask, scale)
    assert_attention_close(out, ref, dtype, "masked")
    assert_lse_close(lse, ref_lse, "masked lse")


def test_non_prefix_masks_and_skipped_tiles(kvd):
    """Random sparse masks, a history + current-slot mask, empty rows and
    mask runs that leave whole tiles empty."""
    B, Hq, Hkv, C, D = 5, 8, 2, 1500, 128
    g = W.generator(7)
    q = W.randn(g, (B, Hq, D))
    k = W.randn(g, (B, Hkv, C, D))
    v = W.randn(g, (B, Hkv, C, D))
    mask = torch.zeros(B, C, dtype=torch.uint8)
    mask[0] = (torch.rand(C, generator=g) < 0.05).to(torch.uint8)
    mask[1, :3] = 1
    mask[1, C - 1] = 1                       # history at the front, current slot last
    mask[2, 100:140] = 1
    mask[2, 1300:1301] = 1                   # tiles in between are all zero
    # row 3 stays empty
    mask[4] = 1
    out, lse = _run_masked(kvd, q, k, v, mask, 0.09)
    ref, ref_lse = oracle.attend_masked(q, k, v, mask, 0.09)
    assert_attention_close(out, ref, torch.bfloat16, "sparse masks")
    assert_lse_close(lse, ref_lse)
    assert torch.all(out[3] == 0) and torch.all(torch.isneginf(lse[3]))


@pytest.mark.parametrize("fill", [float("inf"), float("nan"), 1e3])
@pytest.mark.parametrize("Hq,Hkv", [(8, 4), (16, 2)])  # CUDA-core and tensor-core consumers
def test_garbage_padding_is_ignored(kvd, fill, Hq, Hkv):
    """inf / NaN / large values in mask = 0 slots leave the GPU result
    bit-identical to zero padding, and equal to the oracle within tolerance."""
    B, C, D = 2, 700, 128
    g = W.generator(8)
    q = W.randn(g, (B, Hq, D))
    k = W.randn(g, (B, Hkv, C, D))
    v = W.randn(g, (B, Hkv, C, D))
    mask = W.prefix_mask([650, 37], C)
    mask[0, 10] = 0
    pad = (mask == 0).view(B, 1, C, 1)
    out0, lse0 = _run_masked(kvd, q, k.masked_fill(pad, 0), v.masked_fill(pad, 0), mask, 0.1)
    out1, lse1 = _run_masked(kvd, q, k.masked_fill(pad, fill), v.masked_fill(pad, -fill), mask, 0.1)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    ref, _ = oracle.attend_masked(q, k.masked_fill(pad, fill), v.masked_fill(pad, fill), mask, 0.1)
    assert_attention_close(out1, ref, torch.bfloat16, "garbage")


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (16, 4), (8, 1)])
def test_single_valid_position_is_exact(kvd, Hq, Hkv):
    B, C, D = 2, 300, 128
    gs = Hq // Hkv
    g = W.generator(9)
    q = W.randn(g, (B, Hq, D))
    k = W.randn(g, (B, Hkv, C, D))
    v = W.randn(g, (B, Hkv, C, D))
    mask = torch.zeros(B, C, dtype=torch.uint8)
    mask[0, 0] = 1
    mask[1, 299] = 1
    for ns in (0, 3):
        out, _ = _run_masked(kvd, q, k, v, mask, 0.2, ns)
        out = host(out)
        for h in range(Hq):
            assert torch.equal(out[0, h], v[0, h // gs, 0])
            assert torch.equal(out[1, h], v[1, h // gs, 299])


def test_split_counts_agree(kvd):
    B, Hq, Hkv, C, D = 2, 8, 2, 3000, 128
    g = W.generator(10)
    q = W.randn(g, (B, Hq, D))
    k = W.randn(g, (B, Hkv, C, D))
    v = W.randn(g, (B, Hkv, C, D))
    mask = W.prefix_mask([3000, 1234], C)
    ref, _ = oracle.attend_masked(q, k, v, mask, 0.1)
    for ns in (1, 2, 5, 24):
        out, _ = _run_masked(kvd, q, k, v, mask, 0.1, ns)
        assert_attention_close(out, ref, torch.bfloat16, f"splits={ns}")


def test_append_bit_exact_and_position_errors(kvd):
    B, Hkv, C, D = 4, 8, 64, 128
    g = W.generator(11)
    k = W.randn(g, (B, Hkv, C, D))
    v = W.randn(g, (B, Hkv, C, D))
    kn = W.randn(g, (B, Hkv, D))
    vn = W.randn(g, (B, Hkv, D))
    mask = torch.zeros(B, C, dtype=torch.uint8)
    pos = torch.tensor([0, 63, C, -1], dtype=torch.int32)
    kd, vd, md = k.cuda(), v.cuda(), mask.cuda()
    status = kvd.status_tensor()
    kvd.append(kd, vd, kn.cuda(), vn.cuda(), pos.cuda(), md, status)
    kh = k.view(torch.int16).numpy().copy()
    vh = v.view(torch.int16).numpy().copy()
    mh = mask.numpy().copy()
    err = oracle.append(kh, vh, kn, vn, pos, mh)
    torch.cuda.synchronize()
    assert err == oracle.ERR_POS
    assert int(status.item()) == kvd.DEV_POS_RANGE
    assert np.array_equal(host(kd).view(torch.int16).numpy(), kh)
    assert np.array_equal(host(vd).view(torch.int16).numpy(), vh)
    assert np.array_equal(host(md).numpy(), mh)


def test_combine_matches_oracle(kvd):
    g = W.generator(12)
    R, S, D = 37, 9, 128
    po = W.randn(g, (R, S, D), torch.float32)
    pl = W.randn(g, (R, S), torch.float32) * 3
    pl[0, :] = float("-inf")
    pl[1, 3:] = float("-inf")
    po[1, 3:] = float("nan")  # empty ranges are not read
    lse = torch.empty(R, device="cuda")
    for odt in (torch.float32, torch.bfloat16):
        out = kvd.combine(po.cuda(), pl.cuda(), lse=lse, out_dtype=odt)
        ref, ref_lse = oracle.combine(po.double().numpy(), pl.double().numpy())
        assert_attention_close(out, ref, odt, "combine")
        assert_lse_close(lse, ref_lse)


def test_host_side_errors(kvd):
    q = torch.zeros(1, 4, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 3, 64, 128, dtype=torch.bfloat16, device="cuda")
    m = torch.ones(1, 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvd.KvdError) as e:
        kvd.attend_masked(q, k, k, m, 0.1)
    assert e.value.status == "KVD_ERR_INVALID_ARG"
    q2 = torch.zeros(1, 4, 96, dtype=torch.bfloat16, device="cuda")
    k2 = torch.zeros(1, 4, 64, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvd.KvdError) as e:
        kvd.attend_masked(q2, k2, k2, m, 0.1)
    assert e.value.status == "KVD_ERR_UNSUPPORTED"


@pytest.mark.parametrize("dtype,Hq,Hkv", [(torch.bfloat16, 8, 8), (torch.bfloat16, 8, 2),
                                          (torch.float32, 4, 4)])
def test_skip_scale_paths(kvd, dtype, Hq, Hkv):
    """Scores that climb slowly (the running max rises by less than the
    skip-scale threshold from tile to tile, so the stale max is kept over
    several tiles) and scores that jump (rescale taken), against the oracle.
    The scores are steered through dim 0 of q and k."""
    B, C, D = 3, 1536, 128
    g = W.generator(77, "cpu")
    q = W.randn(g, (B, Hq, D), dtype, scale=0.05)
    k = W.randn(g, (B, Hkv, C, D), dtype, scale=0.05)
    v = W.randn(g, (B, Hkv, C, D), dtype)
    q[:, :, 0] = 4.0
    t = torch.arange(C, dtype=torch.float32)
    # row 0: slow climb of ~0.4 natural-log units per 64 slots (the stale
    # max is kept for about fifteen tiles, then rescaled); row 1: a jump of ~8
    # at slot 1000 (rescaled at once); row 2: a descent (the first tile holds
    # the max).  Scores stay below ~10 so that the fp32 rounding of the scores
    # themselves stays inside the fp32 bar.
    k[0, :, :, 0] = (t * (0.4 / 64.0) * math.sqrt(D) / 4.0).to(dtype)
    k[1, :, :, 0] = torch.where(t >= 1000, 8.0 * math.sqrt(D) / 4.0, 0.0).to(dtype)
    k[2, :, :, 0] = ((C - t) * (0.25 / 64.0) * math.sqrt(D) / 4.0).to(dtype)
    mask = W.prefix_mask([C, 1300, 900], C)
    scale = 1.0 / math.sqrt(D)
    out, lse = _run_masked(kvd, q, k, v, mask, scale)
    ref, ref_lse = oracle.attend_masked(q, k, v, mask, scale)
    assert_attention_close(out, ref, dtype, "skip-scale")
    assert_lse_close(lse, ref_lse, "skip-scale")


@pytest.mark.parametrize("Hq,Hkv", [(32, 32), (32, 8), (16, 2)])
@pytest.mark.parametrize("start", [0, 40, 200, 1000])
def test_leading_tiles_empty_or_valid(kvd, Hq, Hkv, start):
    """Small launches (fewer units than scheduler warps) load the first tiles
    of a CTA's first unit before its mask is read: masks whose valid slots
    start inside or after that unit's tiles ([start, start + 150)), and one
    batch entry whose row is empty, give the oracle's result."""
    B, C, D = 2, 1152, 128
    g = W.generator(900 + start + Hq)
    q = W.randn(g, (B, Hq, D))
    k = W.randn(g, (B, Hkv, C, D))
    v = W.randn(g, (B, Hkv, C, D))
    mask = torch.zeros(B, C, dtype=torch.uint8)
    mask[0, start:start + 150] = 1
    out, lse = _run_masked(kvd, q, k, v, mask, 0.1)
    ref, ref_lse = oracle.attend_masked(q, k, v, mask, 0.1)
    assert_attention_close(out, ref, torch.bfloat16, f"leading tiles from {start}")
    assert_lse_close(lse, ref_lse)
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))


@pytest.mark.parametrize("Hq,Hkv,fused", [(32, 8, False), (32, 8, True), (32, 32, True)])
def test_large_launch_speculated_first_units(kvd, Hq, Hkv, fused):
    """Large launches load the first tiles of a CTA's first unit before its
    mask is read when that unit is a split-0 or split-1 unit.  Rows that are
    empty, hold one slot, or end inside split 0 leave those speculated units
    empty (delivered as empty tiles): every row still equals the oracle, in
    the two-call and the fused append form."""
    B, C, D = 16, 8192, 128
    g = W.generator(1960 + Hq + int(fused))
    q = W.randn(g, (B, Hq, D))
    k = W.randn(g, (B, Hkv, C, D))
    v = W.randn(g, (B, Hkv, C, D))
    # lengths cycle through empty, 1, inside split 0, inside split 1, long
    pattern = [0, 1, 100, 700, 5000, 8192, 37, 300]
    lengths = [pattern[b % len(pattern)] for b in range(B)]
    dev = "cuda"
    plan = kvd.attend_masked_plan(B, Hq, Hkv, C, D)
    assert plan.splits > 2 and plan.launches == 2  # the split kernel, many units
    status = kvd.status_tensor(dev)
    lse = torch.empty(B, Hq, device=dev)
    if fused:
        # the step appends at pos = length (the new slot), rows of length 0
        # get their first slot
        pos = torch.tensor([min(L, C - 1) for L in lengths], dtype=torch.int32)
        mask = W.prefix_mask(lengths, C)
        k_new = W.randn(g, (B, Hkv, D))
        v_new = W.randn(g, (B, Hkv, D))
        kh, vh, mh = k.view(torch.int16).numpy().copy(), v.view(torch.int16).numpy().copy(), \
            mask.numpy().copy()
        assert oracle.append(kh, vh, k_new, v_new, pos, mh) == 0
        kd, vd, md = k.to(dev), v.to(dev), mask.to(dev)
        out = kvd.append_attend_masked(q.to(dev), kd, vd, md, k_new.to(dev), v_new.to(dev),
                                       pos.to(dev), 0.09, lse=lse, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(host(md).numpy(), mh)
        ref, ref_lse = oracle.attend_masked(q, torch.from_numpy(kh).view(torch.bfloat16),
                                            torch.from_numpy(vh).view(torch.bfloat16),
                                            torch.from_numpy(mh), 0.09)
    else:
        mask = W.prefix_mask(lengths, C)
        out = kvd.attend_masked(q.to(dev), k.to(dev), v.to(dev), mask.to(dev), 0.09, lse=lse,
                                dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref, ref_lse = oracle.attend_masked(q, k, v, mask, 0.09)
    assert_attention_close(out, ref, torch.bfloat16, "speculated first units")
    assert_lse_close(lse, ref_lse, "speculated first units")


@pytest.mark.parametrize("dtype,Hq,Hkv,D", [
    (torch.float32, 16, 4, 128), (torch.float32, 16, 2, 64), (torch.bfloat16, 8, 4, 64),
    (torch.bfloat16, 4, 4, 64), (torch.bfloat16, 32, 4, 64), (torch.bfloat16, 24, 1, 128)])
def test_small_launch_matches_split_kernel(kvd, dtype, Hq, Hkv, D):
    """Short buffers take the small-launch kernel (one cluster per row, no
    combine); an explicit split count takes the split kernel.  Both equal the
    oracle, for every group width and head_dim."""
    B, C = 2, 700
    g = W.generator(950 + Hq + D)
    q = W.randn(g, (B, Hq, D), dtype)
    k = W.randn(g, (B, Hkv, C, D), dtype)
    v = W.randn(g, (B, Hkv, C, D), dtype)
    mask = W.prefix_mask([700, 413], C)
    mask[0, 300:360] = 0
    assert kvd.attend_masked_launches(B, Hq, Hkv, C, D, dtype) == 1
    ref, ref_lse = oracle.attend_masked(q, k, v, mask, 0.11)
    for ns in (0, 3):
        out, lse = _run_masked(kvd, q, k, v, mask, 0.11, ns)
        assert_attention_close(out, ref, dtype, f"num_splits {ns}")
        assert_lse_close(lse, ref_lse)


MERGE_CASES = [
    # dtype, B, Hq, Hkv, C, D, num_splits
    (torch.bfloat16, 4, 32, 8, 4096, 128, 0),     # tensor-core consumers
    (torch.bfloat16, 3, 16, 16, 6000, 64, 0),     # CUDA-core consumers, D 64
    (torch.float32, 2, 8, 2, 3000, 128, 24),      # fp32, explicit splits
    (torch.bfloat16, 1, 32, 32, 32768, 128, 0),   # 112 splits per row
]


@pytest.mark.parametrize("dtype,B,Hq,Hkv,C,D,ns", MERGE_CASES)
def test_split_merge_reuses_its_workspace(kvd, dtype, B, Hq, Hkv, C, D, ns):
    """Four calls on one workspace, lengths changing between them: every
    output matches the oracle and every call leaves the workspace's work
    counters at zero."""
    import math
    plan = kvd.attend_masked_plan(B, Hq, Hkv, C, D, dtype, ns)
    assert plan.splits > 1
    need = kvd.attend_masked_workspace_bytes(B, Hq, Hkv, C, D, dtype, ns)
    ws = kvd.workspace(need, "cuda")
    g = W.generator(7700 + C)
    q = W.randn(g, (B, Hq, D), dtype)
    k = W.randn(g, (B, Hkv, C, D), dtype)
    v = W.randn(g, (B, Hkv, C, D), dtype)
    kd, vd = k.cuda(), v.cuda()
    status = kvd.status_tensor()
    gl = W.generator(7800 + C)
    for call in range(4):
        lengths = [int(x) for x in W.randint(gl, B, 0 if call == 3 else 1, C)]
        mask = W.prefix_mask(lengths, C)
        lse = torch.empty(B, Hq, device="cuda")
        out = kvd.attend_masked(q.cuda(), kd, vd, mask.cuda(), 1.0 / math.sqrt(D), lse=lse,
                                num_splits=ns, workspace=ws, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert int(ws[:plan.counter_bytes].count_nonzero()) == 0, f"call {call}: counters left set"
        ref, ref_lse = oracle.attend_masked(q, k, v, mask, 1.0 / math.sqrt(D))
        assert_attention_close(out, ref, dtype, f"call {call}")
        assert_lse_close(lse, ref_lse, f"call {call}")
