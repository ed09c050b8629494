"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (library-planned splits), on outputs sampled so that the
fp64 oracle computes them one by one in seconds.

Workloads (see workloads.py): the 1152-slot static buffer (MHA 32 x 128,
bf16), batched GQA (16 x 32/8 heads, capacity 8192, lengths 512..8192), the
paged cache (8192 blocks of 128 slots x 8 heads x 128, 64 sequences of
1..4096 tokens) and the 32768-token single sequence.
"""
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
    return host(t).view(torch.int16).numpy()


def _masked_step_and_check(kvd, lay, sample, what):
    """Append + attend one layer on the GPU; check the append byte for byte
    over the whole cache and the attention on the sampled (b, h) rows."""
    dev = "cuda"
    B, Hkv, C, D = lay.k_cache.shape
    Hq = lay.q.shape[1]
    g = Hq // Hkv
    kh, vh, mh = _bits(lay.k_cache).copy(), _bits(lay.v_cache).copy(), host(lay.mask).numpy().copy()
    status = kvd.status_tensor(dev)
    kvd.append(lay.k_cache, lay.v_cache, lay.k_new, lay.v_new, lay.pos, lay.mask, status)
    lse = torch.empty(B, Hq, device=dev)
    out = kvd.attend_masked(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.scale, lse=lse,
                            dev_status=status)
    assert oracle.append(kh, vh, host(lay.k_new), host(lay.v_new), host(lay.pos), mh) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(_bits(lay.k_cache), kh), f"{what}: append (K) not bit-exact"
    assert np.array_equal(_bits(lay.v_cache), vh), f"{what}: append (V) not bit-exact"
    assert np.array_equal(host(lay.mask).numpy(), mh)
    qh = host(lay.q)
    outs, refs, lses, rlses = [], [], [], []
    for b, h in sample:
        kvh = h // g
        ref, rl = oracle.attend_masked(
            qh[b:b + 1, h:h + 1], torch.from_numpy(kh[b:b + 1, kvh:kvh + 1]).view(torch.bfloat16),
            torch.from_numpy(vh[b:b + 1, kvh:kvh + 1]).view(torch.bfloat16),
            torch.from_numpy(mh[b:b + 1]), lay.scale, nthreads=0)
        outs.append(out[b, h])
        refs.append(ref[0, 0])
        lses.append(lse[b, h])
        rlses.append(rl[0, 0])
    assert_attention_close(torch.stack(outs), np.stack(refs), torch.bfloat16, what)
    assert_lse_close(torch.stack(lses), np.array(rlses), what)


def test_npuw_default_buffer_steps(kvd):
    """1152-slot buffer: four decode steps (appends at 1024..1027), all 32
    heads compared after each."""
    w = W.npuw(device="cuda", layers=1)
    lay = w.layers[0]
    g = W.generator(77, "cuda")
    for step in range(4):
        if step:
            lay.q = W.randn(g, lay.q.shape, torch.bfloat16, "cuda")
            lay.k_new = W.randn(g, lay.k_new.shape, torch.bfloat16, "cuda")
            lay.v_new = W.randn(g, lay.v_new.shape, torch.bfloat16, "cuda")
            lay.pos = lay.pos + 1
        _masked_step_and_check(kvd, lay, [(0, h) for h in range(32)], f"npuw step {step}")
        assert int(host(lay.mask).sum()) == 1025 + step


def test_batched_gqa_full_size(kvd):
    w = W.gqa(device="cuda", layers=1)
    lay = w.layers[0]
    L = lay.lengths
    order = torch.argsort(L)
    bs = [int(order[0]), int(order[1]), int(order[len(order) // 2]), int(order[-1])]
    sample = [(b, h) for b in bs for h in (0, 3, 4, 17, 31)]
    _masked_step_and_check(kvd, lay, sample, "gqa")


def test_long_context_full_size(kvd):
    w = W.long(device="cuda", layers=1)
    lay = w.layers[0]
    _masked_step_and_check(kvd, lay, [(0, h) for h in (0, 5, 13, 31)], "long")


def test_paged_full_size(kvd):
    pw = W.paged(device="cuda")
    status = kvd.status_tensor()
    lse = torch.empty(pw.q.shape[:2], device="cuda")
    out = kvd.attend_paged(pw.q, pw.key_cache, pw.value_cache, pw.block_tables, pw.seq_lens,
                           pw.seq_offset, pw.scale, lse=lse, dev_status=status)
    ko, vo = kvd.gather_paged(pw.key_cache, pw.value_cache, pw.block_tables, pw.seq_lens,
                              pw.seq_offset, total_tokens=pw.total_tokens, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert ko.shape == (pw.total_tokens, 8, 128)
    L = pw.lengths
    order = torch.argsort(L)
    sample = [int(order[0]), int(order[1]), int(order[32]), int(order[-2]), int(order[-1])]
    bt = host(pw.block_tables)
    sl = host(pw.seq_lens)
    for q in sample:
        n = int(L[q])
        nblk = (n + 127) // 128
        idx = bt[q, :nblk].long()
        kq = host(pw.key_cache.index_select(0, idx.cuda()))
        vq = host(pw.value_cache.index_select(0, idx.cuda()))
        bt_q = torch.arange(nblk, dtype=torch.int32)[None]
        sl_q = torch.tensor([0, n], dtype=torch.int32)
        ref, rl = oracle.attend_paged(host(pw.q[q:q + 1]), kq, vq, bt_q, sl_q, None, pw.scale)
        assert_attention_close(out[q:q + 1], ref, torch.bfloat16, f"paged seq {q} (len {n})")
        assert_lse_close(lse[q:q + 1], rl)
        rk, rv, err = oracle.gather_paged(kq.view(torch.int16).numpy(), vq.view(torch.int16).numpy(),
                                          bt_q, sl_q)
        assert err == 0
        s0 = int(sl[q])
        assert np.array_equal(_bits(ko[s0:s0 + n]), rk), f"gather seq {q}"
        assert np.array_equal(_bits(vo[s0:s0 + n]), rv), f"gather seq {q}"


@pytest.mark.parametrize("name", ["gqa", "long"])
def test_full_size_attention_finishes_far_below_the_wait_limit(kvd, name):
    """A full-size launch takes well under a millisecond of HBM time; one that
    takes anywhere near the kernels' one-second wait limit means some CTA sat
    in a bounded wait (a pipeline bug even if the result is right)."""
    import time
    lay = getattr(W, name)(device="cuda", layers=1).layers[0]
    status = kvd.status_tensor()
    out = torch.empty_like(lay.q)
    kvd.attend_masked(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.scale, out=out,
                      dev_status=status)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(3):
        kvd.attend_masked(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.scale, out=out,
                          dev_status=status)
    torch.cuda.synchronize()
    per_call = (time.perf_counter() - t0) / 3
    assert int(status.item()) == 0
    assert per_call < 0.05, f"{name}: {per_call * 1e3:.1f} ms per attention call"
