"""Parity at the workloads' full sizes, in the launch configurations the
benchmark times (library-planned splits), every output element compared.

Workloads (see workloads.py): the 1152-slot static buffer (MHA 32 x 128,
bf16), batched GQA (16 x 32/8 heads, capacity 8192, lengths 512..8192), the
paged cache (8192 blocks of 128 slots x 8 heads x 128, 64 sequences of
1..4096 tokens; also over E4M3 and E2M1 rows), the 32768-token single
sequence and its 4096-slot sliding window.  The static-buffer steps run both ways a caller can run them: the
append and the attention as two calls, and the fused call the benchmark
times (the append inside the attention launch).  The fp64 oracle computes
the whole layer (every batch entry, every head) on the host cores.
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


def _masked_step_and_check(kvd, lay, what, fused, window=0):
    """Append + attend one layer on the GPU (two calls, or the fused call;
    with ``window``, the sliding-window entries ending at the appended slot);
    the append compared byte for byte over the whole cache and mask, the
    attention over every (batch entry, head) against the oracle's append
    followed by its attention."""
    dev = "cuda"
    B, Hkv, C, D = lay.k_cache.shape
    Hq = lay.q.shape[1]
    kh, vh, mh = _bits(lay.k_cache).copy(), _bits(lay.v_cache).copy(), host(lay.mask).numpy().copy()
    status = kvd.status_tensor(dev)
    lse = torch.empty(B, Hq, device=dev)
    if fused and window:
        out = kvd.append_attend_window(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.k_new,
                                       lay.v_new, lay.pos, window, lay.scale, lse=lse,
                                       dev_status=status)
    elif fused:
        out = kvd.append_attend_masked(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.k_new,
                                       lay.v_new, lay.pos, lay.scale, lse=lse, dev_status=status)
    else:
        kvd.append(lay.k_cache, lay.v_cache, lay.k_new, lay.v_new, lay.pos, lay.mask, status)
        if window:
            out = kvd.attend_window(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.pos, window,
                                    lay.scale, lse=lse, dev_status=status)
        else:
            out = kvd.attend_masked(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.scale,
                                    lse=lse, dev_status=status)
    assert oracle.append(kh, vh, host(lay.k_new), host(lay.v_new), host(lay.pos), mh) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(_bits(lay.k_cache), kh), f"{what}: append (K) not bit-exact"
    assert np.array_equal(_bits(lay.v_cache), vh), f"{what}: append (V) not bit-exact"
    assert np.array_equal(host(lay.mask).numpy(), mh), f"{what}: mask after the append"
    kr, vr = torch.from_numpy(kh).view(torch.bfloat16), torch.from_numpy(vh).view(torch.bfloat16)
    if window:
        ref, rl, err = oracle.attend_window(host(lay.q), kr, vr, torch.from_numpy(mh),
                                            host(lay.pos), window, lay.scale)
        assert err == 0
    else:
        ref, rl = oracle.attend_masked(host(lay.q), kr, vr, torch.from_numpy(mh), lay.scale)
    assert_attention_close(out, ref, torch.bfloat16, what)
    assert_lse_close(lse, rl, what)


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
def test_npuw_default_buffer_steps(kvd, fused):
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
        _masked_step_and_check(kvd, lay, f"npuw step {step}", fused)
        assert int(host(lay.mask).sum()) == 1025 + step


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
def test_batched_gqa_full_size(kvd, fused):
    """All 16 batch entries x 32 query heads (512 rows)."""
    lay = W.gqa(device="cuda", layers=1).layers[0]
    _masked_step_and_check(kvd, lay, "gqa", fused)


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
def test_long_context_full_size(kvd, fused):
    """All 32 heads of the 32768-slot sequence.  The fused call runs the
    append inside the persistent split kernel with CUDA-core consumers (one
    query head per kv head), in the launch the benchmark times."""
    lay = W.long(device="cuda", layers=1).layers[0]
    _masked_step_and_check(kvd, lay, "long", fused)


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
def test_window_full_size(kvd, fused):
    """The 32768-slot sequence with its 4096-slot window, appended at C - 1:
    all 32 heads; the window is the mask after the append."""
    lay = W.window(device="cuda", layers=1).layers[0]
    _masked_step_and_check(kvd, lay, "window", fused)
    mask = host(lay.mask)
    assert int(mask.sum()) == 4096 and int(mask[0, -1]) == 1 and int(mask[0, -4096]) == 1


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
@pytest.mark.parametrize("mask", ["window", "prefix"])
def test_window_entry_full_size(kvd, fused, mask):
    """The sliding-window entries on the 32768-slot sequence, window 4096
    ending at the slot appended at C - 1: over the workload's own mask (the
    benchmark's step), and over the whole prefix, where the window alone
    selects the 4096 newest slots.  All 32 heads."""
    w = W.window(device="cuda", layers=1)
    lay = w.layers[0]
    if mask == "prefix":
        lay.mask = W.prefix_mask([w.C - 1], w.C, "cuda")
    _masked_step_and_check(kvd, lay, f"window entry, {mask} mask", fused, window=w.window)


def test_paged_full_size(kvd):
    """All 64 sequences x 32 query heads of paged attention; the whole
    gathered K and V buffers byte for byte."""
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
    kc, vc = host(pw.key_cache), host(pw.value_cache)
    bt, sl, so = host(pw.block_tables), host(pw.seq_lens), host(pw.seq_offset)
    ref, rl = oracle.attend_paged(host(pw.q), kc, vc, bt, sl, so, pw.scale)
    assert_attention_close(out, ref, torch.bfloat16, "paged attention, all sequences")
    assert_lse_close(lse, rl, "paged attention lse")
    rk, rv, err = oracle.gather_paged(kc.view(torch.int16).numpy(), vc.view(torch.int16).numpy(),
                                      bt, sl, so)
    assert err == 0
    assert np.array_equal(_bits(ko), rk), "gather: key buffer not bit-exact"
    assert np.array_equal(_bits(vo), rv), "gather: value buffer not bit-exact"


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
def test_paged_quant_full_size(kvd, fmt):
    """The paged workload over E4M3 / E2M1 rows, as the benchmark's step
    runs it: the quantising paged append of every sequence's last token
    (both caches byte for byte), then the paged attention of all 64
    sequences x 32 query heads."""
    pw = W.paged_quant(fmt, device="cuda")
    kh, vh = host(pw.key_cache).numpy().copy(), host(pw.value_cache).numpy().copy()
    status = kvd.status_tensor()
    append = kvd.append_paged_fp8 if fmt == "fp8" else kvd.append_paged_fp4
    append(pw.key_cache, pw.value_cache, pw.block_tables, pw.seq_offset, pw.k_new, pw.v_new,
           pw.pos, dev_status=status)
    lse = torch.empty(pw.q.shape[:2], device="cuda")
    out = kvd.attend_paged_quant(fmt, pw.q, pw.key_cache, pw.value_cache, pw.block_tables,
                                 pw.seq_lens, pw.seq_offset, pw.scale, lse=lse, dev_status=status)
    bt, sl, so = host(pw.block_tables), host(pw.seq_lens), host(pw.seq_offset)
    assert oracle.append_paged_quant(kh, vh, bt, so, host(pw.k_new), host(pw.v_new),
                                     host(pw.pos), fmt) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(host(pw.key_cache).numpy(), kh), f"paged {fmt} append (K)"
    assert np.array_equal(host(pw.value_cache).numpy(), vh), f"paged {fmt} append (V)"
    ref, rl = oracle.attend_paged_quant(host(pw.q), kh, vh, bt, sl, so, pw.scale, fmt)
    assert_attention_close(out, ref, torch.bfloat16, f"paged {fmt} attention, all sequences")
    assert_lse_close(lse, rl, f"paged {fmt} attention lse")


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
