"""The sequence-axis split of one decode step across ranks, on the CPU.

Host logic of decode_attention_kv_gb300.seqsplit: the token ranges, the
packed exchange block and the all-gather, run as world-size-2 gloo ranks.
Each rank's partial over its own range comes from the fp64 oracle (rounded
to fp32, as the exchange block holds it); the gathered blocks are merged by
the oracle's log-sum-exp combine and checked against the oracle's attention
over the whole, unsplit sequence ("Intel NPU running LLMs", Part 3, Flash
SDPA path: tiles -- here ranges held by different ranks -- merge exactly
through their running max and sum).  No GPU.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from decode_attention_kv_gb300 import seqsplit  # noqa: E402


def test_token_ranges_cover_the_sequence_in_aligned_pieces():
    for C, world, align in [(32768, 2, 64), (32768, 8, 64), (1000, 3, 64), (100, 4, 64),
                            (7, 2, 1), (0, 2, 64), (4096, 1, 128)]:
        rs = seqsplit.token_ranges(C, world, align)
        assert len(rs) == world
        assert rs[0][0] == 0 and rs[-1][1] == C
        for (a, b), (c, d) in zip(rs, rs[1:]):
            assert b == c  # contiguous, no overlap
        for a, b in rs:
            assert a <= b
            assert a % align == 0 or a == C
        sizes = [b - a for a, b in rs]
        assert max(sizes) - min(sizes) <= align * 2 or C < world * align
    assert seqsplit.token_ranges(32768, 2) == [(0, 16384), (16384, 32768)]
    with pytest.raises(ValueError):
        seqsplit.token_ranges(10, 0)


def test_block_layout():
    R, D = 6, 8
    blk = torch.arange(seqsplit.block_floats(R, D), dtype=torch.float32)
    rows, lse = seqsplit.block_views(blk, R, D)
    assert rows.shape == (R, D) and lse.shape == (R,)
    assert rows[2, 3].item() == 2 * D + 3 and lse[1].item() == R * D + 1
    assert seqsplit.exchange(blk).shape == (1, blk.numel())  # one rank: no process group
    with pytest.raises(ValueError):
        seqsplit.block_views(blk[:-1], R, D)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


# B, Hq, Hkv, C, D, dtype, valid lengths, world; the second case leaves the
# last rank's range without a valid slot for one batch entry (lse = -inf).
CASES = [
    (2, 8, 2, 300, 64, torch.float32, [300, 211], 2),
    (2, 4, 4, 640, 128, torch.bfloat16, [640, 100], 2),
    (1, 6, 3, 1000, 64, torch.float32, [999], 3),
]


def _inputs(B, Hq, Hkv, C, D, dtype, lengths):
    import workloads as W
    g = W.generator(4242 + C)
    q = W.randn(g, (B, Hq, D), dtype)
    k = W.randn(g, (B, Hkv, C, D), dtype)
    v = W.randn(g, (B, Hkv, C, D), dtype)
    mask = W.prefix_mask(lengths, C)
    return q, k, v, mask


def _worker(rank, world, port, case, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        B, Hq, Hkv, C, D, dtype, lengths, _ = case
        q, k, v, mask = _inputs(B, Hq, Hkv, C, D, dtype, lengths)
        start, stop = seqsplit.token_ranges(C, world)[rank]
        # this rank's slice of the cache and mask, its own contiguous buffers
        ks = k[:, :, start:stop].contiguous()
        vs = v[:, :, start:stop].contiguous()
        ms = mask[:, start:stop].contiguous()
        R = B * Hq
        blk = torch.empty(seqsplit.block_floats(R, D), dtype=torch.float32)
        rows, lse = seqsplit.block_views(blk, R, D)
        po, pl = oracle.attend_masked(q, ks, vs, ms, 1.0 / np.sqrt(D))
        rows.copy_(torch.from_numpy(po.reshape(R, D)))
        lse.copy_(torch.from_numpy(pl.reshape(R)))
        gathered = seqsplit.exchange(blk)
        out[rank] = gathered.numpy().copy()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", CASES)
def test_sequence_split_over_gloo_ranks_matches_the_unsplit_oracle(case):
    import oracle
    B, Hq, Hkv, C, D, dtype, lengths, world = case
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, case, out), nprocs=world,
                       start_method="spawn", join=True)
    R = B * Hq
    # every rank gathered the same blocks
    for r in range(1, world):
        assert np.array_equal(out[r], out[0])
    g = out[0]
    assert g.shape == (world, seqsplit.block_floats(R, D))
    part_o = np.stack([g[s, :R * D].reshape(R, D) for s in range(world)], axis=1)  # [R, S, D]
    part_lse = np.stack([g[s, R * D:] for s in range(world)], axis=1)             # [R, S]
    merged, merged_lse = oracle.combine(part_o.astype(np.float64), part_lse.astype(np.float64))
    q, k, v, mask = _inputs(B, Hq, Hkv, C, D, dtype, lengths)
    ref, ref_lse = oracle.attend_masked(q, k, v, mask, 1.0 / np.sqrt(D))
    # the only error is the fp32 rounding of the exchanged partials
    assert np.max(np.abs(merged - ref.reshape(R, D))) <= 1e-6 * max(1.0, np.abs(ref).max())
    assert np.max(np.abs(merged_lse - ref_lse.reshape(R))) <= 1e-5
    if lengths[-1] <= seqsplit.token_ranges(C, world)[-1][0]:
        # the last range of the last batch entry holds no valid slot
        assert np.all(np.isneginf(part_lse[-Hq:, -1]))
