"""GPU parity of the pieces of the sequence-axis split, through the C ABI.

kvd_attend_masked_partial (fp32 rows + log-sum-exp of one token range) and
kvd_combine_gathered (the merge of every range's packed block) against the
fp64 oracle: the attention over the whole sequence, and the oracle's
log-sum-exp combine ("Intel NPU running LLMs", Part 3, Flash SDPA path).
The ranges of several ranks are emulated on one GPU as separate slices of
the cache, each computed by its own call, merged by one combine call -- no
kernel waits on another.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from decode_attention_kv_gb300 import seqsplit
from parity_util import assert_attention_close, assert_lse_close, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvd():
    from decode_attention_kv_gb300 import kvd as _kvd
    _kvd.load()
    return _kvd


PARTIAL_CASES = [
    # dtype, B, Hq, Hkv, C, D, lengths, num_splits
    (torch.bfloat16, 1, 32, 32, 1152, 128, [1100], 0),      # one-launch cluster kernel
    (torch.bfloat16, 2, 32, 8, 8192, 128, [8192, 3000], 0),  # split kernel + combine
    (torch.float32, 2, 4, 2, 700, 64, [700, 0], 1),          # one split: rows written directly
    (torch.bfloat16, 1, 8, 8, 5000, 64, [4999], 0),          # CUDA-core consumers
]


@pytest.mark.parametrize("dtype,B,Hq,Hkv,C,D,lengths,ns", PARTIAL_CASES)
def test_partial_keeps_fp32_rows_and_lse(kvd, dtype, B, Hq, Hkv, C, D, lengths, ns):
    g = W.generator(5100 + C)
    q = W.randn(g, (B, Hq, D), dtype)
    k = W.randn(g, (B, Hkv, C, D), dtype)
    v = W.randn(g, (B, Hkv, C, D), dtype)
    mask = W.prefix_mask(lengths, C)
    status = kvd.status_tensor()
    out, lse = kvd.attend_masked_partial(q.cuda(), k.cuda(), v.cuda(), mask.cuda(),
                                         1.0 / math.sqrt(D), num_splits=ns, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert out.dtype == torch.float32
    ref, ref_lse = oracle.attend_masked(q, k, v, mask, 1.0 / math.sqrt(D))
    # fp32 rows: the fp32 bound for fp32 inputs; for bf16 inputs the rows are
    # never rounded to bf16, so the error is the kernel's fp32 (and bf16-p)
    # arithmetic alone, within the bf16 bound
    assert_attention_close(out, ref, dtype, "partial rows")
    assert_lse_close(lse, ref_lse, "partial lse")
    if dtype == torch.bfloat16:
        # not rounded to the bf16 grid: some element differs from its bf16 rounding
        o = host(out)
        assert not torch.equal(o, o.to(torch.bfloat16).float())


@pytest.mark.parametrize("R,S,D", [(7, 3, 128), (64, 2, 64), (512, 8, 128), (33, 1, 4)])
def test_combine_gathered_matches_the_oracle(kvd, R, S, D):
    g = W.generator(5200 + R * S)
    part_o = W.randn(g, (S, R, D), torch.float32)
    part_lse = W.randn(g, (S, R), torch.float32) * 3
    if S > 1:
        part_lse[0, ::3] = -math.inf               # empty ranges: weight 0
        part_o[0, ::3] = float("nan")              # whose rows are ignored
    part_lse[:, 1] = -math.inf                     # a row with every range empty
    parts = torch.cat([part_o.reshape(S, R * D), part_lse], dim=1).contiguous()
    assert parts.shape == (S, seqsplit.block_floats(R, D))
    lse = torch.empty(R, device="cuda")
    out = kvd.combine_gathered(parts.cuda(), R, D, lse=lse)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.combine(part_o.permute(1, 0, 2).double().numpy(),
                                  part_lse.t().double().numpy())
    assert np.all(host(out)[1].numpy() == 0)
    assert_attention_close(out, ref, torch.float32, "combine_gathered")
    assert_lse_close(lse, ref_lse, "combine_gathered lse")


SPLIT_CASES = [
    # dtype, B, Hq, Hkv, C, D, lengths, ranks
    (torch.bfloat16, 1, 32, 32, 32768, 128, [32768], 2),     # the long-context shape, two GPUs' share
    (torch.bfloat16, 4, 32, 8, 8192, 128, [8192, 5000, 700, 1], 4),
    (torch.float32, 2, 8, 2, 3000, 64, [3000, 1500], 3),     # entry 1 has no slot in the last range
]


@pytest.mark.parametrize("dtype,B,Hq,Hkv,C,D,lengths,ranks", SPLIT_CASES)
def test_ranges_merged_equal_the_unsplit_attention(kvd, dtype, B, Hq, Hkv, C, D, lengths, ranks):
    g = W.generator(5300 + C + ranks, "cuda")
    q = W.randn(g, (B, Hq, D), dtype, "cuda")
    k = W.randn(g, (B, Hkv, C, D), dtype, "cuda")
    v = W.randn(g, (B, Hkv, C, D), dtype, "cuda")
    mask = W.prefix_mask(lengths, C, "cuda")
    R = B * Hq
    parts = torch.empty((ranks, seqsplit.block_floats(R, D)), dtype=torch.float32, device="cuda")
    status = kvd.status_tensor()
    for r, (a, b) in enumerate(seqsplit.token_ranges(C, ranks)):
        rows, lse = seqsplit.block_views(parts[r], R, D)
        kvd.attend_masked_partial(q, k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous(),
                                  mask[:, a:b].contiguous(), 1.0 / math.sqrt(D),
                                  out=rows.view(B, Hq, D), lse=lse.view(B, Hq), dev_status=status)
    out = torch.empty_like(q)
    lse = torch.empty(B, Hq, device="cuda")
    kvd.combine_gathered(parts, R, D, out=out.view(R, D), lse=lse.view(R))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse = oracle.attend_masked(host(q), host(k), host(v), host(mask), 1.0 / math.sqrt(D))
    assert_attention_close(out, ref, dtype, f"{ranks} ranges merged")
    assert_lse_close(lse, ref_lse, f"{ranks} ranges merged, lse")


def test_one_rank_module_equals_the_plain_call(kvd):
    """SequenceSplitAttention without a process group (one rank) is the
    plain attention: the exchange hands back the rank's own block."""
    B, Hq, Hkv, C, D = 2, 16, 4, 2048, 128
    g = W.generator(5400, "cuda")
    q = W.randn(g, (B, Hq, D), torch.bfloat16, "cuda")
    k = W.randn(g, (B, Hkv, C, D), torch.bfloat16, "cuda")
    v = W.randn(g, (B, Hkv, C, D), torch.bfloat16, "cuda")
    mask = W.prefix_mask([2048, 999], C, "cuda")
    att = seqsplit.SequenceSplitAttention(B, Hq, D, device="cuda")
    lse = torch.empty(B, Hq, device="cuda")
    out = att(q, k, v, mask, 1.0 / math.sqrt(D), lse=lse)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attend_masked(host(q), host(k), host(v), host(mask), 1.0 / math.sqrt(D))
    assert_attention_close(out, ref, torch.bfloat16, "one-rank module")
    assert_lse_close(lse, ref_lse, "one-rank module lse")
