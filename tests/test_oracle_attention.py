"""Pins of the fp64 oracle's masked decode attention (CPU only).

Each test fixes the oracle against something other than itself: a closed
form, an invariant the pages state, the pages' printed examples, or a library
routine.  Chosen so that a dropped term, a wrong sign or index, a wrong head
mapping or a forgotten mask fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(seed, B=2, Hq=4, Hkv=2, C=37, D=16, dtype=torch.float32, lengths=None):
    g = W.generator(seed)
    q = W.randn(g, (B, Hq, D), dtype)
    k = W.randn(g, (B, Hkv, C, D), dtype)
    v = W.randn(g, (B, Hkv, C, D), dtype)
    if lengths is None:
        lengths = [C - 5 - b for b in range(B)]
    mask = W.prefix_mask(lengths, C)
    return q, k, v, mask, lengths


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_prefix_recompute_equals_masked(oracle, dtype):
    """Masked full-capacity result == unmasked attention over the valid prefix
    only (the static buffer + mask design of the NPU article, Part 1)."""
    q, k, v, mask, lengths = _rand_case(1, dtype=dtype)
    out, lse = oracle.attend_masked(q, k, v, mask, 0.25)
    for b, L in enumerate(lengths):
        ob, lb = oracle.attend_masked(q[b:b + 1], k[b:b + 1, :, :L].contiguous(),
                                      v[b:b + 1, :, :L].contiguous(),
                                      torch.ones(1, L, dtype=torch.uint8), 0.25)
        assert np.array_equal(ob[0], out[b])
        assert np.array_equal(lb[0], lse[b])


@pytest.mark.parametrize("fill", [1e3, -1e3, float("inf"), float("-inf"), float("nan")])
def test_garbage_in_padding_is_ignored(oracle, fill):
    """Any content of mask=0 slots leaves the result bit-identical."""
    q, k, v, mask, _ = _rand_case(2)
    ref, ref_lse = oracle.attend_masked(q, k, v, mask, 0.3)
    pad = (mask == 0).view(mask.shape[0], 1, mask.shape[1], 1)
    k2 = k.masked_fill(pad, fill)
    v2 = v.masked_fill(pad, -fill if not math.isnan(fill) else fill)
    out, lse = oracle.attend_masked(q, k2, v2, mask, 0.3)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


def test_single_valid_position_returns_its_v_row(oracle):
    q, k, v, _, _ = _rand_case(3, B=1, Hq=4, Hkv=2, C=29, D=8)
    for t in (0, 13, 28):
        mask = torch.zeros(1, 29, dtype=torch.uint8)
        mask[0, t] = 1
        out, lse = oracle.attend_masked(q, k, v, mask, 0.7)
        for h in range(4):
            assert np.array_equal(out[0, h], v[0, h // 2, t].double().numpy())
            s = 0.7 * float(np.dot(q[0, h].double().numpy(), k[0, h // 2, t].double().numpy()))
            assert lse[0, h] == pytest.approx(s, rel=1e-14, abs=1e-14)


def test_identical_keys_give_mean_of_valid_rows(oracle):
    """Equal scores -> uniform weights -> arithmetic mean of the valid V rows;
    lse = s + log(n)."""
    g = W.generator(4)
    B, Hq, Hkv, C, D = 1, 2, 1, 19, 12
    q = W.randn(g, (B, Hq, D), torch.float32)
    k = W.randn(g, (B, Hkv, 1, D), torch.float32).expand(B, Hkv, C, D).contiguous()
    v = W.randn(g, (B, Hkv, C, D), torch.float32)
    mask = torch.zeros(B, C, dtype=torch.uint8)
    valid = [1, 4, 5, 11, 18]
    mask[0, valid] = 1
    out, lse = oracle.attend_masked(q, k, v, mask, 0.9)
    mean = v[0, 0, valid].double().numpy().mean(axis=0)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], mean, rtol=1e-13, atol=1e-13)
        s = 0.9 * float(q[0, h].double() @ k[0, 0, 0].double())
        assert lse[0, h] == pytest.approx(s + math.log(len(valid)), rel=1e-13)


@pytest.mark.parametrize("scale", [0.125, -0.5, 1.0])
def test_two_positions_logistic_weights(oracle, scale):
    """Two valid keys: weights sigma(s1 - s2) and 1 - sigma(s1 - s2)."""
    D = 8
    q = torch.zeros(1, 1, D)
    q[0, 0, 0] = 2.0
    q[0, 0, 3] = -1.0
    k = torch.zeros(1, 1, 6, D)
    k[0, 0, 1, 0] = 3.0        # q.k1 = 6
    k[0, 0, 4, 3] = 2.0        # q.k2 = -2
    k[0, 0, 2] = 1e3           # masked out
    v = torch.arange(6 * D, dtype=torch.float32).reshape(1, 1, 6, D) / 7.0
    mask = torch.tensor([[0, 1, 0, 0, 1, 0]], dtype=torch.uint8)
    out, lse = oracle.attend_masked(q, k, v, mask, scale)
    s1, s2 = 6.0 * scale, -2.0 * scale
    w1 = 1.0 / (1.0 + math.exp(-(s1 - s2)))
    expect = w1 * v[0, 0, 1].double().numpy() + (1.0 - w1) * v[0, 0, 4].double().numpy()
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-13, atol=1e-13)
    assert lse[0, 0] == pytest.approx(math.log(math.exp(s1) + math.exp(s2)), rel=1e-13)


def test_zero_scale_is_uniform_mean(oracle):
    q, k, v, mask, lengths = _rand_case(5)
    out, _ = oracle.attend_masked(q, k, v, mask, 0.0)
    for b, L in enumerate(lengths):
        for h in range(q.shape[1]):
            mean = v[b, h // 2, :L].double().numpy().mean(axis=0)
            np.testing.assert_allclose(out[b, h], mean, rtol=1e-12, atol=1e-13)


def test_permutation_invariance(oracle):
    q, k, v, mask, _ = _rand_case(6)
    mask = mask.clone()
    mask[0, 3] = 0  # make it non-prefix
    perm = torch.randperm(k.shape[2], generator=W.generator(7))
    out, lse = oracle.attend_masked(q, k, v, mask, 0.4)
    out2, lse2 = oracle.attend_masked(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(),
                                      mask[:, perm].contiguous(), 0.4)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=1e-12, atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv(oracle):
    """Query head h reads kv head h // g: same as MHA on repeat-interleaved K/V."""
    q, k, v, mask, _ = _rand_case(8, Hq=6, Hkv=2)
    out, lse = oracle.attend_masked(q, k, v, mask, 0.5)
    k3 = k.repeat_interleave(3, dim=1).contiguous()
    v3 = v.repeat_interleave(3, dim=1).contiguous()
    out2, lse2 = oracle.attend_masked(q, k3, v3, mask, 0.5)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_matches_torch_sdpa_float64(oracle, dtype):
    """Library cross-check: torch's scaled_dot_product_attention in float64
    with a boolean mask (keys with mask=0 not attended)."""
    q, k, v, mask, _ = _rand_case(9, B=3, Hq=8, Hkv=2, C=53, D=32, dtype=dtype,
                                  lengths=[53, 20, 1])
    mask[1, 7] = 0
    out, lse = oracle.attend_masked(q, k, v, mask, 0.17)
    g = q.shape[1] // k.shape[1]
    kk = k.double().repeat_interleave(g, 1)
    vv = v.double().repeat_interleave(g, 1)
    am = (mask != 0).view(mask.shape[0], 1, 1, mask.shape[1])
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.double().unsqueeze(2), kk, vv, attn_mask=am, scale=0.17).squeeze(2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    s = torch.einsum("bhd,bhtd->bht", q.double(), kk) * 0.17
    s = s.masked_fill(~am.squeeze(2), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=1e-12, atol=1e-12)


def test_empty_row_gives_zero_and_minus_inf(oracle):
    q, k, v, mask, _ = _rand_case(10)
    mask[1] = 0
    k[1] = float("nan")
    out, lse = oracle.attend_masked(q, k, v, mask, 0.3)
    assert np.all(out[1] == 0.0) and np.all(lse[1] == -np.inf)
    assert np.all(np.isfinite(out[0]))


def test_generate_loop_mask_from_the_page(oracle):
    """The page's generate-loop mask (history at the front, the current token in
    the last slot) equals prefix attention over [history..., current]."""
    spec = json.load(open(os.path.join(GOLDEN, "generate_loop_mask.json")))
    g = W.generator(11)
    H, D = 2, 16
    for st in spec["steps"]:
        C = st["history"] + st["zeros"] + st["current"]
        q = W.randn(g, (1, H, D), torch.bfloat16)
        k = W.randn(g, (1, H, C, D), torch.bfloat16)
        v = W.randn(g, (1, H, C, D), torch.bfloat16)
        mask = torch.zeros(1, C, dtype=torch.uint8)
        mask[0, :st["history"]] = 1
        mask[0, C - st["current"]:] = 1
        out, _ = oracle.attend_masked(q, k, v, mask, 1 / 4)
        idx = list(range(st["history"])) + list(range(C - st["current"], C))
        n = len(idx)
        out2, _ = oracle.attend_masked(q, k[:, :, idx].contiguous(), v[:, :, idx].contiguous(),
                                       torch.ones(1, n, dtype=torch.uint8), 1 / 4)
        np.testing.assert_allclose(out, out2, rtol=1e-13, atol=1e-14)


def test_tiny_workload_flow(oracle):
    """4-token prompt then 3 appends (pos 4, 5, 6): each step's masked result
    equals attention over the prompt rows plus the appended rows, and the
    +-1e3 padding garbage never leaks in."""
    k, v, mask, steps, scale = W.tiny()
    kc = k.numpy().copy()
    vc = v.numpy().copy()
    m = mask.numpy().copy()
    rows_k = [k[0, :, t].numpy() for t in range(4)]
    rows_v = [v[0, :, t].numpy() for t in range(4)]
    for st in steps:
        assert oracle.append(kc, vc, st["k_new"], st["v_new"], st["pos"], m) == 0
        rows_k.append(st["k_new"][0].numpy())
        rows_v.append(st["v_new"][0].numpy())
        assert int(m.sum()) == st["length"]
        out, _ = oracle.attend_masked(st["q"], torch.from_numpy(kc), torch.from_numpy(vc),
                                      torch.from_numpy(m), scale)
        kk = torch.from_numpy(np.stack(rows_k, axis=1))[None]
        vv = torch.from_numpy(np.stack(rows_v, axis=1))[None]
        ref, _ = oracle.attend_masked(st["q"], kk, vv, torch.ones(1, st["length"],
                                                                  dtype=torch.uint8), scale)
        assert np.array_equal(out, ref)
        assert np.abs(out).max() < 10.0


# ------------------------------------------------------------ index lists

def test_indexed_with_unique_indices_is_masked_attention(oracle):
    """FlashMLA on Ascend, 'Математическая постановка': attention over the
    gathered top-k rows.  With unique indices this is masked attention with
    the mask that marks exactly those slots (the masked oracle is pinned on
    its own)."""
    g = W.generator(41)
    B, Hq, Hkv, C, D = 2, 4, 2, 50, 8
    q = W.randn(g, (B, Hq, D), torch.float32)
    k = W.randn(g, (B, Hkv, C, D), torch.float32)
    v = W.randn(g, (B, Hkv, C, D), torch.float32)
    idx = torch.stack([torch.randperm(C, generator=g)[:12] for _ in range(B)]).to(torch.int32)
    mask = torch.zeros(B, C, dtype=torch.uint8)
    for b in range(B):
        mask[b, idx[b].long()] = 1
    out, lse, err = oracle.attend_indexed(q, k, v, idx, 0.3)
    ref, ref_lse = oracle.attend_masked(q, k, v, mask, 0.3)
    assert err == 0
    assert np.allclose(out, ref, rtol=0, atol=1e-13) and np.allclose(lse, ref_lse, rtol=0, atol=1e-13)


def test_indexed_repeats_unused_entries_and_order(oracle):
    """A repeated entry is one more term (the same as a duplicated K/V row in
    the gathered matrix), -1 entries are ignored, and the order of the list
    does not matter; an out-of-range entry is an error and is skipped."""
    g = W.generator(42)
    B, Hq, Hkv, C, D = 1, 2, 1, 10, 4
    q = W.randn(g, (B, Hq, D), torch.float32)
    k = W.randn(g, (B, Hkv, C, D), torch.float32)
    v = W.randn(g, (B, Hkv, C, D), torch.float32)
    idx = torch.tensor([[3, 7, 3, -1]], dtype=torch.int32)
    out, _, err = oracle.attend_indexed(q, k, v, idx, 0.5)
    assert err == 0
    # the gathered matrix written out: rows 3, 7, 3 of the cache at slots 0, 1, 2
    kg = k[:, :, [3, 7, 3]].contiguous()
    vg = v[:, :, [3, 7, 3]].contiguous()
    ref, _ = oracle.attend_masked(q, kg, vg, torch.ones(B, 3, dtype=torch.uint8), 0.5)
    assert np.allclose(out, ref, rtol=0, atol=1e-13)
    perm, _, _ = oracle.attend_indexed(q, k, v, torch.tensor([[-1, 3, 3, 7]], dtype=torch.int32), 0.5)
    assert np.allclose(perm, out, rtol=0, atol=1e-13)
    bad, _, err = oracle.attend_indexed(q, k, v, torch.tensor([[3, 7, 3, 10]], dtype=torch.int32), 0.5)
    assert err == oracle.ERR_POS and np.allclose(bad, out, rtol=0, atol=1e-13)
    empty, lse, _ = oracle.attend_indexed(q, k, v, torch.full((1, 4), -1, dtype=torch.int32), 0.5)
    assert np.all(empty == 0) and np.all(np.isneginf(lse))


# ------------------------------------------------------------ sliding window

@pytest.mark.parametrize("L,Wn", [(40, 1), (40, 7), (40, 40), (40, 64), (23, 16), (1, 5)])
def test_sliding_window_is_attention_over_the_last_rows(oracle, L, Wn):
    """Sliding-window decode (cuTile on NPU, Part 1, the tile-level variants):
    the step attends to the newest Wn rows only.  The window mask through the
    masked oracle equals float64 softmax attention written out over the slice
    k[L - Wn : L] (torch), and is bit-identical to the masked oracle on that
    slice alone; a window at least as long as the sequence is the prefix."""
    g = W.generator(60 + L + Wn)
    B, Hq, Hkv, C, D = 1, 4, 2, 64, 16
    q = W.randn(g, (B, Hq, D), torch.bfloat16)
    k = W.randn(g, (B, Hkv, C, D), torch.bfloat16)
    v = W.randn(g, (B, Hkv, C, D), torch.bfloat16)
    mask = W.window_mask([L], C, Wn)
    lo = max(0, L - Wn)
    assert int(mask.sum()) == L - lo and int(mask[0, lo]) == 1 and int(mask[0, L - 1]) == 1
    out, lse = oracle.attend_masked(q, k, v, mask, 0.2)
    ks = k[:, :, lo:L].double().repeat_interleave(Hq // Hkv, 1)
    vs = v[:, :, lo:L].double().repeat_interleave(Hq // Hkv, 1)
    s = torch.einsum("bhd,bhtd->bht", q.double(), ks) * 0.2
    ref = torch.einsum("bht,bhtd->bhd", torch.softmax(s, -1), vs)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=1e-12, atol=1e-12)
    o2, l2 = oracle.attend_masked(q, k[:, :, lo:L].contiguous(), v[:, :, lo:L].contiguous(),
                                  torch.ones(1, L - lo, dtype=torch.uint8), 0.2)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)
    if Wn >= L:
        assert np.array_equal(mask, W.prefix_mask([L], C))


@pytest.mark.parametrize("Wn", [1, 5, 16, 33, 64, 200])
def test_window_entry_is_attention_over_the_masked_window(oracle, Wn):
    """The window entry's definition (cuTile on NPU, Part 1's sliding-window
    variant over the mask contract): row b attends to the masked slots of
    [last - Wn + 1, last].  Checked against float64 softmax written out over
    the index set each row selects (a mask with holes, windows clipped at
    slot 0, the newest slot at the buffer's end); W = 1 is the newest row's
    value itself; a newest slot outside the buffer empties the row."""
    g = W.generator(90 + Wn)
    B, Hq, Hkv, C, D = 5, 4, 2, 96, 16
    q = W.randn(g, (B, Hq, D), torch.bfloat16)
    k = W.randn(g, (B, Hkv, C, D), torch.bfloat16)
    v = W.randn(g, (B, Hkv, C, D), torch.bfloat16)
    mask = (torch.rand(B, C, generator=g) < 0.7).to(torch.uint8)
    last = torch.tensor([C - 1, 10, 0, 50, C], dtype=torch.int32)  # the last is outside
    mask[torch.arange(4), last[:4].long()] = 1
    out, lse, err = oracle.attend_window(q, k, v, mask, last, Wn, 0.3)
    assert err == 1
    for b in range(B):
        t = int(last[b])
        if not 0 <= t < C:
            assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
            continue
        sel = [j for j in range(max(0, t - Wn + 1), t + 1) if mask[b, j]]
        for h in range(Hq):
            ks = k[b, h // (Hq // Hkv), sel].double()
            vs = v[b, h // (Hq // Hkv), sel].double()
            s = ks @ q[b, h].double() * 0.3
            ref = torch.softmax(s, 0) @ vs
            np.testing.assert_allclose(out[b, h], ref.numpy(), rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lse[b, h], float(torch.logsumexp(s, 0)), rtol=1e-12)
            if Wn == 1:
                assert sel == [t]
                np.testing.assert_allclose(out[b, h], vs[0].numpy(), rtol=0, atol=1e-15)
