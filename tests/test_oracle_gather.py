"""Pins of the fp64 oracle's paged gather, append, paged attention and combine
(CPU only)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _location_cache(NB, BS, H, Dd, tag):
    """int32 cache whose every row spells out (tag, block, slot, head, dim)."""
    b = np.arange(NB, dtype=np.int64).reshape(NB, 1, 1, 1)
    s = np.arange(BS, dtype=np.int64).reshape(1, BS, 1, 1)
    h = np.arange(H, dtype=np.int64).reshape(1, 1, H, 1)
    d = np.arange(Dd, dtype=np.int64).reshape(1, 1, 1, Dd)
    code = ((((tag * NB + b) * BS + s) * H + h) * Dd + d)
    return code.astype(np.int32)


def _decode(code, NB, BS, H, Dd):
    code = code.astype(np.int64)
    d = code % Dd
    code //= Dd
    h = code % H
    code //= H
    s = code % BS
    code //= BS
    b = code % NB
    return b, s, h, d


def _random_paged_layout(seed, Q, BS, cols, NB, max_len=None, offsets=True):
    rng = np.random.default_rng(seed)
    max_len = max_len or BS * cols
    off = (rng.integers(0, 3, size=Q) * BS) if offsets else np.zeros(Q, np.int64)
    lens = np.array([rng.integers(0, min(max_len, (cols - off[q] // BS) * BS) + 1)
                     for q in range(Q)])
    seq = np.zeros(Q + 1, np.int32)
    seq[1:] = np.cumsum(lens)
    bt = rng.permutation(NB)[: Q * cols].reshape(Q, cols).astype(np.int32)
    return bt, seq, off.astype(np.int32), lens


@pytest.mark.parametrize("BS", [1, 2, 4, 16])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gather_rows_come_from_the_mapped_block(oracle, BS, seed):
    """Each output row decodes to (block_tables[q, off/BS + t//BS], t % BS):
    the row's own contents say where it was read from."""
    Q, cols, NB, Hk, Dk, Hv, Dv = 4, 5, 40, 2, 3, 1, 5
    bt, seq, off, lens = _random_paged_layout(seed, Q, BS, cols, NB)
    kc = _location_cache(NB, BS, Hk, Dk, 1)
    vc = _location_cache(NB, BS, Hv, Dv, 2)
    ko, vo, err = oracle.gather_paged(kc.view(np.float32), vc.view(np.float32), bt, seq, off)
    assert err == 0
    ko, vo = ko.view(np.int32), vo.view(np.int32)
    assert ko.shape == (seq[-1], Hk, Dk) and vo.shape == (seq[-1], Hv, Dv)
    for q in range(Q):
        for t in range(lens[q]):
            row = seq[q] + t
            b, s, h, d = _decode(ko[row] - 1 * NB * BS * Hk * Dk, NB, BS, Hk, Dk)
            assert np.all(b == bt[q, off[q] // BS + t // BS]) and np.all(s == t % BS)
            assert np.array_equal(h[:, 0], np.arange(Hk)) and np.array_equal(d[0], np.arange(Dk))
            b2, s2, _, _ = _decode(vo[row] - 2 * NB * BS * Hv * Dv, NB, BS, Hv, Dv)
            assert np.all(b2 == b[0, 0]) and np.all(s2 == t % BS)


def test_gather_with_identity_tables_is_a_slice(oracle):
    """Consecutive physical blocks and zero offsets: the gather of one sequence
    is a plain slice of the flattened cache (torch slicing as the reference)."""
    NB, BS, H, D = 12, 4, 3, 8
    kc = W.randn(W.generator(3), (NB, BS, H, D), torch.bfloat16)
    vc = W.randn(W.generator(4), (NB, BS, H, D), torch.bfloat16)
    bt = np.array([[0, 1, 2, 3], [4, 5, 6, 7], [8, 9, 10, 11]], np.int32)
    lens = [13, 1, 16]
    seq = np.array([0, 13, 14, 30], np.int32)
    kb = kc.view(torch.int16).numpy()
    vb = vc.view(torch.int16).numpy()
    ko, vo, err = oracle.gather_paged(kb, vb, bt, seq, None)
    assert err == 0
    flat_k = kc.reshape(NB * BS, H, D)
    flat_v = vc.reshape(NB * BS, H, D)
    for q in range(3):
        base = q * 4 * BS
        assert torch.equal(torch.from_numpy(ko[seq[q]:seq[q + 1]]).view(torch.bfloat16),
                           flat_k[base:base + lens[q]])
        assert torch.equal(torch.from_numpy(vo[seq[q]:seq[q + 1]]).view(torch.bfloat16),
                           flat_v[base:base + lens[q]])


def _split_lengths(rng, Q, T, cap):
    """Q lengths summing to T, each <= cap (the page prints only the totals)."""
    while True:
        cuts = np.sort(rng.integers(0, T + 1, size=Q - 1))
        lens = np.diff(np.concatenate([[0], cuts, [T]]))
        if lens.max() <= cap:
            return lens


def test_gather_page_printed_shapes(oracle):
    """Section 8.1 sweep shapes (key [5513,128,1,512], value [5513,128,1,64],
    block_tables [Q,8]) and the section 8.2 hand-picked shapes, checked by
    location decoding.  Only the blocks a case reads are materialised."""
    spec = json.load(open(os.path.join(GOLDEN, "gather_pa_kv_cache_shapes.json")))
    rng = np.random.default_rng(123)
    cases = [(spec["sweep"]["key_cache"], spec["sweep"]["value_cache"], c["Q"], c["T"],
              spec["sweep"]["block_table_cols"]) for c in spec["sweep"]["cases"]]
    cases += [(m["key_cache"], m["value_cache"], 2, m["T"], 4) for m in spec["manual"]]
    for kshape, vshape, Q, T, cols in cases:
        NB, BS, Hk, Dk = kshape
        _, _, Hv, Dv = vshape
        lens = _split_lengths(rng, Q, T, BS * cols)
        seq = np.zeros(Q + 1, np.int32)
        seq[1:] = np.cumsum(lens)
        bt = rng.permutation(NB)[: Q * cols].reshape(Q, cols).astype(np.int32)
        used = sorted(set(bt.reshape(-1).tolist()))
        # compact the cache to the used blocks, remembering the true block id
        remap = {b: i for i, b in enumerate(used)}
        bt_c = np.vectorize(remap.get)(bt).astype(np.int32)
        kc = _location_cache(len(used), BS, Hk, Dk, 0)
        vc = _location_cache(len(used), BS, Hv, Dv, 1)
        ko, vo, err = oracle.gather_paged(kc.view(np.float32), vc.view(np.float32), bt_c, seq)
        assert err == 0 and ko.shape == (T, Hk, Dk) and vo.shape == (T, Hv, Dv)
        ko = ko.view(np.int32)
        vo = vo.view(np.int32)
        for q in range(Q):
            for t in range(lens[q]):
                b, s, _, _ = _decode(ko[seq[q] + t], len(used), BS, Hk, Dk)
                assert used[int(b[0, 0])] == bt[q, t // BS] and int(s[0, 0]) == t % BS
                b, s, _, _ = _decode(vo[seq[q] + t] - len(used) * BS * Hv * Dv,
                                     len(used), BS, Hv, Dv)
                assert used[int(b[0, 0])] == bt[q, t // BS] and int(s[0, 0]) == t % BS


def test_gather_rejections(oracle):
    """Constraints of section 3.3 / 7: bad inputs set their error bit and the
    offending rows are not written."""
    NB, BS, H, D = 6, 4, 1, 4
    kc = _location_cache(NB, BS, H, D, 0).view(np.float32)
    vc = _location_cache(NB, BS, H, D, 0).view(np.float32)
    bt = np.array([[0, 1], [2, 3]], np.int32)
    seq = np.array([0, 5, 8], np.int32)
    _, _, err = oracle.gather_paged(kc, vc, bt, seq)
    assert err == 0
    bad = bt.copy()
    bad[0, 1] = NB
    ko, _, err = oracle.gather_paged(kc, vc, bad, seq)
    assert err == oracle.ERR_BLOCK
    assert np.all(ko[4] == 0) and np.any(ko[3] != 0)
    _, _, err = oracle.gather_paged(kc, vc, bt, np.array([1, 5, 8], np.int32))
    assert err & oracle.ERR_SEQLENS
    _, _, err = oracle.gather_paged(kc, vc, bt, np.array([0, 5, 3], np.int32), total_tokens=8)
    assert err & oracle.ERR_SEQLENS
    _, _, err = oracle.gather_paged(kc, vc, bt, seq, np.array([2, 0], np.int32))
    assert err == oracle.ERR_OFFSET
    _, _, err = oracle.gather_paged(kc, vc, bt, seq, np.array([-4, 0], np.int32))
    assert err == oracle.ERR_OFFSET
    _, _, err = oracle.gather_paged(kc, vc, bt, seq, np.array([4, 0], np.int32))
    assert err == oracle.ERR_COLS
    with pytest.raises(ValueError):
        oracle.gather_paged(kc, vc, bt, np.array([5, 3], np.int32))


# ---------------------------------------------------------------- append

def test_append_writes_only_the_new_row(oracle):
    g = W.generator(20)
    B, H, C, D = 3, 2, 9, 5
    k = W.randn(g, (B, H, C, D), torch.bfloat16).view(torch.int16).numpy().copy()
    v = W.randn(g, (B, H, C, D), torch.bfloat16).view(torch.int16).numpy().copy()
    kn = W.randn(g, (B, H, D), torch.bfloat16)
    vn = W.randn(g, (B, H, D), torch.bfloat16)
    mask = np.zeros((B, C), np.uint8)
    pos = np.array([0, 8, 4], np.int32)
    k0, v0 = k.copy(), v.copy()
    assert oracle.append(k, v, kn, vn, pos, mask) == 0
    for b in range(B):
        for t in range(C):
            if t == pos[b]:
                assert np.array_equal(k[b, :, t], kn[b].view(torch.int16).numpy())
                assert np.array_equal(v[b, :, t], vn[b].view(torch.int16).numpy())
            else:
                assert np.array_equal(k[b, :, t], k0[b, :, t])
                assert np.array_equal(v[b, :, t], v0[b, :, t])
    assert mask.sum() == B and all(mask[b, pos[b]] == 1 for b in range(B))


def test_append_over_capacity_is_an_error(oracle):
    """Over capacity is an error, not a truncation (NPU article, Part 5
    '当前限制'): nothing is written for that sequence."""
    B, H, C, D = 2, 1, 4, 2
    k = np.zeros((B, H, C, D), np.float32)
    v = np.zeros((B, H, C, D), np.float32)
    mask = np.zeros((B, C), np.uint8)
    kn = torch.ones(B, H, D)
    err = oracle.append(k, v, kn, kn, np.array([4, 1], np.int32), mask)
    assert err == oracle.ERR_POS
    assert np.all(k[0] == 0) and np.all(mask[0] == 0) and mask[1, 1] == 1
    err = oracle.append(k, v, kn, kn, np.array([-1, 1], np.int32), None)
    assert err == oracle.ERR_POS


def test_mask_evolution_matches_the_page(oracle):
    """A 4-token prompt in the 1152-slot buffer: 4 valid slots while the first
    token is produced, 5 for the second, 103 for the hundredth (the article's
    printed example); append position = number of stored tokens."""
    spec = json.load(open(os.path.join(GOLDEN, "npuw_mask_evolution.json")))
    C = spec["capacity"]
    assert C == spec["max_prompt_len"] + spec["min_response_len"]
    k = np.zeros((1, 1, C, 2), np.float32)
    v = np.zeros((1, 1, C, 2), np.float32)
    mask = W.prefix_mask([spec["prompt_tokens"]], C).numpy().copy()
    stored = spec["prompt_tokens"]
    seen = {1: int(mask.sum())}
    row = torch.zeros(1, 1, 2)
    for n in range(2, 101):
        assert oracle.append(k, v, row, row, np.array([stored], np.int32), mask) == 0
        stored += 1
        seen[n] = int(mask.sum())
    for ex in spec["examples"]:
        assert seen[ex["generating_token"]] == ex["valid"]
        assert C - seen[ex["generating_token"]] == ex["empty"]


# ---------------------------------------------------------------- combine

def test_split_invariance_of_combine(oracle):
    """Attention over disjoint key ranges, merged by log-sum-exp, equals the
    unsplit attention."""
    g = W.generator(30)
    B, Hq, Hkv, C, D = 2, 4, 2, 50, 16
    q = W.randn(g, (B, Hq, D), torch.float32)
    k = W.randn(g, (B, Hkv, C, D), torch.float32)
    v = W.randn(g, (B, Hkv, C, D), torch.float32)
    mask = W.prefix_mask([50, 23], C)
    full, full_lse = oracle.attend_masked(q, k, v, mask, 0.2)
    bounds = [0, 7, 20, 21, 40, 50]
    parts_o, parts_l = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        m = mask.clone()
        m[:, :a] = 0
        m[:, b:] = 0
        o, l = oracle.attend_masked(q, k, v, m, 0.2)
        parts_o.append(o)
        parts_l.append(l)
    po = np.stack(parts_o, axis=2).reshape(B * Hq, len(parts_o), D)
    pl = np.stack(parts_l, axis=2).reshape(B * Hq, len(parts_l))
    assert np.isneginf(pl).any()  # ranges past the valid length are empty
    out, lse = oracle.combine(po, pl)
    np.testing.assert_allclose(out.reshape(B, Hq, D), full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse.reshape(B, Hq), full_lse, rtol=1e-12, atol=1e-13)


def test_combine_closed_forms(oracle):
    po = np.array([[[1.0, 2.0], [3.0, 6.0]], [[5.0, 5.0], [7.0, 7.0]],
                   [[1.0, 1.0], [2.0, 2.0]]])
    pl = np.array([[0.5, 0.5], [-np.inf, 1.0], [-np.inf, -np.inf]])
    out, lse = oracle.combine(po, pl)
    np.testing.assert_allclose(out[0], [2.0, 4.0], rtol=1e-15)
    assert lse[0] == pytest.approx(0.5 + math.log(2.0), rel=1e-15)
    np.testing.assert_allclose(out[1], [7.0, 7.0], rtol=1e-15)
    assert lse[1] == 1.0
    assert np.all(out[2] == 0.0) and lse[2] == -np.inf


# ---------------------------------------------------------------- paged attention

def test_paged_attention_equals_masked_on_a_static_buffer(oracle):
    """Identity block tables: the paged cache is a static buffer seen through a
    reshape, so paged attention equals masked attention with prefix masks."""
    g = W.generator(40)
    Q, Hq, Hkv, BS, cols, D = 3, 4, 2, 4, 3, 8
    NB = Q * cols
    kc = W.randn(g, (NB, BS, Hkv, D), torch.bfloat16)
    vc = W.randn(g, (NB, BS, Hkv, D), torch.bfloat16)
    q = W.randn(g, (Q, Hq, D), torch.bfloat16)
    lens = [12, 5, 1]
    seq = W.cumsum_lengths(lens)
    bt = torch.arange(NB, dtype=torch.int32).reshape(Q, cols)
    out, lse = oracle.attend_paged(q, kc, vc, bt, seq, None, 0.3)
    C = cols * BS
    ks = kc.reshape(Q, C, Hkv, D).permute(0, 2, 1, 3).contiguous()
    vs = vc.reshape(Q, C, Hkv, D).permute(0, 2, 1, 3).contiguous()
    ref, ref_lse = oracle.attend_masked(q, ks, vs, W.prefix_mask(lens, C), 0.3)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


def test_paged_attention_matches_torch_sdpa(oracle):
    g = W.generator(41)
    Q, Hq, Hkv, BS, cols, D, NB = 3, 8, 2, 16, 4, 32, 20
    kc = W.randn(g, (NB, BS, Hkv, D), torch.float32)
    vc = W.randn(g, (NB, BS, Hkv, D), torch.float32)
    q = W.randn(g, (Q, Hq, D), torch.float32)
    lens = [37, 64, 3]
    seq = W.cumsum_lengths(lens)
    bt = W.permuted_block_tables(W.generator(42), Q, cols, NB)
    out, _ = oracle.attend_paged(q, kc, vc, bt, seq, None, 0.11)
    for i in range(Q):
        t = torch.arange(lens[i])
        phys = bt[i, t // BS].long()
        kk = kc[phys, t % BS].double().permute(1, 0, 2).repeat_interleave(4, 0)
        vv = vc[phys, t % BS].double().permute(1, 0, 2).repeat_interleave(4, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[i].double().unsqueeze(1), kk, vv, scale=0.11).squeeze(1)
        np.testing.assert_allclose(out[i], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_copy_prefix_is_the_slice_assignment(oracle):
    """copy_kvcache (NPU article, Part 2 'NPUW 的核心设计', step 3): the
    prefill present[0:N] becomes the generate past[0:N]; checked against
    numpy slice assignment on the raw 16-bit patterns, plus the prefix mask."""
    g = W.generator(21)
    B, H, Cs, Cd, D = 3, 2, 7, 9, 4
    ks = W.randn(g, (B, H, Cs, D), torch.bfloat16).view(torch.int16).numpy()
    vs = W.randn(g, (B, H, Cs, D), torch.bfloat16).view(torch.int16).numpy()
    kd = W.randn(g, (B, H, Cd, D), torch.bfloat16).view(torch.int16).numpy().copy()
    vd = W.randn(g, (B, H, Cd, D), torch.bfloat16).view(torch.int16).numpy().copy()
    n = np.array([0, 7, 3], np.int32)
    mask = np.full((B, Cd), 7, np.uint8)
    ek, ev = kd.copy(), vd.copy()
    for b in range(B):
        ek[b, :, :n[b]] = ks[b, :, :n[b]]
        ev[b, :, :n[b]] = vs[b, :, :n[b]]
    assert oracle.copy_prefix(ks, vs, kd, vd, n, mask) == 0
    assert np.array_equal(kd, ek) and np.array_equal(vd, ev)
    assert np.array_equal(mask, (np.arange(Cd)[None, :] < n[:, None]).astype(np.uint8))


def test_copy_prefix_longer_than_either_buffer_is_an_error(oracle):
    """A prompt longer than the smaller capacity copies nothing for that
    entry (over capacity is an error, NPU article, Part 5 '当前限制')."""
    B, H, Cs, Cd, D = 2, 1, 6, 4, 2
    ks = np.ones((B, H, Cs, D), np.float32)
    kd = np.zeros((B, H, Cd, D), np.float32)
    vd = np.zeros((B, H, Cd, D), np.float32)
    mask = np.zeros((B, Cd), np.uint8)
    assert oracle.copy_prefix(ks, ks, kd, vd, np.array([5, 2], np.int32), mask) == oracle.ERR_POS
    assert np.all(kd[0] == 0) and np.all(mask[0] == 0)
    assert np.all(kd[1, :, :2] == 1) and np.all(kd[1, :, 2:] == 0)
    assert list(mask[1]) == [1, 1, 0, 0]
    assert oracle.copy_prefix(ks, ks, kd, vd, np.array([-1, 0], np.int32), None) == oracle.ERR_POS
