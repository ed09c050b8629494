"""Pins of the oracle's paged KV append ("Intel NPU running LLMs", Part 2:
update_kvcache_for writes only the new token's row; "PyPTO 实现 AscendC
GatherPaKvCache", section 3.2: token t of sequence q lives in block
block_tables[q, seq_offset[q] / BS + t / BS], slot t % BS).

The append is pinned against the paged gather (itself pinned against
brute-force indexing and the page's shapes in test_oracle_gather.py): after
every sequence appends its next token, gathering the one-token-longer
sequences returns the old rows followed by the new row, and no other byte of
the caches changes.  Error cases write nothing.
"""
import numpy as np
import pytest

import oracle



def _case(seed, Q, NB, BS, cols, H, D, offsets=False):
    rng = np.random.default_rng(seed)
    kc = rng.integers(-2**15, 2**15, size=(NB, BS, H, D), dtype=np.int16)
    vc = rng.integers(-2**15, 2**15, size=(NB, BS, H, D), dtype=np.int16)
    bt = rng.permutation(NB)[:Q * cols].reshape(Q, cols).astype(np.int32)
    off = (rng.integers(0, 2, size=Q) * BS).astype(np.int32) if offsets else np.zeros(Q, np.int32)
    # lengths that leave room for one more token in the table
    lens = np.array([rng.integers(0, (cols - o // BS) * BS) for o in off], np.int32)
    kn = rng.integers(-2**15, 2**15, size=(Q, H, D), dtype=np.int16)
    vn = rng.integers(-2**15, 2**15, size=(Q, H, D), dtype=np.int16)
    return kc, vc, bt, off, lens, kn, vn


@pytest.mark.parametrize("seed,Q,NB,BS,cols,H,D,offsets", [
    (1, 3, 16, 4, 4, 2, 8, False), (2, 4, 32, 1, 6, 1, 4, True), (3, 2, 12, 2, 5, 3, 2, True),
    (4, 5, 40, 8, 3, 2, 16, False)])
def test_appended_token_is_what_the_gather_reads_next(seed, Q, NB, BS, cols, H, D, offsets):
    kc, vc, bt, off, lens, kn, vn = _case(seed, Q, NB, BS, cols, H, D, offsets)
    cum = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    k_before, v_before, err = oracle.gather_paged(kc, vc, bt, cum, off)
    assert err == 0
    kc2, vc2 = kc.copy(), vc.copy()
    assert oracle.append_paged(kc2, vc2, bt, off, kn, vn, lens) == 0
    cum1 = np.concatenate([[0], np.cumsum(lens + 1)]).astype(np.int32)
    k_after, v_after, err = oracle.gather_paged(kc2, vc2, bt, cum1, off)
    assert err == 0
    for q in range(Q):
        a, n = cum1[q], lens[q]
        assert np.array_equal(k_after[a:a + n], k_before[cum[q]:cum[q] + n])
        assert np.array_equal(v_after[a:a + n], v_before[cum[q]:cum[q] + n])
        assert np.array_equal(k_after[a + n], kn[q]) and np.array_equal(v_after[a + n], vn[q])
    # exactly Q token rows changed, nothing else
    changed = np.any(kc2 != kc, axis=(2, 3))
    assert changed.sum() <= Q
    unchanged = ~np.any((kc2 != kc) | (vc2 != vc), axis=(2, 3))
    assert unchanged.sum() >= NB * BS - Q


def test_errors_write_nothing():
    kc, vc, bt, off, lens, kn, vn = _case(9, 4, 16, 4, 3, 2, 8)
    off = np.array([0, 4, 3, -4], np.int32)  # q1 fine, q2 not a multiple of BS, q3 negative
    pos = np.array([-1, 0, 0, 0], np.int32)  # q0 negative position
    kc2, vc2 = kc.copy(), vc.copy()
    err = oracle.append_paged(kc2, vc2, bt, off, kn, vn, pos)
    assert err == oracle.ERR_POS | oracle.ERR_OFFSET
    # only q1's token (table column 1, slot 0) was written
    phys = bt[1, 1]
    assert np.array_equal(kc2[phys, 0], kn[1])
    mask = np.ones((16, 4), bool)
    mask[phys, 0] = False
    assert np.array_equal(kc2[mask], kc[mask]) and np.array_equal(vc2[mask], vc[mask])
    # past the table, or a block id out of range
    bt2 = bt.copy()
    bt2[0, 0] = 99
    kc3 = kc.copy()
    err = oracle.append_paged(kc3, vc.copy(), bt2, None, kn, vn, np.array([0, 12, 0, 1], np.int32))
    assert err == oracle.ERR_BLOCK | oracle.ERR_COLS
    assert np.array_equal(kc3[bt2[2, 0], 0], kn[2]) and np.array_equal(kc3[bt2[3, 0], 1], kn[3])
