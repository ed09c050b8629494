"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports
every entry point include/kvd.h declares, and rejects bad arguments on the
host before any CUDA call (no GPU needed for these paths)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from decode_attention_kv_gb300 import _build, kvd
    _build.build()
    return kvd.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "kvd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvd_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    syms = declared_symbols()
    assert len(syms) >= 10
    from decode_attention_kv_gb300 import kvd
    for s in syms:
        assert hasattr(lib, s), f"{s} not exported"
        assert s in kvd.SIGNATURES, f"{s} has no binding signature"


def test_version_and_status_strings(lib):
    assert lib.kvd_version() == 10000
    assert lib.kvd_status_string(0) == b"KVD_OK"
    assert lib.kvd_status_string(3) == b"KVD_ERR_WORKSPACE"


def _masked(lib, q=1, k=1, v=1, m=1, out=1, B=2, Hq=8, Hkv=2, C=64, D=128, dt=0, ns=0, ws=None,
            wsb=0):
    P = lambda x: None if x is None else ctypes.c_void_p(x * 4096)  # noqa: E731 (aligned fakes)
    return lib.kvd_attend_masked(P(q), P(k), P(v), P(m), P(out), None, B, Hq, Hkv, C, D, 0.1, dt,
                                 ns, P(ws), wsb, None, None)


def test_masked_host_validation(lib):
    assert _masked(lib, Hq=6, Hkv=4) == 1            # Hq not a multiple of Hkv
    assert _masked(lib, D=96) == 2                   # unsupported head_dim
    assert _masked(lib, dt=7) == 1                   # unknown dtype
    assert _masked(lib, q=None) == 1                 # null pointer
    assert _masked(lib, B=0, q=None) == 0            # empty batch: nothing to do
    assert _masked(lib, C=0) == 1
    assert _masked(lib, C=4096, ns=4) == 3           # the call needs a workspace
    assert _masked(lib, C=64, ns=1) == 3             # even with one split (work counters)
    need = lib.kvd_attend_masked_workspace_bytes(2, 8, 2, 4096, 128, 0, 4)
    assert need > 0
    assert _masked(lib, C=4096, ns=4, ws=1, wsb=need - 1) == 3
    msg = lib.kvd_last_error().decode()
    assert "workspace" in msg
    misaligned = lib.kvd_attend_masked(ctypes.c_void_p(4096 + 8), ctypes.c_void_p(4096),
                                       ctypes.c_void_p(4096), ctypes.c_void_p(4096),
                                       ctypes.c_void_p(4096), None, 1, 4, 4, 64, 128, 0.1, 0, 0,
                                       None, 0, None, None)
    assert misaligned == 1


def test_workspace_sizes_follow_the_plan(lib):
    """Workspace = counters | partial log-sum-exps | partial rows, for S
    splits; one split needs only the counters.  The plan depends on the sizes
    only."""
    from decode_attention_kv_gb300 import kvd
    # 16 x 32 heads over capacity 8192: 512 query rows
    ws = lib.kvd_attend_masked_workspace_bytes(16, 32, 8, 8192, 128, 0, 0)
    pl = kvd.attend_masked_plan(16, 32, 8, 8192, 128)
    R, S = 16 * 32, pl.splits
    assert S > 1 and pl.launches == 2
    assert pl.counter_bytes == 256 == pl.lse_offset
    assert pl.o_offset == pl.lse_offset + (R * S * 4 + 255) // 256 * 256
    assert ws == pl.o_offset + R * S * 128 * 4
    # one split: only the 256-byte block of scheduling counters
    assert lib.kvd_attend_masked_workspace_bytes(1, 4, 4, 32, 64, 1, 0) == 256
    # counters | 32 x 16 partial lse | 32 x 16 x 128 partial rows
    assert lib.kvd_attend_masked_workspace_bytes(1, 32, 32, 32768, 128, 0, 16) == \
        256 + 32 * 16 * 4 + 32 * 16 * 128 * 4
    # the short static buffer: the one-launch cluster kernel
    pl = kvd.attend_masked_plan(1, 32, 32, 1152, 128)
    assert pl.splits == 0 and pl.launches == 1
    assert lib.kvd_attend_paged_workspace_bytes(64, 32, 8, 128, 32, 128, 0, 0) > 0
    assert lib.kvd_attend_masked_workspace_bytes(1, 4, 3, 32, 64, 0, 0) == 0  # invalid -> 0


def test_other_entry_points_validate(lib):
    P = lambda x: ctypes.c_void_p(x * 4096)  # noqa: E731
    # append: D*elem not a multiple of 16 bytes
    assert lib.kvd_append(P(1), P(1), P(1), P(1), P(1), None, 1, 1, 8, 6, 0, None, None) == 1
    # gather: elem_bytes must be 2 or 4
    assert lib.kvd_gather_paged(P(1), P(1), P(1), P(1), None, P(1), P(1), 1, 4, 16, 2, 1, 64, 1,
                                64, 10, 8, None, None) == 1
    assert lib.kvd_gather_paged(P(1), P(1), P(1), P(1), None, P(1), P(1), 0, 4, 16, 2, 1, 64, 1,
                                64, 0, 2, None, None) == 0  # no sequences
    # combine: D must be a multiple of 4
    assert lib.kvd_combine(P(1), P(1), P(1), None, 4, 2, 6, 1, None) == 1
    assert lib.kvd_combine(P(1), P(1), P(1), None, 0, 2, 8, 1, None) == 0
    # paged: NB*BS beyond the tensor-map range
    assert lib.kvd_attend_paged(P(1), P(1), P(1), P(1), P(1), None, P(1), None, 1, 4, 4,
                                1 << 24, 256, 4, 128, 0.1, 0, 0, None, 0, None, None) == 2


def test_fp8_entry_points_validate(lib):
    P = lambda x: ctypes.c_void_p(x * 4096)  # noqa: E731
    # head_dim 96 is not supported by the quantiser
    assert lib.kvd_append_fp8(P(1), P(1), P(1), P(1), P(1), None, 1, 1, 8, 96, 0, None, None) == 2
    assert lib.kvd_append_fp8(P(1), P(1), P(1), P(1), None, None, 1, 1, 8, 128, 0, None, None) == 1
    # workspace: one split needs the counters only; many splits need partials
    assert lib.kvd_attend_masked_fp8_workspace_bytes(1, 4, 4, 32, 128, 1) == 256
    assert lib.kvd_attend_masked_fp8_workspace_bytes(16, 32, 8, 8192, 128, 0) > 256
    assert lib.kvd_attend_masked_fp8_workspace_bytes(1, 4, 3, 32, 128, 0) == 0
    assert lib.kvd_attend_masked_fp8(P(1), P(1), P(1), P(1), P(1), None, 2, 8, 2, 4096, 128, 0.1, 4,
                                     None, 0, None, None) == 3


def test_launch_counts(lib):
    """The small static-buffer launch (one cluster kernel) for short buffers,
    the split kernel plus the combine for long ones, none for bad sizes."""
    assert lib.kvd_attend_masked_launches(1, 32, 32, 1152, 128, 0, 0) == 1
    assert lib.kvd_attend_masked_launches(16, 32, 8, 8192, 128, 0, 0) == 2
    assert lib.kvd_attend_masked_launches(1, 32, 32, 1152, 128, 0, 3) == 2  # explicit splits
    assert lib.kvd_attend_masked_launches(1, 4, 4, 32, 64, 0, 0) == 1
    assert lib.kvd_attend_masked_launches(1, 4, 3, 32, 64, 0, 0) == 0


def test_device_status_check():
    """kvd.check names the KVD_DEV_* bits (the same values as kvd.h) and
    passes a clean status word."""
    import torch
    from decode_attention_kv_gb300 import kvd
    text = open(os.path.join(ROOT, "include", "kvd.h")).read()
    defs = {n: int(v) for n, v in re.findall(r"#define (KVD_DEV_\w+) (\d+)u", text)}
    assert {b: n for n, b in defs.items()} == kvd.DEV_BITS
    kvd.check(torch.zeros(1, dtype=torch.int32))
    with pytest.raises(kvd.KvdDeviceError) as e:
        kvd.check(torch.tensor([1 | 32], dtype=torch.int32))
    assert e.value.names == ["KVD_DEV_POS_RANGE", "KVD_DEV_TIMEOUT"]


def test_window_entry_points(lib):
    """The window entries: the plan covers the window's span (W + 63 slots
    at most, never beyond the buffer), never the one-launch kernel; W < 1, a
    null newest-slot array and a short workspace are refused on the host."""
    from decode_attention_kv_gb300 import kvd
    P = lambda x: ctypes.c_void_p(x * 4096)  # noqa: E731
    # the 32768-slot sequence, 32 heads, window 4096: equal splits over the
    # window's span, as many as give each of the 304 persistent CTAs one unit
    # (304 // 32 = 9), against 112 over the whole buffer
    assert kvd.attend_masked_plan(1, 32, 32, 32768, 128).splits == 112
    win = kvd.attend_window_plan(1, 32, 32, 32768, 128, 4096)
    assert win.splits == 9 and win.launches == 2
    R = 32
    assert lib.kvd_attend_window_workspace_bytes(1, 32, 32, 32768, 128, 4096, 0, 0) == \
        256 + (R * 9 * 4 + 255) // 256 * 256 + R * 9 * 128 * 4
    # an explicit split count over the span: 4159 slots in splits of 1056
    assert kvd.attend_window_plan(1, 32, 32, 32768, 128, 4096, num_splits=4).splits == 4
    # 304 or more row units: one split per row, the rows written directly
    pl = kvd.attend_window_plan(64, 32, 8, 8192, 128, 2048)
    assert pl.splits == 1 and pl.launches == 1
    assert lib.kvd_attend_window_workspace_bytes(64, 32, 8, 8192, 128, 2048, 0, 0) == 256
    # a window at least as long as the buffer spans the buffer
    assert kvd.attend_window_plan(1, 32, 32, 1152, 128, 5000).splits >= 1
    assert lib.kvd_attend_window_workspace_bytes(1, 4, 4, 64, 64, 0, 0, 0) == 0  # W < 1
    args = (P(1), P(1), P(1), P(1), P(1), P(1), None, 1, 4, 4, 4096, 128)
    tail = (0.1, 0, 0, P(2), 1 << 20, None, None)
    assert lib.kvd_attend_window(*args, 0, *tail) == 1                       # W < 1
    assert lib.kvd_attend_window(*args[:4], None, *args[5:], 64, *tail) == 1  # no newest slots
    assert lib.kvd_attend_window(*args, 64, 0.1, 0, 3, None, 0, None, None) == 3  # no workspace
    fused = (P(1), P(1), P(1), P(1), P(1), P(1), P(1), P(1), None, 1, 4, 4, 4096, 128)
    assert lib.kvd_append_attend_window(*fused, 0, *tail) == 1
    assert lib.kvd_append_attend_window(*fused[:6], None, *fused[7:], 64, *tail) == 1
    assert kvd.attend_window_plan(2, 8, 8, 1152, 128, 64).splits >= 1


def test_binding_names_follow_the_c_entry_points():
    """Every compute or query entry point of include/kvd.h has a binding
    function of the same name without the kvd_ prefix (the diagnostics
    kvd_status_string, kvd_last_error and kvd_version surface through the
    binding's exceptions instead)."""
    from decode_attention_kv_gb300 import kvd
    header = open(os.path.join(ROOT, "include", "kvd.h")).read()
    names = set(re.findall(r"\b(kvd_[a-z0-9_]+)\s*\(", header))
    skip = {"kvd_status_string", "kvd_last_error", "kvd_version"}
    missing = sorted(n for n in names - skip if not hasattr(kvd, n[len("kvd_"):]))
    assert not missing, missing
