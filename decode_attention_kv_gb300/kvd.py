"""Thin ctypes binding of libkvd (argument marshalling only).

Every function passes torch tensors' device pointers and sizes straight to the
C entry point of the same name (``kvd_<name>``) on the current CUDA stream.
All computation happens in libkvd's kernels; there is no other code path: if
the library is not built, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvd.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA = 0, 1, 2, 3, 4
BF16, F32 = 0, 1

DEV_POS_RANGE = 1
DEV_BLOCK_RANGE = 2
DEV_TABLE_COLS = 4
DEV_SEQLENS = 8
DEV_SEQ_OFFSET = 16
DEV_TIMEOUT = 32

# Entry points of include/kvd.h with their argument types.
_vp, _sz, _i, _f = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
SIGNATURES = {
    "kvd_append": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp], _i),
    "kvd_copy_prefix": ([_vp, _vp, _vp, _vp, _vp, _vp] + [_i] * 7 + [_vp, _vp], _i),
    "kvd_attend_masked_workspace_bytes": ([_i, _i, _i, _i, _i, _i, _i], _sz),
    "kvd_attend_masked_launches": ([_i, _i, _i, _i, _i, _i, _i], _i),
    "kvd_attend_masked": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _vp, _sz,
                           _vp, _vp], _i),
    "kvd_attend_masked_plan": ([_i, _i, _i, _i, _i, _i, _i, _vp], _i),
    "kvd_attend_masked_fp8_plan": ([_i, _i, _i, _i, _i, _i, _vp], _i),
    "kvd_attend_masked_fp4_plan": ([_i, _i, _i, _i, _i, _i, _vp], _i),
    "kvd_attend_indexed_plan": ([_i, _i, _i, _i, _i, _i, _i, _vp], _i),
    "kvd_attend_paged_plan": ([_i, _i, _i, _i, _i, _i, _i, _i, _vp], _i),
    "kvd_attend_masked_partial": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i,
                                   _vp, _sz, _vp, _vp], _i),
    "kvd_attend_masked_noalloc": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i,
                                   _vp, _vp], _i),
    "kvd_append_attend_masked": ([_vp] * 7 + [_vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _vp, _sz,
                                  _vp, _vp], _i),
    "kvd_attend_window_workspace_bytes": ([_i] * 8, _sz),
    "kvd_attend_window_plan": ([_i] * 8 + [_vp], _i),
    "kvd_attend_window": ([_vp] * 7 + [_i] * 6 + [_f, _i, _i, _vp, _sz, _vp, _vp], _i),
    "kvd_append_attend_window": ([_vp] * 9 + [_i] * 6 + [_f, _i, _i, _vp, _sz, _vp, _vp], _i),
    "kvd_append_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp], _i),
    "kvd_attend_masked_fp8_workspace_bytes": ([_i, _i, _i, _i, _i, _i], _sz),
    "kvd_attend_masked_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _sz,
                               _vp, _vp], _i),
    "kvd_append_fp4": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp], _i),
    "kvd_attend_masked_fp4_workspace_bytes": ([_i, _i, _i, _i, _i, _i], _sz),
    "kvd_attend_masked_fp4": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _sz,
                               _vp, _vp], _i),
    "kvd_append_paged_fp8": ([_vp] * 7 + [_i] * 7 + [_vp, _vp], _i),
    "kvd_attend_paged_fp8_workspace_bytes": ([_i] * 7, _sz),
    "kvd_attend_paged_fp8_plan": ([_i] * 7 + [_vp], _i),
    "kvd_attend_paged_fp8": ([_vp] * 8 + [_i] * 7 + [_f, _i, _vp, _sz, _vp, _vp], _i),
    "kvd_attend_indexed_fp8_workspace_bytes": ([_i] * 6, _sz),
    "kvd_attend_indexed_fp8_plan": ([_i] * 6 + [_vp], _i),
    "kvd_attend_indexed_fp8": ([_vp] * 6 + [_i] * 6 + [_f, _i, _vp, _sz, _vp, _vp], _i),
    "kvd_append_paged_fp4": ([_vp] * 7 + [_i] * 7 + [_vp, _vp], _i),
    "kvd_attend_paged_fp4_workspace_bytes": ([_i] * 7, _sz),
    "kvd_attend_paged_fp4_plan": ([_i] * 7 + [_vp], _i),
    "kvd_attend_paged_fp4": ([_vp] * 8 + [_i] * 7 + [_f, _i, _vp, _sz, _vp, _vp], _i),
    "kvd_attend_indexed_fp4_workspace_bytes": ([_i] * 6, _sz),
    "kvd_attend_indexed_fp4_plan": ([_i] * 6 + [_vp], _i),
    "kvd_attend_indexed_fp4": ([_vp] * 6 + [_i] * 6 + [_f, _i, _vp, _sz, _vp, _vp], _i),
    "kvd_attend_indexed_workspace_bytes": ([_i, _i, _i, _i, _i, _i, _i], _sz),
    "kvd_attend_indexed": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp,
                            _sz, _vp, _vp], _i),
    "kvd_attend_paged_workspace_bytes": ([_i, _i, _i, _i, _i, _i, _i, _i], _sz),
    "kvd_attend_paged": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f,
                          _i, _i, _vp, _sz, _vp, _vp], _i),
    "kvd_append_paged": ([_vp] * 7 + [_i] * 7 + [_vp, _vp], _i),
    "kvd_gather_paged": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp] + [_i] * 10 + [_vp, _vp], _i),
    "kvd_combine": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp], _i),
    "kvd_combine_gathered": ([_vp, _vp, _vp, _i, _i, _i, _i, _vp], _i),
    "kvd_status_string": ([_i], ctypes.c_char_p),
    "kvd_last_error": ([], ctypes.c_char_p),
    "kvd_version": ([], _i),
}

_lock = threading.Lock()
_lib = None


class KvdError(RuntimeError):
    def __init__(self, name, status, message):
        super().__init__(f"{name} failed: {status} ({message})")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libkvd.so (built in-tree by ``_build.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libkvd.so not found at {p}: build it first "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(p)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _check(name, status):
    if status != OK:
        L = load()
        msg = L.kvd_last_error().decode(errors="replace")
        raise KvdError(name, L.kvd_status_string(status).decode(), msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _cuda_contig(name, t):
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def status_tensor(device=None):
    """A zeroed int32 device word for the kernels' error bits."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


# the KVD_DEV_* bits of kvd.h
DEV_BITS = {1: "KVD_DEV_POS_RANGE", 2: "KVD_DEV_BLOCK_RANGE", 4: "KVD_DEV_TABLE_COLS",
            8: "KVD_DEV_SEQLENS", 16: "KVD_DEV_SEQ_OFFSET", 32: "KVD_DEV_TIMEOUT",
            64: "KVD_DEV_POINTER"}


class KvdDeviceError(RuntimeError):
    def __init__(self, bits):
        self.bits = bits
        self.names = [n for b, n in DEV_BITS.items() if bits & b]
        super().__init__(f"device status {bits}: {', '.join(self.names) or 'unknown bits'}")


def check(dev_status):
    """Wait for the work queued so far (reading the word synchronises) and
    raise KvdDeviceError naming the bits the kernels set in ``dev_status``."""
    bits = int(dev_status.item())
    if bits:
        raise KvdDeviceError(bits)


# ------------------------------------------------------------------ append

def append(k_cache, v_cache, k_new, v_new, pos, mask=None, dev_status=None):
    """kvd_append: write the step's K/V rows at pos[b]; set mask[b, pos[b]]."""
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_new", k_new), ("v_new", v_new),
                 ("pos", pos)):
        _cuda_contig(n, t)
    B, Hkv, C, D = k_cache.shape
    if v_cache.shape != k_cache.shape or k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D):
        raise ValueError("append: shape mismatch")
    if pos.dtype != torch.int32 or pos.numel() != B:
        raise ValueError("append: pos must be int32 [B]")
    if mask is not None:
        _cuda_contig("mask", mask)
        if mask.dtype != torch.uint8 or mask.shape != (B, C):
            raise ValueError("append: mask must be uint8 [B, C]")
    dt = _dtype_code(k_cache)
    st = load().kvd_append(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(pos),
                           _ptr(mask), B, Hkv, C, D, dt, _ptr(dev_status), _stream(k_cache.device))
    _check("kvd_append", st)


FP8_ROW_PAD = 16  # KVD_FP8_ROW_PAD: bytes after the D codes of a quantised row


FP4_ROW_PAD = 16  # KVD_FP4_ROW_PAD: bytes after the D/2 code bytes of an FP4 row

# code bytes of a row of D elements, per row format
_CODE_BYTES = {"fp8": lambda D: D, "fp4": lambda D: D // 2}
_ROW_D = {"fp8": lambda RB: RB - FP8_ROW_PAD, "fp4": lambda RB: 2 * (RB - FP4_ROW_PAD)}


def _append_quant(fmt, k_cache, v_cache, k_new, v_new, pos, mask, dev_status):
    name = f"append_{fmt}"
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_new", k_new), ("v_new", v_new),
                 ("pos", pos)):
        _cuda_contig(n, t)
    B, Hkv, C, RB = k_cache.shape
    D = _ROW_D[fmt](RB)
    if k_cache.dtype != torch.uint8 or v_cache.shape != k_cache.shape or \
            v_cache.dtype != torch.uint8:
        raise ValueError(f"{name}: caches must be uint8 [B, Hkv, C, row bytes]")
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) or k_new.dtype != v_new.dtype:
        raise ValueError(f"{name}: shape mismatch")
    if pos.dtype != torch.int32 or pos.numel() != B:
        raise ValueError(f"{name}: pos must be int32 [B]")
    if mask is not None:
        _cuda_contig("mask", mask)
        if mask.dtype != torch.uint8 or mask.shape != (B, C):
            raise ValueError(f"{name}: mask must be uint8 [B, C]")
    fn = f"kvd_append_{fmt}"
    st = getattr(load(), fn)(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(pos),
                             _ptr(mask), B, Hkv, C, D, _dtype_code(k_new), _ptr(dev_status),
                             _stream(k_cache.device))
    _check(fn, st)


def append_fp8(k_cache, v_cache, k_new, v_new, pos, mask=None, dev_status=None):
    """kvd_append_fp8: quantise the step's K/V rows (bf16 or fp32 [B, Hkv, D])
    into row pos[b] of the E4M3 caches (uint8 [B, Hkv, C, D + 16]); set
    mask[b, pos[b]]."""
    _append_quant("fp8", k_cache, v_cache, k_new, v_new, pos, mask, dev_status)


def append_fp4(k_cache, v_cache, k_new, v_new, pos, mask=None, dev_status=None):
    """kvd_append_fp4: as append_fp8 into E2M1 caches (uint8
    [B, Hkv, C, D/2 + 16])."""
    _append_quant("fp4", k_cache, v_cache, k_new, v_new, pos, mask, dev_status)


def attend_masked_fp8_workspace_bytes(B, Hq, Hkv, C, D, num_splits=0):
    return load().kvd_attend_masked_fp8_workspace_bytes(B, Hq, Hkv, C, D, num_splits)


def attend_masked_fp4_workspace_bytes(B, Hq, Hkv, C, D, num_splits=0):
    return load().kvd_attend_masked_fp4_workspace_bytes(B, Hq, Hkv, C, D, num_splits)


def _attend_quant(fmt, q, k_cache, v_cache, mask, scale, out, lse, num_splits, workspace,
                  dev_status):
    name = f"attend_masked_{fmt}"
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("mask", mask)):
        _cuda_contig(n, t)
    B, Hq, D = q.shape
    Bk, Hkv, C, RB = k_cache.shape
    pad = FP8_ROW_PAD if fmt == "fp8" else FP4_ROW_PAD
    if Bk != B or RB != _CODE_BYTES[fmt](D) + pad or v_cache.shape != k_cache.shape or \
            mask.shape != (B, C):
        raise ValueError(f"{name}: shape mismatch")
    if q.dtype != torch.bfloat16 or k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8 \
            or mask.dtype != torch.uint8:
        raise TypeError(f"{name}: q bf16, caches and mask uint8")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is not None:
        _cuda_contig("lse", lse)
    L = load()
    fn = f"kvd_attend_masked_{fmt}"
    need = getattr(L, fn + "_workspace_bytes")(B, Hq, Hkv, C, D, num_splits)
    ws, wsb = _workspace(need, q.device, workspace)
    st = getattr(L, fn)(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(mask), _ptr(out), _ptr(lse),
                        B, Hq, Hkv, C, D, float(scale), num_splits, _ptr(ws), wsb,
                        _ptr(dev_status), _stream(q.device))
    _check(fn, st)
    return out


def attend_masked_fp8(q, k_cache, v_cache, mask, scale=None, out=None, lse=None, num_splits=0,
                      workspace=None, dev_status=None):
    """kvd_attend_masked_fp8: decode attention over E4M3 caches.

    q [B, Hq, D] bf16; k_cache, v_cache uint8 [B, Hkv, C, D + 16]; mask [B, C]
    uint8.  Returns out [B, Hq, D] bf16; fills ``lse`` [B, Hq] fp32 if given.
    """
    return _attend_quant("fp8", q, k_cache, v_cache, mask, scale, out, lse, num_splits,
                         workspace, dev_status)


def attend_masked_fp4(q, k_cache, v_cache, mask, scale=None, out=None, lse=None, num_splits=0,
                      workspace=None, dev_status=None):
    """kvd_attend_masked_fp4: decode attention over E2M1 caches (uint8
    [B, Hkv, C, D/2 + 16]); otherwise as attend_masked_fp8."""
    return _attend_quant("fp4", q, k_cache, v_cache, mask, scale, out, lse, num_splits,
                         workspace, dev_status)


# ------------------------------- quantised rows: paged layout, index lists

def _quant_row_d(fmt, RB, name):
    D = _ROW_D[fmt](RB)
    if D not in (64, 128):
        raise ValueError(f"{name}: row bytes {RB} do not give head_dim 64 or 128")
    return D


def _append_paged_quant(fmt, key_cache, value_cache, block_tables, seq_offset, k_new, v_new, pos,
                        dev_status):
    name = f"append_paged_{fmt}"
    for n, t in (("key_cache", key_cache), ("value_cache", value_cache), ("k_new", k_new),
                 ("v_new", v_new), ("block_tables", block_tables), ("pos", pos)):
        _cuda_contig(n, t)
    NB, BS, Hkv, RB = key_cache.shape
    D = _quant_row_d(fmt, RB, name)
    Q, cols = block_tables.shape
    if key_cache.dtype != torch.uint8 or value_cache.dtype != torch.uint8 or \
            value_cache.shape != key_cache.shape:
        raise ValueError(f"{name}: caches must be uint8 [NB, BS, Hkv, row bytes]")
    if k_new.shape != (Q, Hkv, D) or v_new.shape != (Q, Hkv, D) or k_new.dtype != v_new.dtype \
            or pos.numel() != Q:
        raise ValueError(f"{name}: shape mismatch")
    if block_tables.dtype != torch.int32 or pos.dtype != torch.int32 or \
            (seq_offset is not None and seq_offset.dtype != torch.int32):
        raise ValueError(f"{name}: int32 tables, offsets and positions")
    fn = f"kvd_{name}"
    st = getattr(load(), fn)(_ptr(key_cache), _ptr(value_cache), _ptr(k_new), _ptr(v_new),
                             _ptr(block_tables), _ptr(seq_offset), _ptr(pos), Q, NB, BS, cols, Hkv,
                             D, _dtype_code(k_new), _ptr(dev_status), _stream(key_cache.device))
    _check(fn, st)


def append_paged_fp8(key_cache, value_cache, block_tables, seq_offset, k_new, v_new, pos,
                     dev_status=None):
    """kvd_append_paged_fp8: the step's K/V rows (bf16 or fp32 [Q, Hkv, D])
    quantised into token pos[q] of the paged E4M3 caches (uint8
    [NB, BS, Hkv, D + 16])."""
    _append_paged_quant("fp8", key_cache, value_cache, block_tables, seq_offset, k_new, v_new, pos,
                        dev_status)


def append_paged_fp4(key_cache, value_cache, block_tables, seq_offset, k_new, v_new, pos,
                     dev_status=None):
    """kvd_append_paged_fp4: as append_paged_fp8 into E2M1 caches (uint8
    [NB, BS, Hkv, D/2 + 16])."""
    _append_paged_quant("fp4", key_cache, value_cache, block_tables, seq_offset, k_new, v_new, pos,
                        dev_status)


def attend_paged_quant_workspace_bytes(fmt, Q, Hq, Hkv, BS, cols, D, num_splits=0):
    return getattr(load(), f"kvd_attend_paged_{fmt}_workspace_bytes")(Q, Hq, Hkv, BS, cols, D,
                                                                       num_splits)


def attend_paged_quant_plan(fmt, Q, Hq, Hkv, BS, cols, D, num_splits=0):
    return _plan(f"kvd_attend_paged_{fmt}_plan", Q, Hq, Hkv, BS, cols, D, num_splits)


def attend_paged_quant(fmt, q, key_cache, value_cache, block_tables, seq_lens, seq_offset=None,
                       scale=None, out=None, lse=None, num_splits=0, workspace=None,
                       dev_status=None):
    """kvd_attend_paged_fp8 / _fp4 (fmt "fp8" / "fp4"): paged decode attention
    over quantised rows.  q [Q, Hq, D] bf16; caches uint8 [NB, BS, Hkv, RB];
    block_tables [Q, cols], seq_lens [Q + 1], seq_offset [Q] or None, int32."""
    name = f"attend_paged_{fmt}"
    for n, t in (("q", q), ("key_cache", key_cache), ("value_cache", value_cache),
                 ("block_tables", block_tables), ("seq_lens", seq_lens)):
        _cuda_contig(n, t)
    Q, Hq, D = q.shape
    NB, BS, Hkv, RB = key_cache.shape
    if _quant_row_d(fmt, RB, name) != D or value_cache.shape != key_cache.shape:
        raise ValueError(f"{name}: shape mismatch")
    if q.dtype != torch.bfloat16 or key_cache.dtype != torch.uint8 or \
            value_cache.dtype != torch.uint8:
        raise TypeError(f"{name}: q bf16, caches uint8")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != Q:
        raise ValueError(f"{name}: block_tables must be int32 [Q, cols]")
    if seq_lens.dtype != torch.int32 or seq_lens.shape != (Q + 1,):
        raise ValueError(f"{name}: only cumsum seq_lens [Q+1] int32 is supported")
    if seq_offset is not None:
        _cuda_contig("seq_offset", seq_offset)
        if seq_offset.dtype != torch.int32 or seq_offset.shape != (Q,):
            raise ValueError(f"{name}: seq_offset must be int32 [Q]")
    cols = block_tables.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is not None:
        _cuda_contig("lse", lse)
    L = load()
    fn = f"kvd_{name}"
    need = getattr(L, fn + "_workspace_bytes")(Q, Hq, Hkv, BS, cols, D, num_splits)
    ws, wsb = _workspace(need, q.device, workspace)
    st = getattr(L, fn)(_ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
                        _ptr(seq_lens), _ptr(seq_offset), _ptr(out), _ptr(lse), Q, Hq, Hkv, NB,
                        BS, cols, D, float(scale), num_splits, _ptr(ws), wsb, _ptr(dev_status),
                        _stream(q.device))
    _check(fn, st)
    return out


def attend_indexed_quant_workspace_bytes(fmt, B, Hq, Hkv, topk, D, num_splits=0):
    return getattr(load(), f"kvd_attend_indexed_{fmt}_workspace_bytes")(B, Hq, Hkv, topk, D,
                                                                         num_splits)


def attend_indexed_quant_plan(fmt, B, Hq, Hkv, topk, D, num_splits=0):
    return _plan(f"kvd_attend_indexed_{fmt}_plan", B, Hq, Hkv, topk, D, num_splits)


def attend_indexed_quant(fmt, q, k_cache, v_cache, indices, scale=None, out=None, lse=None,
                         num_splits=0, workspace=None, dev_status=None):
    """kvd_attend_indexed_fp8 / _fp4 (fmt "fp8" / "fp4"): index-list decode
    attention over quantised rows.  q [B, Hq, D] bf16; caches uint8
    [B, Hkv, C, RB]; indices [B, topk] int32 (-1 = unused entry)."""
    name = f"attend_indexed_{fmt}"
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("indices", indices)):
        _cuda_contig(n, t)
    B, Hq, D = q.shape
    Bk, Hkv, C, RB = k_cache.shape
    if Bk != B or _quant_row_d(fmt, RB, name) != D or v_cache.shape != k_cache.shape:
        raise ValueError(f"{name}: shape mismatch")
    if q.dtype != torch.bfloat16 or k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError(f"{name}: q bf16, caches uint8")
    if indices.dtype != torch.int32 or indices.dim() != 2 or indices.shape[0] != B:
        raise ValueError(f"{name}: indices must be int32 [B, topk]")
    topk = indices.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is not None:
        _cuda_contig("lse", lse)
    L = load()
    fn = f"kvd_{name}"
    need = getattr(L, fn + "_workspace_bytes")(B, Hq, Hkv, topk, D, num_splits)
    ws, wsb = _workspace(need, q.device, workspace)
    st = getattr(L, fn)(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(indices), _ptr(out), _ptr(lse),
                        B, Hq, Hkv, C, topk, D, float(scale), num_splits, _ptr(ws), wsb,
                        _ptr(dev_status), _stream(q.device))
    _check(fn, st)
    return out


# the C entry points' own names
def attend_paged_fp8_workspace_bytes(Q, Hq, Hkv, BS, cols, D, num_splits=0):
    return attend_paged_quant_workspace_bytes("fp8", Q, Hq, Hkv, BS, cols, D, num_splits)


def attend_paged_fp4_workspace_bytes(Q, Hq, Hkv, BS, cols, D, num_splits=0):
    return attend_paged_quant_workspace_bytes("fp4", Q, Hq, Hkv, BS, cols, D, num_splits)


def attend_paged_fp8_plan(Q, Hq, Hkv, BS, cols, D, num_splits=0):
    return attend_paged_quant_plan("fp8", Q, Hq, Hkv, BS, cols, D, num_splits)


def attend_paged_fp4_plan(Q, Hq, Hkv, BS, cols, D, num_splits=0):
    return attend_paged_quant_plan("fp4", Q, Hq, Hkv, BS, cols, D, num_splits)


def attend_paged_fp8(q, key_cache, value_cache, block_tables, seq_lens, seq_offset=None,
                     scale=None, out=None, lse=None, num_splits=0, workspace=None,
                     dev_status=None):
    """kvd_attend_paged_fp8: paged decode attention over E4M3 rows."""
    return attend_paged_quant("fp8", q, key_cache, value_cache, block_tables, seq_lens,
                              seq_offset, scale, out, lse, num_splits, workspace, dev_status)


def attend_paged_fp4(q, key_cache, value_cache, block_tables, seq_lens, seq_offset=None,
                     scale=None, out=None, lse=None, num_splits=0, workspace=None,
                     dev_status=None):
    """kvd_attend_paged_fp4: paged decode attention over E2M1 rows."""
    return attend_paged_quant("fp4", q, key_cache, value_cache, block_tables, seq_lens,
                              seq_offset, scale, out, lse, num_splits, workspace, dev_status)


def attend_indexed_fp8_workspace_bytes(B, Hq, Hkv, topk, D, num_splits=0):
    return attend_indexed_quant_workspace_bytes("fp8", B, Hq, Hkv, topk, D, num_splits)


def attend_indexed_fp4_workspace_bytes(B, Hq, Hkv, topk, D, num_splits=0):
    return attend_indexed_quant_workspace_bytes("fp4", B, Hq, Hkv, topk, D, num_splits)


def attend_indexed_fp8_plan(B, Hq, Hkv, topk, D, num_splits=0):
    return attend_indexed_quant_plan("fp8", B, Hq, Hkv, topk, D, num_splits)


def attend_indexed_fp4_plan(B, Hq, Hkv, topk, D, num_splits=0):
    return attend_indexed_quant_plan("fp4", B, Hq, Hkv, topk, D, num_splits)


def attend_indexed_fp8(q, k_cache, v_cache, indices, scale=None, out=None, lse=None,
                       num_splits=0, workspace=None, dev_status=None):
    """kvd_attend_indexed_fp8: index-list decode attention over E4M3 rows."""
    return attend_indexed_quant("fp8", q, k_cache, v_cache, indices, scale, out, lse, num_splits,
                                workspace, dev_status)


def attend_indexed_fp4(q, k_cache, v_cache, indices, scale=None, out=None, lse=None,
                       num_splits=0, workspace=None, dev_status=None):
    """kvd_attend_indexed_fp4: index-list decode attention over E2M1 rows."""
    return attend_indexed_quant("fp4", q, k_cache, v_cache, indices, scale, out, lse, num_splits,
                                workspace, dev_status)


def pointer_array(tensors, device):
    """A device int64 tensor holding the data pointers of `tensors` (the
    pointer arrays of kvd_copy_prefix).  Keep it alive until the call has run."""
    return torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64, device=device)


class PrefixCopy:
    """kvd_copy_prefix with its device pointer arrays built once: for every
    layer l, rows [0, n[b]) of k_src[l] / v_src[l] [B, Hkv, C_src, D] go to
    k_dst[l] / v_dst[l] [B, Hkv, C_dst, D], and masks[l] [B, C_dst]
    (optional) become the prefix masks; one launch per run()."""

    def __init__(self, k_src, v_src, k_dst, v_dst, masks=None):
        L = len(k_src)
        if not (L == len(v_src) == len(k_dst) == len(v_dst)) or L < 1:
            raise ValueError("copy_prefix: four lists of the same length >= 1")
        B, Hkv, C_src, D = k_src[0].shape
        C_dst = k_dst[0].shape[2]
        for t in list(k_src) + list(v_src):
            _cuda_contig("source cache", t)
            if t.shape != (B, Hkv, C_src, D) or t.dtype != k_src[0].dtype:
                raise ValueError("copy_prefix: source caches differ in shape or dtype")
        for t in list(k_dst) + list(v_dst):
            _cuda_contig("destination cache", t)
            if t.shape != (B, Hkv, C_dst, D) or t.dtype != k_src[0].dtype:
                raise ValueError("copy_prefix: destination caches differ in shape or dtype")
        if masks is not None:
            if len(masks) != L:
                raise ValueError("copy_prefix: one mask per layer")
            for m in masks:
                _cuda_contig("mask", m)
                if m.dtype != torch.uint8 or m.shape != (B, C_dst):
                    raise ValueError("copy_prefix: masks must be uint8 [B, C_dst]")
        self.dev = k_src[0].device
        # the tensors stay referenced here, so their memory outlives the pointers
        self.tensors = (list(k_src), list(v_src), list(k_dst), list(v_dst), masks)
        self.arrays = [pointer_array(x, self.dev) for x in (k_src, v_src, k_dst, v_dst)]
        self.marr = pointer_array(masks, self.dev) if masks is not None else None
        self.sizes = (L, B, Hkv, C_src, C_dst, D)
        self.dt = _dtype_code(k_src[0])

    def run(self, n, dev_status=None):
        L, B = self.sizes[0], self.sizes[1]
        _cuda_contig("n", n)
        if n.dtype != torch.int32 or n.numel() != B:
            raise ValueError("copy_prefix: n must be int32 [B]")
        st = load().kvd_copy_prefix(*(_ptr(a) for a in self.arrays), _ptr(self.marr), _ptr(n),
                                    *self.sizes, self.dt, _ptr(dev_status), _stream(self.dev))
        _check("kvd_copy_prefix", st)


def copy_prefix(k_src, v_src, k_dst, v_dst, n, masks=None, dev_status=None):
    """One kvd_copy_prefix call (see PrefixCopy); returns the PrefixCopy,
    whose pointer arrays must live until the launch has run."""
    pc = PrefixCopy(k_src, v_src, k_dst, v_dst, masks)
    pc.run(n, dev_status)
    return pc


# ------------------------------------------------------------------ attention

def attend_masked_workspace_bytes(B, Hq, Hkv, C, D, dtype=torch.bfloat16, num_splits=0):
    return load().kvd_attend_masked_workspace_bytes(B, Hq, Hkv, C, D,
                                                    BF16 if dtype == torch.bfloat16 else F32,
                                                    num_splits)


def workspace(nbytes, device=None):
    """A workspace for the attention calls: zero-filled, as the kernels
    require before first use (each call leaves it zeroed again)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def _workspace(nbytes, device, ws):
    if nbytes == 0:
        return None, 0
    if ws is None:
        ws = workspace(nbytes, device)
    have = ws.numel() * ws.element_size()
    if have < nbytes:
        raise ValueError(f"workspace smaller than {nbytes} bytes")
    return ws, have


def attend_masked_launches(B, Hq, Hkv, C, D, dtype=torch.bfloat16, num_splits=0):
    """Kernel launches of one kvd_attend_masked call for these sizes (1 or 2)."""
    return load().kvd_attend_masked_launches(B, Hq, Hkv, C, D,
                                             BF16 if dtype == torch.bfloat16 else F32, num_splits)


def attend_masked(q, k_cache, v_cache, mask, scale=None, out=None, lse=None, num_splits=0,
                  workspace=None, dev_status=None):
    """kvd_attend_masked: decode attention over the static buffer.

    q [B, Hq, D]; k_cache, v_cache [B, Hkv, C, D]; mask [B, C] uint8.
    Returns out [B, Hq, D] (dtype of q); fills ``lse`` [B, Hq] fp32 if given.
    """
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("mask", mask)):
        _cuda_contig(n, t)
    B, Hq, D = q.shape
    Bk, Hkv, C, Dk = k_cache.shape
    if Bk != B or Dk != D or v_cache.shape != k_cache.shape or mask.shape != (B, C):
        raise ValueError("attend_masked: shape mismatch")
    if mask.dtype != torch.uint8:
        raise ValueError("attend_masked: mask must be uint8")
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("attend_masked: q and caches must share a dtype")
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is not None:
        _cuda_contig("lse", lse)
    L = load()
    need = L.kvd_attend_masked_workspace_bytes(B, Hq, Hkv, C, D, dt, num_splits)
    ws, wsb = _workspace(need, q.device, workspace)
    st = L.kvd_attend_masked(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(mask), _ptr(out),
                             _ptr(lse), B, Hq, Hkv, C, D, float(scale), dt, num_splits, _ptr(ws),
                             wsb, _ptr(dev_status), _stream(q.device))
    _check("kvd_attend_masked", st)
    return out


class Plan(ctypes.Structure):
    """kvd_plan (include/kvd.h): how a split attention call runs."""
    _fields_ = [("splits", ctypes.c_int32), ("launches", ctypes.c_int32),
                ("lse_offset", ctypes.c_size_t), ("o_offset", ctypes.c_size_t),
                ("counter_bytes", ctypes.c_size_t)]


def _plan(name, *args):
    pl = Plan()
    st = getattr(load(), name)(*args, ctypes.byref(pl))
    _check(name, st)
    return pl


def attend_masked_plan(B, Hq, Hkv, C, D, dtype=torch.bfloat16, num_splits=0):
    """kvd_attend_masked_plan: the Plan of kvd_attend_masked for these sizes
    (splits 0 = the one-launch cluster kernel, 1 = no merge; launches 1 or 2;
    workspace offsets of the partial rows)."""
    return _plan("kvd_attend_masked_plan", B, Hq, Hkv, C, D,
                 BF16 if dtype == torch.bfloat16 else F32, num_splits)


def attend_masked_fp8_plan(B, Hq, Hkv, C, D, num_splits=0):
    return _plan("kvd_attend_masked_fp8_plan", B, Hq, Hkv, C, D, num_splits)


def attend_masked_fp4_plan(B, Hq, Hkv, C, D, num_splits=0):
    return _plan("kvd_attend_masked_fp4_plan", B, Hq, Hkv, C, D, num_splits)


def attend_indexed_plan(B, Hq, Hkv, topk, D, dtype=torch.bfloat16, num_splits=0):
    return _plan("kvd_attend_indexed_plan", B, Hq, Hkv, topk, D,
                 BF16 if dtype == torch.bfloat16 else F32, num_splits)


def attend_paged_plan(Q, Hq, Hkv, BS, cols, D, dtype=torch.bfloat16, num_splits=0):
    return _plan("kvd_attend_paged_plan", Q, Hq, Hkv, BS, cols, D,
                 BF16 if dtype == torch.bfloat16 else F32, num_splits)


def workspace_partials(ws, plan, R, D):
    """Views of a workspace's partial rows for a Plan from one of the *_plan
    queries: (part_o [R, S, D], part_lse [R, S]) fp32, or None without
    partial rows (splits <= 1)."""
    S, lo, oo = plan.splits, plan.lse_offset, plan.o_offset
    if S <= 1:
        return None
    flat = ws.view(torch.uint8)
    part_lse = flat[lo:lo + R * S * 4].view(torch.float32).view(R, S)
    part_o = flat[oo:oo + R * S * D * 4].view(torch.float32).view(R, S, D)
    return part_o, part_lse


def attend_masked_partial(q, k_cache, v_cache, mask, scale=None, out=None, lse=None, num_splits=0,
                          workspace=None, dev_status=None):
    """kvd_attend_masked_partial: attend_masked with fp32 output rows and
    their log-sum-exp -- the partial of one token range, merged with the
    other ranges' by combine / combine_gathered.  Returns (out [B, Hq, D]
    fp32, lse [B, Hq] fp32)."""
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("mask", mask)):
        _cuda_contig(n, t)
    B, Hq, D = q.shape
    Bk, Hkv, C, Dk = k_cache.shape
    if Bk != B or Dk != D or v_cache.shape != k_cache.shape or mask.shape != (B, C):
        raise ValueError("attend_masked_partial: shape mismatch")
    if mask.dtype != torch.uint8 or not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("attend_masked_partial: uint8 mask and one dtype for q and caches")
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    for n, t in (("out", out), ("lse", lse)):
        _cuda_contig(n, t)
        if t.dtype != torch.float32:
            raise TypeError(f"attend_masked_partial: {n} must be fp32")
    L = load()
    need = L.kvd_attend_masked_workspace_bytes(B, Hq, Hkv, C, D, dt, num_splits)
    ws, wsb = _workspace(need, q.device, workspace)
    st = L.kvd_attend_masked_partial(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(mask), _ptr(out),
                                     _ptr(lse), B, Hq, Hkv, C, D, float(scale), dt, num_splits,
                                     _ptr(ws), wsb, _ptr(dev_status), _stream(q.device))
    _check("kvd_attend_masked_partial", st)
    return out, lse


def append_attend_masked(q, k_cache, v_cache, mask, k_new, v_new, pos, scale=None, out=None,
                         lse=None, num_splits=0, workspace=None, dev_status=None):
    """kvd_append_attend_masked: kvd_append then kvd_attend_masked in one call
    (one launch when Hq / Hkv <= 8).  Returns out [B, Hq, D]."""
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("mask", mask),
                 ("k_new", k_new), ("v_new", v_new), ("pos", pos)):
        _cuda_contig(n, t)
    B, Hq, D = q.shape
    Bk, Hkv, C, Dk = k_cache.shape
    if Bk != B or Dk != D or v_cache.shape != k_cache.shape or mask.shape != (B, C) or \
            k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D):
        raise ValueError("append_attend_masked: shape mismatch")
    if mask.dtype != torch.uint8 or pos.dtype != torch.int32 or pos.numel() != B:
        raise ValueError("append_attend_masked: mask uint8 [B, C], pos int32 [B]")
    if not (q.dtype == k_cache.dtype == v_cache.dtype == k_new.dtype == v_new.dtype):
        raise TypeError("append_attend_masked: q, caches and new rows must share a dtype")
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is not None:
        _cuda_contig("lse", lse)
    L = load()
    need = L.kvd_attend_masked_workspace_bytes(B, Hq, Hkv, C, D, dt, num_splits)
    ws, wsb = _workspace(need, q.device, workspace)
    st = L.kvd_append_attend_masked(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(mask), _ptr(k_new),
                                    _ptr(v_new), _ptr(pos), _ptr(out), _ptr(lse), B, Hq, Hkv, C,
                                    D, float(scale), dt, num_splits, _ptr(ws), wsb,
                                    _ptr(dev_status), _stream(q.device))
    _check("kvd_append_attend_masked", st)
    return out


def attend_window_workspace_bytes(B, Hq, Hkv, C, D, W, dtype=torch.bfloat16, num_splits=0):
    return load().kvd_attend_window_workspace_bytes(B, Hq, Hkv, C, D, W,
                                                    BF16 if dtype == torch.bfloat16 else F32,
                                                    num_splits)


def attend_window_plan(B, Hq, Hkv, C, D, W, dtype=torch.bfloat16, num_splits=0):
    return _plan("kvd_attend_window_plan", B, Hq, Hkv, C, D, W,
                 BF16 if dtype == torch.bfloat16 else F32, num_splits)


def _window_args(fn, q, k_cache, v_cache, mask, W, rows, extra):
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("mask", mask)) + extra:
        _cuda_contig(n, t)
    B, Hq, D = q.shape
    Bk, Hkv, C, Dk = k_cache.shape
    if Bk != B or Dk != D or v_cache.shape != k_cache.shape or mask.shape != (B, C):
        raise ValueError(f"{fn}: shape mismatch")
    if mask.dtype != torch.uint8 or rows.dtype != torch.int32 or rows.numel() != B:
        raise ValueError(f"{fn}: mask uint8 [B, C], positions int32 [B]")
    if int(W) < 1:
        raise ValueError(f"{fn}: W >= 1 required")
    return B, Hq, Hkv, C, D


def attend_window(q, k_cache, v_cache, mask, last, W, scale=None, out=None, lse=None,
                  num_splits=0, workspace=None, dev_status=None):
    """kvd_attend_window: row b attends to the masked slots of
    [last[b] - W + 1, last[b]].  Returns out [B, Hq, D]."""
    B, Hq, Hkv, C, D = _window_args("attend_window", q, k_cache, v_cache, mask, W, last,
                                    (("last", last),))
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("attend_window: q and caches must share a dtype")
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is not None:
        _cuda_contig("lse", lse)
    L = load()
    need = L.kvd_attend_window_workspace_bytes(B, Hq, Hkv, C, D, int(W), dt, num_splits)
    ws, wsb = _workspace(need, q.device, workspace)
    st = L.kvd_attend_window(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(mask), _ptr(last),
                             _ptr(out), _ptr(lse), B, Hq, Hkv, C, D, int(W), float(scale), dt,
                             num_splits, _ptr(ws), wsb, _ptr(dev_status), _stream(q.device))
    _check("kvd_attend_window", st)
    return out


def append_attend_window(q, k_cache, v_cache, mask, k_new, v_new, pos, W, scale=None, out=None,
                         lse=None, num_splits=0, workspace=None, dev_status=None):
    """kvd_append_attend_window: kvd_append then kvd_attend_window with
    last = pos, in one launch when Hq / Hkv <= 8.  Returns out [B, Hq, D]."""
    B, Hq, Hkv, C, D = _window_args("append_attend_window", q, k_cache, v_cache, mask, W, pos,
                                    (("k_new", k_new), ("v_new", v_new), ("pos", pos)))
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D):
        raise ValueError("append_attend_window: shape mismatch")
    if not (q.dtype == k_cache.dtype == v_cache.dtype == k_new.dtype == v_new.dtype):
        raise TypeError("append_attend_window: q, caches and new rows must share a dtype")
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is not None:
        _cuda_contig("lse", lse)
    L = load()
    need = L.kvd_attend_window_workspace_bytes(B, Hq, Hkv, C, D, int(W), dt, num_splits)
    ws, wsb = _workspace(need, q.device, workspace)
    st = L.kvd_append_attend_window(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(mask),
                                    _ptr(k_new), _ptr(v_new), _ptr(pos), _ptr(out), _ptr(lse), B,
                                    Hq, Hkv, C, D, int(W), float(scale), dt, num_splits, _ptr(ws),
                                    wsb, _ptr(dev_status), _stream(q.device))
    _check("kvd_append_attend_window", st)
    return out


def attend_indexed_workspace_bytes(B, Hq, Hkv, topk, D, dtype=torch.bfloat16, num_splits=0):
    return load().kvd_attend_indexed_workspace_bytes(B, Hq, Hkv, topk, D,
                                                     BF16 if dtype == torch.bfloat16 else F32,
                                                     num_splits)


def attend_indexed(q, k_cache, v_cache, indices, scale=None, out=None, lse=None, num_splits=0,
                   workspace=None, dev_status=None):
    """kvd_attend_indexed: decode attention over the cache slots listed in
    indices [B, topk] int32 (-1 = unused entry).

    q [B, Hq, D]; k_cache, v_cache [B, Hkv, C, D].  Returns out [B, Hq, D];
    fills ``lse`` [B, Hq] fp32 if given.
    """
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("indices", indices)):
        _cuda_contig(n, t)
    B, Hq, D = q.shape
    Bk, Hkv, C, Dk = k_cache.shape
    if Bk != B or Dk != D or v_cache.shape != k_cache.shape or indices.dim() != 2 or \
            indices.shape[0] != B:
        raise ValueError("attend_indexed: shape mismatch")
    if indices.dtype != torch.int32:
        raise ValueError("attend_indexed: indices must be int32")
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("attend_indexed: q and caches must share a dtype")
    topk = indices.shape[1]
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is not None:
        _cuda_contig("lse", lse)
    L = load()
    need = L.kvd_attend_indexed_workspace_bytes(B, Hq, Hkv, topk, D, dt, num_splits)
    ws, wsb = _workspace(need, q.device, workspace)
    st = L.kvd_attend_indexed(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(indices), _ptr(out),
                              _ptr(lse), B, Hq, Hkv, C, topk, D, float(scale), dt, num_splits,
                              _ptr(ws), wsb, _ptr(dev_status), _stream(q.device))
    _check("kvd_attend_indexed", st)
    return out


def attend_masked_noalloc(q, k_cache, v_cache, mask, scale=None, out=None, lse=None,
                          num_splits=0, dev_status=None):
    """kvd_attend_masked_noalloc: attend_masked for callers that cannot
    allocate -- the split scratch is the library's built-in array (see
    include/kvd.h for its size limit and sharing rules); ``out`` is the only
    tensor this wrapper creates, and only when none is passed."""
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("mask", mask)):
        _cuda_contig(n, t)
    B, Hq, D = q.shape
    Bk, Hkv, C, Dk = k_cache.shape
    if Bk != B or Dk != D or v_cache.shape != k_cache.shape or mask.shape != (B, C):
        raise ValueError("attend_masked_noalloc: shape mismatch")
    if mask.dtype != torch.uint8 or not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("attend_masked_noalloc: uint8 mask and one dtype for q and caches")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    st = load().kvd_attend_masked_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(mask),
                                          _ptr(out), _ptr(lse), B, Hq, Hkv, C, D, float(scale),
                                          _dtype_code(q), num_splits, _ptr(dev_status),
                                          _stream(q.device))
    _check("kvd_attend_masked_noalloc", st)
    return out


def attend_paged_workspace_bytes(Q, Hq, Hkv, BS, cols, D, dtype=torch.bfloat16, num_splits=0):
    return load().kvd_attend_paged_workspace_bytes(Q, Hq, Hkv, BS, cols, D,
                                                   BF16 if dtype == torch.bfloat16 else F32,
                                                   num_splits)


def attend_paged(q, key_cache, value_cache, block_tables, seq_lens, seq_offset=None, scale=None,
                 out=None, lse=None, num_splits=0, workspace=None, dev_status=None):
    """kvd_attend_paged: decode attention over the paged cache.

    q [Q, Hq, D]; caches [NB, BS, Hkv, D]; block_tables [Q, cols] int32;
    seq_lens [Q + 1] int32 cumsum; seq_offset [Q] int32 or None.
    """
    for n, t in (("q", q), ("key_cache", key_cache), ("value_cache", value_cache),
                 ("block_tables", block_tables), ("seq_lens", seq_lens)):
        _cuda_contig(n, t)
    Q, Hq, D = q.shape
    NB, BS, Hkv, Dk = key_cache.shape
    if Dk != D or value_cache.shape != key_cache.shape:
        raise ValueError("attend_paged: shape mismatch")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != Q:
        raise ValueError("attend_paged: block_tables must be int32 [Q, cols]")
    if seq_lens.dtype != torch.int32 or seq_lens.shape != (Q + 1,):
        raise ValueError("attend_paged: only cumsum seq_lens [Q+1] int32 is supported")
    if seq_offset is not None:
        _cuda_contig("seq_offset", seq_offset)
        if seq_offset.dtype != torch.int32 or seq_offset.shape != (Q,):
            raise ValueError("attend_paged: seq_offset must be int32 [Q]")
    cols = block_tables.shape[1]
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    L = load()
    need = L.kvd_attend_paged_workspace_bytes(Q, Hq, Hkv, BS, cols, D, dt, num_splits)
    ws, wsb = _workspace(need, q.device, workspace)
    st = L.kvd_attend_paged(_ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
                            _ptr(seq_lens), _ptr(seq_offset), _ptr(out), _ptr(lse), Q, Hq, Hkv,
                            NB, BS, cols, D, float(scale), dt, num_splits, _ptr(ws), wsb,
                            _ptr(dev_status), _stream(q.device))
    _check("kvd_attend_paged", st)
    return out


# ------------------------------------------------------------------ gather

def append_paged(key_cache, value_cache, block_tables, seq_offset, k_new, v_new, pos,
                 dev_status=None):
    """kvd_append_paged: token pos[q] of every sequence q into the paged
    caches [NB, BS, Hkv, D] (k_new, v_new [Q, Hkv, D], pos [Q] int32)."""
    for n, t in (("key_cache", key_cache), ("value_cache", value_cache), ("k_new", k_new),
                 ("v_new", v_new), ("block_tables", block_tables), ("pos", pos)):
        _cuda_contig(n, t)
    NB, BS, Hkv, D = key_cache.shape
    Q, cols = block_tables.shape
    if value_cache.shape != key_cache.shape or k_new.shape != (Q, Hkv, D) or \
            v_new.shape != (Q, Hkv, D) or pos.numel() != Q:
        raise ValueError("append_paged: shape mismatch")
    if block_tables.dtype != torch.int32 or pos.dtype != torch.int32 or \
            (seq_offset is not None and seq_offset.dtype != torch.int32):
        raise ValueError("append_paged: int32 tables, offsets and positions")
    if not (key_cache.dtype == value_cache.dtype == k_new.dtype == v_new.dtype):
        raise TypeError("append_paged: caches and new rows must share a dtype")
    st = load().kvd_append_paged(_ptr(key_cache), _ptr(value_cache), _ptr(k_new), _ptr(v_new),
                                 _ptr(block_tables), _ptr(seq_offset), _ptr(pos), Q, NB, BS, cols,
                                 Hkv, D, _dtype_code(key_cache), _ptr(dev_status),
                                 _stream(key_cache.device))
    _check("kvd_append_paged", st)


def gather_paged(key_cache, value_cache, block_tables, seq_lens, seq_offset=None,
                 key_out=None, value_out=None, total_tokens=None, dev_status=None):
    """kvd_gather_paged (gather_pa_kv_cache): copy the pages of every sequence
    into contiguous [total_tokens, H, D] outputs.  Allocates the outputs when
    not given; ``total_tokens`` defaults to seq_lens[-1] (read once to size the
    outputs when they are allocated here)."""
    for n, t in (("key_cache", key_cache), ("value_cache", value_cache),
                 ("block_tables", block_tables), ("seq_lens", seq_lens)):
        _cuda_contig(n, t)
    NB, BS, Hk, Dk = key_cache.shape
    NBv, BSv, Hv, Dv = value_cache.shape
    if (NB, BS) != (NBv, BSv) or key_cache.dtype != value_cache.dtype:
        raise ValueError("gather_paged: caches disagree on blocks or dtype")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2:
        raise ValueError("gather_paged: block_tables must be int32 [Q, cols]")
    Q, cols = block_tables.shape
    if seq_lens.dtype != torch.int32 or seq_lens.shape != (Q + 1,):
        raise ValueError("gather_paged: only cumsum seq_lens [Q+1] int32 is supported")
    if seq_offset is not None:
        _cuda_contig("seq_offset", seq_offset)
    if total_tokens is None:
        total_tokens = int(key_out.shape[0]) if key_out is not None else int(seq_lens[-1].item())
    if key_out is None:
        key_out = torch.empty((total_tokens, Hk, Dk), dtype=key_cache.dtype, device=key_cache.device)
    if value_out is None:
        value_out = torch.empty((total_tokens, Hv, Dv), dtype=value_cache.dtype,
                                device=value_cache.device)
    if key_out.shape != (total_tokens, Hk, Dk) or value_out.shape != (total_tokens, Hv, Dv):
        raise ValueError("gather_paged: output shapes must be [total_tokens, H, D]")
    st = load().kvd_gather_paged(_ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
                                 _ptr(seq_lens), _ptr(seq_offset), _ptr(key_out), _ptr(value_out),
                                 Q, NB, BS, cols, Hk, Dk, Hv, Dv, total_tokens,
                                 key_cache.element_size(), _ptr(dev_status),
                                 _stream(key_cache.device))
    _check("kvd_gather_paged", st)
    return key_out, value_out


# ------------------------------------------------------------------ combine

def combine(part_o, part_lse, out=None, lse=None, out_dtype=torch.float32):
    """kvd_combine: log-sum-exp merge of part_o [R, S, D] by part_lse [R, S]."""
    _cuda_contig("part_o", part_o)
    _cuda_contig("part_lse", part_lse)
    R, S, D = part_o.shape
    if part_lse.shape != (R, S) or part_o.dtype != torch.float32 or part_lse.dtype != torch.float32:
        raise ValueError("combine: part_o [R,S,D] and part_lse [R,S] fp32 required")
    if out is None:
        out = torch.empty((R, D), dtype=out_dtype, device=part_o.device)
    st = load().kvd_combine(_ptr(part_o), _ptr(part_lse), _ptr(out), _ptr(lse), R, S, D,
                            _dtype_code(out), _stream(part_o.device))
    _check("kvd_combine", st)
    return out


def combine_gathered(parts, R, D, out=None, lse=None, out_dtype=torch.float32):
    """kvd_combine_gathered: log-sum-exp merge of S ranges' packed partials,
    parts fp32 [S, R * (D + 1)] (per range: R rows of D, then R lse)."""
    _cuda_contig("parts", parts)
    if parts.dtype != torch.float32 or parts.dim() != 2 or parts.shape[1] != R * (D + 1):
        raise ValueError("combine_gathered: parts fp32 [S, R * (D + 1)] required")
    S = parts.shape[0]
    if out is None:
        out = torch.empty((R, D), dtype=out_dtype, device=parts.device)
    st = load().kvd_combine_gathered(_ptr(parts), _ptr(out), _ptr(lse), R, S, D, _dtype_code(out),
                                     _stream(parts.device))
    _check("kvd_combine_gathered", st)
    return out
