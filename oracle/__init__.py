"""fp64 CPU oracle for decode-phase KV-cache attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package never imports the CUDA library: the two share no code.  The arithmetic
lives in ``kvd_oracle.c`` (plain loops in double); this module only builds it
with gcc and marshals arrays.

Every function states what it computes and the page section it follows:

* ``attend_masked`` -- "Intel NPU running LLMs" (OpenVINO community article
  882), Part 1 "解决方案：预分配 + Attention Mask" and Part 3 "Attention 在 NPU
  上的完整实现"; "FlashMLA на Huawei Ascend", "Математическая постановка".
* ``attend_window`` -- ``attend_masked`` with every mask slot outside the
  sliding window [last - W + 1, last] taken as 0 (Part 3's sliding-window
  tile variant, expressed on Part 1's mask).
* ``append`` -- same article, Part 2 "NPUW 的核心设计" (update_kvcache_for).
* ``gather_paged`` -- "PyPTO 实现 AscendC GatherPaKvCache（Norm/ND 分支）",
  sections 3.1-3.3 and 7.
* ``append_paged`` -- the append of Part 2 ("update_kvcache_for") into the
  paged layout, through the gather's index mapping (section 3.2).
* ``attend_paged`` -- gather (above) followed by ``attend_masked`` with an
  all-ones mask.
* ``e4m3_codes``, ``e4m3_values``, ``quantize_rows``, ``append_fp8``,
  ``attend_masked_fp8`` -- quantised KV rows: "FlashMLA на Huawei Ascend",
  "Ограничение по деквантованию" (decoding reads FP8 KV and dequantises it)
  and "Оптимизация раскладки KV-кэша при decoding" (values and scale of a
  token side by side); the scale encoding is this package's reading: one fp32
  absmax/448 scale per row, after the row's E4M3 codes, rows padded to D + 16
  bytes.
* ``e2m1_codes``, ``e2m1_values``, ``quantize_rows_fp4``, ``append_fp4``,
  ``attend_masked_fp4`` -- the FP4 rows the same section names beside FP8:
  E2M1 codes two per byte (element 2j in the low nibble of byte j), one fp32
  absmax/6 scale per row after them, rows padded to D/2 + 16 bytes.
* ``combine`` -- the log-sum-exp merge of disjoint key ranges (Part 3, "Flash
  SDPA 路径": tiles merged exactly through running max and sum).
* ``append_paged_quant``, ``attend_paged_quant``, ``attend_indexed_quant`` --
  the quantised rows above in the paged layout and through index lists (the
  FlashMLA page motivates the value + scale layout on paged KV blocks):
  compositions of the row quantisers, the paged append and gather (whole
  rows as bytes) and the static-buffer attention over quantised rows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkvd_oracle.so")

BF16 = 0
F32 = 1
FP8_ROW_PAD = 16  # bytes after the D codes of a quantised row: fp32 scale + 12 zero bytes

ERR_POS = 1
ERR_BLOCK = 2
ERR_COLS = 4
ERR_SEQLENS = 8
ERR_OFFSET = 16

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libkvd_oracle.so`` with gcc.

    No fast-math and no floating-point contraction, so the sums are evaluated
    exactly in the order the C source writes them on every host.
    """
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            vp, i32p, dp, u8p = (ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32),
                                 ctypes.POINTER(ctypes.c_double),
                                 ctypes.POINTER(ctypes.c_uint8))
            ci, cd = ctypes.c_int, ctypes.c_double
            L.kvd_oracle_attend_masked.argtypes = [vp, vp, vp, u8p, ci, ci, ci, ci, ci, ci,
                                                   cd, dp, dp, ci]
            L.kvd_oracle_append.argtypes = [vp, vp, vp, vp, i32p, u8p, ci, ci, ci, ci, ci]
            L.kvd_oracle_attend_indexed.argtypes = [vp, vp, vp, i32p, ci, ci, ci, ci, ci, ci, ci,
                                                    cd, dp, dp, ci]
            L.kvd_oracle_copy_prefix.argtypes = [vp, vp, vp, vp, u8p, i32p, ci, ci, ci, ci, ci, ci]
            L.kvd_oracle_gather_paged.argtypes = [vp, vp, i32p, i32p, i32p, vp, vp] + [ci] * 10
            L.kvd_oracle_append_paged.argtypes = [vp, vp, i32p, i32p, vp, vp, i32p] + [ci] * 7
            L.kvd_oracle_attend_paged.argtypes = [vp, vp, vp, i32p, i32p, i32p] + [ci] * 8 + [
                cd, dp, dp, ci]
            L.kvd_oracle_combine.argtypes = [dp, dp, ci, ci, ci, dp, dp]
            L.kvd_oracle_threads.argtypes = []
            cl = ctypes.c_long
            L.kvd_oracle_e4m3_codes.argtypes = [ctypes.POINTER(ctypes.c_float), cl, u8p]
            L.kvd_oracle_e4m3_values.argtypes = [u8p, cl, dp]
            L.kvd_oracle_quantize_rows.argtypes = [vp, ci, cl, ci, u8p]
            L.kvd_oracle_append_fp8.argtypes = [u8p, u8p, vp, vp, ci, i32p, u8p, ci, ci, ci, ci]
            L.kvd_oracle_attend_masked_fp8.argtypes = [vp, ci, u8p, u8p, u8p, ci, ci, ci, ci, ci,
                                                       cd, dp, dp, ci]
            L.kvd_oracle_e2m1_codes.argtypes = [ctypes.POINTER(ctypes.c_float), cl, u8p]
            L.kvd_oracle_e2m1_values.argtypes = [u8p, cl, dp]
            L.kvd_oracle_quantize_rows_fp4.argtypes = [vp, ci, cl, ci, u8p]
            L.kvd_oracle_append_fp4.argtypes = [u8p, u8p, vp, vp, ci, i32p, u8p, ci, ci, ci, ci]
            L.kvd_oracle_attend_masked_fp4.argtypes = [vp, ci, u8p, u8p, u8p, ci, ci, ci, ci, ci,
                                                       cd, dp, dp, ci]
            for f in (L.kvd_oracle_attend_masked, L.kvd_oracle_append, L.kvd_oracle_copy_prefix,
                      L.kvd_oracle_attend_indexed,
                      L.kvd_oracle_gather_paged, L.kvd_oracle_attend_paged,
                      L.kvd_oracle_append_paged,
                      L.kvd_oracle_combine, L.kvd_oracle_threads):
                f.restype = ctypes.c_int
            _lib = L
    return _lib


def threads() -> int:
    """Threads the oracle's parallel loops use by default (OpenMP)."""
    return lib().kvd_oracle_threads()


# ---------------------------------------------------------------- marshalling

def _storage(x):
    """Return (contiguous numpy array holding the raw elements, dtype code).

    Accepts torch CPU tensors (bfloat16 or float32) and numpy float32 arrays;
    bf16 elements travel as their 16-bit patterns and are widened in C.
    """
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.float32:
                return x.numpy(), F32
            raise TypeError(f"oracle: unsupported tensor dtype {x.dtype}")
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    raise TypeError(f"oracle: unsupported array dtype {x.dtype}")


def _bytes_view(x):
    """Contiguous numpy view of the raw bytes of a tensor/array (for copies)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            return x.view(torch.uint8).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x).view(np.uint8)


def _i32(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().to(torch.int32).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.int32)


def _u8(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().to(torch.uint8).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.uint8)


def _p(a, t=None):
    if t is None:
        return a.ctypes.data_as(ctypes.c_void_p)
    return a.ctypes.data_as(ctypes.POINTER(t))


# ------------------------------------------------------------------ functions

def attend_masked(q, k, v, mask, scale: float, nthreads: int = 0):
    """Masked decode attention, fp64.

    q [B, Hq, D]; k, v [B, Hkv, C, D]; mask [B, C] (nonzero = valid).
    Returns (out [B, Hq, D] float64, lse [B, Hq] float64, natural log).
    """
    qa, dt = _storage(q)
    ka, dk = _storage(k)
    va, dv = _storage(v)
    if not (dt == dk == dv):
        raise TypeError("oracle: q, k, v must share one element type")
    B, Hq, D = qa.shape
    _, Hkv, C, Dk = ka.shape
    if Dk != D or va.shape != ka.shape:
        raise ValueError("oracle: shape mismatch")
    m = _u8(mask).reshape(B, C) if C > 0 else np.zeros((B, 1), np.uint8)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = lib().kvd_oracle_attend_masked(_p(qa), _p(ka), _p(va), _p(m, ctypes.c_uint8), dt,
                                        B, Hq, Hkv, C, D, float(scale),
                                        _p(out, ctypes.c_double), _p(lse, ctypes.c_double),
                                        int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle attend_masked failed ({rc})")
    return out, lse


def attend_window(q, k, v, mask, last, W: int, scale: float, nthreads: int = 0):
    """Sliding-window decode attention, fp64: row b attends to the slots j
    with mask[b, j] != 0 and last[b] - W + 1 <= j <= last[b]; a row whose
    last[b] is outside [0, C) attends to nothing.
    Returns (out [B, Hq, D] float64, lse [B, Hq] float64, error bits: 1 when
    some last[b] is outside [0, C))."""
    ka, _ = _storage(k)
    B, C = ka.shape[0], ka.shape[2]
    m = _u8(mask).reshape(B, C).copy()
    lst = _i32(last).reshape(B)
    bad = 0
    j = np.arange(C)
    for b in range(B):
        t = int(lst[b])
        if t < 0 or t >= C:
            bad = 1
            m[b, :] = 0
        else:
            m[b, (j < t - int(W) + 1) | (j > t)] = 0
    out, lse = attend_masked(q, k, v, m, scale, nthreads)
    return out, lse, bad


def attend_indexed(q, k, v, indices, scale: float, nthreads: int = 0):
    """Index-list decode attention, fp64: every entry j with 0 <= idx[b, j] <
    C of indices [B, topk] is one softmax term over k, v [B, Hkv, C, D].
    Returns (out [B, Hq, D] float64, lse [B, Hq] float64, error bits)."""
    qa, dt = _storage(q)
    ka, dk = _storage(k)
    va, dv = _storage(v)
    if not (dt == dk == dv):
        raise TypeError("oracle: q, k, v must share one element type")
    B, Hq, D = qa.shape
    _, Hkv, C, Dk = ka.shape
    if Dk != D or va.shape != ka.shape:
        raise ValueError("oracle: shape mismatch")
    idx = _i32(indices).reshape(B, -1)
    topk = idx.shape[1]
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = lib().kvd_oracle_attend_indexed(_p(qa), _p(ka), _p(va), _p(idx, ctypes.c_int32), dt, B,
                                         Hq, Hkv, C, topk, D, float(scale),
                                         _p(out, ctypes.c_double), _p(lse, ctypes.c_double),
                                         int(nthreads))
    if rc < 0:
        raise RuntimeError(f"oracle attend_indexed failed ({rc})")
    return out, lse, rc


def append(k_cache, v_cache, k_new, v_new, pos, mask=None) -> int:
    """KV append in place on numpy arrays (any element type, byte copy).

    k_cache, v_cache [B, Hkv, C, D] (numpy, modified); k_new, v_new [B, Hkv, D];
    pos [B]; mask [B, C] uint8 numpy (modified) or None.  Returns error bits.
    """
    if not (isinstance(k_cache, np.ndarray) and isinstance(v_cache, np.ndarray)):
        raise TypeError("oracle.append works in place on numpy arrays")
    B, Hkv, C, D = k_cache.shape
    eb = k_cache.dtype.itemsize
    kn = np.ascontiguousarray(_bytes_view(k_new))
    vn = np.ascontiguousarray(_bytes_view(v_new))
    if kn.size != B * Hkv * D * eb or vn.size != kn.size:
        raise ValueError("oracle.append: new rows have the wrong size")
    p = _i32(pos)
    mp = None
    if mask is not None:
        if not (isinstance(mask, np.ndarray) and mask.dtype == np.uint8 and mask.flags.c_contiguous):
            raise TypeError("oracle.append: mask must be a contiguous uint8 numpy array")
        mp = _p(mask, ctypes.c_uint8)
    return lib().kvd_oracle_append(_p(k_cache), _p(v_cache), _p(kn), _p(vn),
                                   _p(p, ctypes.c_int32), mp, B, Hkv, C, D, eb)


def copy_prefix(k_src, v_src, k_dst, v_dst, n, mask=None) -> int:
    """copy_kvcache for one layer, in place on numpy arrays (byte copy):
    rows [0, n[b]) of k_src/v_src [B, Hkv, C_src, D] go to the same rows of
    k_dst/v_dst [B, Hkv, C_dst, D]; mask [B, C_dst] uint8 (or None) becomes
    the prefix mask of n[b].  Returns error bits (ERR_POS for an n[b] outside
    [0, min(C_src, C_dst)])."""
    for name, a in (("k_dst", k_dst), ("v_dst", v_dst)):
        if not (isinstance(a, np.ndarray) and a.flags.c_contiguous):
            raise TypeError(f"oracle.copy_prefix: {name} must be a contiguous numpy array")
    B, Hkv, C_dst, D = k_dst.shape
    ks = np.ascontiguousarray(_bytes_view(k_src))
    vs = np.ascontiguousarray(_bytes_view(v_src))
    eb = k_dst.dtype.itemsize
    C_src = ks.size // (B * Hkv * D * eb)
    if ks.size != B * Hkv * C_src * D * eb or vs.size != ks.size or v_dst.shape != k_dst.shape:
        raise ValueError("oracle.copy_prefix: shape mismatch")
    mp = None
    if mask is not None:
        if not (isinstance(mask, np.ndarray) and mask.dtype == np.uint8 and mask.flags.c_contiguous):
            raise TypeError("oracle.copy_prefix: mask must be a contiguous uint8 numpy array")
        mp = _p(mask, ctypes.c_uint8)
    return lib().kvd_oracle_copy_prefix(_p(ks), _p(vs), _p(k_dst), _p(v_dst), mp,
                                        _p(_i32(n), ctypes.c_int32), B, Hkv, C_src, C_dst, D, eb)


def gather_paged(key_cache, value_cache, block_tables, seq_lens, seq_offset=None,
                 total_tokens=None):
    """gather_pa_kv_cache on numpy arrays (byte copy).

    key_cache [NB, BS, Hk, Dk], value_cache [NB, BS, Hv, Dv] numpy arrays of
    one element type; block_tables [Q, cols]; seq_lens [Q+1] cumsum;
    seq_offset [Q] or None.  Returns (key_out, value_out, error bits).
    Rows that are not written (error cases) stay zero.
    """
    kc = np.ascontiguousarray(key_cache)
    vc = np.ascontiguousarray(value_cache)
    if kc.dtype != vc.dtype:
        raise TypeError("oracle.gather_paged: caches must share one element type")
    NB, BS, Hk, Dk = kc.shape
    NBv, BSv, Hv, Dv = vc.shape
    if (NB, BS) != (NBv, BSv):
        raise ValueError("oracle.gather_paged: caches disagree on blocks")
    bt = _i32(block_tables)
    Q, cols = bt.shape
    sl = _i32(seq_lens)
    if sl.shape != (Q + 1,):
        raise ValueError("oracle.gather_paged: only cumsum seq_lens [Q+1] is supported")
    so = None if seq_offset is None else _i32(seq_offset)
    T = int(sl[-1]) if total_tokens is None else int(total_tokens)
    ko = np.zeros((max(T, 0), Hk, Dk), kc.dtype)
    vo = np.zeros((max(T, 0), Hv, Dv), vc.dtype)
    err = lib().kvd_oracle_gather_paged(_p(kc), _p(vc), _p(bt, ctypes.c_int32),
                                        _p(sl, ctypes.c_int32),
                                        None if so is None else _p(so, ctypes.c_int32),
                                        _p(ko), _p(vo), Q, NB, BS, cols, Hk, Dk, Hv, Dv, T,
                                        kc.dtype.itemsize)
    return ko, vo, err


def append_paged(key_cache, value_cache, block_tables, seq_offset, k_new, v_new, pos) -> int:
    """Paged KV append in place on numpy caches [NB, BS, Hkv, D] (any element
    type, byte copy): token pos[q] of sequence q goes to the block and slot
    the paged gather reads it from (same index mapping); k_new, v_new
    [Q, Hkv, D]; seq_offset [Q] or None.  Returns error bits."""
    if not (isinstance(key_cache, np.ndarray) and isinstance(value_cache, np.ndarray)):
        raise TypeError("oracle.append_paged works in place on numpy arrays")
    NB, BS, Hkv, D = key_cache.shape
    eb = key_cache.dtype.itemsize
    bt = _i32(block_tables)
    Q, cols = bt.shape
    kn = np.ascontiguousarray(_bytes_view(k_new))
    vn = np.ascontiguousarray(_bytes_view(v_new))
    if kn.size != Q * Hkv * D * eb or vn.size != kn.size:
        raise ValueError("oracle.append_paged: new rows have the wrong size")
    p = _i32(pos)
    so = None if seq_offset is None else _i32(seq_offset)
    return lib().kvd_oracle_append_paged(_p(key_cache), _p(value_cache), _p(bt, ctypes.c_int32),
                                         None if so is None else _p(so, ctypes.c_int32),
                                         _p(kn), _p(vn), _p(p, ctypes.c_int32), Q, NB, BS, cols,
                                         Hkv, D, eb)


def attend_paged(q, key_cache, value_cache, block_tables, seq_lens, seq_offset, scale: float,
                 nthreads: int = 0):
    """Paged decode attention, fp64: gather then attend with all-ones masks.

    q [Q, Hq, D]; caches [NB, BS, Hkv, D]; returns (out [Q, Hq, D], lse [Q, Hq]).
    """
    qa, dt = _storage(q)
    ka, dk = _storage(key_cache)
    va, dv = _storage(value_cache)
    if not (dt == dk == dv):
        raise TypeError("oracle: q and caches must share one element type")
    Q, Hq, D = qa.shape
    NB, BS, Hkv, Dk = ka.shape
    if Dk != D or va.shape != ka.shape:
        raise ValueError("oracle: shape mismatch")
    bt = _i32(block_tables)
    cols = bt.shape[1]
    sl = _i32(seq_lens)
    so = None if seq_offset is None else _i32(seq_offset)
    out = np.zeros((Q, Hq, D), np.float64)
    lse = np.zeros((Q, Hq), np.float64)
    rc = lib().kvd_oracle_attend_paged(_p(qa), _p(ka), _p(va), _p(bt, ctypes.c_int32),
                                       _p(sl, ctypes.c_int32),
                                       None if so is None else _p(so, ctypes.c_int32),
                                       dt, Q, Hq, Hkv, NB, BS, cols, D, float(scale),
                                       _p(out, ctypes.c_double), _p(lse, ctypes.c_double),
                                       int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle attend_paged failed ({rc})")
    return out, lse


def combine(part_o, part_lse):
    """Log-sum-exp combine: part_o [R, S, D], part_lse [R, S] -> (out [R, D], lse [R])."""
    po = np.ascontiguousarray(part_o, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    R, S, D = po.shape
    if pl.shape != (R, S):
        raise ValueError("oracle.combine: shape mismatch")
    out = np.zeros((R, D), np.float64)
    lse = np.zeros((R,), np.float64)
    lib().kvd_oracle_combine(_p(po, ctypes.c_double), _p(pl, ctypes.c_double), R, S, D,
                             _p(out, ctypes.c_double), _p(lse, ctypes.c_double))
    return out, lse


# ------------------------------------------------------------ quantised rows

def e4m3_codes(x) -> np.ndarray:
    """float32 values -> E4M3 codes (nearest, ties to even, saturating at 448)."""
    xa = np.ascontiguousarray(x, dtype=np.float32)
    out = np.zeros(xa.shape, np.uint8)
    lib().kvd_oracle_e4m3_codes(_p(xa, ctypes.c_float), xa.size, _p(out, ctypes.c_uint8))
    return out


def e4m3_values(codes) -> np.ndarray:
    """E4M3 codes -> their values (float64; NaN for the NaN codes)."""
    ca = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(ca.shape, np.float64)
    lib().kvd_oracle_e4m3_values(_p(ca, ctypes.c_uint8), ca.size, _p(out, ctypes.c_double))
    return out


def quantize_rows(x) -> np.ndarray:
    """Rows [..., D] (bf16 or fp32) -> quantised rows uint8 [..., D + 16]."""
    xa, dt = _storage(x)
    D = xa.shape[-1]
    rows = xa.size // D
    out = np.zeros(xa.shape[:-1] + (D + FP8_ROW_PAD,), np.uint8)
    rc = lib().kvd_oracle_quantize_rows(_p(xa), dt, rows, D, _p(out, ctypes.c_uint8))
    if rc != 0:
        raise RuntimeError("oracle quantize_rows failed")
    return out


def dequantize_rows(rows) -> np.ndarray:
    """Quantised rows uint8 [..., D + 16] -> float64 [..., D] (scale * value)."""
    ra = np.ascontiguousarray(rows, dtype=np.uint8)
    D = ra.shape[-1] - FP8_ROW_PAD
    scale = ra[..., D:D + 4].copy().view("<f4")[..., 0].astype(np.float64)
    return e4m3_values(ra[..., :D]) * scale[..., None]


def append_fp8(k_cache, v_cache, k_new, v_new, pos, mask=None) -> int:
    """Append into quantised caches in place: k_cache, v_cache uint8 numpy
    [B, Hkv, C, D + 16]; k_new, v_new [B, Hkv, D] (bf16 or fp32); pos [B];
    mask [B, C] uint8 numpy or None.  Returns error bits."""
    for a in (k_cache, v_cache):
        if not (isinstance(a, np.ndarray) and a.dtype == np.uint8 and a.flags.c_contiguous):
            raise TypeError("oracle.append_fp8 works in place on contiguous uint8 numpy arrays")
    B, Hkv, C, RB = k_cache.shape
    D = RB - FP8_ROW_PAD
    kn, dk = _storage(k_new)
    vn, dv = _storage(v_new)
    if dk != dv or kn.size != B * Hkv * D or vn.size != kn.size:
        raise ValueError("oracle.append_fp8: new rows have the wrong size or types")
    p = _i32(pos)
    mp = None
    if mask is not None:
        if not (isinstance(mask, np.ndarray) and mask.dtype == np.uint8 and mask.flags.c_contiguous):
            raise TypeError("oracle.append_fp8: mask must be a contiguous uint8 numpy array")
        mp = _p(mask, ctypes.c_uint8)
    return lib().kvd_oracle_append_fp8(_p(k_cache, ctypes.c_uint8), _p(v_cache, ctypes.c_uint8),
                                       _p(kn), _p(vn), dk, _p(p, ctypes.c_int32), mp, B, Hkv, C, D)


def attend_masked_fp8(q, k_rows, v_rows, mask, scale: float, nthreads: int = 0):
    """Masked decode attention over quantised K/V rows, fp64: q [B, Hq, D]
    (bf16 or fp32); k_rows, v_rows uint8 [B, Hkv, C, D + 16]; mask [B, C].
    Returns (out [B, Hq, D], lse [B, Hq])."""
    qa, dt = _storage(q)
    ka = np.ascontiguousarray(_u8(k_rows))
    va = np.ascontiguousarray(_u8(v_rows))
    B, Hq, D = qa.shape
    _, Hkv, C, RB = ka.shape
    if RB != D + FP8_ROW_PAD or va.shape != ka.shape:
        raise ValueError("oracle: shape mismatch")
    m = _u8(mask).reshape(B, C) if C > 0 else np.zeros((B, 1), np.uint8)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = lib().kvd_oracle_attend_masked_fp8(_p(qa), dt, _p(ka, ctypes.c_uint8),
                                            _p(va, ctypes.c_uint8), _p(m, ctypes.c_uint8), B, Hq,
                                            Hkv, C, D, float(scale), _p(out, ctypes.c_double),
                                            _p(lse, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle attend_masked_fp8 failed ({rc})")
    return out, lse


# ------------------------------------------------------------ FP4 rows

def e2m1_codes(x) -> np.ndarray:
    """float32 values -> E2M1 codes 0..15 (nearest, ties to the even code,
    saturating at 6; NaN -> +6)."""
    xa = np.ascontiguousarray(x, dtype=np.float32)
    out = np.zeros(xa.shape, np.uint8)
    lib().kvd_oracle_e2m1_codes(_p(xa, ctypes.c_float), xa.size, _p(out, ctypes.c_uint8))
    return out


def e2m1_values(codes) -> np.ndarray:
    """E2M1 codes 0..15 -> their values (float64)."""
    ca = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(ca.shape, np.float64)
    lib().kvd_oracle_e2m1_values(_p(ca, ctypes.c_uint8), ca.size, _p(out, ctypes.c_double))
    return out


def quantize_rows_fp4(x) -> np.ndarray:
    """Rows [..., D] (bf16 or fp32) -> FP4 rows uint8 [..., D/2 + 16]."""
    xa, dt = _storage(x)
    D = xa.shape[-1]
    rows = xa.size // D
    out = np.zeros(xa.shape[:-1] + (D // 2 + FP8_ROW_PAD,), np.uint8)
    rc = lib().kvd_oracle_quantize_rows_fp4(_p(xa), dt, rows, D, _p(out, ctypes.c_uint8))
    if rc != 0:
        raise RuntimeError("oracle quantize_rows_fp4 failed")
    return out


def dequantize_rows_fp4(rows) -> np.ndarray:
    """FP4 rows uint8 [..., D/2 + 16] -> float64 [..., D] (scale * value)."""
    ra = np.ascontiguousarray(rows, dtype=np.uint8)
    half = ra.shape[-1] - FP8_ROW_PAD
    scale = ra[..., half:half + 4].copy().view("<f4")[..., 0].astype(np.float64)
    codes = np.stack([ra[..., :half] & 0xF, ra[..., :half] >> 4], axis=-1).reshape(
        ra.shape[:-1] + (2 * half,))
    return e2m1_values(codes) * scale[..., None]


def append_fp4(k_cache, v_cache, k_new, v_new, pos, mask=None) -> int:
    """Append into FP4 caches in place: k_cache, v_cache uint8 numpy
    [B, Hkv, C, D/2 + 16]; k_new, v_new [B, Hkv, D] (bf16 or fp32); pos [B];
    mask [B, C] uint8 numpy or None.  Returns error bits."""
    for a in (k_cache, v_cache):
        if not (isinstance(a, np.ndarray) and a.dtype == np.uint8 and a.flags.c_contiguous):
            raise TypeError("oracle.append_fp4 works in place on contiguous uint8 numpy arrays")
    B, Hkv, C, RB = k_cache.shape
    D = 2 * (RB - FP8_ROW_PAD)
    kn, dk = _storage(k_new)
    vn, dv = _storage(v_new)
    if dk != dv or kn.size != B * Hkv * D or vn.size != kn.size:
        raise ValueError("oracle.append_fp4: new rows have the wrong size or types")
    p = _i32(pos)
    mp = None
    if mask is not None:
        if not (isinstance(mask, np.ndarray) and mask.dtype == np.uint8 and mask.flags.c_contiguous):
            raise TypeError("oracle.append_fp4: mask must be a contiguous uint8 numpy array")
        mp = _p(mask, ctypes.c_uint8)
    return lib().kvd_oracle_append_fp4(_p(k_cache, ctypes.c_uint8), _p(v_cache, ctypes.c_uint8),
                                       _p(kn), _p(vn), dk, _p(p, ctypes.c_int32), mp, B, Hkv, C, D)


def attend_masked_fp4(q, k_rows, v_rows, mask, scale: float, nthreads: int = 0):
    """Masked decode attention over FP4 K/V rows, fp64: q [B, Hq, D] (bf16 or
    fp32); k_rows, v_rows uint8 [B, Hkv, C, D/2 + 16]; mask [B, C].
    Returns (out [B, Hq, D], lse [B, Hq])."""
    qa, dt = _storage(q)
    ka = np.ascontiguousarray(_u8(k_rows))
    va = np.ascontiguousarray(_u8(v_rows))
    B, Hq, D = qa.shape
    _, Hkv, C, RB = ka.shape
    if RB != D // 2 + FP8_ROW_PAD or va.shape != ka.shape:
        raise ValueError("oracle: shape mismatch")
    m = _u8(mask).reshape(B, C) if C > 0 else np.zeros((B, 1), np.uint8)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = lib().kvd_oracle_attend_masked_fp4(_p(qa), dt, _p(ka, ctypes.c_uint8),
                                            _p(va, ctypes.c_uint8), _p(m, ctypes.c_uint8), B, Hq,
                                            Hkv, C, D, float(scale), _p(out, ctypes.c_double),
                                            _p(lse, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle attend_masked_fp4 failed ({rc})")
    return out, lse


# ------------------------------------- quantised rows in the paged layout and
# through index lists: compositions of the functions above (byte copies of
# whole quantised rows, then the static-buffer attention over the copies)

def _quant(fmt):
    if fmt == "fp8":
        return quantize_rows, attend_masked_fp8
    if fmt == "fp4":
        return quantize_rows_fp4, attend_masked_fp4
    raise ValueError(f"oracle: unknown row format {fmt!r}")


def append_paged_quant(key_rows, value_rows, block_tables, seq_offset, k_new, v_new, pos,
                       fmt: str) -> int:
    """Quantising paged append in place: the new rows k_new, v_new [Q, Hkv, D]
    (bf16 or fp32) quantised row by row (``quantize_rows`` / ``_fp4``), then
    written as whole rows through the paged gather's index mapping
    (``append_paged``) into key_rows, value_rows uint8 [NB, BS, Hkv, RB].
    Returns error bits."""
    quantize, _ = _quant(fmt)
    return append_paged(key_rows, value_rows, block_tables, seq_offset, quantize(k_new),
                        quantize(v_new), pos)


def attend_paged_quant(q, key_rows, value_rows, block_tables, seq_lens, seq_offset,
                       scale: float, fmt: str, nthreads: int = 0):
    """Paged decode attention over quantised rows, fp64: the paged gather of
    whole rows (``gather_paged``), then per sequence the static-buffer
    attention over quantised rows (``attend_masked_fp8`` / ``_fp4``) over its
    gathered rows, every one valid.  q [Q, Hq, D]; key_rows, value_rows uint8
    [NB, BS, Hkv, RB].  Returns (out [Q, Hq, D], lse [Q, Hq]); raises on the
    gather's error bits (no result is defined then)."""
    _, attend = _quant(fmt)
    ko, vo, err = gather_paged(_u8(key_rows), _u8(value_rows), block_tables, seq_lens, seq_offset)
    if err:
        raise ValueError(f"oracle.attend_paged_quant: invalid paged inputs (error bits {err})")
    qa, _ = _storage(q)
    Q, Hq, D = qa.shape
    sl = _i32(seq_lens)
    out = np.zeros((Q, Hq, D), np.float64)
    lse = np.full((Q, Hq), -np.inf)
    for s in range(Q):
        a, b = int(sl[s]), int(sl[s + 1])
        if b <= a:
            continue
        kr = np.ascontiguousarray(ko[a:b].transpose(1, 0, 2)[None])  # [1, Hkv, n, RB]
        vr = np.ascontiguousarray(vo[a:b].transpose(1, 0, 2)[None])
        o, l = attend(q[s:s + 1], kr, vr, np.ones((1, b - a), np.uint8), scale, nthreads)
        out[s], lse[s] = o[0], l[0]
    return out, lse


def attend_indexed_quant(q, k_rows, v_rows, indices, scale: float, fmt: str, nthreads: int = 0):
    """Index-list decode attention over quantised rows, fp64: entry j of
    batch entry b with 0 <= indices[b, j] < C contributes row indices[b, j]
    of k_rows, v_rows uint8 [B, Hkv, C, RB] as one softmax term.  Written as
    the copy of every entry's row into a [B, Hkv, topk, RB] buffer whose mask
    marks the valid entries, then ``attend_masked_fp8`` / ``_fp4`` over it.
    Returns (out, lse, error bits: 1 when an entry is outside [-1, C))."""
    _, attend = _quant(fmt)
    ka = np.ascontiguousarray(_u8(k_rows))
    va = np.ascontiguousarray(_u8(v_rows))
    B, Hkv, C, RB = ka.shape
    idx = _i32(indices).reshape(B, -1)
    topk = idx.shape[1]
    err = ERR_POS if np.any((idx < -1) | (idx >= C)) else 0
    valid = (idx >= 0) & (idx < C)
    safe = np.where(valid, idx, 0)
    kg = np.ascontiguousarray(ka[np.arange(B)[:, None, None], np.arange(Hkv)[None, :, None],
                                 safe[:, None, :]])
    vg = np.ascontiguousarray(va[np.arange(B)[:, None, None], np.arange(Hkv)[None, :, None],
                                 safe[:, None, :]])
    out, lse = attend(q, kg, vg, valid.astype(np.uint8), scale, nthreads)
    return out, lse, err
