"""Seeded synthetic inputs for decode-phase KV-cache attention.

The one module that both the fp64 oracle and the CUDA path are fed from.  It
holds random draws and layout construction only (shapes, prefix masks, block
tables, length mixes); none of the method's arithmetic.

Workloads (shapes and value distributions follow the pages' own examples):

* ``tiny``      -- batch 1, 4 heads (MHA), head_dim 64, fp32, capacity 32;
                   a 4-token prompt, then 3 decode steps appending at slots
                   4, 5, 6; padding slots hold uniform +-1e3 garbage; scale
                   1/sqrt(64).  (Mask evolution of "Intel NPU running LLMs",
                   Part 1, shrunk to 32 slots.)
* ``npuw``      -- batch 1, 32 heads (MHA), head_dim 128, bf16, capacity
                   1152 = 1024 + 128 (MAX_PROMPT_LEN + MIN_RESPONSE_LEN,
                   same article, Part 1), 32 layer caches; rows 0..1023
                   N(0,1), the rest zero; decode step i appends at 1024 + i
                   and attends over 1025 + i slots.
* ``gqa``       -- batch 16, 32 query heads / 8 kv heads, head_dim 128, bf16,
                   capacity 8192, valid length per sequence uniform in
                   [512, 8192]; q, k, v ~ N(0,1) with k scaled by 0.5; 32
                   layer caches; one step appends at L_b - 1 and attends
                   over L_b slots.
* ``paged``     -- key/value caches [8192, 128, 8, 128] bf16 N(0,1),
                   block_tables [64, 32] = the first 2048 entries of a random
                   permutation of the 8192 physical blocks, 64 lengths uniform
                   in [1, 4096], seq_lens = their cumsum with a leading 0,
                   seq_offset zeros, 32 query heads; the decode step's new
                   K/V rows N(0,1), appended at each sequence's last token.
                   (Tensor contract of "PyPTO 实现 AscendC GatherPaKvCache",
                   section 3.1.)
* ``long``      -- batch 1, 32 heads (MHA), head_dim 128, bf16, capacity =
                   valid length = 32768, 8 layer caches, N(0,1); one step
                   appends at 32767 and attends over all slots.

Large tensors are drawn on the device passed in (torch's generator for that
device, seeded per workload); tests take host copies of what they compare.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SEEDS = {"tiny": 1, "npuw": 2, "gqa": 3, "paged": 4, "long": 5, "window": 6, "gqa_fp8": 7,
         "gqa_fp4": 8, "paged_fp8": 9, "paged_fp4": 10}


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def randn(g, shape, dtype=torch.bfloat16, device="cpu", scale: float = 1.0):
    """N(0, scale^2) draws in ``dtype`` (drawn in fp32, then rounded)."""
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(dtype)


def uniform(g, shape, lo: float, hi: float, dtype=torch.float32, device="cpu"):
    x = torch.rand(tuple(shape), generator=g, device=device, dtype=torch.float32)
    return (x * (hi - lo) + lo).to(dtype)


def randint(g, n: int, lo: int, hi: int, device="cpu"):
    """n integers uniform in [lo, hi] (both ends included), int64."""
    return torch.randint(lo, hi + 1, (n,), generator=g, device=device, dtype=torch.int64)


FP8_ROW_PAD = 16  # quantised rows: D E4M3 codes, fp32 scale, 12 zero bytes


def fp8_rows(g, shape, D: int, scale_lo: float = 2e-3, scale_hi: float = 2e-2, device="cpu"):
    """uint8 [*shape, D + 16]: quantised K/V rows with random content -- codes
    uniform over the 254 finite E4M3 codes (0x7F and 0xFF are NaN), a scale
    uniform in [scale_lo, scale_hi] as fp32 little-endian bytes, 12 zero
    bytes.  Random bytes, not the result of quantising anything."""
    shape = tuple(shape)
    r = torch.randint(0, 254, shape + (D,), generator=g, device=device, dtype=torch.int32)
    codes = (r + (r >= 0x7F).to(torch.int32)).to(torch.uint8)
    scale = uniform(g, shape + (1,), scale_lo, scale_hi, torch.float32, device)
    out = torch.zeros(shape + (D + FP8_ROW_PAD,), dtype=torch.uint8, device=device)
    out[..., :D] = codes
    out[..., D:D + 4] = scale.contiguous().view(torch.uint8)
    return out


FP4_ROW_PAD = 16  # FP4 rows: D/2 bytes of E2M1 codes, fp32 scale, 12 zero bytes


def fp4_rows(g, shape, D: int, scale_lo: float = 0.1, scale_hi: float = 0.4, device="cpu"):
    """uint8 [*shape, D/2 + 16]: FP4 K/V rows with random content -- code
    bytes uniform over 0..255 (every nibble is a finite E2M1 code), a scale
    uniform in [scale_lo, scale_hi] as fp32 little-endian bytes, 12 zero
    bytes.  Random bytes, not the result of quantising anything."""
    shape = tuple(shape)
    codes = torch.randint(0, 256, shape + (D // 2,), generator=g, device=device,
                          dtype=torch.int32).to(torch.uint8)
    scale = uniform(g, shape + (1,), scale_lo, scale_hi, torch.float32, device)
    out = torch.zeros(shape + (D // 2 + FP4_ROW_PAD,), dtype=torch.uint8, device=device)
    out[..., :D // 2] = codes
    out[..., D // 2:D // 2 + 4] = scale.contiguous().view(torch.uint8)
    return out


def prefix_mask(lengths, capacity: int, device="cpu"):
    """uint8 [B, capacity] with the first lengths[b] slots set to 1."""
    lengths = torch.as_tensor(lengths, dtype=torch.int64, device=device)
    ar = torch.arange(capacity, device=device).unsqueeze(0)
    return (ar < lengths.unsqueeze(1)).to(torch.uint8)


def window_mask(lengths, capacity: int, window: int, device="cpu"):
    """uint8 [B, capacity]: 1 on the last ``window`` slots of each valid
    prefix, [max(0, lengths[b] - window), lengths[b])."""
    lengths = torch.as_tensor(lengths, dtype=torch.int64, device=device)
    ar = torch.arange(capacity, device=device).unsqueeze(0)
    end = lengths.unsqueeze(1)
    return ((ar < end) & (ar >= end - window)).to(torch.uint8)


def index_lists(lengths, topk: int, seed: int = 7):
    """int32 [B, topk]: per entry, min(topk, L) unique slots drawn from its
    valid prefix [0, L) in random order (seeded), -1 after them."""
    g = generator(seed, "cpu")
    rows = []
    for L in lengths:
        L = int(L)
        n = min(topk, L)
        r = torch.full((topk,), -1, dtype=torch.int32)
        r[:n] = torch.randperm(L, generator=g)[:n].to(torch.int32)
        rows.append(r)
    return torch.stack(rows)


def cumsum_lengths(lengths):
    """[Q + 1] int32: 0 followed by the running totals of ``lengths``."""
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    out = torch.zeros(lengths.numel() + 1, dtype=torch.int64, device=lengths.device)
    out[1:] = torch.cumsum(lengths, 0)
    return out.to(torch.int32)


def permuted_block_tables(g, Q: int, cols: int, num_blocks: int, device="cpu"):
    """First Q*cols entries of a random permutation of the physical blocks."""
    perm = torch.randperm(num_blocks, generator=g, device=device)
    return perm[: Q * cols].reshape(Q, cols).to(torch.int32).contiguous()


# ---------------------------------------------------------------- workloads

@dataclass
class MaskedLayer:
    """One layer's static-buffer cache plus the inputs of one decode step."""
    q: torch.Tensor          # [B, Hq, D]
    k_cache: torch.Tensor    # [B, Hkv, C, D]
    v_cache: torch.Tensor    # [B, Hkv, C, D]
    mask: torch.Tensor       # [B, C] uint8, valid slots *before* the append
    k_new: torch.Tensor      # [B, Hkv, D]
    v_new: torch.Tensor      # [B, Hkv, D]
    pos: torch.Tensor        # [B] int32, append position (= valid length - 1)
    lengths: torch.Tensor    # [B] int64, valid length after the append
    scale: float


@dataclass
class MaskedWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    C: int
    D: int
    dtype: torch.dtype
    layers: list = field(default_factory=list)
    window: int = 0  # > 0: each row attends to its last `window` slots only


def masked_layer(g, B, Hq, Hkv, C, D, lengths, dtype=torch.bfloat16, device="cpu",
                 k_scale: float = 1.0, pad: str = "random", pad_garbage: float = 1e3,
                 scale: float | None = None) -> MaskedLayer:
    """A static-buffer layer whose sequences hold lengths[b] - 1 rows before
    the step and ``lengths[b]`` after appending the step's row at
    lengths[b] - 1.

    pad: "random" (padding holds N(0,1) draws), "zero" (zero-filled) or
    "garbage" (uniform +-pad_garbage).  The mask marks the rows present
    before the append; the append sets the new slot.
    """
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    k = randn(g, (B, Hkv, C, D), dtype, device, k_scale)
    v = randn(g, (B, Hkv, C, D), dtype, device)
    before = prefix_mask((lengths - 1).clamp(min=0), C, device)
    if pad != "random":
        pm = (before == 0).view(B, 1, C, 1)
        if pad == "zero":
            k.masked_fill_(pm, 0)
            v.masked_fill_(pm, 0)
        elif pad == "garbage":
            k = torch.where(pm, uniform(g, k.shape, -pad_garbage, pad_garbage, dtype, device), k)
            v = torch.where(pm, uniform(g, v.shape, -pad_garbage, pad_garbage, dtype, device), v)
        else:
            raise ValueError(pad)
    q = randn(g, (B, Hq, D), dtype, device)
    k_new = randn(g, (B, Hkv, D), dtype, device, k_scale)
    v_new = randn(g, (B, Hkv, D), dtype, device)
    pos = (lengths - 1).to(torch.int32).to(device)
    return MaskedLayer(q=q, k_cache=k, v_cache=v, mask=before, k_new=k_new, v_new=v_new,
                       pos=pos, lengths=lengths, scale=scale if scale is not None
                       else 1.0 / math.sqrt(D))


def tiny(device="cpu", seed: int | None = None):
    """The 4-token prompt + 3 decode steps case (fp32, capacity 32).

    Returns (k_cache, v_cache, mask, steps) where k_cache/v_cache [1,4,32,64]
    hold the prompt in slots 0..3 and +-1e3 garbage elsewhere, mask marks the
    4 prompt slots, and each step is a dict with q, k_new, v_new, pos (4, 5,
    6) and the valid length after its append (5, 6, 7).
    """
    g = generator(SEEDS["tiny"] if seed is None else seed, device)
    B, H, C, D = 1, 4, 32, 64
    k = uniform(g, (B, H, C, D), -1e3, 1e3, torch.float32, device)
    v = uniform(g, (B, H, C, D), -1e3, 1e3, torch.float32, device)
    k[:, :, :4] = randn(g, (B, H, 4, D), torch.float32, device)
    v[:, :, :4] = randn(g, (B, H, 4, D), torch.float32, device)
    mask = prefix_mask([4], C, device)
    steps = []
    for i in range(3):
        steps.append(dict(q=randn(g, (B, H, D), torch.float32, device),
                          k_new=randn(g, (B, H, D), torch.float32, device),
                          v_new=randn(g, (B, H, D), torch.float32, device),
                          pos=torch.tensor([4 + i], dtype=torch.int32, device=device),
                          length=5 + i))
    return k, v, mask, steps, 1.0 / math.sqrt(D)


def npuw(device="cpu", layers: int = 32, seed: int | None = None, prompt: int = 1024,
         response: int = 128, B: int = 1, H: int = 32, D: int = 128) -> MaskedWorkload:
    """Static buffer of capacity prompt + response; layer caches hold the
    prompt's rows and zero padding; step 0's append goes to slot ``prompt``."""
    g = generator(SEEDS["npuw"] if seed is None else seed, device)
    C = prompt + response
    w = MaskedWorkload("npuw", B, H, H, C, D, torch.bfloat16)
    lengths = torch.full((B,), prompt + 1, dtype=torch.int64)
    for _ in range(layers):
        w.layers.append(masked_layer(g, B, H, H, C, D, lengths, torch.bfloat16, device,
                                     pad="zero"))
    return w


def gqa(device="cpu", layers: int = 32, seed: int | None = None, B: int = 16,
        Hq: int = 32, Hkv: int = 8, C: int = 8192, D: int = 128, lo: int = 512,
        hi: int = 8192) -> MaskedWorkload:
    """Batched GQA decode: per-sequence lengths uniform in [lo, hi] (drawn once
    on the CPU so that every device sees the same mix), k scaled by 0.5."""
    gl = generator(SEEDS["gqa"] if seed is None else seed, "cpu")
    lengths = randint(gl, B, lo, hi)
    g = generator((SEEDS["gqa"] if seed is None else seed) + 1000, device)
    w = MaskedWorkload("gqa", B, Hq, Hkv, C, D, torch.bfloat16)
    for _ in range(layers):
        w.layers.append(masked_layer(g, B, Hq, Hkv, C, D, lengths, torch.bfloat16, device,
                                     k_scale=0.5))
    return w


def fp8_layer(g, B, Hq, Hkv, C, D, lengths, device="cpu", rows=None) -> MaskedLayer:
    """A static-buffer layer with quantised K/V caches (random rows, see
    fp8_rows; fp4_rows with rows=fp4_rows) holding lengths[b] - 1 rows
    before the step; q and the step's new rows in bf16."""
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    rows = rows or fp8_rows
    k = rows(g, (B, Hkv, C), D, device=device)
    v = rows(g, (B, Hkv, C), D, device=device)
    q = randn(g, (B, Hq, D), torch.bfloat16, device)
    k_new = randn(g, (B, Hkv, D), torch.bfloat16, device, 0.5)
    v_new = randn(g, (B, Hkv, D), torch.bfloat16, device)
    return MaskedLayer(q=q, k_cache=k, v_cache=v,
                       mask=prefix_mask((lengths - 1).clamp(min=0), C, device), k_new=k_new,
                       v_new=v_new, pos=(lengths - 1).to(torch.int32).to(device), lengths=lengths,
                       scale=1.0 / math.sqrt(D))


def gqa_fp8(device="cpu", layers: int = 32, seed: int | None = None, B: int = 16,
            Hq: int = 32, Hkv: int = 8, C: int = 8192, D: int = 128, lo: int = 512,
            hi: int = 8192) -> MaskedWorkload:
    """Batched GQA decode (the gqa shapes and length mix, drawn the same way)
    over quantised caches: rows of D E4M3 codes + fp32 scale + 12 zero bytes."""
    gl = generator(SEEDS["gqa"] if seed is None else seed, "cpu")
    lengths = randint(gl, B, lo, hi)
    g = generator((SEEDS["gqa_fp8"] if seed is None else seed) + 1000, device)
    w = MaskedWorkload("gqa_fp8", B, Hq, Hkv, C, D, torch.uint8)
    for _ in range(layers):
        w.layers.append(fp8_layer(g, B, Hq, Hkv, C, D, lengths, device))
    return w


def gqa_fp4(device="cpu", layers: int = 32, seed: int | None = None, B: int = 16,
            Hq: int = 32, Hkv: int = 8, C: int = 8192, D: int = 128, lo: int = 512,
            hi: int = 8192) -> MaskedWorkload:
    """Batched GQA decode (the gqa shapes and length mix, drawn the same way)
    over FP4 caches: rows of D/2 bytes of E2M1 codes + fp32 scale + 12 zero
    bytes."""
    gl = generator(SEEDS["gqa"] if seed is None else seed, "cpu")
    lengths = randint(gl, B, lo, hi)
    g = generator((SEEDS["gqa_fp4"] if seed is None else seed) + 1000, device)
    w = MaskedWorkload("gqa_fp4", B, Hq, Hkv, C, D, torch.uint8)
    for _ in range(layers):
        w.layers.append(fp8_layer(g, B, Hq, Hkv, C, D, lengths, device, rows=fp4_rows))
    return w


def window(device="cpu", layers: int = 8, seed: int | None = None, C: int = 32768,
           H: int = 32, D: int = 128, W: int = 4096) -> MaskedWorkload:
    """Sliding-window decode over the long caches: one sequence filling its
    capacity, attending to its last W slots (the W - 1 newest rows before the
    step plus the row the step appends at C - 1)."""
    g = generator(SEEDS["window"] if seed is None else seed, device)
    w = MaskedWorkload("window", 1, H, H, C, D, torch.bfloat16, window=W)
    lengths = torch.full((1,), C, dtype=torch.int64)
    for _ in range(layers):
        lay = masked_layer(g, 1, H, H, C, D, lengths, torch.bfloat16, device)
        lay.mask = window_mask(lengths - 1, C, W - 1, device)
        w.layers.append(lay)
    return w


def long(device="cpu", layers: int = 8, seed: int | None = None, C: int = 32768,
         H: int = 32, D: int = 128) -> MaskedWorkload:
    """One sequence filling its whole capacity; the step appends at C - 1."""
    g = generator(SEEDS["long"] if seed is None else seed, device)
    w = MaskedWorkload("long", 1, H, H, C, D, torch.bfloat16)
    lengths = torch.full((1,), C, dtype=torch.int64)
    for _ in range(layers):
        w.layers.append(masked_layer(g, 1, H, H, C, D, lengths, torch.bfloat16, device))
    return w


@dataclass
class PagedWorkload:
    q: torch.Tensor             # [Q, Hq, D]
    key_cache: torch.Tensor     # [NB, BS, Hkv, D]
    value_cache: torch.Tensor   # [NB, BS, Hkv, D]
    block_tables: torch.Tensor  # [Q, cols] int32
    seq_lens: torch.Tensor      # [Q + 1] int32 cumsum
    seq_offset: torch.Tensor    # [Q] int32
    lengths: torch.Tensor       # [Q] int64
    total_tokens: int
    scale: float
    k_new: torch.Tensor = None  # [Q, Hkv, D]: the step's new rows (appended at pos)
    v_new: torch.Tensor = None
    pos: torch.Tensor = None    # [Q] int32 = lengths - 1: the last token of each sequence


def paged(device="cpu", seed: int | None = None, NB: int = 8192, BS: int = 128,
          Hkv: int = 8, D: int = 128, Q: int = 64, cols: int = 32, Hq: int = 32,
          lo: int = 1, hi: int = 4096, dtype=torch.bfloat16, rows: str | None = None,
          content_seed: int | None = None) -> PagedWorkload:
    """Paged cache addressed through a permuted block table.  Lengths, block
    tables and offsets are drawn on the CPU (small), caches and q on
    ``device``.  rows = "fp8" / "fp4": quantised K/V rows (``fp8_rows`` /
    ``fp4_rows``, uint8 [NB, BS, Hkv, row bytes]) instead of `dtype` rows;
    q and the new rows stay bf16."""
    s = SEEDS["paged"] if seed is None else seed
    gl = generator(s, "cpu")
    lengths = randint(gl, Q, lo, hi)
    bt = permuted_block_tables(gl, Q, cols, NB)
    sl = cumsum_lengths(lengths)
    g = generator((s if content_seed is None else content_seed) + 1000, device)
    if rows is None:
        kc = randn(g, (NB, BS, Hkv, D), dtype, device)
        vc = randn(g, (NB, BS, Hkv, D), dtype, device)
    else:
        make = {"fp8": fp8_rows, "fp4": fp4_rows}[rows]
        kc = make(g, (NB, BS, Hkv), D, device=device)
        vc = make(g, (NB, BS, Hkv), D, device=device)
        dtype = torch.bfloat16
    q = randn(g, (Q, Hq, D), dtype, device)
    k_new = randn(g, (Q, Hkv, D), dtype, device)
    v_new = randn(g, (Q, Hkv, D), dtype, device)
    return PagedWorkload(q=q, key_cache=kc, value_cache=vc, block_tables=bt.to(device),
                         seq_lens=sl.to(device),
                         seq_offset=torch.zeros(Q, dtype=torch.int32, device=device),
                         lengths=lengths, total_tokens=int(sl[-1]),
                         scale=1.0 / math.sqrt(D), k_new=k_new, v_new=v_new,
                         pos=(lengths - 1).to(torch.int32).to(device))


def paged_quant(fmt: str, device="cpu") -> PagedWorkload:
    """The paged workload's sequences, tables and offsets over quantised
    caches (E4M3 rows for "fp8", E2M1 rows for "fp4"; the gqa_fp8 / gqa_fp4
    row contents), bf16 q and new rows."""
    return paged(device=device, rows=fmt, content_seed=SEEDS[f"paged_{fmt}"])
