"""Sequence-axis split of one decode step across ranks (one GPU per rank).

A single sequence too long for one GPU's share of the work is cut along its
token axis: rank r keeps slots [start_r, stop_r) of every (batch entry, kv
head) row of the static buffer, as its own cache [B, Hkv, C_r, D] and mask
[B, C_r].  One decode step is then

1. on every rank, the step's query against its own slots
   (``kvd_attend_masked_partial``): fp32 output rows normalised over the
   range and their log-sum-exp, written into one packed block of
   R * (D + 1) floats (R = B * Hq rows of D, then the R log-sum-exps);
2. one all-gather of the blocks -- the only exchange step of the path;
3. on every rank, the exact log-sum-exp merge of the gathered blocks
   (``kvd_combine_gathered``).

The merge is the one the tiles of the Flash SDPA path go through ("Intel NPU
running LLMs", Part 3 "Attention 在 NPU 上的完整实现": each tile's output is
normalised over its own keys and carried with its running max and sum, and
the tiles are merged exactly), applied to ranges held by different GPUs.  A
range with no valid slot contributes lse = -inf, i.e. weight 0.

The exchange works on any ``torch.distributed`` process group: NCCL for GPU
tensors, gloo for host tensors (the tests exercise the exchange with gloo
ranks on the CPU).  Nothing here computes attention: step 1 and step 3 run in
libkvd's kernels, step 2 in the collective library.
"""
from __future__ import annotations

import torch


def token_ranges(C: int, world: int, align: int = 64):
    """Contiguous token ranges [(start, stop), ...] covering [0, C), one per
    rank, as equal as ``align``-slot granules allow (the last range takes the
    remainder; a rank may get an empty range when C is small)."""
    if C < 0 or world < 1 or align < 1:
        raise ValueError("token_ranges: C >= 0, world >= 1, align >= 1 required")
    granules = (C + align - 1) // align
    bounds = [min(C, (granules * r // world) * align) for r in range(world)] + [C]
    return [(bounds[r], bounds[r + 1]) for r in range(world)]


def block_floats(R: int, D: int) -> int:
    """Floats in one rank's packed partial: R rows of D, then R lse."""
    return R * (D + 1)


def block_views(block: torch.Tensor, R: int, D: int):
    """The two parts of a packed block: rows [R, D] and lse [R] (views)."""
    if block.dim() != 1 or block.numel() != block_floats(R, D):
        raise ValueError("block_views: a flat block of R * (D + 1) floats required")
    return block[: R * D].view(R, D), block[R * D:]


def exchange(block: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of every rank's packed block: returns [world, numel], rank
    s's block in row s.  Without an initialised process group (one rank) the
    block itself is the gathered result."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return block.view(1, -1)
    world = dist.get_world_size(group)
    gathered = torch.empty((world, block.numel()), dtype=block.dtype, device=block.device)
    dist.all_gather(list(gathered.unbind(0)), block.contiguous(), group=group)
    return gathered


class SequenceSplitAttention:
    """One rank's side of the sequence-split decode attention.

    Holds the rank's packed partial block (and nothing else); call it with
    the step's query and the rank's slice of the cache and mask.
    """

    def __init__(self, B: int, Hq: int, D: int, device=None, group=None):
        self.B, self.Hq, self.D = B, Hq, D
        self.R = B * Hq
        self.group = group
        self.block = torch.empty(block_floats(self.R, D), dtype=torch.float32,
                                 device=device or "cuda")

    def __call__(self, q, k_slice, v_slice, mask_slice, scale=None, out=None, lse=None,
                 num_splits=0, workspace=None, dev_status=None):
        """out [B, Hq, D] (dtype of q unless given) for the whole sequence;
        fills ``lse`` [B, Hq] fp32 if given."""
        from . import kvd
        B, Hq, D = q.shape
        if (B, Hq, D) != (self.B, self.Hq, self.D):
            raise ValueError("SequenceSplitAttention: q shape differs from the one set up")
        rows, lse_part = block_views(self.block, self.R, D)
        kvd.attend_masked_partial(q, k_slice, v_slice, mask_slice, scale,
                                  out=rows.view(B, Hq, D), lse=lse_part.view(B, Hq),
                                  num_splits=num_splits, workspace=workspace,
                                  dev_status=dev_status)
        gathered = exchange(self.block, self.group)
        if out is None:
            out = torch.empty_like(q)
        kvd.combine_gathered(gathered, self.R, D, out=out.view(self.R, D),
                             lse=None if lse is None else lse.view(self.R))
        return out
