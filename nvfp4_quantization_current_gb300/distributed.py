"""Sharded quantization: the one exchange the quantizers need.

Per-tensor current scaling and NVFP4 use one amax for the whole tensor.
When the tensor is split across ranks (data-parallel master-weight shards,
tensor-parallel sequence shards), every rank computes the amax of its own
shard, the ranks agree on the global amax with a MAX all-reduce of one float,
and each rank then quantizes its shard with that amax, so that the codes do
not depend on the split ("FP8 Current Scaling ...", section "Cost and
multi-GPU use": compute amax, synchronize amax, scale + cast, all-gather;
"Mixed-precision training: fp16 to fp8", section "FP8 communication", TP:
the FP8 tensor must be identical with or without TP).

The block-scaled recipes (MXFP8, blockwise, NVFP4 block scales) need no
exchange when shards split rows on block boundaries.  Delayed scaling
all-reduces the step's recorded amax into every rank's window slot
(``DelayedScaling.quantize(group=...)``), so the windows, and the scales
they give, stay identical.  The random-Hadamard NVFP4 copy of the
weight-gradient inputs all-reduces the amax of the transformed shard; shards
that split rows on 16-row boundaries transform exactly like the slices of
the whole tensor.

Stochastic rounding draws depend only on an element's position in the
whole tensor: element (m, k) takes its random bits from Philox block
offset + (m*K + k)/16 (rowwise) or offset + (m/16)*K + k (columnwise), so a
rank whose shard starts at global row r0 (a multiple of 16) passes
offset + r0*K/16 and draws exactly what the unsharded call draws for those
rows.  The ``quantize_shard_*``
helpers do this by default (``row_base=None`` gathers the shard heights and
takes the rank's first global row).

After the local quantize, the shards' outputs may be all-gathered into the
whole tensor's layout (the FP8 all-gather of the TP path): rowwise codes and
scales concatenate by rows, the transposed copies by columns
(``all_gather_quantized``).

``allreduce_amax_`` and the gathers work on any torch.distributed backend
(NCCL for CUDA tensors, gloo for CPU tensors); the ``quantize_shard_*``
helpers run the library's CUDA kernels around them.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch
import torch.distributed as dist


def allreduce_amax_(amax: torch.Tensor, group=None) -> torch.Tensor:
    """In-place MAX all-reduce of a one-element FP32 amax.  A no-op when
    torch.distributed is not initialized (a single rank)."""
    if amax.numel() != 1 or amax.dtype != torch.float32:
        raise ValueError("amax must be a one-element float32 tensor")
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    return amax


def shard_row_base(rows_local: int, group=None, device=None) -> int:
    """The global index of this rank's first row when the ranks hold
    consecutive row shards in rank order (an exclusive prefix sum of the
    shard heights, from one all-gather of an int64).  0 on a single rank."""
    if not (dist.is_available() and dist.is_initialized()):
        return 0
    world = dist.get_world_size(group)
    n = torch.tensor([int(rows_local)], dtype=torch.int64, device=device)
    sizes = [torch.empty_like(n) for _ in range(world)]
    dist.all_gather(sizes, n, group=group)
    rank = dist.get_rank(group)
    return int(sum(int(v.item()) for v in sizes[:rank]))


def sr_offset(offset: int, row_base: int, K: int) -> int:
    """The Philox counter offset for a row shard that starts at global row
    ``row_base`` (a multiple of 16): the unsharded call's ``offset`` moved by
    the row_base * K elements ahead of the shard (16 draws per counter)."""
    if row_base % 16 != 0 or K % 16 != 0:
        raise ValueError("row_base and K must be multiples of 16")
    return int(offset) + int(row_base) * int(K) // 16


def _shard_offset(x_local, offset, row_base, group):
    if row_base is None:
        row_base = shard_row_base(x_local.shape[0], group, x_local.device if x_local.is_cuda else None)
    return sr_offset(offset, row_base, x_local.shape[1])


def quantize_shard_current_scaling(x_local: torch.Tensor, fmt="e4m3", rowwise=True, colwise=False, group=None,
                                   status: Optional[torch.Tensor] = None):
    """Current scaling of this rank's row shard with the amax of the whole
    (distributed) tensor."""
    from . import q_amax, q_current_scaling
    a = q_amax(x_local, status=status)
    allreduce_amax_(a, group)
    return q_current_scaling(x_local, fmt, rowwise, colwise, amax=a, status=status)


def quantize_shard_nvfp4_rht_colT(x_local: torch.Tensor, sign_mask: int, rounding="rn", seed=0, offset=0, group=None,
                                  status: Optional[torch.Tensor] = None, row_base: Optional[int] = None):
    """The random-Hadamard NVFP4 columnwise copy of this rank's row shard
    (rows split on 16-row boundaries) with the amax of the whole transformed
    tensor.  ``offset`` is the unsharded call's counter offset; the shard's
    own is derived from ``row_base`` (this rank's first global row, gathered
    when None), so stochastic draws match the unsharded copy."""
    from . import q_nvfp4_rht_amax, q_nvfp4_rht_colT
    off = _shard_offset(x_local, offset, row_base, group)
    a = q_nvfp4_rht_amax(x_local, sign_mask, status=status)
    allreduce_amax_(a, group)
    return q_nvfp4_rht_colT(x_local, sign_mask, rounding, seed, off, amax=a, status=status)


def quantize_shard_nvfp4(x_local: torch.Tensor, blk="1x16", rounding="rn", seed=0, offset=0, rowwise=True,
                         colwise=False, group=None, status: Optional[torch.Tensor] = None,
                         row_base: Optional[int] = None):
    """NVFP4 of this rank's row shard with the global amax (so the FP32 tensor
    scale, and therefore every block scale, matches the unsharded tensor).
    ``offset`` is the unsharded call's counter offset; the shard's own is
    derived from ``row_base`` (this rank's first global row, gathered when
    None), so stochastic draws match the unsharded quantization."""
    from . import q_amax, q_nvfp4
    off = _shard_offset(x_local, offset, row_base, group)
    a = q_amax(x_local, status=status)
    allreduce_amax_(a, group)
    return q_nvfp4(x_local, blk, rounding, seed, off, rowwise, colwise, amax=a, status=status)


def quantize_shard_nvfp4_recipe(x_local: torch.Tensor, sign_mask: int, rounding="rn", seed=0, offset=0, group=None,
                                status: Optional[torch.Tensor] = None, row_base: Optional[int] = None):
    """Both NVFP4 recipe copies of this rank's row shard (rows split on 16-row
    boundaries): one read for the two local maxima, a MAX all-reduce of each,
    then the rowwise copy of x and the columnwise copy of its transform with
    the global maxima, both with the shard's counter offset (see
    quantize_shard_nvfp4).  Returns (row, colT) like q_nvfp4_recipe."""
    from . import q_nvfp4_recipe, q_nvfp4_rht_amax2
    off = _shard_offset(x_local, offset, row_base, group)
    a_rht, a_x = q_nvfp4_rht_amax2(x_local, sign_mask, status=status)
    allreduce_amax_(a_rht, group)
    allreduce_amax_(a_x, group)
    return q_nvfp4_recipe(x_local, sign_mask, rounding, seed, off, amax_row=a_x, amax_col=a_rht, status=status)


def all_gather_shards(t_local: torch.Tensor, dim: int = 0, group=None) -> torch.Tensor:
    """The concatenation along ``dim``, in rank order, of every rank's
    ``t_local``.  Shards may differ in size along ``dim`` (they are padded to
    the largest for the collective and trimmed after); every other dimension
    must agree.  Returns ``t_local`` itself when torch.distributed is not
    initialized."""
    if not (dist.is_available() and dist.is_initialized()):
        return t_local
    world = dist.get_world_size(group)
    n = torch.tensor([t_local.shape[dim]], dtype=torch.int64, device=t_local.device)
    sizes = [torch.empty_like(n) for _ in range(world)]
    dist.all_gather(sizes, n, group=group)
    sizes = [int(v.item()) for v in sizes]
    x = t_local.movedim(dim, 0).contiguous()
    if x.shape[0] < max(sizes):
        x = torch.cat([x, x.new_zeros((max(sizes) - x.shape[0],) + tuple(x.shape[1:]))])
    parts = [torch.empty_like(x) for _ in range(world)]
    dist.all_gather(parts, x, group=group)
    return torch.cat([p[:k] for p, k in zip(parts, sizes)]).movedim(0, dim).contiguous()


# Fields of the quantized-tensor classes that follow the rows of the input
# (rowwise codes and scales, and the MXFP8 columnwise copy, which keeps the
# input's [M, K] layout) and those of the transposed copies ([K, M] layouts).
_ROW_FIELDS = ("q_row", "sb_row", "e8m0_row", "s_row", "q_col", "e8m0_col")
_COLT_FIELDS = ("q_colT", "sb_colT", "s_colT", "e8m0_colT")


def all_gather_quantized(t, group=None):
    """The whole tensor's quantized outputs from every rank's row-shard
    outputs ``t`` (a CurrentScalingTensor, MXFP8Tensor, BlockwiseTensor,
    BlockwiseMXTensor or NVFP4Tensor): rowwise fields gathered by rows, transposed copies by
    columns.  Shards must split rows on the recipe's block boundaries (32 for
    MXFP8 columnwise, 16 for NVFP4, 128 for the blockwise columnwise and 2-D
    tiles), for current scaling and NVFP4 share the all-reduced amax, and for
    stochastic rounding use the counter offset of their first global row
    (``sr_offset``; the ``quantize_shard_*`` helpers do both), so that the
    result equals the unsharded quantization.  Tensor-wide fields
    (amax, scale, s_global) are the same on every rank and are kept."""
    upd = {}
    for f in dataclasses.fields(t):
        v = getattr(t, f.name)
        if v is None:
            continue
        if f.name in _ROW_FIELDS:
            upd[f.name] = all_gather_shards(v, 0, group)
        elif f.name in _COLT_FIELDS:
            upd[f.name] = all_gather_shards(v, 1, group)
    return dataclasses.replace(t, **upd)
