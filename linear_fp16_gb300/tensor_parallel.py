"""Tensor-parallel y = FP16(x . W^T) + b over torch.distributed ranks.

"The Graph IR", Primitive operations, the AllReduce / AllGather row
(tensor-parallel collectives; AllGather multiplies the gather axis by the
number of ranks), and "Model and Distributed IR", section "Boundary between
the layers": a linear(x, w) under a tensor-parallel strategy becomes
rank-local matmul tasks, a collective, and a reconstructed result equal to
the one-device result.

* Column split (over the output features N): rank r holds rows
  [begin_r, end_r) of W and of b and computes those columns of y with the
  one-GPU kernel; an all-gather brings every rank's columns together and
  ``poot_linear_gather_columns`` assembles y.  Every column is computed
  exactly as on one GPU, so y is bit-identical to the one-GPU call.
* Row split (over the reduction axis K): rank r holds columns
  [begin_r, end_r) of x and of W and computes the unrounded FP32 partial
  sums S_r (``contract`` with ``out_f32``, no bias); an all-reduce adds them
  in FP32, which is one legal summation order under rule 1 of the contract
  ("Tensor Programs, Part 1", section "One Program and One Numerical
  Contract"), and ``poot_linear_f16_finish`` rounds once:
  y = RN16(RN16(S) + b).  Rounding, or adding b, per rank before the
  reduction would break rule 2.

Shard ranges come from the library's plan (``shard_range``).  The
collectives are torch.distributed's: on an NCCL group the device buffers go
to the collective directly; on a gloo group they are staged through host
memory.  Every arithmetic step runs in the CUDA library.
"""
from __future__ import annotations

from . import binding


def shard_range(extent: int, world: int, rank: int):
    """[begin, end) of `rank`'s shard of an axis of `extent` elements."""
    rc, b, e = binding.poot_linear_tp_shard(extent, world, rank)
    if rc != binding.POOT_OK:
        raise binding.PootLinearError(rc, "poot_linear_tp_shard")
    return b, e


def _group_info(group):
    import torch.distributed as dist
    return dist.get_rank(group), dist.get_world_size(group), dist.get_backend(group)


def all_gather_slots(local, group=None):
    """Every rank's `local` (1-D, the same length on every rank) concatenated
    in rank order, on local's device."""
    import torch
    import torch.distributed as dist
    rank, world, backend = _group_info(group)
    if local.is_cuda and backend != "nccl":
        host = local.cpu()
        parts = [torch.empty_like(host) for _ in range(world)]
        dist.all_gather(parts, host, group=group)
        return torch.cat(parts).to(local.device)
    parts = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(parts, local, group=group)
    return torch.cat(parts)


def all_reduce_sum(S, group=None):
    """S summed over the ranks in place (FP32 adds; the collective's order)."""
    import torch.distributed as dist
    rank, world, backend = _group_info(group)
    if S.is_cuda and backend != "nccl":
        host = S.cpu()
        dist.all_reduce(host, op=dist.ReduceOp.SUM, group=group)
        S.copy_(host)
    else:
        dist.all_reduce(S, op=dist.ReduceOp.SUM, group=group)
    return S


def _stream_of(t):
    import torch
    return torch.cuda.current_stream(t.device).cuda_stream


def column_parallel_linear(x, w_shard, b_shard, N: int, group=None):
    """y [M, N] on every rank from x [M, K] (the same on every rank), this
    rank's W rows w_shard [N_r, K] and bias b_shard [N_r] (fp16 CUDA
    tensors), N_r = end - begin of ``shard_range(N, world, rank)``."""
    import torch
    rank, world, _ = _group_info(group)
    begin, end = shard_range(N, world, rank)
    nr = end - begin
    M, K = x.shape
    if tuple(w_shard.shape) != (nr, K) or tuple(b_shard.shape) != (nr,):
        raise ValueError(f"rank {rank} owns output features [{begin}, {end}): w_shard must be [{nr}, {K}] and "
                         f"b_shard [{nr}], got {tuple(w_shard.shape)} and {tuple(b_shard.shape)}")
    b0, e0 = shard_range(N, world, 0)
    slot = M * (e0 - b0)  # every slot holds the widest shard (rank 0's)
    local = torch.empty(max(slot, 1), dtype=torch.float16, device=x.device)
    if nr > 0 and M > 0:
        binding.linear(x, w_shard, b_shard, out=local[:M * nr].view(M, nr))
    gathered = all_gather_slots(local, group)
    y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    with torch.cuda.device(x.device):
        rc = binding.poot_linear_gather_columns(gathered.data_ptr(), y.data_ptr(), M, N, world, local.numel(),
                                                _stream_of(x))
    if rc != binding.POOT_OK:
        raise binding.PootLinearError(rc, "poot_linear_gather_columns")
    return y


def row_parallel_linear(x_shard, w_shard, b, K: int, group=None):
    """y [M, N] on every rank from this rank's columns of x, x_shard [M, K_r],
    and of W, w_shard [N, K_r], and the full bias b [N] (fp16 CUDA tensors),
    K_r = end - begin of ``shard_range(K, world, rank)``."""
    import torch
    rank, world, _ = _group_info(group)
    begin, end = shard_range(K, world, rank)
    kr = end - begin
    M = x_shard.shape[0]
    N = w_shard.shape[0]
    if tuple(x_shard.shape) != (M, kr) or tuple(w_shard.shape) != (N, kr) or tuple(b.shape) != (N,):
        raise ValueError(f"rank {rank} owns reduction columns [{begin}, {end}): x_shard must be [M, {kr}], "
                         f"w_shard [N, {kr}] and b [N], got {tuple(x_shard.shape)}, {tuple(w_shard.shape)}, "
                         f"{tuple(b.shape)}")
    S = torch.empty((M, N), dtype=torch.float32, device=x_shard.device)
    if kr > 0 and M > 0 and N > 0:
        binding.contract(x_shard, w_shard, None, out=S, out_f32=True)
    else:
        S.zero_()  # an empty shard adds +0
    all_reduce_sum(S, group)
    y = torch.empty((M, N), dtype=torch.float16, device=x_shard.device)
    with torch.cuda.device(x_shard.device):
        rc = binding.poot_linear_f16_finish(S.data_ptr(), b.data_ptr(), y.data_ptr(), M, N, _stream_of(x_shard))
    if rc != binding.POOT_OK:
        raise binding.PootLinearError(rc, "poot_linear_f16_finish")
    return y
