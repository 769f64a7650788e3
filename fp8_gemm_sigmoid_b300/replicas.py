"""Token-parallel replicas of the MoE layer: the host-side glue for N processes, one per GPU.

Every output token depends only on its own input, the weights and the selection bias, so N
replicas of the layer (all weights on every GPU) split a batch's tokens with no exchange of
activations.  The one shared quantity is the selection bias that the top-1 workload updates
from the load it sees: the DeepSeek-V3 co-design teardown (wsisp.com) §2.2 describes the bias
as adjusted from the real-time load of the experts, and under replicas that load is the whole
batch's, so every rank must update from the global per-expert histogram.  One all-reduce of
counts[E] (int32, 1 kB at 256 experts) before the update keeps the ranks' biases identical.

This module holds only process-group plumbing (torch.distributed): the arithmetic of the
update runs in the function it is given (libmoe's moe_bias_update on a GPU).
"""
import torch
import torch.distributed as dist


def token_range(T, world, rank):
    """Contiguous share [start, end) of T tokens for `rank` of `world` (the first T % world
    ranks take one token more)."""
    base, extra = divmod(int(T), int(world))
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def global_counts(counts, T_local, group=None, T_global=None):
    """All-reduce (sum) of this rank's per-expert histogram, in place, and of its token count
    (skipped when the caller already knows T_global, e.g. equal shares: no host sync then).
    counts: int32 tensor on the process group's device (CUDA under NCCL, CPU under gloo).
    Returns the batch's token count over all ranks."""
    if not dist.is_initialized() or dist.get_world_size(group) == 1:
        return int(T_local)
    dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    if T_global is not None:
        return int(T_global)
    t = torch.tensor([int(T_local)], dtype=torch.int64, device=counts.device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return int(t.item())


def global_bias_update(cfg, counts, T_local, bias, update, group=None, T_global=None):
    """The load-driven bias update from the global histogram: all-reduce counts (in place),
    then update(cfg, T_global, counts, bias), which must apply
    bias[i] += 1e-3 * sign(T_global * top_k / E - counts[i]) (libmoe: moe.moe_bias_update).
    Every rank ends with the same bias.  Returns T_global."""
    T_global = global_counts(counts, T_local, group, T_global)
    update(cfg, T_global, counts, bias)
    return T_global
