"""Data parallelism over the batch: one process per GPU, each running the fused
operator on its own contiguous slice of the sequences, then one all-reduce
(sum) of the weight gradients.

The sequences of a batch are independent, and every gradient the operator
returns for them is either per sequence (dx, dh0, dc0: concatenated, no
exchange) or a sum over the sequences (dW, the flat canonical buffer of
W_ih, W_hh, b_ih, b_hh: dW_ih = sum over (t, n) of dG_x^T x, and likewise).
So the whole-batch dW is the sum of the ranks' shard dW, and one all-reduce
of that buffer after backward_weights is the only exchange.  Time, layers and
directions are not sharded.

torch.distributed carries the all-reduce (NCCL between GPUs, gloo on CPU);
the ranks' arithmetic runs in the library's kernels.
"""


def shard_bounds(N, world, rank):
    """Contiguous slice [n0, n1) of N sequences for `rank` of `world`: sizes
    differ by at most one, the first N % world ranks take the extra one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank %r outside a world of %r" % (rank, world))
    base, extra = divmod(int(N), world)
    n0 = rank * base + min(rank, extra)
    return n0, n0 + base + (1 if rank < extra else 0)


def allreduce_grads(dW, dist=None, group=None):
    """Sum dW (a torch tensor: the flat canonical gradient buffer) over the
    ranks of `group`, in place.  With no process group (one process) it is a
    no-op.  bf16 buffers are summed in fp32 and rounded back once, so the
    result does not depend on how the collective splits the sum."""
    if dist is None:
        import torch.distributed as dist  # noqa: F811
    if not dist.is_available() or not dist.is_initialized():
        return dW
    if dist.get_world_size(group) == 1:
        return dW
    import torch
    if dW.dtype == torch.bfloat16:
        acc = dW.float()
        dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
        dW.copy_(acc)
    else:
        dist.all_reduce(dW, op=dist.ReduceOp.SUM, group=group)
    return dW


class DataParallelStep:
    """One training step of the operator on this rank's shard of a batch.

    ``compute(shard) -> dict`` runs forward_training, backward_data and
    backward_weights on the shard (the dict of the rank's inputs, batch
    sliced along dimension 1 of x, dy and the state tensors) and returns the
    shard's outputs, among them the flat ``dW``; the step then all-reduces
    ``dW``.  The per-sequence outputs stay with the rank that owns the
    sequences.
    """

    BATCH_AXIS = {"x": 1, "dy": 1, "h0": 1, "c0": 1, "dhy": 1, "dcy": 1}

    def __init__(self, compute, world, rank, dist=None, group=None):
        self.compute = compute
        self.world = world
        self.rank = rank
        self.dist = dist
        self.group = group

    def shard(self, inputs, N):
        """The rank's slice of a whole-batch input dict (shared tensors such
        as the weights pass through unsliced)."""
        n0, n1 = shard_bounds(N, self.world, self.rank)
        out = {}
        for k, v in inputs.items():
            ax = self.BATCH_AXIS.get(k)
            if v is None or ax is None:
                out[k] = v
            else:
                idx = [slice(None)] * v.ndim
                idx[ax] = slice(n0, n1)
                out[k] = v[tuple(idx)]
        return out, (n0, n1)

    def __call__(self, inputs, N):
        shard, bounds = self.shard(inputs, N)
        out = self.compute(shard)
        out["dW"] = allreduce_grads(out["dW"], self.dist, self.group)
        out["bounds"] = bounds
        return out
