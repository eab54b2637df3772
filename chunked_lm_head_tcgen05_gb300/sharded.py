"""The head across several GPUs: the exchange steps around the library's calls.

Two ways to split the work, each one process per GPU over a torch.distributed
process group.  Every step of the head's arithmetic runs in the library's
kernels on each rank; this module only moves the per-rank results with
collectives.

Vocabulary-parallel (each rank holds a block of rows of the vocabulary table,
``shard_range``): the forward runs ``lmhead_logps_fwd_shard`` on the local rows,
all-gathers the 16 bytes of statistics per token and combines them
(``lmhead_combine_shards``, the log-sum-exp rule by which the "Long Sequences
(SeCO)" guide, section "Efficiency", merges partial results); the backward runs
``lmhead_logps_bwd_shard`` with the combined lse / entropy and all-reduces
d_hidden.  d_weight stays on the rank that owns the rows.

Token-parallel (each rank scores its own tokens against the whole table, as
the pages' sharded head does: it collects the vocabulary table on every
device once and then works through that device's tokens, tunix PR #2876 on
#2873, so a token's log-prob needs nothing from other devices, tunix PR
#2913): the forward is the single-GPU call, and the backward all-reduces
d_weight.

``ops`` selects the per-rank calls; the default runs the library on the
tensors' GPU.  Collectives run on the default stream of torch.distributed's
backend after the library's work on the current stream.
"""
import torch
import torch.distributed as dist

from . import (LmheadError, lmhead_combine_shards, lmhead_logps_bwd, lmhead_logps_bwd_shard,
               lmhead_logps_fwd, lmhead_logps_fwd_shard)
from .autograd import _workspace


def shard_range(vocab_total, rank, world):
    """(vocab_offset, rows) of rank's block of a vocabulary split into `world`
    contiguous blocks, the first vocab_total % world blocks one row longer."""
    base, extra = divmod(int(vocab_total), int(world))
    v0 = rank * base + min(rank, extra)
    return v0, base + (1 if rank < extra else 0)


class LibraryOps:
    """The per-rank calls, run by the library on the tensors' GPU.  Workspaces
    come from one buffer per (device, stream), reused across calls (the
    autograd wrapper's cache), unless the caller passes its own."""

    @staticmethod
    def _ws(T, H, V, chunk_size, device, workspace):
        if workspace is not None:
            return workspace
        return _workspace(T, H, V, chunk_size, device)

    def shard_forward(self, hidden, weight_shard, targets, loss_mask, vocab_offset, vocab_total,
                      temperature, chunk_size, workspace=None):
        T, H = hidden.shape
        part = torch.empty((T, 4), dtype=torch.float32, device=hidden.device)
        ws = self._ws(T, H, weight_shard.shape[0], chunk_size, hidden.device, workspace)
        rc = lmhead_logps_fwd_shard(hidden, weight_shard, targets, loss_mask, vocab_offset,
                                    vocab_total, temperature, chunk_size, part, ws)
        if rc:
            raise LmheadError(rc, "lmhead_logps_fwd_shard")
        return part

    def combine(self, partials, targets, loss_mask, vocab_total):
        T = partials.shape[1]
        dev = partials.device
        logp, ent, lse = (torch.empty(T, dtype=torch.float32, device=dev) for _ in range(3))
        rc = lmhead_combine_shards(partials, targets, loss_mask, vocab_total, logp, ent, lse)
        if rc:
            raise LmheadError(rc, "lmhead_combine_shards")
        return logp, ent, lse

    def shard_backward(self, hidden, weight_shard, targets, loss_mask, vocab_offset, vocab_total,
                       temperature, chunk_size, grad_logp, grad_entropy, lse, entropy,
                       d_weight_shard, accumulate, workspace=None):
        T, H = hidden.shape
        d_hidden = torch.empty((T, H), dtype=torch.float32, device=hidden.device)
        ws = self._ws(T, H, weight_shard.shape[0], chunk_size, hidden.device, workspace)
        rc = lmhead_logps_bwd_shard(hidden, weight_shard, targets, loss_mask, vocab_offset,
                                    vocab_total, temperature, chunk_size, grad_logp, grad_entropy,
                                    lse, entropy if grad_entropy is not None else None, d_hidden,
                                    d_weight_shard, accumulate, ws)
        if rc:
            raise LmheadError(rc, "lmhead_logps_bwd_shard")
        return d_hidden

    def forward(self, hidden, weight, targets, loss_mask, temperature, chunk_size,
                workspace=None):
        T, H = hidden.shape
        dev = hidden.device
        logp, ent, lse = (torch.empty(T, dtype=torch.float32, device=dev) for _ in range(3))
        ws = self._ws(T, H, weight.shape[0], chunk_size, dev, workspace)
        rc = lmhead_logps_fwd(hidden, weight, targets, loss_mask, temperature, chunk_size, logp,
                              ent, lse, ws)
        if rc:
            raise LmheadError(rc, "lmhead_logps_fwd")
        return logp, ent, lse

    def backward(self, hidden, weight, targets, loss_mask, temperature, chunk_size, grad_logp,
                 grad_entropy, lse, entropy, d_weight, accumulate, workspace=None):
        T, H = hidden.shape
        dev = hidden.device
        d_hidden = torch.empty((T, H), dtype=torch.float32, device=dev)
        ws = self._ws(T, H, weight.shape[0], chunk_size, dev, workspace)
        rc = lmhead_logps_bwd(hidden, weight, targets, loss_mask, temperature, chunk_size,
                              grad_logp, grad_entropy, lse,
                              entropy if grad_entropy is not None else None, d_hidden, d_weight,
                              accumulate, ws)
        if rc:
            raise LmheadError(rc, "lmhead_logps_bwd")
        return d_hidden


def _world(group):
    return dist.get_world_size(group), dist.get_rank(group)


def vocab_parallel_forward(hidden, weight_shard, targets, loss_mask, vocab_offset, vocab_total,
                           temperature=1.0, chunk_size=512, group=None, ops=None):
    """(logp, entropy, lse) [T] over the whole vocabulary, on every rank.

    Every rank passes the same tokens (hidden, targets, loss_mask) and its own
    rows of the table; ranks are combined in rank order, so every rank gets the
    same bits."""
    ops = ops or LibraryOps()
    world, _ = _world(group)
    part = ops.shard_forward(hidden, weight_shard, targets, loss_mask, vocab_offset, vocab_total,
                             temperature, chunk_size)
    gathered = [torch.empty_like(part) for _ in range(world)]
    dist.all_gather(gathered, part.contiguous(), group=group)
    return ops.combine(torch.stack(gathered), targets, loss_mask, vocab_total)


def vocab_parallel_backward(hidden, weight_shard, targets, loss_mask, vocab_offset, vocab_total,
                            temperature, chunk_size, grad_logp, grad_entropy, lse, entropy,
                            d_weight_shard=None, accumulate=False, group=None, ops=None):
    """(d_hidden [T, H] summed over ranks, d_weight_shard [rows, H] of this rank)."""
    ops = ops or LibraryOps()
    if d_weight_shard is None:
        d_weight_shard = torch.empty(tuple(weight_shard.shape), dtype=torch.float32,
                                     device=weight_shard.device)
    d_hidden = ops.shard_backward(hidden, weight_shard, targets, loss_mask, vocab_offset,
                                  vocab_total, temperature, chunk_size, grad_logp, grad_entropy,
                                  lse, entropy, d_weight_shard, accumulate)
    dist.all_reduce(d_hidden, op=dist.ReduceOp.SUM, group=group)
    return d_hidden, d_weight_shard


def token_parallel_forward(hidden, weight, targets, loss_mask, temperature=1.0, chunk_size=512,
                           ops=None):
    """(logp, entropy, lse) of this rank's tokens: the single-GPU call, no exchange."""
    ops = ops or LibraryOps()
    return ops.forward(hidden, weight, targets, loss_mask, temperature, chunk_size)


def token_parallel_backward(hidden, weight, targets, loss_mask, temperature, chunk_size,
                            grad_logp, grad_entropy, lse, entropy, d_weight=None,
                            accumulate=False, reduce=True, group=None, ops=None):
    """(d_hidden of this rank's tokens, d_weight).

    The library writes (or, with `accumulate`, adds) the gradient of the table
    from this rank's tokens into d_weight; with `reduce` it is then all-reduced
    in place, so every rank holds the sum over every rank's tokens.  Over
    several micro-batches, accumulate locally with reduce=False and reduce with
    the last one (every rank's d_weight then holds its own tokens' sum, and the
    all-reduce adds the ranks' sums)."""
    ops = ops or LibraryOps()
    if d_weight is None:
        d_weight = torch.empty(tuple(weight.shape), dtype=torch.float32, device=weight.device)
        accumulate = False
    d_hidden = ops.backward(hidden, weight, targets, loss_mask, temperature, chunk_size,
                            grad_logp, grad_entropy, lse, entropy, d_weight, accumulate)
    if reduce:
        dist.all_reduce(d_weight, op=dist.ReduceOp.SUM, group=group)
    return d_hidden, d_weight


class VocabParallelLogps(torch.autograd.Function):
    """Autograd over the vocabulary-parallel head: (hidden [T,H], this rank's
    weight_shard [rows, H], targets, loss_mask, vocab_offset, vocab_total,
    temperature, chunk_size, group, ops, main_grad) -> (logp, entropy) over the
    whole vocabulary.  hidden's gradient is summed over ranks (all-reduce), the
    shard's gradient stays on this rank; with main_grad (fp32 [rows, H]) it is
    added there in fp32 instead of being returned.  As with any collective, every
    rank of the group runs the forward and the backward (the same inputs
    requiring gradients on every rank)."""

    @staticmethod
    def forward(ctx, hidden, weight_shard, targets, loss_mask, vocab_offset, vocab_total,
                temperature, chunk_size, group, ops, main_grad):
        logp, ent, lse = vocab_parallel_forward(hidden, weight_shard, targets, loss_mask,
                                                vocab_offset, vocab_total, temperature,
                                                chunk_size, group=group, ops=ops)
        ctx.save_for_backward(hidden, weight_shard, targets, loss_mask, lse, ent)
        ctx.args = (vocab_offset, vocab_total, temperature, chunk_size, group, ops, main_grad)
        ctx.set_materialize_grads(False)
        return logp, ent

    @staticmethod
    def backward(ctx, g_logp, g_ent):
        hidden, weight_shard, targets, loss_mask, lse, ent = ctx.saved_tensors
        vocab_offset, vocab_total, temperature, chunk_size, group, ops, main_grad = ctx.args
        none = (None,) * 11
        need_h, need_w = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        if (g_logp is None and g_ent is None) or not (need_h or need_w):
            return none
        dt = lse.dtype
        gl = None if g_logp is None else g_logp.to(dt).contiguous()
        ge = None if g_ent is None else g_ent.to(dt).contiguous()
        main = main_grad if need_w else None
        d_hidden, d_w = vocab_parallel_backward(
            hidden, weight_shard, targets, loss_mask, vocab_offset, vocab_total, temperature,
            chunk_size, gl, ge, lse, ent, d_weight_shard=main, accumulate=main is not None,
            group=group, ops=ops)
        return ((d_hidden if need_h else None, d_w if (need_w and main is None) else None)
                + (None,) * 9)


def vocab_parallel_logps(hidden, weight_shard, targets, loss_mask, vocab_offset, vocab_total,
                         temperature=1.0, chunk_size=512, group=None, ops=None, main_grad=None):
    """(logp, entropy) over the whole vocabulary, differentiable in hidden and in
    this rank's weight_shard (main_grad: see VocabParallelLogps)."""
    if main_grad is None:
        main_grad = getattr(weight_shard, "main_grad", None)
    return VocabParallelLogps.apply(hidden, weight_shard, targets, loss_mask, int(vocab_offset),
                                    int(vocab_total), float(temperature), int(chunk_size), group,
                                    ops, main_grad)
