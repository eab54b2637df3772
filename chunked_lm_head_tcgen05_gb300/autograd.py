"""PyTorch autograd wrapper over the C ABI, for use inside training loops
(for instance a chunked-sequence trainer whose per-chunk loss is this head;
"Long Sequences (SeCO)" guide, section "Efficiency").

``lmhead_logps(hidden, weight, targets, ...)`` returns (logp, entropy) and
differentiates both through ``lmhead_logps_bwd``.  When the loss does not use
the entropy, its cotangent is absent and the log-prob-only backward runs
(tunix PR #2913: GRPO stops the entropy's gradient).  All computation happens
in the library's kernels; this module only allocates outputs and workspaces
with torch and moves cotangents in and out.
"""
import torch

from . import (LMHEAD_OP_BWD, LMHEAD_OP_FWD, LmheadError, lmhead_logps_bwd, lmhead_logps_fwd,
               lmhead_workspace_size)


def _workspace(op, T, H, V, chunk_size, device):
    n = lmhead_workspace_size(op, T, H, V, chunk_size)
    if n == 0:
        raise LmheadError(1, "lmhead_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


class LMHeadLogps(torch.autograd.Function):
    """(hidden [T,H] bf16, weight [V,H] bf16, targets [T] int32, loss_mask [T] uint8 or
    None, temperature, chunk_size) -> (logp [T] fp32, entropy [T] fp32)."""

    @staticmethod
    def forward(ctx, hidden, weight, targets, loss_mask, temperature, chunk_size):
        T, H = hidden.shape
        V = weight.shape[0]
        dev = hidden.device
        logp = torch.empty(T, dtype=torch.float32, device=dev)
        ent = torch.empty(T, dtype=torch.float32, device=dev)
        lse = torch.empty(T, dtype=torch.float32, device=dev)
        ws = _workspace(LMHEAD_OP_FWD, T, H, V, chunk_size, dev)
        rc = lmhead_logps_fwd(hidden, weight, targets, loss_mask, temperature, chunk_size, logp,
                              ent, lse, ws)
        if rc:
            raise LmheadError(rc, "lmhead_logps_fwd")
        ctx.save_for_backward(hidden, weight, targets, loss_mask, lse, ent)
        ctx.temperature = temperature
        ctx.chunk_size = chunk_size
        ctx.set_materialize_grads(False)
        ctx.mark_non_differentiable(lse)
        return logp, ent

    @staticmethod
    def backward(ctx, g_logp, g_ent):
        hidden, weight, targets, loss_mask, lse, ent = ctx.saved_tensors
        T, H = hidden.shape
        V = weight.shape[0]
        dev = hidden.device
        need_h, need_w = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        if (g_logp is None and g_ent is None) or not (need_h or need_w):
            return None, None, None, None, None, None
        gl = None if g_logp is None else g_logp.to(torch.float32).contiguous()
        ge = None if g_ent is None else g_ent.to(torch.float32).contiguous()
        d_hidden = torch.empty((T, H), dtype=torch.float32, device=dev)
        d_weight = torch.empty((V, H), dtype=torch.float32, device=dev)
        ws = _workspace(LMHEAD_OP_BWD, T, H, V, ctx.chunk_size, dev)
        rc = lmhead_logps_bwd(hidden, weight, targets, loss_mask, ctx.temperature, ctx.chunk_size,
                              gl, ge, lse, ent if ge is not None else None, d_hidden, d_weight,
                              0, ws)
        if rc:
            raise LmheadError(rc, "lmhead_logps_bwd")
        return (d_hidden if need_h else None, d_weight if need_w else None, None, None, None,
                None)


def lmhead_logps(hidden, weight, targets, loss_mask=None, temperature=1.0, chunk_size=512):
    """Per-token log-prob of the target and entropy, differentiable in hidden and weight."""
    return LMHeadLogps.apply(hidden, weight, targets, loss_mask, float(temperature),
                             int(chunk_size))
