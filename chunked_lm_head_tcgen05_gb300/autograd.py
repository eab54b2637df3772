"""PyTorch autograd wrapper over the C ABI, for use inside training loops
(for instance a chunked-sequence trainer whose per-chunk loss is this head;
"Long Sequences (SeCO)" guide, section "Efficiency").

``lmhead_logps(hidden, weight, targets, ...)`` returns (logp, entropy) and
differentiates both through ``lmhead_logps_bwd``.  When the loss does not use
the entropy, its cotangent is absent and the log-prob-only backward runs
(tunix PR #2913: GRPO stops the entropy's gradient).  All computation happens
in the library's kernels; this module only allocates outputs with torch,
keeps one reusable workspace per device and stream, and moves cotangents in
and out.

Weight gradient precision.  A head called once per sequence chunk contributes
one weight gradient per call.  Returned through autograd, each is cast to the
weight's dtype (bf16) before autograd sums them, so the sum would be formed in
bf16.  Give the call an fp32 ``main_grad`` buffer [V, H] (or set
``weight.main_grad``) and the library adds every call's gradient into it in
fp32 (``accumulate_dweight = 1``) instead; ``weight.grad`` is then left
untouched, as in trainers that keep fp32 main gradients beside bf16
parameters.
"""
import torch

from . import LMHEAD_OP_BWD, LMHEAD_OP_FWD, LmheadError, lmhead_logps_bwd, lmhead_logps_fwd, \
    lmhead_workspace_size

# (device index, stream handle) -> uint8 workspace, grown on demand.  Work on one
# stream runs in order, so every call on that stream can reuse one buffer; the
# backward needs nothing the forward left in it (lse and entropy are passed in).
_workspaces = {}


def _workspace(T, H, V, chunk_size, device):
    n = max(lmhead_workspace_size(LMHEAD_OP_FWD, T, H, V, chunk_size),
            lmhead_workspace_size(LMHEAD_OP_BWD, T, H, V, chunk_size))
    if n == 0:
        raise LmheadError(1, "lmhead_workspace_size")
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    buf = _workspaces.get(key)
    if buf is None or buf.numel() < n:
        # A smaller buffer replaced here may still be read by work queued on this
        # stream; torch's caching allocator gives its memory only to later work on
        # the same stream, so dropping the reference is safe.
        buf = torch.empty(n, dtype=torch.uint8, device=device)
        _workspaces[key] = buf
    return buf


def release_workspaces():
    """Drops the cached workspaces (their memory returns to torch's allocator)."""
    _workspaces.clear()


class LMHeadLogps(torch.autograd.Function):
    """(hidden [T,H] bf16, weight [V,H] bf16, targets [T] int32, loss_mask [T] uint8 or
    None, temperature, chunk_size, main_grad [V,H] fp32 or None) -> (logp [T] fp32,
    entropy [T] fp32)."""

    @staticmethod
    def forward(ctx, hidden, weight, targets, loss_mask, temperature, chunk_size, main_grad):
        T, H = hidden.shape
        V = weight.shape[0]
        dev = hidden.device
        logp = torch.empty(T, dtype=torch.float32, device=dev)
        ent = torch.empty(T, dtype=torch.float32, device=dev)
        lse = torch.empty(T, dtype=torch.float32, device=dev)
        ws = _workspace(T, H, V, chunk_size, dev)
        rc = lmhead_logps_fwd(hidden, weight, targets, loss_mask, temperature, chunk_size, logp,
                              ent, lse, ws)
        if rc:
            raise LmheadError(rc, "lmhead_logps_fwd")
        ctx.save_for_backward(hidden, weight, targets, loss_mask, lse, ent)
        ctx.temperature = temperature
        ctx.chunk_size = chunk_size
        ctx.main_grad = main_grad
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
        main = ctx.main_grad if need_w else None
        if (g_logp is None and g_ent is None) or not (need_h or need_w):
            return (None,) * 7
        gl = None if g_logp is None else g_logp.to(torch.float32).contiguous()
        ge = None if g_ent is None else g_ent.to(torch.float32).contiguous()
        d_hidden = torch.empty((T, H), dtype=torch.float32, device=dev)
        if main is not None:
            d_weight, accumulate = main, 1
        else:
            d_weight, accumulate = torch.empty((V, H), dtype=torch.float32, device=dev), 0
        ws = _workspace(T, H, V, ctx.chunk_size, dev)
        rc = lmhead_logps_bwd(hidden, weight, targets, loss_mask, ctx.temperature, ctx.chunk_size,
                              gl, ge, lse, ent if ge is not None else None, d_hidden, d_weight,
                              accumulate, ws)
        if rc:
            raise LmheadError(rc, "lmhead_logps_bwd")
        d_w = d_weight if (need_w and main is None) else None
        return (d_hidden if need_h else None, d_w, None, None, None, None, None)


def lmhead_logps(hidden, weight, targets, loss_mask=None, temperature=1.0, chunk_size=512,
                 main_grad=None):
    """Per-token log-prob of the target and entropy, differentiable in hidden and weight.

    main_grad: an fp32 [V, H] CUDA tensor that the backward adds the weight's
    gradient to (in fp32, in place); defaults to ``weight.main_grad`` when the
    weight has one.  With it, ``weight.grad`` is not produced."""
    if main_grad is None:
        main_grad = getattr(weight, "main_grad", None)
    if main_grad is not None:
        V, H = weight.shape
        if (main_grad.dtype != torch.float32 or tuple(main_grad.shape) != (V, H)
                or not main_grad.is_contiguous() or main_grad.device != weight.device):
            raise ValueError("main_grad must be a contiguous fp32 [V, H] tensor on the "
                             "weight's device")
    return LMHeadLogps.apply(hidden, weight, targets, loss_mask, float(temperature),
                             int(chunk_size), main_grad)
