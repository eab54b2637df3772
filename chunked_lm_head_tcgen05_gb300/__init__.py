"""Chunked LM-head log-prob + entropy head for GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/lmhead.h`` (``liblmhead.so``,
built by ``buildlib.py``).  The functions named ``lmhead_*`` mirror the C entry
points one to one and only marshal arguments: torch tensors supply device
memory and the CUDA stream, every step of the computation runs in the
library's kernels.  There is no CPU or PyTorch fallback: if the library is
missing or cannot load, every call raises.

``forward`` / ``backward`` are conveniences that allocate the outputs and the
workspace with torch and raise ``LmheadError`` on a non-zero status.
"""
import ctypes
import os

__all__ = [
    "LmheadError", "library", "library_path", "build",
    "LMHEAD_OP_FWD", "LMHEAD_OP_BWD", "STATUS_NAMES",
    "lmhead_workspace_size", "lmhead_logps_fwd", "lmhead_logps_bwd",
    "lmhead_read_device_status", "lmhead_read_scored_count", "lmhead_status_string",
    "lmhead_plan_info", "lmhead_profile_enable", "lmhead_profile_count",
    "lmhead_profile_record", "lmhead_launch_count", "lmhead_logps_fwd_noalloc",
    "NOALLOC_SCRATCH_BYTES", "lmhead_logps_fwd_bwd", "lmhead_fwd_bwd_keeps_logits",
    "LMHEAD_OP_FWD_BWD", "LMHEAD_STRATEGY_AUTO", "LMHEAD_STRATEGY_RECOMPUTE",
    "LMHEAD_STRATEGY_KEEP_LOGITS", "lmhead_score_logits_fwd", "lmhead_score_logits_bwd",
    "lmhead_selftest_bounded_wait", "lmhead_logps_fwd_shard", "lmhead_logps_bwd_shard",
    "lmhead_combine_shards",
    "forward", "backward",
]

LMHEAD_OP_FWD = 0
LMHEAD_OP_BWD = 1
LMHEAD_OP_FWD_BWD = 2
LMHEAD_STRATEGY_AUTO = 0
LMHEAD_STRATEGY_RECOMPUTE = 1
LMHEAD_STRATEGY_KEEP_LOGITS = 2
NOALLOC_SCRATCH_BYTES = 64 << 20   # LMHEAD_NOALLOC_SCRATCH_BYTES in include/lmhead.h
STATUS_NAMES = {
    0: "LMHEAD_OK", 1: "LMHEAD_ERR_INVALID_ARG", 2: "LMHEAD_ERR_UNSUPPORTED",
    3: "LMHEAD_ERR_WORKSPACE_TOO_SMALL", 4: "LMHEAD_ERR_CUDA",
    5: "LMHEAD_ERR_DEVICE_TIMEOUT", 6: "LMHEAD_ERR_BAD_TARGET", 7: "LMHEAD_ERR_INTERNAL",
}

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "liblmhead.so")
_lib = None

_VP = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t

# name -> (restype, argtypes), exactly the declarations of include/lmhead.h
_SIGNATURES = {
    "lmhead_workspace_size": (_SZ, [ctypes.c_int, _I64, _I32, _I32, _I32]),
    "lmhead_logps_fwd": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, ctypes.c_float,
                                        _I32, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "lmhead_logps_bwd": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, ctypes.c_float,
                                        _I32, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_int, _VP,
                                        _SZ, _VP]),
    "lmhead_read_device_status": (ctypes.c_int, [_VP, _VP]),
    "lmhead_read_scored_count": (_I64, [_VP, _VP]),
    "lmhead_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "lmhead_plan_info": (ctypes.c_int, [_I64, _I32, _I32, _I32, ctypes.POINTER(_I32),
                                        ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "lmhead_profile_enable": (None, [ctypes.c_int]),
    "lmhead_profile_count": (ctypes.c_int, []),
    "lmhead_profile_record": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_char_p),
                                             ctypes.POINTER(ctypes.c_float)]),
    "lmhead_launch_count": (ctypes.c_uint64, []),
    "lmhead_logps_fwd_noalloc": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I32, _I32,
                                                ctypes.c_float, _I32, _VP, _VP, _VP, _VP]),
    "lmhead_logps_fwd_bwd": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I32, _I32,
                                            ctypes.c_float, _I32, _VP, _VP, _VP, _VP, _VP, _VP,
                                            _VP, ctypes.c_int, ctypes.c_int, _VP, _SZ, _VP]),
    "lmhead_fwd_bwd_keeps_logits": (ctypes.c_int, [_I64, _I32, _I32, _I32,
                                                   ctypes.POINTER(_I32)]),
    "lmhead_selftest_bounded_wait": (ctypes.c_int, [_VP, _SZ, ctypes.c_uint32, _VP]),
    "lmhead_score_logits_fwd": (ctypes.c_int, [_VP, _VP, _VP, _I64, _I32, ctypes.c_float, _VP,
                                               _VP, _VP, _VP]),
    "lmhead_score_logits_bwd": (ctypes.c_int, [_VP, _VP, _VP, _I64, _I32, ctypes.c_float, _VP,
                                               _VP, _VP, _VP, _VP, _VP]),
    "lmhead_logps_fwd_shard": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, _I32, _I32,
                                              ctypes.c_float, _I32, _VP, _VP, _SZ, _VP]),
    "lmhead_combine_shards": (ctypes.c_int, [_VP, _I32, _VP, _VP, _I64, _I32, _VP, _VP, _VP,
                                             _VP]),
    "lmhead_logps_bwd_shard": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, _I32, _I32,
                                              ctypes.c_float, _I32, _VP, _VP, _VP, _VP, _VP, _VP,
                                              ctypes.c_int, _VP, _SZ, _VP]),
}


class LmheadError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = int(status)
        super().__init__("%s%s" % (where + ": " if where else "",
                                   STATUS_NAMES.get(self.status, "status %d" % self.status)))


def build(force=False):
    """Compile liblmhead.so for sm_103a (nvcc); returns its path."""
    from . import buildlib
    return buildlib.build(force=force)


def library():
    """The loaded liblmhead.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError("liblmhead.so is not built (run chunked_lm_head_tcgen05_gb300.build())")
        lib = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check_tensor(t, name, dtype, shape, allow_none=False):
    import torch
    if t is None:
        if allow_none:
            return
        raise ValueError("%s is required" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    del torch


def _on_device(tensors, stream, fn):
    """Run fn() with the tensors' CUDA device current.  The library launches
    on the current device, so a call whose tensors (or stream) live on
    another device, or on several, is refused here instead of launched."""
    import torch
    devs = {t.device for t in tensors if t is not None}
    if stream is not None and not isinstance(stream, int) and hasattr(stream, "device"):
        devs.add(stream.device)
    if len(devs) > 1:
        raise ValueError("all tensors and the stream of one call must be on one CUDA device, "
                         "got %s" % sorted(str(d) for d in devs))
    if not devs:
        return fn()
    with torch.cuda.device(devs.pop()):
        return fn()


def _check_workspace(ws):
    if ws is None or not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")


def lmhead_workspace_size(op, T, H, V, chunk_size):
    return int(library().lmhead_workspace_size(op, T, H, V, chunk_size))


def lmhead_logps_fwd(hidden, weight, targets, loss_mask, temperature, chunk_size, logp, entropy,
                     lse, workspace, stream=None):
    """C ``lmhead_logps_fwd`` on torch tensors; returns the status code."""
    import torch
    T, H = hidden.shape
    V = weight.shape[0]
    _check_tensor(hidden, "hidden", torch.bfloat16, (T, H))
    _check_tensor(weight, "weight", torch.bfloat16, (V, H))
    _check_tensor(targets, "targets", torch.int32, (T,))
    _check_tensor(loss_mask, "loss_mask", torch.uint8, (T,), allow_none=True)
    _check_tensor(logp, "logp", torch.float32, (T,))
    _check_tensor(entropy, "entropy", torch.float32, (T,), allow_none=True)
    _check_tensor(lse, "lse", torch.float32, (T,))
    _check_workspace(workspace)
    tensors = [hidden, weight, targets, loss_mask, logp, entropy, lse, workspace]
    return _on_device(tensors, stream, lambda: int(library().lmhead_logps_fwd(
        _ptr(hidden), _ptr(weight), _ptr(targets), _ptr(loss_mask), T, H, V, float(temperature),
        int(chunk_size), _ptr(logp), _ptr(entropy), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))))


def lmhead_logps_bwd(hidden, weight, targets, loss_mask, temperature, chunk_size, grad_logp,
                     grad_entropy, lse, entropy, d_hidden, d_weight, accumulate_dweight, workspace,
                     stream=None):
    """C ``lmhead_logps_bwd`` on torch tensors; returns the status code."""
    import torch
    T, H = hidden.shape
    V = weight.shape[0]
    _check_tensor(hidden, "hidden", torch.bfloat16, (T, H))
    _check_tensor(weight, "weight", torch.bfloat16, (V, H))
    _check_tensor(targets, "targets", torch.int32, (T,))
    _check_tensor(loss_mask, "loss_mask", torch.uint8, (T,), allow_none=True)
    _check_tensor(grad_logp, "grad_logp", torch.float32, (T,), allow_none=True)
    _check_tensor(grad_entropy, "grad_entropy", torch.float32, (T,), allow_none=True)
    _check_tensor(lse, "lse", torch.float32, (T,))
    _check_tensor(entropy, "entropy", torch.float32, (T,), allow_none=True)
    _check_tensor(d_hidden, "d_hidden", torch.float32, (T, H))
    _check_tensor(d_weight, "d_weight", torch.float32, (V, H))
    _check_workspace(workspace)
    tensors = [hidden, weight, targets, loss_mask, grad_logp, grad_entropy, lse, entropy,
               d_hidden, d_weight, workspace]
    return _on_device(tensors, stream, lambda: int(library().lmhead_logps_bwd(
        _ptr(hidden), _ptr(weight), _ptr(targets), _ptr(loss_mask), T, H, V, float(temperature),
        int(chunk_size), _ptr(grad_logp), _ptr(grad_entropy), _ptr(lse), _ptr(entropy),
        _ptr(d_hidden), _ptr(d_weight), int(bool(accumulate_dweight)), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))))


def lmhead_logps_fwd_noalloc(hidden, weight, targets, loss_mask, temperature, chunk_size, logp,
                             entropy, lse, stream=None):
    """C ``lmhead_logps_fwd_noalloc`` on torch tensors; returns the status code.

    For callers that cannot allocate device memory: no workspace argument,
    the scratch is the library's static per-GPU array (up to
    LMHEAD_NOALLOC_SCRATCH_BYTES of forward workspace)."""
    import torch
    T, H = hidden.shape
    V = weight.shape[0]
    _check_tensor(hidden, "hidden", torch.bfloat16, (T, H))
    _check_tensor(weight, "weight", torch.bfloat16, (V, H))
    _check_tensor(targets, "targets", torch.int32, (T,))
    _check_tensor(loss_mask, "loss_mask", torch.uint8, (T,), allow_none=True)
    _check_tensor(logp, "logp", torch.float32, (T,))
    _check_tensor(entropy, "entropy", torch.float32, (T,), allow_none=True)
    _check_tensor(lse, "lse", torch.float32, (T,))
    tensors = [hidden, weight, targets, loss_mask, logp, entropy, lse]
    return _on_device(tensors, stream, lambda: int(library().lmhead_logps_fwd_noalloc(
        _ptr(hidden), _ptr(weight), _ptr(targets), _ptr(loss_mask), T, H, V, float(temperature),
        int(chunk_size), _ptr(logp), _ptr(entropy), _ptr(lse), _stream(stream))))


def lmhead_logps_fwd_bwd(hidden, weight, targets, loss_mask, temperature, chunk_size, grad_logp,
                         grad_entropy, logp, entropy, lse, d_hidden, d_weight,
                         accumulate_dweight, strategy, workspace, stream=None):
    """C ``lmhead_logps_fwd_bwd`` on torch tensors; returns the status code."""
    import torch
    T, H = hidden.shape
    V = weight.shape[0]
    _check_tensor(hidden, "hidden", torch.bfloat16, (T, H))
    _check_tensor(weight, "weight", torch.bfloat16, (V, H))
    _check_tensor(targets, "targets", torch.int32, (T,))
    _check_tensor(loss_mask, "loss_mask", torch.uint8, (T,), allow_none=True)
    _check_tensor(grad_logp, "grad_logp", torch.float32, (T,), allow_none=True)
    _check_tensor(grad_entropy, "grad_entropy", torch.float32, (T,), allow_none=True)
    _check_tensor(logp, "logp", torch.float32, (T,))
    _check_tensor(entropy, "entropy", torch.float32, (T,), allow_none=True)
    _check_tensor(lse, "lse", torch.float32, (T,))
    _check_tensor(d_hidden, "d_hidden", torch.float32, (T, H))
    _check_tensor(d_weight, "d_weight", torch.float32, (V, H))
    _check_workspace(workspace)
    tensors = [hidden, weight, targets, loss_mask, grad_logp, grad_entropy, logp, entropy, lse,
               d_hidden, d_weight, workspace]
    return _on_device(tensors, stream, lambda: int(library().lmhead_logps_fwd_bwd(
        _ptr(hidden), _ptr(weight), _ptr(targets), _ptr(loss_mask), T, H, V, float(temperature),
        int(chunk_size), _ptr(grad_logp), _ptr(grad_entropy), _ptr(logp), _ptr(entropy),
        _ptr(lse), _ptr(d_hidden), _ptr(d_weight), int(bool(accumulate_dweight)), int(strategy),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))))


def lmhead_fwd_bwd_keeps_logits(T, H, V, chunk_size):
    """(keeps logits under AUTO: bool, token block of the keep-logits path)."""
    tb = _I32()
    r = int(library().lmhead_fwd_bwd_keeps_logits(T, H, V, chunk_size, ctypes.byref(tb)))
    if r < 0:
        raise LmheadError(1, "lmhead_fwd_bwd_keeps_logits")
    return bool(r), tb.value


def lmhead_score_logits_fwd(logits, targets, loss_mask, temperature, logp, entropy, lse,
                            stream=None):
    """C ``lmhead_score_logits_fwd`` on torch tensors; returns the status code."""
    import torch
    T, V = logits.shape
    _check_tensor(logits, "logits", torch.float32, (T, V))
    _check_tensor(targets, "targets", torch.int32, (T,))
    _check_tensor(loss_mask, "loss_mask", torch.uint8, (T,), allow_none=True)
    _check_tensor(logp, "logp", torch.float32, (T,))
    _check_tensor(entropy, "entropy", torch.float32, (T,), allow_none=True)
    _check_tensor(lse, "lse", torch.float32, (T,))
    tensors = [logits, targets, loss_mask, logp, entropy, lse]
    return _on_device(tensors, stream, lambda: int(library().lmhead_score_logits_fwd(
        _ptr(logits), _ptr(targets), _ptr(loss_mask), T, V, float(temperature), _ptr(logp),
        _ptr(entropy), _ptr(lse), _stream(stream))))


def lmhead_score_logits_bwd(logits, targets, loss_mask, temperature, grad_logp, grad_entropy,
                            lse, entropy, d_logits, stream=None):
    """C ``lmhead_score_logits_bwd`` on torch tensors; returns the status code."""
    import torch
    T, V = logits.shape
    _check_tensor(logits, "logits", torch.float32, (T, V))
    _check_tensor(targets, "targets", torch.int32, (T,))
    _check_tensor(loss_mask, "loss_mask", torch.uint8, (T,), allow_none=True)
    _check_tensor(grad_logp, "grad_logp", torch.float32, (T,), allow_none=True)
    _check_tensor(grad_entropy, "grad_entropy", torch.float32, (T,), allow_none=True)
    _check_tensor(lse, "lse", torch.float32, (T,))
    _check_tensor(entropy, "entropy", torch.float32, (T,), allow_none=True)
    _check_tensor(d_logits, "d_logits", torch.float32, (T, V))
    tensors = [logits, targets, loss_mask, grad_logp, grad_entropy, lse, entropy, d_logits]
    return _on_device(tensors, stream, lambda: int(library().lmhead_score_logits_bwd(
        _ptr(logits), _ptr(targets), _ptr(loss_mask), T, V, float(temperature), _ptr(grad_logp),
        _ptr(grad_entropy), _ptr(lse), _ptr(entropy), _ptr(d_logits), _stream(stream))))


def lmhead_logps_fwd_shard(hidden, weight_shard, targets, loss_mask, vocab_offset, vocab_total,
                           temperature, chunk_size, partials, workspace, stream=None):
    """C ``lmhead_logps_fwd_shard`` on torch tensors (partials: fp32 [T, 4]); returns
    the status code."""
    import torch
    T, H = hidden.shape
    Vs = weight_shard.shape[0]
    _check_tensor(hidden, "hidden", torch.bfloat16, (T, H))
    _check_tensor(weight_shard, "weight_shard", torch.bfloat16, (Vs, H))
    _check_tensor(targets, "targets", torch.int32, (T,))
    _check_tensor(loss_mask, "loss_mask", torch.uint8, (T,), allow_none=True)
    _check_tensor(partials, "partials", torch.float32, (T, 4))
    _check_workspace(workspace)
    tensors = [hidden, weight_shard, targets, loss_mask, partials, workspace]
    return _on_device(tensors, stream, lambda: int(library().lmhead_logps_fwd_shard(
        _ptr(hidden), _ptr(weight_shard), _ptr(targets), _ptr(loss_mask), T, H, Vs,
        int(vocab_offset), int(vocab_total), float(temperature), int(chunk_size), _ptr(partials),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))))


def lmhead_combine_shards(partials, targets, loss_mask, vocab_total, logp, entropy, lse,
                          stream=None):
    """C ``lmhead_combine_shards`` (partials: fp32 [n_shards, T, 4]); returns the status."""
    import torch
    n, T = partials.shape[0], partials.shape[1]
    _check_tensor(partials, "partials", torch.float32, (n, T, 4))
    _check_tensor(targets, "targets", torch.int32, (T,))
    _check_tensor(loss_mask, "loss_mask", torch.uint8, (T,), allow_none=True)
    _check_tensor(logp, "logp", torch.float32, (T,))
    _check_tensor(entropy, "entropy", torch.float32, (T,), allow_none=True)
    _check_tensor(lse, "lse", torch.float32, (T,))
    tensors = [partials, targets, loss_mask, logp, entropy, lse]
    return _on_device(tensors, stream, lambda: int(library().lmhead_combine_shards(
        _ptr(partials), n, _ptr(targets), _ptr(loss_mask), T, int(vocab_total), _ptr(logp),
        _ptr(entropy), _ptr(lse), _stream(stream))))


def lmhead_logps_bwd_shard(hidden, weight_shard, targets, loss_mask, vocab_offset, vocab_total,
                           temperature, chunk_size, grad_logp, grad_entropy, lse, entropy,
                           d_hidden, d_weight_shard, accumulate_dweight, workspace, stream=None):
    """C ``lmhead_logps_bwd_shard`` on torch tensors; returns the status code."""
    import torch
    T, H = hidden.shape
    Vs = weight_shard.shape[0]
    _check_tensor(hidden, "hidden", torch.bfloat16, (T, H))
    _check_tensor(weight_shard, "weight_shard", torch.bfloat16, (Vs, H))
    _check_tensor(targets, "targets", torch.int32, (T,))
    _check_tensor(loss_mask, "loss_mask", torch.uint8, (T,), allow_none=True)
    _check_tensor(grad_logp, "grad_logp", torch.float32, (T,), allow_none=True)
    _check_tensor(grad_entropy, "grad_entropy", torch.float32, (T,), allow_none=True)
    _check_tensor(lse, "lse", torch.float32, (T,))
    _check_tensor(entropy, "entropy", torch.float32, (T,), allow_none=True)
    _check_tensor(d_hidden, "d_hidden", torch.float32, (T, H))
    _check_tensor(d_weight_shard, "d_weight_shard", torch.float32, (Vs, H))
    _check_workspace(workspace)
    tensors = [hidden, weight_shard, targets, loss_mask, grad_logp, grad_entropy, lse, entropy,
               d_hidden, d_weight_shard, workspace]
    return _on_device(tensors, stream, lambda: int(library().lmhead_logps_bwd_shard(
        _ptr(hidden), _ptr(weight_shard), _ptr(targets), _ptr(loss_mask), T, H, Vs,
        int(vocab_offset), int(vocab_total), float(temperature), int(chunk_size),
        _ptr(grad_logp), _ptr(grad_entropy), _ptr(lse), _ptr(entropy), _ptr(d_hidden),
        _ptr(d_weight_shard), int(bool(accumulate_dweight)), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))))


def lmhead_selftest_bounded_wait(workspace, limit_ms, stream=None):
    """C ``lmhead_selftest_bounded_wait``; returns the status code of the launch."""
    _check_workspace(workspace)
    return _on_device([workspace], stream, lambda: int(library().lmhead_selftest_bounded_wait(
        _ptr(workspace), workspace.numel() * workspace.element_size(), int(limit_ms),
        _stream(stream))))


def lmhead_read_device_status(workspace, stream=None):
    _check_workspace(workspace)
    return _on_device([workspace], stream, lambda: int(
        library().lmhead_read_device_status(_ptr(workspace), _stream(stream))))


def lmhead_read_scored_count(workspace, stream=None):
    _check_workspace(workspace)
    return _on_device([workspace], stream, lambda: int(
        library().lmhead_read_scored_count(_ptr(workspace), _stream(stream))))


def lmhead_status_string(status):
    return library().lmhead_status_string(int(status)).decode()


def lmhead_plan_info(T, H, V, chunk_size):
    """(fwd_splits, bwd_tokens, bwd_vocab) for these sizes on the current device."""
    a, b, c = _I32(), _I32(), _I32()
    rc = library().lmhead_plan_info(T, H, V, chunk_size, ctypes.byref(a), ctypes.byref(b),
                                    ctypes.byref(c))
    if rc:
        raise LmheadError(rc, "lmhead_plan_info")
    return a.value, b.value, c.value


def lmhead_profile_enable(on):
    library().lmhead_profile_enable(int(bool(on)))


def lmhead_profile_count():
    return int(library().lmhead_profile_count())


def lmhead_profile_record(i):
    """(kernel name, milliseconds) of the i-th recorded launch."""
    name = ctypes.c_char_p()
    ms = ctypes.c_float()
    rc = library().lmhead_profile_record(i, ctypes.byref(name), ctypes.byref(ms))
    if rc:
        raise LmheadError(rc, "lmhead_profile_record")
    return name.value.decode(), float(ms.value)


def lmhead_launch_count():
    return int(library().lmhead_launch_count())


# ----------------------------------------------------------------- conveniences
def _workspace(op, T, H, V, chunk_size, device):
    import torch
    n = lmhead_workspace_size(op, T, H, V, chunk_size)
    if n == 0:
        raise LmheadError(1, "lmhead_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def forward(hidden, weight, targets, loss_mask=None, temperature=1.0, chunk_size=512,
            with_entropy=True, workspace=None, stream=None):
    """Returns (logp, entropy or None, lse) as fp32 CUDA tensors."""
    import torch
    T, H = hidden.shape
    V = weight.shape[0]
    dev = hidden.device
    logp = torch.empty(T, dtype=torch.float32, device=dev)
    ent = torch.empty(T, dtype=torch.float32, device=dev) if with_entropy else None
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = _workspace(LMHEAD_OP_FWD, T, H, V, chunk_size, dev)
    rc = lmhead_logps_fwd(hidden, weight, targets, loss_mask, temperature, chunk_size, logp, ent,
                          lse, workspace, stream)
    if rc:
        raise LmheadError(rc, "lmhead_logps_fwd")
    return logp, ent, lse


def backward(hidden, weight, targets, loss_mask, temperature, chunk_size, grad_logp,
             grad_entropy, lse, entropy=None, d_weight=None, accumulate_dweight=False,
             workspace=None, stream=None):
    """Returns (d_hidden [T,H] fp32, d_weight [V,H] fp32)."""
    import torch
    T, H = hidden.shape
    V = weight.shape[0]
    dev = hidden.device
    d_hidden = torch.empty((T, H), dtype=torch.float32, device=dev)
    if d_weight is None:
        d_weight = torch.empty((V, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = _workspace(LMHEAD_OP_BWD, T, H, V, chunk_size, dev)
    rc = lmhead_logps_bwd(hidden, weight, targets, loss_mask, temperature, chunk_size, grad_logp,
                          grad_entropy, lse, entropy, d_hidden, d_weight, accumulate_dweight,
                          workspace, stream)
    if rc:
        raise LmheadError(rc, "lmhead_logps_bwd")
    return d_hidden, d_weight
