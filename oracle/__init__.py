"""fp64 CPU oracle for the chunked LM-head log-prob + entropy head.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The product path never
imports this package, and this package imports nothing from the product.

The arithmetic lives in ``lmhead_oracle.c`` (plain double-precision loops,
OpenMP over rows).  This module only marshals numpy arrays into it.

Matrices may be given as float64 arrays, or as uint16 arrays holding raw
bfloat16 bit patterns (decoded exactly inside the C code).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_VP = ctypes.c_void_p


def _matrix(a, rows, cols, name):
    a = np.ascontiguousarray(a)
    if a.shape != (rows, cols):
        raise ValueError("%s has shape %s, expected %s" % (name, a.shape, (rows, cols)))
    if a.dtype == np.uint16:
        return a, 1
    if a.dtype == np.float64:
        return a, 0
    raise TypeError("%s must be float64 or uint16 (bfloat16 bits), got %s" % (name, a.dtype))


def _vec(a, n, dtype, name):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=dtype)
    if a.shape != (n,):
        raise ValueError("%s has shape %s, expected (%d,)" % (name, a.shape, n))
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_VP)


class Oracle:
    """One loaded copy of the oracle library (tests may load variants)."""

    def __init__(self, library_path=None):
        if library_path is None:
            library_path = _build.build()
        self.path = library_path
        lib = ctypes.CDLL(os.path.abspath(library_path))
        lib.lmo_forward.restype = ctypes.c_int
        lib.lmo_forward.argtypes = [_I64, _I32, _I32, _VP, ctypes.c_int, _VP, ctypes.c_int,
                                    _VP, _VP, ctypes.c_double, _VP, _VP, _VP]
        lib.lmo_backward.restype = ctypes.c_int
        lib.lmo_backward.argtypes = [_I64, _I32, _I32, _VP, ctypes.c_int, _VP, ctypes.c_int,
                                     _VP, _VP, ctypes.c_double, _VP, _VP, _VP, _VP]
        lib.lmo_num_threads.restype = ctypes.c_int
        lib.lmo_logits_forward.restype = ctypes.c_int
        lib.lmo_logits_forward.argtypes = [_I64, _I32, _VP, _VP, _VP, ctypes.c_double, _VP, _VP,
                                           _VP]
        lib.lmo_logits_backward.restype = ctypes.c_int
        lib.lmo_logits_backward.argtypes = [_I64, _I32, _VP, _VP, _VP, ctypes.c_double, _VP, _VP,
                                            _VP]
        self._lib = lib

    def num_threads(self):
        return int(self._lib.lmo_num_threads())

    def forward(self, hidden, weight, targets, mask, temperature):
        """Returns (logp, entropy, lse), float64 arrays of length T."""
        T, H = np.shape(hidden)
        V = np.shape(weight)[0]
        h, hb = _matrix(hidden, T, H, "hidden")
        w, wb = _matrix(weight, V, H, "weight")
        y = _vec(targets, T, np.int32, "targets")
        m = _vec(mask, T, np.uint8, "mask")
        logp = np.empty(T, np.float64)
        ent = np.empty(T, np.float64)
        lse = np.empty(T, np.float64)
        rc = self._lib.lmo_forward(T, H, V, _ptr(h), hb, _ptr(w), wb, _ptr(y), _ptr(m),
                                   float(temperature), _ptr(logp), _ptr(ent), _ptr(lse))
        if rc != 0:
            raise ValueError("oracle forward failed with code %d" % rc)
        return logp, ent, lse

    def backward(self, hidden, weight, targets, mask, temperature, grad_logp, grad_entropy,
                 want_dweight=True):
        """Returns (d_hidden [T,H], d_weight [V,H] or None), float64."""
        T, H = np.shape(hidden)
        V = np.shape(weight)[0]
        h, hb = _matrix(hidden, T, H, "hidden")
        w, wb = _matrix(weight, V, H, "weight")
        y = _vec(targets, T, np.int32, "targets")
        m = _vec(mask, T, np.uint8, "mask")
        gl = _vec(grad_logp, T, np.float64, "grad_logp")
        ge = _vec(grad_entropy, T, np.float64, "grad_entropy")
        dh = np.empty((T, H), np.float64)
        dw = np.empty((V, H), np.float64) if want_dweight else None
        rc = self._lib.lmo_backward(T, H, V, _ptr(h), hb, _ptr(w), wb, _ptr(y), _ptr(m),
                                    float(temperature), _ptr(gl), _ptr(ge), _ptr(dh), _ptr(dw))
        if rc != 0:
            raise ValueError("oracle backward failed with code %d" % rc)
        return dh, dw


    def logits_forward(self, logits, targets, mask, temperature):
        """Scoring of given logits [T,V] (float64): (logp, entropy, lse)."""
        logits = np.ascontiguousarray(logits, dtype=np.float64)
        T, V = logits.shape
        y = _vec(targets, T, np.int32, "targets")
        m = _vec(mask, T, np.uint8, "mask")
        out = [np.empty(T, np.float64) for _ in range(3)]
        rc = self._lib.lmo_logits_forward(T, V, _ptr(logits), _ptr(y), _ptr(m), float(temperature),
                                          *[_ptr(a) for a in out])
        if rc != 0:
            raise ValueError("oracle logits forward failed with code %d" % rc)
        return tuple(out)

    def logits_backward(self, logits, targets, mask, temperature, grad_logp, grad_entropy):
        """d loss / d logits [T,V] (float64)."""
        logits = np.ascontiguousarray(logits, dtype=np.float64)
        T, V = logits.shape
        y = _vec(targets, T, np.int32, "targets")
        m = _vec(mask, T, np.uint8, "mask")
        gl = _vec(grad_logp, T, np.float64, "grad_logp")
        ge = _vec(grad_entropy, T, np.float64, "grad_entropy")
        d = np.empty((T, V), np.float64)
        rc = self._lib.lmo_logits_backward(T, V, _ptr(logits), _ptr(y), _ptr(m), float(temperature),
                                           _ptr(gl), _ptr(ge), _ptr(d))
        if rc != 0:
            raise ValueError("oracle logits backward failed with code %d" % rc)
        return d


_default = None


def default():
    """The oracle built from this directory's source."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def forward(*args, **kwargs):
    return default().forward(*args, **kwargs)


def backward(*args, **kwargs):
    return default().backward(*args, **kwargs)
