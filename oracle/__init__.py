"""CPU oracle for the gated delta-rule SSM block (TEST INFRASTRUCTURE ONLY).

A thin ctypes layer over ``gdn_ref.c``: numpy arrays in, numpy arrays out. The
arithmetic lives in C, written step by step from the pages:

* ``decay_gate``      fm_kernel_ssm.m, "Decay gate"; ssm_gated_delta.cu, glue kernels
* ``sigmoid``         ssm_gated_delta.cu, glue kernels (fc_sigmoid)
* ``conv1d_silu_seq`` fm_kernel_ssm.m, "Causal depthwise conv1d + SiLU"; ssm_gated_delta.cu, Kernel 2
* ``l2norm``          ssm_gated_delta.cu, glue kernels (fc_ssm_qknorm_gqa)
* ``recurrence``      fm_kernel_ssm.m, "Delta-rule recurrence"; ssm_gated_delta.cu, Kernel 1;
                      gated_delta_net_decode.metal, "Mathematical recurrence"
* ``gated_norm``      fm_kernel_ssm.m, "Gated RMSNorm"; ssm_gated_delta.cu, Kernel 3
* ``block_decode``    the single-token glue order of ssm_gated_delta.cu

All functions are pinned in tests/test_oracle.py. Only the tests, the smoke
check and the benchmark's CPU-baseline leg may import this package; the
product path (the CUDA library and its binding) never does.

``prec`` selects the float build ("f32", the pages' precision) or the double
build ("f64", used to measure the GPU's error).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIBS = {}
_I32P = ctypes.POINTER(ctypes.c_int32)


def _configure(lib, prec):
    real = ctypes.c_float if prec == "f32" else ctypes.c_double
    rp = ctypes.c_void_p
    i = ctypes.c_int
    lib.gdn_ref_precision.restype = i
    lib.gdn_ref_softplus.argtypes = [real]
    lib.gdn_ref_softplus.restype = real
    lib.gdn_ref_silu.argtypes = [real]
    lib.gdn_ref_silu.restype = real
    lib.gdn_ref_decay_gate.argtypes = [rp, rp, rp, rp, i, i]
    lib.gdn_ref_sigmoid.argtypes = [rp, rp, i]
    lib.gdn_ref_conv1d_silu_seq.argtypes = [rp, rp, rp, rp, i, i, i, i, rp, i, i]
    lib.gdn_ref_conv1d_silu_seq.restype = i
    lib.gdn_ref_l2norm.argtypes = [rp, rp, i, i, real]
    lib.gdn_ref_recurrence.argtypes = [rp, rp, rp, rp, rp, rp, rp, i, i, i, i, i, real, rp, i]
    lib.gdn_ref_recurrence.restype = i
    lib.gdn_ref_gated_norm.argtypes = [rp, rp, rp, rp, i, i, real]
    lib.gdn_ref_block_decode.argtypes = [rp] * 11 + [i, i, i, i, i, real, real, real, rp, i]
    lib.gdn_ref_block_decode.restype = i
    expect = 1 if prec == "f32" else 2
    assert lib.gdn_ref_precision() == expect, "oracle library built with the wrong precision"
    return lib


def _lib(prec):
    if prec not in _LIBS:
        _LIBS[prec] = _configure(ctypes.CDLL(_build.build()[prec]), prec)
    return _LIBS[prec]


def _swap_library(prec, path):
    """Test hook: route `prec` calls to another build of the oracle source (the
    mutation test compiles deliberately broken copies). Returns the previous
    library object, or None; pass it back through _restore_library."""
    prev = _LIBS.get(prec)
    _LIBS[prec] = _configure(ctypes.CDLL(path), prec)
    return prev


def _restore_library(prec, prev):
    if prev is None:
        _LIBS.pop(prec, None)
    else:
        _LIBS[prec] = prev


def _dt(prec):
    return np.float32 if prec == "f32" else np.float64


def _in(x, prec):
    """Contiguous copy (or view) of x in the oracle's real type."""
    return np.ascontiguousarray(np.asarray(x), dtype=_dt(prec))


def _inout(x, prec):
    """An in/out array must already be contiguous and of the oracle's type."""
    if not (isinstance(x, np.ndarray) and x.dtype == _dt(prec) and x.flags.c_contiguous):
        raise TypeError("in/out arrays must be C-contiguous numpy arrays of the oracle dtype")
    return x


def _p(x):
    return None if x is None else ctypes.c_void_p(x.ctypes.data)


def _slots(slots):
    if slots is None:
        return None, None
    s = np.ascontiguousarray(slots, dtype=np.int32)
    return s, ctypes.c_void_p(s.ctypes.data)


def softplus(v, prec="f64"):
    return float(_lib(prec).gdn_ref_softplus(float(v)))


def silu(x, prec="f64"):
    return float(_lib(prec).gdn_ref_silu(float(x)))


def decay_gate(alpha, dt, a, prec="f64"):
    """g[r][h] = a[h] * softplus(alpha[r][h] + dt[h]); alpha is [rows][H]."""
    alpha, dt, a = _in(alpha, prec), _in(dt, prec), _in(a, prec)
    H = dt.shape[0]
    rows = alpha.size // H
    g = np.zeros(alpha.shape, dtype=_dt(prec))
    _lib(prec).gdn_ref_decay_gate(_p(alpha), _p(dt), _p(a), _p(g), H, rows)
    return g


def sigmoid(b, prec="f64"):
    b = _in(b, prec)
    out = np.zeros(b.shape, dtype=_dt(prec))
    _lib(prec).gdn_ref_sigmoid(_p(b), _p(out), b.size)
    return out


def conv1d_silu_seq(qkv, w, conv_state, slots=None, pool=None, apply_silu=True, prec="f64"):
    """qkv [N][T][C], w [C][K], conv_state [pool][C][K-1] (updated in place).

    Returns (out [N][T][C], skipped). Rows of skipped sequences stay zero."""
    qkv, w = _in(qkv, prec), _in(w, prec)
    _inout(conv_state, prec)
    N, T, C = qkv.shape
    K = w.shape[1]
    pool = conv_state.shape[0] if pool is None else pool
    out = np.zeros(qkv.shape, dtype=_dt(prec))
    s, sp = _slots(slots)
    skipped = _lib(prec).gdn_ref_conv1d_silu_seq(_p(qkv), _p(w), _p(conv_state), _p(out), N, T,
                                                 C, K, sp, pool, 1 if apply_silu else 0)
    return out, skipped


def l2norm(x, eps, prec="f64"):
    """Row-wise x / max(||x||, eps) over the last axis."""
    x = _in(x, prec)
    out = np.zeros(x.shape, dtype=_dt(prec))
    dim = x.shape[-1]
    _lib(prec).gdn_ref_l2norm(_p(x), _p(out), x.size // dim, dim, eps)
    return out


def recurrence(state, q, k, v, g, beta, scale, slots=None, pool=None, prec="f64"):
    """state [pool][H][S][S] in place; q,k [N][T][Hk][S]; v [N][T][H][S]; g,beta [N][T][H].

    Returns (y [N][T][H][S], skipped)."""
    _inout(state, prec)
    q, k, v, g, beta = (_in(a, prec) for a in (q, k, v, g, beta))
    N, T, Hk, S = q.shape
    H = v.shape[2]
    pool = state.shape[0] if pool is None else pool
    y = np.zeros(v.shape, dtype=_dt(prec))
    s, sp = _slots(slots)
    skipped = _lib(prec).gdn_ref_recurrence(_p(state), _p(q), _p(k), _p(v), _p(g), _p(beta),
                                            _p(y), N, T, Hk, H, S, scale, sp, pool)
    return y, skipped


def gated_norm(y, w, z, eps, prec="f64"):
    """Row-wise gated RMSNorm over the last axis; w is shared by every row."""
    y, w, z = _in(y, prec), _in(w, prec), _in(z, prec)
    D = y.shape[-1]
    out = np.zeros(y.shape, dtype=_dt(prec))
    _lib(prec).gdn_ref_gated_norm(_p(y), _p(w), _p(z), _p(out), y.size // D, D, eps)
    return out


def block_decode(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, n_k_heads,
                 scale, l2_eps, norm_eps, slots=None, pool=None, prec="f64"):
    """qkv [N][C] raw, conv_state [pool][C][K-1] and state [pool][H][S][S] in place,
    alpha,b [N][H], dt,a [H], z [N][H][S], norm_w [S]. Returns (out [N][H][S], skipped)."""
    qkv, conv_w, alpha, b, dt, a, z, norm_w = (
        _in(x, prec) for x in (qkv, conv_w, alpha, b, dt, a, z, norm_w))
    _inout(conv_state, prec)
    _inout(state, prec)
    N = qkv.shape[0]
    H, S = state.shape[1], state.shape[2]
    K = conv_w.shape[1]
    pool = state.shape[0] if pool is None else pool
    out = np.zeros((N, H, S), dtype=_dt(prec))
    s, sp = _slots(slots)
    skipped = _lib(prec).gdn_ref_block_decode(
        _p(qkv), _p(conv_w), _p(conv_state), _p(alpha), _p(b), _p(dt), _p(a), _p(z),
        _p(norm_w), _p(state), _p(out), N, n_k_heads, H, S, K, scale, l2_eps, norm_eps, sp,
        pool)
    return out, skipped
