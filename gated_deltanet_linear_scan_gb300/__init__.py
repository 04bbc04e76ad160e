"""Python binding of the GB300 gated delta-rule SSM library (libgdn.so).

Argument marshalling only: every function passes tensor data pointers, sizes and
the current CUDA stream to the C ABI of include/gdn.h, checks the returned
status and raises GdnError on failure. All arithmetic runs in the library's
sm_103a kernels; there is no fallback. If libgdn.so has not been built, the
first call raises (``build_if_needed()`` builds it with nvcc).

Tensors are torch CUDA tensors (float32, or int32 for slot ids), contiguous,
with the layouts documented in include/gdn.h.
"""
import ctypes
import os

from . import _build

__all__ = [
    "GdnError", "build_if_needed", "library", "lib_path",
    "gdn_status_str", "gdn_version", "gdn_device_error",
    "gdn_decay_gate", "gdn_beta_sigmoid", "gdn_conv1d_silu", "gdn_conv1d_silu_seq",
    "gdn_qkv_split_norm", "gdn_recurrence_decode", "gdn_recurrence_scan", "gdn_gated_norm",
    "gdn_block_decode", "gdn_recurrence_decode_2pass", "gdn_recurrence_scan_snapshots",
    "gdn_conv1d_silu_seq_snapshots", "gdn_snapshot_restore",
    "gdn_block_prefill_workspace_size", "gdn_block_prefill", "gdn_block_prefill_snapshots",
    "gdn_block_prefill_noalloc", "PREFILL_NOALLOC_SCRATCH_BYTES",
    "gdn_recurrence_scan_chunked", "gdn_block_prefill_chunked",
    "gdn_recurrence_scan_chunked_ws_size", "gdn_recurrence_scan_chunked_ws",
    "gdn_chunked_snapshot_count", "gdn_recurrence_scan_chunked_snapshots",
    "gdn_chunked_prepare", "gdn_chunked_advance", "gdn_block_prefill_chunked_workspace_size",
    "gdn_recurrence_scan_varlen", "gdn_recurrence_scan_chunked_varlen_ws_size",
    "gdn_recurrence_scan_chunked_varlen", "gdn_recurrence_scan_chunked_snapshots_varlen",
    "gdn_block_prefill_varlen_workspace_size",
    "gdn_block_prefill_chunked_varlen_workspace_size", "gdn_block_prefill_varlen",
    "gdn_block_prefill_chunked_varlen", "gdn_block_prefill_snapshots_varlen",
    "gdn_snapshot_restore_varlen", "gdn_selftest_bounded_wait",
]

STATUS = {0: "GDN_OK", 1: "GDN_ERR_NULL", 2: "GDN_ERR_SHAPE", 3: "GDN_ERR_UNSUPPORTED",
          4: "GDN_ERR_ALIGN", 5: "GDN_ERR_LAUNCH", 6: "GDN_ERR_DEVICE"}


class GdnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


_LIB = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float

_SIGS = {
    "gdn_status_str": ([_I], ctypes.c_char_p),
    "gdn_version": ([], _I),
    "gdn_device_error": ([_P], _I),
    "gdn_selftest_bounded_wait": ([ctypes.c_uint, ctypes.c_uint, _P, _P], _I),
    "gdn_decay_gate": ([_P, _P, _P, _P, _I, _I, _P], _I),
    "gdn_beta_sigmoid": ([_P, _P, _I, _P], _I),
    "gdn_conv1d_silu": ([_P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _P], _I),
    "gdn_conv1d_silu_seq": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _P], _I),
    "gdn_qkv_split_norm": ([_P, _P, _P, _P, _I, _I, _I, _I, _F, _P], _I),
    "gdn_recurrence_decode": ([_P] * 7 + [_I, _I, _I, _I, _F, _P, _I, _P, _P], _I),
    "gdn_recurrence_scan": ([_P] * 7 + [_I, _I, _I, _I, _I, _F, _P, _I, _P, _P], _I),
    "gdn_gated_norm": ([_P, _P, _P, _P, _I, _I, _F, _P], _I),
    "gdn_block_decode": ([_P] * 11 + [_I, _I, _I, _I, _I, _F, _F, _F, _P, _I, _P, _P], _I),
    "gdn_recurrence_decode_2pass": ([_P] * 7 + [_I, _I, _I, _I, _F, _P, _I, _P, _P], _I),
    "gdn_recurrence_scan_snapshots": ([_P] * 8 + [_I, _I, _I, _I, _I, _F, _P, _I, _P, _P], _I),
    "gdn_conv1d_silu_seq_snapshots": ([_P] * 5 + [_I, _I, _I, _I, _P, _I, _P, _P], _I),
    "gdn_snapshot_restore": ([_P] * 5 + [_I] * 6 + [_P, _I, _P, _P], _I),
    "gdn_block_prefill_workspace_size": ([_I, _I, _I, _I, _I], ctypes.c_size_t),
    "gdn_block_prefill": ([_P] * 11 + [_I, _I, _I, _I, _I, _I, _F, _F, _F, _P, _I, _P, _P,
                                       ctypes.c_size_t, _P], _I),
    "gdn_block_prefill_noalloc": ([_P] * 11 + [_I, _I, _I, _I, _I, _I, _F, _F, _F, _P, _I, _P,
                                               _P], _I),
    "gdn_block_prefill_snapshots": ([_P] * 13 + [_I, _I, _I, _I, _I, _I, _F, _F, _F, _P, _I, _P,
                                                 _P, ctypes.c_size_t, _P], _I),
    "gdn_recurrence_scan_chunked": ([_P] * 7 + [_I, _I, _I, _I, _I, _F, _P, _I, _P, _P], _I),
    "gdn_recurrence_scan_chunked_ws_size": ([_I, _I, _I, _I], ctypes.c_size_t),
    "gdn_recurrence_scan_chunked_ws": ([_P] * 7 + [_I, _I, _I, _I, _I, _F, _P, _I, _P, _P,
                                                   ctypes.c_size_t, _P], _I),
    "gdn_chunked_snapshot_count": ([_I, _I], _I),
    "gdn_recurrence_scan_chunked_snapshots": ([_P] * 8 + [_I] * 6 + [_F, _P, _I, _P, _P,
                                                                  ctypes.c_size_t, _P], _I),
    "gdn_chunked_prepare": ([_P] * 5 + [_P, ctypes.c_size_t] + [_I] * 7 + [_P], _I),
    "gdn_chunked_advance": ([_P] * 5 + [ctypes.c_size_t, _P] + [_I] * 5 + [_F, _I, _I, _P, _I,
                                                                          _P, _P], _I),
    "gdn_block_prefill_chunked_workspace_size": ([_I, _I, _I, _I, _I], ctypes.c_size_t),
    "gdn_block_prefill_chunked": ([_P] * 11 + [_I, _I, _I, _I, _I, _I, _F, _F, _F, _P, _I, _P, _P,
                                               ctypes.c_size_t, _P], _I),
    "gdn_recurrence_scan_varlen": ([_P] * 8 + [_I] * 6 + [_F, _P, _I, _P, _P], _I),
    "gdn_recurrence_scan_chunked_varlen_ws_size": ([_I, _I, _I, _I], ctypes.c_size_t),
    "gdn_recurrence_scan_chunked_snapshots_varlen": ([_P] * 9 + [_I, _I, _P] + [_I] * 6 +
                                                     [_F, _P, _I, _P, _P, ctypes.c_size_t, _P],
                                                     _I),
    "gdn_recurrence_scan_chunked_varlen": ([_P] * 8 + [_I] * 6 + [_F, _P, _I, _P, _P,
                                                                ctypes.c_size_t, _P], _I),
    "gdn_block_prefill_varlen_workspace_size": ([_I, _I, _I, _I, _I], ctypes.c_size_t),
    "gdn_block_prefill_chunked_varlen_workspace_size": ([_I, _I, _I, _I, _I], ctypes.c_size_t),
    "gdn_block_prefill_varlen": ([_P] * 12 + [_I] * 7 + [_F, _F, _F, _P, _I, _P, _P,
                                                       ctypes.c_size_t, _P], _I),
    "gdn_block_prefill_chunked_varlen": ([_P] * 12 + [_I] * 7 + [_F, _F, _F, _P, _I, _P, _P,
                                                               ctypes.c_size_t, _P], _I),
    "gdn_block_prefill_snapshots_varlen": ([_P] * 14 + [_I] * 7 + [_F, _F, _F, _P, _I, _P, _P,
                                                                 ctypes.c_size_t, _P], _I),
    "gdn_snapshot_restore_varlen": ([_P] * 6 + [_I] * 7 + [_P, _I, _P, _P], _I),
}

# Size of the fixed device scratch of gdn_block_prefill_noalloc (include/gdn.h).
PREFILL_NOALLOC_SCRATCH_BYTES = 32 << 20


def lib_path():
    return _build.LIB


def build_if_needed(force=False):
    """Compile libgdn.so for sm_103a if it is missing or older than its sources."""
    return _build.build(force=force)


def library():
    """The loaded libgdn.so (ctypes.CDLL). Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libgdn.so is not built ({_build.LIB}); run "
                               "gated_deltanet_linear_scan_gb300.build_if_needed()")
        lib = ctypes.CDLL(_build.LIB)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = lib
    return _LIB


# ------------------------------------------------------------------ marshalling helpers

_TORCH = None


def _torch():
    """torch, imported on first use (the package itself imports without it)."""
    global _TORCH
    if _TORCH is None:
        import torch
        _TORCH = torch
    return _TORCH


def _stream(stream):
    """The stream argument of a call: the caller's, else torch's current stream (read
    through the raw-stream accessor when this torch has it: a tenth of the cost of building
    a Stream object, which matters at decode-step rates)."""
    if stream is not None:
        return int(stream)
    torch = _torch()
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _ptr(t, name, dtype=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    want = dtype or torch.float32
    if t.dtype != want:
        raise TypeError(f"{name} must be {want}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _slots(slots):
    return None if slots is None else _ptr(slots, "slots", _torch().int32)


def _errc(err_count):
    return None if err_count is None else _ptr(err_count, "err_count", _torch().int32)


def _ws_check(workspace):
    torch = _torch()
    if not (isinstance(workspace, torch.Tensor) and workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")


def _ws_ptr(workspace):
    _ws_check(workspace)
    return workspace.data_ptr()


def _ws_bytes(workspace):
    return workspace.numel() * workspace.element_size()


def _pool(pool, n_seqs, slots):
    if pool is not None:
        return int(pool)
    if slots is not None:
        raise ValueError("pool (the number of slots the state buffers hold) is required with slots")
    return max(1, int(n_seqs))


def _check(fn, status):
    if status != 0:
        raise GdnError(fn, status)


# ------------------------------------------------------------------ the C ABI

def gdn_status_str(status):
    return library().gdn_status_str(int(status)).decode()


def gdn_version():
    return library().gdn_version()


def gdn_device_error(stream=None):
    """Synchronise the stream; raise GdnError if a kernel's bounded wait gave up."""
    _check("gdn_device_error", library().gdn_device_error(_stream(stream)))


def gdn_selftest_bounded_wait(arm_mask, limit_us, out, stream=None):
    """Enqueue the bounded-wait self-test: probe i (bit i of arm_mask) waits at most
    limit_us for a copy that never comes and raises the device flag; `out` is a CUDA
    float32 tensor of 4 elements (unarmed probes write 1.0 there)."""
    _check("gdn_selftest_bounded_wait", library().gdn_selftest_bounded_wait(
        int(arm_mask), int(limit_us), _ptr(out, "out"), _stream(stream)))


def gdn_decay_gate(alpha, dt, a, g, n_heads, rows, stream=None):
    _check("gdn_decay_gate", library().gdn_decay_gate(
        _ptr(alpha, "alpha"), _ptr(dt, "dt"), _ptr(a, "a"), _ptr(g, "g"), n_heads, rows,
        _stream(stream)))


def gdn_beta_sigmoid(b, beta, n, stream=None):
    _check("gdn_beta_sigmoid", library().gdn_beta_sigmoid(_ptr(b, "b"), _ptr(beta, "beta"), n,
                                                         _stream(stream)))


def gdn_conv1d_silu(qkv, w, conv_state, out, n_seqs, conv_dim, conv_kernel, slots=None,
                    pool=None, err_count=None, stream=None):
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_conv1d_silu", library().gdn_conv1d_silu(
        _ptr(qkv, "qkv"), _ptr(w, "w"), _ptr(conv_state, "conv_state"), _ptr(out, "out"),
        n_seqs, conv_dim, conv_kernel, _slots(slots), pool, _errc(err_count), _stream(stream)))


def gdn_conv1d_silu_seq(qkv, w, conv_state, out, n_seqs, n_tokens, conv_dim, conv_kernel,
                        slots=None, pool=None, err_count=None, stream=None):
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_conv1d_silu_seq", library().gdn_conv1d_silu_seq(
        _ptr(qkv, "qkv"), _ptr(w, "w"), _ptr(conv_state, "conv_state"), _ptr(out, "out"),
        n_seqs, n_tokens, conv_dim, conv_kernel, _slots(slots), pool, _errc(err_count),
        _stream(stream)))


def gdn_qkv_split_norm(conv_out, q, k, v, rows, n_k_heads, n_v_heads, state_size, eps,
                       stream=None):
    _check("gdn_qkv_split_norm", library().gdn_qkv_split_norm(
        _ptr(conv_out, "conv_out"), _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), rows, n_k_heads,
        n_v_heads, state_size, eps, _stream(stream)))


def gdn_recurrence_decode(state, q, k, v, g, beta, y, n_seqs, n_k_heads, n_v_heads, state_size,
                          scale, slots=None, pool=None, err_count=None, stream=None):
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_recurrence_decode", library().gdn_recurrence_decode(
        _ptr(state, "state"), _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g"),
        _ptr(beta, "beta"), _ptr(y, "y"), n_seqs, n_k_heads, n_v_heads, state_size, scale,
        _slots(slots), pool, _errc(err_count), _stream(stream)))


def gdn_recurrence_scan(state, q, k, v, g, beta, y, n_seqs, n_tokens, n_k_heads, n_v_heads,
                        state_size, scale, slots=None, pool=None, err_count=None, stream=None):
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_recurrence_scan", library().gdn_recurrence_scan(
        _ptr(state, "state"), _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g"),
        _ptr(beta, "beta"), _ptr(y, "y"), n_seqs, n_tokens, n_k_heads, n_v_heads, state_size,
        scale, _slots(slots), pool, _errc(err_count), _stream(stream)))


def gdn_recurrence_scan_chunked(state, q, k, v, g, beta, y, n_seqs, n_tokens, n_k_heads,
                                n_v_heads, state_size, scale, slots=None, pool=None,
                                err_count=None, stream=None):
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_recurrence_scan_chunked", library().gdn_recurrence_scan_chunked(
        _ptr(state, "state"), _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g"),
        _ptr(beta, "beta"), _ptr(y, "y"), n_seqs, n_tokens, n_k_heads, n_v_heads, state_size,
        scale, _slots(slots), pool, _errc(err_count), _stream(stream)))


def gdn_recurrence_scan_chunked_ws_size(n_seqs, n_tokens, n_v_heads, state_size):
    return library().gdn_recurrence_scan_chunked_ws_size(n_seqs, n_tokens, n_v_heads, state_size)


def gdn_recurrence_scan_chunked_ws(state, q, k, v, g, beta, y, n_seqs, n_tokens, n_k_heads,
                                   n_v_heads, state_size, scale, workspace, slots=None, pool=None,
                                   err_count=None, stream=None):
    """The two-phase chunked scan; `workspace` is a CUDA tensor (any dtype, contiguous)
    whose byte size sets how many chunks each wave prepares."""
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_recurrence_scan_chunked_ws", library().gdn_recurrence_scan_chunked_ws(
        _ptr(state, "state"), _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g"),
        _ptr(beta, "beta"), _ptr(y, "y"), n_seqs, n_tokens, n_k_heads, n_v_heads, state_size,
        scale, _slots(slots), pool, _errc(err_count), _ws_ptr(workspace),
        _ws_bytes(workspace), _stream(stream)))


def gdn_chunked_snapshot_count(n_tokens, snap_every):
    return library().gdn_chunked_snapshot_count(n_tokens, snap_every)


def gdn_recurrence_scan_chunked_snapshots(state, q, k, v, g, beta, y, snaps, snap_every, n_seqs,
                                          n_tokens, n_k_heads, n_v_heads, state_size, scale,
                                          workspace, slots=None, pool=None, err_count=None,
                                          stream=None):
    """The two-phase chunked scan, also writing the state every 32 * snap_every positions
    into snaps [n_seqs][n_snaps][H][S][S]; snaps may be None when n_snaps is 0."""
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_recurrence_scan_chunked_snapshots",
           library().gdn_recurrence_scan_chunked_snapshots(
               _ptr(state, "state"), _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g"),
               _ptr(beta, "beta"), _ptr(y, "y"), _ptr(snaps, "snaps", optional=True),
               snap_every, n_seqs, n_tokens, n_k_heads, n_v_heads, state_size, scale,
               _slots(slots), pool, _errc(err_count), _ws_ptr(workspace), _ws_bytes(workspace),
               _stream(stream)))


def gdn_chunked_prepare(q, k, v, g, beta, workspace, n_seqs, n_tokens, n_k_heads, n_v_heads,
                        state_size, chunk_begin, n_chunks, stream=None):
    """Phase 1 of the two-phase chunked scan over chunks chunk_begin .. + n_chunks - 1."""
    _check("gdn_chunked_prepare", library().gdn_chunked_prepare(
        _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g"), _ptr(beta, "beta"),
        _ws_ptr(workspace), _ws_bytes(workspace), n_seqs, n_tokens, n_k_heads, n_v_heads,
        state_size, chunk_begin, n_chunks, _stream(stream)))


def gdn_chunked_advance(state, q, k, g, workspace, y, n_seqs, n_tokens, n_k_heads, n_v_heads,
                        state_size, scale, chunk_begin, n_chunks, slots=None, pool=None,
                        err_count=None, stream=None):
    """Phase 2: advance the state over the prepared chunks, writing their y."""
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_chunked_advance", library().gdn_chunked_advance(
        _ptr(state, "state"), _ptr(q, "q"), _ptr(k, "k"), _ptr(g, "g"), _ws_ptr(workspace),
        _ws_bytes(workspace), _ptr(y, "y"), n_seqs, n_tokens, n_k_heads, n_v_heads, state_size,
        scale, chunk_begin, n_chunks, _slots(slots), pool, _errc(err_count), _stream(stream)))


def gdn_gated_norm(y, w, z, out, rows, head_dim, eps, stream=None):
    _check("gdn_gated_norm", library().gdn_gated_norm(
        _ptr(y, "y"), _ptr(w, "w"), _ptr(z, "z"), _ptr(out, "out"), rows, head_dim, eps,
        _stream(stream)))


def gdn_block_decode(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out, n_seqs,
                     n_k_heads, n_v_heads, state_size, conv_kernel, scale, l2_eps, norm_eps,
                     slots=None, pool=None, err_count=None, stream=None):
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_block_decode", library().gdn_block_decode(
        _ptr(qkv, "qkv"), _ptr(conv_w, "conv_w"), _ptr(conv_state, "conv_state"),
        _ptr(alpha, "alpha"), _ptr(b, "b"), _ptr(dt, "dt"), _ptr(a, "a"), _ptr(z, "z"),
        _ptr(norm_w, "norm_w"), _ptr(state, "state"), _ptr(out, "out"), n_seqs, n_k_heads,
        n_v_heads, state_size, conv_kernel, scale, l2_eps, norm_eps, _slots(slots), pool,
        _errc(err_count), _stream(stream)))


def gdn_recurrence_decode_2pass(state, q, k, v, g, beta, y, n_seqs, n_k_heads, n_v_heads,
                                state_size, scale, slots=None, pool=None, err_count=None,
                                stream=None):
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_recurrence_decode_2pass", library().gdn_recurrence_decode_2pass(
        _ptr(state, "state"), _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g"),
        _ptr(beta, "beta"), _ptr(y, "y"), n_seqs, n_k_heads, n_v_heads, state_size, scale,
        _slots(slots), pool, _errc(err_count), _stream(stream)))


def gdn_recurrence_scan_snapshots(state, q, k, v, g, beta, y, snaps, n_seqs, n_tokens,
                                  n_k_heads, n_v_heads, state_size, scale, slots=None, pool=None,
                                  err_count=None, stream=None):
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_recurrence_scan_snapshots", library().gdn_recurrence_scan_snapshots(
        _ptr(state, "state"), _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g"),
        _ptr(beta, "beta"), _ptr(y, "y"), _ptr(snaps, "snaps"), n_seqs, n_tokens, n_k_heads,
        n_v_heads, state_size, scale, _slots(slots), pool, _errc(err_count), _stream(stream)))


def gdn_conv1d_silu_seq_snapshots(qkv, w, conv_state, out, snaps, n_seqs, n_tokens, conv_dim,
                                  conv_kernel, slots=None, pool=None, err_count=None,
                                  stream=None):
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_conv1d_silu_seq_snapshots", library().gdn_conv1d_silu_seq_snapshots(
        _ptr(qkv, "qkv"), _ptr(w, "w"), _ptr(conv_state, "conv_state"), _ptr(out, "out"),
        _ptr(snaps, "snaps"), n_seqs, n_tokens, conv_dim, conv_kernel, _slots(slots), pool,
        _errc(err_count), _stream(stream)))


def gdn_snapshot_restore(state, snaps, accepted, n_seqs, n_tokens, n_v_heads, state_size,
                         conv_state=None, conv_snaps=None, conv_dim=0, conv_kernel=0,
                         slots=None, pool=None, err_count=None, stream=None):
    """Roll each sequence back to the snapshot after its accepted[n]-th position (int32
    CUDA tensor of n_seqs counts in [1, n_tokens]); the conv history too when conv_state
    and conv_snaps are given."""
    import torch
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_snapshot_restore", library().gdn_snapshot_restore(
        _ptr(state, "state"), _ptr(snaps, "snaps"), _ptr(conv_state, "conv_state", optional=True),
        _ptr(conv_snaps, "conv_snaps", optional=True), _ptr(accepted, "accepted", torch.int32),
        n_seqs, n_tokens, n_v_heads, state_size, conv_dim, conv_kernel, _slots(slots), pool,
        _errc(err_count), _stream(stream)))


def gdn_block_prefill_workspace_size(n_seqs, n_tokens, n_k_heads, n_v_heads, state_size):
    return library().gdn_block_prefill_workspace_size(n_seqs, n_tokens, n_k_heads, n_v_heads,
                                                      state_size)


def gdn_block_prefill_chunked_workspace_size(n_seqs, n_tokens, n_k_heads, n_v_heads, state_size):
    return library().gdn_block_prefill_chunked_workspace_size(n_seqs, n_tokens, n_k_heads,
                                                              n_v_heads, state_size)


def _block_prefill(name, qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out, n_seqs,
                   n_tokens, n_k_heads, n_v_heads, state_size, conv_kernel, scale, l2_eps,
                   norm_eps, workspace, slots, pool, err_count, stream):
    pool = _pool(pool, n_seqs, slots)
    _ws_check(workspace)
    _check(name, getattr(library(), name)(
        _ptr(qkv, "qkv"), _ptr(conv_w, "conv_w"), _ptr(conv_state, "conv_state"),
        _ptr(alpha, "alpha"), _ptr(b, "b"), _ptr(dt, "dt"), _ptr(a, "a"), _ptr(z, "z"),
        _ptr(norm_w, "norm_w"), _ptr(state, "state"), _ptr(out, "out"), n_seqs, n_tokens,
        n_k_heads, n_v_heads, state_size, conv_kernel, scale, l2_eps, norm_eps, _slots(slots),
        pool, _errc(err_count), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def gdn_block_prefill(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out, n_seqs,
                      n_tokens, n_k_heads, n_v_heads, state_size, conv_kernel, scale, l2_eps,
                      norm_eps, workspace, slots=None, pool=None, err_count=None, stream=None):
    """`workspace`: a CUDA tensor of at least gdn_block_prefill_workspace_size() bytes."""
    _block_prefill("gdn_block_prefill", qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w,
                   state, out, n_seqs, n_tokens, n_k_heads, n_v_heads, state_size, conv_kernel,
                   scale, l2_eps, norm_eps, workspace, slots, pool, err_count, stream)


def gdn_block_prefill_snapshots(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out,
                                snaps, conv_snaps, n_seqs, n_tokens, n_k_heads, n_v_heads,
                                state_size, conv_kernel, scale, l2_eps, norm_eps, workspace,
                                slots=None, pool=None, err_count=None, stream=None):
    """gdn_block_prefill keeping the state and the conv history after every position
    (snaps [n][t][H][S][S], conv_snaps [n][t][C][K-1]) for speculative-decoding rollback."""
    pool = _pool(pool, n_seqs, slots)
    _ws_check(workspace)
    _check("gdn_block_prefill_snapshots", library().gdn_block_prefill_snapshots(
        _ptr(qkv, "qkv"), _ptr(conv_w, "conv_w"), _ptr(conv_state, "conv_state"),
        _ptr(alpha, "alpha"), _ptr(b, "b"), _ptr(dt, "dt"), _ptr(a, "a"), _ptr(z, "z"),
        _ptr(norm_w, "norm_w"), _ptr(state, "state"), _ptr(out, "out"), _ptr(snaps, "snaps"),
        _ptr(conv_snaps, "conv_snaps"), n_seqs, n_tokens, n_k_heads, n_v_heads, state_size,
        conv_kernel, scale, l2_eps, norm_eps, _slots(slots), pool, _errc(err_count),
        _ws_ptr(workspace), _ws_bytes(workspace), _stream(stream)))


def gdn_block_prefill_chunked(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out,
                              n_seqs, n_tokens, n_k_heads, n_v_heads, state_size, conv_kernel,
                              scale, l2_eps, norm_eps, workspace, slots=None, pool=None,
                              err_count=None, stream=None):
    """gdn_block_prefill with the chunked tensor-core scan (state_size 128)."""
    _block_prefill("gdn_block_prefill_chunked", qkv, conv_w, conv_state, alpha, b, dt, a, z,
                   norm_w, state, out, n_seqs, n_tokens, n_k_heads, n_v_heads, state_size,
                   conv_kernel, scale, l2_eps, norm_eps, workspace, slots, pool, err_count,
                   stream)


def gdn_block_prefill_noalloc(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out,
                              n_seqs, n_tokens, n_k_heads, n_v_heads, state_size, conv_kernel,
                              scale, l2_eps, norm_eps, slots=None, pool=None, err_count=None,
                              stream=None):
    """gdn_block_prefill working in the library's fixed device scratch instead of a
    caller workspace, for callers that cannot allocate device memory."""
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_block_prefill_noalloc", library().gdn_block_prefill_noalloc(
        _ptr(qkv, "qkv"), _ptr(conv_w, "conv_w"), _ptr(conv_state, "conv_state"),
        _ptr(alpha, "alpha"), _ptr(b, "b"), _ptr(dt, "dt"), _ptr(a, "a"), _ptr(z, "z"),
        _ptr(norm_w, "norm_w"), _ptr(state, "state"), _ptr(out, "out"), n_seqs, n_tokens,
        n_k_heads, n_v_heads, state_size, conv_kernel, scale, l2_eps, norm_eps, _slots(slots),
        pool, _errc(err_count), _stream(stream)))


# ------------------------------------------------------------------ ragged batches
# Sequences of different lengths packed token-major ([total_tokens][...] arrays);
# `cu_seqlens` is an int32 CUDA tensor of n_seqs + 1 offsets (sequence n owns positions
# cu_seqlens[n] .. cu_seqlens[n+1] - 1), `max_tokens` an upper bound on one length.

def _cu(cu_seqlens):
    import torch
    return _ptr(cu_seqlens, "cu_seqlens", torch.int32)


def gdn_recurrence_scan_varlen(state, q, k, v, g, beta, y, cu_seqlens, n_seqs, total_tokens,
                               max_tokens, n_k_heads, n_v_heads, state_size, scale, slots=None,
                               pool=None, err_count=None, stream=None):
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_recurrence_scan_varlen", library().gdn_recurrence_scan_varlen(
        _ptr(state, "state"), _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g"),
        _ptr(beta, "beta"), _ptr(y, "y"), _cu(cu_seqlens), n_seqs, total_tokens, max_tokens,
        n_k_heads, n_v_heads, state_size, scale, _slots(slots), pool, _errc(err_count),
        _stream(stream)))


def gdn_recurrence_scan_chunked_varlen_ws_size(n_seqs, total_tokens, n_v_heads, state_size):
    return library().gdn_recurrence_scan_chunked_varlen_ws_size(n_seqs, total_tokens, n_v_heads,
                                                                state_size)


def gdn_recurrence_scan_chunked_varlen(state, q, k, v, g, beta, y, cu_seqlens, n_seqs,
                                       total_tokens, max_tokens, n_k_heads, n_v_heads,
                                       state_size, scale, workspace=None, slots=None, pool=None,
                                       err_count=None, stream=None):
    """`workspace` None: the one-kernel form; a CUDA tensor of at least
    gdn_recurrence_scan_chunked_varlen_ws_size() bytes: the two-phase form."""
    pool = _pool(pool, n_seqs, slots)
    ws, nbytes = (None, 0) if workspace is None else (_ws_ptr(workspace), _ws_bytes(workspace))
    _check("gdn_recurrence_scan_chunked_varlen", library().gdn_recurrence_scan_chunked_varlen(
        _ptr(state, "state"), _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g"),
        _ptr(beta, "beta"), _ptr(y, "y"), _cu(cu_seqlens), n_seqs, total_tokens, max_tokens,
        n_k_heads, n_v_heads, state_size, scale, _slots(slots), pool, _errc(err_count), ws,
        nbytes, _stream(stream)))


def gdn_recurrence_scan_chunked_snapshots_varlen(state, q, k, v, g, beta, y, snaps, snap_base,
                                                 snap_pool, snap_every, cu_seqlens, n_seqs,
                                                 total_tokens, max_tokens, n_k_heads, n_v_heads,
                                                 state_size, scale, workspace, slots=None,
                                                 pool=None, err_count=None, stream=None):
    """The ragged chunked scan keeping snapshots: sequence n's snapshot j in slot
    snap_base[n] + j of `snaps` ([snap_pool][H][S][S]); snaps and snap_base may be None
    when no sequence can reach a snapshot."""
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_recurrence_scan_chunked_snapshots_varlen",
           library().gdn_recurrence_scan_chunked_snapshots_varlen(
               _ptr(state, "state"), _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g"),
               _ptr(beta, "beta"), _ptr(y, "y"), _ptr(snaps, "snaps", optional=True),
               _ptr(snap_base, "snap_base", _torch().int32, optional=True), snap_pool,
               snap_every, _cu(cu_seqlens), n_seqs, total_tokens, max_tokens, n_k_heads,
               n_v_heads, state_size, scale, _slots(slots), pool, _errc(err_count),
               _ws_ptr(workspace), _ws_bytes(workspace), _stream(stream)))


def gdn_block_prefill_varlen_workspace_size(n_seqs, total_tokens, n_k_heads, n_v_heads,
                                            state_size):
    return library().gdn_block_prefill_varlen_workspace_size(n_seqs, total_tokens, n_k_heads,
                                                             n_v_heads, state_size)


def gdn_block_prefill_chunked_varlen_workspace_size(n_seqs, total_tokens, n_k_heads, n_v_heads,
                                                    state_size):
    return library().gdn_block_prefill_chunked_varlen_workspace_size(
        n_seqs, total_tokens, n_k_heads, n_v_heads, state_size)


def _block_prefill_varlen(name, qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out,
                          extra, cu_seqlens, n_seqs, total_tokens, max_tokens, n_k_heads,
                          n_v_heads, state_size, conv_kernel, scale, l2_eps, norm_eps, workspace,
                          slots, pool, err_count, stream):
    pool = _pool(pool, n_seqs, slots)
    _ws_check(workspace)
    _check(name, getattr(library(), name)(
        _ptr(qkv, "qkv"), _ptr(conv_w, "conv_w"), _ptr(conv_state, "conv_state"),
        _ptr(alpha, "alpha"), _ptr(b, "b"), _ptr(dt, "dt"), _ptr(a, "a"), _ptr(z, "z"),
        _ptr(norm_w, "norm_w"), _ptr(state, "state"), _ptr(out, "out"), *extra,
        _cu(cu_seqlens), n_seqs, total_tokens, max_tokens, n_k_heads, n_v_heads, state_size,
        conv_kernel, scale, l2_eps, norm_eps, _slots(slots), pool, _errc(err_count),
        _ws_ptr(workspace), _ws_bytes(workspace), _stream(stream)))


def gdn_block_prefill_varlen(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out,
                             cu_seqlens, n_seqs, total_tokens, max_tokens, n_k_heads, n_v_heads,
                             state_size, conv_kernel, scale, l2_eps, norm_eps, workspace,
                             slots=None, pool=None, err_count=None, stream=None):
    """gdn_block_prefill over a ragged batch; `workspace` of at least
    gdn_block_prefill_varlen_workspace_size() bytes."""
    _block_prefill_varlen("gdn_block_prefill_varlen", qkv, conv_w, conv_state, alpha, b, dt, a,
                          z, norm_w, state, out, (), cu_seqlens, n_seqs, total_tokens,
                          max_tokens, n_k_heads, n_v_heads, state_size, conv_kernel, scale,
                          l2_eps, norm_eps, workspace, slots, pool, err_count, stream)


def gdn_block_prefill_chunked_varlen(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state,
                                     out, cu_seqlens, n_seqs, total_tokens, max_tokens,
                                     n_k_heads, n_v_heads, state_size, conv_kernel, scale, l2_eps,
                                     norm_eps, workspace, slots=None, pool=None, err_count=None,
                                     stream=None):
    """gdn_block_prefill_chunked over a ragged batch (state_size 128)."""
    _block_prefill_varlen("gdn_block_prefill_chunked_varlen", qkv, conv_w, conv_state, alpha, b,
                          dt, a, z, norm_w, state, out, (), cu_seqlens, n_seqs, total_tokens,
                          max_tokens, n_k_heads, n_v_heads, state_size, conv_kernel, scale,
                          l2_eps, norm_eps, workspace, slots, pool, err_count, stream)


def gdn_block_prefill_snapshots_varlen(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state,
                                       out, snaps, conv_snaps, cu_seqlens, n_seqs, total_tokens,
                                       max_tokens, n_k_heads, n_v_heads, state_size, conv_kernel,
                                       scale, l2_eps, norm_eps, workspace, slots=None, pool=None,
                                       err_count=None, stream=None):
    """gdn_block_prefill_snapshots over a ragged batch: snaps [total][H][S][S], conv_snaps
    [total][C][K-1], packed as the positions are."""
    _block_prefill_varlen("gdn_block_prefill_snapshots_varlen", qkv, conv_w, conv_state, alpha,
                          b, dt, a, z, norm_w, state, out,
                          (_ptr(snaps, "snaps"), _ptr(conv_snaps, "conv_snaps")), cu_seqlens,
                          n_seqs, total_tokens, max_tokens, n_k_heads, n_v_heads, state_size,
                          conv_kernel, scale, l2_eps, norm_eps, workspace, slots, pool,
                          err_count, stream)


def gdn_snapshot_restore_varlen(state, snaps, accepted, cu_seqlens, n_seqs, total_tokens,
                                max_tokens, n_v_heads, state_size, conv_state=None,
                                conv_snaps=None, conv_dim=0, conv_kernel=0, slots=None,
                                pool=None, err_count=None, stream=None):
    """Roll each sequence of a ragged batch back to the snapshot after its accepted[n]-th
    position (snapshots packed as the positions are)."""
    import torch
    pool = _pool(pool, n_seqs, slots)
    _check("gdn_snapshot_restore_varlen", library().gdn_snapshot_restore_varlen(
        _ptr(state, "state"), _ptr(snaps, "snaps"), _ptr(conv_state, "conv_state", optional=True),
        _ptr(conv_snaps, "conv_snaps", optional=True), _ptr(accepted, "accepted", torch.int32),
        _cu(cu_seqlens), n_seqs, total_tokens, max_tokens, n_v_heads, state_size, conv_dim,
        conv_kernel, _slots(slots), pool, _errc(err_count), _stream(stream)))
