"""Python binding of libra (blockwise exact attention, ring-emulated, sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/ra.h.  PyTorch supplies device
memory and streams.  The compiled library is loaded on first use (the first
call, or the first access to ``lib``), so that importing the package for its
seeded input generators maps no product code; if the library is missing that
first use raises ImportError.  There is no other implementation to fall back
to.

Functions with the C names (``ra_block_fwd``, ``ra_merge``, ``ra_ring_fwd``,
``ra_ring_bwd``, ...) take torch tensors in the [B, N, H, d] layout and raise
``RAError`` on a non-OK status.  ``ring_attention_fwd`` / ``ring_attention_bwd``
additionally allocate outputs and workspace with torch.
"""
import ctypes
import os
import threading

import torch

__all__ = [
    "RAError", "RaShape", "lib", "shape_of", "empty_like_layout",
    "ra_acc_init", "ra_block_fwd", "ra_block_fwd_workspace_bytes", "ra_merge", "ra_finalize",
    "ra_ring_fwd", "ra_ring_fwd_workspace_bytes", "ra_ring_bwd", "ra_ring_bwd_workspace_bytes",
    "ra_ring_fwd_noalloc", "ra_ring_fwd_varlen", "ra_ring_bwd_varlen", "ra_ring_step_host",
    "ra_ring_step_host_workspace_bytes", "ra_ffn_workspace_bytes", "ra_ffn_fwd", "ra_ffn_bwd",
    "ra_sync_status", "ra_last_error", "ra_launch_count", "ra_selftest_timeout", "ra_debug_visit_log",
    "ra_kernel_timing", "ra_kernel_timing_read",
    "ring_attention_fwd", "ring_attention_bwd", "RA_F32", "RA_BF16", "RA_F16",
    "RA_CAUSAL", "RA_PRECISE", "RA_STRIPED",
]

RA_F32, RA_BF16, RA_F16 = 0, 1, 2
RA_CAUSAL, RA_PRECISE, RA_STRIPED = 1, 2, 4
STATUS = {0: "RA_OK", 1: "RA_ERR_INVALID_ARG", 2: "RA_ERR_UNSUPPORTED", 3: "RA_ERR_CUDA",
          4: "RA_ERR_RANGE", 5: "RA_ERR_TIMEOUT"}
_DTYPES = {torch.float32: RA_F32, torch.bfloat16: RA_BF16, torch.float16: RA_F16}
_TORCH = {v: k for k, v in _DTYPES.items()}

# RA_LIBRARY may name another build of the same library (e.g. an instrumented one).
_LIBPATH = os.environ.get("RA_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)),
                                                        "libra.so")


class RAError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class RaShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("N_q", ctypes.c_int), ("N_kv", ctypes.c_int),
                ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("d", ctypes.c_int),
                ("q_bstride", ctypes.c_longlong), ("kv_bstride", ctypes.c_longlong),
                ("q_rstride", ctypes.c_longlong), ("q_hstride", ctypes.c_longlong),
                ("kv_rstride", ctypes.c_longlong), ("kv_hstride", ctypes.c_longlong)]


def _load():
    if not os.path.exists(_LIBPATH):
        raise ImportError(
            f"{_LIBPATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(or python blockwise_exact_attention_ra_gb300/build.py)")
    L = ctypes.CDLL(_LIBPATH)
    vp, i, f, ll, sz, sh = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong,
                            ctypes.c_size_t, RaShape)
    sig = {
        "ra_acc_init": (i, [vp, vp, vp, sh, vp]),
        "ra_block_fwd": (i, [vp, vp, vp, i, vp, vp, vp, sh, ll, ll, i, f, vp, sz, vp]),
        "ra_block_fwd_workspace_bytes": (sz, [i, sh]),
        "ra_merge": (i, [vp, vp, vp, vp, vp, vp, sh, vp]),
        "ra_finalize": (i, [vp, vp, vp, vp, i, vp, sh, vp]),
        "ra_ring_fwd": (i, [vp, vp, vp, i, sh, i, i, f, vp, i, vp, vp, sz, vp]),
        "ra_ring_fwd_workspace_bytes": (sz, [i, sh, i]),
        "ra_ring_fwd_noalloc": (i, [vp, vp, vp, i, sh, i, i, f, vp, i, vp, vp]),
        "ra_ring_fwd_varlen": (i, [vp, vp, vp, i, sh, i, vp, i, f, vp, i, vp, vp, sz, vp]),
        "ra_ring_step_host": (i, [vp, vp, vp, vp, i, sh, i, i, f, vp, i, vp, vp, vp, vp, i, vp, sz, vp]),
        "ra_ring_step_host_workspace_bytes": (sz, [i, i, i, sh, i]),
        "ra_ffn_workspace_bytes": (sz, [i, ctypes.c_longlong, i, i, i, i]),
        "ra_ffn_fwd": (i, [vp, vp, vp, i, ctypes.c_longlong, i, i, i, vp, i, vp, sz, vp]),
        "ra_ffn_bwd": (i, [vp, vp, vp, vp, i, ctypes.c_longlong, i, i, i, vp, i, vp, vp, vp, sz, vp]),
        "ra_ring_bwd_varlen": (i, [vp, vp, vp, vp, i, vp, vp, i, sh, i, vp, i, f, vp, vp, vp, i, vp, sz, vp]),
        "ra_ring_bwd": (i, [vp, vp, vp, vp, i, vp, vp, i, sh, i, i, f, vp, vp, vp, i, vp, sz, vp]),
        "ra_ring_bwd_workspace_bytes": (sz, [i, i, sh, i]),
        "ra_sync_status": (i, [vp]),
        "ra_last_error": (ctypes.c_char_p, []),
        "ra_launch_count": (ctypes.c_ulonglong, []),
        "ra_debug_visit_log": (i, [vp, sz, vp]),
        "ra_selftest_timeout": (i, [ctypes.c_uint, vp]),
        "ra_kernel_timing": (i, [i]),
        "ra_kernel_timing_read": (i, [i, ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(ctypes.c_ulonglong)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


_LIB = None
_LIB_LOCK = threading.Lock()


def _lib():
    """The loaded library (loaded on the first call)."""
    global _LIB
    if _LIB is None:
        with _LIB_LOCK:
            if _LIB is None:
                _LIB = _load()
    return _LIB


def __getattr__(name):
    if name == "lib":
        return _lib()
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")


def ra_last_error():
    return _lib().ra_last_error().decode()


def ra_launch_count():
    return int(_lib().ra_launch_count())


def _check(code):
    if code != 0:
        raise RAError(code, ra_last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dt(t):
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise RAError(1, f"unsupported dtype {t.dtype}") from None


def _bstride(t):
    return t.stride(0)


def _strides(t):
    """(batch, row, head) strides of a [B, N, H, d] tensor; an axis of extent
    1 passes 0 (the library's default), since torch leaves its stride free."""
    return tuple(t.stride(i) if t.shape[i] > 1 else 0 for i in range(3))


def _check_layout(t, name):
    """Tensors are [B, N, H, d] with d contiguous; batch, row and head strides
    are passed to the library, which checks them."""
    if t.dim() != 4:
        raise RAError(1, f"{name} must be [B, N, H, d]")
    if t.stride(3) != 1 and t.shape[3] > 1:
        raise RAError(1, f"{name} must have a contiguous last (head) dimension (strides {t.stride()})")


def _same_layout(t, ref, name, ref_name):
    """o, dO, dq share q's layout and v, dk, dv share k's: the library takes one
    set of strides per group."""
    if t is None:
        return
    _check_layout(t, name)
    if tuple(t.shape) != tuple(ref.shape) or _strides(t) != _strides(ref):
        raise RAError(1, f"{name} must have the shape and strides of {ref_name} "
                         f"({tuple(t.shape)} {t.stride()} vs {tuple(ref.shape)} {ref.stride()})")


def shape_of(q, k):
    """RaShape for q [B, Nq, Hq, d] and k [B, Nkv, Hkv, d], with the batch,
    row and head strides of the tensors."""
    _check_layout(q, "q")
    _check_layout(k, "k")
    B, Nq, Hq, d = q.shape
    _, Nkv, Hkv, _ = k.shape
    qb, qr, qh = _strides(q)
    kb, kr, kh = _strides(k)
    return RaShape(B, Nq, Nkv, Hq, Hkv, d, qb, kb, qr, qh, kr, kh)


def empty_like_layout(t, dtype=None):
    """A new tensor with t's shape and strides (outputs of a group must share
    its layout)."""
    return torch.empty_strided(tuple(t.shape), t.stride(), dtype=dtype or t.dtype, device=t.device)


RA_KERNEL_FWD_TC, RA_KERNEL_BWD_TC, RA_KERNEL_FWD_F32, RA_KERNEL_BWD_F32, RA_KERNEL_GEMM_TC = 0, 1, 2, 3, 4
RA_COPY_H2D, RA_COPY_D2H = 5, 6


def ra_kernel_timing(enable):
    _check(_lib().ra_kernel_timing(int(bool(enable))))


def ra_kernel_timing_read(kernel):
    """(total device ms, launches) of one kernel since timing was enabled."""
    ms = ctypes.c_double()
    n = ctypes.c_ulonglong()
    _check(_lib().ra_kernel_timing_read(int(kernel), ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, int(n.value)


def ra_debug_visit_log(entries, count):
    """Start recording the ring schedule into `entries` (int32 device tensor
    [capacity, 4]) and `count` (one zeroed int32 device element); pass None
    for both to stop.  See include/ra.h."""
    if entries is None:
        _check(_lib().ra_debug_visit_log(None, 0, None))
        return
    if entries.dim() != 2 or entries.shape[1] != 4 or entries.element_size() != 4 or not entries.is_contiguous():
        raise RAError(1, "visit log entries must be a contiguous [capacity, 4] tensor of 32-bit integers")
    _check(_lib().ra_debug_visit_log(_ptr(entries), entries.shape[0], _ptr(count)))


def ra_sync_status(stream=None):
    _check(_lib().ra_sync_status(_stream(stream)))


def ra_selftest_timeout(timeout_us, stream=None):
    _check(_lib().ra_selftest_timeout(int(timeout_us), _stream(stream)))


def ra_acc_init(o_acc, m_acc, l_acc, shape, stream=None):
    _check(_lib().ra_acc_init(_ptr(o_acc), _ptr(m_acc), _ptr(l_acc), shape, _stream(stream)))


def ra_block_fwd_workspace_bytes(dtype, shape):
    return int(_lib().ra_block_fwd_workspace_bytes(dtype, shape))


def ra_block_fwd(q, k_blk, v_blk, o_acc, m_acc, l_acc, q_off, kv_off, causal, scale,
                 workspace=None, shape=None, stream=None, precise=False):
    """Fold one key/value block into the running state of a query block."""
    shape = shape or shape_of(q, k_blk)
    dt = _dt(q)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().ra_block_fwd(_ptr(q), _ptr(k_blk), _ptr(v_blk), dt, _ptr(o_acc), _ptr(m_acc),
                            _ptr(l_acc), shape, int(q_off), int(kv_off), _flags(causal, precise),
                            float(scale), _ptr(workspace), ws_bytes, _stream(stream)))


def ra_merge(o_a, m_a, l_a, o_b, m_b, l_b, shape, stream=None):
    _check(_lib().ra_merge(_ptr(o_a), _ptr(m_a), _ptr(l_a), _ptr(o_b), _ptr(m_b), _ptr(l_b),
                        shape, _stream(stream)))


def ra_finalize(o_acc, m_acc, l_acc, o_out, lse, shape, stream=None):
    _check(_lib().ra_finalize(_ptr(o_acc), _ptr(m_acc), _ptr(l_acc), _ptr(o_out), _dt(o_out),
                           _ptr(lse), shape, _stream(stream)))


def _fwd_shape(q, k, v, o, lse):
    shape = shape_of(q, k)
    _same_layout(v, k, "v", "k")
    _same_layout(o, q, "o", "q")
    if lse is not None and not lse.is_contiguous():
        raise RAError(1, "lse must be packed [B, Hq, N]")
    return shape


def _bwd_shape(q, k, v, o, dO, lse, dq, dk, dv):
    shape = _fwd_shape(q, k, v, o, lse)
    for t, name in ((dO, "dO"), (dq, "dq")):
        _same_layout(t, q, name, "q")
    for t, name in ((dk, "dk"), (dv, "dv")):
        _same_layout(t, k, name, "k")
    return shape


def ra_ring_fwd_workspace_bytes(dtype, shape, P):
    return int(_lib().ra_ring_fwd_workspace_bytes(dtype, shape, P))


def ra_ring_fwd(q, k, v, P, causal, scale, o, lse, workspace=None, stream=None, precise=False,
                striped=False):
    shape = _fwd_shape(q, k, v, o, lse)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().ra_ring_fwd(_ptr(q), _ptr(k), _ptr(v), _dt(q), shape, int(P), _flags(causal, precise, striped),
                           float(scale), _ptr(o), _dt(o), _ptr(lse), _ptr(workspace), ws_bytes,
                           _stream(stream)))


def ra_ring_fwd_noalloc(q, k, v, P, causal, scale, o, lse, stream=None, precise=False, striped=False):
    """ra_ring_fwd without a workspace, for callers that cannot allocate device
    memory: the library's own 32 MiB per-device scratch buffer is used instead
    (shapes needing more are rejected).  Calls that overlap on the GPU race on
    that buffer."""
    shape = _fwd_shape(q, k, v, o, lse)
    _check(_lib().ra_ring_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _dt(q), shape, int(P),
                                   _flags(causal, precise, striped), float(scale), _ptr(o), _dt(o),
                                   _ptr(lse), _stream(stream)))


def ra_ring_fwd_varlen(q, k, v, P, host_len, causal, scale, o, lse, workspace=None, stream=None,
                       precise=False):
    """Ring forward where host i's first host_len[i] rows are valid (host_len:
    int32 device tensor of P entries) and the rest is padding."""
    shape = _fwd_shape(q, k, v, o, lse)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().ra_ring_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _dt(q), shape, int(P), _ptr(host_len),
                                  _flags(causal, precise), float(scale), _ptr(o), _dt(o), _ptr(lse),
                                  _ptr(workspace), ws_bytes, _stream(stream)))


def ra_ring_bwd_varlen(q, k, v, o, dO, lse, P, host_len, causal, scale, dq, dk, dv, workspace,
                       stream=None, precise=False):
    shape = _bwd_shape(q, k, v, o, dO, lse, dq, dk, dv)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().ra_ring_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dt(o), _ptr(dO), _ptr(lse),
                                  _dt(q), shape, int(P), _ptr(host_len), _flags(causal, precise),
                                  float(scale), _ptr(dq), _ptr(dk), _ptr(dv), _dt(dq), _ptr(workspace),
                                  ws_bytes, _stream(stream)))


def ra_ring_step_host_workspace_bytes(dtype, o_dtype, grad_dtype, shape, P):
    return int(_lib().ra_ring_step_host_workspace_bytes(dtype, o_dtype, grad_dtype, shape, int(P)))


def ra_ring_step_host(q, k, v, dO, P, causal, scale, o, lse, dq, dk, dv, workspace, stream=None,
                      precise=False, striped=False):
    """Forward + backward with q, k, v, dO and the outputs o, lse, dq, dk, dv in
    host (CPU) memory; the library uploads, computes and downloads on `stream`
    (pinned tensors make the copies asynchronous).  workspace: device uint8
    tensor of ra_ring_step_host_workspace_bytes() bytes."""
    for t in (q, k, v, dO, o, lse, dq, dk, dv):
        if t.is_cuda:
            raise RAError(1, "ra_ring_step_host takes host tensors")
    # one layout per group: q's for dO, o, dq; k's for v, dk, dv (the library
    # takes host tensors with packed rows and any batch stride)
    shape = _bwd_shape(q, k, v, o, dO, lse, dq, dk, dv)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib().ra_ring_step_host(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _dt(q), shape, int(P),
                                 _flags(causal, precise, striped), float(scale), _ptr(o), _dt(o),
                                 _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _dt(dq), _ptr(workspace),
                                 ws_bytes, _stream(stream)))


def ra_ffn_workspace_bytes(dtype, T, d_model, d_hidden, block, backward):
    return int(_lib().ra_ffn_workspace_bytes(dtype, int(T), int(d_model), int(d_hidden), int(block),
                                          1 if backward else 0))


def _ffn_check(x, w1, w2):
    if x.dim() != 2 or w1.dim() != 2 or w2.dim() != 2:
        raise RAError(1, "feed-forward tensors are 2-D: x [T, d_model], w1 [d_hidden, d_model], w2 [d_model, d_hidden]")
    T, dm = x.shape
    dh = w1.shape[0]
    if tuple(w1.shape) != (dh, dm) or tuple(w2.shape) != (dm, dh):
        raise RAError(1, f"weight shapes {tuple(w1.shape)}, {tuple(w2.shape)} do not match x {tuple(x.shape)}")
    for t in (x, w1, w2):
        if not t.is_contiguous():
            raise RAError(1, "feed-forward tensors must be contiguous")
    return T, dm, dh


def ra_ffn_fwd(x, w1, w2, block, y, workspace, stream=None):
    """y = GELU(x w1^T) w2^T one block of `block` tokens at a time."""
    T, dm, dh = _ffn_check(x, w1, w2)
    _check(_lib().ra_ffn_fwd(_ptr(x), _ptr(w1), _ptr(w2), _dt(x), T, dm, dh, int(block), _ptr(y), _dt(y),
                          _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def ra_ffn_bwd(x, w1, w2, dy, block, dx, dw1, dw2, workspace, stream=None):
    """Gradients of sum(y * dy): dx, and fp32 dw1, dw2 (overwritten)."""
    T, dm, dh = _ffn_check(x, w1, w2)
    _check(_lib().ra_ffn_bwd(_ptr(x), _ptr(w1), _ptr(w2), _ptr(dy), _dt(x), T, dm, dh, int(block), _ptr(dx),
                          _dt(dx), _ptr(dw1), _ptr(dw2), _ptr(workspace),
                          workspace.numel() * workspace.element_size(), _stream(stream)))


def ffn_fwd(x, w1, w2, block=None, y_dtype=None, stream=None):
    """Convenience wrapper: allocates y and the workspace."""
    T, dm, dh = _ffn_check(x, w1, w2)
    block = T if block is None else block
    y = torch.empty(T, dm, dtype=y_dtype or x.dtype, device=x.device)
    ws = _workspace(ra_ffn_workspace_bytes(_dt(x), T, dm, dh, block, False), x.device)
    ra_ffn_fwd(x, w1, w2, block, y, ws, stream)
    return y


def ffn_bwd(x, w1, w2, dy, block=None, dx_dtype=torch.float32, stream=None):
    T, dm, dh = _ffn_check(x, w1, w2)
    block = T if block is None else block
    dx = torch.empty(T, dm, dtype=dx_dtype, device=x.device)
    dw1 = torch.empty(dh, dm, dtype=torch.float32, device=x.device)
    dw2 = torch.empty(dm, dh, dtype=torch.float32, device=x.device)
    ws = _workspace(ra_ffn_workspace_bytes(_dt(x), T, dm, dh, block, True), x.device)
    ra_ffn_bwd(x, w1, w2, dy, block, dx, dw1, dw2, ws, stream)
    return dx, dw1, dw2


def ra_ring_bwd_workspace_bytes(dtype, grad_dtype, shape, P):
    return int(_lib().ra_ring_bwd_workspace_bytes(dtype, grad_dtype, shape, P))


def ra_ring_bwd(q, k, v, o, dO, lse, P, causal, scale, dq, dk, dv, workspace, stream=None,
                precise=False, striped=False):
    shape = _bwd_shape(q, k, v, o, dO, lse, dq, dk, dv)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().ra_ring_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dt(o), _ptr(dO), _ptr(lse),
                           _dt(q), shape, int(P), _flags(causal, precise, striped), float(scale), _ptr(dq),
                           _ptr(dk), _ptr(dv), _dt(dq), _ptr(workspace), ws_bytes,
                           _stream(stream)))


def _flags(causal, precise, striped=False):
    return (RA_CAUSAL if causal else 0) | (RA_PRECISE if precise else 0) | (RA_STRIPED if striped else 0)


def _workspace(nbytes, device):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def ring_attention_fwd(q, k, v, P, causal=True, scale=None, o_dtype=torch.float32,
                       stream=None, precise=False, striped=False, host_len=None):
    """Allocate O [B,N,Hq,d] (o_dtype) and LSE [B,Hq,N] fp32 and run the ring forward."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    B, N, Hq, d = q.shape
    o = empty_like_layout(q, o_dtype)  # the q group's layout
    lse = torch.empty(B, Hq, N, dtype=torch.float32, device=q.device)
    ws = _workspace(ra_ring_fwd_workspace_bytes(_dt(q), shape_of(q, k), P), q.device)
    if host_len is not None:
        if striped:
            raise RAError(1, "striped layouts do not combine with per-host lengths")
        ra_ring_fwd_varlen(q, k, v, P, host_len, causal, scale, o, lse, ws, stream, precise)
    else:
        ra_ring_fwd(q, k, v, P, causal, scale, o, lse, ws, stream, precise, striped)
    return o, lse


def ring_attention_bwd(q, k, v, o, lse, dO, P, causal=True, scale=None,
                       grad_dtype=torch.float32, stream=None, precise=False, striped=False,
                       host_len=None):
    """Allocate dQ, dK, dV (grad_dtype) and workspace and run the ring backward."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    dq = empty_like_layout(q, grad_dtype)
    dk = empty_like_layout(k, grad_dtype)
    dv = empty_like_layout(k, grad_dtype)
    ws = _workspace(ra_ring_bwd_workspace_bytes(_dt(q), _DTYPES[grad_dtype], shape_of(q, k), P),
                    q.device)
    if host_len is not None:
        if striped:
            raise RAError(1, "striped layouts do not combine with per-host lengths")
        ra_ring_bwd_varlen(q, k, v, o, dO, lse, P, host_len, causal, scale, dq, dk, dv, ws, stream, precise)
    else:
        ra_ring_bwd(q, k, v, o, dO, lse, P, causal, scale, dq, dk, dv, ws, stream, precise, striped)
    return dq, dk, dv
