"""GB300 chunkwise gated delta rule forward -- Python binding of the C ABI.

The binding only marshals arguments: every step of the forward runs in the
CUDA kernels of ``libdnchunk.so`` (declared in ``include/dn_chunk_fwd.h``).
There is no CPU path: if the library is missing, :func:`load` raises.
PyTorch supplies device memory and streams.

Names follow the C ABI: :func:`dn_chunk_fwd`,
:func:`dn_chunk_fwd_workspace_bytes`, :func:`dn_chunk_fwd_noalloc`,
:func:`dn_recurrent_fwd`, :func:`dn_chunk_bwd`,
:func:`dn_chunk_bwd_workspace_bytes`, :func:`dn_check`,
:func:`dn_status_str`, :func:`dn_last_kernel`.  :func:`recurrent_fwd` and
:func:`chunk_bwd` are conveniences for the token-serial entry point and the
backward.  :func:`chunk_fwd` is a convenience that allocates
``o``, ``ht`` and the workspace with torch and calls :func:`dn_chunk_fwd`.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdnchunk.so")

DN_OK = 0
DN_ERR_INVALID_ARG = 1
DN_ERR_UNSUPPORTED = 2
DN_ERR_CUDA = 3
DN_ERR_TIMEOUT = 4
DN_ERR_DEVICE_ARG = 5

DN_BF16 = 0
DN_F32 = 1

# Option bits of the ``flags`` argument.
DN_QK_L2NORM = 1

# Every symbol the public header declares.
ABI_SYMBOLS = ("dn_chunk_fwd", "dn_chunk_fwd_workspace_bytes", "dn_chunk_fwd_noalloc",
               "dn_recurrent_fwd", "dn_chunk_bwd", "dn_chunk_bwd_workspace_bytes", "dn_check",
               "dn_status_str", "dn_last_kernel")

# Size of the library's fixed scratch array used by dn_chunk_fwd_noalloc.
DN_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024

_lib = None
_lock = threading.Lock()


class DnError(RuntimeError):
    def __init__(self, status: int, what: str = "dn_chunk_fwd"):
        self.status = status
        super().__init__("%s failed: %s" % (what, dn_status_str(status)))


def load(path: str | None = None):
    """Load ``libdnchunk.so`` (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                "libdnchunk.so is not built (%s); run `python -c \"import __graft_entry__ as g; "
                "g.build()\"` -- there is no fallback path" % p)
        lib = ctypes.CDLL(p)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        Z, U = ctypes.c_size_t, ctypes.c_uint
        lib.dn_chunk_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, U, I, P, P, P, Z,
                                     P]
        lib.dn_chunk_fwd.restype = I
        lib.dn_chunk_fwd_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I, I]
        lib.dn_chunk_fwd_workspace_bytes.restype = Z
        lib.dn_chunk_fwd_noalloc.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, U, I, P,
                                             P, P]
        lib.dn_chunk_fwd_noalloc.restype = I
        lib.dn_recurrent_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, U, P, P, P]
        lib.dn_recurrent_fwd.restype = I
        lib.dn_chunk_bwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, U, P, P, P, P,
                                     P, P, P, P, P, Z, P]
        lib.dn_chunk_bwd.restype = I
        lib.dn_chunk_bwd_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I]
        lib.dn_chunk_bwd_workspace_bytes.restype = Z
        lib.dn_check.argtypes = [P]
        lib.dn_check.restype = I
        lib.dn_status_str.argtypes = [I]
        lib.dn_status_str.restype = ctypes.c_char_p
        lib.dn_last_kernel.argtypes = []
        lib.dn_last_kernel.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def _ptr(x):
    """Device pointer of a tensor (or an int address, or None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    if not x.is_contiguous():
        raise ValueError("tensors passed to dn_chunk_fwd must be contiguous")
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dn_chunk_fwd(q, k, v, beta, g, h0, cu_seqlens, n_seqs, B, T, Nk, Nv, dk, dv, dtype,
                 scale, chunk, o, ht, workspace=None, workspace_bytes=None, stream=None,
                 flags=0) -> int:
    """Call the C entry point as is; returns its status code.

    ``workspace`` is a device tensor (its byte size is passed unless
    ``workspace_bytes`` is given), an int address, or None.  ``flags`` is the
    C argument of that name (0 or :data:`DN_QK_L2NORM`).
    """
    lib = load()
    if workspace_bytes is None:
        workspace_bytes = 0
        if workspace is not None and not isinstance(workspace, int):
            workspace_bytes = workspace.numel() * workspace.element_size()
    return lib.dn_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                            _ptr(cu_seqlens), int(n_seqs), int(B), int(T), int(Nk), int(Nv),
                            int(dk), int(dv), int(dtype), float(scale), int(flags), int(chunk),
                            _ptr(o), _ptr(ht), _ptr(workspace), int(workspace_bytes),
                            _stream(stream))


def dn_chunk_fwd_noalloc(q, k, v, beta, g, h0, cu_seqlens, n_seqs, B, T, Nk, Nv, dk, dv, dtype,
                         scale, chunk, o, ht, stream=None, flags=0) -> int:
    """Call the C entry point that takes no workspace (it uses the library's
    fixed scratch array and allocates nothing); returns its status code."""
    lib = load()
    return lib.dn_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                                    _ptr(cu_seqlens), int(n_seqs), int(B), int(T), int(Nk),
                                    int(Nv), int(dk), int(dv), int(dtype), float(scale), int(flags),
                                    int(chunk), _ptr(o), _ptr(ht), _stream(stream))


def dn_recurrent_fwd(q, k, v, beta, g, h0, cu_seqlens, n_seqs, B, T, Nk, Nv, dk, dv, dtype,
                     scale, o, ht, stream=None, flags=0) -> int:
    """Call the token-serial C entry point as is; returns its status code."""
    lib = load()
    return lib.dn_recurrent_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                                _ptr(cu_seqlens), int(n_seqs), int(B), int(T), int(Nk), int(Nv),
                                int(dk), int(dv), int(dtype), float(scale), int(flags), _ptr(o),
                                _ptr(ht), _stream(stream))


def recurrent_fwd(q, k, v, beta, g=None, h0=None, cu_seqlens=None, scale=None,
                  output_final_state=True, stream=None, o=None, ht=None,
                  use_qk_l2norm_in_kernel=False):
    """Allocate ``o`` (and ``ht``) and run :func:`dn_recurrent_fwd` (shapes
    and options as for :func:`chunk_fwd`)."""
    import torch
    B, T, Nk, dk = q.shape
    Nv, dv = v.shape[2], v.shape[3]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    if o is None:
        o = torch.empty(B, T, Nv, dv, dtype=q.dtype, device=q.device)
    if ht is None and output_final_state:
        ht = torch.empty(N, Nv, dk, dv, dtype=torch.float32, device=q.device)
    st = dn_recurrent_fwd(q, k, v, beta, g, h0, cu_seqlens, N, B, T, Nk, Nv, dk, dv,
                          dtype_code(q.dtype), 0.0 if scale is None else scale, o,
                          ht if output_final_state else None, stream,
                          flags=DN_QK_L2NORM if use_qk_l2norm_in_kernel else 0)
    if st != DN_OK:
        raise DnError(st, "dn_recurrent_fwd")
    return o, (ht if output_final_state else None)


def dn_chunk_fwd_workspace_bytes(n_seqs, B, T, Nk, Nv, dk, dv, dtype, chunk=64) -> int:
    return int(load().dn_chunk_fwd_workspace_bytes(int(n_seqs), int(B), int(T), int(Nk), int(Nv),
                                                   int(dk), int(dv), int(dtype), int(chunk)))


def workspace_for(q, v, n_seqs, chunk=64):
    """A uint8 device tensor of the workspace size for these inputs (or None)."""
    import torch
    B, T, Nk, dk = q.shape
    Nv, dv = v.shape[2], v.shape[3]
    nbytes = dn_chunk_fwd_workspace_bytes(n_seqs, B, T, Nk, Nv, dk, dv, dtype_code(q.dtype), chunk)
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=q.device)


def dn_check(stream=None) -> int:
    return load().dn_check(_stream(stream))


def dn_status_str(status: int) -> str:
    try:
        return load().dn_status_str(int(status)).decode()
    except RuntimeError:
        return "status %d" % status


def dn_last_kernel() -> str:
    return load().dn_last_kernel().decode()


def dtype_code(dtype) -> int:
    import torch
    if dtype == torch.bfloat16:
        return DN_BF16
    if dtype == torch.float32:
        return DN_F32
    raise ValueError("unsupported dtype %s (bf16 or fp32)" % dtype)


def chunk_fwd(q, k, v, beta, g=None, h0=None, cu_seqlens=None, scale=None,
              output_final_state=True, chunk=64, stream=None, o=None, ht=None, workspace=None,
              use_qk_l2norm_in_kernel=False):
    """Allocate ``o`` (and ``ht``, and the workspace) and run :func:`dn_chunk_fwd`.

    q, k ``[B, T, Nk, dk]``; v ``[B, T, Nv, dv]``; beta, g ``[B, T, Nv]`` fp32;
    h0 ``[N, Nv, dk, dv]`` fp32; cu_seqlens int64 ``[N+1]`` on the device.
    ``use_qk_l2norm_in_kernel`` sets :data:`DN_QK_L2NORM` (the kernels
    normalise every q and k row).  Returns ``(o, ht)`` (``ht`` is None unless
    ``output_final_state``).
    """
    import torch
    B, T, Nk, dk = q.shape
    Nv, dv = v.shape[2], v.shape[3]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    if o is None:
        o = torch.empty(B, T, Nv, dv, dtype=q.dtype, device=q.device)
    if ht is None and output_final_state:
        ht = torch.empty(N, Nv, dk, dv, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = workspace_for(q, v, N, chunk)
    st = dn_chunk_fwd(q, k, v, beta, g, h0, cu_seqlens, N, B, T, Nk, Nv, dk, dv,
                      dtype_code(q.dtype), 0.0 if scale is None else scale, chunk, o,
                      ht if output_final_state else None, workspace, stream=stream,
                      flags=DN_QK_L2NORM if use_qk_l2norm_in_kernel else 0)
    if st != DN_OK:
        raise DnError(st)
    return o, (ht if output_final_state else None)


def dn_chunk_bwd(q, k, v, beta, g, h0, cu_seqlens, n_seqs, B, T, Nk, Nv, dk, dv, dtype, scale,
                 flags, d_o, d_ht, d_q, d_k, d_v, d_beta, d_g, d_h0, workspace,
                 workspace_bytes=None, stream=None) -> int:
    """Call the backward C entry point as is; returns its status code."""
    lib = load()
    if workspace_bytes is None:
        workspace_bytes = 0
        if workspace is not None and not isinstance(workspace, int):
            workspace_bytes = workspace.numel() * workspace.element_size()
    return lib.dn_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                            _ptr(cu_seqlens), int(n_seqs), int(B), int(T), int(Nk), int(Nv),
                            int(dk), int(dv), int(dtype), float(scale), int(flags), _ptr(d_o),
                            _ptr(d_ht), _ptr(d_q), _ptr(d_k), _ptr(d_v), _ptr(d_beta), _ptr(d_g),
                            _ptr(d_h0), _ptr(workspace), int(workspace_bytes), _stream(stream))


def dn_chunk_bwd_workspace_bytes(n_seqs, B, T, Nk, Nv, dk, dv, dtype) -> int:
    return int(load().dn_chunk_bwd_workspace_bytes(int(n_seqs), int(B), int(T), int(Nk),
                                                   int(Nv), int(dk), int(dv), int(dtype)))


def chunk_bwd(q, k, v, beta, g=None, h0=None, cu_seqlens=None, scale=None, do=None, dht=None,
              stream=None, workspace=None, use_qk_l2norm_in_kernel=False):
    """Gradients of :func:`chunk_fwd`'s loss ``sum(do * o) + sum(dht * ht)``
    (with the same ``use_qk_l2norm_in_kernel``).

    Allocates the fp32 gradients and the workspace with torch and runs
    :func:`dn_chunk_bwd`.  Returns a dict with ``dq``, ``dk``, ``dv``,
    ``dbeta``, ``dg`` (None when g is None) and ``dh0`` (None when h0 is None).
    """
    import torch
    B, T, Nk, dk = q.shape
    Nv, dv = v.shape[2], v.shape[3]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    f32 = dict(dtype=torch.float32, device=q.device)
    out = dict(dq=torch.empty(q.shape, **f32), dk=torch.empty(k.shape, **f32),
               dv=torch.empty(v.shape, **f32), dbeta=torch.empty(beta.shape, **f32),
               dg=None if g is None else torch.empty(beta.shape, **f32),
               dh0=None if h0 is None else torch.empty(N, Nv, dk, dv, **f32))
    if workspace is None:
        nbytes = dn_chunk_bwd_workspace_bytes(N, B, T, Nk, Nv, dk, dv, dtype_code(q.dtype))
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = dn_chunk_bwd(q, k, v, beta, g, h0, cu_seqlens, N, B, T, Nk, Nv, dk, dv,
                      dtype_code(q.dtype), 0.0 if scale is None else scale,
                      DN_QK_L2NORM if use_qk_l2norm_in_kernel else 0, do, dht,
                      out["dq"], out["dk"], out["dv"], out["dbeta"], out["dg"], out["dh0"],
                      workspace, stream=stream)
    if st != DN_OK:
        raise DnError(st, "dn_chunk_bwd")
    return out
