"""fp64 CPU oracle for the chunkwise gated delta rule forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never loads it, and it shares no code with the CUDA library.

Functions follow the pages' notation:

* :func:`recurrent` -- the definition, a token-by-token recurrence
  ("flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现" §1;
  "01 · 数学原理:ChunkGatedDeltaRule 在算什么" §1), decayed read.
* :func:`chunked` -- the chunk algorithm in the pages' order (same pages,
  §2.3-§2.4 and §3.1-§3.3), with a dense forward-substitution solve.
* :func:`wy_chunk` -- steps a1-a4 of one chunk (G, T, W, U), exposed so the
  tests can check W and U against brute-force Householder-like products.
* :func:`recurrent_bwd` -- the gradient of :func:`recurrent` (reverse mode
  through the token recurrence) for given output and final-state gradients;
  :func:`l2norm_bwd` is the gradient of :func:`l2norm`.
* :func:`l2norm` -- the row normalisation that ``use_qk_l2norm_in_kernel``
  applies to q and k ("flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与
  Triton 内核实现" §5, §6); :func:`recurrent` and :func:`chunked` take the
  same option and normalise q and k with it before anything else.

All arithmetic is fp64 (``dn_oracle.c``; :func:`l2norm` in numpy).  Every function here is pinned by
``tests/test_oracle_pins.py``; none is marked "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``dn_oracle.c`` into ``liboracle.so`` (gcc, -O2, pthreads)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.dn_oracle_recurrent.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, D,
                                                P, P, I, P, I, I]
            lib.dn_oracle_recurrent.restype = I
            lib.dn_oracle_chunked.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, D, I,
                                              P, P, P, I, I]
            lib.dn_oracle_chunked.restype = I
            lib.dn_oracle_wy_chunk.argtypes = [I, I, I, P, ctypes.c_long, P, ctypes.c_long,
                                               P, ctypes.c_long, P, ctypes.c_long, P, P, P, P]
            lib.dn_oracle_wy_chunk.restype = None
            lib.dn_oracle_recurrent_bwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, D,
                                                    P, P, P, P, P, P, P, P, P, I, I]
            lib.dn_oracle_recurrent_bwd.restype = I
            lib.dn_oracle_default_threads.argtypes = []
            lib.dn_oracle_default_threads.restype = I
            _lib = lib
    return _lib


def default_threads() -> int:
    """Threads the oracle uses when ``threads=0`` (the host's online cores)."""
    return int(_load().dn_oracle_default_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: exact upcast on the CPU
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _shapes(q, v, cu_seqlens):
    B, T, Nk, dk = q.shape
    Nv, dv = v.shape[2], v.shape[3]
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens), dtype=np.int64)
        N = len(cu) - 1
    else:
        cu, N = None, B
    return B, T, Nk, dk, Nv, dv, cu, N


def _units(units):
    if units is None:
        return None, 0
    u = np.ascontiguousarray(np.asarray(units), dtype=np.int32)
    return u, len(u)


def l2norm(x):
    """Each row (last axis) of ``x`` divided by ``max(||row||_2, 1e-12)``, fp64.

    The pages' tests L2-normalise k along the head dimension with
    ``F.normalize(p=2, dim=-1)`` (whose guard is 1e-12), and the option
    ``use_qk_l2norm_in_kernel`` moves that normalisation, for q and k, into
    the kernels ("flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton
    内核实现" §5 parameter table, §6).
    """
    x = _f64(x)
    norm = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(norm, 1e-12)


def recurrent(q, k, v, beta, g=None, h0=None, cu_seqlens=None, scale=None,
              units=None, threads=0, read_mode=0, use_qk_l2norm_in_kernel=False):
    """Token recurrence in fp64.

    Shapes: q, k ``[B, T, Nk, dk]``; v ``[B, T, Nv, dv]``; beta, g ``[B, T, Nv]``;
    h0 ``[N, Nv, dk, dv]``.  Returns ``(o [B, T, Nv, dv], ht [N, Nv, dk, dv])``
    in fp64.  ``units`` restricts the work to the listed ``n * Nv + h``
    (sequence, v-head) pairs; other outputs stay NaN.  ``read_mode=1`` is the
    literal undecayed read, kept only to show the chunk form rejects it.
    ``use_qk_l2norm_in_kernel`` first replaces q and k by :func:`l2norm` of them.
    """
    lib = _load()
    q, k, v, beta, g, h0 = map(_f64, (q, k, v, beta, g, h0))
    if use_qk_l2norm_in_kernel:
        q, k = l2norm(q), l2norm(k)
    B, T, Nk, dk, Nv, dv, cu, N = _shapes(q, v, cu_seqlens)
    if scale is None:
        scale = dk ** -0.5
    o = np.full((B, T, Nv, dv), np.nan)
    ht = np.full((N, Nv, dk, dv), np.nan)
    u, nu = _units(units)
    rc = lib.dn_oracle_recurrent(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                                 _ptr(cu), N, B, T, Nk, Nv, dk, dv, float(scale),
                                 _ptr(o), _ptr(ht), int(read_mode), _ptr(u), nu, int(threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (rc=%d)" % rc)
    return o, ht


def chunked(q, k, v, beta, g=None, h0=None, cu_seqlens=None, scale=None, chunk=64,
            units=None, threads=0, use_qk_l2norm_in_kernel=False):
    """Chunk algorithm in fp64 (steps a1-a6); same shapes and options as
    :func:`recurrent`."""
    lib = _load()
    q, k, v, beta, g, h0 = map(_f64, (q, k, v, beta, g, h0))
    if use_qk_l2norm_in_kernel:
        q, k = l2norm(q), l2norm(k)
    B, T, Nk, dk, Nv, dv, cu, N = _shapes(q, v, cu_seqlens)
    if scale is None:
        scale = dk ** -0.5
    o = np.full((B, T, Nv, dv), np.nan)
    ht = np.full((N, Nv, dk, dv), np.nan)
    u, nu = _units(units)
    rc = lib.dn_oracle_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                               _ptr(cu), N, B, T, Nk, Nv, dk, dv, float(scale), int(chunk),
                               _ptr(o), _ptr(ht), _ptr(u), nu, int(threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (rc=%d)" % rc)
    return o, ht


def wy_chunk(k, v, beta, g=None):
    """Steps a1-a4 of one chunk: k ``[L, dk]``, v ``[L, dv]``, beta/g ``[L]``.

    Returns ``(G [L], T [L, L], W [L, dk], U [L, dv])`` in fp64 with
    ``T = (I - A)^-1``, ``W = T diag(beta e^G) K``, ``U = T diag(beta) V``.
    """
    lib = _load()
    k, v, beta, g = map(_f64, (k, v, beta, g))
    L, dk = k.shape
    dv = v.shape[1]
    G = np.zeros(L)
    Tm = np.zeros((L, L))
    W = np.zeros((L, dk))
    U = np.zeros((L, dv))
    lib.dn_oracle_wy_chunk(L, dk, dv, _ptr(k), dk, _ptr(v), dv, _ptr(beta), 1,
                           _ptr(g), 1, _ptr(G), _ptr(Tm), _ptr(W), _ptr(U))
    return G, Tm, W, U


def l2norm_bwd(x, dy):
    """Gradient with respect to ``x`` of ``sum(dy * l2norm(x))``, row by row, fp64.

    For a row with ``||x|| > 1e-12``: ``(dy - y (y . dy)) / ||x||`` with
    ``y = x / ||x||`` (the derivative of x / ||x||); below the guard the
    divisor is the constant 1e-12, so the gradient is ``dy / 1e-12``.
    """
    x, dy = _f64(x), _f64(dy)
    norm = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    big = norm > 1e-12
    y = x / np.where(big, norm, 1.0)
    proj = np.sum(y * dy, axis=-1, keepdims=True)
    return np.where(big, (dy - y * proj) / np.where(big, norm, 1.0), dy / 1e-12)


def recurrent_bwd(q, k, v, beta, g=None, h0=None, cu_seqlens=None, scale=None, do=None,
                  dht=None, groups=None, threads=0, use_qk_l2norm_in_kernel=False):
    """Gradient of the forward in fp64, reverse mode through the token recurrence.

    For the loss ``sum(do * o) + sum(dht * ht)`` of :func:`recurrent` (same
    shapes; ``do`` like o, ``dht`` like ht or None), returns a dict with
    ``dq``, ``dk`` (``[B, T, Nk, dk]``), ``dv`` (like v), ``dbeta``, ``dg``
    (``[B, T, Nv]``) and ``dh0`` (``[N, Nv, dk, dv]``).  ``groups`` restricts
    the work to the listed ``n * Nk + hk`` (sequence, key head) groups, each
    with all value heads that read key head hk; other entries stay NaN.
    ("flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现" §3.4
    lists these gradients; the pages print no formula for them, so this is
    the chain rule through each step of the definition.)  With
    ``use_qk_l2norm_in_kernel`` the forward normalises q and k first
    (:func:`l2norm`), and dq, dk go back through :func:`l2norm_bwd`.
    """
    lib = _load()
    q, k, v, beta, g, h0, do, dht = map(_f64, (q, k, v, beta, g, h0, do, dht))
    if use_qk_l2norm_in_kernel:
        out = recurrent_bwd(l2norm(q), l2norm(k), v, beta, g, h0, cu_seqlens, scale, do, dht,
                            groups, threads)
        out["dq"] = l2norm_bwd(q, out["dq"])
        out["dk"] = l2norm_bwd(k, out["dk"])
        return out
    B, T, Nk, dk, Nv, dv, cu, N = _shapes(q, v, cu_seqlens)
    if scale is None:
        scale = dk ** -0.5
    out = dict(dq=np.full(q.shape, np.nan), dk=np.full(k.shape, np.nan),
               dv=np.full(v.shape, np.nan), dbeta=np.full(beta.shape, np.nan),
               dg=np.full(beta.shape, np.nan), dh0=np.full((N, Nv, dk, dv), np.nan))
    gr, ng = _units(groups)
    rc = lib.dn_oracle_recurrent_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                                     _ptr(cu), N, B, T, Nk, Nv, dk, dv, float(scale),
                                     _ptr(do), _ptr(dht), _ptr(out["dq"]), _ptr(out["dk"]),
                                     _ptr(out["dv"]), _ptr(out["dbeta"]), _ptr(out["dg"]),
                                     _ptr(out["dh0"]), _ptr(gr), ng, int(threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (rc=%d)" % rc)
    return out
