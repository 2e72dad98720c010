"""Boundary tests that need no GPU: the library loads, exports exactly the
entry points its headers declare, and rejects bad arguments on the host
before anything reaches the device."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

import chunkwise_gated_delta_chunk_gb300 as dn
from chunkwise_gated_delta_chunk_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def clib():
    _build.build()
    return dn.load()


def declared_symbols():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(dn_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_abi():
    assert set(dn.ABI_SYMBOLS) <= declared_symbols()


def test_library_exports_every_declared_symbol(clib):
    for name in declared_symbols():
        assert getattr(clib, name) is not None


def test_library_exports_nothing_else():
    _build.build()
    out = subprocess.run(["nm", "-D", "--defined-only", dn.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    ours = {line.split()[-1] for line in out.splitlines()
            if line.split() and line.split()[-1].startswith("dn_")}
    assert ours == declared_symbols()


def test_status_strings(clib):
    for code, name in [(0, "DN_OK"), (1, "DN_ERR_INVALID_ARG"), (2, "DN_ERR_UNSUPPORTED"),
                       (3, "DN_ERR_CUDA"), (4, "DN_ERR_TIMEOUT"), (5, "DN_ERR_DEVICE_ARG")]:
        assert clib.dn_status_str(code).decode() == name
    assert clib.dn_status_str(99).decode() == "DN_ERR_UNKNOWN"


# Fake, 16-byte aligned "device" addresses: validation rejects the call before
# any pointer could be used, so nothing is ever dereferenced.
A = 1 << 20


def call(clib, **over):
    args = dict(q=A, k=A, v=A, beta=A, g=None, h0=None, cu=None, n=2, B=2, T=64, Nk=2, Nv=4,
                dk=64, dv=64, dtype=dn.DN_BF16, scale=0.0, flags=0, chunk=64, o=A, ht=None,
                ws=None, wsb=0)
    args.update(over)
    return clib.dn_chunk_fwd(args["q"], args["k"], args["v"], args["beta"], args["g"], args["h0"],
                             args["cu"], args["n"], args["B"], args["T"], args["Nk"], args["Nv"],
                             args["dk"], args["dv"], args["dtype"], args["scale"], args["flags"],
                             args["chunk"], args["o"], args["ht"], args["ws"], args["wsb"], None)


@pytest.mark.parametrize("over,code", [
    (dict(Nv=3), dn.DN_ERR_INVALID_ARG),                 # Nv % Nk != 0
    (dict(Nk=0), dn.DN_ERR_INVALID_ARG),
    (dict(n=3), dn.DN_ERR_INVALID_ARG),                  # N != B without cu_seqlens
    (dict(cu=A, n=2, B=2), dn.DN_ERR_INVALID_ARG),       # cu_seqlens needs B == 1
    (dict(q=None), dn.DN_ERR_INVALID_ARG),
    (dict(beta=None), dn.DN_ERR_INVALID_ARG),
    (dict(o=None), dn.DN_ERR_INVALID_ARG),
    (dict(q=A + 8), dn.DN_ERR_INVALID_ARG),              # misaligned
    (dict(ht=A + 4), dn.DN_ERR_INVALID_ARG),
    (dict(T=-1), dn.DN_ERR_INVALID_ARG),
    (dict(dtype=7), dn.DN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), dn.DN_ERR_INVALID_ARG),
    (dict(flags=2), dn.DN_ERR_INVALID_ARG),              # unknown option bit
    (dict(flags=dn.DN_QK_L2NORM | 4), dn.DN_ERR_INVALID_ARG),
    (dict(chunk=0), dn.DN_ERR_INVALID_ARG),
    (dict(chunk=48), dn.DN_ERR_UNSUPPORTED),             # C in {16, 32, 64} is built
    (dict(chunk=128), dn.DN_ERR_UNSUPPORTED),
    (dict(dk=96), dn.DN_ERR_UNSUPPORTED),
    (dict(dv=512), dn.DN_ERR_UNSUPPORTED),
    (dict(dtype=dn.DN_F32, dk=256), dn.DN_ERR_UNSUPPORTED),
])
def test_invalid_arguments_rejected_on_host(clib, over, code):
    assert call(clib, **over) == code


def test_workspace_size(clib):
    """One slot per (floor(tokens/C) + N) x Nv on the tensor-core path (C the chunk
    length; 25088 bytes for dk = 128, 49664 for dk = 256, which holds -W), none
    elsewhere."""
    ws = clib.dn_chunk_fwd_workspace_bytes
    assert ws(4, 4, 2048, 16, 16, 128, 128, dn.DN_BF16, 64) == (4 * 2048 // 64 + 4) * 16 * 25088
    assert ws(3, 1, 300, 2, 8, 128, 256, dn.DN_BF16, 64) == (300 // 64 + 3) * 8 * 25088
    assert ws(8, 8, 8192, 8, 8, 256, 256, dn.DN_BF16, 64) == (8 * 8192 // 64 + 8) * 8 * 49664
    assert ws(2, 2, 100, 2, 4, 256, 128, dn.DN_BF16, 32) == (2 * 100 // 32 + 2) * 4 * 49664
    assert ws(2, 2, 64, 2, 4, 256, 64, dn.DN_BF16, 64) == 0      # dv not a multiple of 128
    assert ws(2, 2, 64, 2, 4, 64, 64, dn.DN_BF16, 64) == 0       # CUDA-core path
    assert ws(2, 2, 64, 2, 2, 128, 128, dn.DN_F32, 64) == 0      # fp32: CUDA-core path
    assert ws(2, 2, 0, 2, 2, 128, 128, dn.DN_BF16, 64) == 0      # no tokens
    assert ws(0, 0, 0, 2, 2, 128, 128, dn.DN_BF16, 64) == 0
    assert ws(2, 2, 64, 2, 2, 128, 128, dn.DN_BF16, 32) == (2 * 64 // 32 + 2) * 2 * 25088
    assert ws(1, 1, 100, 2, 2, 128, 128, dn.DN_BF16, 16) == (100 // 16 + 1) * 2 * 25088
    assert ws(2, 2, 64, 2, 2, 128, 128, dn.DN_F32, 32) == 0      # fp32: CUDA-core path
    assert ws(2, 2, 64, 2, 2, 128, 128, dn.DN_BF16, 48) == 0     # rejected chunk size


@pytest.mark.parametrize("ws,wsb", [(None, 0), (A, 1024), (A + 8, 1 << 30), (None, 1 << 30)])
def test_workspace_checked_on_host(clib, ws, wsb):
    """The tensor-core path rejects a missing, small or misaligned workspace before any launch."""
    assert call(clib, dk=128, dv=128, Nk=2, Nv=4, ws=ws, wsb=wsb) == dn.DN_ERR_INVALID_ARG


def rec_call(clib, **over):
    args = dict(q=A, k=A, v=A, beta=A, g=None, h0=None, cu=None, n=2, B=2, T=64, Nk=2, Nv=4,
                dk=64, dv=64, dtype=dn.DN_BF16, scale=0.0, flags=0, o=A, ht=None)
    args.update(over)
    return clib.dn_recurrent_fwd(args["q"], args["k"], args["v"], args["beta"], args["g"],
                                 args["h0"], args["cu"], args["n"], args["B"], args["T"], args["Nk"],
                                 args["Nv"], args["dk"], args["dv"], args["dtype"], args["scale"],
                                 args["flags"], args["o"], args["ht"], None)


@pytest.mark.parametrize("over,code", [
    (dict(Nv=3), dn.DN_ERR_INVALID_ARG),
    (dict(n=3), dn.DN_ERR_INVALID_ARG),
    (dict(cu=A, n=2, B=2), dn.DN_ERR_INVALID_ARG),
    (dict(k=None), dn.DN_ERR_INVALID_ARG),
    (dict(v=A + 8), dn.DN_ERR_INVALID_ARG),
    (dict(dtype=3), dn.DN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), dn.DN_ERR_INVALID_ARG),
    (dict(flags=8), dn.DN_ERR_INVALID_ARG),
    (dict(dk=96), dn.DN_ERR_UNSUPPORTED),
    (dict(dv=512), dn.DN_ERR_UNSUPPORTED),
])
def test_recurrent_invalid_arguments_rejected_on_host(clib, over, code):
    assert rec_call(clib, **over) == code


def test_recurrent_zero_sequences_is_a_noop(clib):
    assert rec_call(clib, n=0, B=0, T=0, q=None, k=None, v=None, beta=None, o=None) == dn.DN_OK


def test_zero_sequences_is_a_noop(clib):
    assert call(clib, n=0, B=0, T=0, q=None, k=None, v=None, beta=None, o=None) == dn.DN_OK
    assert call(clib, n=0, B=1, T=5, cu=A) == dn.DN_OK


def test_product_path_has_no_fallback(tmp_path):
    """The binding refuses to run without the CUDA library (no CPU path)."""
    with pytest.raises(RuntimeError, match="no fallback"):
        dn.load(str(tmp_path / "missing.so"))


def bwd_call(clib, **over):
    args = dict(q=A, k=A, v=A, beta=A, g=None, h0=None, cu=None, n=2, B=2, T=64, Nk=2, Nv=4,
                dk=64, dv=64, dtype=dn.DN_BF16, scale=0.0, flags=0, do=A, dht=None, dq=A, dkk=A,
                dvv=A, dbeta=A, dg=None, dh0=None, ws=A, wsb=1 << 30)
    args.update(over)
    return clib.dn_chunk_bwd(args["q"], args["k"], args["v"], args["beta"], args["g"], args["h0"],
                             args["cu"], args["n"], args["B"], args["T"], args["Nk"], args["Nv"],
                             args["dk"], args["dv"], args["dtype"], args["scale"], args["flags"],
                             args["do"], args["dht"], args["dq"], args["dkk"], args["dvv"],
                             args["dbeta"], args["dg"], args["dh0"], args["ws"], args["wsb"], None)


@pytest.mark.parametrize("over,code", [
    (dict(Nv=3), dn.DN_ERR_INVALID_ARG),
    (dict(n=3), dn.DN_ERR_INVALID_ARG),
    (dict(do=None), dn.DN_ERR_INVALID_ARG),              # gradient of o is required
    (dict(dq=None), dn.DN_ERR_INVALID_ARG),
    (dict(dbeta=A + 4), dn.DN_ERR_INVALID_ARG),          # misaligned
    (dict(flags=2), dn.DN_ERR_INVALID_ARG),
    (dict(ws=None), dn.DN_ERR_INVALID_ARG),              # the workspace is required
    (dict(wsb=1024), dn.DN_ERR_INVALID_ARG),             # and must be large enough
    (dict(dk=256), dn.DN_ERR_UNSUPPORTED),
    (dict(dv=48), dn.DN_ERR_UNSUPPORTED),
    (dict(n=0, B=0), dn.DN_OK),                           # nothing to do, nothing launched
])
def test_bwd_host_validation(clib, over, code):
    """dn_chunk_bwd rejects bad arguments on the host before any CUDA call."""
    assert bwd_call(clib, **over) == code


def test_bwd_workspace_bytes(clib):
    """One fp32 dk x dv state per (floor(tokens/64) + N) x Nv, plus the forward's
    WY slots where that forward runs on the tensor cores; 0 for rejected sizes."""
    ws = clib.dn_chunk_bwd_workspace_bytes
    slots = 4 * 2048 // 64 + 4
    assert ws(4, 4, 2048, 16, 16, 128, 128, dn.DN_BF16) == slots * 16 * (128 * 128 * 4 + 25088 + 3 * 64 * 64 * 4)
    assert ws(4, 4, 2048, 16, 16, 128, 128, dn.DN_F32) == slots * 16 * 128 * 128 * 4
    assert ws(4, 4, 2048, 16, 16, 64, 128, dn.DN_BF16) == slots * 16 * 64 * 128 * 4
    assert ws(3, 1, 300, 2, 8, 64, 32, dn.DN_F32) == (300 // 64 + 3) * 8 * 64 * 32 * 4
    assert ws(1, 1, 64, 1, 1, 256, 64, dn.DN_BF16) == 0
