"""dn_chunk_fwd_noalloc: the forward for callers that cannot allocate device
memory where they run it (a plugin host whose execute path may not allocate,
or a runtime whose device memory is all committed to its own pool).  It takes
no workspace and uses the library's fixed scratch array instead.

This file is collected last on purpose, so that a stop-at-first-failure run
has already run every other test when it gets here.
"""
import pytest
import torch

import workloads
from conftest import cuda_ok
from parity_util import TOL, metrics

A = 1 << 20  # fake, 16-byte aligned device address: rejected before any use


@pytest.mark.gpu
@pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")
def test_noalloc_matches_workspace_entry_point(lib):
    """Two calls in a row through the C ABI agree with dn_chunk_fwd (given a
    torch-allocated workspace) within the parity tolerance."""
    dn = lib
    inp = workloads.make_inputs(1, 0, 2, 4, 128, 128, dtype=torch.bfloat16, gate_mu=3.0, h0=True,
                                seed=900, lengths=[300, 64, 1, 0, 129, 2000])
    d = workloads.to_device(inp, "cuda")
    B, T, Nk, dk = d["q"].shape
    Nv, dv = d["v"].shape[2], d["v"].shape[3]
    N = inp["N"]
    o_ref, ht_ref = dn.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                 d["cu_seqlens"], scale=inp["scale"])
    assert dn.dn_check() == dn.DN_OK
    tol = TOL[torch.bfloat16]
    for call in range(2):
        o = torch.full_like(o_ref, float("nan"))
        ht = torch.full_like(ht_ref, float("nan"))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        st = dn.dn_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                     d["cu_seqlens"], N, B, T, Nk, Nv, dk, dv, dn.DN_BF16,
                                     inp["scale"], 64, o, ht)
        assert st == dn.DN_OK, dn.dn_status_str(st)
        assert dn.dn_check() == dn.DN_OK
        if call == 1:
            # the array was reserved by the first call; the second takes no
            # device memory at all
            assert torch.cuda.mem_get_info()[0] == free_before
        for got, ref in ((o, o_ref), (ht, ht_ref)):
            m = metrics(got.cpu().double().numpy(), ref.cpu().double().numpy())
            assert m["max_abs"] <= tol["max_abs"] and m["rel_l2"] <= tol["rel_l2"], m


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Sizes that need more than the fixed scratch are refused on the host,
    before anything is launched (no GPU needed)."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    dn.load()
    Nv = 16
    slots = dn.DN_NOALLOC_SCRATCH_BYTES // (25088 * Nv)  # whole slots per value head that fit
    T = slots * 64  # floor(T / 64) + N = slots + 1 slots: one too many
    assert dn.dn_chunk_fwd_workspace_bytes(1, 1, T, Nv, Nv, 128, 128, dn.DN_BF16) > \
        dn.DN_NOALLOC_SCRATCH_BYTES
    st = dn.dn_chunk_fwd_noalloc(A, A, A, A, None, None, None, 1, 1, T, Nv, Nv, 128, 128,
                                 dn.DN_BF16, 0.0, 64, A, None, 0)
    assert st == dn.DN_ERR_UNSUPPORTED
    # one chunk fewer fits
    assert dn.dn_chunk_fwd_workspace_bytes(1, 1, T - 64, Nv, Nv, 128, 128, dn.DN_BF16) <= \
        dn.DN_NOALLOC_SCRATCH_BYTES


def test_noalloc_checks_arguments_before_sizes():
    """A bad argument is reported as DN_ERR_INVALID_ARG even when the sizes
    would also exceed the scratch array (no GPU needed: nothing launches)."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    dn.load()
    Nv = 16
    T = 1 << 20  # far beyond the scratch array
    assert dn.dn_chunk_fwd_workspace_bytes(1, 1, T, Nv, Nv, 128, 128, dn.DN_BF16) > \
        dn.DN_NOALLOC_SCRATCH_BYTES
    bad = [
        # Nv not a multiple of Nk
        dict(Nk=3),
        # cu_seqlens given with B != 1
        dict(cu=A, B=2, n_seqs=2),
        # a pointer that is not 16-byte aligned
        dict(q=A + 8),
        # a required pointer missing
        dict(v=None),
    ]
    for over in bad:
        a = dict(q=A, k=A, v=A, beta=A, cu=None, n_seqs=1, B=1, Nk=Nv)
        a.update(over)
        st = dn.dn_chunk_fwd_noalloc(a["q"], a["k"], a["v"], a["beta"], None, None, a["cu"],
                                     a["n_seqs"], a["B"], T, a["Nk"], Nv, 128, 128, dn.DN_BF16,
                                     0.0, 64, A, None, 0)
        assert st == dn.DN_ERR_INVALID_ARG, (over, dn.dn_status_str(st))
