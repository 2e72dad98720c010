"""Bounded waits of the tensor-core kernels, exercised.

Every mbarrier wait of the WY and scan kernels gives up after a time limit:
the CTA records a timeout in the status word, stops its other roles, waits
for its own copies and MMAs in flight, frees its tensor memory and returns, so
the context stays usable and dn_check reports DN_ERR_TIMEOUT.

These tests use the failure-path build of the library (compiled with
-DDN_TEST_STALL into _build/stall/, never the library's own build): its wait
limit is 2 ms and it has a hook, dn_test_stall_next, that makes one wait of
the next call run out
  1: the scan kernel's first chunk never becomes ready (dk = 128: its first
     stage never receives its second arrival; dk = 256: its gate scalars are
     never announced);
  2: the WY kernel's first item on one CTA expects 16 bytes more than its
     copies bring.
In both cases the bytes that were requested still land before the kernel
returns.  The call must end with DN_ERR_TIMEOUT, and the next call must be
bit-identical to a clean call made before.
"""
import contextlib

import pytest
import torch

import workloads
from conftest import cuda_ok
from parity_util import check

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


@contextlib.contextmanager
def stall_build():
    """The binding's functions, routed to the failure-path build."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    from chunkwise_gated_delta_chunk_gb300 import _build
    dn.load()
    lib = dn.load(_build.build_stall_variant())
    import ctypes
    lib.dn_test_stall_next.argtypes = [ctypes.c_uint]
    lib.dn_test_stall_next.restype = None
    saved = dn._lib
    dn._lib = lib
    try:
        yield dn, lib
    finally:
        dn._lib = saved


@pytest.mark.parametrize("mode,where,dk", [(1, "scan", 128), (2, "wy", 128), (1, "scan", 256), (2, "wy", 256)])
def test_wait_runs_out_then_next_call_is_clean(mode, where, dk):
    inp = workloads.make_inputs(2, 200, 2, 2, dk, 128, gate_mu=3.0, h0=True, seed=600 + mode + dk)
    d = workloads.to_device(inp, "cuda")
    with stall_build() as (dn, lib):
        def call():
            o, ht = dn.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], None,
                                 scale=inp["scale"])
            return o, ht, dn.dn_check()

        o_ref, ht_ref, st = call()
        assert st == dn.DN_OK, dn.dn_status_str(st)
        assert dn.dn_last_kernel() == ("wy_fwd+tc_fwd" if dk == 128 else "wy_fwd+tc_wide_fwd")
        lib.dn_test_stall_next(mode)
        _, _, st = call()
        assert st == dn.DN_ERR_TIMEOUT, (where, dn.dn_status_str(st))
        o2, ht2, st = call()
        assert st == dn.DN_OK, (where, dn.dn_status_str(st))
        assert torch.equal(o2, o_ref) and torch.equal(ht2, ht_ref), where
    # and the clean result is the recurrence's
    check(inp, o_ref, ht_ref, label="stall build, clean call")

