"""GPU parity of in-kernel q / k L2 normalisation (DN_QK_L2NORM, the pages'
use_qk_l2norm_in_kernel, "flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导
与 Triton 内核实现" §5 and §6) against the fp64 oracle with the same option:
raw q and k whose row norms spread over about a factor of e, on the
tensor-core path, the CUDA-core kernel (chunk 16 / 32 / 64, fp32 and bf16)
and the token-serial kernel, through the C ABI."""
import pytest
import torch

import workloads
from conftest import cuda_ok
from parity_util import check, run_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


def inputs(B=2, T=150, Nk=2, Nv=2, dk=128, dv=128, dtype=torch.bfloat16, gate=3.0, h0=True,
           seed=0, lengths=None):
    return workloads.make_inputs(B, T, Nk, Nv, dk, dv, dtype=dtype, gate_mu=gate, h0=h0,
                                 seed=seed, lengths=lengths, raw_qk=True)


def run_rec(inp):
    import chunkwise_gated_delta_chunk_gb300 as dn
    d = workloads.to_device(inp, "cuda")
    o, ht = dn.recurrent_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["cu_seqlens"],
                             scale=inp["scale"], use_qk_l2norm_in_kernel=True)
    assert dn.dn_check() == dn.DN_OK
    return o, ht


@pytest.mark.parametrize("dv", [128, 256])
def test_tensor_core_path(lib, dv):
    """bf16, dk = 128, chunk 64: the WY + scan kernels, ragged tails."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    inp = inputs(B=2, T=300, dv=dv, seed=700 + dv)
    o, ht = run_gpu(inp)
    assert dn.dn_last_kernel() == "wy_fwd+tc_fwd"
    check(inp, o, ht, label="tc l2norm dv=%d" % dv)


@pytest.mark.parametrize("nv_per_nk", [1, 4])
def test_tensor_core_varlen_gqa(lib, nv_per_nk):
    """Packed sequences (empty, length 1, chunk-aligned, ragged) with shared
    key heads: the norms follow the key head, the slots the value head."""
    inp = inputs(B=1, Nk=2, Nv=2 * nv_per_nk, lengths=[1, 0, 64, 65, 130, 3],
                 seed=710 + nv_per_nk)
    o, ht = run_gpu(inp)
    check(inp, o, ht, label="tc l2norm varlen r=%d" % nv_per_nk)


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("dtype,dk,dv", [(torch.float32, 64, 64), (torch.bfloat16, 128, 128),
                                         (torch.bfloat16, 256, 64), (torch.float32, 16, 32)])
def test_cuda_core_path(lib, chunk, dtype, dk, dv):
    """The CUDA-core kernel (every shape the tensor-core path does not take,
    and chunk 16 / 32)."""
    if chunk == 64 and dtype == torch.bfloat16 and dk == 128:
        pytest.skip("tensor-core path, covered above")
    inp = inputs(B=2, T=150, dk=dk, dv=dv, dtype=dtype, seed=720 + chunk + dk + dv)
    o, ht = run_gpu(inp, chunk=chunk)
    check(inp, o, ht, label="simt l2norm C=%d %s %dx%d" % (chunk, dtype, dk, dv))


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.float32, 16, 16),
                                         (torch.bfloat16, 256, 64), (torch.float32, 64, 256)])
def test_recurrent_path(lib, dtype, dk, dv):
    inp = inputs(B=2, T=37, dk=dk, dv=dv, dtype=dtype, seed=740 + dk + dv)
    o, ht = run_rec(inp)
    check(inp, o, ht, label="rec l2norm %s %dx%d" % (dtype, dk, dv))
    inp = inputs(B=1, Nk=2, Nv=4, dk=dk, dv=dv, dtype=dtype, lengths=[1, 0, 17, 3],
                 seed=750 + dk + dv)
    o, ht = run_rec(inp)
    check(inp, o, ht, label="rec l2norm varlen %s %dx%d" % (dtype, dk, dv))


def test_power_of_two_row_scales_change_nothing(lib):
    """Multiplying q and k rows by powers of two (exact in bf16) leaves the
    normalised forward unchanged, on the tensor-core path and the token-serial
    kernel."""
    inp = inputs(B=2, T=200, seed=760)
    gen = torch.Generator().manual_seed(760)
    e = lambda x: torch.pow(2.0, torch.randint(-6, 7, x.shape[:-1] + (1,), generator=gen).float())
    scaled = dict(inp, q=(inp["q"].float() * e(inp["q"])).to(inp["q"].dtype),
                  k=(inp["k"].float() * e(inp["k"])).to(inp["k"].dtype))
    for runner in (run_gpu, run_rec):
        o1, h1 = runner(inp)
        o2, h2 = runner(scaled)
        assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
        assert (h1 - h2).abs().max().item() <= 1e-4


def test_flag_off_differs(lib):
    """The option is not a no-op: on raw q / k the unnormalised forward is a
    different function (guards against the flag being dropped on the way)."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    inp = inputs(B=1, T=130, seed=770)
    d = workloads.to_device(inp, "cuda")
    o1, _ = run_gpu(inp)
    o2, _ = dn.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], None,
                         scale=inp["scale"])
    assert dn.dn_check() == dn.DN_OK
    # (raw keys of norm ~ 11 may well make the unnormalised recurrence blow up)
    assert not torch.allclose(o1.float(), o2.float(), rtol=0, atol=0.1)
