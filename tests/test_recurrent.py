"""GPU parity of the token-serial entry point (dn_recurrent_fwd, "flash linear
attention" notes, Attention: fused recurrent forward) against the fp64
oracle, through the C ABI: decoding steps with a carried state, short
prompts, varlen and GQA batches, every head size and both dtypes."""
import pytest
import torch

import workloads
from conftest import cuda_ok
from parity_util import TOL, check

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


def inputs(B=2, T=5, Nk=2, Nv=2, dk=128, dv=128, dtype=torch.bfloat16, gate=3.0, h0=True, seed=0,
           lengths=None):
    return workloads.make_inputs(B, T, Nk, Nv, dk, dv, dtype=dtype, gate_mu=gate, h0=h0, seed=seed,
                                 lengths=lengths)


def run(inp, output_final_state=True):
    import chunkwise_gated_delta_chunk_gb300 as dn
    d = workloads.to_device(inp, "cuda")
    o, ht = dn.recurrent_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["cu_seqlens"],
                             scale=inp["scale"], output_final_state=output_final_state,
                             use_qk_l2norm_in_kernel=inp.get("qk_l2norm", False))
    assert dn.dn_check() == dn.DN_OK
    return o, ht


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("dk,dv", [(16, 16), (64, 32), (128, 128), (256, 64), (64, 256)])
def test_dims(lib, dtype, dk, dv):
    inp = inputs(T=37, dk=dk, dv=dv, dtype=dtype, seed=500 + dk + dv)
    o, ht = run(inp)
    check(inp, o, ht, label="rec %s %dx%d" % (dtype, dk, dv))


@pytest.mark.parametrize("T", [1, 2, 64, 65])
def test_lengths(lib, T):
    inp = inputs(B=3, T=T, seed=510 + T)
    o, ht = run(inp)
    check(inp, o, ht, label="rec T=%d" % T)


def test_decode_steps_chain(lib):
    """Eight single-token calls, each from the previous call's ht, equal one
    eight-token call."""
    inp = inputs(B=4, T=8, Nk=2, Nv=4, seed=520)
    o_all, ht_all = run(inp)
    h = inp["h0"]
    outs = []
    for t in range(8):
        step = dict(inp)
        for key in ("q", "k", "v", "beta", "g"):
            step[key] = inp[key][:, t:t + 1].contiguous()
        step["h0"] = h
        o, ht = run(step)
        outs.append(o)
        h = ht.cpu()
    tol = TOL[torch.bfloat16]
    assert (torch.cat(outs, 1).float() - o_all.float()).abs().max().item() <= tol["max_abs"]
    assert (h.cuda() - ht_all).abs().max().item() <= tol["max_abs"]
    check(inp, o_all, ht_all, label="rec chain")


@pytest.mark.parametrize("nv_per_nk", [1, 4])
def test_varlen_gqa(lib, nv_per_nk):
    inp = inputs(B=1, Nk=2, Nv=2 * nv_per_nk, lengths=[1, 0, 17, 64, 3], seed=530 + nv_per_nk)
    o, ht = run(inp)
    check(inp, o, ht, label="rec varlen r=%d" % nv_per_nk)


@pytest.mark.parametrize("gate,h0,final", [(None, False, True), (3.0, True, False)])
def test_optional_inputs(lib, gate, h0, final):
    inp = inputs(T=20, gate=gate, h0=h0, seed=540)
    o, ht = run(inp, output_final_state=final)
    assert (ht is None) == (not final)
    check(inp, o, ht, label="rec gate=%s h0=%s" % (gate, h0))


def test_matches_chunk_path(lib):
    """On a 300-token input the token-serial and the chunk (tensor-core) paths
    agree to the bf16 tolerance."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    inp = inputs(B=2, T=300, seed=550)
    d = workloads.to_device(inp, "cuda")
    o1, h1 = run(inp)
    o2, h2 = dn.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], None, scale=inp["scale"])
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (h1 - h2).abs().max().item() <= 2e-2


def test_decode_workload_full_size(lib):
    """The decoding-step workload (64 sequences x 16 heads, T = 1, state in and
    out) in the configuration bench.py --mode recurrent times: every output."""
    inp = workloads.workload_inputs("gdn_decode_bf16_b64_h16_t1_d128")
    o, ht = run(inp)
    check(inp, o, ht, label="decode")
