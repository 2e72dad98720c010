"""GPU parity of the backward (dn_chunk_bwd, "flash-linear-attention 中 DeltaNet
的分块并行化WY 表示推导与 Triton 内核实现" §3.4 and §6: dq, dk, dv, dbeta, dh0, and
dg of the gated form) against the fp64 oracle's reverse pass, through the C
ABI.  The oracle's gradient is itself pinned by finite differences of the
forward definition (tests/test_oracle_pins.py).

Tolerance.  The reverse walk computes in fp32 from the same (exactly upcast)
inputs the oracle sees.  Where the chunk-start states come from the fp32
CUDA-core forward, the only error is fp32 rounding through the chunk algebra
and the cross-tile atomic sums: rel-L2 <= 1e-4 per gradient tensor (the fp32
forward bound) and max-abs <= 1e-3 * max(1, max |reference|).  For bf16 with
dk = 128 and dv a multiple of 128 the states come from the tensor-core
forward, as the page's backward recomputes them with its forward kernels
(§3.4); they carry that forward's bf16 operand rounding, so these cases take
the forward's bf16 bound, rel-L2 <= 5e-3, with max-abs <= 2e-2 * max(1, max
|reference|) (the page's own gradient checks allow 0.006-0.008, §6).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from conftest import cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

NAMES = ("dq", "dk", "dv", "dbeta", "dg", "dh0")


def inputs(B=2, T=150, Nk=2, Nv=2, dk=64, dv=64, dtype=torch.bfloat16, gate=3.0, h0=True,
           seed=0, lengths=None, dht=True, raw_qk=False):
    inp = workloads.make_inputs(B, T, Nk, Nv, dk, dv, dtype=dtype, gate_mu=gate, h0=h0,
                                seed=seed, lengths=lengths, raw_qk=raw_qk)
    gen = torch.Generator().manual_seed(seed + 99)
    inp["do"] = torch.randn(inp["v"].shape, generator=gen).to(dtype)
    N = inp["N"]
    inp["dht"] = torch.randn(N, Nv, dk, dv, generator=gen) if dht else None
    return inp


def run(inp):
    import chunkwise_gated_delta_chunk_gb300 as dn
    d = workloads.to_device(inp, "cuda")
    out = dn.chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["cu_seqlens"],
                       scale=inp["scale"], do=d["do"], dht=d["dht"],
                       use_qk_l2norm_in_kernel=inp.get("qk_l2norm", False))
    assert dn.dn_check() == dn.DN_OK
    return out


def tc_states(inp):
    """True where the backward's forward pass runs on the tensor cores."""
    dk, dv = inp["q"].shape[-1], inp["v"].shape[-1]
    return inp["q"].dtype == torch.bfloat16 and dk == 128 and dv % 128 == 0


def check(inp, out, groups=None, label=""):
    ref = oracle.recurrent_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["h0"],
                               inp["cu_seqlens"], inp["scale"], do=inp["do"], dht=inp["dht"],
                               groups=groups,
                               use_qk_l2norm_in_kernel=inp.get("qk_l2norm", False))
    res = {}
    for name in NAMES:
        if out[name] is None:
            continue
        got = out[name].detach().cpu().double().numpy()
        want = ref[name]
        mask = ~np.isnan(want)  # entries of the groups the oracle computed
        assert mask.any(), (label, name)
        g, w = got[mask], want[mask]
        assert np.isfinite(g).all(), (label, name)
        err = g - w
        rel = float(np.linalg.norm(err) / max(np.linalg.norm(w), 1e-30))
        mx = float(np.abs(err).max())
        res[name] = (mx, rel)
        rel_tol, max_tol = (5e-3, 2e-2) if tc_states(inp) else (1e-4, 1e-3)
        assert rel <= rel_tol, (label, name, mx, rel)
        assert mx <= max_tol * max(1.0, float(np.abs(w).max())), (label, name, mx, rel)
    print(label, {k: "%.1e / %.1e" % v for k, v in res.items()})
    return res


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 16, 16), (torch.bfloat16, 32, 64),
                                         (torch.bfloat16, 64, 64), (torch.bfloat16, 128, 128),
                                         (torch.bfloat16, 64, 256), (torch.bfloat16, 128, 32),
                                         (torch.float32, 64, 64), (torch.float32, 16, 32)])
def test_dims(lib, dtype, dk, dv):
    import chunkwise_gated_delta_chunk_gb300 as dn
    inp = inputs(dk=dk, dv=dv, dtype=dtype, seed=800 + dk + dv)
    out = run(inp)
    assert ("tc_fwd" in dn.dn_last_kernel()) == tc_states(inp), dn.dn_last_kernel()
    check(inp, out, label="bwd %s %dx%d" % (dtype, dk, dv))


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130])
def test_lengths(lib, T):
    inp = inputs(B=2, T=T, dk=128, dv=128, seed=820 + T)
    check(inp, run(inp), label="bwd T=%d" % T)


@pytest.mark.parametrize("nv_per_nk,d", [(1, 64), (4, 64), (2, 128)])
def test_varlen_gqa(lib, nv_per_nk, d):
    """Packed sequences (empty, length 1, one chunk, ragged) with value heads
    sharing a key head: dq and dk sum over those heads.  d = 128 takes the
    tensor-core forward for the states (its slots follow the packed layout)."""
    inp = inputs(B=1, Nk=2, Nv=2 * nv_per_nk, dk=d, dv=d, lengths=[1, 0, 64, 65, 130, 3],
                 seed=840 + nv_per_nk + d)
    check(inp, run(inp), label="bwd varlen r=%d d=%d" % (nv_per_nk, d))


@pytest.mark.parametrize("gate,h0,dht", [(None, False, False), (None, True, True),
                                         (3.0, False, True), (3.0, True, False)])
def test_optional_inputs(lib, gate, h0, dht):
    """No gate (dg is then the gradient at g = 0), no h0, no dht."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    inp = inputs(B=2, T=100, dk=64, dv=32, gate=gate, h0=h0, dht=dht, seed=860)
    d = workloads.to_device(inp, "cuda")
    out = run(inp)
    if gate is None:
        # dg at g = 0, asked for explicitly
        g0 = torch.zeros_like(d["beta"])
        full = dn.chunk_bwd(d["q"], d["k"], d["v"], d["beta"], g0, d["h0"], None,
                            scale=inp["scale"], do=d["do"], dht=d["dht"])
        assert dn.dn_check() == dn.DN_OK
        assert torch.allclose(full["dq"], out["dq"], rtol=1e-5, atol=1e-6)
        inp_g0 = dict(inp, g=g0.cpu())
        check(inp_g0, full, label="bwd g=0 explicit")
    check(inp, out, label="bwd gate=%s h0=%s dht=%s" % (gate, h0, dht))


def test_extreme_gates(lib):
    """Strong decay (g = -30 on some tokens) and no decay with beta = 1."""
    inp = inputs(B=1, T=130, dk=64, dv=64, seed=870)
    g = inp["g"].clone()
    g[:, ::7] = -30.0
    g[:, 1::5] = 0.0
    inp["g"] = g
    inp["beta"][:, 1::5] = 1.0
    check(inp, run(inp), label="bwd extreme gates")


def test_headline_sampled_groups(lib):
    """The headline shapes (B=4, H=16, T=2048, d=128, bf16) at full size;
    the oracle computes three (sequence, key head) groups."""
    inp = inputs(B=4, T=2048, Nk=16, Nv=16, dk=128, dv=128, seed=880)
    out = run(inp)
    res = check(inp, out, groups=[0, 37, 63], label="bwd headline")
    for name in ("dq", "dk", "dv", "dbeta", "dg"):
        assert torch.isfinite(out[name]).all()
    print(res)


def test_repeatable(lib):
    """Two calls agree to fp32 rounding (the cross-tile sums are atomic)."""
    inp = inputs(B=2, T=200, Nk=1, Nv=2, dk=128, dv=128, seed=890)
    a, b = run(inp), run(inp)
    for name in NAMES:
        assert torch.allclose(a[name], b[name], rtol=1e-5, atol=1e-5), name
    assert torch.equal(a["dv"], b["dv"]) and torch.equal(a["dh0"], b["dh0"])


@pytest.mark.parametrize("dtype,dk,dv,lengths", [(torch.bfloat16, 128, 128, None),
                                                 (torch.float32, 64, 32, None),
                                                 (torch.bfloat16, 64, 64, [1, 0, 64, 65, 130])])
def test_qk_l2norm(lib, dtype, dk, dv, lengths):
    """DN_QK_L2NORM: the gradient of the forward that normalises raw q / k rows
    in the kernels; dq and dk go back through the normalisation."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    if lengths is None:
        inp = inputs(B=2, T=150, dk=dk, dv=dv, dtype=dtype, seed=900 + dk, raw_qk=True)
    else:
        inp = inputs(B=1, Nk=2, Nv=4, dk=dk, dv=dv, dtype=dtype, lengths=lengths, seed=905,
                     raw_qk=True)
    out = run(inp)
    assert dn.dn_last_kernel().endswith("l2norm_bwd_rows<%s>" % ("bf16" if dtype == torch.bfloat16
                                                                 else "f32"))
    check(inp, out, label="bwd l2norm %s %dx%d" % (dtype, dk, dv))
