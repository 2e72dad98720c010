"""GPU parity: the CUDA path (called through the C ABI) against the fp64 oracle,
element by element on the same seeded inputs.

Small cases compare every output and span several chunks plus a ragged tail;
the named full-size workloads compare every output of sampled (sequence,
value-head) units, which the oracle computes one by one, in the same launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import workloads
from conftest import cuda_ok
from parity_util import TOL, check, run_gpu

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


def inputs(B=2, T=130, Nk=2, Nv=2, dk=64, dv=64, dtype=torch.bfloat16, gate=3.0, h0=True,
           seed=0, lengths=None, **kw):
    return workloads.make_inputs(B, T, Nk, Nv, dk, dv, dtype=dtype, gate_mu=gate, h0=h0,
                                 seed=seed, lengths=lengths, **kw)


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 64), (64, 64), (64, 128), (128, 64),
                                   (128, 128), (256, 128), (128, 256), (256, 256)])
def test_dims_bf16(lib, dk, dv):
    inp = inputs(dk=dk, dv=dv, seed=dk + dv)
    o, ht = run_gpu(inp)
    check(inp, o, ht, label="bf16 %dx%d" % (dk, dv))


@pytest.mark.parametrize("dk,dv", [(16, 16), (64, 32), (64, 64), (128, 128)])
def test_dims_fp32(lib, dk, dv):
    inp = inputs(dk=dk, dv=dv, dtype=torch.float32, seed=7 + dk)
    o, ht = run_gpu(inp)
    check(inp, o, ht, label="f32 %dx%d" % (dk, dv))


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 129, 200])
def test_lengths(lib, T):
    inp = inputs(B=3, T=T, dk=128, dv=128, seed=100 + T)
    o, ht = run_gpu(inp)
    check(inp, o, ht, label="T=%d" % T)


@pytest.mark.parametrize("chunk", [16, 32])
@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.bfloat16, 64, 256),
                                         (torch.float32, 64, 64)])
def test_chunk_sizes(lib, chunk, dtype, dk, dv):
    """C = 16 and 32 ([WY] §5 chunk_size) give the recurrence's result: ragged
    tails, a varlen GQA batch with empty and length-1 sequences."""
    inp = inputs(B=2, T=150, dk=dk, dv=dv, dtype=dtype, seed=400 + chunk + dk)
    o, ht = run_gpu(inp, chunk=chunk)
    check(inp, o, ht, label="C=%d %s %dx%d" % (chunk, dtype, dk, dv))
    inp = inputs(B=1, Nk=2, Nv=4, dk=dk, dv=dv, dtype=dtype, lengths=[1, 0, 33, 64, 97],
                 seed=450 + chunk + dk)
    o, ht = run_gpu(inp, chunk=chunk)
    check(inp, o, ht, label="C=%d varlen" % chunk)


@pytest.mark.parametrize("chunk", [16, 32])
def test_chunk_sizes_tensor_core_path(lib, chunk):
    """bf16 with dk = 128 runs C = 16 and 32 on the tensor-core kernels (a chunk
    fills the first C rows of their 64-row tiles): extreme gates, many short
    packed sequences, in-kernel q / k normalisation, and dv = 256."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    cases = []
    inp = inputs(B=2, T=150, dk=128, dv=128, seed=470 + chunk)
    inp["g"] = torch.full_like(inp["g"], -30.0)
    cases.append(("g=-30", inp))
    inp = inputs(B=2, T=150, dk=128, dv=128, seed=471 + chunk)
    inp["g"] = torch.zeros_like(inp["g"])
    inp["beta"] = torch.ones_like(inp["beta"])
    cases.append(("g=0 beta=1", inp))
    cases.append(("many short", inputs(B=1, Nk=2, Nv=4, dk=128, dv=128, seed=472 + chunk,
                                       lengths=[16, 15, 17, 1, 0, 33, 31, 64, 65, 2, 130])))
    cases.append(("qk l2norm", inputs(B=2, T=140, dk=128, dv=128, seed=473 + chunk, raw_qk=True)))
    cases.append(("dv=256 no gate", inputs(B=1, T=200, dk=128, dv=256, gate=None, seed=474 + chunk)))
    for label, inp in cases:
        o, ht = run_gpu(inp, chunk=chunk)
        assert dn.dn_last_kernel().startswith("wy_fwd"), dn.dn_last_kernel()
        check(inp, o, ht, label="C=%d %s" % (chunk, label))


@pytest.mark.parametrize("chunk", [16, 32])
def test_chunk_sizes_wide_heads(lib, chunk):
    """dk = dv = 256 at C = 16 and 32 on the wide tensor-core kernels, whose WY
    items then hold two or four chunks of a 64-token tile: ragged tails, a
    varlen GQA batch of short sequences, extreme gates, in-kernel q / k
    normalisation."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    cases = [("ragged", inputs(B=2, T=150, dk=256, dv=256, seed=480 + chunk)),
             ("varlen gqa", inputs(B=1, Nk=1, Nv=2, dk=256, dv=256, seed=481 + chunk,
                                   lengths=[16, 1, 0, 33, 97, 64, 15])),
             ("qk l2norm", inputs(B=1, T=140, dk=256, dv=256, seed=482 + chunk, raw_qk=True))]
    inp = inputs(B=1, T=100, dk=256, dv=256, seed=483 + chunk)
    inp["g"] = torch.full_like(inp["g"], -30.0)
    cases.append(("g=-30", inp))
    for label, inp in cases:
        o, ht = run_gpu(inp, chunk=chunk)
        assert dn.dn_last_kernel() == "wy_fwd+tc_wide_fwd", dn.dn_last_kernel()
        check(inp, o, ht, label="C=%d dk=dv=256 %s" % (chunk, label))


@pytest.mark.parametrize("chunk", [16, 32])
def test_chunk_sizes_headline_full_size(lib, chunk):
    """The headline shapes (B = 4, H = 16, T = 2048, d = 128) at C = 16 and 32,
    on sampled (sequence, head) units, in the launch configuration the
    benchmark times with --chunk."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    inp = workloads.workload_inputs("gdn_bf16_b4_h16_t2048_d128")
    o, ht = run_gpu(inp, chunk=chunk)
    assert dn.dn_last_kernel().startswith("wy_fwd"), dn.dn_last_kernel()
    res = check(inp, o, ht, units=[0, 21, 63], label="headline C=%d" % chunk)
    print("headline C=%d" % chunk, res)


@pytest.mark.parametrize("case", ["gated_h0", "varlen_gqa", "ungated", "chunk16", "chunk32",
                                  "qk_l2norm", "dv256"])
def test_wide_heads_tensor_core_path(lib, case):
    """dk = 256 (bf16) runs on the tensor-core kernels, with -W^T formed by
    the WY kernel: several chunks and a ragged tail, a varlen GQA batch with
    empty and length-1 sequences, no gates, the shorter chunks, in-kernel q / k
    normalisation and two value tiles per head."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    chunk = {"chunk16": 16, "chunk32": 32}.get(case, 64)
    if case == "varlen_gqa":
        inp = inputs(B=1, Nk=2, Nv=4, dk=256, dv=128, lengths=[1, 0, 65, 200, 64, 130], seed=520)
    elif case == "ungated":
        inp = inputs(B=2, T=300, dk=256, dv=128, gate=None, seed=521)
    elif case == "qk_l2norm":
        inp = inputs(B=2, T=150, dk=256, dv=128, seed=522, raw_qk=True)
    elif case == "dv256":
        inp = inputs(B=2, T=190, dk=256, dv=256, seed=523)
    else:
        inp = inputs(B=2, T=200, dk=256, dv=128, seed=524 + chunk)
    o, ht = run_gpu(inp, chunk=chunk)
    assert dn.dn_last_kernel() == "wy_fwd+tc_wide_fwd", dn.dn_last_kernel()
    check(inp, o, ht, label="wide %s" % case)


@pytest.mark.parametrize("case", ["chunk16", "chunk32", "ungated", "qk_l2norm", "varlen_gqa"])
def test_wide_heads_full_size(lib, case):
    """The wide-head shapes (B = 8, H = 8, T = 8192, d = 256) in the modes of
    the smaller tests: the shorter chunks, no gates, in-kernel q / k
    normalisation, and a varlen GQA batch with long and short sequences; on
    sampled (sequence, head) units."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    chunk = {"chunk16": 16, "chunk32": 32}.get(case, 64)
    if case == "varlen_gqa":
        inp = workloads.make_inputs(1, 0, 4, 8, 256, 256, gate_mu=3.0, h0=True, seed=530,
                                    lengths=[8192, 1, 3000, 64, 12289, 0, 700, 4097])
        units = [4 * 8 + 0, 4 * 8 + 7, 1 * 8 + 3, 2 * 8 + 5]
    else:
        inp = workloads.make_inputs(8, 8192, 8, 8, 256, 256, gate_mu=None if case == "ungated" else 3.0,
                                    h0=True, seed=531, raw_qk=case == "qk_l2norm")
        units = [0, 37, 63]
    o, ht = run_gpu(inp, chunk=chunk)
    assert dn.dn_last_kernel() == "wy_fwd+tc_wide_fwd", dn.dn_last_kernel()
    res = check(inp, o, ht, units=units, label="wide full %s" % case)
    assert torch.isfinite(o.float()).all() and torch.isfinite(ht).all()
    print("wide full", case, res)


def test_wide_heads_state_carry(lib):
    """dk = 256: a second call from the first call's ht equals one call on the
    whole sequence."""
    inp = inputs(B=2, T=300, dk=256, dv=128, seed=525)
    o, ht = run_gpu(inp)
    cut = 100
    p1, p2 = dict(inp), dict(inp)
    for key in ("q", "k", "v", "beta", "g"):
        p1[key] = inp[key][:, :cut].contiguous()
        p2[key] = inp[key][:, cut:].contiguous()
    o1, h1 = run_gpu(p1)
    p2["h0"] = h1.cpu()
    o2, h2 = run_gpu(p2)
    both = torch.cat([o1, o2], dim=1).float()
    tol = TOL[torch.bfloat16]
    assert (both - o.float()).abs().max().item() <= tol["max_abs"]
    assert (h2 - ht).abs().max().item() <= tol["max_abs"]


def test_chunk_sizes_agree(lib):
    """The same inputs at C = 16, 32 and 64 agree with each other to the
    rounding of the two paths (the chunk form is exact, [WY] §6)."""
    inp = inputs(B=2, T=300, dk=128, dv=128, seed=460)
    outs = [run_gpu(inp, chunk=c) for c in (16, 32, 64)]
    for (o, ht) in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= 2e-2
        assert (ht - outs[0][1]).abs().max().item() <= 2e-2


@pytest.mark.parametrize("nv_per_nk", [1, 2, 4])
def test_varlen_gqa(lib, nv_per_nk):
    lengths = [1, 63, 64, 65, 0, 200, 128, 3]
    inp = inputs(B=1, Nk=2, Nv=2 * nv_per_nk, dk=128, dv=128, lengths=lengths,
                 seed=200 + nv_per_nk)
    o, ht = run_gpu(inp)
    check(inp, o, ht, label="varlen r=%d" % nv_per_nk)


@pytest.mark.parametrize("gate,h0,final", [(None, False, True), (None, True, True),
                                           (3.0, False, True), (3.0, True, False)])
def test_optional_inputs(lib, gate, h0, final):
    inp = inputs(dk=128, dv=128, gate=gate, h0=h0, seed=300)
    o, ht = run_gpu(inp, output_final_state=final)
    assert (ht is None) == (not final)
    check(inp, o, ht, label="gate=%s h0=%s" % (gate, h0))


@pytest.mark.parametrize("dv,h0", [(128, False), (128, True), (256, False), (256, True)])
def test_ungated_long_bf16(lib, dv, h0):
    """Plain DeltaNet (g = NULL, [WY] §1) in bf16 at T = 8192 on the tensor-core
    path: without gates the state never forgets, so rounding error is not
    damped and this is the case closest to the bf16 bound."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    inp = inputs(B=1, T=8192, Nk=2, Nv=2, dk=128, dv=dv, gate=None, h0=h0, seed=320 + dv + h0)
    o, ht = run_gpu(inp)
    assert dn.dn_last_kernel().startswith("wy_fwd")
    res = check(inp, o, ht, label="ungated T=8192 dv=%d h0=%s" % (dv, h0))
    print("ungated T=8192 dv=%d h0=%s" % (dv, h0), res)


def test_ungated_long_varlen_gqa_bf16(lib):
    """Plain DeltaNet, packed GQA batch with sequences longer than 4096."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    inp = inputs(B=1, Nk=2, Nv=4, dk=128, dv=128, gate=None, h0=True,
                 lengths=[5000, 1, 8200, 4097, 63], seed=330)
    o, ht = run_gpu(inp)
    assert dn.dn_last_kernel().startswith("wy_fwd")
    res = check(inp, o, ht, label="ungated varlen GQA")
    print("ungated varlen GQA", res)


def test_custom_scale(lib):
    inp = inputs(dk=128, dv=128, seed=301)
    inp["scale"] = 0.37
    o, ht = run_gpu(inp)
    check(inp, o, ht, label="scale")


@pytest.mark.parametrize("dk", [128, 256])
def test_extreme_gates(lib, dk):
    """Very strong decay (e^g ~ 1e-13 per token), no decay, and beta = 1;
    for dk = 256 also a weak decay over many chunks, which the wide kernel
    carries as a running product (renormalised when it leaves [2^-40, 2^40])."""
    inp = inputs(dk=dk, dv=128, seed=302, T=150)
    inp["g"] = torch.full_like(inp["g"], -30.0)
    o, ht = run_gpu(inp)
    check(inp, o, ht, label="g=-30")
    inp = inputs(dk=dk, dv=128, seed=303, T=150)
    inp["g"] = torch.zeros_like(inp["g"])
    inp["beta"] = torch.ones_like(inp["beta"])
    o, ht = run_gpu(inp)
    check(inp, o, ht, label="g=0 beta=1")
    inp = inputs(dk=dk, dv=128, seed=304, T=150)
    inp["g"] = -torch.rand(inp["g"].shape, generator=torch.Generator().manual_seed(9)) * 4.0
    o, ht = run_gpu(inp)
    check(inp, o, ht, label="g~U(-4,0)")
    if dk == 256:
        # e^{G_L} ~ e^-0.6 per chunk: the product crosses 2^-40 after ~45 chunks
        inp = inputs(B=1, dk=dk, dv=128, seed=305, T=64 * 120 + 17)
        inp["g"] = torch.full_like(inp["g"], -0.01)
        o, ht = run_gpu(inp)
        check(inp, o, ht, label="g=-0.01 long")
        # strong and weak chunks alternating
        inp = inputs(B=1, dk=dk, dv=128, seed=306, T=64 * 12)
        g = torch.full_like(inp["g"], -0.02)
        g[:, 64 * 3:64 * 4] = -2.0
        g[:, 64 * 7:64 * 8] = -30.0
        inp["g"] = g
        o, ht = run_gpu(inp)
        check(inp, o, ht, label="g mixed")


def test_state_carry(lib):
    """Second call from the first call's ht equals one call on the whole."""
    inp = inputs(B=2, T=300, dk=128, dv=128, seed=305)
    o, ht = run_gpu(inp)
    cut = 100
    p1, p2 = dict(inp), dict(inp)
    for key in ("q", "k", "v", "beta", "g"):
        p1[key] = inp[key][:, :cut].contiguous()
        p2[key] = inp[key][:, cut:].contiguous()
    o1, h1 = run_gpu(p1)
    p2["h0"] = h1.cpu()
    o2, h2 = run_gpu(p2)
    both = torch.cat([o1, o2], dim=1).float()
    tol = TOL[torch.bfloat16]
    assert (both - o.float()).abs().max().item() <= tol["max_abs"]
    assert (h2 - ht).abs().max().item() <= tol["max_abs"]


def test_deterministic(lib):
    inp = inputs(dk=128, dv=128, seed=306, T=257)
    o1, h1 = run_gpu(inp)
    o2, h2 = run_gpu(inp)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_guard_regions_untouched(lib):
    """The kernel writes exactly o and ht: sentinels around them survive."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    inp = inputs(B=2, T=70, dk=128, dv=128, seed=307)
    d = workloads.to_device(inp, "cuda")
    n_o = d["v"].numel()
    n_h = 2 * 2 * 128 * 128
    o_buf = torch.full((n_o + 4096,), 12345.0, dtype=torch.bfloat16, device="cuda")
    h_buf = torch.full((n_h + 4096,), -777.0, dtype=torch.float32, device="cuda")
    o = o_buf[:n_o].view_as(d["v"])
    ht = h_buf[:n_h].view(2, 2, 128, 128)
    dn.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], None, o=o, ht=ht,
                 scale=inp["scale"])
    torch.cuda.synchronize()
    assert bool((o_buf[n_o:] == 12345.0).all()) and bool((h_buf[n_h:] == -777.0).all())
    check(inp, o, ht, label="guards")


def test_workspace_bounds_and_contents(lib):
    """The WY kernel writes inside the queried workspace size only, and the
    result does not depend on what the workspace held before the call."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    inp = inputs(B=1, Nk=2, Nv=4, dk=128, dv=128, lengths=[64, 1, 130, 0, 65], seed=311)
    d = workloads.to_device(inp, "cuda")
    nbytes = dn.workspace_for(d["q"], d["v"], inp["N"]).numel()
    buf = torch.full((nbytes + 65536,), 0xA5, dtype=torch.uint8, device="cuda")
    o1, h1 = dn.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["cu_seqlens"],
                          scale=inp["scale"], workspace=buf[:nbytes])
    assert dn.dn_check() == dn.DN_OK
    assert bool((buf[nbytes:] == 0xA5).all())
    buf[:nbytes].fill_(0xFF)  # NaN bit patterns everywhere
    o2, h2 = dn.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["cu_seqlens"],
                          scale=inp["scale"], workspace=buf[:nbytes])
    assert dn.dn_check() == dn.DN_OK
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    check(inp, o1, h1, label="workspace")


def test_varlen_many_short(lib):
    """Many sequences, aligned and ragged, packed: every chunk keeps its own
    workspace slot."""
    lengths = [64, 64, 64, 1, 1, 1, 1, 1, 130, 0, 0, 65, 127, 63, 2, 256]
    inp = inputs(B=1, Nk=2, Nv=4, dk=128, dv=128, lengths=lengths, seed=312)
    o, ht = run_gpu(inp)
    check(inp, o, ht, label="many short")


def test_empty_sequences_keep_h0(lib):
    inp = inputs(B=1, dk=128, dv=128, lengths=[0, 5, 0], seed=308)
    o, ht = run_gpu(inp)
    assert torch.equal(ht[0].cpu(), inp["h0"][0]) and torch.equal(ht[2].cpu(), inp["h0"][2])
    check(inp, o, ht, label="empty")


def test_zero_tokens(lib):
    inp = inputs(B=2, T=0, dk=64, dv=64, seed=309)
    o, ht = run_gpu(inp)
    assert o.numel() == 0 and torch.equal(ht.cpu(), inp["h0"])


@pytest.mark.parametrize("dk", [64, 128])
def test_malformed_cu_seqlens_reported(lib, dk):
    """A decreasing cu_seqlens is caught by the kernels' own bounds checks and
    reported by dn_check; the bad sequence is skipped, the others computed."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    inp = inputs(B=1, dk=dk, dv=dk, lengths=[10, 20, 30], seed=310)
    d = workloads.to_device(inp, "cuda")
    cu = torch.tensor([0, 10, 5, 60], dtype=torch.int64, device="cuda")
    o, ht = dn.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], cu,
                         scale=inp["scale"])
    assert dn.dn_check() == dn.DN_ERR_DEVICE_ARG
    assert dn.dn_check() == dn.DN_OK  # the status word was cleared


# ---------------------------------------------------------------------------
# The named workloads at full size, sampled units.
# ---------------------------------------------------------------------------
SAMPLES = {
    "deltanet_fp32_h2_t256_d64": None,
    "gdn_bf16_b4_h16_t2048_d128": [0, 17, 40, 63],
    "gdn_gqa_varlen_bf16_n8_nk8_nv32_d128": "longest_shortest",
    "gdn_long_bf16_b1_h32_t32768_d128": [0, 31],
    "gdn_wide_bf16_b8_h8_t8192_d256": [0, 63],
    "gdn_wide_bf16_b2_h8_t8192_d256": [5],
    "gdn_decode_bf16_b64_h16_t1_d128": None,
    "gdn_l2norm_bf16_b4_h16_t2048_d128": [0, 33, 63],
}


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_workload_full_size(lib, name):
    inp = workloads.workload_inputs(name)
    o, ht = run_gpu(inp)
    units = SAMPLES[name]
    if units == "longest_shortest":
        cu = inp["cu_seqlens"]
        lens = (cu[1:] - cu[:-1]).tolist()
        Nv = inp["v"].shape[2]
        nl, ns = int(np.argmax(lens)), int(np.argmin(lens))
        units = [nl * Nv, nl * Nv + Nv - 1, ns * Nv + 1]
    if name.startswith("gdn_wide"):
        import chunkwise_gated_delta_chunk_gb300 as dn
        assert dn.dn_last_kernel() == "wy_fwd+tc_wide_fwd", dn.dn_last_kernel()
    res = check(inp, o, ht, units=units, label=name)
    # every output of every unit is finite
    assert torch.isfinite(o.float()).all() and torch.isfinite(ht).all()
    print(name, res)


@pytest.mark.parametrize("nseq", [64, 65])
def test_many_sequences_longest_first(lib, nseq):
    """Packed batches at and just past the number of sequences the kernels order
    longest first (64; beyond it units run in sequence order): random lengths,
    empty ones included, on the tensor-core forward and the backward's walk."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    rng = np.random.default_rng(800 + nseq)
    lengths = [int(x) for x in rng.integers(0, 260, size=nseq)]
    lengths[3] = 0
    inp = inputs(B=1, Nk=1, Nv=2, dk=128, dv=128, lengths=lengths, seed=810 + nseq)
    o, ht = run_gpu(inp)
    assert dn.dn_last_kernel() == "wy_fwd+tc_fwd", dn.dn_last_kernel()
    check(inp, o, ht, label="%d sequences" % nseq)
