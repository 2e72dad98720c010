"""Seeded random configurations of the tensor-core forward against the oracle.

Each case draws, from its own seed, the sizes and options the library takes
on its tensor-core path (dk in {128, 256}, dv a multiple of 128, GQA ratio,
chunk length, gates / h0 / final state present or not, in-kernel q / k
normalisation, dense or packed varlen batches with empty and length-1
sequences) and compares every output with the fp64 oracle at the bf16 bound.
"""
import random

import pytest

import workloads
from conftest import cuda_ok
from parity_util import check, run_gpu

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


def draw(seed):
    r = random.Random(seed)
    dk = r.choice([128, 256])
    dv = r.choice([128, 256])
    nk = r.choice([1, 2])
    nv = nk * r.choice([1, 2, 4])
    chunk = r.choice([16, 32, 64, 64])
    gate = r.choice([None, 3.0, 5.0, 1.0])
    h0 = r.random() < 0.6
    raw_qk = r.random() < 0.3
    if r.random() < 0.5:
        lengths = [r.choice([0, 1, r.randint(2, 63), r.randint(64, 400)]) for _ in range(r.randint(1, 5))]
        lengths.append(r.randint(65, 300))  # at least one sequence of several chunks
        r.shuffle(lengths)
        kw = dict(B=1, T=0, lengths=lengths)
    else:
        kw = dict(B=r.randint(1, 3), T=r.randint(1, 330), lengths=None)
    final = r.random() < 0.8
    return dict(dk=dk, dv=dv, nk=nk, nv=nv, chunk=chunk, gate=gate, h0=h0, raw_qk=raw_qk, final=final, **kw)


@pytest.mark.parametrize("seed", range(700, 716))
def test_random_configuration(lib, seed):
    import chunkwise_gated_delta_chunk_gb300 as dn
    c = draw(seed)
    inp = workloads.make_inputs(c["B"], c["T"], c["nk"], c["nv"], c["dk"], c["dv"], gate_mu=c["gate"],
                                h0=c["h0"], seed=seed, lengths=c["lengths"], raw_qk=c["raw_qk"])
    o, ht = run_gpu(inp, chunk=c["chunk"], output_final_state=c["final"])
    assert dn.dn_last_kernel().startswith("wy_fwd"), (c, dn.dn_last_kernel())
    check(inp, o, ht, label="fuzz %d %s" % (seed, c))
