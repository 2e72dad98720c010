"""GPU: the forward captured in a CUDA graph (the scan is launched as a
programmatic dependent of the WY kernel, a dependency the capture must keep)
and replayed, against eager calls on the same inputs, bit for bit."""
import pytest
import torch

import workloads
from conftest import cuda_ok

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


@pytest.mark.parametrize("dk,dv", [(128, 128), (256, 256)])
def test_forward_replayed_from_a_cuda_graph(lib, dk, dv):
    import chunkwise_gated_delta_chunk_gb300 as dn

    def make(seed):
        return workloads.make_inputs(2, 700, 2, 4, dk, dv, gate_mu=3.0, h0=True, seed=seed)

    inp = make(1200 + dk)
    d = workloads.to_device(inp, "cuda")

    def call():
        return dn.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], None,
                            scale=inp["scale"])

    o_ref, ht_ref = call()  # eager, also sets up the library's per-device state
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            o, ht = call()
    torch.cuda.current_stream().wait_stream(stream)
    graph.replay()
    torch.cuda.synchronize()
    assert dn.dn_check() == dn.DN_OK
    assert torch.equal(o, o_ref) and torch.equal(ht, ht_ref)
    # new inputs through the captured buffers
    inp2 = make(1300 + dk)
    for key in ("q", "k", "v", "beta", "g", "h0"):
        d[key].copy_(inp2[key].to("cuda"))
    graph.replay()
    torch.cuda.synchronize()
    o2_ref, ht2_ref = call()
    torch.cuda.synchronize()
    assert dn.dn_check() == dn.DN_OK
    assert torch.equal(o, o2_ref) and torch.equal(ht, ht2_ref)
    assert not torch.equal(o2_ref, o_ref)
