"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it element by element with the fp64 oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

# Tolerances against the fp64 oracle, on o and ht:
#   bf16 q/k/v with fp32 accumulation: max-abs <= 2e-2 and rel-L2 <= 5e-3;
#   fp32 inputs (fp32 arithmetic throughout): rel-L2 <= 1e-4.
TOL = {
    torch.bfloat16: dict(max_abs=2e-2, rel_l2=5e-3),
    torch.float32: dict(max_abs=1e-3, rel_l2=1e-4),
}


def run_gpu(inp: dict, device="cuda", output_final_state=True, scale=None, chunk=64):
    """dn_chunk_fwd on the inputs (with in-kernel q / k normalisation when the
    inputs ask for it), then dn_check."""
    import chunkwise_gated_delta_chunk_gb300 as dn
    d = workloads.to_device(inp, device)
    o, ht = dn.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["cu_seqlens"],
                         scale=inp["scale"] if scale is None else scale,
                         output_final_state=output_final_state, chunk=chunk,
                         use_qk_l2norm_in_kernel=inp.get("qk_l2norm", False))
    st = dn.dn_check()
    assert st == dn.DN_OK, dn.dn_status_str(st)
    return o, ht


def unit_index(inp: dict, u: int):
    """Index tuples of unit u = n*Nv + h in o [B,T,Nv,dv] and ht [N,Nv,dk,dv]."""
    Nv = inp["v"].shape[2]
    n, h = divmod(u, Nv)
    if inp["cu_seqlens"] is not None:
        cu = inp["cu_seqlens"]
        return (0, slice(int(cu[n]), int(cu[n + 1])), h), (n, h)
    return (n, slice(None), h), (n, h)


def metrics(got: np.ndarray, ref: np.ndarray) -> dict:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return dict(max_abs=0.0, rel_l2=0.0)
    err = got - ref
    return dict(max_abs=float(np.abs(err).max()),
                rel_l2=float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)))


def check(inp: dict, o_gpu, ht_gpu, units=None, threads=0, tol=None, label=""):
    """Compare the GPU outputs with the oracle on `units` (all when None)."""
    dtype = inp["q"].dtype
    tol = tol or TOL[dtype]
    o_ref, ht_ref = oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"],
                                     inp["h0"], inp["cu_seqlens"], inp["scale"], units=units,
                                     threads=threads,
                                     use_qk_l2norm_in_kernel=inp.get("qk_l2norm", False))
    o_g = o_gpu.detach().to("cpu", torch.float64).numpy()
    ht_g = None if ht_gpu is None else ht_gpu.detach().to("cpu", torch.float64).numpy()
    Nv = inp["v"].shape[2]
    N = inp["N"]
    uu = list(range(N * Nv)) if units is None else list(units)
    og, orf, hg, hrf = [], [], [], []
    for u in uu:
        oi, hi = unit_index(inp, u)
        og.append(o_g[oi].ravel())
        orf.append(o_ref[oi].ravel())
        if ht_g is not None:
            hg.append(ht_g[hi].ravel())
            hrf.append(ht_ref[hi].ravel())
    res = {"o": metrics(np.concatenate(og), np.concatenate(orf))}
    if ht_g is not None:
        res["ht"] = metrics(np.concatenate(hg), np.concatenate(hrf))
    for key, m in res.items():
        assert np.isfinite(m["max_abs"]), (label, key, m)
        assert m["max_abs"] <= tol["max_abs"], (label, key, m)
        assert m["rel_l2"] <= tol["rel_l2"], (label, key, m)
    return res
