"""Seeded synthetic inputs for the chunkwise gated delta rule forward.

This module is shared by the tests, the benchmark and the smoke check.  It
draws random inputs only: it holds none of the method's arithmetic, and it
imports neither the CUDA package nor the oracle.

Recipe (all draws on a CPU ``torch.Generator`` seeded per workload):

* q, v ~ N(0, 1), drawn in fp32 and cast to the workload dtype (RNE);
* k ~ N(0, 1) in fp32, L2-normalised per (token, head) in fp32, then cast;
  for the in-kernel normalisation workloads (``qk_l2norm``) k is left as
  drawn, and every q and k row is multiplied by exp(0.5 z), z ~ N(0, 1), so
  the row norms spread over about a factor of e around sqrt(d);
* beta = sigmoid(N(0, 1)) in fp32;
* g = log(sigmoid(N(mu, 1))) in fp32 (mu = 3, or 5 for the long-context
  workload), so every per-token decay e^g lies in (0, 1);
* h0 ~ N(0, 0.02^2) in fp32 (standard deviation 0.02);
* varlen: sequence lengths uniform in [1, 4096], drawn from the same seed.

The named workloads follow the pages' shapes: plain DeltaNet in fp32, gated
DeltaNet at H=16/T=2048/d=128, GQA + varlen, long context and wide heads, and
one decoding step (T = 1, state in and out) for the token-serial path.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int               # per-sequence length (ignored when lengths is set)
    Nk: int
    Nv: int
    dk: int
    dv: int
    dtype: torch.dtype
    gate_mu: Optional[float]   # None: no gate (g = 0, plain DeltaNet)
    h0: bool                   # False: zero initial state (passed as null)
    seed: int
    n_varlen: int = 0          # > 0: that many packed sequences, B must be 1
    max_len: int = 4096
    chunk: int = 64
    qk_l2norm: bool = False    # q and k left raw; the kernels normalise them


WORKLOADS = {
    w.name: w
    for w in [
        Workload("deltanet_fp32_h2_t256_d64", B=1, T=256, Nk=2, Nv=2, dk=64, dv=64,
                 dtype=torch.float32, gate_mu=None, h0=False, seed=1),
        Workload("gdn_bf16_b4_h16_t2048_d128", B=4, T=2048, Nk=16, Nv=16, dk=128, dv=128,
                 dtype=torch.bfloat16, gate_mu=3.0, h0=True, seed=2),
        Workload("gdn_gqa_varlen_bf16_n8_nk8_nv32_d128", B=1, T=0, Nk=8, Nv=32, dk=128,
                 dv=128, dtype=torch.bfloat16, gate_mu=3.0, h0=True, seed=3, n_varlen=8),
        Workload("gdn_long_bf16_b1_h32_t32768_d128", B=1, T=32768, Nk=32, Nv=32, dk=128,
                 dv=128, dtype=torch.bfloat16, gate_mu=5.0, h0=False, seed=4),
        Workload("gdn_wide_bf16_b8_h8_t8192_d256", B=8, T=8192, Nk=8, Nv=8, dk=256, dv=256,
                 dtype=torch.bfloat16, gate_mu=3.0, h0=True, seed=5),
        # the wide-head shapes at a quarter of the batch (profiling case: its
        # inputs still exceed L2)
        Workload("gdn_wide_bf16_b2_h8_t8192_d256", B=2, T=8192, Nk=8, Nv=8, dk=256, dv=256,
                 dtype=torch.bfloat16, gate_mu=3.0, h0=True, seed=8),
        # one decoding step of 64 sequences: the state comes in and goes out
        Workload("gdn_decode_bf16_b64_h16_t1_d128", B=64, T=1, Nk=16, Nv=16, dk=128, dv=128,
                 dtype=torch.bfloat16, gate_mu=3.0, h0=True, seed=6),
        # the gated DeltaNet shapes with raw q / k normalised inside the kernels
        Workload("gdn_l2norm_bf16_b4_h16_t2048_d128", B=4, T=2048, Nk=16, Nv=16, dk=128,
                 dv=128, dtype=torch.bfloat16, gate_mu=3.0, h0=True, seed=7, qk_l2norm=True),
    ]
}

# The headline workload the benchmark times.
HEADLINE = "gdn_bf16_b4_h16_t2048_d128"


def varlen_lengths(n: int, max_len: int, gen: torch.Generator) -> list[int]:
    return [int(x) for x in torch.randint(1, max_len + 1, (n,), generator=gen)]


def make_inputs(B: int, T: int, Nk: int, Nv: int, dk: int, dv: int,
                dtype: torch.dtype = torch.bfloat16, gate_mu: Optional[float] = 3.0,
                h0: bool = True, seed: int = 0,
                lengths: Optional[Sequence[int]] = None,
                beta_range: Optional[tuple] = None, raw_qk: bool = False) -> dict:
    """Draw one input set on the CPU.

    With ``lengths`` the sequences are packed (B must be 1, T = sum(lengths))
    and ``cu_seqlens`` (int64, ``[N+1]``) is returned.  Keys: q, k, v, beta,
    g (or None), h0 (or None), cu_seqlens (or None), scale, N, qk_l2norm
    (= ``raw_qk``: q and k are not normalised and need the in-kernel option).
    """
    gen = torch.Generator().manual_seed(seed)
    cu = None
    if lengths is not None:
        assert B == 1
        lengths = [int(x) for x in lengths]
        T = sum(lengths)
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int64)
        if lengths:
            cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0)
        N = len(lengths)
    else:
        N = B
    q = torch.randn(B, T, Nk, dk, generator=gen)
    k = torch.randn(B, T, Nk, dk, generator=gen)
    if not raw_qk:
        k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    v = torch.randn(B, T, Nv, dv, generator=gen)
    beta = torch.sigmoid(torch.randn(B, T, Nv, generator=gen))
    if beta_range is not None:
        lo, hi = beta_range
        beta = lo + (hi - lo) * beta
    g = None
    if gate_mu is not None:
        g = torch.nn.functional.logsigmoid(gate_mu + torch.randn(B, T, Nv, generator=gen))
    s0 = None
    if h0:
        s0 = 0.02 * torch.randn(N, Nv, dk, dv, generator=gen)
    if raw_qk:
        q = q * torch.exp(0.5 * torch.randn(B, T, Nk, 1, generator=gen))
        k = k * torch.exp(0.5 * torch.randn(B, T, Nk, 1, generator=gen))
    return dict(q=q.to(dtype), k=k.to(dtype), v=v.to(dtype), beta=beta.float(),
                g=None if g is None else g.float(), h0=s0, cu_seqlens=cu,
                scale=1.0 / math.sqrt(dk), N=N, qk_l2norm=bool(raw_qk))


def workload_inputs(name: str) -> dict:
    """Inputs of a named workload (deterministic for its seed)."""
    w = WORKLOADS[name]
    lengths = None
    if w.n_varlen:
        gen = torch.Generator().manual_seed(w.seed)
        lengths = varlen_lengths(w.n_varlen, w.max_len, gen)
        # separate stream for the tensors so the lengths do not shift them
    return make_inputs(w.B, w.T, w.Nk, w.Nv, w.dk, w.dv, dtype=w.dtype, gate_mu=w.gate_mu,
                       h0=w.h0, seed=w.seed + (1000 if w.n_varlen else 0), lengths=lengths,
                       raw_qk=w.qk_l2norm)


def to_device(inp: dict, device) -> dict:
    out = {}
    for key, val in inp.items():
        out[key] = val.to(device) if isinstance(val, torch.Tensor) else val
    return out


def tokens(inp: dict) -> int:
    return int(inp["q"].shape[0] * inp["q"].shape[1])
