"""Pins for the fp64 oracle, against what the pages and the mathematics fix.

None of these retypes the oracle's own formula: each compares it with an
independent statement -- brute-force products of the Householder-like factors,
a closed form, an invariant, or a second independently written form.

Pages: [WY] "flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现";
[CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么".
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads


def _small(B=1, T=37, Nk=2, Nv=2, dk=8, dv=6, gate=True, h0=True, seed=0, lengths=None,
           dtype=torch.float64):
    inp = workloads.make_inputs(B, T, Nk, Nv, dk, dv, dtype=torch.float32,
                                gate_mu=1.0 if gate else None, h0=h0, seed=seed,
                                lengths=lengths)
    return inp


def _rel(a, b):
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-300))


def _call(fn, inp, **kw):
    return fn(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["h0"],
              inp["cu_seqlens"], inp["scale"], **kw)


# --------------------------------------------------------------------------
# Chunk algebra ([WY] §2.4, [CGDR] §3.2): the chunk form equals the token
# recurrence for every chunk size, including C=1 and C >= T.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [1, 5, 16, 32, 64, 1000])
@pytest.mark.parametrize("gate", [False, True])
def test_chunk_invariance(chunk, gate):
    inp = _small(T=77, gate=gate, seed=11)
    o_r, h_r = _call(oracle.recurrent, inp)
    o_c, h_c = _call(oracle.chunked, inp, chunk=chunk)
    assert _rel(o_c, o_r) < 1e-12
    assert _rel(h_c, h_r) < 1e-12


def test_chunk_invariance_varlen_gqa():
    inp = _small(B=1, Nk=2, Nv=6, lengths=[1, 64, 65, 130, 3], seed=12)
    o_r, h_r = _call(oracle.recurrent, inp)
    o_c, h_c = _call(oracle.chunked, inp, chunk=64)
    assert _rel(o_c, o_r) < 1e-12
    assert _rel(h_c, h_r) < 1e-12


def test_literal_read_rejected_by_chunk_form():
    """Reading 1: with a gate, the chunk form of [CGDR] §3 matches only the
    decayed read; without a gate the two readings coincide."""
    inp = _small(T=70, gate=True, seed=13)
    o_c, h_c = _call(oracle.chunked, inp, chunk=64)
    o_l, h_l = _call(oracle.recurrent, inp, read_mode=1)
    assert _rel(o_l, o_c) > 1e-3
    assert _rel(h_l, h_c) > 1e-3
    inp = _small(T=70, gate=False, seed=13)
    o_c, h_c = _call(oracle.chunked, inp, chunk=64)
    o_l, h_l = _call(oracle.recurrent, inp, read_mode=1)
    assert _rel(o_l, o_c) < 1e-12 and _rel(h_l, h_c) < 1e-12


# --------------------------------------------------------------------------
# WY representation ([WY] §2.1-§2.2): brute-force products of the factors
# (I - b_i k_i k_i^T) against the W and U the oracle's chunk step produces.
# With a gate the factors become e^{g_i}(I - b_i k_i k_i^T) (decay first).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("gate", [False, True])
@pytest.mark.parametrize("L,dk,dv", [(1, 3, 2), (5, 4, 3), (8, 16, 5), (12, 6, 7)])
def test_wy_identities_brute_force(L, dk, dv, gate):
    rng = np.random.default_rng(100 + L * 7 + dk)
    K = rng.standard_normal((L, dk))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    V = rng.standard_normal((L, dv))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    g = np.log(1.0 / (1.0 + np.exp(-(1.0 + rng.standard_normal(L))))) if gate else None
    G, Tm, W, U = oracle.wy_chunk(K, V, b, g)
    a = np.exp(g) if gate else np.ones(L)
    P = np.eye(dk)
    H = np.zeros((dk, dv))
    for r in range(L):
        F = a[r] * (np.eye(dk) - b[r] * np.outer(K[r], K[r]))
        P = F @ P                                     # P^r = F_r P^{r-1}
        H = F @ H + b[r] * np.outer(K[r], V[r])       # H^r = F_r H^{r-1} + b_r k_r v_r^T
        dec = np.exp(G[r] - G[: r + 1])               # e^{G_r - G_i}, i <= r
        P_wy = math.exp(G[r]) * np.eye(dk) - (K[: r + 1] * dec[:, None]).T @ W[: r + 1]
        H_wy = (K[: r + 1] * dec[:, None]).T @ U[: r + 1]
        assert np.abs(P_wy - P).max() < 1e-12
        assert np.abs(H_wy - H).max() < 1e-12


def test_T_is_unit_lower_inverse():
    rng = np.random.default_rng(5)
    L, dk, dv = 64, 32, 4
    K = rng.standard_normal((L, dk))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    V = rng.standard_normal((L, dv))
    b = rng.uniform(0, 1, L)
    g = -rng.uniform(0, 0.3, L)
    G, Tm, W, U = oracle.wy_chunk(K, V, b, g)
    assert np.allclose(np.diag(Tm), 1.0)
    assert np.abs(np.triu(Tm, 1)).max() == 0.0
    # T^-1 = I - A is unit lower triangular with the strictly lower part
    # -b_i (k_i.k_j) e^{G_i-G_j}, i.e. T^-1 has that off-diagonal.
    Tinv = np.linalg.inv(Tm)
    expect = np.tril(b[:, None] * (K @ K.T) * np.exp(G[:, None] - G[None, :]), -1)
    assert np.abs(Tinv - (np.eye(L) + expect)).max() < 1e-10


# --------------------------------------------------------------------------
# Closed forms and invariants.
# --------------------------------------------------------------------------
def test_beta_zero_only_decays():
    """beta = 0: nothing is written, so ht = e^{sum g} h0 and
    o_t = scale e^{sum_{s<=t} g_s} q_t^T h0."""
    inp = _small(T=50, seed=21)
    inp["beta"] = torch.zeros_like(inp["beta"])
    o, ht = _call(oracle.recurrent, inp)
    q = inp["q"].double().numpy()[0]
    g = inp["g"].double().numpy()[0]
    h0 = inp["h0"].double().numpy()[0]
    Gs = np.cumsum(g, axis=0)                             # [T, Nv]
    for h in range(2):
        ht_cf = math.exp(Gs[-1, h]) * h0[h]
        o_cf = inp["scale"] * np.exp(Gs[:, h])[:, None] * (q[:, h] @ h0[h])
        assert np.abs(ht[0, h] - ht_cf).max() < 1e-13
        assert np.abs(o[0, :, h] - o_cf).max() < 1e-13
    oc, hc = _call(oracle.chunked, inp, chunk=16)
    assert _rel(oc, o) < 1e-12 and _rel(hc, ht) < 1e-12


@pytest.mark.parametrize("gate", [False, True])
def test_orthonormal_keys_overwrite(gate):
    """Orthonormal k with beta = 1 ([CGDR] §1 steps 2-3): writing key k_s puts
    exactly v_s in its slot; later writes to orthogonal keys only decay it.
    So o_t for q_t = k_s is scale e^{G_t - G_s} v_s (s <= t)."""
    T, dk, dv = 24, 32, 5
    rng = np.random.default_rng(3)
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:, :T].T                                    # T orthonormal rows
    v = rng.standard_normal((T, dv))
    g = -rng.uniform(0.0, 0.5, T) if gate else np.zeros(T)
    h0 = rng.standard_normal((dk, dv))
    src = rng.integers(0, T, T)
    src = np.minimum(src, np.arange(T))                   # query an earlier key
    q = keys[src]
    t_ = lambda x: torch.from_numpy(np.ascontiguousarray(x))
    o, ht = oracle.recurrent(t_(q[None, :, None]), t_(keys[None, :, None]),
                             t_(v[None, :, None]), t_(np.ones((1, T, 1))),
                             t_(g[None, :, None]), t_(h0[None, None]), None, 0.5)
    G = np.cumsum(g)
    expect = 0.5 * np.exp(G - G[src])[:, None] * v[src]
    assert np.abs(o[0, :, 0] - expect).max() < 1e-12
    # the final state holds every written slot exactly (decayed), plus the
    # decayed part of h0 outside the written subspace
    proj = np.eye(dk) - keys.T @ keys
    expect_ht = math.exp(G[-1]) * proj @ h0 + (keys * np.exp(G[-1] - G)[:, None]).T @ v
    assert np.abs(ht[0, 0] - expect_ht).max() < 1e-12


def test_scalar_state_closed_form():
    """dk = dv = 1: the state is a scalar first-order linear recurrence
    s_t = c_t s_{t-1} + b_t k_t v_t with c_t = e^{g_t} (1 - b_t k_t^2), whose
    closed form is s_T = (prod c) s_0 + sum_t (prod_{r>t} c_r) b_t k_t v_t."""
    rng = np.random.default_rng(8)
    T = 40
    k = rng.uniform(-1, 1, T)
    v = rng.standard_normal(T)
    q = rng.standard_normal(T)
    b = rng.uniform(0, 1, T)
    g = -rng.uniform(0, 0.2, T)
    s0 = 0.7
    c = np.exp(g) * (1 - b * k * k)
    s = np.empty(T)
    for t in range(T):
        s[t] = np.prod(c[: t + 1]) * s0 + sum(np.prod(c[r + 1: t + 1]) * b[r] * k[r] * v[r]
                                              for r in range(t + 1))
    t_ = lambda x: torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=np.float64)))
    o, ht = oracle.recurrent(t_(q.reshape(1, T, 1, 1)), t_(k.reshape(1, T, 1, 1)),
                             t_(v.reshape(1, T, 1, 1)), t_(b.reshape(1, T, 1)),
                             t_(g.reshape(1, T, 1)), t_([[[[s0]]]]), None, 1.3)
    assert np.abs(o[0, :, 0, 0] - 1.3 * q * s).max() < 1e-13
    assert abs(ht[0, 0, 0, 0] - s[-1]) < 1e-13


def test_single_token_by_hand():
    """One token, exact binary fractions: decay 1/2 (g = -ln 2), beta = 1/2,
    k = e_1, v = (1, 2), h0 = [[1, 0], [0, 4]], q = (1, 1), scale 1.
    S = 1/2 h0 + 1/2 e_1 ((1, 2) - 1/2 (1, 0))^T = [[3/4, 1], [0, 2]];
    o = S^T q = (3/4, 3)."""
    t_ = lambda x: torch.tensor(x, dtype=torch.float64)
    o, ht = oracle.recurrent(t_([[[[1.0, 1.0]]]]), t_([[[[1.0, 0.0]]]]), t_([[[[1.0, 2.0]]]]),
                             t_([[[0.5]]]), t_([[[-math.log(2.0)]]]),
                             t_([[[[1.0, 0.0], [0.0, 4.0]]]]), None, 1.0)
    assert np.allclose(ht[0, 0], [[0.75, 1.0], [0.0, 2.0]], atol=1e-15, rtol=0)
    assert np.allclose(o[0, 0, 0], [0.75, 3.0], atol=1e-15, rtol=0)


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(path):
    """`name: values` lines of a worked-example fixture (fractions allowed)."""
    rec = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                name, vals = line.split(":", 1)
                rec[name.strip()] = [float(Fraction(x)) for x in vals.split()]
    return rec


@pytest.mark.parametrize("name", sorted(f for f in os.listdir(GOLDEN) if f.endswith(".txt")))
def test_golden_worked_examples(name):
    """Hand-derived worked examples (exact fractions, derivation in each
    fixture) against the token recurrence and the chunk form."""
    rec = _read_golden(os.path.join(GOLDEN, name))
    dk, dv = (int(x) for x in rec["dims"])
    T = len(rec["beta"])
    t_ = lambda x, *shape: torch.tensor(x, dtype=torch.float64).reshape(*shape)
    args = (t_(rec["q"], 1, T, 1, dk), t_(rec["k"], 1, T, 1, dk), t_(rec["v"], 1, T, 1, dv),
            t_(rec["beta"], 1, T, 1), t_([math.log(d) for d in rec["decay"]], 1, T, 1),
            t_(rec["h0"], 1, 1, dk, dv), None, rec["scale"][0])
    want_o, want_ht = np.array(rec["o"]).reshape(T, dv), np.array(rec["ht"]).reshape(dk, dv)
    runs = [oracle.recurrent(*args)] + [oracle.chunked(*args, chunk=c) for c in (1, 2, 64)]
    for o, ht in runs:
        assert np.abs(o[0, :, 0] - want_o).max() < 1e-14
        assert np.abs(ht[0, 0] - want_ht).max() < 1e-14


def test_linearity():
    """o and ht are jointly linear in (v, h0); o is linear in q and in scale."""
    a = {k: (v.double() if isinstance(v, torch.Tensor) and v.is_floating_point() else v)
         for k, v in _small(T=45, seed=31).items()}
    b = {k: (v.double() if isinstance(v, torch.Tensor) and v.is_floating_point() else v)
         for k, v in _small(T=45, seed=32).items()}
    mix = dict(a)
    mix["v"] = a["v"] + 2.0 * b["v"]
    mix["h0"] = a["h0"] + 2.0 * b["h0"]
    bb = dict(a)
    bb["v"], bb["h0"] = b["v"], b["h0"]
    oa, ha = _call(oracle.recurrent, a)
    ob, hb = _call(oracle.recurrent, bb)
    om, hm = _call(oracle.recurrent, mix)
    assert _rel(om, oa + 2 * ob) < 1e-12 and _rel(hm, ha + 2 * hb) < 1e-12
    q3 = dict(a)
    q3["q"] = 3.0 * a["q"]
    o3, h3 = _call(oracle.recurrent, q3)
    assert _rel(o3, 3 * oa) < 1e-13 and _rel(h3, ha) < 1e-15
    s2 = dict(a)
    s2["scale"] = 2 * a["scale"]
    o2, _ = _call(oracle.recurrent, s2)
    assert _rel(o2, 2 * oa) < 1e-13


def test_varlen_equals_separate_runs():
    lengths = [5, 64, 1, 70]
    inp = _small(Nk=1, Nv=3, lengths=lengths, seed=41)
    o, ht = _call(oracle.recurrent, inp)
    cu = inp["cu_seqlens"]
    for n in range(len(lengths)):
        s, e = int(cu[n]), int(cu[n + 1])
        part = dict(inp)
        for key in ("q", "k", "v", "beta", "g"):
            part[key] = inp[key][:, s:e]
        part["h0"] = inp["h0"][n: n + 1]
        part["cu_seqlens"] = None
        op, hp = _call(oracle.recurrent, part)
        assert np.abs(op[0] - o[0, s:e]).max() < 1e-14
        assert np.abs(hp[0] - ht[n]).max() < 1e-14


def test_gqa_equals_head_expansion():
    """nvPerNk = Nv/Nk: v-head h reads q/k head h // nvPerNk ([CGDR] §1)."""
    inp = _small(Nk=2, Nv=6, T=30, seed=51)
    o, ht = _call(oracle.recurrent, inp)
    exp_ = dict(inp)
    idx = torch.arange(6) // 3
    exp_["q"] = inp["q"][:, :, idx]
    exp_["k"] = inp["k"][:, :, idx]
    oe, he = _call(oracle.recurrent, exp_)
    assert np.abs(oe - o).max() == 0.0 and np.abs(he - ht).max() == 0.0


def test_state_carry_split():
    """Two calls, the second starting from the first's final state, equal one
    call on the whole sequence (initial_state / output_final_state, [WY] §5)."""
    inp = _small(T=90, seed=61)
    o, ht = _call(oracle.recurrent, inp)
    cut = 37
    p1, p2 = dict(inp), dict(inp)
    for key in ("q", "k", "v", "beta", "g"):
        p1[key] = inp[key][:, :cut]
        p2[key] = inp[key][:, cut:]
    o1, h1 = _call(oracle.chunked, p1, chunk=16)
    p2["h0"] = torch.from_numpy(h1)
    o2, h2 = _call(oracle.chunked, p2, chunk=16)
    assert _rel(np.concatenate([o1, o2], axis=1), o) < 1e-12
    assert _rel(h2, ht) < 1e-12


def test_units_subset_matches_full():
    inp = _small(B=3, Nk=1, Nv=2, T=20, seed=71)
    o, ht = _call(oracle.recurrent, inp)
    os_, hs = _call(oracle.recurrent, inp, units=[5, 0])
    assert np.array_equal(os_[2, :, 1], o[2, :, 1]) and np.array_equal(hs[2, 1], ht[2, 1])
    assert np.array_equal(os_[0, :, 0], o[0, :, 0])
    assert np.isnan(os_[1]).all()


def test_empty_sequence_keeps_h0():
    inp = _small(Nk=1, Nv=2, lengths=[0, 4, 0], seed=81)
    o, ht = _call(oracle.recurrent, inp)
    h0 = inp["h0"].double().numpy()
    assert np.array_equal(ht[0], h0[0]) and np.array_equal(ht[2], h0[2])


# --------------------------------------------------------------------------
# In-kernel q / k normalisation ([WY] §5 use_qk_l2norm_in_kernel; [WY] §6:
# the tests L2-normalise k along the head dimension, F.normalize(p=2,
# dim=-1), or leave it to the kernels with the option on).
# --------------------------------------------------------------------------
def test_l2norm_closed_forms():
    """Pythagorean rows by hand, the zero row, and a row below the 1e-12 guard
    (divided by the guard, not by its own norm)."""
    x = np.array([[3.0, 4.0, 0.0], [1.0, 2.0, 2.0], [0.0, 0.0, 0.0], [-1e-13, 0.0, 0.0],
                  [0.0, -12.0, 5.0]])
    want = np.array([[0.6, 0.8, 0.0], [1 / 3, 2 / 3, 2 / 3], [0.0, 0.0, 0.0], [-0.1, 0.0, 0.0],
                     [0.0, -12 / 13, 5 / 13]])
    assert np.allclose(oracle.l2norm(x), want, rtol=0, atol=1e-15)


def test_l2norm_unit_rows_same_direction():
    """Random rows of every head size come out with norm 1 and a positive
    multiple of the input (x^ . x = ||x||), over arbitrary leading axes."""
    rng = np.random.default_rng(5)
    for d in (1, 16, 128, 256):
        x = rng.standard_normal((3, 7, 2, d)) * np.exp(rng.standard_normal((3, 7, 2, 1)))
        y = oracle.l2norm(x)
        assert y.shape == x.shape
        assert np.allclose(np.sqrt((y * y).sum(-1)), 1.0, rtol=0, atol=1e-14)
        assert np.allclose((y * x).sum(-1), np.sqrt((x * x).sum(-1)), rtol=1e-13, atol=0)


@pytest.mark.parametrize("fn", ["recurrent", "chunked"])
def test_qk_l2norm_ignores_row_scale(fn):
    """With the option on, rescaling every q row and every k row by its own
    positive factor leaves o and ht unchanged; with it off they change.  A
    normalisation that misses q or k, or normalises along the wrong axis,
    fails this."""
    f = getattr(oracle, fn)
    inp = _small(B=1, Nk=2, Nv=4, dk=8, dv=5, lengths=[9, 70, 1], seed=91)
    rng = np.random.default_rng(91)
    sq = torch.tensor(np.exp(rng.standard_normal(inp["q"].shape[:-1] + (1,))))
    sk = torch.tensor(np.exp(rng.standard_normal(inp["k"].shape[:-1] + (1,))))
    scaled = dict(inp, q=inp["q"].double() * sq, k=inp["k"].double() * sk)
    o1, h1 = _call(f, inp, use_qk_l2norm_in_kernel=True)
    o2, h2 = _call(f, scaled, use_qk_l2norm_in_kernel=True)
    assert _rel(o2, o1) < 1e-12 and _rel(h2, h1) < 1e-12
    o3, _ = _call(f, scaled)
    assert _rel(o3, o1) > 1e-2


def test_qk_l2norm_reduces_to_plain_on_unit_rows():
    """Rows that already have unit norm are left alone: the option changes
    nothing (up to fp64 rounding) when q and k are unit rows."""
    inp = _small(B=2, T=40, Nk=1, Nv=2, dk=16, dv=4, seed=92)
    q, k = inp["q"].double(), inp["k"].double()
    inp = dict(inp, q=q / q.norm(dim=-1, keepdim=True), k=k / k.norm(dim=-1, keepdim=True))
    o1, h1 = _call(oracle.recurrent, inp)
    o2, h2 = _call(oracle.recurrent, inp, use_qk_l2norm_in_kernel=True)
    assert _rel(o2, o1) < 1e-13 and _rel(h2, h1) < 1e-13


@pytest.mark.parametrize("chunk", [16, 64])
def test_qk_l2norm_chunk_equals_recurrent(chunk):
    """The chunk form and the token recurrence agree with the option on, on
    raw (unnormalised, widely scaled) q and k."""
    inp = workloads.make_inputs(1, 0, 2, 4, 16, 8, dtype=torch.float32, gate_mu=3.0, h0=True,
                                seed=93, lengths=[5, 64, 100], raw_qk=True)
    o_r, h_r = _call(oracle.recurrent, inp, use_qk_l2norm_in_kernel=True)
    o_c, h_c = _call(oracle.chunked, inp, chunk=chunk, use_qk_l2norm_in_kernel=True)
    assert _rel(o_c, o_r) < 1e-12 and _rel(h_c, h_r) < 1e-12


# --------------------------------------------------------------------------
# Gradient of the forward ([WY] §3.4 lists dq, dk, dv, dbeta and dh0; the
# gated form adds dg).  The pages print no backward formula, so the oracle's
# reverse pass is pinned by central finite differences of the forward oracle
# (the definition), element by element, on tiny inputs that cross the
# reverse pass's 64-token checkpoints.
# --------------------------------------------------------------------------
def _loss(inp, do, dht, l2=False, **over):
    d = dict(inp, **over)
    o, ht = oracle.recurrent(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                             d["cu_seqlens"], d["scale"], threads=1, use_qk_l2norm_in_kernel=l2)
    return float((o * do).sum() + (0.0 if dht is None else (ht * dht).sum()))


@pytest.mark.parametrize("gate,h0,with_dht", [(True, True, True), (False, False, True),
                                              (True, True, False)])
def test_bwd_matches_finite_differences(gate, h0, with_dht):
    inp = _small(B=1, Nk=2, Nv=4, dk=5, dv=3, gate=gate, h0=h0, lengths=[7, 0, 70, 2], seed=95)
    inp = {key: (val.double().numpy().copy() if hasattr(val, "numpy") and key != "cu_seqlens"
                 else val) for key, val in inp.items()}
    if inp["g"] is None:
        inp["g"] = np.zeros_like(inp["beta"])   # differentiate at g = 0
    if inp["h0"] is None:
        inp["h0"] = np.zeros((4, 4, 5, 3))
    rng = np.random.default_rng(95)
    o, ht = _call(oracle.recurrent, inp)
    do = rng.standard_normal(o.shape)
    dht = rng.standard_normal(ht.shape) if with_dht else None
    gr = oracle.recurrent_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["h0"],
                              inp["cu_seqlens"], inp["scale"], do=do, dht=dht)
    eps = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "dbeta"), ("g", "dg"),
                        ("h0", "dh0")):
        x = inp[name].copy()
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(inp, do, dht, **{name: x})
            x[idx] = old - eps
            lm = _loss(inp, do, dht, **{name: x})
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        an = gr[gname]
        assert np.abs(fd - an).max() <= 1e-7 * max(np.abs(an).max(), 1.0), (name, gate, h0)


def test_bwd_groups_subset_matches_full():
    """Restricting the work to (sequence, key head) groups gives those groups'
    gradients bit for bit and leaves the rest NaN."""
    inp = _small(B=2, T=30, Nk=2, Nv=4, dk=6, dv=4, seed=96)
    rng = np.random.default_rng(96)
    o, ht = _call(oracle.recurrent, inp)
    do, dht = rng.standard_normal(o.shape), rng.standard_normal(ht.shape)
    args = (inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["h0"], inp["cu_seqlens"],
            inp["scale"])
    full = oracle.recurrent_bwd(*args, do=do, dht=dht)
    part = oracle.recurrent_bwd(*args, do=do, dht=dht, groups=[3])  # n = 1, hk = 1
    assert np.array_equal(part["dq"][1, :, 1], full["dq"][1, :, 1])
    assert np.array_equal(part["dv"][1, :, 2:], full["dv"][1, :, 2:])
    assert np.array_equal(part["dh0"][1, 2:], full["dh0"][1, 2:])
    assert np.isnan(part["dq"][0]).all() and np.isnan(part["dbeta"][1, :, :2]).all()


def test_bwd_l2norm_matches_finite_differences():
    """With in-kernel q / k normalisation, dq and dk (through the normalisation)
    and the other gradients against central differences of the normalised
    forward, on raw q / k rows of widely varying norm."""
    inp = workloads.make_inputs(1, 0, 2, 4, 5, 3, dtype=torch.float32, gate_mu=1.0, h0=True,
                                seed=97, lengths=[7, 0, 70, 2], raw_qk=True)
    inp = {key: (val.double().numpy().copy() if hasattr(val, "numpy") and key != "cu_seqlens"
                 else val) for key, val in inp.items()}
    rng = np.random.default_rng(97)
    o, ht = _call(oracle.recurrent, inp, use_qk_l2norm_in_kernel=True)
    do, dht = rng.standard_normal(o.shape), rng.standard_normal(ht.shape)
    gr = oracle.recurrent_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["h0"],
                              inp["cu_seqlens"], inp["scale"], do=do, dht=dht,
                              use_qk_l2norm_in_kernel=True)
    eps = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("beta", "dbeta"), ("g", "dg")):
        x = inp[name].copy()
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(inp, do, dht, True, **{name: x})
            x[idx] = old - eps
            lm = _loss(inp, do, dht, True, **{name: x})
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        an = gr[gname]
        assert np.abs(fd - an).max() <= 1e-7 * max(np.abs(an).max(), 1.0), name


def test_l2norm_bwd_closed_forms():
    """The gradient of x / ||x|| is orthogonal to x and scales as 1 / ||x||;
    below the guard it is dy / 1e-12."""
    rng = np.random.default_rng(98)
    x = rng.standard_normal((5, 7))
    dy = rng.standard_normal((5, 7))
    g = oracle.l2norm_bwd(x, dy)
    assert np.allclose((g * x).sum(-1), 0.0, atol=1e-13)
    assert np.allclose(oracle.l2norm_bwd(3.0 * x, dy), g / 3.0, rtol=1e-13)
    tiny = np.array([[1e-14, 0.0, 0.0]])
    assert np.allclose(oracle.l2norm_bwd(tiny, np.array([[1.0, 2.0, 3.0]])), [[1e12, 2e12, 3e12]])
