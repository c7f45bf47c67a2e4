"""Pins of the float64 backward oracle (no GPU).

The gradient oracles (oracle_tc_backward, oracle_delta_backward) are
hand-written reverse-mode passes of the per-token recurrences.  They are
pinned here against what does not share their derivation:
  * central finite differences of the forward oracle (which is pinned on its
    own in test_oracle_tc.py / test_oracle_delta.py);
  * torch float64 autograd through forward formulas written in a different
    form (dense masked matrices for the Tensor Cache layer, a chunk of torch
    ops per token for the delta rule), themselves checked against the forward
    oracle first;
  * for eta = 0, torch's scaled_dot_product_attention with a band mask (a
    library routine) under autograd;
  * exact identities of the layers: y is linear in v, m is linear in eta, the
    delta rule's output is linear in q and jointly linear in (v, S0), and
    the chain rule across a split of the sequence.
A dropped term, a wrong sign, a transposed state or an off-by-one in the
eviction step fails at least one of these.
"""
import numpy as np
import pytest
import torch

from outer_product_associative_chunked_b300 import synth

F64 = torch.float64


def _dy(shape, seed):
    return torch.randn(*shape, generator=torch.Generator().manual_seed(seed), dtype=F64)


# ------------------------------------------------------------------ Tensor Cache
def _tc_loss(oracle, q, k, v, lam, eta, gate, W, dy):
    y = oracle.tc_prefill(q, k, v, lam, eta, gate, W)["y"]
    return float((y * oracle.f64(dy)).sum())


TC_CASES = [
    # B, H, T, d_k, d_v, W
    (1, 1, 9, 3, 2, 1),
    (1, 2, 20, 4, 3, 5),
    (2, 1, 17, 2, 4, 16),
    (1, 1, 12, 3, 3, 40),   # W >= T: no eviction
]


@pytest.mark.parametrize("B,H,T,dk,dv,W", TC_CASES)
def test_tc_backward_finite_differences(oracle_mod, B, H, T, dk, dv, W):
    inp = synth.tc_inputs(B, H, T, dk, dv, W, dtype="f32", seed=T + W)
    dy = _dy((B, H, T, dv), 3)
    g = oracle_mod.tc_backward(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W, dy)
    base = {n: oracle_mod.f64(getattr(inp, n)) for n in ("q", "k", "v", "lam", "eta", "gate")}
    rng = np.random.default_rng(T)
    h = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("lam", "dlam"), ("eta", "deta"),
                        ("gate", "dgate")):
        x = base[name]
        picks = [tuple(rng.integers(0, s) for s in x.shape) for _ in range(4)]
        for idx in picks:
            args = dict(base)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args[name] = xp
            lp = _tc_loss(oracle_mod, args["q"], args["k"], args["v"], args["lam"], args["eta"], args["gate"],
                          W, dy)
            args[name] = xm
            lm = _tc_loss(oracle_mod, args["q"], args["k"], args["v"], args["lam"], args["eta"], args["gate"],
                          W, dy)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[gname][idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, g[gname][idx])


def _tc_dense_torch(q, k, v, lam, eta, gate, W, scale):
    """The layer in a dense form (no recurrence): a band-masked softmax and
    the L2 read m = (D * Q K^T) V with D[t, s] = eta lambda^(t-W-s) for
    s <= t-W; float64 torch ops, differentiable."""
    B, H, T, dk = q.shape
    t = torch.arange(T).view(T, 1)
    s = torch.arange(T).view(1, T)
    band = (s <= t) & (s > t - W)
    scores = scale * q @ k.transpose(-1, -2)
    p = torch.softmax(scores.masked_fill(~band, float("-inf")), dim=-1)
    y_loc = p @ v
    n = (t - W - s).to(F64)                           # exponent t-W-s
    mask = (s <= t - W)
    lam_b = lam.view(1, H, 1, 1)
    D = torch.where(mask, eta.view(1, H, 1, 1) * lam_b ** n.clamp_min(0), torch.zeros((), dtype=F64))
    m = (D * (q @ k.transpose(-1, -2))) @ v
    return y_loc + torch.sigmoid(gate).view(1, H, 1, 1) * m


@pytest.mark.parametrize("B,H,T,dk,dv,W", TC_CASES + [(2, 3, 40, 8, 6, 7)])
def test_tc_backward_matches_autograd_of_dense_form(oracle_mod, B, H, T, dk, dv, W):
    inp = synth.tc_inputs(B, H, T, dk, dv, W, dtype="f32", seed=100 + T)
    dy = _dy((B, H, T, dv), 4)
    xs = [getattr(inp, n).to(F64).requires_grad_(True) for n in ("q", "k", "v", "lam", "eta", "gate")]
    y = _tc_dense_torch(*xs, W, 1.0 / np.sqrt(dk))
    ref_y = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W)["y"]
    assert np.abs(y.detach().numpy() - ref_y).max() < 1e-12   # the dense form is the same layer
    (y * dy).sum().backward()
    g = oracle_mod.tc_backward(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W, dy)
    for x, name in zip(xs, ("dq", "dk", "dv", "dlam", "deta", "dgate")):
        np.testing.assert_allclose(g[name], x.grad.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)


def test_tc_backward_eta_zero_is_windowed_sdpa(oracle_mod):
    """With eta = 0 the layer is band-masked softmax attention, whose gradient
    torch computes through scaled_dot_product_attention."""
    B, H, T, d, W = 2, 2, 33, 8, 6
    inp = synth.tc_inputs(B, H, T, d, d, W, dtype="f32", seed=8, eta=0.0)
    dy = _dy((B, H, T, d), 5)
    q, k, v = (getattr(inp, n).to(F64).requires_grad_(True) for n in ("q", "k", "v"))
    t = torch.arange(T).view(T, 1)
    s = torch.arange(T).view(1, T)
    band = (s <= t) & (s > t - W)
    y = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=band)
    (y * dy).sum().backward()
    g = oracle_mod.tc_backward(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W, dy)
    for x, name in zip((q, k, v), ("dq", "dk", "dv")):
        np.testing.assert_allclose(g[name], x.grad.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)
    assert np.all(g["dgate"] == 0.0)


def test_tc_backward_identities(oracle_mod):
    B, H, T, dk, dv, W = 2, 3, 50, 5, 4, 9
    inp = synth.tc_inputs(B, H, T, dk, dv, W, dtype="f32", seed=12)
    dy = _dy((B, H, T, dv), 6)
    g = oracle_mod.tc_backward(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W, dy)
    fw = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W, want_m=True)
    dyn = dy.numpy()
    # y is linear in v: <dL/dv, v> = L
    assert np.isclose((g["dv"] * oracle_mod.f64(inp.v)).sum(), (fw["y"] * dyn).sum(), rtol=1e-10)
    # m is linear in eta: eta dL/deta = sigmoid(g) sum <dy, m> per head, and
    # dL/dg = sigmoid'(g) sum <dy, m>
    dym = (dyn * fw["m"]).sum(axis=(0, 2, 3))
    sg = 1.0 / (1.0 + np.exp(-oracle_mod.f64(inp.gate)))
    np.testing.assert_allclose(oracle_mod.f64(inp.eta) * g["deta"], sg * dym, rtol=1e-10)
    np.testing.assert_allclose(g["dgate"], sg * (1 - sg) * dym, rtol=1e-10)


# ------------------------------------------------------------------ DeltaNet
def _delta_loss(oracle, q, k, v, beta, S0, dy):
    y = oracle.delta(q, k, v, beta, S0=S0)["y"]
    return float((y * oracle.f64(dy)).sum())


def _delta_torch(q, k, v, beta, S0):
    """Per-token torch ops: S (d_v x d_k) <- S + beta (v - S k) k^T, o = S q."""
    B, H, T, dk = q.shape
    S = S0.transpose(-1, -2)                          # key-major [d_k, d_v] -> S [d_v, d_k]
    outs = []
    for t in range(T):
        kt = k[:, :, t].unsqueeze(-1)
        err = v[:, :, t].unsqueeze(-1) - S @ kt
        S = S + beta[:, :, t].view(B, H, 1, 1) * err @ kt.transpose(-1, -2)
        outs.append((S @ q[:, :, t].unsqueeze(-1)).squeeze(-1))
    return torch.stack(outs, dim=2), S.transpose(-1, -2)


DELTA_CASES = [(1, 1, 6, 3, 2), (2, 2, 13, 4, 5), (1, 3, 20, 6, 6)]


@pytest.mark.parametrize("B,H,T,dk,dv", DELTA_CASES)
def test_delta_backward_matches_autograd(oracle_mod, B, H, T, dk, dv):
    inp = synth.delta_inputs(B, H, T, dk, dv, dtype="f32", seed=T)
    S0 = torch.randn(B, H, dk, dv, generator=torch.Generator().manual_seed(T), dtype=F64) * 0.3
    dy = _dy((B, H, T, dv), 7)
    dST = _dy((B, H, dk, dv), 8)
    xs = [getattr(inp, n).to(F64).requires_grad_(True) for n in ("q", "k", "v", "beta")]
    s0 = S0.clone().requires_grad_(True)
    y, ST = _delta_torch(*xs, s0)
    ref = oracle_mod.delta(inp.q, inp.k, inp.v, inp.beta, S0=S0, want_state=True)
    assert np.abs(y.detach().numpy() - ref["y"]).max() < 1e-12
    ((y * dy).sum() + (ST * dST).sum()).backward()
    g = oracle_mod.delta_backward(inp.q, inp.k, inp.v, inp.beta, dy, S0=S0, dS_T=dST)
    for x, name in zip(xs + [s0], ("dq", "dk", "dv", "dbeta", "dS0")):
        np.testing.assert_allclose(g[name], x.grad.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)


def test_delta_backward_finite_differences(oracle_mod):
    B, H, T, dk, dv = 1, 2, 11, 4, 3
    inp = synth.delta_inputs(B, H, T, dk, dv, dtype="f32", seed=31)
    S0 = oracle_mod.f64(torch.randn(B, H, dk, dv, generator=torch.Generator().manual_seed(2)) * 0.5)
    dy = _dy((B, H, T, dv), 9)
    g = oracle_mod.delta_backward(inp.q, inp.k, inp.v, inp.beta, dy, S0=S0)
    base = {n: oracle_mod.f64(getattr(inp, n)) for n in ("q", "k", "v", "beta")}
    base["S0"] = S0
    rng = np.random.default_rng(5)
    h = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "dbeta"), ("S0", "dS0")):
        x = base[name]
        for _ in range(5):
            idx = tuple(rng.integers(0, s) for s in x.shape)
            args = dict(base)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args[name] = xp
            lp = _delta_loss(oracle_mod, args["q"], args["k"], args["v"], args["beta"], args["S0"], dy)
            args[name] = xm
            lm = _delta_loss(oracle_mod, args["q"], args["k"], args["v"], args["beta"], args["S0"], dy)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[gname][idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, g[gname][idx])


def test_delta_backward_identities_and_chain_rule(oracle_mod):
    B, H, T, dk, dv = 2, 2, 24, 5, 4
    inp = synth.delta_inputs(B, H, T, dk, dv, dtype="f32", seed=41)
    S0 = oracle_mod.f64(torch.randn(B, H, dk, dv, generator=torch.Generator().manual_seed(3)) * 0.4)
    dy = _dy((B, H, T, dv), 10).numpy()
    g = oracle_mod.delta_backward(inp.q, inp.k, inp.v, inp.beta, dy, S0=S0)
    y = oracle_mod.delta(inp.q, inp.k, inp.v, inp.beta, S0=S0)["y"]
    L = (y * dy).sum()
    q, v = oracle_mod.f64(inp.q), oracle_mod.f64(inp.v)
    # o is linear in q, and jointly linear in (v, S0)
    assert np.isclose((g["dq"] * q).sum(), L, rtol=1e-10)
    assert np.isclose((g["dv"] * v).sum() + (g["dS0"] * S0).sum(), L, rtol=1e-10)
    # chain rule across a split at T0: the second half's dS0 is the first
    # half's final-state gradient
    T0 = 10
    sl = lambda x, a, b: x[:, :, a:b]  # noqa: E731
    first = oracle_mod.delta(sl(inp.q, 0, T0), sl(inp.k, 0, T0), sl(inp.v, 0, T0), sl(inp.beta, 0, T0), S0=S0,
                             want_state=True)
    g2 = oracle_mod.delta_backward(sl(inp.q, T0, T), sl(inp.k, T0, T), sl(inp.v, T0, T), sl(inp.beta, T0, T),
                                   dy[:, :, T0:], S0=first["S"])
    g1 = oracle_mod.delta_backward(sl(inp.q, 0, T0), sl(inp.k, 0, T0), sl(inp.v, 0, T0), sl(inp.beta, 0, T0),
                                   dy[:, :, :T0], S0=S0, dS_T=g2["dS0"])
    for name in ("dq", "dk", "dv", "dbeta"):
        np.testing.assert_allclose(np.concatenate([g1[name], g2[name]], axis=2), g[name], rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(g1["dS0"], g["dS0"], rtol=1e-9, atol=1e-12)
    # beta = 0: the state never changes, so o_t = S0 q_t; v and k get no gradient
    z = oracle_mod.delta_backward(inp.q, inp.k, inp.v, np.zeros((B, H, T)), dy, S0=S0)
    assert np.all(z["dv"] == 0.0) and np.all(z["dk"] == 0.0)
    np.testing.assert_allclose(z["dq"], np.einsum("bhji,bhti->bhtj", S0, dy), rtol=1e-12)
