"""Pins for the BDH-style additive linear-attention oracle (CPU only).

Pages: ainews.random.gg BDH memory-architecture post (keys and queries are
non-negative neuron activations in a very wide space; the state is the
accumulated connectivity and reading it is propagation; it acts like a noisy
fixed-size hash table that sparse keys write a few buckets of) and mo.ai.kr
"Hebbian memory MLP", simple MLP construction (W = sum_i v_i k_i^T, read as a
similarity-weighted sum of values).  molayo1419.me, "the additive-write
problem of linear attention": after writing v_t under a unit-norm key,
re-reading that key gives S_{t-1} k_t + v_t.
"""
import numpy as np
import pytest
import torch

from helpers import load_golden
from outer_product_associative_chunked_b300 import synth


def test_hand_worked_onehot_buckets(oracle_mod):
    g = load_golden("bdh_onehot_n4.txt")
    out = oracle_mod.sparse_linattn(g["q"][None, None], g["k"][None, None], g["v"][None, None])
    np.testing.assert_allclose(out["y"][0, 0], g["y"], rtol=0, atol=0)


def _brute(q, k, v):
    T, N, dv = len(q), len(q[0]), len(v[0])
    ys = []
    for t in range(T):
        y = [0.0] * dv
        for s in range(t + 1):
            d = sum(k[s][j] * q[t][j] for j in range(N))
            for i in range(dv):
                y[i] += d * v[s][i]
        ys.append(y)
    return np.array(ys)


@pytest.mark.parametrize("T,N,dv", [(16, 12, 3), (1, 5, 2), (9, 40, 4)])
def test_bruteforce_small(oracle_mod, T, N, dv):
    rng = np.random.default_rng(T + N)
    q = np.maximum(rng.standard_normal((1, 1, T, N)) - 1.0, 0)
    k = np.maximum(rng.standard_normal((1, 1, T, N)) - 1.0, 0)
    v = rng.standard_normal((1, 1, T, dv))
    out = oracle_mod.sparse_linattn(q, k, v)
    ref = _brute(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist())
    np.testing.assert_allclose(out["y"][0, 0], ref, rtol=1e-12, atol=1e-12)


def test_additive_reread(oracle_mod):
    """Unit-norm key: S_t k_t = S_{t-1} k_t + v_t ('+=' not '='); in general
    the new value comes back scaled by ||k_t||^2."""
    rng = np.random.default_rng(9)
    T, N, dv = 6, 10, 4
    q = rng.random((1, 1, T, N))
    k = rng.random((1, 1, T, N))
    v = rng.standard_normal((1, 1, T, dv))
    k[0, 0, T - 1] /= np.linalg.norm(k[0, 0, T - 1])
    prev = oracle_mod.sparse_linattn(q[:, :, :T - 1], k[:, :, :T - 1], v[:, :, :T - 1], want_state=True)
    cur = oracle_mod.sparse_linattn(q, k, v, want_state=True)
    kt = k[0, 0, T - 1].copy()
    Sp, St = prev["S"][0, 0].T, cur["S"][0, 0].T
    np.testing.assert_allclose(St @ kt, Sp @ kt + v[0, 0, T - 1], rtol=1e-13, atol=1e-14)
    k2 = 3.0 * kt
    k[0, 0, T - 1] = k2
    cur2 = oracle_mod.sparse_linattn(q, k, v, want_state=True)
    np.testing.assert_allclose(cur2["S"][0, 0].T @ kt, Sp @ kt + 3.0 * v[0, 0, T - 1], rtol=1e-13)


def test_dense_causal_form_with_initial_state(oracle_mod):
    """Unrolled: o = Q S0^T + tril(Q K^T) V, and S_T = S0 + V^T K."""
    rng = np.random.default_rng(10)
    B, H, T, N, dv = 1, 2, 30, 25, 6
    q = np.maximum(rng.standard_normal((B, H, T, N)), 0)
    k = np.maximum(rng.standard_normal((B, H, T, N)), 0)
    v = rng.standard_normal((B, H, T, dv))
    S0 = rng.standard_normal((B, H, N, dv))
    out = oracle_mod.sparse_linattn(q, k, v, S0=S0, want_state=True)
    for h in range(H):
        ref = q[0, h] @ S0[0, h] + np.tril(q[0, h] @ k[0, h].T) @ v[0, h]
        np.testing.assert_allclose(out["y"][0, h], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(out["S"][0, h], S0[0, h] + k[0, h].T @ v[0, h], rtol=1e-12, atol=1e-12)


def test_closed_form_positions(oracle_mod):
    inp = synth.sparse_inputs(1, 1, 40, 256, 8, seed=11)
    S0 = np.random.default_rng(11).standard_normal((1, 1, 256, 8))
    out = oracle_mod.sparse_linattn(inp.q, inp.k, inp.v, S0=S0)
    ts = [0, 1, 17, 39]
    y = oracle_mod.sparse_linattn_output_at(inp.q[0, 0], inp.k[0, 0], inp.v[0, 0], ts, S0=S0[0, 0])
    np.testing.assert_allclose(y, out["y"][0, 0, ts], rtol=1e-12, atol=1e-12)


def test_synthetic_keys_are_sparse_and_nonnegative():
    inp = synth.sparse_inputs(1, 2, 64, 4096, 8, seed=12)
    for x in (inp.q, inp.k):
        assert torch.all(x >= 0)
        dens = float((x > 0).double().mean())
        assert 0.04 < dens < 0.06, dens


# ------------------------------------------------------------------ key generation
def test_bdh_keys_match_library_matmul(oracle_mod):
    """oracle.bdh_keys against torch's float64 matmul and ReLU."""
    import torch
    g = torch.Generator().manual_seed(3)
    x = torch.randn(2, 3, 5, 16, generator=g, dtype=torch.float64)
    U = torch.randn(3, 16, 40, generator=g, dtype=torch.float64) / 4
    for theta in (-0.5, 0.0, 0.7):
        ref = torch.relu(torch.einsum("bhtr,hrn->bhtn", x, U) - theta).numpy()
        np.testing.assert_allclose(oracle_mod.bdh_keys(x, U, theta), ref, rtol=1e-13, atol=1e-14)


def test_bdh_keys_reproduce_the_recipe(oracle_mod):
    """From the same inputs, the oracle's keys are the recipe's float32 keys
    up to float32 rounding, and the 95th-percentile threshold keeps about 5%
    of the entries; a very low threshold keeps every positive pre-activation
    (shifted), a very high one none."""
    from outer_product_associative_chunked_b300 import synth
    import torch
    kg = synth.sparse_keygen_inputs(1, 2, 64, 4096, 8, seed=7)
    keys = oracle_mod.bdh_keys(kg.xk, kg.U, kg.theta)
    f32 = torch.relu(torch.einsum("bhtr,hrn->bhtn", kg.xk.float(), kg.U.float()) - kg.theta).double().numpy()
    assert np.abs(keys - f32).max() < 1e-5
    dens = float((keys > 0).mean())
    assert 0.04 < dens < 0.06, dens
    assert np.all(oracle_mod.bdh_keys(kg.xk, kg.U, 1e3) == 0.0)
    low = oracle_mod.bdh_keys(kg.xk, kg.U, -1e3)
    pre = np.einsum("bhtr,hrn->bhtn", oracle_mod.f64(kg.xk), oracle_mod.f64(kg.U))
    np.testing.assert_allclose(low, pre + 1e3, rtol=1e-14)
