"""Pins of the oracle's linear layer and attention block (CPU only).

The linear layer is pinned against a hand-worked product, against the
definition summed element by element in plain Python (brute force on a tiny
case), against identities that fix the operand order (identity and
permutation weights, the transpose), and against torch.nn.functional.linear
in float64; the block against the composition of its parts and the attention
oracle's own pins (first query row = v of token 0 projected).
"""
import numpy as np
import pytest

import oracle


def test_hand_worked_example():
    # inp (2 x 3), weight (OC = 2, K = 3), bias (2)
    inp = np.array([[1.0, 2.0, 3.0], [-1.0, 0.5, 4.0]])
    w = np.array([[1.0, 0.0, -1.0], [2.0, 1.0, 0.5]])
    b = np.array([0.25, -1.0])
    # row 0: 1-3 = -2 (+0.25) ; 2+2+1.5 = 5.5 (-1)
    # row 1: -1-4 = -5 (+0.25); -2+0.5+2 = 0.5 (-1)
    want = np.array([[-1.75, 4.5], [-4.75, -0.5]])
    assert np.array_equal(oracle.linear(inp, w, b), want)


def test_brute_force_tiny():
    rng = np.random.default_rng(3)
    inp = rng.standard_normal((3, 5))
    w = rng.standard_normal((4, 5))
    b = rng.standard_normal(4)
    got = oracle.linear(inp, w, b)
    for m in range(3):
        for o in range(4):
            s = b[o]
            for k in range(5):
                s += inp[m, k] * w[o, k]
            assert abs(got[m, o] - s) <= 1e-12


def test_operand_order_identities():
    rng = np.random.default_rng(4)
    inp = rng.standard_normal((6, 8))
    assert np.allclose(oracle.linear(inp, np.eye(8)), inp, rtol=0, atol=1e-15)
    perm = rng.permutation(8)
    w = np.eye(8)[perm]                      # out[:, o] = inp[:, perm[o]]
    assert np.array_equal(oracle.linear(inp, w), inp[:, perm])
    w2 = rng.standard_normal((3, 8))
    assert np.allclose(oracle.linear(inp, w2), (w2 @ inp.T).T, rtol=0, atol=1e-12)
    assert np.array_equal(oracle.linear(inp, w2, np.zeros(3)), oracle.linear(inp, w2))


def test_against_torch_float64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    inp = rng.standard_normal((2, 7, 16))
    w = rng.standard_normal((48, 16))
    b = rng.standard_normal(48)
    ref = torch.nn.functional.linear(torch.from_numpy(inp), torch.from_numpy(w), torch.from_numpy(b)).numpy()
    assert np.allclose(oracle.linear(inp, w, b), ref, rtol=0, atol=1e-12)


def test_block_is_the_composition_and_row0_is_projected_v0():
    rng = np.random.default_rng(6)
    B, T, C, NH = 2, 9, 16, 2
    x = rng.standard_normal((B, T, C))
    w_attn, b_attn = rng.standard_normal((3 * C, C)) * 0.2, rng.standard_normal(3 * C) * 0.1
    w_proj, b_proj = rng.standard_normal((C, C)) * 0.2, rng.standard_normal(C) * 0.1
    y, qkv, out, lse = oracle.block_forward(x, w_attn, b_attn, w_proj, b_proj, NH, True)
    assert np.allclose(qkv, oracle.linear(x, w_attn, b_attn), rtol=0, atol=1e-12)
    o2, l2 = oracle.forward(qkv, B, T, C, NH, True)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)
    assert np.allclose(y, oracle.linear(out, w_proj, b_proj), rtol=0, atol=1e-12)
    # causal: token 0 attends only to itself, so out_0 = v_0 and y_0 = proj(v_0)
    v0 = qkv[:, 0, 2 * C:]
    assert np.allclose(y[:, 0], oracle.linear(v0, w_proj, b_proj), rtol=0, atol=1e-12)
