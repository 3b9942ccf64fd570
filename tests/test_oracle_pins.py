"""Pins for the CPU oracle: checks against facts that do not come from the oracle itself.

Each test names the fact it relies on: a hand-worked example, a closed form, an
invariant of softmax attention, a library routine (torch float64 SDPA and
autograd), or finite differences. A last test plants mistakes in the oracle and
checks that the pins catch every one.
"""
import json
import math
import pathlib
import types

import numpy as np
import pytest

import oracle
import oracle.attention as oa
from causal_head_attention_fwd_gb300 import inputs

GOLDEN = pathlib.Path(__file__).parent / "golden"


def _ev(x):
    if isinstance(x, (int, float)):
        return float(x)
    names = {"ln3": math.log(3), "ln4": math.log(4), "ln5": math.log(5), "ln8": math.log(8)}
    return float(eval(x, {"__builtins__": {}}, names))  # fixture expressions only


def _arr(rows):
    return np.array([[_ev(x) for x in r] for r in rows], dtype=np.float64)


def _qkv_from(q, k, v):
    return np.concatenate([q, k, v], axis=1)[None]  # (1, T, 3C)


def _rand(B, T, C, NH, seed=7, sigma=1.0):
    x, _ = inputs.draw((B, T, 3 * C), sigma, seed, "f32")
    d, _ = inputs.draw((B, T, C), 1.0, seed + 1, "f32")
    return x.astype(np.float64), d.astype(np.float64)


# ---------------------------------------------------------------- worked example
def test_worked_example_forward_and_backward():
    g = json.loads((GOLDEN / "worked_example_T3.json").read_text())
    q, k, v, dout = _arr(g["q"]), _arr(g["k"]), _arr(g["v"]), _arr(g["dout"])
    qkv = _qkv_from(q, k, v)
    B, T, C, NH = g["B"], g["T"], g["C"], g["NH"]
    out, lse = oracle.forward(qkv, B, T, C, NH, causal=True)
    np.testing.assert_allclose(out[0], _arr(g["causal"]["out"]), atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [_ev(x) for x in g["causal"]["lse"]], atol=1e-14)
    out, lse = oracle.forward(qkv, B, T, C, NH, causal=False)
    np.testing.assert_allclose(out[0], _arr(g["noncausal"]["out"]), atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [_ev(x) for x in g["noncausal"]["lse"]], atol=1e-14)
    dqkv = oracle.backward(dout[None], qkv, B, T, C, NH, causal=True)
    np.testing.assert_allclose(dqkv[0, :, 0:C], _arr(g["causal"]["dq"]), atol=1e-14)
    np.testing.assert_allclose(dqkv[0, :, C:2 * C], _arr(g["causal"]["dk"]), atol=1e-14)
    np.testing.assert_allclose(dqkv[0, :, 2 * C:], _arr(g["causal"]["dv"]), atol=1e-14)


# ---------------------------------------------------------------- forward invariants
@pytest.mark.parametrize("causal", [True, False])
def test_att_rows_sum_to_one_and_mask(causal):
    x, _ = _rand(1, 37, 64, 2)
    q, k, v = oracle.split_heads(x, 64, 2)
    _, _, att, _ = oracle.head_forward(q[0, 1], k[0, 1], v[0, 1], causal, return_att=True)
    np.testing.assert_allclose(att.sum(axis=1), 1.0, atol=1e-14)
    assert np.all(att >= 0)
    if causal:
        assert np.all(att[np.triu_indices(37, 1)] == 0.0)
    else:
        assert np.all(att > 0)


@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_first_row_is_v0_for_every_workload_shape(name):
    """Causal row t=0 sees only key 0, so out[b, 0] = v_0 exactly (for ViT, the
    non-causal shape, the same holds with the causal mask switched on)."""
    w = inputs.WORKLOADS[name]
    T = min(w.T, 9)
    x, _ = _rand(2, T, w.C, w.NH, seed=11)
    out, _ = oracle.forward(x, 2, T, w.C, w.NH, causal=True)
    np.testing.assert_array_equal(out[:, 0, :], x[:, 0, 2 * w.C:])


def test_T1_closed_form():
    x, d = _rand(3, 1, 96, 3)
    out, lse = oracle.forward(x, 3, 1, 96, 3, causal=True)
    np.testing.assert_array_equal(out, x[:, :, 192:])
    q, k, _ = oracle.split_heads(x, 96, 3)
    np.testing.assert_allclose(lse[:, :, 0], (q * k).sum(-1)[:, :, 0] / math.sqrt(32), rtol=1e-14)
    dqkv = oracle.backward(d, x, 3, 1, 96, 3, causal=True)
    assert np.all(dqkv[:, :, :192] == 0.0)
    np.testing.assert_array_equal(dqkv[:, :, 192:], d)


@pytest.mark.parametrize("causal", [True, False])
def test_uniform_keys_give_prefix_mean(causal):
    B, T, C, NH = 2, 23, 32, 2
    x, _ = _rand(B, T, C, NH, seed=5)
    x[:, :, C:2 * C] = x[:, :1, C:2 * C]          # every key equal to key 0
    out, lse = oracle.forward(x, B, T, C, NH, causal)
    v = x[:, :, 2 * C:]
    if causal:
        expect = np.cumsum(v, axis=1) / np.arange(1, T + 1)[None, :, None]
        count = np.arange(1, T + 1)
    else:
        expect = np.broadcast_to(v.mean(axis=1, keepdims=True), v.shape)
        count = np.full(T, T)
    np.testing.assert_allclose(out, expect, atol=1e-13)
    q, k, _ = oracle.split_heads(x, C, NH)
    s = (q * k[:, :, :1]).sum(-1) / math.sqrt(C // NH)
    np.testing.assert_allclose(lse, s + np.log(count)[None, None], atol=1e-12)


def test_key_shift_invariance():
    B, T, C, NH = 1, 19, 64, 2
    x, _ = _rand(B, T, C, NH, seed=9)
    out0, lse0 = oracle.forward(x, B, T, C, NH, True)
    c = np.linspace(-1, 1, C)
    y = x.copy()
    y[:, :, C:2 * C] += c
    out1, lse1 = oracle.forward(y, B, T, C, NH, True)
    np.testing.assert_allclose(out1, out0, atol=1e-12)
    q, _, _ = oracle.split_heads(x, C, NH)
    shift = np.einsum("bhti,hi->bht", q, c.reshape(NH, C // NH)) / math.sqrt(C // NH)
    np.testing.assert_allclose(lse1, lse0 + shift, atol=1e-12)


def test_out_linear_in_v():
    B, T, C, NH = 1, 17, 64, 4
    x, _ = _rand(B, T, C, NH, seed=2)
    y = x.copy()
    y[:, :, 2 * C:] = np.random.default_rng(0).normal(size=(B, T, C))
    z = x.copy()
    z[:, :, 2 * C:] = 2.0 * x[:, :, 2 * C:] - 3.0 * y[:, :, 2 * C:]
    ox, _ = oracle.forward(x, B, T, C, NH, True)
    oy, _ = oracle.forward(y, B, T, C, NH, True)
    oz, _ = oracle.forward(z, B, T, C, NH, True)
    np.testing.assert_allclose(oz, 2 * ox - 3 * oy, atol=1e-12)


# ---------------------------------------------------------------- library cross-check
@pytest.mark.parametrize("causal", [True, False])
def test_against_torch_sdpa_float64(causal):
    torch = pytest.importorskip("torch")
    B, T, C, NH = 2, 29, 96, 3
    x, d = _rand(B, T, C, NH, seed=21)
    out, lse = oracle.forward(x, B, T, C, NH, causal)
    dqkv = oracle.backward(d, x, B, T, C, NH, causal)
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    q, k, v = xt.split(C, dim=2)
    sh = lambda t: t.view(B, T, NH, C // NH).transpose(1, 2)
    o = torch.nn.functional.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=causal)
    o = o.transpose(1, 2).reshape(B, T, C)
    o.backward(torch.tensor(d, dtype=torch.float64))
    np.testing.assert_allclose(out, o.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(dqkv, xt.grad.numpy(), atol=1e-12)
    # lse against torch.logsumexp of the scaled, masked scores
    s = sh(q) @ sh(k).transpose(-1, -2) / math.sqrt(C // NH)
    if causal:
        s = s.masked_fill(torch.ones(T, T, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).detach().numpy(), atol=1e-12)


# ---------------------------------------------------------------- backward
def test_finite_differences_all_elements_tiny():
    """Central differences of L = <dout, out(qkv)> w.r.t. every qkv element."""
    B, T, C, NH = 1, 6, 8, 2
    x, d = _rand(B, T, C, NH, seed=3)
    g = oracle.backward(d, x, B, T, C, NH, causal=True)
    eps = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += eps
        xm[idx] -= eps
        lp = (oracle.forward(xp, B, T, C, NH, True)[0] * d).sum()
        lm = (oracle.forward(xm, B, T, C, NH, True)[0] * d).sum()
        fd[idx] = (lp - lm) / (2 * eps)
    np.testing.assert_allclose(g, fd, atol=1e-8)


@pytest.mark.parametrize("causal", [True, False])
def test_directional_derivative_larger_shape(causal):
    B, T, C, NH = 2, 70, 64, 2
    x, d = _rand(B, T, C, NH, seed=13)
    g = oracle.backward(d, x, B, T, C, NH, causal)
    delta = np.random.default_rng(1).normal(size=x.shape)
    eps = 1e-5
    lp = (oracle.forward(x + eps * delta, B, T, C, NH, causal)[0] * d).sum()
    lm = (oracle.forward(x - eps * delta, B, T, C, NH, causal)[0] * d).sum()
    assert abs((lp - lm) / (2 * eps) - (g * delta).sum()) < 1e-7 * max(1.0, abs((g * delta).sum()))


@pytest.mark.parametrize("causal", [True, False])
def test_jacobian_form_equals_rowsum_form(causal):
    x, d = _rand(1, 31, 64, 2, seed=4)
    q, k, v = oracle.split_heads(x, 64, 2)
    do = d.reshape(1, 31, 2, 32).transpose(0, 2, 1, 3)
    _, _, _, parts = oracle.head_backward(q[0, 0], k[0, 0], v[0, 0], do[0, 0], causal, return_parts=True)
    jac = oracle.head_dpreatt_jacobian(parts["att"], parts["datt"], causal) / math.sqrt(32)
    np.testing.assert_allclose(jac, parts["dpreatt"], atol=1e-14, rtol=1e-12)


def test_backward_structural_identities():
    B, T, C, NH = 2, 45, 64, 2
    x, d = _rand(B, T, C, NH, seed=17)
    g = oracle.backward(d, x, B, T, C, NH, causal=True)
    hs = C // NH
    dq = g[:, :, :C].reshape(B, T, NH, hs)
    dk = g[:, :, C:2 * C].reshape(B, T, NH, hs)
    dv = g[:, :, 2 * C:].reshape(B, T, NH, hs)
    assert np.all(dq[:, 0] == 0.0)                    # query 0 sees one key: no gradient
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)      # each dS row sums to 0
    np.testing.assert_allclose(dv.sum(axis=1), d.reshape(B, T, NH, hs).sum(axis=1), atol=1e-12)
    g2 = oracle.backward(-2.5 * d, x, B, T, C, NH, causal=True)
    np.testing.assert_allclose(g2, -2.5 * g, atol=1e-12)


def test_row_stat_D_equals_local_sum():
    B, T, C, NH = 1, 33, 64, 2
    x, d = _rand(B, T, C, NH, seed=23)
    out, _ = oracle.forward(x, B, T, C, NH, True)
    D = oracle.row_stat_D(d, out, B, T, C, NH)
    q, k, v = oracle.split_heads(x, C, NH)
    do = d.reshape(B, T, NH, C // NH).transpose(0, 2, 1, 3)
    for h in range(NH):
        _, _, _, parts = oracle.head_backward(q[0, h], k[0, h], v[0, h], do[0, h], True, return_parts=True)
        np.testing.assert_allclose(D[0, h], parts["D"], atol=1e-13)


# ---------------------------------------------------------------- planted mistakes
def _pins_pass():
    try:
        test_worked_example_forward_and_backward()
        test_against_torch_sdpa_float64(True)
        test_against_torch_sdpa_float64(False)
        test_uniform_keys_give_prefix_mean(True)
        test_finite_differences_all_elements_tiny()
    except AssertionError:
        return False
    return True


class _NpProxy(types.SimpleNamespace):
    def __getattr__(self, name):
        return getattr(np, name)


@pytest.mark.parametrize("mutation", ["scale_1_over_hs", "mask_transposed", "lse_log2",
                                      "exp_base2", "att_not_normalised"])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    pytest.importorskip("torch")
    assert _pins_pass()
    if mutation == "scale_1_over_hs":
        monkeypatch.setattr(oa, "math", types.SimpleNamespace(sqrt=lambda x: x))
    elif mutation == "mask_transposed":
        monkeypatch.setattr(oa, "_allowed", lambda T, c: np.triu(np.ones((T, T), bool)) if c else np.ones((T, T), bool))
    elif mutation == "lse_log2":
        monkeypatch.setattr(oa, "np", _NpProxy(log=np.log2))
    elif mutation == "exp_base2":
        monkeypatch.setattr(oa, "np", _NpProxy(exp=np.exp2))
    elif mutation == "att_not_normalised":
        real = oa.head_forward

        def broken(q, k, v, causal, return_att=False):
            out, lse, att, pre = real(q, k, v, causal, return_att=True)
            att = att * (1.0 + 1e-3)
            out = att @ v
            return (out, lse, att, pre) if return_att else (out, lse)
        monkeypatch.setattr(oa, "head_forward", broken)
    assert not _pins_pass(), f"mutation {mutation} was not caught by the pins"
