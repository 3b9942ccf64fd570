"""llm.c drop-in mode: attn_fwd_att materialises preatt and att (B, NH, T, T).

Checked against the oracle's per-head preatt (q.k without the scale, the full
matrix) and att (softmax over J(t), zeros elsewhere) on the same seeded inputs:
- bf16 inputs: products are exact in fp32, so preatt matches to fp32 rounding
  (1e-4 of its largest magnitude) and att to 1e-4 absolute (att <= 1; the
  rest is ex2.approx and the fp32 lse);
- fp32 inputs: the tensor core reads q and k as tf32 (each loses < 2^-10 of its
  magnitude), so each preatt moves by at most 2^-9 * sum_i |q_i k_i|; att, an
  exponential of scale*preatt - lse, moves by at most twice the scaled bound
  (its own preatt and, through lse, the row's largest one).
Masked entries must be exactly 0 and every row of att must sum to 1.
"""
import numpy as np
import pytest

import oracle
from causal_head_attention_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_head_attention_fwd_gb300 import build
    build.build()
    from causal_head_attention_fwd_gb300 import api, ops
    return torch, api, ops


def _oracle_mats(x, B, T, C, NH, causal):
    hs = C // NH
    pre = np.zeros((B, NH, T, T))
    att = np.zeros((B, NH, T, T))
    w = np.zeros((B, NH))
    q, k, v = oracle.split_heads(x, C, NH)              # each (B, NH, T, hs)
    for b in range(B):
        for h in range(NH):
            _, _, a, p = oracle.head_forward(q[b, h], k[b, h], v[b, h], causal, return_att=True)
            att[b, h], pre[b, h] = a, p
            w[b, h] = np.max(np.abs(q[b, h]) @ np.abs(k[b, h]).T)
    return pre, att, w


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,T,C,NH,causal", [
    (1, 1, 128, 2, 1), (2, 64, 128, 4, 1), (1, 130, 128, 2, 1), (2, 127, 64, 1, 0),
    (1, 257, 64, 1, 1), (1, 300, 128, 2, 0), (1, 333, 128, 2, 1),
])
def test_matrices_match_the_oracle(env, dtype, B, T, C, NH, causal):
    torch, api, ops = env
    host = inputs.make_inputs(B, T, C, NH, dtype, 0.5, 1e-2, 50 + T, 60 + T)
    qkv = ops.upload(host.qkv_dev, dtype)
    out, lse = ops.attention_forward(qkv, NH, bool(causal))
    pre, att = ops.attention_matrices(qkv, lse, NH, bool(causal))
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    rpre, ratt, w = _oracle_mats(host.qkv.astype(np.float64), B, T, C, NH, bool(causal))
    gpre, gatt = ops.download_f64(pre), ops.download_f64(att)
    assert np.isfinite(gpre).all() and np.isfinite(gatt).all()
    hs = C // NH
    if dtype == "bf16":
        assert np.max(np.abs(gpre - rpre)) <= 1e-4 * max(np.max(np.abs(rpre)), 1e-30)
        assert np.max(np.abs(gatt - ratt)) <= 1e-4
    else:
        bound = 2.0 ** -9 * w.max()
        assert np.max(np.abs(gpre - rpre)) <= bound + 1e-5
        assert np.max(np.abs(gatt - ratt)) <= 2 * bound / np.sqrt(hs) + 1e-4
    np.testing.assert_allclose(gatt.sum(axis=-1), 1.0, atol=1e-3)
    if causal:
        upper = np.triu(np.ones((T, T), dtype=bool), 1)
        assert np.all(gatt[:, :, upper] == 0.0)


def test_one_output_may_be_skipped_and_no_out_of_bounds_writes(env):
    torch, api, ops = env
    B, T, C, NH, G = 1, 250, 128, 2, 1024
    host = inputs.make_inputs(B, T, C, NH, "bf16", 0.5, 1e-2, 71, 72)
    qkv = ops.upload(host.qkv_dev, "bf16")
    out, lse = ops.attention_forward(qkv, NH, True)
    n = B * NH * T * T
    big = torch.full((n + 2 * G,), float("nan"), dtype=torch.float32, device="cuda")
    att = big[G:G + n].view(B, NH, T, T)
    pre, got = ops.attention_matrices(qkv, lse, NH, True, preatt=False, att=att)
    torch.cuda.synchronize()
    assert pre is None and got is att
    assert not torch.isnan(big[G:G + n]).any()
    assert torch.isnan(big[:G]).all() and torch.isnan(big[G + n:]).all()
    _, ratt, _ = _oracle_mats(host.qkv.astype(np.float64), B, T, C, NH, True)
    assert np.max(np.abs(ops.download_f64(att) - ratt)) <= 1e-4
