"""The forward's deal of causal work items over its CTAs (host logic, no GPU).

An item is two 128-row query tiles of one head; item i starts at query row
256*(P-1-i/(B*NH)) with P = ceil(T/256), and its two tiles see (causal) one
key tile per 128 rows up to their own. The deal must run every item exactly
once, longest first on each CTA, give every CTA work, and leave the busiest
CTA no busier than the snake order it replaced (rounds of G items, CTA c
taking c, 2G-1-c, ...)."""
import math

import pytest

api = pytest.importorskip("causal_head_attention_fwd_gb300.api")

BOUNDARY = 1.7   # the deal's start-up weight per item, in key-tile steps


def n_steps(i, B, T, NH):
    P = (T + 255) // 256
    q0 = 256 * (P - 1 - i // (B * NH))
    tiles = [q for q in (q0, q0 + 128) if q < T]
    return max(q // 128 + 1 for q in tiles)


def snake_max(B, T, NH, G):
    n = B * NH * ((T + 255) // 256)
    loads = [0.0] * G
    for k in range(math.ceil(n / G)):
        for c in range(G):
            i = k * G + (G - 1 - c if k & 1 else c)
            if i < n:
                loads[c] += n_steps(i, B, T, NH) + BOUNDARY
    return max(loads)


@pytest.mark.parametrize("B,T,C,NH,n_cta", [
    (16, 1024, 768, 12, 152),   # GPT-2 small training shape
    (8, 1024, 1600, 25, 152),   # GPT-2 XL heads
    (2, 8192, 768, 12, 152),    # long context
    (2, 1000, 768, 12, 152),    # ragged T, fewer items than CTAs
    (2, 333, 128, 2, 6),        # tiny, several items per CTA
    (1, 64, 128, 2, 152),       # one item per head
])
def test_deal_is_complete_and_balanced(B, T, C, NH, n_cta):
    got = api.attn_fwd_schedule(B, T, C, NH, n_cta)
    assert got is not None
    off, items = got
    n = B * NH * ((T + 255) // 256)
    G = min(n, n_cta)
    assert len(off) == G + 1 and off[0] == 0 and off[-1] == n
    assert sorted(items) == list(range(n))                       # each item exactly once
    loads = []
    for c in range(G):
        mine = items[off[c]:off[c + 1]]
        assert mine, f"CTA {c} has no work"
        steps = [n_steps(i, B, T, NH) for i in mine]
        assert steps == sorted(steps, reverse=True)              # longest first
        loads.append(sum(s + BOUNDARY for s in steps))
    assert max(loads) <= snake_max(B, T, NH, G) + 1e-9
    # greedy longest-first is within one item of the average load
    assert max(loads) <= sum(loads) / G + max(n_steps(i, B, T, NH) for i in range(n)) + BOUNDARY + 1e-9


def test_deal_beats_snake_on_the_training_shape():
    off, items = api.attn_fwd_schedule(16, 1024, 768, 12, 152)  # 152 SMs
    loads = [sum(n_steps(i, 16, 1024, 12) + BOUNDARY for i in items[off[c]:off[c + 1]]) for c in range(152)]
    assert max(loads) < snake_max(16, 1024, 12, 152) - 1.0     # 36.2 against 38.2


def test_no_table_beyond_the_parameter_space_and_bad_arguments():
    assert api.attn_fwd_schedule(64, 2048, 768, 12, 152) is None   # 6144 items: snake order
    with pytest.raises(api.AttnError):
        api.attn_fwd_schedule(2, 64, 100, 3, 152)                  # C % NH != 0
    with pytest.raises(api.AttnError):
        api.attn_fwd_schedule(2, 64, 128, 2, 0)
