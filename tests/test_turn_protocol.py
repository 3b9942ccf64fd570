"""The forward kernels' turns at the exponentials, modelled on the CPU.

In attn_fwd_kernel (and the FP8 forward without a mask) the two softmax
warpgroups hand the exponentials to each other through two named barriers
(ids 3 and 4, 256 threads each): the warpgroup whose turn it is waits with
bar.sync, the other signals with bar.arrive. A named barrier has no time
limit, so the hand-overs must pair up on every path, including the ones where
a bounded mbarrier wait gives up. The kernels keep them paired by construction:

  * tile 1 takes the first turn (tile 0 arrives on barrier 4 once at the
    start; tile 1 takes one extra bar.sync on 4 at the end);
  * every warp takes exactly one turn per key step of every item: a warp whose
    tile has no such step, or whose wait gave up before its turn, takes the
    missing turns with no work before the item's epilogue;
  * a warpgroup that fails at an item's epilogue leaves the item loop and takes
    the turns of the items it did not walk.

This test replays each of the eight softmax warps' barrier operations for
random item lists and failure points and runs them against a model of named
barriers (a barrier completes when 256 threads have arrived; bar.sync blocks
until then). Every replay must run to the end with no barrier left half full.
"""
import random

import pytest

WARPS_PER_WG = 4
THREADS_PER_BAR = 256


def warp_ops(wg, items, fail, wg_fail_item):
    """Barrier operations of one softmax warp of warpgroup `wg`.

    items: list of (n_tile0, n_tile1, n_max) per work item.
    fail: None or (item, step, where): this warp's wait gives up at that key
          step, before its turn ('S') or inside it ('PV', the P.V wait).
    wg_fail_item: the item at whose epilogue the warpgroup leaves (a failure
          of any of its warps is combined there), or None.
    """
    my, other = 3 + wg, 4 - wg
    ops = []
    if wg == 0:
        ops.append(("arrive", 4))                 # tile 1 takes the first turn
    ic = 0
    ok = True
    while ok and ic < len(items):
        n, n_max = items[ic][wg], items[ic][2]
        turns = 0
        for j in range(n):
            if fail and fail[:2] == (ic, j) and fail[2] == "S":
                break                             # gave up before its turn
            ops.append(("sync", my))
            gave_up = bool(fail and fail[:2] == (ic, j) and fail[2] == "PV" and j > 0)
            ops.append(("arrive", other))
            turns += 1
            if gave_up:
                break
        ops += [("sync", my), ("arrive", other)] * (n_max - turns)
        if n > 0 and wg_fail_item == ic:
            ok = False                            # the epilogue's combined decision
            break
        ic += 1
    if not ok:
        for k in range(ic + 1, len(items)):
            ops += [("sync", my), ("arrive", other)] * items[k][2]
    if wg == 1:
        ops.append(("sync", 4))                   # the other warpgroup's last hand-over
    return ops


def run_barriers(seqs):
    """Replay the warps' operations against named barriers 3 and 4."""
    pos = [0] * len(seqs)
    count = {3: 0, 4: 0}
    waiting = {3: [], 4: []}
    progress = True
    while progress:
        progress = False
        for w, ops in enumerate(seqs):
            if pos[w] >= len(ops) or w in waiting[3] or w in waiting[4]:
                continue
            op, bar = ops[pos[w]]
            count[bar] += 32
            if op == "sync":
                waiting[bar].append(w)
            else:
                pos[w] += 1
            progress = True
            if count[bar] == THREADS_PER_BAR:
                count[bar] = 0
                for x in waiting[bar]:
                    pos[x] += 1
                waiting[bar] = []
            elif count[bar] > THREADS_PER_BAR:
                return "more than 256 threads at one barrier"
    if any(pos[w] < len(ops) for w, ops in enumerate(seqs)):
        return "deadlock"
    if count[3] or count[4]:
        return f"barrier left with {count}"
    return "ok"


def random_items(rng):
    items = []
    for _ in range(rng.randint(1, 6)):
        if rng.random() < 0.7:                    # causal pair: tile 1 one key step longer
            n0 = rng.randint(1, 8)
            n1 = n0 + 1 if rng.random() < 0.8 else 0     # 0: tile 1 past T
        else:                                     # no mask: equal steps
            n0 = n1 = rng.randint(1, 8)
        items.append((n0, n1, max(n0, n1)))
    return items


def random_failures(rng, items):
    """Per warp: None or a failure point; per warpgroup: the item it leaves at."""
    fails = [None] * (2 * WARPS_PER_WG)
    wg_fail = {0: None, 1: None}
    if rng.random() < 0.5:
        for w in range(2 * WARPS_PER_WG):
            if rng.random() < 0.3:
                wg = w // WARPS_PER_WG
                points = [(ic, j) for ic, it in enumerate(items) for j in range(it[wg])]
                if points:
                    ic, j = rng.choice(points)
                    where = rng.choice(["S", "PV"])
                    if where == "PV" and j == 0:
                        continue                  # no P.V wait at an item's first step
                    fails[w] = (ic, j, where)
                    if wg_fail[wg] is None or ic < wg_fail[wg]:
                        wg_fail[wg] = ic
    # a warp's failure after its warpgroup already left changes nothing
    for w in range(2 * WARPS_PER_WG):
        wg = w // WARPS_PER_WG
        if fails[w] and fails[w][0] > wg_fail[wg]:
            fails[w] = None
    return fails, wg_fail


def test_turns_pair_up_without_failures():
    rng = random.Random(7)
    for _ in range(2000):
        items = random_items(rng)
        seqs = [warp_ops(w // WARPS_PER_WG, items, None, None) for w in range(2 * WARPS_PER_WG)]
        assert run_barriers(seqs) == "ok", items


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_turns_pair_up_when_waits_give_up(seed):
    rng = random.Random(seed)
    for _ in range(5000):
        items = random_items(rng)
        fails, wg_fail = random_failures(rng, items)
        seqs = [warp_ops(w // WARPS_PER_WG, items, fails[w], wg_fail[w // WARPS_PER_WG])
                for w in range(2 * WARPS_PER_WG)]
        assert run_barriers(seqs) == "ok", (items, fails, wg_fail)


def test_a_missing_idle_turn_is_caught():
    """The model is not vacuous: dropping the idle turns of a shorter tile deadlocks."""
    items = [(2, 3, 3)]
    full = [warp_ops(w // WARPS_PER_WG, items, None, None) for w in range(2 * WARPS_PER_WG)]
    assert run_barriers(full) == "ok"
    # tile 0: the first arrive and its two real turns, without the idle third turn
    short = [ops[:-2] if w < WARPS_PER_WG else ops for w, ops in enumerate(full)]
    assert full[0][-2:] == [("sync", 3), ("arrive", 4)]
    assert run_barriers(short) != "ok"
