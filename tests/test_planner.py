"""Pins for the oracle's bucket planner and readiness rule.

Hand-counted plans (tests/golden/plan_small.txt), bucket counts for the
BERT-large parameter list worked out separately in the design analysis
(148/98/22/6/2 buckets at 1/4/25/100/500 MiB), and invariants of the rule
checked on random tensor lists.
"""
import random

import pytest

import oracle
from gradient_reduce_optimizer_gb300 import workloads as wl
from plan_fixtures import load_cases

CASES = load_cases()


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_hand_counted_plans(case):
    offsets, buckets, n_padded = oracle.plan_buckets(case["numel"],
                                                     case["bucket_bytes"])
    assert offsets == case["offsets"]
    assert buckets == case["buckets"]
    assert n_padded == case["n_padded"]
    ready = oracle.bucket_ready_layers(case["numel"], case["layer"], offsets,
                                       buckets)
    assert ready == case["ready"]


def check_invariants(numel, layer_of, cap):
    offsets, buckets, n_padded = oracle.plan_buckets(numel, cap)
    T = len(numel)
    span = [(k + 7) // 8 * 8 for k in numel]
    # reverse layer order, contiguous, 8-element aligned
    assert offsets[T - 1] == 0
    for t in range(T - 1):
        assert offsets[t] == offsets[t + 1] + span[t + 1]
    assert all(o % 8 == 0 for o in offsets)
    assert n_padded == sum(span)
    # buckets tile [0, n_padded) in order, on tensor boundaries
    starts = {offsets[t] for t in range(T)} | {n_padded}
    pos = 0
    for b, e in buckets:
        assert b == pos and e > b and b in starts and e in starts
        pos = e
    assert pos == n_padded
    # the greedy closing rule
    for i, (b, e) in enumerate(buckets):
        inside = [t for t in range(T) if b <= offsets[t] < e and span[t] > 0]
        nbytes = 2 * (e - b)
        last = max(inside, key=lambda t: offsets[t])
        if cap > 0 and i < len(buckets) - 1:
            assert nbytes >= cap
        if cap > 0:
            assert nbytes - 2 * span[last] < cap   # closed at the first chance
    # readiness: buckets launch in reverse layer order
    ready = oracle.bucket_ready_layers(numel, layer_of, offsets, buckets)
    assert ready == sorted(ready, reverse=True)
    return buckets


@pytest.mark.parametrize("seed", range(30))
def test_invariants_random_lists(seed):
    rnd = random.Random(seed)
    T = rnd.randint(1, 60)
    numel = [rnd.choice([0, 1, 2, 7, 8, 9, 100, 1000, 4096, 65537])
             for _ in range(T)]
    if sum(numel) == 0:
        numel[0] = 3
    layer_of = sorted(rnd.randint(0, 9) for _ in range(T))
    cap = rnd.choice([0, 1, 2, 16, 100, 2048, 10 ** 6])
    check_invariants(numel, layer_of, cap)


@pytest.mark.parametrize("mib,count", [(1, 148), (4, 98), (25, 22), (100, 6),
                                       (500, 2)])
def test_bert_large_bucket_counts(mib, count):
    t = wl.bert_large_tensors()
    numel = [x[1] for x in t]
    layer_of = [x[2] for x in t]
    assert len(t) == 398 and sum(numel) == 336_226_108
    buckets = check_invariants(numel, layer_of, mib * wl.MiB)
    assert len(buckets) == count
    _, _, n_padded = oracle.plan_buckets(numel, mib * wl.MiB)
    assert n_padded == 336_226_120   # 30522 -> 30528 and 2 -> 8


def test_bert_large_25mib_last_bucket_holds_word_embedding():
    """The 62.5 MB word embedding is never split, so the final bucket (the
    first layer's) is far above the 25 MiB cap."""
    t = wl.bert_large_tensors()
    numel = [x[1] for x in t]
    offsets, buckets, _ = oracle.plan_buckets(numel, 25 * wl.MiB)
    b, e = buckets[-1]
    assert b <= offsets[0] < e
    assert e - b >= 30522 * 1024 and 2 * (e - b) > 2 * 25 * wl.MiB


def test_gpt2_slice_sizes():
    t = wl.gpt2_slice_tensors()
    assert len(t) == 288 and sum(x[1] for x in t) == 2_718_867_456


# ---------------------------------------------------------------------------
# The shard plan of the sharded (multi-GPU) form
# ---------------------------------------------------------------------------

# Worked by hand: a bucket of u whole 8-element units gives rank q units
# floor(u q / W) .. floor(u (q + 1) / W) - 1; the last rank also takes a
# ragged tail; each rank's state holds its shards back to back.
SHARD_CASES = [
    # 5 units over 2 ranks: 2 and 3 units
    ([(0, 40)], 2, [[(0, 16), (16, 40)]], [[0, 0]], [16, 24]),
    # 5 units over 3 ranks: 1, 2, 2 units
    ([(0, 40)], 3, [[(0, 8), (8, 24), (24, 40)]], [[0, 0, 0]], [8, 16, 16]),
    # a one-unit bucket leaves rank 0 empty; a ragged last bucket:
    # 119 units + 3 elements over 2 ranks: 59 units, then 60 units + 3
    ([(0, 40), (40, 48), (48, 1003)], 2,
     [[(0, 16), (16, 40)], [(40, 40), (40, 48)], [(48, 520), (520, 1003)]],
     [[0, 0], [16, 24], [16, 32]], [488, 515]),
    # one unit over three ranks: only the last rank holds anything
    ([(0, 8)], 3, [[(0, 0), (0, 0), (0, 8)]], [[0, 0, 0]], [0, 0, 8]),
    # only a tail (5 elements) over two ranks
    ([(0, 5)], 2, [[(0, 0), (0, 5)]], [[0, 0]], [0, 5]),
]


@pytest.mark.parametrize("buckets,world,shards,offsets,elems", SHARD_CASES)
def test_shard_plan_hand_worked(buckets, world, shards, offsets, elems):
    assert oracle.shard_plan(buckets, world) == (shards, offsets, elems)


def check_shard_invariants(buckets, world):
    shards, offsets, elems = oracle.shard_plan(buckets, world)
    used = [0] * world
    for (b, e), row, offs in zip(buckets, shards, offsets):
        # the shards tile the bucket in rank order, each 16-byte aligned
        assert row[0][0] == b and row[-1][1] == e
        for (lo, hi), (lo2, _) in zip(row, row[1:]):
            assert hi == lo2
        assert all(lo % 8 == 0 and hi >= lo for lo, hi in row)
        whole = [(hi - lo) // 8 for lo, hi in row]
        assert max(whole) - min(whole) <= 1          # balanced to one unit
        for q, (lo, hi) in enumerate(row):
            assert offs[q] == used[q]
            used[q] += hi - lo
    assert elems == used
    assert sum(elems) == sum(e - b for b, e in buckets)
    if world == 1:
        assert shards == [[bk] for bk in buckets]


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("mib", [1, 25, 500])
def test_shard_plan_invariants_bert_large(world, mib):
    w = wl.bert_large_r8()
    _, buckets, _ = oracle.plan_buckets(w.numel(), mib << 20)
    check_shard_invariants(buckets, world)


def test_shard_plan_invariants_random():
    rng = random.Random(13)
    for _ in range(40):
        numel = [rng.choice([1, 7, 8, 9, 64, 1000, 4099]) for _ in range(rng.randint(1, 12))]
        _, buckets, _ = oracle.plan_buckets(numel, rng.choice([0, 16, 64, 4096]))
        check_shard_invariants(buckets, rng.randint(1, 9))
