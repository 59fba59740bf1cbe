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
