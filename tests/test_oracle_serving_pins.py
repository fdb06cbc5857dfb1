"""Pins of the serving oracle (oracle/serving.py): the KV block pool and the
continuous-batching decode step.

Two kinds of evidence, neither of which reuses the oracle's code:
  * traces worked out by hand from the stated policy
    (tests/golden/serving_trace.json);
  * invariants checked by brute force on every step of seeded random request
    streams, including pools small enough to force preemption: every block
    is free or owned by exactly one sequence, a sequence of n tokens owns
    ceil(n / block_size) blocks, each slot is the table entry of position
    len-1 times block_size plus the offset, first admissions follow arrival
    order, a preempted sequence is the next one admitted, the per-step prompt
    budget holds, a sequence leaves with
    prompt + max_new tokens after exactly max_new decode steps in a row, and
    the pool is empty once every request has finished (forge-engine README,
    "What it implements": deterministic cleanup, zero blocks at the end).
"""
import json
import os

import pytest

from oracle import serving as S
from paged_kv_gqa_06_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "serving_trace.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_pool_case_by_hand():
    c = _golden()["pool_case"]
    pool = S.BlockPool(c["num_blocks"], c["block_size"], c["max_blocks_per_seq"])
    slots = []
    for op, seq, *arg in c["ops"]:
        if op == "add":
            pool.add(seq, arg[0])
        elif op == "release":
            pool.release(seq)
        else:
            slots.append(pool.grow(seq)[0])
    assert slots == c["grow_slots"]
    assert {str(k): v for k, v in pool.tables.items()} == c["tables"]
    assert len(pool.free) == c["free_after"]


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["name"])
def test_trace_by_hand(case):
    pool = S.BlockPool(case["num_blocks"], case["block_size"], case["max_blocks_per_seq"])
    batch = S.DecodeBatch(pool, case["rows"], case["token_budget"])
    for req in case["requests"]:
        batch.submit(*req)
    for i, want in enumerate(case["steps"]):
        got = batch.step()
        for key in ("seq_ids", "context_lens", "slots", "new_blocks"):
            assert got[key] == want[key], (i, key)
        for key in ("admitted", "retired", "preempted"):
            assert [list(e) for e in got[key]] == want[key], (i, key)
        assert got["report"]["free_blocks"] == want["free_blocks"], i
        assert got["report"]["waiting"] == want["waiting"], i
    assert pool.used() == 0


def drive(stream, pool, batch, max_steps=100000):
    """Submit each request before its arrival step and step until all are done."""
    trace, step = [], 0
    n = len(stream.seq_ids)
    while True:
        for req in stream.arriving(step):
            batch.submit(*req)
        rec = batch.step()
        trace.append(rec)
        step += 1
        done = sum(len(r["retired"]) for r in trace)
        if done == n and rec["report"]["running"] == 0:
            return trace
        assert step < max_steps, "stream did not drain"


# (pool blocks, block size, rows, budget, prompt median, decode max): the last
# two are small enough to preempt often
PRESSURES = [(4096, 16, 8, 4096, 200.0, 64), (200, 16, 8, 512, 150.0, 64), (40, 4, 6, 64, 20.0, 40),
             (12, 4, 4, 16, 6.0, 20)]


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("nb,bs,rows,budget,median,new_max", PRESSURES)
def test_invariants_on_random_streams(seed, nb, bs, rows, budget, median, new_max):
    mbps = 64
    stream = W.request_stream(60, seed, prompt_median=median, prompt_max=min(mbps * bs - new_max, nb * bs // 2),
                              new_max=new_max, arrivals_per_step=0.7)
    pool = S.BlockPool(nb, bs, mbps)
    batch = S.DecodeBatch(pool, rows, budget)
    prompt_of = {int(s): int(p) for s, p in zip(stream.seq_ids, stream.prompts)}
    new_of = {int(s): int(m) for s, m in zip(stream.seq_ids, stream.max_new)}
    arrival_order = [int(s) for s in stream.seq_ids]

    first_admission, steps_in_row, preempted_any = [], {}, False
    queue_front = []   # preempted sequences, in the order they must come back
    order_of, counter = {}, 0
    trace, step = [], 0
    while True:
        for req in stream.arriving(step):
            batch.submit(*req)
        running_before = {s: order_of[s] for s in batch.seq if s >= 0}
        rec = batch.step()
        trace.append(rec)
        step += 1

        # ownership: every block exactly once among the free stack and the tables
        owned = [b for t in pool.tables.values() for b in t]
        assert sorted(owned + pool.free) == list(range(nb))
        # rows, lengths, tables and slots
        for r in range(rows):
            s, L = rec["seq_ids"][r], rec["context_lens"][r]
            if s < 0:
                assert L == 0 and rec["slots"][r] == -1 and rec["new_blocks"][r] == -1
                continue
            t = pool.tables[s]
            assert len(t) == -(-L // bs) and pool.lens[s] == L
            assert rec["slots"][r] == t[(L - 1) // bs] * bs + (L - 1) % bs
            assert rec["new_blocks"][r] == (t[-1] if (L - 1) % bs == 0 else -1)
            steps_in_row[s] = steps_in_row.get(s, 0) + 1
        assert len(set(s for s in rec["seq_ids"] if s >= 0)) == rec["report"]["running"]
        # admissions: budget, first-come order, lowest free rows
        prompts = [p for _, _, p in rec["admitted"]]
        assert len(prompts) <= 1 or sum(prompts) <= budget
        for s, r, p in rec["admitted"]:
            if queue_front:     # a preempted sequence comes back before anyone else
                assert s == queue_front.pop(0)
            counter += 1
            order_of[s] = counter
            if s not in first_admission:
                first_admission.append(s)
                assert p == prompt_of[s]
        # preemption takes the latest admitted of the rows running before the step
        for s, _, L in rec["preempted"]:
            preempted_any = True
            assert order_of[s] == max(o for q, o in running_before.items()
                                      if q not in [x for x, _, _ in rec["retired"]])
            running_before.pop(s)
            queue_front.insert(0, s)
        # a sequence retires with prompt + max_new tokens after max_new decode steps
        for s, _, L in rec["retired"]:
            assert L == prompt_of[s] + new_of[s]
            assert steps_in_row[s] == new_of[s]

        done = sum(len(x["retired"]) for x in trace)
        if done == len(arrival_order) and rec["report"]["running"] == 0:
            break
        assert step < 100000

    assert first_admission == arrival_order
    assert pool.used() == 0 and sorted(pool.free) == list(range(nb)) and not pool.tables
    if nb <= 40:
        assert preempted_any, "the small pools are meant to preempt"


def test_same_calls_give_the_same_trace():
    stream = W.request_stream(40, 9, prompt_median=30.0, prompt_max=60, new_max=30)
    traces = []
    for _ in range(2):
        pool = S.BlockPool(30, 4, 64)
        traces.append(drive(stream, pool, S.DecodeBatch(pool, 4, 64)))
    assert traces[0] == traces[1]


def test_submit_rejects_what_can_never_run():
    pool = S.BlockPool(4, 16, 2)
    batch = S.DecodeBatch(pool, 2, 100)
    with pytest.raises(ValueError):
        batch.submit(1, 30, 3)          # 33 tokens > 2 blocks of 16
    with pytest.raises(ValueError):
        batch.submit(1, 3, 0)           # no decode step
    batch.submit(1, 3, 1)
    with pytest.raises(ValueError):
        batch.submit(1, 3, 1)           # id already live
    big = S.DecodeBatch(S.BlockPool(1, 16, 4), 2, 100)
    with pytest.raises(MemoryError):
        big.submit(2, 16, 1)            # 17 tokens need 2 blocks; the pool has 1
