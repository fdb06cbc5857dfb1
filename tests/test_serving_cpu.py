"""The KV block pool and the continuous-batching step driver of
libforge_paged.so (include/forge_serving.h) on the host: no GPU needed,
since everything but forge_batch_apply makes no CUDA call.

The library's per-step row state (sequence, context length, slot, opened
block), its events (admitted, retired, preempted) and its report must equal
the oracle's (oracle/serving.py) exactly, on the hand-worked traces and on
seeded random request streams, including pools small enough to preempt.
"""
import ctypes
import json
import os

import numpy as np
import pytest
import torch

from oracle import serving as S
from paged_kv_gqa_06_gb300 import binding as B
from paged_kv_gqa_06_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "serving_trace.json")
EVENT_KINDS = {"admitted": B.FORGE_BATCH_ADMITTED, "retired": B.FORGE_BATCH_RETIRED,
               "preempted": B.FORGE_BATCH_PREEMPTED}


@pytest.fixture(scope="module", autouse=True)
def lib():
    from paged_kv_gqa_06_gb300 import build
    build.build()
    return B.load_library()


class Lib:
    """The library's pool + batch, stepped like the oracle's."""

    def __init__(self, nb, bs, mbps, rows, budget):
        self.rows = rows
        self.pool = B.forge_kv_pool_create(nb, bs, mbps)
        self.batch = B.forge_batch_create(self.pool, rows, budget)

    def submit(self, *req):
        B.forge_batch_submit(self.batch, *req)

    def step(self):
        rep = B.forge_batch_step(self.batch)
        rows = B.forge_batch_rows(self.batch, self.rows)
        rec = {k: v.tolist() for k, v in rows.items()}
        for name, kind in EVENT_KINDS.items():
            rec[name] = B.forge_batch_events(self.batch, kind)
        rec["report"] = rep
        return rec

    def close(self):
        B.forge_batch_destroy(self.batch)
        used = B.forge_kv_pool_used_blocks(self.pool)
        B.forge_kv_pool_destroy(self.pool)
        return used


def test_pool_case_by_hand():
    c = json.load(open(GOLDEN))["pool_case"]
    pool = B.forge_kv_pool_create(c["num_blocks"], c["block_size"], c["max_blocks_per_seq"])
    slots = []
    for op, seq, *arg in c["ops"]:
        if op == "add":
            B.forge_kv_pool_add(pool, seq, arg[0])
        elif op == "release":
            B.forge_kv_pool_release(pool, seq)
        else:
            slots.append(B.forge_kv_pool_grow(pool, seq))
    assert slots == c["grow_slots"]
    for seq, blocks in c["tables"].items():
        assert B.forge_kv_pool_sequence(pool, int(seq))[1] == blocks
    assert B.forge_kv_pool_free_blocks(pool) == c["free_after"]
    B.forge_kv_pool_destroy(pool)


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_trace_by_hand(case):
    lib = Lib(case["num_blocks"], case["block_size"], case["max_blocks_per_seq"], case["rows"],
              case["token_budget"])
    for req in case["requests"]:
        lib.submit(*req)
    for i, want in enumerate(case["steps"]):
        got = lib.step()
        for key in ("seq_ids", "context_lens", "slots", "new_blocks"):
            assert got[key] == want[key], (i, key)
        for key in EVENT_KINDS:
            assert [list(e) for e in got[key]] == want[key], (i, key)
        assert got["report"]["free_blocks"] == want["free_blocks"]
        assert got["report"]["waiting"] == want["waiting"]
    assert lib.close() == 0


PRESSURES = [(4096, 16, 32, 4096, 300.0, 128), (300, 16, 16, 1024, 150.0, 64), (40, 4, 6, 64, 20.0, 40),
             (12, 4, 4, 16, 6.0, 20)]


@pytest.mark.parametrize("seed", [11, 12])
@pytest.mark.parametrize("nb,bs,rows,budget,median,new_max", PRESSURES)
def test_matches_the_oracle_step_by_step(seed, nb, bs, rows, budget, median, new_max):
    mbps = 64
    stream = W.request_stream(80, seed, prompt_median=median, prompt_max=min(mbps * bs - new_max, nb * bs // 2),
                              new_max=new_max, arrivals_per_step=0.8)
    pool = S.BlockPool(nb, bs, mbps)
    ref = S.DecodeBatch(pool, rows, budget)
    lib = Lib(nb, bs, mbps, rows, budget)
    retired, step, preempted = 0, 0, 0
    while retired < len(stream.seq_ids):
        for req in stream.arriving(step):
            ref.submit(*req)
            lib.submit(*req)
        want, got = ref.step(), lib.step()
        step += 1
        for key in ("seq_ids", "context_lens", "slots", "new_blocks"):
            assert got[key] == want[key], (step, key)
        for key in EVENT_KINDS:
            assert got[key] == want[key], (step, key)
        assert got["report"] == want["report"], step
        for r in range(rows):
            s = want["seq_ids"][r]
            if s >= 0:
                assert B.forge_kv_pool_sequence(lib.pool, s) == (pool.lens[s], pool.tables[s])
        retired += len(want["retired"])
        preempted += len(want["preempted"])
        assert step < 100000
    assert lib.close() == 0 and pool.used() == 0
    if nb <= 40:
        assert preempted > 0


def test_submit_and_pool_errors():
    pool = B.forge_kv_pool_create(4, 16, 2)
    batch = B.forge_batch_create(pool, 2, 100)
    with pytest.raises(B.ForgeError) as e:
        B.forge_batch_submit(batch, 1, 30, 3)        # 33 tokens > 2 blocks of 16
    assert e.value.status == -8
    with pytest.raises(B.ForgeError):
        B.forge_batch_submit(batch, 1, 3, 0)         # no decode step
    with pytest.raises(B.ForgeError):
        B.forge_batch_submit(batch, 1, -1, 1)        # negative prompt
    B.forge_batch_submit(batch, 1, 3, 1)
    with pytest.raises(B.ForgeError):
        B.forge_batch_submit(batch, 1, 3, 1)         # id already live
    B.forge_batch_destroy(batch)
    B.forge_kv_pool_destroy(pool)

    small = B.forge_kv_pool_create(1, 16, 4)
    batch = B.forge_batch_create(small, 2, 100)
    with pytest.raises(B.ForgeError) as e:
        B.forge_batch_submit(batch, 2, 16, 1)        # 17 tokens need 2 blocks; the pool has 1
    assert e.value.status == -9
    B.forge_batch_destroy(batch)

    B.forge_kv_pool_add(small, 5, 16)
    with pytest.raises(B.ForgeError) as e:
        B.forge_kv_pool_add(small, 6, 1)             # no block left
    assert e.value.status == -9
    with pytest.raises(B.ForgeError) as e:
        B.forge_kv_pool_grow(small, 5)               # token 16 needs a second block
    assert e.value.status == -9
    assert B.forge_kv_pool_sequence(small, 5) == (16, [0])   # nothing changed
    with pytest.raises(B.ForgeError):
        B.forge_kv_pool_add(small, 5, 1)             # id already present
    with pytest.raises(B.ForgeError):
        B.forge_kv_pool_release(small, 77)           # unknown id
    B.forge_kv_pool_release(small, 5)
    assert B.forge_kv_pool_used_blocks(small) == 0
    B.forge_kv_pool_destroy(small)

    with pytest.raises(ValueError):
        B.forge_kv_pool_create(4, 0, 2)
    assert B.load_library().forge_batch_step(None, None) == -1
    assert B.load_library().forge_kv_pool_used_blocks(None) == -1


def test_destroying_a_batch_returns_its_blocks():
    lib = Lib(64, 16, 8, 4, 1000)
    for i in range(6):
        lib.submit(100 + i, 20 + i, 50)
    for _ in range(3):
        lib.step()
    assert B.forge_kv_pool_used_blocks(lib.pool) > 0
    assert lib.close() == 0


def test_apply_validates_before_touching_cuda():
    lib = Lib(64, 16, 8, 4, 1000)
    lib.submit(1, 5, 2)
    lib.step()
    tables = torch.zeros(4, 8, dtype=torch.int32)
    lens = torch.zeros(4, dtype=torch.int32)
    slots = torch.zeros(4, dtype=torch.int64)
    bad = [
        (tables.to(torch.int64), lens, slots, -2),
        (tables, lens.to(torch.int64), slots, -2),
        (tables, lens, slots.to(torch.int32), -2),
        (torch.zeros(4, 7, dtype=torch.int32), lens, slots, -3),        # narrower than a table row
        (torch.zeros(3, 8, dtype=torch.int32), lens, slots, -3),        # wrong batch width
        (tables.t().contiguous().t(), lens, slots, -3),                 # inner stride not 1
        (tables, torch.zeros(8, dtype=torch.int32)[::2], slots, -3),    # strided lengths
    ]
    def desc(t):  # a descriptor of a host tensor, straight to the C ABI (the binding refuses host tensors)
        d = B.ForgeTensor()
        d.data, d.dtype, d.ndim = t.data_ptr(), B._DTYPES[t.dtype], t.dim()
        for i in range(t.dim()):
            d.shape[i], d.stride[i] = t.shape[i], t.stride(i)
        return d

    for t, l, s, status in bad:
        dt, dl, ds = desc(t), desc(l), desc(s)
        rc = B.load_library().forge_batch_apply(lib.batch, ctypes.byref(dt), ctypes.byref(dl), ctypes.byref(ds),
                                                None)
        assert rc == status
    with pytest.raises(ValueError, match="CUDA device memory"):
        B.forge_batch_apply(lib.batch, tables, lens, slots, stream=0)
    assert lib.close() == 0


def _drive(seed, nb=300, bs=16, rows=16, budget=1024):
    """Every step's record of one pool + batch driven by a seeded request stream."""
    stream = W.request_stream(60, seed, prompt_median=150.0, prompt_max=min(64 * bs - 64, nb * bs // 2),
                              new_max=64, arrivals_per_step=0.8)
    lib = Lib(nb, bs, 64, rows, budget)
    records, retired, step = [], 0, 0
    while retired < len(stream.seq_ids):
        for req in stream.arriving(step):
            lib.submit(*req)
        rec = lib.step()
        records.append(rec)
        retired += len(rec["retired"])
        step += 1
        assert step < 100000
    assert lib.close() == 0
    return records


def test_batches_driven_from_threads_match_the_single_threaded_run():
    # separate pools and batches from separate host threads at once (the
    # header says every function is thread-safe): no state is shared
    import threading
    seeds = [31, 32, 33, 34]
    want = [_drive(s) for s in seeds]
    got, errors = [None] * len(seeds), []

    def work(i):
        try:
            got[i] = _drive(seeds[i])
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(seeds))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert got == want
