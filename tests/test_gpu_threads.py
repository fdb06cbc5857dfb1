"""The library used from several host threads at once, each on its own CUDA
stream (the C ABI is documented as thread-safe).

The library-owned split scratch is per (device, stream), and the per-device
state and scratch caches are shared under locks.  Each thread decodes its
own workload repeatedly on its own stream; every thread's result must equal
the single-threaded run's bit for bit (the split merge has a fixed order, so
one plan gives one result), and the single-threaded run must match the
oracle within the tolerance.
"""
import threading

import pytest
import torch

from gpu_util import TOL, DeviceLayer, assert_device_clean, max_abs_err, oracle_appended, oracle_decode, out_tensor
from paged_kv_gqa_06_gb300 import binding
from paged_kv_gqa_06_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


def test_threads_on_their_own_streams_match_the_single_threaded_run():
    names = ["qwen3_0_6b", "skewed", "tiny", "qwen3_0_6b", "skewed_bf16", "tiny"]
    jobs = []
    for name in names:
        wl = W.make_workload(name)
        t = wl.layer(0)
        d = DeviceLayer(wl, t)
        d.append()
        ref = out_tensor(wl)
        d.decode(ref)
        torch.cuda.synchronize()
        kc, vc = oracle_appended(wl, t)
        assert max_abs_err(ref, oracle_decode(wl, t, kc, vc)) <= TOL[wl.spec.out_dtype], name
        jobs.append((wl, d, ref))

    results = [None] * len(jobs)
    errors = []
    start = threading.Barrier(len(jobs))

    def work(i):
        try:
            wl, d, _ = jobs[i]
            stream = torch.cuda.Stream()
            out = out_tensor(wl)
            start.wait()
            for _ in range(25):
                binding.forge_paged_gqa_decode(d.q, d.k_cache, d.v_cache, d.tables, d.lens, wl.scale, out,
                                               stream=stream)
            stream.synchronize()
            results[i] = out
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for (wl, _, ref), out in zip(jobs, results):
        assert torch.equal(out, ref), wl.spec.name
    assert_device_clean()


def test_threads_sharing_one_stream_grow_its_scratch():
    """Four host threads decode on ONE stream, with problems whose split scratch
    grows from one to the next, so the stream's library-owned scratch is grown
    (stream-ordered: new buffer allocated, old one released after the work
    queued before it) while other threads' calls on the same stream are in
    flight.  Every result must equal the single-threaded run's bit for bit and
    match the oracle."""
    grow = W.custom_spec("grow", B=16, Hq=32, Hkv=8, D=128, fixed_lens=(2000,) * 16, out_dtype="bf16", seed=5)
    names = ["qwen3_0_6b", grow, "skewed", "qwen3_4b"]
    jobs = []
    for name in names:
        wl = W.make_workload(name)
        t = wl.layer(0)
        d = DeviceLayer(wl, t)
        d.append()
        ref = out_tensor(wl)
        d.decode(ref)
        torch.cuda.synchronize()
        kc, vc = oracle_appended(wl, t)
        assert max_abs_err(ref, oracle_decode(wl, t, kc, vc)) <= TOL[wl.spec.out_dtype], name
        need = binding.forge_paged_gqa_decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.D, wl.MB, 0)
        jobs.append((wl, d, ref, need))
    assert len({j[3] for j in jobs}) == len(jobs), "each problem should need a different scratch size"

    for order in (range(4), reversed(range(4))):
        shared = torch.cuda.Stream()        # a fresh stream: its scratch starts empty
        results = [None] * len(jobs)
        errors = []
        turn = threading.Semaphore(1)
        start = threading.Barrier(len(jobs))
        order = list(order)

        def work(i):
            try:
                wl, d, _, _ = jobs[i]
                out = out_tensor(wl)
                start.wait()
                for rep in range(20):
                    if rep == 0:            # first calls in the given order: the scratch grows in turn
                        while True:
                            with turn:
                                if order[0] == i:
                                    order.pop(0)
                                    break
                    binding.forge_paged_gqa_decode(d.q, d.k_cache, d.v_cache, d.tables, d.lens, wl.scale, out,
                                                   stream=shared)
                results[i] = out
            except Exception as e:  # reported below, on the main thread
                errors.append(e)
                with turn:
                    if i in order:
                        order.remove(i)

        threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
        for th in threads:
            th.start()
        for th in threads:
            th.join()
        shared.synchronize()
        assert not errors, errors
        for (wl, _, ref, _), out in zip(jobs, results):
            assert torch.equal(out, ref), wl.spec.name
    assert_device_clean()
