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
