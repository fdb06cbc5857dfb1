"""The continuous-batching step driver on the GPU.

forge_batch_apply must leave the device block tables, context lengths and
slot mapping equal to the oracle's (oracle/serving.py) after every step,
bit for bit; and a whole serving loop -- requests arriving, prompts written
into their blocks on admission, one appended token and one decode per
running row per step, retirement and preemption -- must give decode outputs
within the parity tolerance of the CPU oracle run over the oracle's own
tables, with the caches bit-identical at the end.  Admitted prompts go
through forge_paged_prefill, checked against the oracle's prefill.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import serving as S
from gpu_util import DEV, TOL, bits_host
from paged_kv_gqa_06_gb300 import binding as B
from paged_kv_gqa_06_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


class Driver:
    """Library pool + batch, the oracle's twin, and the device index tensors."""

    def __init__(self, nb, bs, mbps, rows, budget):
        self.rows, self.mbps = rows, mbps
        self.pool = B.forge_kv_pool_create(nb, bs, mbps)
        self.batch = B.forge_batch_create(self.pool, rows, budget)
        self.ref_pool = S.BlockPool(nb, bs, mbps)
        self.ref = S.DecodeBatch(self.ref_pool, rows, budget)
        self.tables = torch.full((rows, mbps), -7, dtype=torch.int32, device=DEV)
        self.lens = torch.full((rows,), -7, dtype=torch.int32, device=DEV)
        self.slots = torch.full((rows,), -7, dtype=torch.int64, device=DEV)

    def submit(self, req):
        self.ref.submit(*req)
        B.forge_batch_submit(self.batch, *req)

    def step(self, apply=True, stream=None):
        want = self.ref.step()
        B.forge_batch_step(self.batch)
        if apply:
            B.forge_batch_apply(self.batch, self.tables, self.lens, self.slots, stream=stream)
        return want

    def host_tables(self):
        t = np.full((self.rows, self.mbps), -1, dtype=np.int32)
        for r in range(self.rows):
            row = self.ref.table(r)
            t[r, :len(row)] = row
        return t

    def check_device(self, want):
        torch.cuda.synchronize()
        assert self.lens.cpu().tolist() == want["context_lens"]
        assert self.slots.cpu().tolist() == want["slots"]
        dev = self.tables.cpu().numpy()
        admitted = {r for _, r, _ in want["admitted"]}
        for r in range(self.rows):
            row = self.ref.table(r)
            if not row:
                continue
            assert dev[r, :len(row)].tolist() == row, r
            if r in admitted:
                assert np.all(dev[r, len(row):] == -1), r

    def close(self):
        B.forge_batch_destroy(self.batch)
        used = B.forge_kv_pool_used_blocks(self.pool)
        B.forge_kv_pool_destroy(self.pool)
        return used


@pytest.mark.parametrize("nb,bs,rows,budget", [(4096, 16, 64, 8192), (40, 4, 6, 64), (300, 16, 16, 512)])
def test_apply_matches_the_oracle_tables(nb, bs, rows, budget):
    mbps = 64
    stream = W.request_stream(120, 21 + rows, prompt_median=100.0 if bs == 16 else 20.0,
                              prompt_max=min(mbps * bs - 64, nb * bs // 2), new_max=64 if bs == 16 else 40,
                              arrivals_per_step=1.5)
    d = Driver(nb, bs, mbps, rows, budget)
    retired, step, preempted = 0, 0, 0
    while retired < len(stream.seq_ids):
        for req in stream.arriving(step):
            d.submit(req)
        want = d.step()
        d.check_device(want)
        retired += len(want["retired"])
        preempted += len(want["preempted"])
        step += 1
    assert d.close() == 0
    if nb == 40:
        assert preempted > 0


def test_a_skipped_apply_is_repaired_by_the_next():
    d = Driver(64, 16, 16, 4, 1000)
    for i in range(4):
        d.submit((50 + i, 14 + 5 * i, 40))
    want = d.step()
    d.check_device(want)
    for _ in range(5):                 # tokens cross block boundaries while the device is not told
        d.step(apply=False)
    want = d.step()
    d.check_device(want)
    assert d.close() == 0


def _bf16(rng, shape):
    return W.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


@pytest.mark.parametrize("mode", ["fused", "separate", "graph"])
def test_serving_loop_matches_the_oracle(mode):
    Hq, Hkv, D, bs, nb, mbps, rows = 8, 2, 128, 16, 96, 32, 6
    scale = 1.0 / np.sqrt(D)
    rng = np.random.Generator(np.random.PCG64(77))
    stream = W.request_stream(30, 5, prompt_median=60.0, prompt_max=300, new_max=40, arrivals_per_step=0.5)
    d = Driver(nb, bs, mbps, rows, 256)
    nan = np.full((nb, Hkv, bs, D), W.BF16_NAN, dtype=np.uint16)
    kc_h, vc_h = nan.copy(), nan.copy()
    kc_d, vc_d = _dev(nan), _dev(nan)
    out = torch.zeros(rows, Hq, D, dtype=torch.float32, device=DEV)

    side = torch.cuda.Stream()
    if mode == "graph":   # the decode step captured once, over fixed buffers the loop refills
        q_s = torch.zeros(rows, Hq, D, dtype=torch.bfloat16, device=DEV)
        kn_s = torch.zeros(rows, Hkv, D, dtype=torch.bfloat16, device=DEV)
        vn_s = torch.zeros_like(kn_s)
        d.lens.zero_()
        d.tables.fill_(-1)

        def launch():
            B.forge_paged_append_gqa_decode(q_s, kn_s, vn_s, kc_d, vc_d, d.tables, d.lens, scale, out, stream=side)
        with torch.cuda.stream(side):
            launch()                   # sizes the split workspace on this stream before capture
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            launch()

    retired, step, errs, prefilled = 0, 0, [], 0
    while retired < len(stream.seq_ids):
        for req in stream.arriving(step):
            d.submit(req)
        with torch.cuda.stream(side):
            want = d.step(stream=side)
        host_tables = d.host_tables()
        # prefill of the admitted prompts: their K/V written into the blocks the
        # driver gave them, then one forge_paged_prefill over all of them
        pf = [(r, p) for _, r, p in want["admitted"] if p > 0]
        for r, p in pf:
            table = d.ref.table(r)
            slots = np.array([table[t // bs] * bs + t % bs for t in range(p)], dtype=np.int64)
            k, v = _bf16(rng, (p, Hkv, D)), _bf16(rng, (p, Hkv, D))
            oracle.paged_kv_append(k, v, slots, kc_h, vc_h)
            with torch.cuda.stream(side):
                B.forge_paged_kv_append(_dev(k), _dev(v), torch.from_numpy(slots).to(DEV), kc_d, vc_d, stream=side)
        if pf:
            pf_tables = np.ascontiguousarray(host_tables[[r for r, _ in pf]])
            pf_lens = np.array([p for _, p in pf], dtype=np.int32)
            pf_qs = np.concatenate([[0], np.cumsum(pf_lens)]).astype(np.int32)
            pq = _bf16(rng, (int(pf_qs[-1]), Hq, D))
            pf_ref = oracle.paged_prefill(pq, kc_h, vc_h, pf_tables, pf_lens, pf_qs, scale)
            pf_out = torch.empty(int(pf_qs[-1]), Hq, D, dtype=torch.float32, device=DEV)
            with torch.cuda.stream(side):
                B.forge_paged_prefill(_dev(pq), kc_d, vc_d, torch.from_numpy(pf_tables).to(DEV),
                                      torch.from_numpy(pf_lens).to(DEV), torch.from_numpy(pf_qs).to(DEV), scale,
                                      pf_out, stream=side)
            side.synchronize()
            prefilled += len(pf)
            errs.append(float(np.max(np.abs(pf_out.double().cpu().numpy() - pf_ref))))
        # this step's token of every running row, then the decode
        q, kn, vn = _bf16(rng, (rows, Hq, D)), _bf16(rng, (rows, Hkv, D)), _bf16(rng, (rows, Hkv, D))
        oracle.paged_kv_append(kn, vn, np.array(want["slots"], dtype=np.int64), kc_h, vc_h)
        ref = oracle.paged_gqa_decode(q, kc_h, vc_h, host_tables, np.array(want["context_lens"], np.int32), scale)
        with torch.cuda.stream(side):
            if mode == "fused":
                B.forge_paged_append_gqa_decode(_dev(q), _dev(kn), _dev(vn), kc_d, vc_d, d.tables, d.lens, scale,
                                                out, stream=side)
            elif mode == "separate":
                B.forge_paged_kv_append(_dev(kn), _dev(vn), d.slots, kc_d, vc_d, stream=side)
                B.forge_paged_gqa_decode(_dev(q), kc_d, vc_d, d.tables, d.lens, scale, out, stream=side)
            else:
                q_s.copy_(_dev(q))
                kn_s.copy_(_dev(kn))
                vn_s.copy_(_dev(vn))
                graph.replay()
        side.synchronize()
        got = out.double().cpu().numpy()
        assert np.all(np.isfinite(got)), step
        errs.append(float(np.max(np.abs(got - ref))))
        retired += len(want["retired"])
        step += 1

    assert prefilled > 0
    assert max(errs) <= TOL["f32"], max(errs)
    assert np.array_equal(bits_host(kc_d), kc_h) and np.array_equal(bits_host(vc_d), vc_h)
    assert B.forge_paged_get_device_error() == 0
    assert d.close() == 0


def test_applies_alternating_between_two_streams():
    """Applies of one batch go to two streams in turn, ordered by events but
    never synchronised with the host between checks, for many more steps than
    the staging ring has buffers: a buffer is refilled only once the apply
    kernel that last read it has ended, so the device state stays the
    oracle's."""
    d = Driver(300, 16, 16, 8, 512)
    reqs = W.request_stream(60, 33, prompt_median=100.0, prompt_max=200, new_max=30, arrivals_per_step=1.0)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    retired, step, prev, checks = 0, 0, None, 0
    while retired < len(reqs.seq_ids):
        for req in reqs.arriving(step):
            d.submit(req)
        s = streams[step % 2]
        if prev is not None:
            s.wait_event(prev)
        want = d.step(stream=s)
        prev = torch.cuda.Event()
        prev.record(s)
        retired += len(want["retired"])
        step += 1
        if step % 9 == 0:               # the 8 applies before this check ran without a host sync
            d.check_device(want)
            checks += 1
    d.check_device(want)
    assert checks >= 2
    assert d.close() == 0
