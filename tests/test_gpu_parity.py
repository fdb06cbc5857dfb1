"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Append must be bit-exact over the entire caches; decode within max-abs
2e-3 (fp32 out) or 1.6e-2 (bf16 out) of the oracle on the same seeded inputs.
Every cache slot that holds no token is NaN, so reading one shows up as NaN.
"""
import gc

import numpy as np
import pytest
import torch

from gpu_util import (DEV, TOL, DeviceLayer, assert_device_clean, bits_host, max_abs_err, oracle_appended,
                      oracle_decode, out_tensor)
from paged_kv_gqa_06_gb300 import binding
from paged_kv_gqa_06_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("decode_kernel")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


_cache = {}


def _config(name):
    """(workload, host layer, oracle caches after append), cached per module."""
    if name not in _cache:
        wl = W.make_workload(name)
        t = wl.layer(0)
        _cache[name] = (wl, t, oracle_appended(wl, t))
    return _cache[name]


@pytest.mark.parametrize("name", ["tiny", "qwen3_0_6b", "qwen3_4b", "skewed"])
def test_append_bit_exact(name):
    wl, t, (kc_ref, vc_ref) = _config(name)
    d = DeviceLayer(wl, t)
    d.append()
    assert np.array_equal(bits_host(d.k_cache), kc_ref)
    assert np.array_equal(bits_host(d.v_cache), vc_ref)
    assert_device_clean()


@pytest.mark.parametrize("name,out_dtype", [("tiny", "f32"), ("tiny", "bf16"), ("qwen3_0_6b", "bf16"),
                                            ("qwen3_0_6b", "f32"), ("qwen3_4b", "bf16"), ("qwen3_4b", "f32"),
                                            ("skewed", "f32"), ("skewed", "bf16")])
def test_append_then_decode_matches_oracle(name, out_dtype):
    wl, t, (kc_ref, vc_ref) = _config(name)
    d = DeviceLayer(wl, t)
    d.append()
    out = out_tensor(wl, out_dtype)
    d.decode(out)
    ref = oracle_decode(wl, t, kc_ref, vc_ref)
    err = max_abs_err(out, ref)
    assert err <= TOL[out_dtype], f"{name}/{out_dtype}: max-abs error {err}"
    assert_device_clean()


@pytest.mark.parametrize("split_tokens", [16, 48, 128, 512, 1024])
def test_split_length_does_not_change_result(split_tokens):
    wl, t, (kc_ref, vc_ref) = _config("skewed")
    d = DeviceLayer(wl, t)
    d.append()
    out = out_tensor(wl, "f32")
    d.decode(out, split_tokens=split_tokens)
    err = max_abs_err(out, oracle_decode(wl, t, kc_ref, vc_ref))
    assert err <= TOL["f32"], f"split {split_tokens}: {err}"
    assert_device_clean()


def test_block_placement_gives_identical_bits():
    wl, t, _ = _config("qwen3_0_6b")
    d = DeviceLayer(wl, t)
    d.append()
    a = out_tensor(wl, "f32")
    d.decode(a, split_tokens=256)
    perm = torch.from_numpy(np.random.default_rng(11).permutation(wl.NB)).to(DEV)
    kc2 = torch.empty_like(d.k_cache)
    vc2 = torch.empty_like(d.v_cache)
    kc2[perm] = d.k_cache
    vc2[perm] = d.v_cache
    d.k_cache, d.v_cache = kc2, vc2
    d.tables = torch.where(d.tables >= 0, perm[d.tables.clamp(min=0).long()].int(), d.tables)
    b = out_tensor(wl, "f32")
    d.decode(b, split_tokens=256)
    assert torch.equal(a, b)


def test_query_heads_use_only_their_group():
    wl, t, _ = _config("tiny")
    d = DeviceLayer(wl, t)
    d.append()
    ref = out_tensor(wl, "f32")
    d.decode(ref)
    G = wl.Hq // wl.Hkv
    for g in range(wl.Hkv):
        e = DeviceLayer(wl, t)
        e.append()
        e.v_cache[:, g] *= 2.0
        got = out_tensor(wl, "f32")
        e.decode(got)
        changed = (got != ref).any(dim=2).any(dim=0).cpu().numpy()
        assert np.array_equal(changed, np.arange(wl.Hq) // G == g)
        # doubling V of a group doubles exactly the outputs of that group
        hs = slice(g * G, (g + 1) * G)
        torch.testing.assert_close(got[:, hs], 2 * ref[:, hs], rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 8, 8), (64, 8, 4), (64, 16, 2), (128, 8, 1), (128, 32, 8),
                                      (128, 16, 8), (128, 64, 8)])
@pytest.mark.parametrize("split_tokens", [None, 16, 64])
def test_shapes_and_ragged_lengths(D, Hq, Hkv, split_tokens):
    lens = (1, 15, 16, 17, 31, 32, 33, 100, 255, 256, 257, 700)
    spec = W.custom_spec(f"ragged{D}_{Hq}_{Hkv}", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, fixed_lens=lens,
                         free_frac=0.2, seed=D * 1000 + Hq * 10 + Hkv)
    wl = W.make_workload(spec)
    t = wl.layer(0)
    kc_ref, vc_ref = oracle_appended(wl, t)
    ref = oracle_decode(wl, t, kc_ref, vc_ref)
    d = DeviceLayer(wl, t)
    d.append()
    for out_dtype in ("f32", "bf16"):
        out = out_tensor(wl, out_dtype)
        d.decode(out, split_tokens=split_tokens)
        err = max_abs_err(out, ref)
        assert err <= TOL[out_dtype], f"{out_dtype}: {err}"
    assert_device_clean()


def test_single_token_and_empty_sequences_are_exact():
    spec = W.custom_spec("edge", B=4, Hq=32, Hkv=8, D=128, fixed_lens=(1, 1, 3, 1), seed=17)
    wl = W.make_workload(spec)
    t = wl.layer(0)
    d = DeviceLayer(wl, t)
    d.append()
    d.lens[2] = 0   # an empty sequence: output defined as zero
    for out_dtype in ("f32", "bf16"):
        out = out_tensor(wl, out_dtype)
        d.decode(out)
        G = wl.Hq // wl.Hkv
        vnew = torch.from_numpy(W.bf16_bits_to_f32(t["v_new"]))
        for b in (0, 1, 3):
            want = vnew[b].repeat_interleave(G, 0)
            assert torch.equal(out[b].float().cpu(), want), f"L=1 row {b} ({out_dtype}) is not V exactly"
        assert torch.all(out[2] == 0)
    assert_device_clean()


def test_strided_views_and_layer_slices():
    """Caches as views into a [layers, NB, Hkv, BS, D] pool; q and out inside larger buffers."""
    wl, t, (kc_ref, vc_ref) = _config("tiny")
    d = DeviceLayer(wl, t)
    pool_k = torch.full((3,) + tuple(d.k_cache.shape), float("nan"), dtype=torch.bfloat16, device=DEV)
    pool_v = torch.full_like(pool_k, float("nan"))
    pool_k[1] = d.k_cache
    pool_v[1] = d.v_cache
    qbig = torch.zeros(wl.B, wl.Hq + 3, wl.D + 16, dtype=torch.bfloat16, device=DEV)
    qbig[:, 1:1 + wl.Hq, 8:8 + wl.D] = d.q
    obig = torch.full((wl.B, wl.Hq, 2 * wl.D), float("nan"), dtype=torch.float32, device=DEV)
    out = obig[:, :, wl.D:]
    binding.forge_paged_kv_append(d.k_new, d.v_new, d.slots, pool_k[1], pool_v[1])
    binding.forge_paged_gqa_decode(qbig[:, 1:1 + wl.Hq, 8:8 + wl.D], pool_k[1], pool_v[1], d.tables, d.lens,
                                   wl.scale, out)
    assert np.array_equal(bits_host(pool_k[1]), kc_ref)
    assert torch.isnan(pool_k[0].float()).all() and torch.isnan(pool_k[2].float()).all()
    assert max_abs_err(out, oracle_decode(wl, t, kc_ref, vc_ref)) <= TOL["f32"]
    assert torch.isnan(obig[:, :, : wl.D]).all()


def test_cuda_graph_replay_matches_eager():
    wl, t, (kc_ref, vc_ref) = _config("qwen3_0_6b")
    d = DeviceLayer(wl, t)
    out_eager = out_tensor(wl, "bf16")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d.append()
        d.decode(out_eager)      # first call on this stream sizes the library's workspace
    torch.cuda.synchronize()
    out = out_tensor(wl, "bf16")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            d.append()
            d.decode(out)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, out_eager)
    assert max_abs_err(out, oracle_decode(wl, t, kc_ref, vc_ref)) <= TOL["bf16"]


def test_lengths_written_by_the_previous_kernel():
    """Each decode's lengths are written by the kernel just before it in the
    stream: an append whose destination row is the length array (an int32
    view of a scratch bf16 cache).  That append lets its dependent launch
    start early, so a decode CTA may read the previous lengths before
    griddepcontrol.wait and predict the wrong first blocks.  Every call must
    still decode the lengths that the append wrote."""
    wl, t, (kc_ref, vc_ref) = _config("qwen3_0_6b")
    d = DeviceLayer(wl, t)
    d.append()
    lens_a = wl.context_lens.astype(np.int32)
    lens_b = np.maximum(lens_a - 37, 1).astype(np.int32)  # other block counts, so other split boundaries
    scratch_k = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16, device=DEV)
    scratch_v = torch.zeros_like(scratch_k)
    lens_dev = scratch_k.view(torch.int32).view(-1)[: wl.B]  # row 0 of block 0, head 0
    zero_slot = torch.zeros(1, dtype=torch.int64, device=DEV)

    def row_of(lens):
        r = np.zeros(32, dtype=np.int32)
        r[: wl.B] = lens
        return torch.from_numpy(r.view(np.int16).copy()).view(torch.bfloat16).reshape(1, 1, 64).to(DEV)

    rows = {"a": row_of(lens_a), "b": row_of(lens_b)}
    order = ["a", "b"] * 8
    outs = [out_tensor(wl, "bf16") for _ in order]
    for key, out in zip(order, outs):  # back to back, no host sync in between
        binding.forge_paged_kv_append(rows[key], rows[key], zero_slot, scratch_k, scratch_v)
        binding.forge_paged_gqa_decode(d.q, d.k_cache, d.v_cache, d.tables, lens_dev, wl.scale, out)
    torch.cuda.synchronize()
    assert_device_clean()
    refs = {"a": oracle_decode(wl, t, kc_ref, vc_ref, lens=lens_a),
            "b": oracle_decode(wl, t, kc_ref, vc_ref, lens=lens_b)}
    for key, out in zip(order, outs):
        assert max_abs_err(out, refs[key]) <= TOL["bf16"], key


def test_device_side_precondition_checks_report_errors():
    wl, t, _ = _config("tiny")
    d = DeviceLayer(wl, t)
    assert binding.forge_paged_get_device_error() == 0
    bad_slots = d.slots.clone()
    bad_slots[0] = wl.NB * 16 + 5           # outside the pool: skipped, flagged
    before = d.k_cache.clone()
    binding.forge_paged_kv_append(d.k_new, d.v_new, bad_slots, d.k_cache, d.v_cache)
    assert binding.forge_paged_get_device_error() == 3
    changed = (d.k_cache.view(torch.int16) != before.view(torch.int16)).any(dim=(1, 3))
    assert int(changed.sum()) == wl.B - 1

    out = out_tensor(wl, "f32")
    bad_tables = d.tables.clone()
    bad_tables[3, 1] = wl.NB + 100          # a used entry outside the pool: not read, flagged
    binding.forge_paged_gqa_decode(d.q, d.k_cache, d.v_cache, bad_tables, d.lens, wl.scale, out)
    assert binding.forge_paged_get_device_error() == 1

    long_lens = d.lens.clone()
    assert int(long_lens[3]) == wl.MB * 16  # sequence 3 fills its table row
    long_lens[3] = wl.MB * 16 + 1           # longer than the table row: clamped, flagged
    binding.forge_paged_gqa_decode(d.q, d.k_cache, d.v_cache, d.tables, long_lens, wl.scale, out)
    assert binding.forge_paged_get_device_error() == 2
    assert binding.forge_paged_get_device_error() == 0


def test_continuous_batching_36_layer_step():
    """One step of the 36-layer config: per layer, append then decode, all
    layers in one shared pool; every layer's caches and output checked
    against the oracle."""
    wl = W.make_workload("cb36")
    L = wl.layers
    shape = (L, wl.NB, wl.Hkv, 16, wl.D)
    pool_k = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
    pool_v = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
    qs, kns, vns, outs = [], [], [], []
    from gpu_util import bf16_dev
    for l in range(L):
        t = wl.layer(l)
        pool_k[l].copy_(bf16_dev(t["k_cache"]))
        pool_v[l].copy_(bf16_dev(t["v_cache"]))
        qs.append(bf16_dev(t["q"]))
        kns.append(bf16_dev(t["k_new"]))
        vns.append(bf16_dev(t["v_new"]))
        outs.append(out_tensor(wl, "bf16"))
        del t
    slots = torch.from_numpy(wl.slot_mapping).to(DEV)
    tables = torch.from_numpy(wl.block_tables).to(DEV)
    lens = torch.from_numpy(wl.context_lens).to(DEV)
    crossing = int(((wl.context_lens - 1) % 16 == 0).sum())
    assert crossing > 0, "some sequences should start a new block this step"
    for l in range(L):
        binding.forge_paged_kv_append(kns[l], vns[l], slots, pool_k[l], pool_v[l])
        binding.forge_paged_gqa_decode(qs[l], pool_k[l], pool_v[l], tables, lens, wl.scale, outs[l])
    torch.cuda.synchronize()
    assert_device_clean()
    worst = 0.0
    for l in range(L):                   # the inputs again, from the same seeds
        t = wl.layer(l)
        kc_ref, vc_ref = oracle_appended(wl, t)
        assert np.array_equal(bits_host(pool_k[l]), kc_ref), f"layer {l}: K cache"
        assert np.array_equal(bits_host(pool_v[l]), vc_ref), f"layer {l}: V cache"
        err = max_abs_err(outs[l], oracle_decode(wl, t, kc_ref, vc_ref))
        assert err <= TOL["bf16"], f"layer {l}: {err}"
        worst = max(worst, err)
    print(f"36-layer step: every layer within {worst:.3e} of the oracle")


def test_one_workspace_serves_changing_shapes():
    """A workspace zeroed once serves calls of different shapes in any order:
    split arrival counters live in a fixed prefix that no call's data overlaps."""
    names = ["skewed", "qwen3_4b", "tiny", "skewed", "qwen3_0_6b", "qwen3_4b"]
    need = 0
    for name in set(names):
        wl = _config(name)[0]
        need = max(need, binding.forge_paged_gqa_decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.D, wl.MB, 64))
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    refs = {}
    for name in names:
        wl, t, (kc_ref, vc_ref) = _config(name)
        if name not in refs:
            refs[name] = oracle_decode(wl, t, kc_ref, vc_ref)
        d = DeviceLayer(wl, t)
        d.append()
        out = out_tensor(wl)
        binding.forge_paged_gqa_decode_ex(d.q, d.k_cache, d.v_cache, d.tables, d.lens, wl.scale, out, ws, 64)
        err = max_abs_err(out, refs[name])
        assert err <= TOL[wl.spec.out_dtype], f"{name}: {err}"
    assert_device_clean()


def test_scratch_cannot_grow_during_capture():
    """The library-owned scratch grows in stream order, but not while the
    stream is being captured: the call refuses with FORGE_ERR_WORKSPACE and
    enqueues nothing; after an eager call of that size, capture works."""
    wl, t, (kc_ref, vc_ref) = _config("skewed")
    d = DeviceLayer(wl, t)
    d.append()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    out = out_tensor(wl, "f32")
    g = torch.cuda.CUDAGraph()
    # Earlier tests' graphs and buffers are released before the capture
    # window, not by a garbage collection inside it; the refusal capture is
    # relaxed, so that only an operation on the captured stream (which a
    # refused call must not enqueue) could invalidate it.
    gc.collect()
    torch.cuda.synchronize()
    with pytest.raises(binding.ForgeError) as info:
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            binding.forge_paged_gqa_decode(d.q, d.k_cache, d.v_cache, d.tables, d.lens, wl.scale, out, stream=s)
    assert info.value.status == -7
    del info  # its traceback holds this frame
    with torch.cuda.stream(s):
        binding.forge_paged_gqa_decode(d.q, d.k_cache, d.v_cache, d.tables, d.lens, wl.scale, out, stream=s)
    s.synchronize()
    g2 = torch.cuda.CUDAGraph()
    out2 = out_tensor(wl, "f32")
    with torch.cuda.graph(g2, stream=s, capture_error_mode="thread_local"):
        binding.forge_paged_gqa_decode(d.q, d.k_cache, d.v_cache, d.tables, d.lens, wl.scale, out2, stream=s)
    g2.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    assert max_abs_err(out2, oracle_decode(wl, t, kc_ref, vc_ref)) <= TOL["f32"]
    assert_device_clean()
