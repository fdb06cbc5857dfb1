"""Pins for the CPU oracle: checks against things other than the oracle itself.

* hand-derived worked examples (tests/golden/hand_worked.json);
* brute-force dense attention that finds each token by scanning the physical
  pool (not by walking the block table), with KV heads repeated per group;
* torch's scaled_dot_product_attention in fp64 (a library routine);
* closed forms: one token returns its V; equal keys or scale 0 give the mean
  of V; a dominant key returns its V; all-ones V gives ones;
* invariants: block placement, group isolation, linearity in V, NaN poison,
  threading.

The attention definition these follow: "Make the Engine Talk" section 1.3
(grouped-query attention) and the forge-engine README "What it implements"
(paged block pool).  Append follows section 1.2 (the cache grows by the one
new token of each decode pass).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from paged_kv_gqa_06_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _bits(x):
    return W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def _small(name="pins", **kw):
    spec = W.custom_spec(name, **kw)
    wl = W.make_workload(spec)
    return wl, wl.layer(0)


def _appended(oracle_mod, wl, t):
    """Caches after the oracle's append (the state decode reads)."""
    kc, vc = t["k_cache"].copy(), t["v_cache"].copy()
    oracle_mod.paged_kv_append(t["k_new"], t["v_new"], wl.slot_mapping, kc, vc)
    return kc, vc


def _decode(oracle_mod, wl, t, kc, vc, scale=None, tables=None, lens=None, nthreads=2):
    return oracle_mod.paged_gqa_decode(
        t["q"], kc, vc, wl.block_tables if tables is None else tables,
        wl.context_lens if lens is None else lens,
        wl.scale if scale is None else scale, nthreads=nthreads)


# ---------------------------------------------------------------- worked examples

def _golden_inputs(case):
    BS, NB, Hq, Hkv, D = (case[k] for k in ("BS", "NB", "Hq", "Hkv", "D"))
    kc = np.full((NB, Hkv, BS, D), W.BF16_NAN, dtype=np.uint16)
    vc = kc.copy()
    table = np.array(case["block_tables"], dtype=np.int32)
    L = case["context_lens"][0]
    if "tokens" in case:
        per_head = [case["tokens"]] * Hkv
    else:
        tp = case["tokens_per_head"]
        per_head = [{"k": tp["k"][g], "v": tp["v"][g]} for g in range(Hkv)]
    for g in range(Hkv):
        for t in range(L):
            p, o = table[0, t // BS], t % BS
            kc[p, g, o] = _bits(per_head[g]["k"][t])
            vc[p, g, o] = _bits(per_head[g]["v"][t])
    scale = {"ln3": math.log(3.0), "ln2": math.log(2.0), "1": 1.0}[case["scale"]]
    return (_bits(case["q"]), kc, vc, table, np.array(case["context_lens"], np.int32), scale)


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_hand_worked_examples(oracle_mod, idx):
    case = json.load(open(GOLDEN))["cases"][idx]
    q, kc, vc, table, lens, scale = _golden_inputs(case)
    out = oracle_mod.paged_gqa_decode(q, kc, vc, table, lens, scale, nthreads=1)
    np.testing.assert_allclose(out, np.array(case["expected"], dtype=np.float64),
                               rtol=0, atol=1e-12)


# ---------------------------------------------------------------- brute force / library

def _dense_by_pool_scan(wl, kc, vc):
    """Dense [B, Lmax, Hkv, D] K/V found by scanning every physical block and
    asking which (sequence, logical block) owns it."""
    owner = {}
    for b in range(wl.B):
        for j in range(wl.MB):
            p = int(wl.block_tables[b, j])
            if p >= 0:
                owner[p] = (b, j)
    Lmax = int(wl.context_lens.max())
    Kd = np.zeros((wl.B, Lmax, wl.Hkv, wl.D))
    Vd = np.zeros_like(Kd)
    for p in range(wl.NB):
        if p not in owner:
            continue
        b, j = owner[p]
        for o in range(wl.BS):
            t = j * wl.BS + o
            if t < wl.context_lens[b]:
                Kd[b, t] = _f64(kc[p, :, o, :])
                Vd[b, t] = _f64(vc[p, :, o, :])
    return Kd, Vd


def _brute_force(wl, q_bits, kc, vc, scale):
    G = wl.Hq // wl.Hkv
    Kd, Vd = _dense_by_pool_scan(wl, kc, vc)
    Kr = np.repeat(Kd, G, axis=2)          # KV head g serves query heads gG .. gG+G-1
    Vr = np.repeat(Vd, G, axis=2)
    q = _f64(q_bits)
    logits = np.einsum("bhd,bthd->bht", q, Kr) * scale
    Lmax = Kd.shape[1]
    mask = np.arange(Lmax)[None, None, :] < wl.context_lens[:, None, None]
    logits = np.where(mask, logits, -np.inf)
    w = scipy.special.softmax(logits, axis=-1)
    return np.einsum("bht,bthd->bhd", w, Vr)


@pytest.mark.parametrize("kw", [
    dict(B=4, Hq=8, Hkv=2, D=64, fixed_lens=(7, 16, 33, 64), nb_fixed=32),
    dict(B=3, Hq=8, Hkv=8, D=128, fixed_lens=(40, 1, 17)),
    dict(B=2, Hq=16, Hkv=2, D=64, fixed_lens=(50, 31), free_frac=0.3),
])
def test_oracle_matches_brute_force(oracle_mod, kw):
    wl, t = _small(**kw)
    kc, vc = _appended(oracle_mod, wl, t)
    got = _decode(oracle_mod, wl, t, kc, vc)
    want = _brute_force(wl, t["q"], kc, vc, wl.scale)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_oracle_matches_torch_sdpa_fp64(oracle_mod):
    wl, t = _small(B=3, Hq=8, Hkv=2, D=64, fixed_lens=(5, 47, 16))
    kc, vc = _appended(oracle_mod, wl, t)
    got = _decode(oracle_mod, wl, t, kc, vc)
    G = wl.Hq // wl.Hkv
    for b in range(wl.B):
        L = int(wl.context_lens[b])
        rows = [(int(wl.block_tables[b, i // wl.BS]), i % wl.BS) for i in range(L)]
        K = torch.tensor(np.stack([_f64(kc[p, :, o]) for p, o in rows], 1))  # [Hkv, L, D]
        V = torch.tensor(np.stack([_f64(vc[p, :, o]) for p, o in rows], 1))
        q = torch.tensor(_f64(t["q"][b]))[:, None, :]                          # [Hq, 1, D]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None], K.repeat_interleave(G, 0)[None], V.repeat_interleave(G, 0)[None],
            scale=wl.scale)[0, :, 0, :].numpy()
        np.testing.assert_allclose(got[b], ref, rtol=0, atol=1e-10)


# ---------------------------------------------------------------- closed forms

def test_single_token_returns_its_value_exactly(oracle_mod):
    wl, t = _small(B=3, Hq=8, Hkv=2, D=64, fixed_lens=(1, 1, 1))
    kc, vc = _appended(oracle_mod, wl, t)
    out = _decode(oracle_mod, wl, t, kc, vc)
    G = wl.Hq // wl.Hkv
    for b in range(wl.B):
        for h in range(wl.Hq):
            assert np.array_equal(out[b, h], _f64(t["v_new"][b, h // G]))


@pytest.mark.parametrize("mode", ["equal_keys", "zero_scale"])
def test_uniform_weights_give_mean_of_values(oracle_mod, mode):
    wl, t = _small(B=2, Hq=8, Hkv=2, D=64, fixed_lens=(21, 48))
    kc, vc = _appended(oracle_mod, wl, t)
    scale = wl.scale
    if mode == "equal_keys":
        kc[:] = _bits(0.75)
    else:
        scale = 0.0
    out = _decode(oracle_mod, wl, t, kc, vc, scale=scale)
    G = wl.Hq // wl.Hkv
    for b in range(wl.B):
        L = int(wl.context_lens[b])
        rows = np.stack([_f64(vc[wl.block_tables[b, i // 16], :, i % 16]) for i in range(L)])
        for h in range(wl.Hq):
            np.testing.assert_allclose(out[b, h], rows[:, h // G].mean(0), rtol=0, atol=1e-12)


def test_dominant_key_returns_its_value(oracle_mod):
    wl, t = _small(B=1, Hq=4, Hkv=1, D=64, fixed_lens=(37,))
    kc, vc = _appended(oracle_mod, wl, t)
    q = t["q"].copy()
    q[0] = _bits(np.sign(_f64(q[0, 0]))[None, :] * np.ones((4, 64)))  # all heads: same +-1 query
    qs = np.sign(_f64(q[0, 0]))
    kc[:] = _bits(np.zeros(64))
    star = 29
    p, o = wl.block_tables[0, star // 16], star % 16
    kc[p, 0, o] = _bits(8.0 * qs)        # logit 8*64/8 = 64 vs 0 for every other token
    out = oracle_mod.paged_gqa_decode(q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    np.testing.assert_allclose(out[0], np.repeat(_f64(vc[p, 0, o])[None], 4, 0), rtol=0, atol=1e-20 + 1e-12)


def test_all_ones_values_give_ones(oracle_mod):
    wl, t = _small(B=2, Hq=8, Hkv=2, D=64, fixed_lens=(19, 64))
    kc, vc = _appended(oracle_mod, wl, t)
    vc = np.where(vc == W.BF16_NAN, vc, _bits(1.0)).astype(np.uint16)
    out = _decode(oracle_mod, wl, t, kc, vc)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-14)


def test_output_is_linear_in_values(oracle_mod):
    # For a fixed q and K the softmax weights do not depend on V, so
    # out(a V1 + b V2) = a out(V1) + b out(V2).  Small integers keep every
    # combination exact in bf16, which leaves only fp64 rounding.
    wl, t = _small(B=3, Hq=8, Hkv=2, D=64, fixed_lens=(7, 33, 64))
    kc, vc = _appended(oracle_mod, wl, t)
    live = vc != W.BF16_NAN
    rng = np.random.default_rng(11)
    v1 = rng.integers(-4, 5, size=vc.shape).astype(np.float32)
    v2 = rng.integers(-4, 5, size=vc.shape).astype(np.float32)

    def cache_of(x):
        return np.where(live, _bits(x), vc).astype(np.uint16)

    o1 = _decode(oracle_mod, wl, t, kc, cache_of(v1))
    o2 = _decode(oracle_mod, wl, t, kc, cache_of(v2))
    o12 = _decode(oracle_mod, wl, t, kc, cache_of(2 * v1 - 3 * v2))
    assert np.abs(o1 - o2).max() > 0.1  # the two parts differ
    np.testing.assert_allclose(o12, 2 * o1 - 3 * o2, rtol=0, atol=1e-12)


def test_zero_length_gives_zeros(oracle_mod):
    wl, t = _small(B=2, Hq=8, Hkv=2, D=64, fixed_lens=(9, 20))
    kc, vc = _appended(oracle_mod, wl, t)
    lens = wl.context_lens.copy()
    lens[1] = 0
    out = _decode(oracle_mod, wl, t, kc, vc, lens=lens)
    assert np.all(out[1] == 0.0)
    assert np.all(np.isfinite(out[0]))


# ---------------------------------------------------------------- invariants

def test_block_placement_does_not_matter(oracle_mod):
    wl, t = _small(B=3, Hq=8, Hkv=2, D=64, fixed_lens=(33, 64, 2), free_frac=0.25)
    kc, vc = _appended(oracle_mod, wl, t)
    ref = _decode(oracle_mod, wl, t, kc, vc)
    perm = np.random.default_rng(5).permutation(wl.NB)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    tables = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
    got = _decode(oracle_mod, wl, t, kc2, vc2, tables=tables)
    assert np.array_equal(got, ref)


def test_query_heads_use_only_their_group(oracle_mod):
    wl, t = _small(B=2, Hq=8, Hkv=2, D=64, fixed_lens=(25, 40))
    kc, vc = _appended(oracle_mod, wl, t)
    ref = _decode(oracle_mod, wl, t, kc, vc)
    G = wl.Hq // wl.Hkv
    for g in range(wl.Hkv):
        kc2, vc2 = kc.copy(), vc.copy()
        live = kc2[:, g] != W.BF16_NAN
        kc2[:, g][live] ^= np.uint16(0x0040)   # flip a mantissa bit of every live K of head g
        vc2[:, g][live] ^= np.uint16(0x0040)
        got = _decode(oracle_mod, wl, t, kc2, vc2)
        changed = np.any(got != ref, axis=(0, 2))
        assert np.array_equal(changed, np.arange(wl.Hq) // G == g)


def test_unowned_slots_never_read(oracle_mod):
    wl, t = _small(B=3, Hq=8, Hkv=2, D=64, fixed_lens=(5, 17, 30), free_frac=0.4)
    kc, vc = _appended(oracle_mod, wl, t)
    out_nan = _decode(oracle_mod, wl, t, kc, vc)
    assert np.all(np.isfinite(out_nan))
    rng = np.random.default_rng(3)
    kc2, vc2 = kc.copy(), vc.copy()
    for c in (kc2, vc2):
        nanm = c == W.BF16_NAN
        c[nanm] = _bits(rng.standard_normal(int(nanm.sum())))
    assert np.array_equal(_decode(oracle_mod, wl, t, kc2, vc2), out_nan)


def test_threads_do_not_change_results(oracle_mod):
    wl, t = _small(B=4, Hq=8, Hkv=2, D=64, fixed_lens=(7, 16, 33, 64), nb_fixed=32)
    kc, vc = _appended(oracle_mod, wl, t)
    a = _decode(oracle_mod, wl, t, kc, vc, nthreads=1)
    b = _decode(oracle_mod, wl, t, kc, vc, nthreads=5)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- append

def test_append_writes_exactly_the_new_rows(oracle_mod):
    wl = W.make_workload("tiny")
    t = wl.layer(0)
    kc, vc = _appended(oracle_mod, wl, t)
    # worked positions: L=16 -> last slot of the first block; L=33 -> first slot of the third
    assert wl.slot_mapping[1] == wl.block_tables[1, 0] * 16 + 15
    assert wl.slot_mapping[2] == wl.block_tables[2, 2] * 16 + 0
    changed = np.any(kc != t["k_cache"], axis=(1, 3))   # [NB, BS]
    expect = np.zeros_like(changed)
    for b in range(wl.B):
        s = int(wl.slot_mapping[b])
        expect[s // 16, s % 16] = True
    assert np.array_equal(changed, expect)
    assert np.array_equal(np.any(vc != t["v_cache"], axis=(1, 3)), expect)
    for b in range(wl.B):
        s = int(wl.slot_mapping[b])
        assert np.array_equal(kc[s // 16, :, s % 16], t["k_new"][b])
        assert np.array_equal(vc[s // 16, :, s % 16], t["v_new"][b])


def test_append_skips_negative_slots_and_rejects_out_of_pool(oracle_mod):
    wl = W.make_workload("tiny")
    t = wl.layer(0)
    kc, vc = t["k_cache"].copy(), t["v_cache"].copy()
    oracle_mod.paged_kv_append(t["k_new"], t["v_new"], np.full(wl.B, -1, np.int64), kc, vc)
    assert np.array_equal(kc, t["k_cache"]) and np.array_equal(vc, t["v_cache"])
    with pytest.raises(ValueError):
        oracle_mod.paged_kv_append(t["k_new"], t["v_new"],
                                   np.array([0, 0, 0, wl.NB * 16], np.int64), kc, vc)


def test_decode_rejects_bad_tables(oracle_mod):
    wl, t = _small(B=1, Hq=4, Hkv=1, D=64, fixed_lens=(20,))
    kc, vc = _appended(oracle_mod, wl, t)
    bad = wl.block_tables.copy()
    bad[0, 1] = -1
    with pytest.raises(ValueError):
        _decode(oracle_mod, wl, t, kc, vc, tables=bad)
    with pytest.raises(ValueError):
        _decode(oracle_mod, wl, t, kc, vc, lens=np.array([wl.MB * 16 + 1], np.int32))
