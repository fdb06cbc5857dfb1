"""Pins of the oracle's paged prefill (oracle_paged_prefill).

The prefill runs one pass over a run of new tokens and fills the cache
("Make the Engine Talk", 1.2); each query token attends causally to the
cached tokens up to its own position.  Pinned by:
  * hand-derived examples (tests/golden/hand_worked.json, "prefill_cases");
  * the decode, which is the one-query-token case and is itself pinned:
    identical results, bit for bit;
  * torch's scaled_dot_product_attention in fp64 with a causal mask, over
    K/V found by scanning the physical pool, for whole prompts;
  * invariants: a chunk's outputs equal the same rows of a whole-prompt
    prefill; changing K/V after a token's position leaves that token's
    output alone, changing it before does not; NaN in unheld slots never
    reaches an output.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from paged_kv_gqa_06_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")
SCALES = {"ln2": math.log(2.0), "ln3": math.log(3.0)}


def _f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def _bits(x):
    return W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["prefill_cases"], ids=lambda c: c["name"])
def test_prefill_hand_worked(oracle_mod, case):
    BS, NB, Hkv, D = case["BS"], case["NB"], case["Hkv"], case["D"]
    kc = np.full((NB, Hkv, BS, D), W.BF16_NAN, dtype=np.uint16)
    vc = kc.copy()
    tables = np.array(case["block_tables"], dtype=np.int32)
    for b, tok in case["tokens"].items():
        for t, (k, v) in enumerate(zip(tok["k"], tok["v"])):
            p = tables[int(b), t // BS]
            kc[p, 0, t % BS] = _bits(k)
            vc[p, 0, t % BS] = _bits(v)
    out = oracle_mod.paged_prefill(_bits(case["q"]), kc, vc, tables, np.array(case["context_lens"], np.int32),
                                   np.array(case["query_start"], np.int32), SCALES[case["scale"]])
    np.testing.assert_allclose(out, np.array(case["expected"]), rtol=0, atol=1e-12)


def _appended(oracle_mod, pw, t):
    kc, vc = t["k_cache"].copy(), t["v_cache"].copy()
    oracle_mod.paged_kv_append(t["k_new"], t["v_new"], pw.slot_mapping, kc, vc)
    return kc, vc


def _prefill(oracle_mod, pw, q, kc, vc, **kw):
    return oracle_mod.paged_prefill(q, kc, vc, pw.block_tables, pw.context_lens, pw.query_start,
                                    kw.get("scale", pw.scale), nthreads=kw.get("nthreads"))


def _spec(**kw):
    return W.custom_spec("pf", **kw)


def test_one_query_token_is_the_decode(oracle_mod):
    pw = W.make_prefill(_spec(B=5, Hq=8, Hkv=2, D=64, fixed_lens=(1, 16, 17, 40, 3), free_frac=0.2),
                        chunk_lens=(1, 1, 1, 1, 1))
    t = pw.layer(0)
    kc, vc = _appended(oracle_mod, pw, t)
    got = _prefill(oracle_mod, pw, t["q"], kc, vc)
    want = oracle_mod.paged_gqa_decode(t["q"], kc, vc, pw.block_tables, pw.context_lens, pw.scale)
    assert np.array_equal(got, want)


def _dense_by_pool_scan(pw, kc, vc, b):
    """[L, Hkv, D] K/V of sequence b found by scanning every physical block for
    the (sequence, logical block) that owns it."""
    L = int(pw.context_lens[b])
    K = np.full((L, pw.Hkv, pw.D), np.nan)
    V = np.full_like(K, np.nan)
    for p in range(pw.NB):
        hits = np.nonzero(pw.block_tables[b] == p)[0]
        for j in hits:
            for o in range(pw.BS):
                tok = int(j) * pw.BS + o
                if tok < L:
                    K[tok] = _f64(kc[p, :, o, :])
                    V[tok] = _f64(vc[p, :, o, :])
    assert not np.isnan(K).any()
    return K, V


@pytest.mark.parametrize("kw", [dict(B=3, Hq=8, Hkv=2, D=64, fixed_lens=(33, 1, 20)),
                                dict(B=2, Hq=4, Hkv=4, D=128, fixed_lens=(17, 48), free_frac=0.3),
                                dict(B=1, Hq=16, Hkv=2, D=64, fixed_lens=(70,))])
def test_whole_prompt_matches_torch_causal_sdpa(oracle_mod, kw):
    pw = W.make_prefill(_spec(**kw))            # chunk 0: every token is a query
    t = pw.layer(0)
    kc, vc = _appended(oracle_mod, pw, t)
    got = _prefill(oracle_mod, pw, t["q"], kc, vc)
    G = pw.Hq // pw.Hkv
    for b in range(pw.B):
        K, V = _dense_by_pool_scan(pw, kc, vc, b)
        q0, q1 = int(pw.query_start[b]), int(pw.query_start[b + 1])
        q = torch.tensor(_f64(t["q"][q0:q1])).transpose(0, 1)                  # [Hq, n, D]
        Kt = torch.tensor(K).transpose(0, 1).repeat_interleave(G, 0)           # [Hq, L, D]
        Vt = torch.tensor(V).transpose(0, 1).repeat_interleave(G, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(q[None], Kt[None], Vt[None], is_causal=True,
                                                               scale=pw.scale)[0].transpose(0, 1).numpy()
        np.testing.assert_allclose(got[q0:q1], ref, rtol=0, atol=1e-10)


def test_chunks_equal_the_whole_prompt(oracle_mod):
    spec = _spec(B=3, Hq=8, Hkv=2, D=64, fixed_lens=(50, 31, 64), free_frac=0.1)
    whole = W.make_prefill(spec)
    t = whole.layer(0)
    kc, vc = _appended(oracle_mod, whole, t)
    full = _prefill(oracle_mod, whole, t["q"], kc, vc)
    chunks = (7, 31, 16)                        # the last n_b tokens of each sequence as queries
    part = W.make_prefill(spec, chunk_lens=chunks)
    rows = np.concatenate([np.arange(int(whole.query_start[b + 1]) - n, int(whole.query_start[b + 1]))
                           for b, n in enumerate(chunks)])
    got = _prefill(oracle_mod, part, t["q"][rows], kc, vc)
    assert np.array_equal(got, full[rows])


def test_causality(oracle_mod):
    pw = W.make_prefill(_spec(B=1, Hq=8, Hkv=2, D=64, fixed_lens=(40,)))
    t = pw.layer(0)
    kc, vc = _appended(oracle_mod, pw, t)
    base = _prefill(oracle_mod, pw, t["q"], kc, vc)
    cut = 25                                    # change the cache from this position on
    kc2, vc2 = kc.copy(), vc.copy()
    for tok in range(cut, 40):
        p, o = int(pw.block_tables[0, tok // 16]), tok % 16
        kc2[p, :, o, :] = _bits(np.full((pw.Hkv, pw.D), 3.0))
        vc2[p, :, o, :] = _bits(np.full((pw.Hkv, pw.D), -5.0))
    moved = _prefill(oracle_mod, pw, t["q"], kc2, vc2)
    assert np.array_equal(moved[:cut], base[:cut])          # earlier queries never see the change
    assert np.all(np.abs(moved[cut:] - base[cut:]).max(axis=(1, 2)) > 1e-3)


def test_unheld_slots_never_reach_the_output(oracle_mod):
    pw = W.make_prefill("prefill_tiny")
    t = pw.layer(0)
    kc, vc = _appended(oracle_mod, pw, t)
    out = _prefill(oracle_mod, pw, t["q"], kc, vc)
    assert np.isfinite(out).all() and np.isnan(W.bf16_bits_to_f32(kc)).any()


def test_thread_count_does_not_change_the_result(oracle_mod):
    pw = W.make_prefill("prefill_tiny")
    t = pw.layer(0)
    kc, vc = _appended(oracle_mod, pw, t)
    assert np.array_equal(_prefill(oracle_mod, pw, t["q"], kc, vc, nthreads=1),
                          _prefill(oracle_mod, pw, t["q"], kc, vc, nthreads=7))


def test_bad_arguments_are_rejected(oracle_mod):
    pw = W.make_prefill("prefill_tiny")
    t = pw.layer(0)
    kc, vc = _appended(oracle_mod, pw, t)
    qs = pw.query_start.copy()
    qs[1] = qs[0] + int(pw.context_lens[0]) + 1           # more queries than context
    qs[2:] += qs[1] - pw.query_start[1]
    q = np.zeros((int(qs[-1]), pw.Hq, pw.D), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle_mod.paged_prefill(q, kc, vc, pw.block_tables, pw.context_lens, qs, pw.scale)
    with pytest.raises(ValueError):                         # query_start not ending at T
        oracle_mod.paged_prefill(t["q"][:-1], kc, vc, pw.block_tables, pw.context_lens, pw.query_start,
                                 pw.scale)
