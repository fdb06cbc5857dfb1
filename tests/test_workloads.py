"""The seeded input generator: structure the parity tests rely on."""
import numpy as np
import pytest
import torch

from paged_kv_gqa_06_gb300 import workloads as W


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(100_000).astype(np.float32) * 3
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0]   # exact ties
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(W.f32_to_bf16_bits(W.bf16_bits_to_f32(ours)), ours)


@pytest.mark.parametrize("name", list(W.SPECS))
def test_tables_are_a_valid_allocation(name):
    wl = W.make_workload(name)
    s = wl.spec
    assert wl.context_lens.shape == (s.B,) and wl.context_lens.dtype == np.int32
    nblk = -(-wl.context_lens.astype(np.int64) // 16)
    assert wl.MB == max(1, int(nblk.max()))
    used = []
    for b in range(s.B):
        row = wl.block_tables[b]
        assert np.all(row[: nblk[b]] >= 0) and np.all(row[: nblk[b]] < wl.NB)
        assert np.all(row[nblk[b]:] == -1)
        used.extend(row[: nblk[b]].tolist())
    assert len(used) == len(set(used))          # no block shared between sequences
    if s.free_frac:
        free = wl.NB - len(used)
        assert free == wl.NB - int(nblk.sum())
        assert abs(free / wl.NB - s.free_frac) < max(0.01, 1.0 / wl.NB)   # NB = ceil(needed / (1 - f))
    if s.nb_fixed:
        assert wl.NB == s.nb_fixed
    # the appended token's slot is position L-1 of its sequence
    for b in range(s.B):
        t = int(wl.context_lens[b]) - 1
        assert wl.slot_mapping[b] == wl.block_tables[b, t // 16] * 16 + t % 16


def test_length_recipes():
    assert W.make_workload("tiny").context_lens.tolist() == [7, 16, 33, 64]
    assert W.make_workload("skewed").context_lens.tolist() == [32768, 1024, 256, 17]
    l4 = W.make_workload("qwen3_4b").context_lens
    assert l4.min() >= 512 and l4.max() <= 8192
    l6 = W.make_workload("qwen3_0_6b").context_lens
    assert l6.min() >= 128 and l6.max() <= 2048
    lc = W.make_workload("cb36").context_lens
    assert lc.min() >= 1 and lc.max() <= 16384 and 300 < np.median(lc) < 3000


def test_seeded_and_deterministic():
    a, b = W.make_workload("tiny"), W.make_workload("tiny")
    assert np.array_equal(a.block_tables, b.block_tables)
    la, lb = a.layer(0), b.layer(0)
    for k in la:
        assert np.array_equal(la[k], lb[k])
    c = W.make_workload("tiny", seed=99)
    assert not np.array_equal(c.block_tables, a.block_tables)
    assert not np.array_equal(a.layer(1)["q"], la["q"])


def test_poison_covers_exactly_the_unheld_slots():
    wl = W.make_workload("tiny")
    t = wl.layer(0)
    nan = t["k_cache"] == W.BF16_NAN
    assert np.array_equal(nan, t["v_cache"] == W.BF16_NAN)
    held = np.zeros((wl.NB, 16), bool)
    for b in range(wl.B):
        for pos in range(int(wl.context_lens[b]) - 1):
            held[wl.block_tables[b, pos // 16], pos % 16] = True
    assert np.array_equal(nan.all(axis=(1, 3)), ~held)
    assert not np.any(nan[held.nonzero()[0], :, held.nonzero()[1], :])


def test_qwen3_4b_key_scale_doubles_values():
    spec = W.custom_spec(B=1, Hq=4, Hkv=1, D=64, fixed_lens=(40,), k_mul=2.0)
    t = W.make_workload(spec).layer(0)
    k = W.bf16_bits_to_f32(t["k_cache"])
    k = k[np.isfinite(k)]
    assert 1.6 < k.std() < 2.4
    # doubling is exact: halving every value gives back a bf16 number
    half = k / 2
    assert np.array_equal(W.bf16_bits_to_f32(W.f32_to_bf16_bits(half)), half)


def test_byte_accounting():
    wl = W.make_workload("tiny")
    tok = 7 + 16 + 33 + 64
    assert wl.bytes_decode() == 4 * 8 * 64 * 2 + tok * 2 * 64 * 2 * 2 + 4 * 8 * 64 * 4
    assert wl.bytes_append() == 4 * 2 * 64 * 2 * 2 * 2
