"""forge_paged_qk_append_gqa_decode: RMSNorm and RoPE on q and the new k,
then append + decode, in one launch, against the oracle.

The oracle takes each step from its own fp64 definition (oracle.rmsnorm,
oracle.rope), rounds q' and k' to bf16 once, appends k' and decodes with q'.
The kernel computes q' and k' in fp32 and rounds once, so an element whose
exact value sits within fp32 error of a bf16 rounding boundary may round the
other way: the appended cache rows are compared within one bf16 ulp, every
other cache byte exactly, and the output within the parity tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, TOL, DeviceLayer, bits_host, max_abs_err, out_tensor
from paged_kv_gqa_06_gb300 import binding
from paged_kv_gqa_06_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("decode_kernel")]

THETA = 1e6   # Qwen3's rotary base
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


def _reference(wl, t, qw, kw, rope):
    """Oracle caches after the append of k' and the decode output with q'."""
    pos = wl.context_lens.astype(np.int64) - 1

    def path(x, w):
        y = oracle.rmsnorm(x, w, EPS) if w is not None else W.bf16_bits_to_f32(x).astype(np.float64)
        if rope:
            y = oracle.rope(y, pos, THETA)
        return oracle.bf16_round(y)

    q2, k2 = path(t["q"], qw), path(t["k_new"], kw)
    kc, vc = t["k_cache"].copy(), t["v_cache"].copy()
    oracle.paged_kv_append(k2, t["v_new"], wl.slot_mapping, kc, vc)
    out = oracle.paged_gqa_decode(q2, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    return kc, vc, out


def _run(wl, t, qw, kw, rope, out_dtype, rows=None):
    d = DeviceLayer(wl, t)
    out = out_tensor(wl, out_dtype)
    to_dev = lambda a: None if a is None else torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(DEV)
    table = None
    if rope:
        table = binding.forge_rope_cos_sin_table(THETA, wl.D, rows or wl.MB * 16).to(DEV)
    binding.forge_paged_qk_append_gqa_decode(d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.tables, d.lens,
                                             wl.scale, out, q_norm_weight=to_dev(qw), k_norm_weight=to_dev(kw),
                                             norm_eps=EPS, rope_cos_sin=table)
    return d, out


def _check_cache(got, want, wl):
    """Equal everywhere except the appended rows, which may be one bf16 ulp off."""
    diff = got != want
    held = np.zeros(got.shape, dtype=bool)
    for b in range(wl.B):
        s = int(wl.slot_mapping[b])
        if s >= 0:
            held[s // 16, :, s % 16, :] = True
    assert not np.any(diff & ~held), "bytes outside the appended rows changed"
    g, w = got[diff].astype(np.int32), want[diff].astype(np.int32)
    assert np.all((g >> 15) == (w >> 15)) and np.all(np.abs(g - w) <= 1), "appended row off by more than 1 ulp"
    assert diff.sum() <= max(8, held.sum() // 1000)


CASES = [("tiny", "f32"), ("qwen3_4b", "bf16"), ("skewed", "f32")]


@pytest.mark.parametrize("name,out_dtype", CASES)
@pytest.mark.parametrize("norm,rope", [(True, True), (False, True), (True, False)])
def test_qk_path_matches_oracle(name, out_dtype, norm, rope):
    wl = W.make_workload(name)
    t = wl.layer(0)
    qw, kw = wl.qk_norm_weights(0) if norm else (None, None)
    kc_ref, vc_ref, ref = _reference(wl, t, qw, kw, rope)
    d, out = _run(wl, t, qw, kw, rope, out_dtype)
    _check_cache(bits_host(d.k_cache), kc_ref, wl)
    assert np.array_equal(bits_host(d.v_cache), vc_ref)          # V is appended untouched
    err = max_abs_err(out, ref)
    assert err <= TOL[out_dtype], f"{name}/{out_dtype} norm={norm} rope={rope}: {err}"
    assert binding.forge_paged_get_device_error() == 0


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 64, 8), (128, 8, 8), (64, 16, 2)])
def test_qk_path_ragged_shapes(D, Hq, Hkv):
    lens = (1, 15, 16, 17, 33, 100, 257, 700, 0)
    spec = W.custom_spec(f"qk{D}_{Hq}_{Hkv}", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, fixed_lens=lens, free_frac=0.2,
                         seed=300 + Hq)
    wl = W.make_workload(spec)
    t = wl.layer(0)
    qw, kw = wl.qk_norm_weights(0)
    kc_ref, vc_ref, ref = _reference(wl, t, qw, kw, True)
    for out_dtype in ("f32", "bf16"):
        d, out = _run(wl, t, qw, kw, True, out_dtype)
        _check_cache(bits_host(d.k_cache), kc_ref, wl)
        assert max_abs_err(out, ref) <= TOL[out_dtype]
        assert torch.all(out[-1] == 0)
    assert binding.forge_paged_get_device_error() == 0


def test_no_options_is_the_plain_fused_call():
    wl = W.make_workload("qwen3_0_6b")
    t = wl.layer(0)
    a, b = DeviceLayer(wl, t), DeviceLayer(wl, t)
    out_a, out_b = out_tensor(wl), out_tensor(wl)
    binding.forge_paged_append_gqa_decode(a.q, a.k_new, a.v_new, a.k_cache, a.v_cache, a.tables, a.lens, wl.scale,
                                          out_a)
    binding.forge_paged_qk_append_gqa_decode(b.q, b.k_new, b.v_new, b.k_cache, b.v_cache, b.tables, b.lens,
                                             wl.scale, out_b)
    assert torch.equal(out_a, out_b)
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))


def test_position_past_the_table_skips_rotation_and_is_flagged():
    wl = W.make_workload("tiny")
    t = wl.layer(0)
    qw, kw = wl.qk_norm_weights(0)
    # a table too short for every sequence: rotation skipped everywhere, norm still applied
    _, _, ref_norm_only = _reference(wl, t, qw, kw, False)
    assert binding.forge_paged_get_device_error() == 0
    d, out = _run(wl, t, qw, kw, True, "f32", rows=2)
    assert binding.forge_paged_get_device_error() == 5
    assert max_abs_err(out, ref_norm_only) <= TOL["f32"]
