"""forge_paged_append_gqa_decode: append + decode in one launch, against the
oracle's append followed by the oracle's decode."""
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


def _fused(d, out):
    return binding.forge_paged_append_gqa_decode(d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.tables, d.lens,
                                                 d.wl.scale, out)


@pytest.mark.parametrize("name,out_dtype", [("tiny", "f32"), ("qwen3_0_6b", "bf16"), ("qwen3_4b", "bf16"),
                                            ("skewed", "f32"), ("skewed", "bf16")])
def test_fused_matches_append_then_decode(name, out_dtype):
    wl = W.make_workload(name)
    t = wl.layer(0)
    kc_ref, vc_ref = oracle_appended(wl, t)
    d = DeviceLayer(wl, t)
    out = out_tensor(wl, out_dtype)
    _fused(d, out)
    assert np.array_equal(bits_host(d.k_cache), kc_ref)      # the new rows landed in their slots, nothing else
    assert np.array_equal(bits_host(d.v_cache), vc_ref)
    err = max_abs_err(out, oracle_decode(wl, t, kc_ref, vc_ref))
    assert err <= TOL[out_dtype], f"{name}/{out_dtype}: {err}"
    assert_device_clean()


def test_fused_ragged_lengths_block_crossing_and_empty_rows():
    lens = (1, 15, 16, 17, 31, 32, 33, 100, 255, 256, 257, 700, 0)
    spec = W.custom_spec("fused_ragged", B=len(lens), Hq=32, Hkv=8, D=128, fixed_lens=lens, free_frac=0.2, seed=77)
    wl = W.make_workload(spec)
    t = wl.layer(0)
    kc_ref, vc_ref = oracle_appended(wl, t)     # slot -1 for the empty row: nothing appended
    d = DeviceLayer(wl, t)
    for out_dtype in ("f32", "bf16"):
        e = DeviceLayer(wl, t)
        out = out_tensor(wl, out_dtype)
        _fused(e, out)
        assert np.array_equal(bits_host(e.k_cache), kc_ref)
        assert np.array_equal(bits_host(e.v_cache), vc_ref)
        err = max_abs_err(out, oracle_decode(wl, t, kc_ref, vc_ref))
        assert err <= TOL[out_dtype], f"{out_dtype}: {err}"
        assert torch.all(out[-1] == 0)
    assert_device_clean()


def test_fused_equals_separate_calls_bit_for_bit():
    wl = W.make_workload("qwen3_4b")
    t = wl.layer(0)
    a, b = DeviceLayer(wl, t), DeviceLayer(wl, t)
    out_a, out_b = out_tensor(wl), out_tensor(wl)
    a.append()
    a.decode(out_a)
    _fused(b, out_b)
    bits = lambda x: x.view(torch.int16)     # the caches hold NaN poison: compare bit patterns
    assert torch.equal(bits(a.k_cache), bits(b.k_cache)) and torch.equal(bits(a.v_cache), bits(b.v_cache))
    assert torch.equal(out_a, out_b)
