"""Worst case of the decode's output precision, on the GPU against the oracle.

The values come from workloads.rounding_stress_values.  Every softmax weight
but one per block sits just above 0.5, where rounding it to bf16 would drop
about 0.26 % of it, and always in the same direction.  Every V value has
magnitude in [7, 8), so the outputs are near +-7.5, where a bf16 output's own
rounding already takes up to 2^-6 = 0.015625 of the 1.6e-2 bound.  Contexts
are long (up to 8192 tokens), so sequences span several splits and the split
merge is exercised too.  With the weights entering P V at about 16 bits, the
fp32 output stays near 1e-5 of exact and the bf16 output within its rounding.
A weight rounded to bf16 once would add about 0.017 and break the bound.

Each case prints its measured max-abs error (run pytest with -s to see it).
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, DeviceLayer, assert_device_clean, max_abs_err, oracle_appended, oracle_decode, out_tensor
from paged_kv_gqa_06_gb300 import binding
from paged_kv_gqa_06_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("decode_kernel")]

LENS = (8192, 8000, 3000, 1100)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


_cache = {}


def _stress(G, D):
    key = (G, D)
    if key not in _cache:
        Hkv = 8 if G == 4 else 2
        spec = W.custom_spec(f"stress_g{G}_d{D}", B=len(LENS), Hq=G * Hkv, Hkv=Hkv, D=D, fixed_lens=LENS,
                             free_frac=0.1, seed=900 + 10 * G + D, values="rounding_stress")
        wl = W.make_workload(spec)
        t = wl.layer(0)
        kc, vc = oracle_appended(wl, t)
        _cache[key] = (wl, t, oracle_decode(wl, t, kc, vc))
    return _cache[key]


def test_stress_outputs_are_large():
    """The case is what it claims: outputs near 7.5 in magnitude."""
    for G in (4, 8):
        ref = _stress(G, 128)[2]
        assert np.abs(ref).min() > 7.0 and np.abs(ref).max() < 8.0


@pytest.mark.parametrize("G,D", [(4, 128), (1, 128), (2, 128), (8, 128), (4, 64), (8, 64)])
@pytest.mark.parametrize("split_tokens", [None, 128])
def test_decode_rounding_stress(G, D, split_tokens, decode_kernel):
    wl, t, ref = _stress(G, D)
    d = DeviceLayer(wl, t)
    d.append()
    for od in ("f32", "bf16"):
        out = out_tensor(wl, od)
        d.decode(out, split_tokens=split_tokens)
        err = max_abs_err(out, ref)
        print(f"rounding stress G={G} D={D} split={split_tokens} kernel={decode_kernel} out={od}: "
              f"max-abs error {err:.3e} (bound {TOL[od]})")
        assert err <= TOL[od], f"{od}: {err}"
        if od == "f32":
            assert err <= 1e-4, f"weights lost precision: {err}"
    assert_device_clean()


def test_fused_path_rounding_stress(decode_kernel):
    """The benchmark's entry point (append fused into the decode) on the same case."""
    wl, t, ref = _stress(4, 128)
    d = DeviceLayer(wl, t)
    out = out_tensor(wl, "bf16")
    binding.forge_paged_append_gqa_decode(d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.tables, d.lens,
                                          wl.scale, out)
    err = max_abs_err(out, ref)
    print(f"rounding stress fused kernel={decode_kernel} out=bf16: max-abs error {err:.3e}")
    assert err <= TOL["bf16"]
    assert_device_clean()
