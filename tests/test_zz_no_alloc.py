"""forge_paged_gqa_decode_noalloc: the decode for callers that cannot allocate.

Such callers -- a process whose device memory was fixed at start-up (a
serving loop that gave the rest to its KV-block pool), or code running under
a memory manager of its own that forbids allocations it did not make -- call
this entry point instead of forge_paged_gqa_decode, which may allocate its
split scratch on first use.
These tests call it through the C ABI twice in a row (the static scratch keeps
the first call's contents) and check both results against the regular entry
point's within the parity tolerance, with shapes alternating over the one
scratch, and with the device's free memory unchanged across calls.  They live
in a file of their own that pytest collects last, and build their own inputs
so they also pass alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import TOL, DeviceLayer, max_abs_err, oracle_appended, oracle_decode, out_tensor
from paged_kv_gqa_06_gb300 import binding
from paged_kv_gqa_06_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("decode_kernel")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


def _call_noalloc(lib, d, out):
    descs = [binding.describe(t) for t in (d.q, d.k_cache, d.v_cache, d.tables, d.lens, out)]
    rc = lib.forge_paged_gqa_decode_noalloc(*(ctypes.byref(x) for x in descs[:5]), ctypes.c_float(d.wl.scale),
                                            ctypes.byref(descs[5]), torch.cuda.current_stream().cuda_stream)
    return rc


@pytest.mark.parametrize("name", ["qwen3_4b", "skewed"])
def test_noalloc_matches_regular_decode_twice(name):
    lib = binding.load_library()
    wl = W.make_workload(name)
    t = wl.layer(0)
    d = DeviceLayer(wl, t)
    d.append()
    ref = out_tensor(wl)
    d.decode(ref)
    tol = TOL[wl.spec.out_dtype]
    first = None
    for call in range(2):
        out = out_tensor(wl)
        assert _call_noalloc(lib, d, out) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        diff = (out.float() - ref.float()).abs().max().item()
        assert diff <= tol, f"call {call}: max-abs difference {diff} from forge_paged_gqa_decode"
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out, first)     # same inputs, same scratch reuse: same bits
    assert binding.forge_paged_get_device_error() == 0
    # and it is the attention the oracle defines
    kc_ref, vc_ref = oracle_appended(wl, t)
    assert max_abs_err(first, oracle_decode(wl, t, kc_ref, vc_ref)) <= tol


def test_noalloc_alternating_shapes_share_the_scratch():
    """Calls of different shapes in turn reuse the one static scratch."""
    lib = binding.load_library()
    cases = {}
    for name in ("skewed", "qwen3_0_6b", "qwen3_4b"):
        wl = W.make_workload(name)
        t = wl.layer(0)
        d = DeviceLayer(wl, t)
        d.append()
        ref = out_tensor(wl)
        d.decode(ref)
        cases[name] = (wl, d, ref)
    for name in ("qwen3_4b", "skewed", "qwen3_0_6b", "qwen3_4b", "skewed"):
        wl, d, ref = cases[name]
        out = out_tensor(wl)
        assert _call_noalloc(lib, d, out) == 0
        torch.cuda.synchronize()
        diff = (out.float() - ref.float()).abs().max().item()
        assert diff <= TOL[wl.spec.out_dtype], f"{name}: {diff}"


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = binding.load_library()
    spec = W.custom_spec("too_big", B=64, Hq=64, Hkv=8, D=128, fixed_lens=(16384,) * 64, seed=3)
    wl = W.make_workload(spec)
    B, Hq, D, MB = wl.B, wl.Hq, wl.D, wl.MB
    # descriptors only: the call must refuse on the host before touching these buffers
    q = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.empty(16, wl.Hkv, 16, D, dtype=torch.bfloat16, device="cuda")
    tables = torch.zeros(B, MB, dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    descs = [binding.describe(x) for x in (q, kc, kc, tables, lens, out)]
    rc = lib.forge_paged_gqa_decode_noalloc(*(ctypes.byref(x) for x in descs[:5]), ctypes.c_float(0.1),
                                            ctypes.byref(descs[5]), torch.cuda.current_stream().cuda_stream)
    assert rc == -7   # FORGE_ERR_WORKSPACE: needs more than the static scratch holds


def test_noalloc_calls_leave_device_free_memory_unchanged():
    """After one warm-up call (which may load the kernel's code), further
    calls allocate nothing: the device's free memory is the same after them.
    The output tensors are made before the measurement, and nothing else in
    this process allocates in between."""
    lib = binding.load_library()
    wl = W.make_workload("skewed")
    t = wl.layer(0)
    d = DeviceLayer(wl, t)
    d.append()
    outs = [out_tensor(wl) for _ in range(4)]
    assert _call_noalloc(lib, d, outs[0]) == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for out in outs[1:]:
        assert _call_noalloc(lib, d, out) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert binding.forge_paged_get_device_error() == 0
    for out in outs[1:]:
        assert torch.equal(out, outs[0])
