"""The C ABI on a machine without a GPU: the library loads, exports every
entry point include/*.h declares, and rejects bad arguments on the host
before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from paged_kv_gqa_06_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    from paged_kv_gqa_06_gb300 import build
    build.build()
    return binding.load_library()


def _declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"FORGE_API\s+[\w\s\*]*?\b(forge_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    assert len(HEADERS) >= 2
    names = _declared_functions()
    assert len(names) >= 25 and "forge_batch_apply" in names and "forge_paged_gqa_decode" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings_and_version(lib):
    for code in range(-9, 1):
        assert lib.forge_status_string(code)
    assert lib.forge_status_string(-99) == b"unknown forge status"
    assert lib.forge_paged_version() == b"0.1.0"


def test_workspace_bytes_is_host_only(lib):
    f = binding.forge_paged_gqa_decode_workspace_bytes
    r256 = lambda x: (x + 255) // 256 * 256
    assert f(32, 32, 8, 128, 512, 512) == 65536 * 4 + r256(32 * 32 * 16 * 128 * 4) + 32 * 32 * 16 * 2 * 4
    assert f(4, 8, 2, 64, 4, 1024) == 0      # one split: no scratch
    assert f(4, 8, 2, 64, 4, 17) == 0        # invalid split length
    assert f(-1, 8, 2, 64, 4, 0) == 0


def _desc(shape, dtype, data=16, stride=None):
    d = binding.ForgeTensor()
    d.data = data
    d.dtype = dtype
    d.ndim = len(shape)
    st = stride
    if st is None:
        st, acc = [], 1
        for s in reversed(shape):
            st.insert(0, acc)
            acc *= s
    for i, s in enumerate(shape):
        d.shape[i] = s
        d.stride[i] = st[i]
    return d


BF16, F32, I32, I64 = binding.FORGE_BF16, binding.FORGE_F32, binding.FORGE_I32, binding.FORGE_I64


def _decode_args(**over):
    B, Hq, Hkv, D, NB, MB = 2, 8, 2, 64, 8, 4
    a = dict(q=_desc([B, Hq, D], BF16), k=_desc([NB, Hkv, 16, D], BF16), v=_desc([NB, Hkv, 16, D], BF16),
             bt=_desc([B, MB], I32), cl=_desc([B], I32), scale=0.125, out=_desc([B, Hq, D], F32))
    a.update(over)
    return a


def _call_decode(lib, a):
    r = lambda d: ctypes.byref(d) if d is not None else None
    return lib.forge_paged_gqa_decode(r(a["q"]), r(a["k"]), r(a["v"]), r(a["bt"]), r(a["cl"]), a["scale"],
                                      r(a["out"]), None)


@pytest.mark.parametrize("over,status", [
    (dict(q=None), -1),
    (dict(q=_desc([2, 8, 64], F32)), -2),
    (dict(q=_desc([2, 8, 64, 1], BF16)), -3),
    (dict(out=_desc([2, 8, 64], I32)), -2),
    (dict(out=_desc([2, 4, 64], F32)), -3),
    (dict(k=_desc([8, 2, 8, 64], BF16), v=_desc([8, 2, 8, 64], BF16)), -4),     # block size 8
    (dict(q=_desc([2, 8, 96], BF16), k=_desc([8, 2, 16, 96], BF16), v=_desc([8, 2, 16, 96], BF16),
          out=_desc([2, 8, 96], F32)), -4),                                        # D = 96
    (dict(q=_desc([2, 6, 64], BF16), out=_desc([2, 6, 64], F32)), -4),             # Hq % Hkv != 0
    (dict(q=_desc([2, 32, 64], BF16), out=_desc([2, 32, 64], F32)), -4),           # G = 16
    (dict(bt=_desc([3, 4], I32)), -3),
    (dict(cl=_desc([2], I64)), -2),
    (dict(scale=float("nan")), -8),
    (dict(q=_desc([2, 8, 64], BF16, data=8)), -5),                                 # misaligned
    (dict(q=_desc([2, 8, 64], BF16, stride=[512, 60, 1])), -5),                    # stride not x8
    (dict(q=_desc([2, 8, 64], BF16, stride=[1, 128, 2])), -3),                     # inner stride
    (dict(k=_desc([8, 2, 16, 64], BF16, stride=[4096, 2048, 65, 1])), -3),        # tile not contiguous
    (dict(v=_desc([8, 4, 16, 64], BF16)), -3),
])
def test_decode_rejects_bad_arguments(lib, over, status):
    assert _call_decode(lib, _decode_args(**over)) == status


def test_decode_with_valid_arguments_reaches_cuda(lib):
    rc = _call_decode(lib, _decode_args())
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the GPU tests cover real calls")
    assert rc == -6        # no device here: the first CUDA call fails cleanly


def test_empty_batch_is_a_no_op(lib):
    a = _decode_args(q=_desc([0, 8, 64], BF16, data=0), bt=_desc([0, 4], I32, data=0), cl=_desc([0], I32, data=0),
                     out=_desc([0, 8, 64], F32, data=0))
    assert _call_decode(lib, a) == 0


def _call_append(lib, kn, vn, sm, kc, vc):
    r = lambda d: ctypes.byref(d) if d is not None else None
    return lib.forge_paged_kv_append(r(kn), r(vn), r(sm), r(kc), r(vc), None)


@pytest.mark.parametrize("over,status", [
    (dict(kn=None), -1),
    (dict(sm=_desc([2], I32)), -2),
    (dict(sm=_desc([3], I64)), -3),
    (dict(kn=_desc([2, 2, 64], F32)), -2),
    (dict(kc=_desc([8, 2, 32, 64], BF16)), -4),
    (dict(kn=_desc([2, 2, 64], BF16, data=4)), -5),
    (dict(vn=_desc([2, 3, 64], BF16)), -3),
])
def test_append_rejects_bad_arguments(lib, over, status):
    a = dict(kn=_desc([2, 2, 64], BF16), vn=_desc([2, 2, 64], BF16), sm=_desc([2], I64),
             kc=_desc([8, 2, 16, 64], BF16), vc=_desc([8, 2, 16, 64], BF16))
    a.update(over)
    assert _call_append(lib, a["kn"], a["vn"], a["sm"], a["kc"], a["vc"]) == status


def test_python_binding_raises_on_bad_status(lib):
    with pytest.raises(binding.ForgeError) as e:
        binding._raise(-4, "forge_paged_gqa_decode")
    assert e.value.status == -4
    assert "forge_paged_gqa_decode" in str(e.value)
    binding._raise(binding.FORGE_OK, "no error")  # no exception


def test_python_binding_refuses_host_tensors(lib):
    # a host pointer would reach the kernels as a device address: refused
    # before the C call
    q = torch.zeros(2, 8, 64, dtype=torch.bfloat16)
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16)
    out = torch.zeros(2, 8, 64)
    with pytest.raises(ValueError, match="CUDA device memory"):
        binding.forge_paged_gqa_decode(q, kc, kc, torch.zeros(2, 4, dtype=torch.int32),
                                       torch.zeros(2, dtype=torch.int32), 0.1, out, stream=0)


def test_fused_entry_rejects_bad_new_rows(lib):
    a = _decode_args()
    r = lambda d: ctypes.byref(d) if d is not None else None
    good = _desc([2, 2, 64], BF16)

    def call(kn, vn):
        return lib.forge_paged_append_gqa_decode(r(a["q"]), r(kn), r(vn), r(a["k"]), r(a["v"]), r(a["bt"]),
                                                 r(a["cl"]), a["scale"], r(a["out"]), None)
    assert call(None, good) == -1
    assert call(_desc([2, 2, 64], F32), good) == -2
    assert call(good, _desc([2, 3, 64], BF16)) == -3
    assert call(_desc([3, 2, 64], BF16), _desc([3, 2, 64], BF16)) == -3
    assert call(_desc([2, 2, 64], BF16, data=8), good) == -5


def test_rope_table_matches_its_definition(lib):
    for theta, D, rows in [(1e6, 128, 300), (1e4, 64, 17), (10.0, 2, 5)]:
        t = binding.forge_rope_cos_sin_table(theta, D, rows).numpy()
        r = np.arange(rows, dtype=np.float64)[:, None]
        a = r * theta ** (-2.0 * np.arange(D // 2) / D)
        np.testing.assert_array_equal(t[:, : D // 2], np.cos(a).astype(np.float32))
        np.testing.assert_array_equal(t[:, D // 2:], np.sin(a).astype(np.float32))
    with pytest.raises(binding.ForgeError):
        binding.forge_rope_cos_sin_table(1e4, 63, 4)


def test_qk_options_are_validated(lib):
    a = _decode_args()
    r = lambda d: ctypes.byref(d) if d is not None else None
    kn = _desc([2, 2, 64], BF16)

    def call(**kw):
        o = binding.ForgeQKOptions()
        o.norm_eps = kw.get("eps", 1e-6)
        for name in ("q_norm_weight", "k_norm_weight", "rope_cos_sin"):
            if name in kw:
                setattr(o, name, ctypes.pointer(kw[name]))
        return lib.forge_paged_qk_append_gqa_decode(r(a["q"]), r(kn), r(kn), ctypes.byref(o), r(a["k"]), r(a["v"]),
                                                    r(a["bt"]), r(a["cl"]), a["scale"], r(a["out"]), None)
    assert call(q_norm_weight=_desc([64], F32)) == -2
    assert call(k_norm_weight=_desc([32], BF16)) == -3
    assert call(q_norm_weight=_desc([64], BF16), eps=float("nan")) == -8
    assert call(rope_cos_sin=_desc([10, 64], BF16)) == -2
    assert call(rope_cos_sin=_desc([10, 32], F32)) == -3
    assert call(rope_cos_sin=_desc([10, 64], F32, stride=[128, 1])) == -3
    expect = -6 if not torch.cuda.is_available() else None
    if expect is not None:   # valid options reach CUDA (absent here)
        assert call(q_norm_weight=_desc([64], BF16), k_norm_weight=_desc([64], BF16),
                    rope_cos_sin=_desc([10, 64], F32)) == -6


def _prefill_args(**over):
    a = dict(q=_desc([10, 8, 64], BF16), k=_desc([8, 2, 16, 64], BF16), v=_desc([8, 2, 16, 64], BF16),
             bt=_desc([2, 4], I32), cl=_desc([2], I32), qs=_desc([3], I32), scale=0.125,
             out=_desc([10, 8, 64], F32))
    a.update(over)
    return a


def _call_prefill(lib, a):
    r = lambda d: ctypes.byref(d) if d is not None else None
    return lib.forge_paged_prefill(r(a["q"]), r(a["k"]), r(a["v"]), r(a["bt"]), r(a["cl"]), r(a["qs"]),
                                   a["scale"], r(a["out"]), None)


@pytest.mark.parametrize("over,status", [
    (dict(qs=None), -1),
    (dict(qs=_desc([3], I64)), -2),
    (dict(qs=_desc([2], I32)), -3),                                                 # not B + 1 entries
    (dict(out=_desc([9, 8, 64], F32)), -3),                                         # not T rows
    (dict(bt=_desc([3, 4], I32)), -3),
    (dict(q=_desc([10, 8, 96], BF16), k=_desc([8, 2, 16, 96], BF16), v=_desc([8, 2, 16, 96], BF16),
          out=_desc([10, 8, 96], F32)), -4),                                        # D = 96
    (dict(q=_desc([10, 32, 64], BF16), out=_desc([10, 32, 64], F32)), -4),         # G = 16
    (dict(scale=float("inf")), -8),
    (dict(q=_desc([10, 8, 64], BF16, data=8)), -5),
    (dict(qs=_desc([3], I32, stride=[2])), -3),
])
def test_prefill_rejects_bad_arguments(lib, over, status):
    assert _call_prefill(lib, _prefill_args(**over)) == status


def test_prefill_empty_is_a_no_op(lib):
    a = _prefill_args(q=_desc([0, 8, 64], BF16, data=0), out=_desc([0, 8, 64], F32, data=0))
    assert _call_prefill(lib, a) == 0


# (B, Hkv, table width in blocks) of the Qwen3-4B / 36-layer / skewed / Qwen3-0.6B decode
# workloads, and the plan the policy gives on 152 SMs: 1024-token splits while
# B * Hkv * ceil(MB * 16 / split) >= 4 * 152, else the longest shorter split that gets
# there; the single-pass kernel either way.
@pytest.mark.parametrize("B,Hkv,MB,want", [
    (32, 8, 498, (1024, "online")),      # 256 * 8 = 2048 CTAs at 1024 tokens
    (64, 8, 457, (1024, "online")),      # 512 * 8
    (4, 8, 2048, (1024, "online")),      # 32 * 32 = 1024
    (8, 8, 116, (128, "online")),        # 64 * 2 < 608, ... 64 * 15 = 960 at 128 tokens
    (16, 8, 128, (256, "online")),       # 128 * 8 = 1024 at 256 tokens
    (32, 8, 64, (256, "online")),        # 256 * 2 = 512 < 608 at 512 tokens
    (0, 8, 10, (64, "online")),          # nothing to run: the shortest split
])
def test_decode_plan_policy(lib, monkeypatch, B, Hkv, MB, want):
    monkeypatch.delenv("FORGE_DECODE_KERNEL", raising=False)
    assert binding.forge_paged_gqa_decode_plan(B, Hkv, MB, 0, num_sms=152) == want


def test_decode_plan_explicit_split_and_override(lib, monkeypatch):
    monkeypatch.delenv("FORGE_DECODE_KERNEL", raising=False)
    assert binding.forge_paged_gqa_decode_plan(32, 8, 498, 512, num_sms=152) == (512, "online")
    assert binding.forge_paged_gqa_decode_plan(32, 8, 498, 496, num_sms=152) == (496, "online")
    monkeypatch.setenv("FORGE_DECODE_KERNEL", "two_pass")   # automatic two-pass splits stop at 512
    assert binding.forge_paged_gqa_decode_plan(32, 8, 498, 0, num_sms=152) == (512, "two_pass")
    assert binding.forge_paged_gqa_decode_plan(32, 8, 498, 1024, num_sms=152) == (1024, "two_pass")
    monkeypatch.setenv("FORGE_DECODE_KERNEL", "online")
    assert binding.forge_paged_gqa_decode_plan(8, 8, 116, 0, num_sms=152) == (128, "online")


@pytest.mark.parametrize("args,status", [((32, 8, 498, 0, 0), -8), ((32, 8, 498, 17, 152), -8),
                                         ((32, 8, 498, 2048, 152), -8), ((-1, 8, 498, 0, 152), -3),
                                         ((32, 0, 498, 0, 152), -3)])
def test_decode_plan_rejects_bad_arguments(lib, args, status):
    st, kern = ctypes.c_int(0), ctypes.c_int(0)
    assert lib.forge_paged_gqa_decode_plan(*args, ctypes.byref(st), ctypes.byref(kern)) == status
