"""Helpers for the GPU parity tests: move generator arrays to the device and
compare device results with the CPU oracle."""
import numpy as np
import torch

import oracle
from paged_kv_gqa_06_gb300 import binding
from paged_kv_gqa_06_gb300 import workloads as W

TOL = {"f32": 2e-3, "bf16": 1.6e-2}   # max-abs error bound against the fp64 oracle
DEV = "cuda:0"


def bf16_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)


def bits_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def out_tensor(wl, out_dtype=None):
    dt = torch.float32 if (out_dtype or wl.spec.out_dtype) == "f32" else torch.bfloat16
    return torch.full((wl.B, wl.Hq, wl.D), float("nan"), dtype=dt, device=DEV)


class DeviceLayer:
    """One layer's inputs on the GPU (caches in their pre-append state)."""

    def __init__(self, wl, t):
        self.wl = wl
        self.q = bf16_dev(t["q"])
        self.k_new = bf16_dev(t["k_new"])
        self.v_new = bf16_dev(t["v_new"])
        self.k_cache = bf16_dev(t["k_cache"])
        self.v_cache = bf16_dev(t["v_cache"])
        self.slots = torch.from_numpy(wl.slot_mapping).to(DEV)
        self.tables = torch.from_numpy(wl.block_tables).to(DEV)
        self.lens = torch.from_numpy(wl.context_lens).to(DEV)

    def append(self):
        binding.forge_paged_kv_append(self.k_new, self.v_new, self.slots, self.k_cache, self.v_cache)

    def decode(self, out, split_tokens=None):
        if split_tokens is None:
            return binding.forge_paged_gqa_decode(self.q, self.k_cache, self.v_cache, self.tables, self.lens,
                                                  self.wl.scale, out)
        nbytes = binding.forge_paged_gqa_decode_workspace_bytes(self.wl.B, self.wl.Hq, self.wl.Hkv, self.wl.D,
                                                                self.wl.MB, split_tokens)
        ws = torch.zeros(max(nbytes, 1), dtype=torch.uint8, device=DEV)
        return binding.forge_paged_gqa_decode_ex(self.q, self.k_cache, self.v_cache, self.tables, self.lens,
                                                 self.wl.scale, out, ws, split_tokens)


def oracle_appended(wl, t):
    kc, vc = t["k_cache"].copy(), t["v_cache"].copy()
    oracle.paged_kv_append(t["k_new"], t["v_new"], wl.slot_mapping, kc, vc)
    return kc, vc


def oracle_decode(wl, t, kc, vc, **kw):
    return oracle.paged_gqa_decode(t["q"], kc, vc, kw.get("tables", wl.block_tables),
                                   kw.get("lens", wl.context_lens), kw.get("scale", wl.scale))


def max_abs_err(out: torch.Tensor, ref: np.ndarray) -> float:
    got = out.detach().double().cpu().numpy()
    assert np.all(np.isfinite(got)), "non-finite output"
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


def assert_device_clean():
    code = binding.forge_paged_get_device_error()
    assert code == 0, f"device error: {binding.DEVICE_ERRORS.get(code, code)}"
