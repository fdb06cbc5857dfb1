"""CPU oracle for paged-KV append, paged GQA decode and paged prefill.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs may import this package.  It
shares no code with the CUDA library and never imports it.

The arithmetic lives in ``forge_oracle.c`` (fp64, written the plain way:
gather the sequence's K/V into contiguous rows, dot products, max-subtracted
softmax with libm ``exp``, weighted sum).  This module only compiles that file
with gcc and marshals numpy arrays into it.

Citations (page title, section):
  * forge-engine README, "What it implements" (KV cache row): the cache is a
    paged pool of fixed-size blocks.
  * "Make the Engine Talk", 1.2 "The loop behind it": one new token per decode
    pass; the cache grows by that token.  1.3: attention is grouped-query
    attention.

Pins: every function here is pinned by CPU tests against brute-force dense
attention, torch's scaled_dot_product_attention in fp64, closed forms,
hand-derived examples and invariants (``tests/test_oracle_pins.py``,
``tests/test_oracle_qk_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "forge_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

STATUS = {
    0: "ok",
    -1: "bad argument",
    -2: "block table entry outside the pool",
    -3: "context length longer than the block table row",
    -4: "slot outside the pool",
    -5: "out of memory",
}


def build(force: bool = False) -> str:
    """Compile ``forge_oracle.c`` into ``oracle/_build/liboracle.so`` with gcc.

    ``-ffp-contract=off`` keeps a*b+c unfused so x86 and Arm hosts round the
    same way.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_paged_kv_append.argtypes = [P, P, P, P, P, i, i, i, i, i]
            lib.oracle_paged_kv_append.restype = i
            lib.oracle_paged_gqa_decode.argtypes = [P, P, P, P, P, ctypes.c_double, P,
                                                    i, i, i, i, i, i, i, i]
            lib.oracle_paged_gqa_decode.restype = i
            lib.oracle_rmsnorm.argtypes = [P, P, ctypes.c_double, P, i, i]
            lib.oracle_rmsnorm.restype = None
            lib.oracle_rope.argtypes = [P, P, ctypes.c_double, i, i]
            lib.oracle_rope.restype = None
            lib.oracle_paged_prefill.argtypes = [P, P, P, P, P, P, ctypes.c_double, P,
                                                 i, i, i, i, i, i, i, i]
            lib.oracle_paged_prefill.restype = i
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: {STATUS.get(rc, rc)}")


def host_cores() -> int:
    """Threads the oracle uses by default: the cores this process may run on."""
    return len(os.sched_getaffinity(0))


def paged_kv_append(k_new, v_new, slot_mapping, k_cache, v_cache) -> None:
    """Scatter each row's new K/V token into its cache slot, in place.

    k_new, v_new: uint16 (bf16 bits) [B, Hkv, D]; slot_mapping: int64 [B]
    (negative = skip); k_cache, v_cache: uint16 [NB, Hkv, BS, D], C-contiguous,
    modified in place.
    """
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    for c in (k_cache, v_cache):
        if c.dtype != np.uint16 or not c.flags["C_CONTIGUOUS"]:
            raise ValueError("caches must be C-contiguous uint16 arrays")
    B, Hkv, D = k_new.shape
    NB, Hkv2, BS, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or v_cache.shape != k_cache.shape or v_new.shape != k_new.shape:
        raise ValueError("shape mismatch")
    rc = _load().oracle_paged_kv_append(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                        _ptr(k_cache), _ptr(v_cache), B, Hkv, D, NB, BS)
    _check(rc, "append")


def paged_gqa_decode(q, k_cache, v_cache, block_tables, context_lens, scale,
                     nthreads: int | None = None) -> np.ndarray:
    """fp64 decode attention; returns out [B, Hq, D] float64.

    q: uint16 [B, Hq, D]; k_cache, v_cache: uint16 [NB, Hkv, BS, D];
    block_tables: int32 [B, MB]; context_lens: int32 [B]; scale: float.
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint16)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint16)
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.ndim != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables / context_lens shape mismatch")
    MB = block_tables.shape[1]
    out = np.zeros((B, Hq, D), dtype=np.float64)
    if nthreads is None:
        nthreads = host_cores()
    rc = _load().oracle_paged_gqa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                         _ptr(block_tables), _ptr(context_lens),
                                         float(scale), _ptr(out),
                                         B, Hq, Hkv, D, NB, BS, MB, int(nthreads))
    _check(rc, "decode")
    return out


def paged_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale,
                  nthreads: int | None = None) -> np.ndarray:
    """fp64 causal prefill over the paged cache; returns out [T, Hq, D] float64.

    q: uint16 [T, Hq, D] packed by query_start (int32 [B+1], starting at 0);
    sequence b's query tokens sit at the last n_b positions of its
    context_lens[b] tokens.  Other arguments as in paged_gqa_decode.
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint16)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint16)
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    query_start = np.ascontiguousarray(query_start, dtype=np.int32)
    T, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_cache.shape
    B = context_lens.shape[0]
    if D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.ndim != 2 or block_tables.shape[0] != B or query_start.shape != (B + 1,):
        raise ValueError("block_tables / query_start shape mismatch")
    if B and int(query_start[-1]) != T:
        raise ValueError("query_start[B] must equal the number of query tokens")
    out = np.zeros((T, Hq, D), dtype=np.float64)
    if nthreads is None:
        nthreads = host_cores()
    rc = _load().oracle_paged_prefill(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                      _ptr(context_lens), _ptr(query_start), float(scale), _ptr(out),
                                      B, Hq, Hkv, D, NB, BS, block_tables.shape[1], int(nthreads))
    _check(rc, "prefill")
    return out


def rmsnorm(x, weight, eps) -> np.ndarray:
    """fp64 RMSNorm of each last-axis row of x (bf16 bits); weight [D] bf16 bits or None."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    D = x.shape[-1]
    rows = x.size // D
    y = np.empty(x.shape, dtype=np.float64)
    w = None if weight is None else np.ascontiguousarray(weight, dtype=np.uint16)
    _load().oracle_rmsnorm(_ptr(x), None if w is None else _ptr(w), float(eps), _ptr(y), rows, D)
    return y


def rope(x, positions, theta) -> np.ndarray:
    """Rotate-half rotary embedding of fp64 rows x [..., D] at per-row positions
    (broadcast over the rows of each leading index); returns a new array."""
    x = np.array(x, dtype=np.float64, order="C", copy=True)
    D = x.shape[-1]
    rows = x.size // D
    pos = np.ascontiguousarray(np.broadcast_to(np.asarray(positions, dtype=np.int64).reshape(
        np.asarray(positions).shape + (1,) * (x.ndim - 1 - np.asarray(positions).ndim)), x.shape[:-1]),
        dtype=np.int64).reshape(rows)
    _load().oracle_rope(_ptr(x), _ptr(pos), float(theta), rows, D)
    return x


def bf16_round(x) -> np.ndarray:
    """Round fp64 values straight to bf16 (nearest, ties to even) and return the
    bf16 bits.  Rounding via float32 first could round twice; this takes the
    8-bit quantum of each value's binade directly.  Normal-range values only."""
    x = np.asarray(x, dtype=np.float64)
    b = x.view(np.uint64)
    sign = (b >> np.uint64(63)).astype(np.uint16)
    a = np.abs(x)
    out = np.zeros(x.shape, dtype=np.uint16)
    nz = a > 0
    m, e = np.frexp(a[nz])                    # a = m * 2^e, m in [0.5, 1)
    # bf16 normal: 8 significant bits -> quantum 2^(e-8) for |x| in [2^(e-1), 2^e)
    q = np.ldexp(np.ones_like(m), e - 8)
    r = np.rint(a[nz] / q) * q                # rint: ties to even
    out[nz] = (np.asarray(r, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    return out | (sign << np.uint16(15))
