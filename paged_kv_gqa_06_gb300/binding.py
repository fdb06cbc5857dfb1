"""ctypes binding of libforge_paged.so: argument marshalling only.

Each function has the name of the C entry point it calls, takes torch CUDA
tensors, builds the ``forge_tensor`` descriptors (data pointer, dtype,
shape, element strides), passes the current torch CUDA stream unless one is
given, and turns a negative status into an exception.  No arithmetic of the
operations happens here, and there is no fallback: if the library is not
built the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libforge_paged.so")

FORGE_BF16, FORGE_F32, FORGE_I32, FORGE_I64 = 1, 2, 3, 4
_DTYPES = {torch.bfloat16: FORGE_BF16, torch.float32: FORGE_F32,
           torch.int32: FORGE_I32, torch.int64: FORGE_I64}

FORGE_OK = 0
STATUS_NAMES = {0: "FORGE_OK", -1: "FORGE_ERR_NULL", -2: "FORGE_ERR_DTYPE", -3: "FORGE_ERR_SHAPE",
                -4: "FORGE_ERR_UNSUPPORTED", -5: "FORGE_ERR_ALIGN", -6: "FORGE_ERR_CUDA",
                -7: "FORGE_ERR_WORKSPACE", -8: "FORGE_ERR_VALUE", -9: "FORGE_ERR_CAPACITY"}
DEVICE_ERRORS = {0: "none", 1: "block id outside the pool", 2: "context length longer than the table row",
                 3: "slot outside the pool", 4: "pipeline wait timed out", 5: "position beyond the rotary table",
                 6: "prefill query_start out of order or longer than the context"}


class ForgeTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class ForgeQKOptions(ctypes.Structure):
    _fields_ = [("q_norm_weight", ctypes.POINTER(ForgeTensor)), ("k_norm_weight", ctypes.POINTER(ForgeTensor)),
                ("norm_eps", ctypes.c_float), ("rope_cos_sin", ctypes.POINTER(ForgeTensor))]


class ForgeBatchReport(ctypes.Structure):
    _fields_ = [("running", ctypes.c_int32), ("waiting", ctypes.c_int32), ("admitted", ctypes.c_int32),
                ("retired", ctypes.c_int32), ("preempted", ctypes.c_int32), ("free_blocks", ctypes.c_int32),
                ("tokens", ctypes.c_int64)]


class ForgeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load (once) and type the C entry points.  Raises if the library is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
                "(the CUDA library is required: there is no CPU path)")
        lib = ctypes.CDLL(path)
        T = ctypes.POINTER(ForgeTensor)
        P = ctypes.c_void_p
        lib.forge_paged_kv_append.argtypes = [T, T, T, T, T, P]
        lib.forge_paged_kv_append.restype = ctypes.c_int
        lib.forge_paged_gqa_decode.argtypes = [T, T, T, T, T, ctypes.c_float, T, P]
        lib.forge_paged_gqa_decode.restype = ctypes.c_int
        lib.forge_paged_gqa_decode_ex.argtypes = [T, T, T, T, T, ctypes.c_float, T, P, ctypes.c_size_t,
                                                  ctypes.c_int, P]
        lib.forge_paged_gqa_decode_ex.restype = ctypes.c_int
        lib.forge_paged_qk_append_gqa_decode.argtypes = [T, T, T, ctypes.POINTER(ForgeQKOptions), T, T, T, T,
                                                         ctypes.c_float, T, P]
        lib.forge_paged_qk_append_gqa_decode.restype = ctypes.c_int
        lib.forge_rope_cos_sin_table.argtypes = [ctypes.c_double, ctypes.c_int, ctypes.c_int,
                                                 ctypes.POINTER(ctypes.c_float)]
        lib.forge_rope_cos_sin_table.restype = ctypes.c_int
        lib.forge_paged_append_gqa_decode.argtypes = [T, T, T, T, T, T, T, ctypes.c_float, T, P]
        lib.forge_paged_append_gqa_decode.restype = ctypes.c_int
        lib.forge_paged_prefill.argtypes = [T, T, T, T, T, T, ctypes.c_float, T, P]
        lib.forge_paged_prefill.restype = ctypes.c_int
        lib.forge_paged_gqa_decode_noalloc.argtypes = [T, T, T, T, T, ctypes.c_float, T, P]
        lib.forge_paged_gqa_decode_noalloc.restype = ctypes.c_int
        lib.forge_paged_gqa_decode_workspace_bytes.argtypes = [ctypes.c_int] * 6
        lib.forge_paged_gqa_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.forge_paged_gqa_decode_plan.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int)] * 2
        lib.forge_paged_gqa_decode_plan.restype = ctypes.c_int
        lib.forge_status_string.argtypes = [ctypes.c_int]
        lib.forge_status_string.restype = ctypes.c_char_p
        lib.forge_paged_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
        lib.forge_paged_get_device_error.restype = ctypes.c_int
        lib.forge_paged_version.argtypes = []
        lib.forge_paged_version.restype = ctypes.c_char_p
        _type_serving(lib)
        _lib = lib
        return lib


_desc_cache: dict = {}
_DESC_CACHE_MAX = 4096


def describe(t: torch.Tensor | None) -> ForgeTensor | None:
    """forge_tensor descriptor of a torch tensor (no copy).

    Descriptors are cached by (address, dtype, shape, strides): a decode loop
    passes the same tensors every step, and filling a ctypes struct costs
    more host time than the lookup.  The C side only reads them.  A tensor
    must be on the current CUDA device (checked when its descriptor is
    made); ValueError otherwise.
    """
    if t is None:
        return None
    key = (t.data_ptr(), t.dtype, t.shape, t.stride())
    d = _desc_cache.get(key)
    if d is not None:
        return d
    if t.dim() > 4:
        raise ValueError("forge tensors have at most 4 dims")
    # The kernels dereference these pointers on the device: a host tensor
    # would be a memory fault there, not an error status, so it stops here.
    if not t.is_cuda:
        raise ValueError(f"forge tensors are CUDA device memory; got a tensor on {t.device}")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensor on {t.device}, but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()}")
    if len(_desc_cache) >= _DESC_CACHE_MAX:
        _desc_cache.clear()
    d = ForgeTensor()
    d.data = t.data_ptr() if t.numel() > 0 else 0
    d.dtype = _DTYPES.get(t.dtype, 0)
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    _desc_cache[key] = d
    return d


def _ref(d):
    return ctypes.byref(d) if d is not None else None


def _stream_ptr(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _raise(status: int, what: str):
    if status != FORGE_OK:
        msg = load_library().forge_status_string(status).decode()
        raise ForgeError(status, f"{what}: {msg}")


def forge_paged_kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, stream=None) -> None:
    """Scatter the new K/V token of every row into its slot (in place)."""
    lib = load_library()
    rc = lib.forge_paged_kv_append(_ref(describe(k_new)), _ref(describe(v_new)), _ref(describe(slot_mapping)),
                                   _ref(describe(k_cache)), _ref(describe(v_cache)), _stream_ptr(stream))
    _raise(rc, "forge_paged_kv_append")


def forge_paged_gqa_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, stream=None):
    """Paged GQA decode into ``out`` (bf16 or fp32 [B, Hq, D]); returns ``out``."""
    lib = load_library()
    rc = lib.forge_paged_gqa_decode(_ref(describe(q)), _ref(describe(k_cache)), _ref(describe(v_cache)),
                                    _ref(describe(block_tables)), _ref(describe(context_lens)),
                                    float(scale), _ref(describe(out)), _stream_ptr(stream))
    _raise(rc, "forge_paged_gqa_decode")
    return out


def forge_paged_append_gqa_decode(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, out,
                                  stream=None):
    """Append each sequence's new K/V at position L-1 and decode, in one launch."""
    lib = load_library()
    rc = lib.forge_paged_append_gqa_decode(_ref(describe(q)), _ref(describe(k_new)), _ref(describe(v_new)),
                                           _ref(describe(k_cache)), _ref(describe(v_cache)),
                                           _ref(describe(block_tables)), _ref(describe(context_lens)),
                                           float(scale), _ref(describe(out)), _stream_ptr(stream))
    _raise(rc, "forge_paged_append_gqa_decode")
    return out


def qk_options(q_norm_weight=None, k_norm_weight=None, norm_eps=1e-6, rope_cos_sin=None) -> ForgeQKOptions:
    """forge_qk_options for forge_paged_qk_append_gqa_decode (tensors may be None)."""
    o = ForgeQKOptions()
    o.norm_eps = float(norm_eps)
    for name, t in (("q_norm_weight", q_norm_weight), ("k_norm_weight", k_norm_weight),
                    ("rope_cos_sin", rope_cos_sin)):
        setattr(o, name, ctypes.pointer(describe(t)) if t is not None else None)
    return o


def forge_paged_qk_append_gqa_decode(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, out,
                                     q_norm_weight=None, k_norm_weight=None, norm_eps=1e-6, rope_cos_sin=None,
                                     stream=None):
    """Append + decode in one launch, with RMSNorm / RoPE on q and the new k first."""
    lib = load_library()
    o = qk_options(q_norm_weight, k_norm_weight, norm_eps, rope_cos_sin)
    rc = lib.forge_paged_qk_append_gqa_decode(_ref(describe(q)), _ref(describe(k_new)), _ref(describe(v_new)),
                                              ctypes.byref(o), _ref(describe(k_cache)), _ref(describe(v_cache)),
                                              _ref(describe(block_tables)), _ref(describe(context_lens)),
                                              float(scale), _ref(describe(out)), _stream_ptr(stream))
    _raise(rc, "forge_paged_qk_append_gqa_decode")
    return out


def forge_rope_cos_sin_table(theta: float, D: int, rows: int) -> torch.Tensor:
    """The rotary cos/sin table [rows, D] (f32, host) built by the library."""
    t = torch.empty(rows, D, dtype=torch.float32)
    rc = load_library().forge_rope_cos_sin_table(float(theta), int(D), int(rows),
                                                 ctypes.cast(t.data_ptr(), ctypes.POINTER(ctypes.c_float)))
    _raise(rc, "forge_rope_cos_sin_table")
    return t


def forge_paged_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale, out, stream=None):
    """Causal prefill of the query rows packed by ``query_start`` into ``out``; returns ``out``."""
    lib = load_library()
    rc = lib.forge_paged_prefill(_ref(describe(q)), _ref(describe(k_cache)), _ref(describe(v_cache)),
                                 _ref(describe(block_tables)), _ref(describe(context_lens)),
                                 _ref(describe(query_start)), float(scale), _ref(describe(out)), _stream_ptr(stream))
    _raise(rc, "forge_paged_prefill")
    return out


def forge_paged_gqa_decode_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale, out, stream=None):
    """Decode for callers that cannot allocate device memory: the split scratch
    is a static array inside the library (see include/forge_paged.h)."""
    lib = load_library()
    rc = lib.forge_paged_gqa_decode_noalloc(_ref(describe(q)), _ref(describe(k_cache)), _ref(describe(v_cache)),
                                            _ref(describe(block_tables)), _ref(describe(context_lens)),
                                            float(scale), _ref(describe(out)), _stream_ptr(stream))
    _raise(rc, "forge_paged_gqa_decode_noalloc")
    return out


def forge_paged_gqa_decode_workspace_bytes(B, Hq, Hkv, D, max_blocks_per_seq, split_tokens=0) -> int:
    return int(load_library().forge_paged_gqa_decode_workspace_bytes(B, Hq, Hkv, D, max_blocks_per_seq,
                                                                      split_tokens))


FORGE_DECODE_TWO_PASS, FORGE_DECODE_ONLINE = 0, 1
DECODE_KERNEL_NAMES = {FORGE_DECODE_TWO_PASS: "two_pass", FORGE_DECODE_ONLINE: "online"}


def forge_paged_gqa_decode_plan(B, Hkv, max_blocks_per_seq, split_tokens=0, num_sms=None):
    """(split length in tokens, kernel name) that decode calls of these sizes
    use; num_sms defaults to the current CUDA device's SM count."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    st, kern = ctypes.c_int(0), ctypes.c_int(0)
    rc = load_library().forge_paged_gqa_decode_plan(B, Hkv, max_blocks_per_seq, split_tokens, num_sms,
                                                    ctypes.byref(st), ctypes.byref(kern))
    _raise(rc, "forge_paged_gqa_decode_plan")
    return st.value, DECODE_KERNEL_NAMES[kern.value]


def forge_paged_gqa_decode_ex(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                              workspace=None, split_tokens=0, stream=None):
    """Decode with caller-owned scratch (a uint8 CUDA tensor) and an explicit split length."""
    lib = load_library()
    ws_ptr = workspace.data_ptr() if workspace is not None and workspace.numel() > 0 else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib.forge_paged_gqa_decode_ex(_ref(describe(q)), _ref(describe(k_cache)), _ref(describe(v_cache)),
                                       _ref(describe(block_tables)), _ref(describe(context_lens)),
                                       float(scale), _ref(describe(out)), ws_ptr, ws_bytes,
                                       int(split_tokens), _stream_ptr(stream))
    _raise(rc, "forge_paged_gqa_decode_ex")
    return out


def forge_paged_get_device_error(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device error code."""
    code = ctypes.c_int(0)
    rc = load_library().forge_paged_get_device_error(_stream_ptr(stream), ctypes.byref(code))
    _raise(rc, "forge_paged_get_device_error")
    return code.value


# ---------------------------------------------------------------- KV block pool and batch driver
# (include/forge_serving.h).  Handles are opaque pointers (Python ints); the
# caller destroys what it creates.

FORGE_BATCH_ADMITTED, FORGE_BATCH_RETIRED, FORGE_BATCH_PREEMPTED = 0, 1, 2


def _type_serving(lib):
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    pi32, pi64 = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
    T = ctypes.POINTER(ForgeTensor)
    sig = {
        "forge_kv_pool_create": ([i32, i32, i32], P),
        "forge_kv_pool_destroy": ([P], None),
        "forge_kv_pool_add": ([P, i64, i32], ctypes.c_int),
        "forge_kv_pool_grow": ([P, i64, pi64], ctypes.c_int),
        "forge_kv_pool_release": ([P, i64], ctypes.c_int),
        "forge_kv_pool_free_blocks": ([P], i32),
        "forge_kv_pool_used_blocks": ([P], i32),
        "forge_kv_pool_sequence": ([P, i64, pi32, pi32, i32, pi32], ctypes.c_int),
        "forge_batch_create": ([P, i32, i32], P),
        "forge_batch_destroy": ([P], None),
        "forge_batch_submit": ([P, i64, i32, i32], ctypes.c_int),
        "forge_batch_step": ([P, ctypes.POINTER(ForgeBatchReport)], ctypes.c_int),
        "forge_batch_rows": ([P, pi64, pi32, pi64, pi32], ctypes.c_int),
        "forge_batch_events": ([P, ctypes.c_int, i32, pi64, pi32, pi32], ctypes.c_int),
        "forge_batch_apply": ([P, T, T, T, P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = args, res


def _np_ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def forge_kv_pool_create(num_blocks: int, block_size: int, max_blocks_per_seq: int) -> int:
    h = load_library().forge_kv_pool_create(num_blocks, block_size, max_blocks_per_seq)
    if not h:
        raise ValueError("forge_kv_pool_create: bad sizes or out of memory")
    return h


def forge_kv_pool_destroy(pool: int) -> None:
    load_library().forge_kv_pool_destroy(pool)


def forge_kv_pool_add(pool: int, seq_id: int, num_tokens: int) -> None:
    _raise(load_library().forge_kv_pool_add(pool, seq_id, num_tokens), "forge_kv_pool_add")


def forge_kv_pool_grow(pool: int, seq_id: int) -> int:
    """Add one token to seq_id; returns its cache slot."""
    slot = ctypes.c_int64(-1)
    _raise(load_library().forge_kv_pool_grow(pool, seq_id, ctypes.byref(slot)), "forge_kv_pool_grow")
    return slot.value


def forge_kv_pool_release(pool: int, seq_id: int) -> None:
    _raise(load_library().forge_kv_pool_release(pool, seq_id), "forge_kv_pool_release")


def forge_kv_pool_free_blocks(pool: int) -> int:
    return load_library().forge_kv_pool_free_blocks(pool)


def forge_kv_pool_used_blocks(pool: int) -> int:
    return load_library().forge_kv_pool_used_blocks(pool)


def forge_kv_pool_sequence(pool: int, seq_id: int):
    """(token count, list of block ids) of seq_id."""
    lib = load_library()
    n, length = ctypes.c_int32(0), ctypes.c_int32(0)
    _raise(lib.forge_kv_pool_sequence(pool, seq_id, ctypes.byref(length), None, 0, ctypes.byref(n)),
           "forge_kv_pool_sequence")
    blocks = np.zeros(max(1, n.value), dtype=np.int32)
    _raise(lib.forge_kv_pool_sequence(pool, seq_id, None, _np_ptr(blocks, ctypes.c_int32), n.value, None),
           "forge_kv_pool_sequence")
    return length.value, blocks[: n.value].tolist()


def forge_batch_create(pool: int, rows: int, token_budget: int) -> int:
    h = load_library().forge_batch_create(pool, rows, token_budget)
    if not h:
        raise ValueError("forge_batch_create: bad arguments or out of memory")
    return h


def forge_batch_destroy(batch: int) -> None:
    load_library().forge_batch_destroy(batch)


def forge_batch_submit(batch: int, seq_id: int, prompt_tokens: int, max_new_tokens: int) -> None:
    _raise(load_library().forge_batch_submit(batch, seq_id, prompt_tokens, max_new_tokens), "forge_batch_submit")


def forge_batch_step(batch: int) -> dict:
    """One host step; returns the forge_batch_report fields as a dict."""
    rep = ForgeBatchReport()
    _raise(load_library().forge_batch_step(batch, ctypes.byref(rep)), "forge_batch_step")
    return {name: getattr(rep, name) for name, _ in ForgeBatchReport._fields_}


def forge_batch_rows(batch: int, rows: int) -> dict:
    """The last step's per-row state as numpy arrays of length ``rows``."""
    out = {"seq_ids": np.zeros(rows, np.int64), "context_lens": np.zeros(rows, np.int32),
           "slots": np.zeros(rows, np.int64), "new_blocks": np.zeros(rows, np.int32)}
    _raise(load_library().forge_batch_rows(batch, _np_ptr(out["seq_ids"], ctypes.c_int64),
                                           _np_ptr(out["context_lens"], ctypes.c_int32),
                                           _np_ptr(out["slots"], ctypes.c_int64),
                                           _np_ptr(out["new_blocks"], ctypes.c_int32)), "forge_batch_rows")
    return out


def forge_batch_events(batch: int, kind: int) -> list:
    """The last step's events of one kind as (seq_id, row, tokens) tuples."""
    lib = load_library()
    n = lib.forge_batch_events(batch, kind, 0, None, None, None)
    _raise(min(n, 0), "forge_batch_events")
    seq, row, tok = np.zeros(max(1, n), np.int64), np.zeros(max(1, n), np.int32), np.zeros(max(1, n), np.int32)
    lib.forge_batch_events(batch, kind, n, _np_ptr(seq, ctypes.c_int64), _np_ptr(row, ctypes.c_int32),
                           _np_ptr(tok, ctypes.c_int32))
    return [(int(seq[i]), int(row[i]), int(tok[i])) for i in range(n)]


def forge_batch_apply(batch: int, block_tables, context_lens, slot_mapping, stream=None) -> None:
    rc = load_library().forge_batch_apply(batch, _ref(describe(block_tables)), _ref(describe(context_lens)),
                                          _ref(describe(slot_mapping)), _stream_ptr(stream))
    _raise(rc, "forge_batch_apply")
