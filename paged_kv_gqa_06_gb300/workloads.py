"""Seeded synthetic inputs for paged-KV append + paged GQA decode.

This module is the one thing the CUDA path and the CPU oracle share: it makes
the inputs (numpy arrays of bf16 bit patterns and int32/int64 index arrays)
and holds none of the method's arithmetic -- no dot products, no softmax, no
address translation of cache rows.  It plays the host-side block allocator of
a serving engine (forge-engine README, "What it implements": a paged block
allocator owns the KV pool) so that each sequence owns a list of physical
blocks and the new token of this step has a slot.

Shapes follow the attention layers of the two model sizes the pages name
(Qwen3-4B in the forge-engine README, Qwen3-0.6B in "Make the Engine Talk"),
plus a tiny case, a skewed long-context case and a 36-layer batch step.

Recipe (every config):
  * context_lens: the lengths AFTER this step's append; the appended token
    sits at position L-1.
  * Blocks: BS = 16 tokens.  The pool holds NB blocks.  Physical ids are a
    seeded random permutation of range(NB), handed out to sequences in order;
    ids the permutation leaves over are free blocks scattered through the
    pool.  Unused block-table entries are -1.
  * Values: float32 N(0, 1) draws from numpy's PCG64 (one stream per
    4 Mi-element chunk, seeded by (seed, layer, tensor, chunk)), rounded to
    bf16 with round-to-nearest-even.  Config "qwen3_4b" doubles K (an exact power-of-two
    scale) so that logits reach about +-8.
  * Values "rounding_stress" (tests only): structured q/K/V for the worst
    case of the output precision -- see rounding_stress_values.
  * Poison: every cache slot that holds no token before the append -- free
    blocks, the tail of each sequence's last block, and the append target
    itself -- is bf16 NaN (0x7FC0), so a kernel that reads a slot it should
    not read, or skips the append, produces NaN.
"""
from __future__ import annotations

import dataclasses
import math
import os

import numpy as np

BF16_NAN = np.uint16(0x7FC0)
BLOCK_SIZE = 16


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits.

    Inputs are finite normal draws here, so NaN/Inf handling is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_CHUNK = 1 << 22
_pool = None


def _threads():
    global _pool
    if _pool is None:
        from concurrent.futures import ThreadPoolExecutor
        _pool = ThreadPoolExecutor(max_workers=max(1, min(16, len(os.sched_getaffinity(0)))))
    return _pool


def _normal_bf16(key, shape, mul: float = 1.0) -> np.ndarray:
    """bf16 bits of mul * N(0,1) (mul a power of two, so the scaling is exact).

    Chunk c of the array draws from its own PCG64 stream seeded by
    (*key, c), so the values do not depend on how many threads fill it.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)

    def fill(c):
        s, e = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        x = np.random.default_rng([*key, c]).standard_normal(e - s, dtype=np.float32)
        if mul != 1.0:
            x *= np.float32(mul)
        out[s:e] = f32_to_bf16_bits(x)

    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        list(_threads().map(fill, range(nchunks)))
    return out.reshape(shape)


@dataclasses.dataclass
class Spec:
    """Shape recipe for one named workload."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    out_dtype: str            # "f32" or "bf16"
    lens: str                 # "fixed", "uniform", "lognormal"
    fixed_lens: tuple = ()
    lo: int = 1
    hi: int = 1
    median: float = 1.0
    sigma: float = 1.0
    k_mul: float = 1.0
    free_frac: float = 0.0    # fraction of the pool left free (interleaved)
    nb_fixed: int = 0         # pool size when fixed by the recipe
    layers: int = 1
    seed: int = 0
    chunk: int = 0            # prefill: new tokens per sequence (0 = the whole context)
    values: str = "normal"    # "normal" or "rounding_stress" (see rounding_stress_values)
    description: str = ""


SPECS = {
    "tiny": Spec(
        "tiny", B=4, Hq=8, Hkv=2, D=64, out_dtype="f32", lens="fixed",
        fixed_lens=(7, 16, 33, 64), nb_fixed=32, seed=1001,
        description="batch 4, lens {7,16,33,64}, 8/2 heads, D 64, 32-block pool, fp32 out"),
    "qwen3_0_6b": Spec(
        "qwen3_0_6b", B=8, Hq=16, Hkv=8, D=128, out_dtype="bf16", lens="uniform",
        lo=128, hi=2048, seed=1002,
        description="Qwen3-0.6B-shaped layer: batch 8, lens U[128,2048], 16/8 heads, D 128, bf16 out"),
    "qwen3_4b": Spec(
        "qwen3_4b", B=32, Hq=32, Hkv=8, D=128, out_dtype="bf16", lens="uniform",
        lo=512, hi=8192, k_mul=2.0, free_frac=0.10, seed=1003,
        description="Qwen3-4B-shaped layer: batch 32, lens U[512,8192], 32/8 heads, D 128, "
                    "10% free blocks interleaved, K x2, bf16 out"),
    "skewed": Spec(
        "skewed", B=4, Hq=32, Hkv=8, D=128, out_dtype="f32", lens="fixed",
        fixed_lens=(32768, 1024, 256, 17), seed=1004,
        description="skewed long context: lens {32768,1024,256,17}, 32/8 heads, D 128, fp32 out"),
    "skewed_bf16": Spec(
        "skewed_bf16", B=4, Hq=32, Hkv=8, D=128, out_dtype="bf16", lens="fixed",
        fixed_lens=(32768, 1024, 256, 17), seed=1004,
        description="skewed long context, bf16 out"),
    "prefill_tiny": Spec(
        "prefill_tiny", B=4, Hq=8, Hkv=2, D=64, out_dtype="f32", lens="fixed",
        fixed_lens=(20, 45, 7, 64), chunk=24, free_frac=0.2, seed=1011,
        description="prefill: batch 4, lens {20,45,7,64}, last min(24, L) tokens new, 8/2 heads, D 64, fp32"),
    "prefill_4b": Spec(
        "prefill_4b", B=8, Hq=32, Hkv=8, D=128, out_dtype="bf16", lens="uniform",
        lo=512, hi=4096, chunk=512, k_mul=2.0, free_frac=0.10, seed=1012,
        description="Qwen3-4B-shaped chunked prefill: batch 8, a 512-token chunk ending contexts U[512,4096], "
                    "32/8 heads, D 128, 10% free blocks, K x2, bf16 out"),
    "cb36": Spec(
        "cb36", B=64, Hq=32, Hkv=8, D=128, out_dtype="bf16", lens="lognormal",
        lo=1, hi=16384, median=1024.0, sigma=1.0, layers=36, seed=1005,
        description="continuous-batching step over 36 layers: batch 64, lens lognormal "
                    "(median 1024, sigma 1) clipped to [1,16384], 32/8 heads, D 128, bf16"),
}


# Logit gap of the rounding-stress values: exp(-7.8125 / sqrt(128)) = 0.50131,
# just above 0.5, so a softmax weight rounded to bf16 (steps of 2^-8 there)
# loses 0.26 % of itself.  7.8125 is exact in bf16.
STRESS_GAP = 7.8125


def rounding_stress_values(spec: Spec, key, rows: int, slot_of_row, nb: int):
    """q [rows, Hq, D], k/v of the new rows [rows, Hkv, D] and caches [nb, Hkv, 16, D]
    (bf16 bits) for the worst case of the output precision: every softmax
    weight but one per block sits just above 0.5, where rounding it to bf16
    drops about 2^-8.6 of it in the same direction, and every V value is
    large (magnitude in [7, 8), one sign per (KV head, dim)), so the output
    is too.  Query head h has a single 1 at dim h % G; key dims < G hold
    STRESS_GAP in slot 0 of every block and 0 elsewhere, so slot 0 of each
    block is the maximum and the other 15 tokens get weight exp(-gap scale).
    ``slot_of_row(r)`` is the cache slot (0..15) of new row r."""
    G, D = spec.Hq // spec.Hkv, spec.D
    rng = np.random.default_rng([*key, 0x5735])
    q = np.zeros((rows, spec.Hq, D), dtype=np.float32)
    for h in range(spec.Hq):
        q[:, h, h % G] = 1.0
    kc = rng.standard_normal((nb, spec.Hkv, BLOCK_SIZE, D), dtype=np.float32)
    kc[:, :, :, :G] = 0.0
    kc[:, :, 0, :G] = STRESS_GAP
    kn = rng.standard_normal((rows, spec.Hkv, D), dtype=np.float32)
    kn[:, :, :G] = 0.0
    for r in range(rows):
        if slot_of_row(r) == 0:
            kn[r, :, :G] = STRESS_GAP
    sign = np.where(rng.random((spec.Hkv, D)) < 0.5, -1.0, 1.0).astype(np.float32)
    vc = sign[None, :, None, :] * rng.uniform(7.0, 7.97, (nb, spec.Hkv, BLOCK_SIZE, D)).astype(np.float32)
    vn = sign[None, :, :] * rng.uniform(7.0, 7.97, (rows, spec.Hkv, D)).astype(np.float32)
    return tuple(f32_to_bf16_bits(x) for x in (q, kn, vn, kc, vc))


@dataclasses.dataclass
class Workload:
    """One batch of decode inputs.  Arrays are numpy; bf16 tensors are uint16 bits.

    Per-layer tensors come from ``layer(l)`` so that a many-layer step can be
    produced (and checked) one layer at a time.
    """
    spec: Spec
    seed: int
    NB: int
    MB: int
    context_lens: np.ndarray   # int32 [B]
    block_tables: np.ndarray   # int32 [B, MB]
    slot_mapping: np.ndarray   # int64 [B]
    scale: float               # float32 value, passed to both sides

    @property
    def B(self): return self.spec.B

    @property
    def Hq(self): return self.spec.Hq

    @property
    def Hkv(self): return self.spec.Hkv

    @property
    def D(self): return self.spec.D

    @property
    def BS(self): return BLOCK_SIZE

    @property
    def layers(self): return self.spec.layers

    def layer(self, l: int = 0) -> dict:
        """q, k_new, v_new and the pre-append (poisoned) caches of layer ``l``."""
        s = self.spec
        key = (self.seed, 1 + l)
        if s.values == "rounding_stress":
            q, k_new, v_new, k_cache, v_cache = rounding_stress_values(
                s, key, s.B, lambda b: (int(self.context_lens[b]) - 1) % BLOCK_SIZE, self.NB)
        else:
            q = _normal_bf16((*key, 0), (s.B, s.Hq, s.D))
            k_new = _normal_bf16((*key, 1), (s.B, s.Hkv, s.D), s.k_mul)
            v_new = _normal_bf16((*key, 2), (s.B, s.Hkv, s.D))
            shape = (self.NB, s.Hkv, BLOCK_SIZE, s.D)
            k_cache = _normal_bf16((*key, 3), shape, s.k_mul)
            v_cache = _normal_bf16((*key, 4), shape)
        pb, po = np.nonzero(self.poison_mask())
        k_cache[pb, :, po, :] = BF16_NAN
        v_cache[pb, :, po, :] = BF16_NAN
        return dict(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache)

    def qk_norm_weights(self, l: int = 0):
        """bf16 bits of the per-head RMSNorm weights of layer ``l`` for q and k:
        [D] each, 1 + 0.25 * N(0, 1) (learned weights hover around one)."""
        key = (self.seed, 1 + l, 5)
        w = _normal_bf16(key, (2, self.spec.D))
        x = bf16_bits_to_f32(w) * np.float32(0.25) + np.float32(1.0)
        out = f32_to_bf16_bits(x)
        return out[0], out[1]

    def poison_mask(self, new_tokens=None) -> np.ndarray:
        """bool [NB, BS]: slots holding no token before this step's append
        (of one token per sequence, or of ``new_tokens[b]``)."""
        holds = np.zeros((self.NB, BLOCK_SIZE), dtype=bool)
        for b in range(self.B):
            n_new = 1 if new_tokens is None else int(new_tokens[b])
            n_before = int(self.context_lens[b]) - n_new   # tokens already cached
            for j in range(-(-n_before // BLOCK_SIZE) if n_before > 0 else 0):
                p = int(self.block_tables[b, j])
                cnt = min(BLOCK_SIZE, n_before - j * BLOCK_SIZE)
                holds[p, :cnt] = True
        return ~holds

    def bytes_decode(self, out_bytes: int | None = None) -> int:
        """Algorithmic bytes of one decode call: q + K/V rows of every cached
        token + the output.  (Accounting, not arithmetic of the method.)"""
        s = self.spec
        ob = out_bytes if out_bytes is not None else (4 if s.out_dtype == "f32" else 2)
        tok = int(self.context_lens.astype(np.int64).sum())
        return s.B * s.Hq * s.D * 2 + tok * s.Hkv * s.D * 2 * 2 + s.B * s.Hq * s.D * ob

    def bytes_append(self) -> int:
        """Bytes one append call moves: new K/V rows read and written."""
        rows = int((self.slot_mapping >= 0).sum())
        return rows * self.Hkv * self.D * 2 * 2 * 2


def _lengths(spec: Spec, rng: np.random.Generator) -> np.ndarray:
    if spec.lens == "fixed":
        return np.array(spec.fixed_lens, dtype=np.int32)
    if spec.lens == "uniform":
        return rng.integers(spec.lo, spec.hi, size=spec.B, endpoint=True).astype(np.int32)
    if spec.lens == "lognormal":
        x = np.exp(rng.normal(math.log(spec.median), spec.sigma, size=spec.B))
        return np.clip(np.rint(x), spec.lo, spec.hi).astype(np.int32)
    raise ValueError(spec.lens)


def make_workload(name_or_spec, seed: int | None = None, context_lens=None) -> Workload:
    """Build the index structures of a named (or custom) workload.

    ``context_lens`` overrides the recipe's lengths (edge-case tests).
    """
    spec = SPECS[name_or_spec] if isinstance(name_or_spec, str) else name_or_spec
    seed = spec.seed if seed is None else int(seed)
    rng = np.random.default_rng([seed, 0])
    lens = _lengths(spec, rng) if context_lens is None else np.asarray(context_lens, np.int32)
    if lens.shape != (spec.B,):
        raise ValueError("context_lens must have one entry per sequence")
    nblk = [-(-int(L) // BLOCK_SIZE) for L in lens]
    needed = sum(nblk)
    if spec.nb_fixed:
        NB = spec.nb_fixed
        if NB < needed:
            raise ValueError("pool too small for these lengths")
    elif spec.free_frac > 0:
        NB = math.ceil(needed / (1.0 - spec.free_frac))
    else:
        NB = needed
    MB = max(1, max(nblk) if nblk else 1)
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((spec.B, MB), -1, dtype=np.int32)
    slots = np.full(spec.B, -1, dtype=np.int64)
    pos = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[pos:pos + n]
        pos += n
        L = int(lens[b])
        if L > 0:
            t = L - 1                     # the appended token's position
            slots[b] = int(tables[b, t // BLOCK_SIZE]) * BLOCK_SIZE + t % BLOCK_SIZE
    scale = float(np.float32(1.0 / math.sqrt(spec.D)))
    return Workload(spec=spec, seed=seed, NB=NB, MB=MB, context_lens=lens.astype(np.int32),
                    block_tables=tables, slot_mapping=slots, scale=scale)


def custom_spec(name="custom", **kw) -> Spec:
    """A Spec for tests: any field of ``Spec`` may be given."""
    base = dict(B=2, Hq=8, Hkv=2, D=64, out_dtype="f32", lens="fixed", fixed_lens=(1, 1), seed=7)
    base.update(kw)
    return Spec(name, **base)


@dataclasses.dataclass
class RequestStream:
    """Requests for the continuous-batching step driver, in arrival order."""
    seq_ids: np.ndarray   # int64 [n]
    prompts: np.ndarray   # int32 [n] prompt tokens
    max_new: np.ndarray   # int32 [n] decode steps
    arrive: np.ndarray    # int32 [n] step before which the request is submitted (non-decreasing)

    def arriving(self, step: int):
        """(seq_id, prompt, max_new) of the requests submitted before ``step``."""
        idx = np.nonzero(self.arrive == step)[0]
        return [(int(self.seq_ids[i]), int(self.prompts[i]), int(self.max_new[i])) for i in idx]


def request_stream(n: int, seed: int, prompt_median: float = 1024.0, prompt_sigma: float = 1.0,
                   prompt_max: int = 16383, new_min: int = 1, new_max: int = 256,
                   arrivals_per_step: float = 1.0) -> RequestStream:
    """n seeded requests: prompt lengths round(exp(N(ln median, sigma))) clipped
    to [0, prompt_max], decode lengths uniform in [new_min, new_max], arrival
    steps from exponential gaps of mean 1/arrivals_per_step steps (several
    requests can arrive before the same step)."""
    rng = np.random.Generator(np.random.PCG64([seed, 0x5e7]))
    prompts = np.clip(np.rint(np.exp(rng.normal(math.log(prompt_median), prompt_sigma, n))), 0, prompt_max)
    max_new = rng.integers(new_min, new_max, size=n, endpoint=True)
    gaps = rng.exponential(1.0 / arrivals_per_step, n)
    arrive = np.floor(np.cumsum(gaps) - gaps[0]).astype(np.int32)
    ids = np.arange(n, dtype=np.int64) * 7 + 1000   # not the row numbers: ids are opaque
    return RequestStream(ids, prompts.astype(np.int32), max_new.astype(np.int32), arrive)


@dataclasses.dataclass
class PrefillWorkload:
    """A chunked-prefill batch over the same paged layout: sequence b ends with
    n_b = chunk_lens[b] new tokens at positions L_b - n_b .. L_b - 1, packed in
    ``query_start`` order.  Their K/V go into the cache one slot per token
    (``slot_mapping``, int64 [T]) before the prefill attends over all L_b
    tokens; every slot that holds no token before that append is NaN."""
    base: Workload
    chunk_lens: np.ndarray    # int32 [B]
    query_start: np.ndarray   # int32 [B + 1]
    slot_mapping: np.ndarray  # int64 [T]

    def __getattr__(self, name):          # shapes, tables, lens and scale come from the base batch
        if name == "base":
            raise AttributeError(name)
        return getattr(self.base, name)

    @property
    def T(self): return int(self.query_start[-1])

    def layer(self, l: int = 0) -> dict:
        """q [T,Hq,D], the chunk's k/v [T,Hkv,D] and the pre-append caches of layer ``l``."""
        s = self.base.spec
        key = (self.base.seed, 1 + l)
        if s.values == "rounding_stress":
            q, k_new, v_new, k_cache, v_cache = rounding_stress_values(
                s, key, self.T, lambda r: int(self.slot_mapping[r]) % BLOCK_SIZE, self.base.NB)
        else:
            q = _normal_bf16((*key, 10), (self.T, s.Hq, s.D))
            k_new = _normal_bf16((*key, 11), (self.T, s.Hkv, s.D), s.k_mul)
            v_new = _normal_bf16((*key, 12), (self.T, s.Hkv, s.D))
            shape = (self.base.NB, s.Hkv, BLOCK_SIZE, s.D)
            k_cache = _normal_bf16((*key, 3), shape, s.k_mul)
            v_cache = _normal_bf16((*key, 4), shape)
        pb, po = np.nonzero(self.base.poison_mask(self.chunk_lens))
        k_cache[pb, :, po, :] = BF16_NAN
        v_cache[pb, :, po, :] = BF16_NAN
        return dict(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache)

    def attended_pairs(self) -> int:
        """(query token, cached token) pairs the causal prefill visits: sum over
        sequences and query tokens of position + 1.  (Accounting only.)"""
        n = self.chunk_lens.astype(np.int64)
        L = self.base.context_lens.astype(np.int64)
        return int(np.sum(n * (L - n) + n * (n + 1) // 2))


def make_prefill(name_or_spec, seed: int | None = None, context_lens=None, chunk_lens=None) -> PrefillWorkload:
    """A prefill batch: tables and lengths as ``make_workload`` builds them,
    n_b = min(chunk, L_b) new tokens per sequence (all L_b when the spec's
    chunk is 0) unless ``chunk_lens`` gives them."""
    base = make_workload(name_or_spec, seed, context_lens)
    L = base.context_lens
    if chunk_lens is None:
        n = np.minimum(L, base.spec.chunk) if base.spec.chunk > 0 else L.copy()
    else:
        n = np.asarray(chunk_lens, dtype=np.int32)
        if n.shape != L.shape or np.any(n < 0) or np.any(n > L):
            raise ValueError("chunk_lens must satisfy 0 <= n_b <= context_lens[b]")
    n = n.astype(np.int32)
    qs = np.zeros(base.B + 1, dtype=np.int32)
    qs[1:] = np.cumsum(n)
    slots = np.empty(int(qs[-1]), dtype=np.int64)
    for b in range(base.B):
        for i in range(int(n[b])):
            t = int(L[b]) - int(n[b]) + i
            slots[qs[b] + i] = int(base.block_tables[b, t // BLOCK_SIZE]) * BLOCK_SIZE + t % BLOCK_SIZE
    return PrefillWorkload(base=base, chunk_lens=n, query_start=qs, slot_mapping=slots)
