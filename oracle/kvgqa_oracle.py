"""FP64 CPU oracle for the positions-aware cached GQA + RoPE decode step and
the equal-length prefill into empty cache rows.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or call this module.  The product
path (the CUDA library and its Python binding) never imports it, and this
module imports nothing from the product package: the two share no code.

What it computes is the plain definition of each step, in float64, with plain
numpy operations (a matrix product is the only library primitive used):

* split-half rotary position embedding (microLLM-rocm ARCHITECTURE.md, section
  "Attention layout boundary": the bias + split-half RoPE kernel requires an even
  head width D, a nonnegative position offset and a positive base);
* the positions-aware K/V store and cached attention of the active-row decode
  step (same page, section "Tensor ownership boundary": device ``positions[A]``
  and ``cache_rows[A]`` parameterise decode RoPE, K/V store and cached attention;
  inactive full-capacity rows stay untouched);
* the equal-length prefill whose prefixes land in their target empty cache rows
  (same section: one [A, T] batch runs, then each prefix is mapped into its
  target empty shared-cache row), and its generalisation to prompts of
  different lengths at nonnegative position offsets into rows that already
  hold a prefix (chunked prefill; prompts of other lengths form separate
  groups there, one call here).

Storage is BF16 (16-bit patterns in numpy ``uint16`` arrays), or IEEE
binary16 where a function is given ``fmt="f16"`` (the FP16 cached rows that
microLLM-rocm operator-development.md, section "Public interfaces", has its
typed softmax serve beside BF16); arithmetic is float64; results that the
path stores are rounded once, directly from float64, to nearest-even in the
storage format.

Readings taken where the pages are silent:
  - pair i of a head is (x[i], x[i + D/2]) and rotates by angle pos * theta^(-2i/D),
    y[i] = x[i] cos - x[i+D/2] sin, y[i+D/2] = x[i+D/2] cos + x[i] sin;
  - the decode token attends to keys 0..pos inclusive (its own K/V is stored first);
  - q is rounded to BF16 after rotation, before attention;
  - the softmax scale multiplies the float score q.k (it is not folded into q);
  - query head h reads KV head floor(h / G), G = H_q / H_kv;
  - prefill positions start at 0 (the target rows are empty); a chunk's
    positions start at its offset and see the row's prefix before it.

Parity pins: every function here is checked by ``tests/test_oracle_pins.py``
against closed forms, invariants and brute force; none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_to_f64", "f64_to_bf16", "rope_inv_freq", "rope_split_half",
    "rope_split_half_bf16", "rope_kv_store", "cached_gqa_attention",
    "cached_gqa_attention_one", "prefill_gqa_cached_rows", "prefill_varlen_gqa_cached_rows",
    "prefill_attention_one", "ulp_distance_bf16", "f16_to_f64", "f64_to_f16", "widen", "codec",
]


# ---------------------------------------------------------------- BF16 codec
def bf16_to_f64(bits) -> np.ndarray:
    """BF16 bit patterns -> float64 (exact: BF16 is the top half of FP32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round float64 values to BF16, nearest-even, in one rounding step.

    BF16 keeps 8 significant bits and FP32's exponent range (normal numbers
    down to 2^-126, subnormal spacing 2^-133).  A value is scaled by a power of
    two so that its last kept bit has weight 1, rounded with ``np.rint`` (ties
    to even), scaled back, and reinterpreted.  Rounding happens once, from
    float64: there is no intermediate FP32 rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    _, e = np.frexp(ax)                       # ax = m * 2^e, m in [0.5, 1)
    quantum = np.where(e >= -125, e - 8, -133)
    y = np.ldexp(np.rint(np.ldexp(ax, -quantum)), quantum)
    with np.errstate(over="ignore", invalid="ignore"):
        y32 = y.astype(np.float32)            # exact: y has at most 8 significant bits
    bits = (y32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = np.where(np.isnan(x), np.uint16(0x7FC0), bits)
    bits = np.where(np.signbit(x), bits | np.uint16(0x8000), bits)
    return bits.astype(np.uint16)


def f16_to_f64(bits) -> np.ndarray:
    """IEEE binary16 bit patterns -> float64 (exact: every half value is a
    double; the widening is numpy's, which preserves the value)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def f64_to_f16(x) -> np.ndarray:
    """Round float64 values to IEEE binary16, nearest-even, in one step.

    Binary16 keeps 11 significant bits, normal numbers from 2^-14, subnormal
    spacing 2^-24, largest finite 65504.  As for BF16: scale so that the last
    kept bit has weight 1, round with ``np.rint`` (ties to even), scale back.
    A result above 65504 (from 65520 up) is out of range and becomes infinity.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    _, e = np.frexp(ax)                       # ax = m * 2^e, m in [0.5, 1)
    quantum = np.maximum(e - 11, -24)
    y = np.ldexp(np.rint(np.ldexp(ax, -quantum)), quantum)
    y = np.where(y > 65504.0, np.inf, y)
    with np.errstate(over="ignore", invalid="ignore"):
        bits = y.astype(np.float16).view(np.uint16)   # exact: y is a binary16 value or inf
    bits = np.where(np.isnan(x), np.uint16(0x7E00), bits)
    bits = np.where(np.signbit(x), bits | np.uint16(0x8000), bits)
    return bits.astype(np.uint16)


def codec(fmt: str):
    """(widen, round) of a storage format: "bf16" or "f16"."""
    return {"bf16": (bf16_to_f64, f64_to_bf16), "f16": (f16_to_f64, f64_to_f16)}[fmt]


def widen(bits, fmt: str = "bf16") -> np.ndarray:
    return codec(fmt)[0](bits)


def ulp_distance_bf16(a_bits, b_bits) -> np.ndarray:
    """Distance between BF16 patterns counted in representable values
    (ordered-integer difference; +0 and -0 are the same point).  The same
    ordering holds for binary16 patterns, so it serves both formats."""
    def ordered(b):
        b = np.asarray(b, dtype=np.uint16).astype(np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(ordered(a_bits) - ordered(b_bits))


# ---------------------------------------------------------------- RoPE
def rope_inv_freq(D: int, theta: float) -> np.ndarray:
    """Angular frequency of pair i: theta^(-2i/D), i = 0..D/2-1."""
    if D % 2:
        raise ValueError("split-half RoPE needs an even head width")
    if not theta > 0:
        raise ValueError("RoPE base must be positive")
    i = np.arange(D // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / D)


def rope_split_half(x, positions, theta: float) -> np.ndarray:
    """Split-half rotation of float64 vectors.

    ``x`` has shape [..., D]; ``positions`` broadcasts against x[..., 0].
    Pair i is (x[i], x[i + D/2]); it turns by phi = pos * theta^(-2i/D):
        y[i]       = x[i] cos(phi) - x[i + D/2] sin(phi)
        y[i + D/2] = x[i + D/2] cos(phi) + x[i] sin(phi)
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    pos = np.asarray(positions)
    if np.any(pos < 0):
        raise ValueError("RoPE positions must be nonnegative")
    phi = pos.astype(np.float64)[..., None] * rope_inv_freq(D, theta)
    c, s = np.cos(phi), np.sin(phi)
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_split_half_bf16(x_bits, positions, theta: float, fmt: str = "bf16") -> np.ndarray:
    """Stored format in, stored format out (BF16 unless ``fmt`` says "f16"):
    widen, rotate in float64, round once."""
    to64, round16 = codec(fmt)
    return round16(rope_split_half(to64(x_bits), positions, theta))


# ---------------------------------------------------------------- decode store
def rope_kv_store(q, k, v, positions, cache_rows, theta, k_cache, v_cache, fmt="bf16"):
    """Decode RoPE + K/V store for A active tokens.

    q [A, H_q, D], k/v [A, H_kv, D] (BF16 bits); positions, cache_rows [A];
    k_cache/v_cache [S, H_kv, max_seq, D] (BF16 bits, not modified).
    Returns (q_rot, k_cache', v_cache'): q rotated at its own position, and
    copies of the caches in which cell [cache_rows[a], :, positions[a], :] of
    each active token holds its rotated K and its V bytes unchanged.  Every
    other byte of the caches is left as it was.
    """
    positions = np.asarray(positions, dtype=np.int64)
    rows = np.asarray(cache_rows, dtype=np.int64)
    S, H_kv, max_seq, D = k_cache.shape
    if np.any((positions < 0) | (positions >= max_seq)) or np.any((rows < 0) | (rows >= S)):
        raise ValueError("position or cache row out of range")
    if len(set(rows.tolist())) != len(rows):
        raise ValueError("cache rows of one step must be distinct")
    q_rot = rope_split_half_bf16(q, positions[:, None], theta, fmt)
    k_rot = rope_split_half_bf16(k, positions[:, None], theta, fmt)
    kc = np.array(k_cache, dtype=np.uint16, copy=True)
    vc = np.array(v_cache, dtype=np.uint16, copy=True)
    for a in range(len(rows)):
        kc[rows[a], :, positions[a], :] = k_rot[a]
        vc[rows[a], :, positions[a], :] = np.asarray(v[a], dtype=np.uint16)
    return q_rot, kc, vc


# ---------------------------------------------------------------- attention
def softmax(s: np.ndarray) -> np.ndarray:
    """Softmax over the last axis in float64 (max-shifted, exact definition)."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def cached_gqa_attention_one(q_vec, keys, values, scale: float) -> np.ndarray:
    """softmax(keys @ q * scale) @ values for one query (all float64)."""
    s = (keys @ q_vec) * scale
    return softmax(s) @ values


def cached_gqa_attention(q_rot, k_cache, v_cache, positions, cache_rows,
                         scale: float, heads=None, fmt="bf16") -> np.ndarray:
    """Cached GQA attention of the decode step, float64 result.

    Token a, query head h attends to keys 0..positions[a] (inclusive) of KV head
    floor(h / G) in cache row cache_rows[a].  ``heads`` optionally lists the
    (a, h) pairs to compute; the others stay NaN.  Result [A, H_q, D].
    """
    q_rot = np.asarray(q_rot, dtype=np.uint16)
    A, H_q, D = q_rot.shape
    H_kv = k_cache.shape[1]
    G = H_q // H_kv
    out = np.full((A, H_q, D), np.nan)
    pairs = [(a, h) for a in range(A) for h in range(H_q)] if heads is None else heads
    for a, h in pairs:
        r, p, g = int(cache_rows[a]), int(positions[a]), h // G
        keys = widen(k_cache[r, g, : p + 1], fmt)
        vals = widen(v_cache[r, g, : p + 1], fmt)
        out[a, h] = cached_gqa_attention_one(widen(q_rot[a, h], fmt), keys, vals, scale)
    return out


# ---------------------------------------------------------------- prefill
def prefill_attention_one(q_rot_bits, k_rows, v_rows, t: int, scale: float, fmt="bf16") -> np.ndarray:
    """Causal attention of prompt position t over cached positions 0..t."""
    return cached_gqa_attention_one(widen(q_rot_bits, fmt), widen(k_rows[: t + 1], fmt),
                                    widen(v_rows[: t + 1], fmt), scale)


def prefill_gqa_cached_rows(q, k, v, cache_rows, theta, scale, k_cache, v_cache,
                            select=None, fmt="bf16"):
    """Equal-length prefill of A prompts into empty cache rows.

    q [A, T, H_q, D], k/v [A, T, H_kv, D] (BF16 bits, token-major BTHD), positions
    0..T-1.  Rotated K and raw V of prompt a go to cache row cache_rows[a],
    positions [0, T); nothing else in the caches changes.  Causal GQA attention
    (position t sees 0..t) reads them back from the cache rows.

    Returns (q_rot [A, T, H_q, D] bits, out float64 [A, T, H_q, D], k_cache',
    v_cache').  ``select`` optionally lists the (a, t, h) outputs to compute
    (others NaN); without it every output is computed, one (a, h) at a time.
    """
    q = np.asarray(q, dtype=np.uint16)
    A, T, H_q, D = q.shape
    S, H_kv, max_seq, _ = k_cache.shape
    G = H_q // H_kv
    rows = np.asarray(cache_rows, dtype=np.int64)
    if T > max_seq:
        raise ValueError("prompt longer than the cache")
    if np.any((rows < 0) | (rows >= S)) or len(set(rows.tolist())) != len(rows):
        raise ValueError("cache rows must be distinct and in range")
    pos = np.arange(T)
    q_rot = rope_split_half_bf16(q, pos[None, :, None], theta, fmt)
    k_rot = rope_split_half_bf16(k, pos[None, :, None], theta, fmt)
    kc = np.array(k_cache, dtype=np.uint16, copy=True)
    vc = np.array(v_cache, dtype=np.uint16, copy=True)
    for a in range(A):
        kc[rows[a], :, :T, :] = np.transpose(k_rot[a], (1, 0, 2))
        vc[rows[a], :, :T, :] = np.transpose(np.asarray(v[a], dtype=np.uint16), (1, 0, 2))
    out = np.full((A, T, H_q, D), np.nan)
    if select is None:
        mask = np.tril(np.ones((T, T), dtype=bool))
        for a in range(A):
            for h in range(H_q):
                g = h // G
                Q = widen(q_rot[a, :, h], fmt)
                K = widen(kc[rows[a], g, :T], fmt)
                V = widen(vc[rows[a], g, :T], fmt)
                s = (Q @ K.T) * scale
                s = np.where(mask, s, -np.inf)
                out[a, :, h] = softmax(s) @ V
    else:
        for a, t, h in select:
            g = h // G
            out[a, t, h] = prefill_attention_one(q_rot[a, t, h], kc[rows[a], g, :T],
                                                 vc[rows[a], g, :T], t, scale, fmt)
    return q_rot, out, kc, vc


def prefill_varlen_gqa_cached_rows(q, k, v, offsets, lengths, cache_rows, theta, scale, k_cache, v_cache,
                                   select=None, fmt="bf16"):
    """Prefill of A prompts of different lengths into rows that may already
    hold a prefix (chunked prefill).

    microLLM-rocm ARCHITECTURE.md, "Tensor ownership boundary" (prompts of
    other lengths form separate equal-length groups there; here one call takes
    them together) and "Attention layout boundary" (RoPE takes a nonnegative
    position offset).  Prompt a has lengths[a] tokens (the first ones of the
    padded [A, T] batch); token t sits at position p = offsets[a] + t of row
    cache_rows[a].  Q and K are rotated at p, rotated K and raw V are stored at
    (row, :, p, :), and query (a, t, h) attends causally over keys 0..p of its
    row: the row's existing prefix [0, offsets[a]) and the prompt's tokens up
    to itself.  Outputs for t >= lengths[a] are NaN; nothing else in the
    caches changes.

    Returns (q_rot [A, T, H_q, D] bits (rows past a prompt's length 0),
    out float64 [A, T, H_q, D], k_cache', v_cache').  ``select`` optionally
    lists the (a, t, h) outputs to compute.
    """
    q = np.asarray(q, dtype=np.uint16)
    k = np.asarray(k, dtype=np.uint16)
    v = np.asarray(v, dtype=np.uint16)
    A, T, H_q, D = q.shape
    S, H_kv, max_seq, _ = k_cache.shape
    G = H_q // H_kv
    rows = np.asarray(cache_rows, dtype=np.int64)
    off = np.asarray(offsets, dtype=np.int64)
    lens = np.asarray(lengths, dtype=np.int64)
    if np.any((rows < 0) | (rows >= S)) or len(set(rows.tolist())) != len(rows):
        raise ValueError("cache rows must be distinct and in range")
    if np.any(lens < 0) or np.any(lens > T) or np.any(off < 0) or np.any(off + lens > max_seq):
        raise ValueError("offsets/lengths out of range")
    q_rot = np.zeros_like(q)
    kc = np.array(k_cache, dtype=np.uint16, copy=True)
    vc = np.array(v_cache, dtype=np.uint16, copy=True)
    for a in range(A):
        L, o = int(lens[a]), int(off[a])
        pos = o + np.arange(L)
        q_rot[a, :L] = rope_split_half_bf16(q[a, :L], pos[:, None], theta, fmt)
        k_rot = rope_split_half_bf16(k[a, :L], pos[:, None], theta, fmt)
        kc[rows[a], :, o:o + L, :] = np.transpose(k_rot, (1, 0, 2))
        vc[rows[a], :, o:o + L, :] = np.transpose(v[a, :L], (1, 0, 2))
    out = np.full((A, T, H_q, D), np.nan)
    if select is None:
        for a in range(A):
            L, o = int(lens[a]), int(off[a])
            if L == 0:
                continue
            n = o + L
            mask = np.arange(n)[None, :] <= (o + np.arange(L))[:, None]   # key j visible to query t
            for h in range(H_q):
                g = h // G
                Q = widen(q_rot[a, :L, h], fmt)
                K = widen(kc[rows[a], g, :n], fmt)
                V = widen(vc[rows[a], g, :n], fmt)
                s = np.where(mask, (Q @ K.T) * scale, -np.inf)
                out[a, :L, h] = softmax(s) @ V
    else:
        for a, t, h in select:
            if t >= lens[a]:
                continue
            g = h // G
            p = int(off[a]) + t
            out[a, t, h] = cached_gqa_attention_one(widen(q_rot[a, t, h], fmt), widen(kc[rows[a], g, :p + 1], fmt),
                                                    widen(vc[rows[a], g, :p + 1], fmt), scale)
    return q_rot, out, kc, vc
