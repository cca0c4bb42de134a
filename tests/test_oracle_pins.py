"""The FP64 oracle against closed forms, invariants, a library rounding routine
and brute force; then planted mistakes in copies of the oracle, each of which
must be caught by at least one of those checks."""
import importlib.util
import math
import os
import types

import numpy as np
import pytest

import oracle
import oracle_pins as pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "kvgqa_oracle.py")


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle.kvgqa_oracle)


def fresh_oracle(patch=None):
    """A private copy of the oracle module; ``patch`` = (old, new) replaces one
    source fragment (it must occur exactly once) before the copy is loaded, to
    plant a mistake inside a function rather than around it."""
    if patch is None:
        spec = importlib.util.spec_from_file_location("kvgqa_oracle_mutant", ORACLE_SRC)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        return mod
    src = open(ORACLE_SRC).read()
    old, new = patch
    assert src.count(old) == 1, f"patch target not unique: {old!r}"
    mod = types.ModuleType("kvgqa_oracle_mutant")
    exec(compile(src.replace(old, new), ORACLE_SRC, "exec"), mod.__dict__)
    return mod


def mutant_rope_direction(m):
    def rope(x, positions, theta):
        x = np.asarray(x, dtype=np.float64); D = x.shape[-1]
        phi = np.asarray(positions).astype(np.float64)[..., None] * m.rope_inv_freq(D, theta)
        c, s = np.cos(phi), np.sin(phi)
        x1, x2 = x[..., : D // 2], x[..., D // 2:]
        return np.concatenate([x1 * c + x2 * s, x2 * c - x1 * s], axis=-1)
    m.rope_split_half = rope


def mutant_rope_interleaved(m):
    def rope(x, positions, theta):
        x = np.asarray(x, dtype=np.float64); D = x.shape[-1]
        phi = np.asarray(positions).astype(np.float64)[..., None] * m.rope_inv_freq(D, theta)
        c, s = np.cos(phi), np.sin(phi)
        x1, x2 = x[..., 0::2], x[..., 1::2]
        y = np.empty_like(x)
        y[..., 0::2] = x1 * c - x2 * s
        y[..., 1::2] = x2 * c + x1 * s
        return y
    m.rope_split_half = rope


def mutant_rope_frequency(m):
    m.rope_inv_freq = lambda D, theta: np.power(float(theta), -np.arange(D // 2) / D)


def mutant_gqa_modulo(m):
    def attn(q_rot, k_cache, v_cache, positions, cache_rows, scale, heads=None):
        A, H_q, D = q_rot.shape
        H_kv = k_cache.shape[1]
        out = np.full((A, H_q, D), np.nan)
        for a in range(A):
            for h in range(H_q):
                r, p, g = int(cache_rows[a]), int(positions[a]), h % H_kv
                out[a, h] = m.cached_gqa_attention_one(
                    m.bf16_to_f64(q_rot[a, h]), m.bf16_to_f64(k_cache[r, g, : p + 1]),
                    m.bf16_to_f64(v_cache[r, g, : p + 1]), scale)
        return out
    m.cached_gqa_attention = attn


def mutant_exclusive_prefix(m):
    orig = m.cached_gqa_attention
    m.cached_gqa_attention = lambda q, kc, vc, pos, rows, scale, heads=None: orig(
        q, kc, vc, np.maximum(np.asarray(pos) - 1, 0), rows, scale, heads)


def mutant_scale_ignored(m):
    m.cached_gqa_attention_one = lambda q, keys, values, scale: m.softmax(keys @ q) @ values


def mutant_double_rounding(m):
    def f(x):
        import torch
        x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
        return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    m.f64_to_bf16 = f


def mutant_prefill_not_causal(m):
    orig_one = m.cached_gqa_attention_one

    def prefill(q, k, v, cache_rows, theta, scale, k_cache, v_cache, select=None):
        q = np.asarray(q, dtype=np.uint16)
        A, T, H_q, D = q.shape
        G = H_q // k_cache.shape[1]
        pos = np.arange(T)
        q_rot = m.rope_split_half_bf16(q, pos[None, :, None], theta)
        k_rot = m.rope_split_half_bf16(k, pos[None, :, None], theta)
        kc, vc = k_cache.copy(), v_cache.copy()
        rows = np.asarray(cache_rows)
        out = np.zeros((A, T, H_q, D))
        for a in range(A):
            kc[rows[a], :, :T] = np.transpose(k_rot[a], (1, 0, 2))
            vc[rows[a], :, :T] = np.transpose(v[a], (1, 0, 2))
            for t in range(T):
                for h in range(H_q):
                    out[a, t, h] = orig_one(m.bf16_to_f64(q_rot[a, t, h]),
                                            m.bf16_to_f64(kc[rows[a], h // G, :T]),
                                            m.bf16_to_f64(vc[rows[a], h // G, :T]), scale)
        return q_rot, out, kc, vc
    m.prefill_gqa_cached_rows = prefill


def mutant_store_row_index(m):
    orig = m.rope_kv_store

    def store(q, k, v, positions, cache_rows, theta, k_cache, v_cache):
        return orig(q, k, v, positions, np.arange(len(cache_rows)), theta, k_cache, v_cache)
    m.rope_kv_store = store


def mutant_prefill_offset(m):
    orig = m.rope_split_half

    def rope(x, positions, theta):
        return orig(x, np.asarray(positions) + 1, theta)
    m.rope_split_half = rope


def mutant_softmax_no_shift_sign(m):
    m.softmax = lambda s: np.exp(-s) / np.sum(np.exp(-s), axis=-1, keepdims=True)


def mutant_varlen_mask_ignores_offset(m):
    """The causal mask taken relative to the prompt (query t sees keys 0..t)
    instead of the absolute position offset + t."""
    orig = m.prefill_varlen_gqa_cached_rows

    def varlen(q, k, v, offsets, lengths, cache_rows, theta, scale, k_cache, v_cache, select=None):
        q_rot, out, kc, vc = orig(q, k, v, offsets, lengths, cache_rows, theta, scale, k_cache, v_cache, select)
        A, T, H_q, D = q.shape
        G = H_q // k_cache.shape[1]
        for a in range(A):
            for t in range(int(lengths[a])):
                for h in range(H_q):
                    r, g = int(cache_rows[a]), h // G
                    out[a, t, h] = m.cached_gqa_attention_one(m.bf16_to_f64(q_rot[a, t, h]),
                                                              m.bf16_to_f64(kc[r, g, : t + 1]),
                                                              m.bf16_to_f64(vc[r, g, : t + 1]), scale)
        return q_rot, out, kc, vc
    m.prefill_varlen_gqa_cached_rows = varlen


def mutant_varlen_rope_at_t(m):
    """Tokens rotated at their index in the prompt, not at offset + index."""
    orig = m.prefill_varlen_gqa_cached_rows

    def varlen(q, k, v, offsets, lengths, *rest, **kw):
        return orig(q, k, v, np.zeros_like(np.asarray(offsets)), lengths, *rest, **kw)
    m.prefill_varlen_gqa_cached_rows = varlen


def mutant_f16_double_rounding(m):
    m.f64_to_f16 = lambda x: np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float16).view(np.uint16)


def mutant_f16_no_subnormals(m):
    def f(x):
        x = np.asarray(x, dtype=np.float64)
        _, e = np.frexp(np.abs(x))
        q = e - 11                                  # subnormal spacing forgotten
        y = np.ldexp(np.rint(np.ldexp(np.abs(x), -q)), q)
        y = np.where(y > 65504.0, np.inf, y)
        b = y.astype(np.float16).view(np.uint16)
        return np.where(np.signbit(x), b | np.uint16(0x8000), b).astype(np.uint16)
    m.f64_to_f16 = f


def mutant_f16_read_as_bf16(m):
    m.f16_to_f64 = m.bf16_to_f64


MUTANTS = [mutant_rope_direction, mutant_rope_interleaved, mutant_rope_frequency,
           mutant_gqa_modulo, mutant_exclusive_prefix, mutant_scale_ignored,
           mutant_double_rounding, mutant_prefill_not_causal, mutant_store_row_index,
           mutant_prefill_offset, mutant_softmax_no_shift_sign, mutant_varlen_mask_ignores_offset,
           mutant_varlen_rope_at_t, mutant_f16_double_rounding, mutant_f16_no_subnormals,
           mutant_f16_read_as_bf16]


# Mistakes planted inside a branch of a function (source fragment -> its
# broken form), for branches that no function-level replacement reaches.
SOURCE_MUTANTS = {
    # the per-output chunked prefill drops the prompt's position offset
    "varlen_select_drops_offset": ("p = int(off[a]) + t", "p = t"),
    # the per-output equal-length prefill stops one key early
    "prefill_select_exclusive": ("vc[rows[a], g, :T], t, scale, fmt)", "vc[rows[a], g, :T], max(t - 1, 0), scale, fmt)"),
    # the listed (token, head) pairs read transposed
    "decode_heads_transposed": ("if heads is None else heads", "if heads is None else [(h, a) for a, h in heads]"),
}


def caught_by(m):
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(m)
        except Exception:  # an assertion, or a crash of the broken copy
            caught.append(check.__name__)
    return caught


@pytest.mark.parametrize("mutate", MUTANTS, ids=lambda f: f.__name__)
def test_planted_mistake_is_caught(mutate):
    m = fresh_oracle()
    mutate(m)
    assert caught_by(m), f"no pin catches {mutate.__name__}"


@pytest.mark.parametrize("name", sorted(SOURCE_MUTANTS))
def test_planted_branch_mistake_is_caught(name):
    m = fresh_oracle(SOURCE_MUTANTS[name])
    assert caught_by(m), f"no pin catches {name}"


def test_unpatched_copy_passes_every_pin():
    """The patching loader itself changes nothing: an identity patch passes."""
    m = fresh_oracle(("p = int(off[a]) + t", "p = int(off[a]) + t"))
    assert caught_by(m) == []
