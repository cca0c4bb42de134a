"""Checks that pin the FP64 oracle to facts other than itself.

Each check takes the oracle module as an argument so that the same check can
be run against deliberately broken copies of the oracle (planted mistakes, on
the CPU) to show that it would catch them.  Every check raises AssertionError
on failure.

Sources of truth used here: closed forms (rotation by a known angle, exact
frequencies for a power-of-two base, two-key softmax as a logistic function,
the mean of V for equal scores), invariants (norm preservation, composition of
rotations, softmax normalisation, causality, untouched cache bytes), special
cases that reduce to a library routine (torch's FP32 -> BF16 rounding), and
brute force in scalar Python loops on tiny inputs.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def rng(seed=0):
    return np.random.default_rng(seed)


def random_bf16_bits(shape, seed=0, scale=1.0):
    x = torch.from_numpy(rng(seed).standard_normal(shape).astype(np.float32) * scale)
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------ BF16 codec
def check_bf16_matches_torch_rounding(o):
    """For FP32-representable inputs, direct FP64->BF16 nearest-even must equal
    torch's FP32->BF16 conversion (a library routine)."""
    r = rng(1)
    bits = r.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    # ties: low 16 bits exactly 0x8000, with even and odd kept mantissas
    ties = (r.integers(0, 2**16, size=20000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    near = np.concatenate([bits, ties, np.array([0x00000001, 0x00008000, 0x00018000, 0x7F7F8000,
                                                 0x7F7FFFFF, 0x7F7F7FFF, 0x80000000, 0x7F800000,
                                                 0xFF800000], dtype=np.uint32)])
    f32 = near.view(np.float32)
    keep = ~np.isnan(f32)
    f32 = f32[keep]
    ref = torch.from_numpy(f32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = o.f64_to_bf16(f32.astype(np.float64))
    assert np.array_equal(got, ref), int(np.sum(got != ref))


def check_bf16_single_rounding(o):
    """Hand-derived: 1 + 2^-8 is a tie (-> even, 1.0); 1 + 3*2^-8 is a tie
    (-> even mantissa, 1 + 2^-6); 1 + 2^-8 + 2^-40 lies above the tie and must
    round up to 1 + 2^-7, which a detour through FP32 (that drops 2^-40) would
    miss."""
    vals = np.array([1 + 2.0**-8, 1 + 3 * 2.0**-8, 1 + 2.0**-8 + 2.0**-40, -(1 + 2.0**-8 + 2.0**-40)])
    want = np.array([0x3F80, 0x3F82, 0x3F81, 0xBF81], dtype=np.uint16)
    assert np.array_equal(o.f64_to_bf16(vals), want)


def check_bf16_roundtrip(o):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = o.bf16_to_f64(allbits)
    ok = ~np.isnan(f)
    assert np.array_equal(o.f64_to_bf16(f[ok]), allbits[ok])
    assert o.bf16_to_f64(np.array([0x3F80], dtype=np.uint16))[0] == 1.0
    assert o.bf16_to_f64(np.array([0x7F7F], dtype=np.uint16))[0] == float.fromhex("0x1.fep127")


# ------------------------------------------------------------------ binary16 codec
def check_f16_matches_torch_rounding(o):
    """For FP32-representable inputs, direct FP64 -> binary16 nearest-even must
    equal torch's FP32 -> FP16 conversion (a library routine), across normal,
    subnormal, overflowing and tie inputs."""
    r = rng(11)
    mags = np.ldexp(r.uniform(1, 2, 150000), r.integers(-30, 18, 150000))
    signs = np.where(r.integers(0, 2, 150000) == 1, -1.0, 1.0)
    x = (signs * mags).astype(np.float32)
    # ties: 12 significant bits with the last set, at normal and subnormal scales
    m = (r.integers(2048, 4096, 20000) | 1).astype(np.float64)
    ties = np.concatenate([np.ldexp(m, r.integers(-20, 5, 20000)), np.ldexp(m, -36)]).astype(np.float32)
    edge = np.array([65504, 65519.99, 65520, 65536, 2.0**-24, 2.0**-25, 3 * 2.0**-26, 2.0**-14,
                     2.0**-14 - 2.0**-25, 0.0, -0.0, np.inf, -np.inf], dtype=np.float32)
    f32 = np.concatenate([x, ties, edge])
    ref = torch.from_numpy(f32.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    got = o.f64_to_f16(f32.astype(np.float64))
    assert np.array_equal(got, ref), int(np.sum(got != ref))


def check_f16_single_rounding(o):
    """Hand-derived: 1 + 2^-11 is a tie (-> even, 1.0); 1 + 3*2^-11 is a tie
    (-> 1 + 2^-9); 1 + 2^-11 + 2^-40 lies above the tie and rounds up to
    1 + 2^-10, which a detour through FP32 (that drops 2^-40) would miss;
    65520 overflows to infinity, 65519.99 does not; 2^-25 is a tie between 0
    and the smallest subnormal (-> 0); 3*2^-26 rounds up to 2^-24."""
    vals = np.array([1 + 2.0**-11, 1 + 3 * 2.0**-11, 1 + 2.0**-11 + 2.0**-40, -(1 + 2.0**-11 + 2.0**-40),
                     65520.0, 65519.99, 2.0**-25, 3 * 2.0**-26])
    want = np.array([0x3C00, 0x3C02, 0x3C01, 0xBC01, 0x7C00, 0x7BFF, 0x0000, 0x0001], dtype=np.uint16)
    assert np.array_equal(o.f64_to_f16(vals), want), o.f64_to_f16(vals)


def check_f16_roundtrip(o):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = o.f16_to_f64(allbits)
    ok = ~np.isnan(f)
    assert np.array_equal(o.f64_to_f16(f[ok]), allbits[ok])
    assert o.f16_to_f64(np.array([0x3C00], dtype=np.uint16))[0] == 1.0
    assert o.f16_to_f64(np.array([0x7BFF], dtype=np.uint16))[0] == 65504.0
    assert o.f16_to_f64(np.array([0x0001], dtype=np.uint16))[0] == 2.0**-24


def check_f16_storage_paths(o):
    """With fmt="f16" the store writes binary16 patterns of the rotated K
    (a unit vector turned by a known angle, so the exact values are cos/sin
    rounded once to binary16) and attention reads the cache as binary16:
    one key returns V exactly, and it equals the BF16 path's result on data
    that both formats hold exactly (small integers)."""
    D, pos, theta = 8, 3, 16.0
    k = np.zeros((1, 1, D))
    k[0, 0, 0] = 1.0
    kb = o.f64_to_f16(k)
    q = o.f64_to_f16(np.zeros((1, 1, D)))
    kc = np.zeros((1, 1, 8, D), dtype=np.uint16)
    vc = np.zeros_like(kc)
    v = o.f64_to_f16(np.arange(D, dtype=np.float64).reshape(1, 1, D))
    _, kc2, vc2 = o.rope_kv_store(q, kb, v, np.array([pos]), np.array([0]), theta, kc, vc, fmt="f16")
    phi = pos * 1.0   # frequency of pair 0 is 1
    want = o.f64_to_f16(np.array([math.cos(phi), 0, 0, 0, math.sin(phi), 0, 0, 0]))
    assert np.array_equal(kc2[0, 0, pos], want)
    assert np.array_equal(vc2[0, 0, pos], v[0, 0])
    out = o.cached_gqa_attention(o.f64_to_f16(np.ones((1, 1, D))), kc2, vc2, np.array([0]), np.array([0]),
                                 0.5, fmt="f16")
    assert np.array_equal(out[0, 0], o.f16_to_f64(vc2[0, 0, 0]))
    ints = np.array([[1.0, -2.0, 3.0, 4.0], [0.5, 2.0, -1.0, 8.0]])
    a16 = o.f64_to_f16(ints)
    a_bf = o.f64_to_bf16(ints)
    assert np.array_equal(o.f16_to_f64(a16), o.bf16_to_f64(a_bf))
    kcx = a16[None, None]                              # [1 slot, 1 kv head, 2 positions, 4]
    kcb = a_bf[None, None]
    qx = np.array([[[1.0, 0.5, -1.0, 2.0]]])
    r16 = o.cached_gqa_attention(o.f64_to_f16(qx), kcx, kcx, np.array([1]), np.array([0]), 0.25, fmt="f16")
    rbf = o.cached_gqa_attention(o.f64_to_bf16(qx), kcb, kcb, np.array([1]), np.array([0]), 0.25)
    assert np.allclose(r16, rbf, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ RoPE
def check_rope_frequencies(o):
    """theta = 16, D = 8 gives frequencies 16^(-2i/8) = 2^-i exactly; theta =
    10000, D = 4 gives 1 and 1/100."""
    assert np.array_equal(o.rope_inv_freq(8, 16.0), np.array([1.0, 0.5, 0.25, 0.125]))
    f = o.rope_inv_freq(4, 10000.0)
    assert f[0] == 1.0 and abs(f[1] - 0.01) < 1e-17


def check_rope_pairing_and_direction(o):
    """A unit vector on dim i turns toward dim i + D/2 by angle pos * 2^-i
    (theta = 16, D = 8): e_i -> cos e_i + sin e_{i+4}; e_{i+4} -> -sin e_i + cos e_{i+4}."""
    D = 8
    for i, pos in [(0, 1), (1, 2), (2, 4), (3, 8), (1, 5)]:
        ang = pos * 2.0**-i
        e = np.zeros(D); e[i] = 1.0
        want = np.zeros(D); want[i] = math.cos(ang); want[i + 4] = math.sin(ang)
        assert np.allclose(o.rope_split_half(e, pos, 16.0), want, atol=1e-15)
        e2 = np.zeros(D); e2[i + 4] = 1.0
        want2 = np.zeros(D); want2[i] = -math.sin(ang); want2[i + 4] = math.cos(ang)
        assert np.allclose(o.rope_split_half(e2, pos, 16.0), want2, atol=1e-15)


def check_rope_identity_at_zero(o):
    x = random_bf16_bits((5, 7, 64), seed=2)
    assert np.array_equal(o.rope_split_half_bf16(x, np.zeros((5, 7)), 10000.0), x)


def check_rope_norm_and_composition(o):
    r = rng(3)
    x = r.standard_normal((64, 128))
    p1 = r.integers(0, 40000, size=64)
    p2 = r.integers(0, 25000, size=64)
    y = o.rope_split_half(x, p1, 500000.0)
    n_in = x[:, :64] ** 2 + x[:, 64:] ** 2
    n_out = y[:, :64] ** 2 + y[:, 64:] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-12, atol=0)
    z = o.rope_split_half(y, p2, 500000.0)
    w = o.rope_split_half(x, p1 + p2, 500000.0)
    assert np.allclose(z, w, rtol=0, atol=1e-9)


def check_rope_matches_complex_rotation(o):
    """Pair (x_i, x_{i+D/2}) read as the complex number x_i + j x_{i+D/2}
    is multiplied by exp(j phi) (numpy's complex exponential)."""
    r = rng(4)
    x = r.standard_normal((16, 64))
    pos = r.integers(0, 65536, size=16)
    phi = pos[:, None] * np.power(10000.0, -np.arange(32) / 32.0)
    zc = (x[:, :32] + 1j * x[:, 32:]) * np.exp(1j * phi)
    y = o.rope_split_half(x, pos, 10000.0)
    assert np.allclose(y[:, :32], zc.real, atol=1e-10) and np.allclose(y[:, 32:], zc.imag, atol=1e-10)


# ------------------------------------------------------------------ K/V store
def check_store_slot_mapping_and_untouched(o):
    S, H_kv, L, D, H_q, A = 6, 2, 16, 8, 4, 3
    kc = random_bf16_bits((S, H_kv, L, D), seed=5)
    vc = random_bf16_bits((S, H_kv, L, D), seed=6)
    q = random_bf16_bits((A, H_q, D), seed=7)
    k = random_bf16_bits((A, H_kv, D), seed=8)
    v = random_bf16_bits((A, H_kv, D), seed=9)
    pos = np.array([0, 7, 15]); rows = np.array([4, 1, 2])
    q_rot, kc2, vc2 = o.rope_kv_store(q, k, v, pos, rows, 16.0, kc, vc)
    touched = np.zeros((S, H_kv, L), dtype=bool)
    for a in range(A):
        touched[rows[a], :, pos[a]] = True
        assert np.array_equal(vc2[rows[a], :, pos[a]], v[a])
        want_k = o.f64_to_bf16(np.stack([o.rope_split_half(o.bf16_to_f64(k[a, g]), pos[a], 16.0)
                                         for g in range(H_kv)]))
        assert np.array_equal(kc2[rows[a], :, pos[a]], want_k)
    assert np.array_equal(kc2[~touched], kc[~touched])
    assert np.array_equal(vc2[~touched], vc[~touched])
    assert np.array_equal(q_rot[0], q[0])          # position 0 rotates by nothing
    assert np.array_equal(kc2[4, :, 0], k[0])


# ------------------------------------------------------------------ attention
def _tiny_cache(S=3, H_kv=2, L=9, D=8, seed=10):
    return (random_bf16_bits((S, H_kv, L, D), seed=seed),
            random_bf16_bits((S, H_kv, L, D), seed=seed + 1))


def check_single_key_returns_v(o):
    kc, vc = _tiny_cache()
    q = random_bf16_bits((2, 4, 8), seed=12)
    out = o.cached_gqa_attention(q, kc, vc, np.array([0, 0]), np.array([2, 0]), 0.35)
    for a, r in enumerate([2, 0]):
        for h in range(4):
            assert np.array_equal(o.f64_to_bf16(out[a, h]), vc[r, h // 2, 0])


def check_equal_scores_give_mean(o):
    kc, vc = _tiny_cache()
    kc = np.zeros_like(kc)                       # every score is 0
    q = random_bf16_bits((1, 4, 8), seed=13)
    out = o.cached_gqa_attention(q, kc, vc, np.array([6]), np.array([1]), 0.35)
    for h in range(4):
        assert np.allclose(out[0, h], o.bf16_to_f64(vc[1, h // 2, :7]).mean(axis=0), atol=1e-15)


def check_two_key_logistic(o):
    """Two keys: out = v0 + (v1 - v0) * sigmoid(scale * (s1 - s0))."""
    D = 4
    kc = np.zeros((1, 1, 2, D), dtype=np.uint16)
    vc = np.zeros((1, 1, 2, D), dtype=np.uint16)
    k0 = np.array([1.0, 0, 0, 0]); k1 = np.array([0, 2.0, 0, 0])
    v0 = np.array([1.0, -2.0, 0.5, 0]); v1 = np.array([0.25, 4.0, -1.0, 3.0])
    kc[0, 0, 0] = o.f64_to_bf16(k0); kc[0, 0, 1] = o.f64_to_bf16(k1)
    vc[0, 0, 0] = o.f64_to_bf16(v0); vc[0, 0, 1] = o.f64_to_bf16(v1)
    qv = np.array([0.5, 1.5, 0, 0])
    q = o.f64_to_bf16(qv)[None, None]
    scale = 0.75
    d = scale * (qv @ k1 - qv @ k0)
    want = v0 + (v1 - v0) / (1.0 + math.exp(-d))
    out = o.cached_gqa_attention(q, kc, vc, np.array([1]), np.array([0]), scale)
    assert np.allclose(out[0, 0], want, atol=1e-14)


def check_softmax_normalised(o):
    s = rng(14).standard_normal((5, 333)) * 30
    p = o.kvgqa_oracle.softmax(s) if hasattr(o, "kvgqa_oracle") else o.softmax(s)
    assert np.allclose(p.sum(axis=-1), 1.0, atol=1e-12) and np.all(p >= 0)


def check_brute_force_tiny(o):
    """Scalar Python loops with math.exp on a D=4, 3-key, G=2 case."""
    S, H_kv, L, D, H_q = 2, 2, 4, 4, 4
    kc, vc = _tiny_cache(S, H_kv, L, D, seed=15)
    q = random_bf16_bits((1, H_q, D), seed=17)
    scale = 0.5
    out = o.cached_gqa_attention(q, kc, vc, np.array([2]), np.array([1]), scale)
    f = lambda b: float(o.bf16_to_f64(np.array([b], dtype=np.uint16))[0])
    for h in range(H_q):
        g = h // 2
        scores = []
        for j in range(3):
            acc = 0.0
            for d in range(D):
                acc += f(q[0, h, d]) * f(kc[1, g, j, d])
            scores.append(acc * scale)
        m = max(scores)
        w = [math.exp(sv - m) for sv in scores]
        tot = sum(w)
        for d in range(D):
            want = sum(w[j] * f(vc[1, g, j, d]) for j in range(3)) / tot
            assert abs(out[0, h, d] - want) < 1e-13


def check_gqa_equals_repeated_mha(o):
    S, H_kv, L, D, G = 3, 2, 12, 8, 3
    kc, vc = _tiny_cache(S, H_kv, L, D, seed=18)
    q = random_bf16_bits((2, H_kv * G, D), seed=20)
    pos, rows = np.array([11, 4]), np.array([2, 0])
    out = o.cached_gqa_attention(q, kc, vc, pos, rows, 0.3)
    out_mha = o.cached_gqa_attention(q, np.repeat(kc, G, axis=1), np.repeat(vc, G, axis=1),
                                     pos, rows, 0.3)
    assert np.array_equal(out, out_mha)
    # and the heads of one group really do differ from another group's
    assert not np.allclose(out[0, 0], out[0, G])


def check_prefix_is_inclusive_and_bounded(o):
    """Keys past the position are not read; the key at the position is."""
    kc, vc = _tiny_cache(seed=21)
    q = random_bf16_bits((1, 4, 8), seed=23)
    out1 = o.cached_gqa_attention(q, kc, vc, np.array([4]), np.array([1]), 0.35)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[1, :, 5:] = 0x7F7F; vc2[1, :, 5:] = 0x7F7F
    out2 = o.cached_gqa_attention(q, kc2, vc2, np.array([4]), np.array([1]), 0.35)
    assert np.array_equal(out1, out2)
    vc3 = vc.copy(); vc3[1, :, 4] = 0
    out3 = o.cached_gqa_attention(q, kc, vc3, np.array([4]), np.array([1]), 0.35)
    assert not np.allclose(out1, out3)


# ------------------------------------------------------------------ prefill
def _prefill_case(A=2, T=6, H_q=4, H_kv=2, D=8, S=4, L=10, seed=30):
    q = random_bf16_bits((A, T, H_q, D), seed=seed)
    k = random_bf16_bits((A, T, H_kv, D), seed=seed + 1)
    v = random_bf16_bits((A, T, H_kv, D), seed=seed + 2)
    kc = np.full((S, H_kv, L, D), 0x7F7F, dtype=np.uint16)
    vc = np.full((S, H_kv, L, D), 0x7F7F, dtype=np.uint16)
    return q, k, v, kc, vc


def check_prefill_rows_and_first_position(o):
    q, k, v, kc, vc = _prefill_case()
    rows = np.array([3, 0])
    q_rot, out, kc2, vc2 = o.prefill_gqa_cached_rows(q, k, v, rows, 16.0, 0.4, kc, vc)
    for a in range(2):
        r = rows[a]
        assert np.array_equal(vc2[r, :, :6], np.transpose(v[a], (1, 0, 2)))
        assert np.array_equal(kc2[r, :, 0], k[a, 0])        # position 0 is unrotated
        for h in range(4):                                   # position 0 sees only itself
            assert np.array_equal(o.f64_to_bf16(out[a, 0, h]), v[a, 0, h // 2])
    untouched = np.ones(kc.shape[:3], dtype=bool)
    untouched[rows, :, :6] = False
    assert np.array_equal(kc2[untouched], kc[untouched])
    assert np.array_equal(vc2[untouched], vc[untouched])


def check_prefill_causal(o):
    q, k, v, kc, vc = _prefill_case(seed=40)
    rows = np.array([1, 2])
    _, out, _, _ = o.prefill_gqa_cached_rows(q, k, v, rows, 16.0, 0.4, kc, vc)
    k2, v2 = k.copy(), v.copy()
    k2[:, 4:] = random_bf16_bits(k2[:, 4:].shape, seed=99)
    v2[:, 4:] = random_bf16_bits(v2[:, 4:].shape, seed=98)
    _, out2, _, _ = o.prefill_gqa_cached_rows(q, k2, v2, rows, 16.0, 0.4, kc, vc)
    assert np.array_equal(out[:, :4], out2[:, :4])
    assert not np.allclose(out[:, 4:], out2[:, 4:])


def check_prefill_matches_decode(o):
    """Decoding the token at position p after prefilling positions 0..p-1 gives
    the same result as row p of one prefill of positions 0..T-1."""
    A, T, H_q, H_kv, D = 2, 7, 4, 2, 8
    q, k, v, kc, vc = _prefill_case(A, T, H_q, H_kv, D, seed=50)
    rows = np.array([2, 0])
    _, out_full, _, _ = o.prefill_gqa_cached_rows(q, k, v, rows, 16.0, 0.4, kc, vc)
    for p in (1, 3, 6):
        _, _, kcp, vcp = o.prefill_gqa_cached_rows(q[:, :p], k[:, :p], v[:, :p], rows, 16.0, 0.4, kc, vc)
        pos = np.full(A, p)
        q_rot, kc3, vc3 = o.rope_kv_store(q[:, p], k[:, p], v[:, p], pos, rows, 16.0, kcp, vcp)
        out = o.cached_gqa_attention(q_rot, kc3, vc3, pos, rows, 0.4)
        assert np.allclose(out, out_full[:, p], rtol=0, atol=1e-13)


def check_prefill_select_matches_full(o):
    q, k, v, kc, vc = _prefill_case(seed=60)
    rows = np.array([0, 3])
    _, full, _, _ = o.prefill_gqa_cached_rows(q, k, v, rows, 16.0, 0.4, kc, vc)
    sel = [(0, 0, 0), (1, 5, 3), (0, 3, 2)]
    _, part, _, _ = o.prefill_gqa_cached_rows(q, k, v, rows, 16.0, 0.4, kc, vc, select=sel)
    for a, t, h in sel:
        assert np.allclose(part[a, t, h], full[a, t, h], rtol=0, atol=1e-14)


def check_varlen_select_matches_full(o):
    """The per-output path of the chunked prefill (``select``) gives the values
    of the whole-prompt path for prompts at nonzero offsets and of different
    lengths; an output past its prompt's length stays NaN in both."""
    A, T, H_q, H_kv, D, S, L = 3, 6, 4, 2, 8, 5, 14
    q, k, v, _, _ = _prefill_case(A, T, H_q, H_kv, D, S, L, seed=110)
    kc = random_bf16_bits((S, H_kv, L, D), seed=111)
    vc = random_bf16_bits((S, H_kv, L, D), seed=112)
    rows, offs, lens = np.array([3, 0, 4]), np.array([0, 5, 8]), np.array([6, 2, 4])
    _, full, kc1, vc1 = o.prefill_varlen_gqa_cached_rows(q, k, v, offs, lens, rows, 16.0, 0.4, kc, vc)
    sel = [(a, t, h) for a in range(A) for t in range(T) for h in range(H_q)]
    _, part, kc2, vc2 = o.prefill_varlen_gqa_cached_rows(q, k, v, offs, lens, rows, 16.0, 0.4, kc, vc, select=sel)
    assert np.array_equal(kc1, kc2) and np.array_equal(vc1, vc2)
    assert np.array_equal(np.isnan(part), np.isnan(full))
    seen = ~np.isnan(full)
    assert seen.sum() == int(np.sum(lens)) * H_q * D
    assert np.allclose(part[seen], full[seen], rtol=0, atol=1e-13)


def check_decode_heads_matches_full(o):
    """Attention of listed (token, head) pairs (``heads``) equals those entries
    of the call over every pair; the unlisted entries stay NaN."""
    kc, vc = _tiny_cache(S=3, H_kv=2, L=9, D=8, seed=120)
    q = random_bf16_bits((3, 4, 8), seed=121)
    pos, rows = np.array([8, 0, 4]), np.array([2, 0, 1])
    full = o.cached_gqa_attention(q, kc, vc, pos, rows, 0.3)
    heads = [(2, 3), (0, 1), (1, 0), (0, 2)]
    part = o.cached_gqa_attention(q, kc, vc, pos, rows, 0.3, heads=heads)
    listed = np.zeros((3, 4), dtype=bool)
    for a, h in heads:
        listed[a, h] = True
        assert np.array_equal(part[a, h], full[a, h])
    assert np.all(np.isnan(part[~listed]))


def check_varlen_equal_lengths_is_prefill(o):
    """Zero offsets and full lengths: the equal-length prefill."""
    q, k, v, kc, vc = _prefill_case(seed=70)
    rows = np.array([1, 3])
    A, T = q.shape[:2]
    qr1, out1, kc1, vc1 = o.prefill_gqa_cached_rows(q, k, v, rows, 16.0, 0.4, kc, vc)
    qr2, out2, kc2, vc2 = o.prefill_varlen_gqa_cached_rows(q, k, v, np.zeros(A, int), np.full(A, T), rows, 16.0,
                                                            0.4, kc, vc)
    assert np.array_equal(qr1, qr2) and np.array_equal(kc1, kc2) and np.array_equal(vc1, vc2)
    assert np.allclose(out1, out2, rtol=0, atol=1e-13)


def check_varlen_length_one_is_decode(o):
    """One token at offset p: the decode step at position p (store, then
    attention over keys 0..p of the row)."""
    A, T, H_q, H_kv, D, S, L = 3, 4, 4, 2, 8, 5, 12
    q, k, v, _, _ = _prefill_case(A, T, H_q, H_kv, D, S, L, seed=80)
    kc = random_bf16_bits((S, H_kv, L, D), seed=81)
    vc = random_bf16_bits((S, H_kv, L, D), seed=82)
    rows = np.array([4, 0, 2])
    offs = np.array([0, 5, 11])
    qr, out, kc2, vc2 = o.prefill_varlen_gqa_cached_rows(q, k, v, offs, np.ones(A, int), rows, 16.0, 0.4, kc, vc)
    q_rot, kc3, vc3 = o.rope_kv_store(q[:, 0], k[:, 0], v[:, 0], offs, rows, 16.0, kc, vc)
    ref = o.cached_gqa_attention(q_rot, kc3, vc3, offs, rows, 0.4)
    assert np.array_equal(kc2, kc3) and np.array_equal(vc2, vc3) and np.array_equal(qr[:, 0], q_rot)
    assert np.allclose(out[:, 0], ref, rtol=0, atol=1e-13)
    assert np.all(np.isnan(out[:, 1:]))


def check_varlen_chunks_compose(o):
    """Prefilling L1 tokens and then the next L2 at offset L1 gives the same
    cache and the same outputs as one prefill of L1 + L2 tokens; prompts of
    different lengths in one call behave as separate calls."""
    A, T, H_q, H_kv, D, S, L = 2, 7, 4, 2, 8, 4, 12
    q, k, v, kc, vc = _prefill_case(A, T, H_q, H_kv, D, S, L, seed=90)
    rows = np.array([2, 1])
    _, out_full, kcf, vcf = o.prefill_gqa_cached_rows(q, k, v, rows, 16.0, 0.4, kc, vc)
    L1 = np.array([3, 5])
    _, out1, kc1, vc1 = o.prefill_varlen_gqa_cached_rows(q, k, v, np.zeros(A, int), L1, rows, 16.0, 0.4, kc, vc)
    q2 = np.zeros_like(q); k2 = np.zeros_like(k); v2 = np.zeros_like(v)
    for a in range(A):
        n = T - L1[a]
        q2[a, :n], k2[a, :n], v2[a, :n] = q[a, L1[a]:], k[a, L1[a]:], v[a, L1[a]:]
    _, out2, kc2, vc2 = o.prefill_varlen_gqa_cached_rows(q2, k2, v2, L1, T - L1, rows, 16.0, 0.4, kc1, vc1)
    assert np.array_equal(kc2, kcf) and np.array_equal(vc2, vcf)
    for a in range(A):
        assert np.allclose(out1[a, :L1[a]], out_full[a, :L1[a]], rtol=0, atol=1e-13)
        assert np.allclose(out2[a, :T - L1[a]], out_full[a, L1[a]:], rtol=0, atol=1e-13)
    # bytes past each prompt's tokens untouched
    untouched = np.ones(kc.shape[:3], dtype=bool)
    for a in range(A):
        untouched[rows[a], :, :L1[a]] = False
    assert np.array_equal(kc1[untouched], kc[untouched]) and np.array_equal(vc1[untouched], vc[untouched])


ALL_CHECKS = [
    check_bf16_matches_torch_rounding, check_bf16_single_rounding, check_bf16_roundtrip,
    check_f16_matches_torch_rounding, check_f16_single_rounding, check_f16_roundtrip, check_f16_storage_paths,
    check_rope_frequencies, check_rope_pairing_and_direction, check_rope_identity_at_zero,
    check_rope_norm_and_composition, check_rope_matches_complex_rotation,
    check_store_slot_mapping_and_untouched, check_single_key_returns_v,
    check_equal_scores_give_mean, check_two_key_logistic, check_softmax_normalised,
    check_brute_force_tiny, check_gqa_equals_repeated_mha, check_prefix_is_inclusive_and_bounded,
    check_prefill_rows_and_first_position, check_prefill_causal, check_prefill_matches_decode,
    check_prefill_select_matches_full, check_varlen_equal_lengths_is_prefill, check_varlen_length_one_is_decode,
    check_varlen_chunks_compose, check_varlen_select_matches_full, check_decode_heads_matches_full,
]
