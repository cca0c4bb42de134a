"""Seeded synthetic workloads for the cached GQA + RoPE decode/prefill path.

This module only draws inputs: random BF16 tensors, integer metadata and the
sentinel fill of unused cache cells.  It holds none of the method's arithmetic
(no rotation, no attention, no rounding rule beyond the one torch applies when
an FP32 draw is cast to BF16), so both the CUDA path and the oracle can be fed
from it without sharing any computation.

The five workloads follow the serving situation described in microLLM-rocm
ARCHITECTURE.md, section "Tensor ownership boundary": A survivor tokens with
their own device ``positions[A]`` and ``cache_rows[A]`` over a shared slot KV
cache whose capacity is ``[slots, max_seq]``, plus the equal-length prefill of A
prompts into empty rows.

Cache layout (one layer): K and V are each ``[slots, H_kv, max_seq, D]`` BF16.
Every cell that holds no token is filled with the 16-bit pattern 0x7F7F (a
finite BF16 value of about 3.39e38), so a kernel that reads past a row's prefix
produces a visibly wrong result.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

SENTINEL_BITS = 0x7F7F
BASE_SEED = 20261202


@dataclass(frozen=True)
class DecodeWorkload:
    """One decode step: A active rows of a [slots, max_seq] shared cache."""
    name: str
    index: int
    slots: int
    max_seq: int
    A: int
    H_q: int
    H_kv: int
    D: int
    theta: float
    positions: str          # "fixed" | "uniform" | "loguniform"
    pos_lo: int = 0
    pos_hi: int = 0         # exclusive
    fixed_positions: tuple = ()
    fixed_rows: tuple = ()
    k_head_scale: Optional[tuple] = None   # (lo, hi) of U(lo, hi) per (row, kv head)

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


@dataclass(frozen=True)
class PrefillWorkload:
    """Equal-length prefill of A prompts of T tokens into empty cache rows."""
    name: str
    index: int
    slots: int
    max_seq: int
    A: int
    T: int
    H_q: int
    H_kv: int
    D: int
    theta: float

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


# The five synthetic workloads.  Sizes, position laws and RoPE bases are the
# ones the measured configurations name; theta for the divergent-length case is
# not stated there and takes the Llama-style value of the neighbouring case.
TINY_DECODE = DecodeWorkload(
    name="tiny_decode_s4_a2_hq4_hkv2_d64", index=0, slots=4, max_seq=128, A=2,
    H_q=4, H_kv=2, D=64, theta=10000.0, positions="fixed",
    fixed_positions=(5, 17), fixed_rows=(0, 2))
LLAMA_DECODE = DecodeWorkload(
    name="llama_decode_s64_ms4096_a32_hq32_hkv8_d128", index=1, slots=64,
    max_seq=4096, A=32, H_q=32, H_kv=8, D=128, theta=500000.0,
    positions="uniform", pos_lo=1, pos_hi=4096)
DIVERGENT_DECODE = DecodeWorkload(
    name="divergent_decode_s256_ms8192_a128_hq32_hkv8_d128", index=2, slots=256,
    max_seq=8192, A=128, H_q=32, H_kv=8, D=128, theta=500000.0,
    positions="loguniform", pos_lo=16, pos_hi=8192, k_head_scale=(0.5, 2.0))
LONG_DECODE = DecodeWorkload(
    name="long_decode_s8_ms65536_a8_hq64_hkv8_d128", index=3, slots=8,
    max_seq=65536, A=8, H_q=64, H_kv=8, D=128, theta=1000000.0,
    positions="uniform", pos_lo=32768, pos_hi=65536)
PREFILL = PrefillWorkload(
    name="prefill_a16_t1024_hq32_hkv8_d128_s32_ms2048", index=4, slots=32,
    max_seq=2048, A=16, T=1024, H_q=32, H_kv=8, D=128, theta=500000.0)

DECODE_WORKLOADS = (TINY_DECODE, LLAMA_DECODE, DIVERGENT_DECODE, LONG_DECODE)

# The Llama-style decode workload (same seed: same slots, positions and draws)
# with the other head shapes the kernels take: head width 64, and one query
# head per KV head (multi-head attention, G = 1) at widths 128 and 64.
HEAD_SHAPE_DECODE = tuple(
    DecodeWorkload(name=f"llama_decode_s64_ms4096_a32_hq{hq}_hkv8_d{d}", index=1, slots=64, max_seq=4096, A=32,
                   H_q=hq, H_kv=8, D=d, theta=500000.0, positions="uniform", pos_lo=1, pos_hi=4096)
    for hq, d in ((32, 64), (8, 128), (8, 64)))
ALL_WORKLOADS = DECODE_WORKLOADS + (PREFILL,)


def generator(index: int, salt: int = 0) -> torch.Generator:
    return torch.Generator("cpu").manual_seed(BASE_SEED + index + 1000 * salt)


def randn_bf16(shape, g: torch.Generator, scale: Optional[torch.Tensor] = None) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if scale is not None:
        x = x * scale
    return x.to(torch.bfloat16)


def sentinel_fill(shape, device="cpu") -> torch.Tensor:
    t = torch.empty(*shape, dtype=torch.int16, device=device)
    t.fill_(SENTINEL_BITS)
    return t.view(torch.bfloat16)


@dataclass
class DecodeInputs:
    """Inputs of one decode step, held on the host.

    ``k_prefix[a]`` / ``v_prefix[a]`` hold the cached tokens of active row a,
    shape ``[H_kv, n_a, D]``.  With ``include_current`` the prefix already holds
    position ``positions[a]`` (n_a = p_a + 1) and ``q`` serves directly as the
    rotated query, which is the input of the attention step alone; otherwise
    n_a = p_a and the new token's K/V still have to be stored.
    """
    wl: DecodeWorkload
    q: torch.Tensor            # [A, H_q, D] bf16
    k: torch.Tensor            # [A, H_kv, D] bf16
    v: torch.Tensor            # [A, H_kv, D] bf16
    positions: torch.Tensor    # [A] int32
    cache_rows: torch.Tensor   # [A] int32
    k_prefix: List[torch.Tensor] = field(default_factory=list)
    v_prefix: List[torch.Tensor] = field(default_factory=list)
    include_current: bool = False

    def build_cache(self, device="cpu", rows_subset=None):
        """Full ``[slots, H_kv, max_seq, D]`` K and V caches, sentinel filled,
        with every active prefix scattered into its row (plain copies)."""
        wl = self.wl
        shape = (wl.slots, wl.H_kv, wl.max_seq, wl.D)
        kc = sentinel_fill(shape, device)
        vc = sentinel_fill(shape, device)
        for a in range(wl.A) if rows_subset is None else rows_subset:
            r = int(self.cache_rows[a])
            n = self.k_prefix[a].shape[1]
            if n:
                kc[r, :, :n].copy_(self.k_prefix[a].to(device))
                vc[r, :, :n].copy_(self.v_prefix[a].to(device))
        return kc, vc

    def compact_cache(self, rows, length: Optional[int] = None):
        """Host caches holding only the given active rows, in the given order,
        each ``length`` positions long (sentinel past the prefix).  Row i of the
        result stands for slot ``cache_rows[rows[i]]``."""
        wl = self.wl
        if length is None:
            length = max(int(self.positions[a]) + 1 for a in rows)
        shape = (len(rows), wl.H_kv, length, wl.D)
        kc = sentinel_fill(shape)
        vc = sentinel_fill(shape)
        for i, a in enumerate(rows):
            n = self.k_prefix[a].shape[1]
            kc[i, :, :n] = self.k_prefix[a]
            vc[i, :, :n] = self.v_prefix[a]
        return kc, vc


def draw_positions(wl: DecodeWorkload, g: torch.Generator) -> torch.Tensor:
    if wl.positions == "fixed":
        return torch.tensor(wl.fixed_positions, dtype=torch.int32)
    if wl.positions == "uniform":
        return torch.randint(wl.pos_lo, wl.pos_hi, (wl.A,), generator=g, dtype=torch.int64).to(torch.int32)
    if wl.positions == "loguniform":
        u = torch.rand(wl.A, generator=g, dtype=torch.float64)
        lo, hi = math.log(wl.pos_lo), math.log(wl.pos_hi)
        p = torch.floor(torch.exp(lo + u * (hi - lo))).to(torch.int64)
        return p.clamp(wl.pos_lo, wl.pos_hi - 1).to(torch.int32)
    raise ValueError(wl.positions)


def make_decode_inputs(wl: DecodeWorkload, include_current: bool = False,
                       salt: int = 0) -> DecodeInputs:
    g = generator(wl.index, salt)
    if wl.fixed_rows:
        rows = torch.tensor(wl.fixed_rows, dtype=torch.int32)
    else:
        rows = torch.randperm(wl.slots, generator=g)[: wl.A].to(torch.int32)
    positions = draw_positions(wl, g)
    kscale = None
    if wl.k_head_scale is not None:
        lo, hi = wl.k_head_scale
        kscale = lo + (hi - lo) * torch.rand(wl.A, wl.H_kv, generator=g, dtype=torch.float32)
    q = randn_bf16((wl.A, wl.H_q, wl.D), g)
    k = randn_bf16((wl.A, wl.H_kv, wl.D), g,
                   None if kscale is None else kscale[:, :, None])
    v = randn_bf16((wl.A, wl.H_kv, wl.D), g)
    kp, vp = [], []
    for a in range(wl.A):
        n = int(positions[a]) + (1 if include_current else 0)
        ks = None if kscale is None else kscale[a][:, None, None]
        kp.append(randn_bf16((wl.H_kv, n, wl.D), g, ks))
        vp.append(randn_bf16((wl.H_kv, n, wl.D), g))
    return DecodeInputs(wl, q, k, v, positions, rows, kp, vp, include_current)


@dataclass
class PrefillInputs:
    wl: PrefillWorkload
    q: torch.Tensor           # [A, T, H_q, D] bf16
    k: torch.Tensor           # [A, T, H_kv, D] bf16
    v: torch.Tensor           # [A, T, H_kv, D] bf16
    cache_rows: torch.Tensor  # [A] int32

    def build_cache(self, device="cpu", fill_other_rows: bool = False, salt: int = 7):
        """Empty ``[slots, H_kv, max_seq, D]`` caches (sentinel everywhere).
        With ``fill_other_rows`` the slots that receive no prompt hold random
        BF16 data instead, standing for other requests' live rows."""
        wl = self.wl
        shape = (wl.slots, wl.H_kv, wl.max_seq, wl.D)
        kc = sentinel_fill(shape, device)
        vc = sentinel_fill(shape, device)
        if fill_other_rows:
            g = generator(wl.index, salt)
            used = set(int(r) for r in self.cache_rows)
            for r in range(wl.slots):
                if r not in used:
                    kc[r].copy_(randn_bf16(shape[1:], g).to(device))
                    vc[r].copy_(randn_bf16(shape[1:], g).to(device))
        return kc, vc


def make_prefill_inputs(wl: PrefillWorkload, salt: int = 0) -> PrefillInputs:
    g = generator(wl.index, salt)
    rows = torch.randperm(wl.slots, generator=g)[: wl.A].to(torch.int32)
    q = randn_bf16((wl.A, wl.T, wl.H_q, wl.D), g)
    k = randn_bf16((wl.A, wl.T, wl.H_kv, wl.D), g)
    v = randn_bf16((wl.A, wl.T, wl.H_kv, wl.D), g)
    return PrefillInputs(wl, q, k, v, rows)


NAN_BITS = 0x7FC0  # a quiet NaN in BF16


@dataclass
class VarlenInputs:
    """Prompts of different lengths at their own offsets (chunked prefill).

    Prompt a holds ``lengths[a]`` tokens, padded to T in q/k/v (the padding
    is random too), at positions ``offsets[a]`` .. of row ``cache_rows[a]``,
    whose cells ``[0, offsets[a])`` already hold a random prefix (earlier
    chunks or decode steps)."""
    wl: PrefillWorkload
    q: torch.Tensor           # [A, T, H_q, D] bf16
    k: torch.Tensor           # [A, T, H_kv, D] bf16
    v: torch.Tensor           # [A, T, H_kv, D] bf16
    offsets: torch.Tensor     # [A] int32
    lengths: torch.Tensor     # [A] int32
    cache_rows: torch.Tensor  # [A] int32
    salt: int = 0

    def build_cache(self, device="cpu", tail: str = "sentinel"):
        """``[slots, H_kv, max_seq, D]`` caches: each target row's prefix
        random, the cells from ``offsets[a]`` on ``tail`` ("sentinel" or
        "nan"), every other slot random (other requests' live rows)."""
        wl = self.wl
        shape = (wl.slots, wl.H_kv, wl.max_seq, wl.D)
        g = generator(wl.index, 100 + self.salt)
        kc = randn_bf16(shape, g)
        vc = randn_bf16(shape, g)
        fill = {"sentinel": SENTINEL_BITS, "nan": NAN_BITS}[tail]
        for a in range(self.offsets.shape[0]):
            r, o = int(self.cache_rows[a]), min(max(int(self.offsets[a]), 0), wl.max_seq)
            if 0 <= r < wl.slots:
                kc[r, :, o:].view(torch.int16).fill_(fill)
                vc[r, :, o:].view(torch.int16).fill_(fill)
        return kc.to(device), vc.to(device)


def make_varlen_inputs(wl: PrefillWorkload, offsets, lengths, salt: int = 0, rows=None) -> VarlenInputs:
    g = generator(wl.index, salt)
    perm = torch.randperm(wl.slots, generator=g)[: wl.A].to(torch.int32)
    q = randn_bf16((wl.A, wl.T, wl.H_q, wl.D), g)
    k = randn_bf16((wl.A, wl.T, wl.H_kv, wl.D), g)
    v = randn_bf16((wl.A, wl.T, wl.H_kv, wl.D), g)
    cache_rows = perm if rows is None else torch.tensor(rows, dtype=torch.int32)
    return VarlenInputs(wl, q, k, v, torch.tensor(offsets, dtype=torch.int32),
                        torch.tensor(lengths, dtype=torch.int32), cache_rows, salt)


def random_offsets_lengths(wl: PrefillWorkload, salt: int = 0):
    """A mix of chunk shapes for A prompts: lengths uniform in [1, T], offsets
    uniform in [0, max_seq - length] (a prompt continuing a prefix of any
    size, not aligned to any tile)."""
    g = generator(wl.index, 200 + salt)
    lengths = torch.randint(1, wl.T + 1, (wl.A,), generator=g)
    offsets = torch.stack([torch.randint(0, wl.max_seq - int(n) + 1, (1,), generator=g)[0] for n in lengths])
    return offsets.tolist(), lengths.tolist()


def scaled_decode(wl: DecodeWorkload, **kw) -> DecodeWorkload:
    """A copy of a decode workload with some sizes replaced (test cases)."""
    d = dict(wl.__dict__)
    d.update(kw)
    return DecodeWorkload(**d)


def scaled_prefill(wl: PrefillWorkload, **kw) -> PrefillWorkload:
    d = dict(wl.__dict__)
    d.update(kw)
    return PrefillWorkload(**d)


F16_SENTINEL_BITS = 0x7BFF  # 65504, the largest finite binary16 value


def to_f16(t: torch.Tensor) -> torch.Tensor:
    """The FP16-storage form of a BF16 workload tensor: every value converted
    (BF16 draws of N(0, 1) are binary16 values, except the rare ones below
    2^-14, which round), and unused-cell sentinels mapped to the largest
    finite binary16 value (0x7F7F itself would overflow to infinity)."""
    bits = t.view(torch.int16)
    out = t.to(torch.float16)
    out.view(torch.int16)[bits == SENTINEL_BITS] = F16_SENTINEL_BITS
    return out


def bits16(t: torch.Tensor):
    """16-bit tensor (BF16 or FP16) -> numpy uint16 array of its patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def bf16_bits(t: torch.Tensor):
    """BF16 tensor -> numpy uint16 array of its bit patterns (a view copy)."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def from_bf16_bits(a) -> torch.Tensor:
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
