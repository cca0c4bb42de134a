"""Shared pieces of the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, and compare with the stated
tolerances."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import workloads as W

# Attention output tolerances versus the FP64 oracle: max-abs and RMS as the
# acceptance bar states them, plus relative RMS.  The GPU result is rounded to
# BF16 once (relative error <= 2^-9, RMS about 2^-9/sqrt(3) of the value) and
# accumulates in FP32 over at most 65536 keys (relative error well below
# 1e-5), so a relative RMS above 5e-3 means a real defect.
MAX_ABS, RMS, REL_RMS = 1e-2, 2e-3, 5e-3


def bits(t: torch.Tensor) -> np.ndarray:
    return W.bf16_bits(t.detach().cpu())


def assert_ulp(gpu_bf16: torch.Tensor, oracle_bits: np.ndarray, what: str, max_ulp: int = 1):
    d = oracle.ulp_distance_bf16(bits(gpu_bf16), oracle_bits)
    assert d.max() <= max_ulp, f"{what}: {int((d > max_ulp).sum())} values beyond {max_ulp} ulp (max {int(d.max())})"


def attention_errors(gpu_bf16: torch.Tensor, ref: np.ndarray, mask=None):
    g = gpu_bf16.detach().float().cpu().numpy().astype(np.float64)
    if mask is not None:
        g, ref = g[mask], ref[mask]
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    err = g - ref
    rms_ref = math.sqrt(float(np.mean(ref * ref)))
    rms = math.sqrt(float(np.mean(err * err)))
    return float(np.max(np.abs(err))), rms, rms / rms_ref


def assert_attention_close(gpu_bf16, ref, what, mask=None):
    mx, rms, rel = attention_errors(gpu_bf16, ref, mask)
    assert mx <= MAX_ABS and rms <= RMS and rel <= REL_RMS, \
        f"{what}: max-abs {mx:.3e} rms {rms:.3e} rel-rms {rel:.3e}"
    return mx, rms, rel


class DecodeRun:
    """Device buffers of one decode step plus the calls of the C ABI."""

    def __init__(self, inp: W.DecodeInputs, device="cuda", cache_guard: int = 0):
        import kv_cached_gqa_rope_gb300 as kv
        self.kv, self.inp, wl = kv, inp, inp.wl
        self.q = inp.q.to(device)
        self.k = inp.k.to(device)
        self.v = inp.v.to(device)
        self.positions = inp.positions.to(device)
        self.cache_rows = inp.cache_rows.to(device)
        kc, vc = inp.build_cache(device)
        self.guard = cache_guard
        if cache_guard:
            # caches as views in the middle of larger sentinel-filled buffers
            n = kc.numel()
            self.kbuf = torch.full((n + 2 * cache_guard,), 0x5A5A, dtype=torch.int16, device=device).view(torch.bfloat16)
            self.vbuf = torch.full((n + 2 * cache_guard,), 0x5A5A, dtype=torch.int16, device=device).view(torch.bfloat16)
            self.kbuf[cache_guard:cache_guard + n] = kc.view(-1)
            self.vbuf[cache_guard:cache_guard + n] = vc.view(-1)
            self.k_cache = self.kbuf[cache_guard:cache_guard + n].view(kc.shape)
            self.v_cache = self.vbuf[cache_guard:cache_guard + n].view(vc.shape)
            del kc, vc
        else:
            self.k_cache, self.v_cache = kc, vc
        self.q_out = torch.empty_like(self.q)
        self.out = torch.empty(wl.A, wl.H_q, wl.D, dtype=torch.bfloat16, device=device)
        self.ws_store = kv.new_workspace(kv.rope_kv_store_workspace_size(), device)
        self.ws_attn = kv.new_workspace(
            kv.cached_gqa_attention_workspace_size(wl.A, wl.H_q, wl.H_kv, wl.D), device)

    def guards_intact(self) -> bool:
        if not self.guard:
            return True
        g = self.guard
        ok = True
        for buf in (self.kbuf, self.vbuf):
            b = buf.view(torch.int16)
            ok &= bool((b[:g] == 0x5A5A).all()) and bool((b[-g:] == 0x5A5A).all())
        return ok

    def store(self):
        self.kv.rope_kv_store_out_(self.q, self.k, self.v, self.positions, self.cache_rows, self.inp.wl.theta,
                                   self.q_out, self.k_cache, self.v_cache, self.ws_store)

    def attention(self, q_rot=None):
        self.kv.cached_gqa_attention_out_(self.q if q_rot is None else q_rot, self.k_cache, self.v_cache,
                                          self.positions, self.cache_rows, self.inp.wl.scale,
                                          self.out, self.ws_attn)

    def status(self):
        return self.kv.kvgqa_read_status(self.ws_store), self.kv.kvgqa_read_status(self.ws_attn)


def oracle_attention(inp: W.DecodeInputs, rows, heads=None, q_rot_bits=None, extra_cell=None):
    """Oracle output for active tokens `rows` (all heads unless `heads` lists
    (row_index_in_rows, h) pairs), from a compact host cache of those rows.
    ``extra_cell`` = (k_rot_bits [A,H_kv,D], v_bits) writes the new token's K/V
    at its position first (the chain case)."""
    wl = inp.wl
    kc, vc = inp.compact_cache(rows)
    kc_b, vc_b = W.bf16_bits(kc), W.bf16_bits(vc)
    pos = inp.positions.numpy()[rows]
    if extra_cell is not None:
        k_rot, v_new = extra_cell
        for i, a in enumerate(rows):
            kc_b[i, :, pos[i]] = k_rot[a]
            vc_b[i, :, pos[i]] = v_new[a]
    q = W.bf16_bits(inp.q)[rows] if q_rot_bits is None else q_rot_bits[rows]
    return oracle.cached_gqa_attention(q, kc_b, vc_b, pos, np.arange(len(rows)), wl.scale, heads=heads)


def whole_step(run: DecodeRun, out=None, ws=None, single_launch=False):
    """decode_step_out_ (or its single-launch form) on the buffers of `run`
    (its own workspace by default)."""
    kv, wl = run.kv, run.inp.wl
    if ws is None:
        if not hasattr(run, "ws_step"):
            run.ws_step = kv.new_workspace(kv.decode_step_workspace_size(wl.A, wl.H_q, wl.H_kv, wl.D))
        ws = run.ws_step
    fn = kv.decode_step_single_launch_out_ if single_launch else kv.decode_step_out_
    fn(run.q, run.k, run.v, run.positions, run.cache_rows, wl.theta, wl.scale,
       run.k_cache, run.v_cache, run.out if out is None else out, ws)
