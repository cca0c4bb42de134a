"""The attention entry point for callers that cannot allocate device memory.

Such callers (code running where cudaMalloc is unavailable or forbidden, or
under a runtime that hands out only its inputs and outputs) cannot provide
the workspace that cached_gqa_attention_out_ needs for its split-K partials.
cached_gqa_attention_static_scratch_out_ keeps those partials in the
library's own static device array instead.  Its result must match the
workspace entry point's, within the attention tolerance of the other tests,
on two calls in a row (the second call reuses the scratch the first one left).

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import DecodeRun, assert_attention_close, oracle_attention

pytestmark = pytest.mark.gpu


def call_static(run: DecodeRun, out: torch.Tensor):
    kv = run.kv
    ds = [kv.describe(t) for t in (run.q, run.k_cache, run.v_cache, run.positions, run.cache_rows)]
    o = kv.describe(out)
    st = kv.library().cached_gqa_attention_static_scratch_out_(
        *(ctypes.byref(d) for d in ds), ctypes.c_float(run.inp.wl.scale), ctypes.byref(o),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, kv.library().kvgqa_last_error()


@pytest.mark.parametrize("wl", [W.LLAMA_DECODE, W.scaled_decode(W.TINY_DECODE, H_q=4, H_kv=4)],
                         ids=["llama_decode", "tiny_G1"])
def test_static_scratch_matches_workspace_entry(wl):
    inp = W.make_decode_inputs(wl, include_current=True)
    run = DecodeRun(inp)
    run.attention()                       # the workspace entry point
    torch.cuda.synchronize()
    want = run.out.clone()
    for call in range(2):                 # two calls in a row on the shared scratch
        got = torch.full_like(run.out, float("nan"))
        call_static(run, got)
        torch.cuda.synchronize()
        mx = (got.float() - want.float()).abs().max().item()
        assert mx <= 1e-2, f"call {call}: max difference {mx} from the workspace entry point"
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    rows = list(range(min(wl.A, 8)))
    assert_attention_close(got.cpu()[rows], oracle_attention(inp, rows), "static scratch vs oracle")


def _zeros(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype, device="cuda")


def test_static_scratch_rejects_too_many_rows():
    """More active rows than the decode kernels take: refused before the
    scratch is considered."""
    import kv_cached_gqa_rope_gb300 as kv
    wl = W.scaled_decode(W.TINY_DECODE, A=3000, slots=3000, max_seq=4)
    q = _zeros(wl.A, wl.H_q, wl.D)
    kc = _zeros(wl.slots, wl.H_kv, wl.max_seq, wl.D)
    pos = _zeros(wl.A, dtype=torch.int32)
    with pytest.raises(kv.KvgqaError) as e:
        kv.cached_gqa_attention_static_scratch_out_(q, kc, kc.clone(), pos, pos.clone(), 0.1, q.clone())
    assert e.value.code == "EUNSUPPORTED"
    assert "active rows" in str(e.value)


def test_static_scratch_rejects_oversize():
    """A legal shape inside the row limit whose counters and partials do not
    fit the 4 MiB static array: 1024 rows x 1024 KV heads need 4 MiB of
    counters alone.  Refused with a message naming the static scratch, and
    nothing is launched (the output keeps its bytes)."""
    import kv_cached_gqa_rope_gb300 as kv
    A, H, D = 1024, 1024, 64
    q = _zeros(A, H, D)
    kc = _zeros(1, H, 1, D)
    pos = _zeros(A, dtype=torch.int32)
    out = torch.full((A, H, D), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kv.KvgqaError) as e:
        kv.cached_gqa_attention_static_scratch_out_(q, kc, kc.clone(), pos, pos.clone(), 0.125, out)
    assert e.value.code == "EUNSUPPORTED"
    assert "static scratch" in str(e.value)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
