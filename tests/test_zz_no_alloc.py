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

from kv_cached_gqa_rope_gb300 import workloads as W
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


def test_static_scratch_rejects_oversize():
    import kv_cached_gqa_rope_gb300 as kv
    wl = W.scaled_decode(W.TINY_DECODE, A=3000, slots=3000, max_seq=4)   # beyond the active-row limit
    q = torch.zeros(wl.A, wl.H_q, wl.D, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(wl.slots, wl.H_kv, wl.max_seq, wl.D, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(wl.A, dtype=torch.int32, device="cuda")
    with pytest.raises(kv.KvgqaError) as e:
        kv.cached_gqa_attention_static_scratch_out_(q, kc, kc.clone(), pos, pos.clone(), 0.1, q.clone())
    assert e.value.code == "EUNSUPPORTED"
