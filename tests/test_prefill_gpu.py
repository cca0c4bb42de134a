"""GPU parity of the equal-length prefill into empty rows (K1 in prefill mode
+ K4 tcgen05 causal attention) against the FP64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_attention_close, bits

pytestmark = pytest.mark.gpu


class PrefillRun:
    def __init__(self, pin: W.PrefillInputs, fill_other_rows=True):
        import kv_cached_gqa_rope_gb300 as kv
        self.kv, self.pin, wl = kv, pin, pin.wl
        self.q, self.k, self.v = pin.q.cuda(), pin.k.cuda(), pin.v.cuda()
        self.rows = pin.cache_rows.cuda()
        self.k_cache, self.v_cache = pin.build_cache("cuda", fill_other_rows=fill_other_rows)
        self.k0, self.v0 = self.k_cache.clone(), self.v_cache.clone()
        self.out = torch.empty(wl.A, wl.T, wl.H_q, wl.D, dtype=torch.bfloat16, device="cuda")
        self.ws = kv.new_workspace(kv.prefill_gqa_cached_rows_workspace_size(wl.A, wl.T, wl.H_q, wl.H_kv, wl.D))

    def run(self):
        wl = self.pin.wl
        self.kv.prefill_gqa_cached_rows_out_(self.q, self.k, self.v, self.rows, wl.theta, wl.scale,
                                             self.k_cache, self.v_cache, self.out, self.ws)
        torch.cuda.synchronize()


def check_cache(run: PrefillRun):
    """Target rows [0, T) hold rotated K (<= 1 ulp) and V (bit-exact); every
    other byte of both caches is unchanged."""
    pin, wl = run.pin, run.pin.wl
    pos = np.arange(wl.T)
    k_rot = oracle.rope_split_half_bf16(W.bf16_bits(pin.k), pos[None, :, None], wl.theta)  # [A,T,H_kv,D]
    rows = pin.cache_rows.long().cuda()
    k_cells = run.k_cache[rows, :, : wl.T]        # [A, H_kv, T, D]
    v_cells = run.v_cache[rows, :, : wl.T]
    d = oracle.ulp_distance_bf16(bits(k_cells), np.transpose(k_rot, (0, 2, 1, 3)))
    assert d.max() <= 1, f"K cells beyond 1 ulp: {int((d > 1).sum())}"
    assert np.array_equal(bits(v_cells), np.transpose(W.bf16_bits(pin.v), (0, 2, 1, 3)))
    k0, v0 = run.k0, run.v0
    k0[rows, :, : wl.T] = k_cells
    v0[rows, :, : wl.T] = v_cells
    assert torch.equal(k0.view(torch.int16), run.k_cache.view(torch.int16)), "K cache bytes outside the prompts changed"
    assert torch.equal(v0.view(torch.int16), run.v_cache.view(torch.int16)), "V cache bytes outside the prompts changed"


def oracle_prefill(pin: W.PrefillInputs, select=None):
    wl = pin.wl
    # the oracle only needs the target rows: a compact cache whose row i is slot rows[i]
    kc = np.full((wl.A, wl.H_kv, wl.T, wl.D), 0x7F7F, dtype=np.uint16)
    vc = kc.copy()
    _, out, _, _ = oracle.prefill_gqa_cached_rows(W.bf16_bits(pin.q), W.bf16_bits(pin.k), W.bf16_bits(pin.v),
                                                  np.arange(wl.A), wl.theta, wl.scale, kc, vc, select=select)
    return out


SMALL = [
    dict(A=2, T=40, H_q=8, H_kv=2, D=128, slots=4, max_seq=64),
    dict(A=3, T=128, H_q=4, H_kv=4, D=128, slots=5, max_seq=128),
    dict(A=2, T=129, H_q=8, H_kv=1, D=128, slots=3, max_seq=200),
    dict(A=1, T=255, H_q=16, H_kv=2, D=128, slots=2, max_seq=256),
    dict(A=2, T=300, H_q=6, H_kv=2, D=64, slots=4, max_seq=320),
    dict(A=2, T=160, H_q=8, H_kv=2, D=64, slots=3, max_seq=192),  # D = 64 with head pairs
    dict(A=1, T=1, H_q=4, H_kv=2, D=64, slots=2, max_seq=8),
]


@pytest.mark.parametrize("kw", SMALL, ids=lambda k: f"A{k['A']}_T{k['T']}_G{k['H_q'] // k['H_kv']}_D{k['D']}")
def test_prefill_small_full(kw):
    wl = W.scaled_prefill(W.PREFILL, index=20, **kw)
    pin = W.make_prefill_inputs(wl)
    run = PrefillRun(pin)
    run.run()
    check_cache(run)
    ref = oracle_prefill(pin)
    assert_attention_close(run.out.cpu(), ref, f"prefill {kw}")
    assert run.kv.kvgqa_read_status(run.ws) == 0


def test_prefill_first_position_is_v():
    """Row 0 attends to itself only: out[:, 0, h] == V[:, 0, h // G] bit for bit."""
    wl = W.scaled_prefill(W.PREFILL, index=21, A=3, T=130, H_q=16, H_kv=4, D=128, slots=4, max_seq=256)
    pin = W.make_prefill_inputs(wl)
    run = PrefillRun(pin)
    run.run()
    want = pin.v[:, 0].repeat_interleave(wl.G, dim=1)
    assert torch.equal(run.out[:, 0].cpu().view(torch.int16), want.view(torch.int16))


def test_prefill_full_workload():
    """16 prompts x 1024 tokens, H_q 32 / H_kv 8, D 128: the whole cache and
    every one of the 67M output values against the oracle, element by
    element; a second call gives the same bytes."""
    wl = W.PREFILL
    pin = W.make_prefill_inputs(wl)
    run = PrefillRun(pin, fill_other_rows=True)
    run.run()
    check_cache(run)
    ref = oracle_prefill(pin)
    assert not np.isnan(ref).any()
    assert_attention_close(run.out.cpu(), ref, "prefill 16x1024, every output")
    # per prompt too, so that a wrong prompt cannot hide in the average
    for a in range(wl.A):
        assert_attention_close(run.out[a].cpu(), ref[a], f"prefill 16x1024, prompt {a}")
    del ref
    first = run.out.clone()
    run.run()
    assert torch.equal(first.view(torch.int16), run.out.view(torch.int16))
    assert run.kv.kvgqa_read_status(run.ws) == 0


def test_prefill_invalid_row_flagged():
    wl = W.scaled_prefill(W.PREFILL, index=22, A=2, T=64, H_q=8, H_kv=2, D=128, slots=3, max_seq=64)
    pin = W.make_prefill_inputs(wl)
    run = PrefillRun(pin)
    run.rows[1] = 7
    run.out.view(torch.int16).fill_(0x1234)
    run.run()
    assert run.kv.kvgqa_read_status(run.ws) == run.kv.FLAG_ROW_RANGE
    assert bool((run.out[1].view(torch.int16) == 0x1234).all())   # skipped prompt untouched
    r0 = int(pin.cache_rows[0])
    ref = oracle_prefill(W.PrefillInputs(W.scaled_prefill(wl, A=1), pin.q[:1], pin.k[:1], pin.v[:1],
                                         pin.cache_rows[:1]))
    assert_attention_close(run.out[:1].cpu(), ref, "valid prompt next to an invalid one")
    k0 = run.k0
    k0[r0, :, : wl.T] = run.k_cache[r0, :, : wl.T]
    assert torch.equal(k0.view(torch.int16), run.k_cache.view(torch.int16))


def test_prefill_output_16_byte_aligned():
    """The output only needs 16-byte alignment: an output that starts 16 bytes
    past a 32-byte boundary (whose rows then take 16-byte stores instead of
    whole 32-byte sectors) gets the same bytes as an aligned one, and nothing
    around it is written."""
    pw = W.scaled_prefill(W.PREFILL, A=2, T=200, H_q=8, H_kv=2, D=128, slots=3, max_seq=256)
    pin = W.make_prefill_inputs(pw)
    a = PrefillRun(pin)
    a.run()
    b = PrefillRun(pin)
    n = a.out.numel()
    big = torch.full((n + 32,), 7.0, dtype=torch.bfloat16, device="cuda")
    b.out = big[8:8 + n].view(a.out.shape)  # 16 bytes past the allocation's start
    assert b.out.data_ptr() % 32 == 16
    b.run()
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert bool((big[:8] == 7.0).all()) and bool((big[8 + n:] == 7.0).all())
