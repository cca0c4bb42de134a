"""GPU parity of the whole decode step (decode_step_out_, two launches with
an early start, and decode_step_single_launch_out_): the same bytes as
rope_kv_store_out_ followed by cached_gqa_attention_out_ (caches and output),
and the oracle's results, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import DecodeRun, assert_attention_close, assert_ulp, bits, oracle_attention, whole_step

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[False, True], ids=["two_launch", "single_launch"])
def single(request):
    return request.param


def two_call_and_step(inp, single, guard=0):
    """Run the two-call path and the whole step on separate copies of the same
    inputs; return both runs."""
    a = DecodeRun(inp, cache_guard=guard)
    a.store()
    a.attention(q_rot=a.q_out)
    b = DecodeRun(inp, cache_guard=guard)
    whole_step(b, single_launch=single)
    torch.cuda.synchronize()
    return a, b


def assert_same_bytes(a, b, what):
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16)), what + ": K cache differs"
    assert torch.equal(a.v_cache.view(torch.int16), b.v_cache.view(torch.int16)), what + ": V cache differs"
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16)), what + ": output differs"


@pytest.mark.parametrize("wl", [W.TINY_DECODE, W.LLAMA_DECODE, W.DIVERGENT_DECODE], ids=lambda w: w.name)
def test_step_equals_two_calls(wl, single):
    inp = W.make_decode_inputs(wl)
    a, b = two_call_and_step(inp, single)
    assert_same_bytes(a, b, wl.name)
    assert b.kv.kvgqa_read_status(b.ws_step) == 0


def test_step_tiny_against_oracle(single):
    inp = W.make_decode_inputs(W.TINY_DECODE)
    wl = inp.wl
    run = DecodeRun(inp)
    whole_step(run, single_launch=single)
    torch.cuda.synchronize()
    pos = inp.positions.numpy()
    rows = inp.cache_rows.numpy()
    q_rot_o = oracle.rope_split_half_bf16(W.bf16_bits(inp.q), pos[:, None], wl.theta)
    k_rot_o = oracle.rope_split_half_bf16(W.bf16_bits(inp.k), pos[:, None], wl.theta)
    r_t = torch.as_tensor(rows, device="cuda", dtype=torch.long)
    p_t = torch.as_tensor(pos, device="cuda", dtype=torch.long)
    assert_ulp(run.k_cache[r_t, :, p_t], k_rot_o, "k_rot in cache")
    assert np.array_equal(bits(run.v_cache[r_t, :, p_t]), W.bf16_bits(inp.v))
    ref = oracle_attention(inp, list(range(wl.A)), q_rot_bits=q_rot_o, extra_cell=(k_rot_o, W.bf16_bits(inp.v)))
    assert_attention_close(run.out.cpu(), ref, "step tiny")


EDGE_POSITIONS = [0, 1, 2, 7, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 1023]


@pytest.mark.parametrize("D,H_q,H_kv", [(128, 32, 8), (128, 8, 8), (128, 64, 8), (128, 24, 8), (64, 8, 2),
                                         (64, 4, 4), (128, 14, 2)])
def test_step_edge_positions_and_groups(D, H_q, H_kv, single):
    wl = W.DecodeWorkload(name="edge", index=11, slots=24, max_seq=1024, A=len(EDGE_POSITIONS),
                          H_q=H_q, H_kv=H_kv, D=D, theta=10000.0, positions="fixed",
                          fixed_positions=tuple(EDGE_POSITIONS),
                          fixed_rows=tuple(range(23, 23 - len(EDGE_POSITIONS), -1)))
    inp = W.make_decode_inputs(wl)
    a, b = two_call_and_step(inp, single, guard=4096)
    assert_same_bytes(a, b, f"edge D={D} G={H_q // H_kv}")
    assert b.guards_intact()
    # and against the oracle directly
    pos = inp.positions.numpy()
    q_rot_o = oracle.rope_split_half_bf16(W.bf16_bits(inp.q), pos[:, None], wl.theta)
    k_rot_o = oracle.rope_split_half_bf16(W.bf16_bits(inp.k), pos[:, None], wl.theta)
    ref = oracle_attention(inp, list(range(wl.A)), q_rot_bits=q_rot_o, extra_cell=(k_rot_o, W.bf16_bits(inp.v)))
    assert_attention_close(b.out.cpu(), ref, f"step edge D={D} G={H_q // H_kv}")


def test_step_long_context_sampled(single):
    """Long rows split over many CTAs: the cut segments merge, and the cell at
    the last position is written by exactly one CTA before its tile is read."""
    inp = W.make_decode_inputs(W.LONG_DECODE)
    a, b = two_call_and_step(inp, single)
    assert_same_bytes(a, b, "long")


def test_step_invalid_metadata_is_flagged_and_skipped(single):
    wl = W.DecodeWorkload(name="bad", index=13, slots=6, max_seq=256, A=4, H_q=8, H_kv=2, D=128,
                          theta=10000.0, positions="fixed", fixed_positions=(10, 20, 30, 40),
                          fixed_rows=(0, 1, 2, 3))
    inp = W.make_decode_inputs(wl)
    run = DecodeRun(inp)
    run.positions[1] = 256
    run.cache_rows[2] = 6
    run.positions[3] = -1
    k_before, v_before = run.k_cache.clone(), run.v_cache.clone()
    sentinel = torch.full_like(run.out.view(torch.int16), 0x1234)
    run.out.view(torch.int16).copy_(sentinel)
    whole_step(run, single_launch=single)
    assert run.kv.kvgqa_read_status(run.ws_step) == (run.kv.FLAG_POSITION_RANGE | run.kv.FLAG_ROW_RANGE)
    k_before[0, :, 10] = run.k_cache[0, :, 10]
    v_before[0, :, 10] = run.v_cache[0, :, 10]
    assert torch.equal(k_before.view(torch.int16), run.k_cache.view(torch.int16))
    assert torch.equal(v_before.view(torch.int16), run.v_cache.view(torch.int16))
    assert torch.equal(run.out.view(torch.int16)[1:], sentinel[1:])


def test_step_repeats_are_idempotent(single):
    """The bench repeats one step: rewriting the same cells gives the same bytes."""
    inp = W.make_decode_inputs(W.LLAMA_DECODE)
    run = DecodeRun(inp)
    whole_step(run, single_launch=single)
    first_out, first_k = run.out.clone(), run.k_cache.clone()
    whole_step(run, single_launch=single)
    torch.cuda.synchronize()
    assert torch.equal(first_out.view(torch.int16), run.out.view(torch.int16))
    assert torch.equal(first_k.view(torch.int16), run.k_cache.view(torch.int16))


@pytest.mark.parametrize("single", [False, True], ids=["two_launch", "single_launch"])
def test_step_captured_in_a_cuda_graph(single):
    """The whole step, prepared on a stream of its own and captured once as a
    CUDA graph (its programmatic launches included), replays to the same
    caches and output as direct calls, and leaves no status flag."""
    import kv_cached_gqa_rope_gb300 as kv
    inp = W.make_decode_inputs(W.LLAMA_DECODE)
    wl = inp.wl
    a = DecodeRun(inp)
    whole_step(a, single_launch=single)
    torch.cuda.synchronize()
    b = DecodeRun(inp)
    ws = kv.new_workspace(kv.decode_step_workspace_size(wl.A, wl.H_q, wl.H_kv, wl.D))
    s = torch.cuda.Stream()
    call = kv.prepare_decode_step_out_(b.q, b.k, b.v, b.positions, b.cache_rows, wl.theta, wl.scale,
                                       b.k_cache, b.v_cache, b.out, ws, s, single_launch=single)
    with torch.cuda.stream(s):
        call()  # first use outside the capture
    torch.cuda.synchronize()
    b.out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
        call()
    for _ in range(2):
        with torch.cuda.stream(s):
            g.replay()
    torch.cuda.synchronize()
    assert_same_bytes(a, b, "graph replay")
    assert kv.kvgqa_read_status(ws) == 0
