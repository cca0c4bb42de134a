"""GPU parity of the decode step (K1 rope_kv_store, K2+K3 cached attention)
against the FP64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import DecodeRun, assert_attention_close, assert_ulp, bits, oracle_attention

pytestmark = pytest.mark.gpu


def check_store(inp: W.DecodeInputs, run: DecodeRun):
    """K1 against the oracle: q_out and K cells within 1 BF16 ulp, V cells and
    every other cache byte bit-exact."""
    wl = inp.wl
    k_before = run.k_cache.clone()
    v_before = run.v_cache.clone()
    run.store()
    torch.cuda.synchronize()
    pos = inp.positions.numpy()
    rows = inp.cache_rows.numpy()
    q_rot_o = oracle.rope_split_half_bf16(W.bf16_bits(inp.q), pos[:, None], wl.theta)
    k_rot_o = oracle.rope_split_half_bf16(W.bf16_bits(inp.k), pos[:, None], wl.theta)
    assert_ulp(run.q_out, q_rot_o, "q_rot")
    r_t = torch.as_tensor(rows, device="cuda", dtype=torch.long)
    p_t = torch.as_tensor(pos, device="cuda", dtype=torch.long)
    k_cells = run.k_cache[r_t, :, p_t]          # [A, H_kv, D]
    v_cells = run.v_cache[r_t, :, p_t]
    assert_ulp(k_cells, k_rot_o, "k_rot in cache")
    assert np.array_equal(bits(v_cells), W.bf16_bits(inp.v)), "V cells not bit-exact"
    # every other byte untouched: put the new cells into the before-copies
    k_before[r_t, :, p_t] = k_cells
    v_before[r_t, :, p_t] = v_cells
    assert torch.equal(k_before.view(torch.int16), run.k_cache.view(torch.int16)), "K cache bytes changed"
    assert torch.equal(v_before.view(torch.int16), run.v_cache.view(torch.int16)), "V cache bytes changed"
    return q_rot_o, k_rot_o


@pytest.fixture(scope="module")
def tiny():
    return W.make_decode_inputs(W.TINY_DECODE)


def test_store_tiny_whole_cache(tiny):
    run = DecodeRun(tiny)
    check_store(tiny, run)
    # whole-cache comparison with the oracle's own store
    kc, vc = tiny.build_cache()
    q_rot, kc_o, vc_o = oracle.rope_kv_store(W.bf16_bits(tiny.q), W.bf16_bits(tiny.k), W.bf16_bits(tiny.v),
                                             tiny.positions.numpy(), tiny.cache_rows.numpy(),
                                             tiny.wl.theta, W.bf16_bits(kc), W.bf16_bits(vc))
    assert np.array_equal(bits(run.v_cache), vc_o)
    assert oracle.ulp_distance_bf16(bits(run.k_cache), kc_o).max() <= 1
    assert run.status() == (0, 0)


@pytest.mark.parametrize("wl", W.DECODE_WORKLOADS[1:], ids=lambda w: w.name)
def test_store_workloads(wl):
    inp = W.make_decode_inputs(wl)
    run = DecodeRun(inp)
    check_store(inp, run)
    assert run.status()[0] == 0


def test_attention_tiny(tiny):
    inp = W.make_decode_inputs(W.TINY_DECODE, include_current=True)
    run = DecodeRun(inp)
    run.attention()
    torch.cuda.synchronize()
    ref = oracle_attention(inp, list(range(inp.wl.A)))
    assert_attention_close(run.out.cpu(), ref, "tiny attention")
    assert run.status() == (0, 0)


def sampled_rows(inp, k):
    """The k active rows with the longest, the shortest and evenly spread prefixes."""
    order = np.argsort(inp.positions.numpy())
    if k >= len(order):
        return sorted(order.tolist())
    idx = np.unique(np.linspace(0, len(order) - 1, k).round().astype(int))
    return sorted(order[idx].tolist())


@pytest.mark.parametrize("wl,k", [(W.LLAMA_DECODE, 32), (W.DIVERGENT_DECODE, 128), (W.LONG_DECODE, 8)]
                         + [(w, 32) for w in W.HEAD_SHAPE_DECODE],
                         ids=lambda x: getattr(x, "name", str(x)))
def test_attention_workloads(wl, k):
    """Every active row (k = A) and every query head of the decode workloads
    against the oracle, element by element, and row by row."""
    inp = W.make_decode_inputs(wl, include_current=True)
    run = DecodeRun(inp)
    run.attention()
    torch.cuda.synchronize()
    rows = sampled_rows(inp, k)
    assert len(rows) == wl.A
    ref = oracle_attention(inp, rows)
    out = run.out.cpu()[rows]
    assert not np.isnan(ref).any()
    assert_attention_close(out, ref, wl.name)
    for i, a in enumerate(rows):   # a row with a short prefix cannot hide in the average
        assert_attention_close(out[i], ref[i], f"{wl.name} row {a} (position {int(inp.positions[a])})")
    assert run.status() == (0, 0)
    # deterministic: a second call gives the same bytes
    first = run.out.clone()
    run.attention()
    assert torch.equal(first.view(torch.int16), run.out.view(torch.int16))


@pytest.mark.parametrize("wl", [W.TINY_DECODE, W.LLAMA_DECODE], ids=lambda w: w.name)
def test_decode_chain(wl):
    """K1 then K2+K3 on the same buffers versus the oracle chain."""
    inp = W.make_decode_inputs(wl)
    run = DecodeRun(inp)
    q_rot_o, k_rot_o = check_store(inp, run)
    run.attention(q_rot=run.q_out)
    torch.cuda.synchronize()
    rows = list(range(wl.A))
    ref = oracle_attention(inp, rows, q_rot_bits=q_rot_o, extra_cell=(k_rot_o, W.bf16_bits(inp.v)))
    assert_attention_close(run.out.cpu(), ref, wl.name + " chain")


EDGE_POSITIONS = [0, 1, 2, 7, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 1023]


@pytest.mark.parametrize("D,H_q,H_kv", [(128, 32, 8), (128, 8, 8), (128, 16, 8), (128, 64, 8),
                                         (128, 24, 8), (64, 8, 2), (64, 16, 2), (64, 4, 4), (128, 14, 2)])
def test_edge_positions_and_groups(D, H_q, H_kv):
    max_seq = 1024
    wl = W.DecodeWorkload(name="edge", index=11, slots=24, max_seq=max_seq, A=len(EDGE_POSITIONS),
                          H_q=H_q, H_kv=H_kv, D=D, theta=10000.0, positions="fixed",
                          fixed_positions=tuple(EDGE_POSITIONS),
                          fixed_rows=tuple(range(23, 23 - len(EDGE_POSITIONS), -1)))
    inp = W.make_decode_inputs(wl)
    run = DecodeRun(inp, cache_guard=4096)
    q_rot_o, k_rot_o = check_store(inp, run)
    run.attention(q_rot=run.q_out)
    torch.cuda.synchronize()
    ref = oracle_attention(inp, list(range(wl.A)), q_rot_bits=q_rot_o, extra_cell=(k_rot_o, W.bf16_bits(inp.v)))
    assert_attention_close(run.out.cpu(), ref, f"edge D={D} G={H_q // H_kv}")
    assert run.guards_intact()
    assert run.status() == (0, 0)


@pytest.mark.parametrize("step", [False, True], ids=["two_calls", "decode_step"])
def test_max_active_rows(step):
    """The largest batch the decode kernels take (1024 active rows, every
    slot of a 1024-slot cache active, positions spread over the whole row),
    checked in full against the oracle; the whole-step call must give the
    same bytes as the two calls."""
    wl = W.DecodeWorkload(name="max_rows", index=16, slots=1024, max_seq=160, A=1024, H_q=8, H_kv=2, D=64,
                          theta=10000.0, positions="uniform", pos_lo=0, pos_hi=160)
    inp = W.make_decode_inputs(wl)
    run = DecodeRun(inp, cache_guard=4096)
    q_rot_o, k_rot_o = check_store(inp, run)
    run.attention(q_rot=run.q_out)
    torch.cuda.synchronize()
    ref = oracle_attention(inp, list(range(wl.A)), q_rot_bits=q_rot_o, extra_cell=(k_rot_o, W.bf16_bits(inp.v)))
    assert_attention_close(run.out.cpu(), ref, "1024 active rows")
    assert run.guards_intact()
    assert run.status() == (0, 0)
    if step:
        import kv_cached_gqa_rope_gb300 as kv
        kc, vc = inp.build_cache("cuda")
        out2 = torch.empty_like(run.out)
        ws = kv.new_workspace(kv.decode_step_workspace_size(wl.A, wl.H_q, wl.H_kv, wl.D), "cuda")
        kv.decode_step_out_(run.q, run.k, run.v, run.positions, run.cache_rows, wl.theta, wl.scale, kc, vc,
                            out2, ws)
        torch.cuda.synchronize()
        assert kv.kvgqa_read_status(ws) == 0
        assert torch.equal(out2.view(torch.int16), run.out.view(torch.int16))
        assert torch.equal(kc.view(torch.int16), run.k_cache.view(torch.int16))
        assert torch.equal(vc.view(torch.int16), run.v_cache.view(torch.int16))


def test_single_key_returns_v_exactly():
    """Position 0: the only key is the token itself, so out == V bit for bit."""
    wl = W.DecodeWorkload(name="pos0", index=12, slots=8, max_seq=64, A=5, H_q=32, H_kv=8, D=128,
                          theta=500000.0, positions="fixed", fixed_positions=(0,) * 5, fixed_rows=(7, 0, 3, 5, 1))
    inp = W.make_decode_inputs(wl)
    run = DecodeRun(inp)
    run.store()
    run.attention(q_rot=run.q_out)
    torch.cuda.synchronize()
    want = inp.v.repeat_interleave(wl.G, dim=1)
    assert torch.equal(run.out.cpu().view(torch.int16), want.view(torch.int16))


def test_invalid_metadata_is_flagged_and_skipped():
    wl = W.DecodeWorkload(name="bad", index=13, slots=6, max_seq=256, A=4, H_q=8, H_kv=2, D=128,
                          theta=10000.0, positions="fixed", fixed_positions=(10, 20, 30, 40),
                          fixed_rows=(0, 1, 2, 3))
    inp = W.make_decode_inputs(wl)
    run = DecodeRun(inp)
    run.positions[1] = 256          # == max_seq: out of range
    run.cache_rows[2] = 6           # == S: out of range
    run.positions[3] = -1
    k_before, v_before = run.k_cache.clone(), run.v_cache.clone()
    sentinel_out = torch.full_like(run.out.view(torch.int16), 0x1234)
    run.out.view(torch.int16).copy_(sentinel_out)
    run.store()
    run.attention(q_rot=run.q_out)
    flags_store, flags_attn = run.status()
    assert flags_store == (run.kv.FLAG_POSITION_RANGE | run.kv.FLAG_ROW_RANGE)
    assert flags_attn == (run.kv.FLAG_POSITION_RANGE | run.kv.FLAG_ROW_RANGE)
    assert run.status() == (0, 0)                 # reading clears the word
    # only token 0's cells changed
    k_before[0, :, 10] = run.k_cache[0, :, 10]
    v_before[0, :, 10] = run.v_cache[0, :, 10]
    assert torch.equal(k_before.view(torch.int16), run.k_cache.view(torch.int16))
    assert torch.equal(v_before.view(torch.int16), run.v_cache.view(torch.int16))
    # skipped rows leave their outputs unwritten; the valid row is correct
    assert torch.equal(run.out.view(torch.int16)[1:], sentinel_out[1:])
    pos0 = inp.positions.numpy()
    q_rot_o = oracle.rope_split_half_bf16(W.bf16_bits(inp.q), pos0[:, None], wl.theta)
    k_rot_o = oracle.rope_split_half_bf16(W.bf16_bits(inp.k), pos0[:, None], wl.theta)
    ref = oracle_attention(inp, [0], q_rot_bits=q_rot_o, extra_cell=(k_rot_o, W.bf16_bits(inp.v)))
    assert_attention_close(run.out.cpu()[:1], ref, "valid row next to invalid ones")


def test_zero_active_rows_is_noop():
    import kv_cached_gqa_rope_gb300 as kv
    wl = W.DecodeWorkload(name="empty", index=14, slots=2, max_seq=16, A=0, H_q=4, H_kv=2, D=64,
                          theta=10000.0, positions="fixed", fixed_positions=(), fixed_rows=())
    inp = W.make_decode_inputs(wl)
    run = DecodeRun(inp)
    kb = run.k_cache.clone()
    run.store()
    run.attention()
    torch.cuda.synchronize()
    assert torch.equal(kb.view(torch.int16), run.k_cache.view(torch.int16))
    assert run.status() == (0, 0)


def test_host_errors_on_device_tensors():
    import kv_cached_gqa_rope_gb300 as kv
    inp = W.make_decode_inputs(W.TINY_DECODE)
    run = DecodeRun(inp)
    with pytest.raises(kv.KvgqaError) as e:        # a host tensor among device ones
        kv.rope_kv_store_out_(inp.q, run.k, run.v, run.positions, run.cache_rows, 1e4,
                              run.q_out, run.k_cache, run.v_cache, run.ws_store)
    assert e.value.code == "EDEVICE"
    small = kv.new_workspace(256)
    with pytest.raises(kv.KvgqaError) as e:
        kv.cached_gqa_attention_out_(run.q, run.k_cache, run.v_cache, run.positions, run.cache_rows, 0.1,
                                     run.out, small)
    assert e.value.code == "EWORKSPACE"


def test_theta_with_an_infinite_frequency_is_refused():
    """A positive, finite base so small that theta^(-2i/D) overflows: refused
    on the host before anything is queued (the cache keeps its bytes)."""
    import kv_cached_gqa_rope_gb300 as kv
    inp = W.make_decode_inputs(W.TINY_DECODE)
    run = DecodeRun(inp)
    before = run.k_cache.clone()
    with pytest.raises(kv.KvgqaError) as e:
        kv.rope_kv_store_out_(run.q, run.k, run.v, run.positions, run.cache_rows, 1e-320,
                              run.q_out, run.k_cache, run.v_cache, run.ws_store)
    assert e.value.code == "EINVAL"
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int16), run.k_cache.view(torch.int16))
