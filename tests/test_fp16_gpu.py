"""GPU parity of the FP16-storage path (IEEE binary16 Q, K, V, caches and
outputs; FP32 softmax and accumulation) against the FP64 oracle run with
fmt="f16", through the C ABI: the decode store and attention, the whole-step
calls (bit-identical to the two calls), the equal-length prefill and the
prefill of prompts at offsets."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import DecodeRun, assert_attention_close, whole_step

pytestmark = pytest.mark.gpu

F16 = "f16"


def b16(t):
    return W.bits16(t)


def f16_decode_run(inp):
    """A DecodeRun whose 16-bit tensors are all FP16 (same seeded values)."""
    run = DecodeRun(inp)
    run.q, run.k, run.v = (W.to_f16(t) for t in (run.q, run.k, run.v))
    run.k_cache, run.v_cache = W.to_f16(run.k_cache), W.to_f16(run.v_cache)
    run.q_out = torch.empty_like(run.q)
    run.out = torch.empty(inp.wl.A, inp.wl.H_q, inp.wl.D, dtype=torch.float16, device="cuda")
    return run


def test_f16_decode_tiny_against_oracle():
    inp = W.make_decode_inputs(W.TINY_DECODE)
    wl = inp.wl
    run = f16_decode_run(inp)
    kc0, vc0 = b16(run.k_cache), b16(run.v_cache)
    run.store()
    run.attention(q_rot=run.q_out)
    torch.cuda.synchronize()
    pos, rows = inp.positions.numpy(), inp.cache_rows.numpy()
    q_rot, kc, vc = oracle.rope_kv_store(b16(run.q), b16(run.k), b16(run.v), pos, rows, wl.theta, kc0, vc0, fmt=F16)
    assert oracle.ulp_distance_bf16(b16(run.q_out), q_rot).max() <= 1
    assert oracle.ulp_distance_bf16(b16(run.k_cache), kc).max() <= 1
    assert np.array_equal(b16(run.v_cache), vc)
    ref = oracle.cached_gqa_attention(q_rot, kc, vc, pos, rows, wl.scale, fmt=F16)
    assert_attention_close(run.out.cpu(), ref, "f16 decode tiny", fmt="f16")
    assert run.status() == (0, 0)


@pytest.mark.parametrize("wl", [W.LLAMA_DECODE, W.DIVERGENT_DECODE, W.HEAD_SHAPE_DECODE[0]], ids=lambda w: w.name)
def test_f16_decode_workloads_sampled(wl):
    """Full-size decode workloads: the new cells of every active row against
    the oracle's rotation, the output of sampled (row, head) pairs against the
    oracle over those rows' whole prefixes."""
    inp = W.make_decode_inputs(wl)
    run = f16_decode_run(inp)
    run.store()
    run.attention(q_rot=run.q_out)
    torch.cuda.synchronize()
    pos = inp.positions.numpy()
    r_t = inp.cache_rows.long().cuda()
    p_t = inp.positions.long().cuda()
    k_rot = oracle.rope_split_half_bf16(b16(run.k), pos[:, None], wl.theta, fmt=F16)
    q_rot = oracle.rope_split_half_bf16(b16(run.q), pos[:, None], wl.theta, fmt=F16)
    assert oracle.ulp_distance_bf16(b16(run.k_cache[r_t, :, p_t]), k_rot).max() <= 1
    assert np.array_equal(b16(run.v_cache[r_t, :, p_t]), b16(run.v))
    assert oracle.ulp_distance_bf16(b16(run.q_out), q_rot).max() <= 1
    rng = np.random.default_rng(5)
    rows = sorted(rng.choice(wl.A, size=min(6, wl.A), replace=False).tolist())
    kc = b16(run.k_cache[r_t[rows]])                  # compact cache of the sampled rows
    vc = b16(run.v_cache[r_t[rows]])
    heads = [(i, int(h)) for i in range(len(rows)) for h in rng.choice(wl.H_q, size=3, replace=False)]
    ref = oracle.cached_gqa_attention(b16(run.q_out)[rows], kc, vc, pos[rows], np.arange(len(rows)), wl.scale,
                                      heads=heads, fmt=F16)
    got = run.out.float().cpu().numpy()[rows]
    idx = tuple(np.array(heads).T)
    err = np.abs(got[idx] - ref[idx])
    assert np.all(np.isfinite(got[idx]))
    assert err.max() <= 1e-2 and np.sqrt(np.mean(err ** 2)) <= 2e-3, err.max()
    assert run.status() == (0, 0)


@pytest.mark.parametrize("single", [False, True], ids=["two_launch", "single_launch"])
def test_f16_step_equals_two_calls(single):
    inp = W.make_decode_inputs(W.LLAMA_DECODE)
    a = f16_decode_run(inp)
    a.store()
    a.attention(q_rot=a.q_out)
    b = f16_decode_run(inp)
    whole_step(b, single_launch=single)
    torch.cuda.synchronize()
    for x, y, what in ((a.k_cache, b.k_cache, "K cache"), (a.v_cache, b.v_cache, "V cache"), (a.out, b.out, "output")):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16)), what
    assert b.kv.kvgqa_read_status(b.ws_step) == 0


PREFILL_CASES = [
    dict(A=2, T=200, H_q=8, H_kv=2, D=128, slots=4, max_seq=256),
    dict(A=2, T=130, H_q=6, H_kv=2, D=64, slots=3, max_seq=160),
]


@pytest.mark.parametrize("kw", PREFILL_CASES, ids=lambda k: f"T{k['T']}_G{k['H_q'] // k['H_kv']}_D{k['D']}")
def test_f16_prefill_against_oracle(kw):
    import kv_cached_gqa_rope_gb300 as kv
    wl = W.scaled_prefill(W.PREFILL, index=40, **kw)
    pin = W.make_prefill_inputs(wl)
    q, k, v = (W.to_f16(t).cuda() for t in (pin.q, pin.k, pin.v))
    rows = pin.cache_rows.cuda()
    kcb, vcb = pin.build_cache("cuda", fill_other_rows=True)
    kc, vc = W.to_f16(kcb), W.to_f16(vcb)
    kc0, vc0 = b16(kc), b16(vc)
    out = torch.empty(wl.A, wl.T, wl.H_q, wl.D, dtype=torch.float16, device="cuda")
    ws = kv.new_workspace(kv.prefill_gqa_cached_rows_workspace_size(wl.A, wl.T, wl.H_q, wl.H_kv, wl.D))
    kv.prefill_gqa_cached_rows_out_(q, k, v, rows, wl.theta, wl.scale, kc, vc, out, ws)
    torch.cuda.synchronize()
    _, ref, kco, vco = oracle.prefill_gqa_cached_rows(b16(q), b16(k), b16(v), pin.cache_rows.numpy(), wl.theta,
                                                      wl.scale, kc0, vc0, fmt=F16)
    assert oracle.ulp_distance_bf16(b16(kc), kco).max() <= 1
    assert np.array_equal(b16(vc), vco)
    assert_attention_close(out.cpu(), ref, f"f16 prefill {kw}", fmt="f16")
    assert kv.kvgqa_read_status(ws) == 0


def test_f16_varlen_against_oracle():
    import kv_cached_gqa_rope_gb300 as kv
    wl = W.scaled_prefill(W.PREFILL, index=41, A=3, T=160, H_q=8, H_kv=2, D=128, slots=4, max_seq=512)
    inp = W.make_varlen_inputs(wl, [100, 0, 257], [160, 33, 129])
    q, k, v = (W.to_f16(t).cuda() for t in (inp.q, inp.k, inp.v))
    kcb, vcb = inp.build_cache("cuda", tail="sentinel")
    kc, vc = W.to_f16(kcb), W.to_f16(vcb)
    kc0, vc0 = b16(kc), b16(vc)
    out = torch.zeros(wl.A, wl.T, wl.H_q, wl.D, dtype=torch.float16, device="cuda")
    ws = kv.new_workspace(kv.prefill_gqa_cached_rows_workspace_size(wl.A, wl.T, wl.H_q, wl.H_kv, wl.D))
    kv.prefill_varlen_gqa_cached_rows_out_(q, k, v, inp.offsets.cuda(), inp.lengths.cuda(), inp.cache_rows.cuda(),
                                           wl.theta, wl.scale, kc, vc, out, ws)
    torch.cuda.synchronize()
    _, ref, kco, vco = oracle.prefill_varlen_gqa_cached_rows(b16(q), b16(k), b16(v), inp.offsets.numpy(),
                                                             inp.lengths.numpy(), inp.cache_rows.numpy(), wl.theta,
                                                             wl.scale, kc0, vc0, fmt=F16)
    assert oracle.ulp_distance_bf16(b16(kc), kco).max() <= 1
    assert np.array_equal(b16(vc), vco)
    mask = np.zeros(out.shape, dtype=bool)
    for a in range(wl.A):
        mask[a, : int(inp.lengths[a])] = True
    assert_attention_close(out.cpu(), np.nan_to_num(ref), "f16 varlen", mask=mask, fmt="f16")
    assert kv.kvgqa_read_status(ws) == 0
