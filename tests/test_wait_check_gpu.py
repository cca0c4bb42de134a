"""The bounded waits end on the GPU: a kernel whose only wait can never
complete gives up after the wait's bound, reports KVGQA_FLAG_TIMEOUT through
the workspace status word, frees its tensor memory and returns; the context
stays usable, so a decode step right after it still matches the oracle.
Nothing here faults, traps or spins without limit."""
import time

import pytest
import torch

import kv_cached_gqa_rope_gb300 as kv
import oracle
import workloads as W
from gpu_helpers import DecodeRun, assert_attention_close, oracle_attention

pytestmark = pytest.mark.gpu


def test_wait_gives_up_and_context_stays_usable():
    ws = kv.new_workspace(kv.STATUS_BYTES)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kv.kvgqa_check_bounded_wait(ws)
    flags = kv.kvgqa_read_status(ws)   # synchronises
    waited = time.perf_counter() - t0
    assert flags == kv.FLAG_TIMEOUT
    assert 1.5 < waited < 30.0, f"the wait ended after {waited:.2f} s (bound: 2 s)"
    assert kv.kvgqa_read_status(ws) == 0  # read_status clears the word

    # the same context runs a decode step correctly afterwards
    inp = W.make_decode_inputs(W.TINY_DECODE)
    run = DecodeRun(inp)
    run.store()
    run.attention(q_rot=run.q_out)
    torch.cuda.synchronize()
    pos = inp.positions.numpy()
    q_rot_o = oracle.rope_split_half_bf16(W.bf16_bits(inp.q), pos[:, None], inp.wl.theta)
    k_rot_o = oracle.rope_split_half_bf16(W.bf16_bits(inp.k), pos[:, None], inp.wl.theta)
    ref = oracle_attention(inp, list(range(inp.wl.A)), q_rot_bits=q_rot_o, extra_cell=(k_rot_o, W.bf16_bits(inp.v)))
    assert_attention_close(run.out.cpu(), ref, "decode after the bounded-wait check")
    assert run.status() == (0, 0)


def test_wait_check_rejects_host_workspace():
    raw = torch.zeros(512, dtype=torch.uint8)      # a 256-byte aligned host buffer
    off = (-raw.data_ptr()) % 256
    with pytest.raises(kv.KvgqaError) as e:
        kv.kvgqa_check_bounded_wait(raw[off:off + 256])
    assert e.value.code == "EDEVICE"


def test_timeout_status_read_restores_the_workspace():
    """A decode call whose bounded wait gave up leaves the status word with
    KVGQA_FLAG_TIMEOUT and may leave split-K counters short of their count.
    That state is made on the host here (a set timeout bit and non-zero
    counters written into the workspace): reading the status returns the
    flag and zero-fills the workspace, after which an attention call on it
    matches the oracle."""
    inp = W.make_decode_inputs(W.LLAMA_DECODE, include_current=True)
    run = DecodeRun(inp)
    ws = run.ws_attn
    wl = inp.wl
    counters = ws[kv.STATUS_BYTES:kv.STATUS_BYTES + 4 * wl.A * wl.H_kv].view(torch.int32)
    counters.fill_(1)
    ws[:4].view(torch.int32).fill_(kv.FLAG_TIMEOUT)
    assert kv.kvgqa_read_status(ws) == kv.FLAG_TIMEOUT
    assert int(ws.count_nonzero()) == 0, "workspace not zero-filled after a timeout was read"
    run.attention()
    torch.cuda.synchronize()
    rows = list(range(wl.A))
    assert_attention_close(run.out.cpu(), oracle_attention(inp, rows), "attention after the workspace was restored")
    assert kv.kvgqa_read_status(ws) == 0
