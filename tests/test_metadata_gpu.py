"""Decode steps driven by the host slot table: one [3, capacity] host-to-device
copy per step, positions and cache_rows as zero-copy views of the device copy.
Each step's metadata is checked against hand-derived values (lowest free row
on admission, position = the row's length), its results against the FP64
oracle run on the same metadata with its own cache state carried from step to
step, and against the same calls on separately built metadata tensors."""
import numpy as np
import pytest
import torch

import kv_cached_gqa_rope_gb300 as kv
import oracle
import workloads as W
from gpu_helpers import assert_attention_close, bits

pytestmark = pytest.mark.gpu


def make_step_inputs(A, H_q, H_kv, D, seed):
    g = torch.Generator().manual_seed(seed)
    bf = torch.bfloat16
    return (torch.randn(A, H_q, D, generator=g).to(bf).cuda(), torch.randn(A, H_kv, D, generator=g).to(bf).cuda(),
            torch.randn(A, H_kv, D, generator=g).to(bf).cuda())


def test_slot_table_driven_steps_match_explicit_metadata():
    S, L, H_q, H_kv, D = 6, 64, 8, 2, 128
    g = torch.Generator().manual_seed(20261202)
    kc0 = torch.randn(S, H_kv, L, D, generator=g).to(torch.bfloat16).cuda()
    vc0 = torch.randn(S, H_kv, L, D, generator=g).to(torch.bfloat16).cuda()
    kc_a, vc_a, kc_b, vc_b = kc0.clone(), vc0.clone(), kc0.clone(), vc0.clone()
    table = kv.SlotTable(S, L)
    meta = kv.StepMetadata(capacity=S)
    lengths = {100: 10, 101: 40, 102: 0, 103: 61}
    for r, n in lengths.items():
        table.admit(r, n)
    ws_s = kv.new_workspace(kv.rope_kv_store_workspace_size())
    ws_a = kv.new_workspace(kv.cached_gqa_attention_workspace_size(S, H_q, H_kv, D))
    scale, theta = D ** -0.5, 10000.0
    order = [[103, 100, 102, 101], [101, 103, 100], [104, 100, 103]]
    # rows: 100..103 take the lowest free rows 0..3 in admission order, 104
    # (admitted before step 2, no row released yet) row 4; positions: each
    # row's length, which every step advances by one
    want_pos = [[61, 10, 0, 40], [41, 62, 11], [5, 12, 63]]
    want_rows = [[3, 0, 2, 1], [1, 3, 0], [4, 0, 3]]
    kc_o, vc_o = bits(kc0), bits(vc0)   # the oracle's own cache state
    for step, reqs in enumerate(order):
        if step == 2:
            table.admit(104, 5)                       # admission at a step boundary
        A, fin = table.step(reqs, [7] * len(reqs), meta.host)
        tokens, positions, rows = meta.upload(A)
        torch.cuda.synchronize()
        assert positions.data_ptr() == meta.device[1].data_ptr()   # views, no copies
        assert meta.host[0, :A].tolist() == [7] * A
        assert meta.host[1, :A].tolist() == want_pos[step]
        assert meta.host[2, :A].tolist() == want_rows[step]
        q, k, v = make_step_inputs(A, H_q, H_kv, D, seed=step)
        q_rot_a, out_a = torch.empty_like(q), torch.empty_like(q)
        kv.rope_kv_store_out_(q, k, v, positions, rows, theta, q_rot_a, kc_a, vc_a, ws_s)
        kv.cached_gqa_attention_out_(q_rot_a, kc_a, vc_a, positions, rows, scale, out_a, ws_a)
        # the oracle on the same step: store, then attention over each row's prefix
        pos_h, rows_h = np.array(want_pos[step]), np.array(want_rows[step])
        q_rot_o, kc_o, vc_o = oracle.rope_kv_store(bits(q), bits(k), bits(v), pos_h, rows_h, theta, kc_o, vc_o)
        ref = oracle.cached_gqa_attention(q_rot_o, kc_o, vc_o, pos_h, rows_h, scale)
        torch.cuda.synchronize()
        assert oracle.ulp_distance_bf16(bits(q_rot_a), q_rot_o).max() <= 1
        assert oracle.ulp_distance_bf16(bits(kc_a), kc_o).max() <= 1, "K cache beyond 1 ulp of the oracle"
        assert np.array_equal(bits(vc_a), vc_o), "V cache differs from the oracle"
        assert_attention_close(out_a.cpu(), ref, f"slot-table step {step}")
        # the same step on explicitly built device tensors
        pos_b = torch.tensor(meta.host[1, :A].tolist(), dtype=torch.int32, device="cuda")
        rows_b = torch.tensor(meta.host[2, :A].tolist(), dtype=torch.int32, device="cuda")
        q_rot_b, out_b = torch.empty_like(q), torch.empty_like(q)
        kv.rope_kv_store_out_(q, k, v, pos_b, rows_b, theta, q_rot_b, kc_b, vc_b, ws_s)
        kv.cached_gqa_attention_out_(q_rot_b, kc_b, vc_b, pos_b, rows_b, scale, out_b, ws_a)
        torch.cuda.synchronize()
        assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
        assert torch.equal(kc_a.view(torch.int16), kc_b.view(torch.int16))
        assert torch.equal(vc_a.view(torch.int16), vc_b.view(torch.int16))
        assert kv.kvgqa_read_status(ws_s) == 0 and kv.kvgqa_read_status(ws_a) == 0
        if step == 2:
            assert fin.tolist() == [False, False, True]   # request 103 wrote position 63: its row is full
    assert table.query()["released"]["length"] == 1
