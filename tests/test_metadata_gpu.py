"""Decode steps driven by the host slot table: one [3, capacity] host-to-device
copy per step, positions and cache_rows as zero-copy views of the device copy;
the results equal the same calls on separately built metadata tensors."""
import pytest
import torch

import kv_cached_gqa_rope_gb300 as kv

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
    for step, reqs in enumerate(order):
        if step == 2:
            table.admit(104, 5)                       # admission at a step boundary
        A, fin = table.step(reqs, [7] * len(reqs), meta.host)
        tokens, positions, rows = meta.upload(A)
        torch.cuda.synchronize()
        assert positions.data_ptr() == meta.device[1].data_ptr()   # views, no copies
        q, k, v = make_step_inputs(A, H_q, H_kv, D, seed=step)
        q_rot_a, out_a = torch.empty_like(q), torch.empty_like(q)
        kv.rope_kv_store_out_(q, k, v, positions, rows, theta, q_rot_a, kc_a, vc_a, ws_s)
        kv.cached_gqa_attention_out_(q_rot_a, kc_a, vc_a, positions, rows, scale, out_a, ws_a)
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
