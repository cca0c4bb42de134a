"""The tiny decode step against its stored fixture (tests/golden/tiny_decode.json).

The fixture holds seeded inputs and the FP64 oracle's results, written by
tests/golden/make_golden.py (the pages print no worked values for this path).
On the CPU the oracle must reproduce it exactly (it pins the oracle against
changes to itself); on the GPU the CUDA path, fed the stored inputs, must
match it within the parity bars: rotated Q and K within 1 BF16 ulp, V cells
and every other cache byte exact, the output within max-abs 1e-2 / RMS 2e-3
/ relative RMS 5e-3.
"""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def unhex(s, shape):
    return np.frombuffer(bytes.fromhex(s), dtype=">u2").astype(np.uint16).reshape(shape)


@pytest.fixture(scope="module")
def fx():
    with open(os.path.join(HERE, "golden", "tiny_decode.json")) as f:
        d = json.load(f)
    w = d["workload"]
    A, H_q, H_kv, D, S, L = w["A"], w["H_q"], w["H_kv"], w["D"], w["slots"], w["max_seq"]
    pos = np.array(d["positions"], dtype=np.int64)
    rows = np.array(d["cache_rows"], dtype=np.int64)
    kc = np.full((S, H_kv, L, D), w["sentinel"], dtype=np.uint16)
    vc = np.full((S, H_kv, L, D), w["sentinel"], dtype=np.uint16)
    for a in range(A):
        kc[rows[a], :, : pos[a]] = unhex(d["k_prefix"][a], (H_kv, pos[a], D))
        vc[rows[a], :, : pos[a]] = unhex(d["v_prefix"][a], (H_kv, pos[a], D))
    return dict(w=w, pos=pos, rows=rows, kc=kc, vc=vc,
                q=unhex(d["q"], (A, H_q, D)), k=unhex(d["k"], (A, H_kv, D)), v=unhex(d["v"], (A, H_kv, D)),
                q_rot=unhex(d["q_rot"], (A, H_q, D)), k_rot=unhex(d["k_rot"], (A, H_kv, D)),
                out=np.array(d["out_f64"]).reshape(A, H_q, D), out_bf16=unhex(d["out_bf16"], (A, H_q, D)))


def test_oracle_reproduces_fixture(fx):
    w = fx["w"]
    q_rot, kc, vc = oracle.rope_kv_store(fx["q"], fx["k"], fx["v"], fx["pos"], fx["rows"], w["theta"],
                                         fx["kc"], fx["vc"])
    assert np.array_equal(q_rot, fx["q_rot"])
    for a in range(w["A"]):
        r, p = fx["rows"][a], fx["pos"][a]
        assert np.array_equal(kc[r, :, p], fx["k_rot"][a])
        assert np.array_equal(vc[r, :, p], fx["v"][a])
    out = oracle.cached_gqa_attention(q_rot, kc, vc, fx["pos"], fx["rows"], w["scale"])
    assert np.max(np.abs(out - fx["out"])) <= 1e-13
    assert np.array_equal(oracle.f64_to_bf16(out), fx["out_bf16"])


@pytest.mark.gpu
@pytest.mark.parametrize("call", ["two_calls", "decode_step"])
def test_cuda_path_matches_fixture(fx, call):
    import torch

    import kv_cached_gqa_rope_gb300 as kv
    from gpu_helpers import assert_attention_close

    w = fx["w"]
    dev = torch.device("cuda")

    def t16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v = t16(fx["q"]), t16(fx["k"]), t16(fx["v"])
    pos = torch.as_tensor(fx["pos"], dtype=torch.int32, device=dev)
    rows = torch.as_tensor(fx["rows"], dtype=torch.int32, device=dev)
    kc, vc = t16(fx["kc"]), t16(fx["vc"])
    out = torch.empty_like(q)
    q_rot = torch.empty_like(q)
    if call == "two_calls":
        ws1 = kv.new_workspace(kv.rope_kv_store_workspace_size(), dev)
        ws2 = kv.new_workspace(kv.cached_gqa_attention_workspace_size(w["A"], w["H_q"], w["H_kv"], w["D"]), dev)
        kv.rope_kv_store_out_(q, k, v, pos, rows, w["theta"], q_rot, kc, vc, ws1)
        kv.cached_gqa_attention_out_(q_rot, kc, vc, pos, rows, w["scale"], out, ws2)
        torch.cuda.synchronize()
        assert kv.kvgqa_read_status(ws1) == 0 and kv.kvgqa_read_status(ws2) == 0
        bits = q_rot.cpu().view(torch.int16).numpy().view(np.uint16)
        assert oracle.ulp_distance_bf16(bits, fx["q_rot"]).max() <= 1
    else:
        ws = kv.new_workspace(kv.decode_step_workspace_size(w["A"], w["H_q"], w["H_kv"], w["D"]), dev)
        kv.decode_step_out_(q, k, v, pos, rows, w["theta"], w["scale"], kc, vc, out, ws)
        torch.cuda.synchronize()
        assert kv.kvgqa_read_status(ws) == 0
    kc_b = kc.cpu().view(torch.int16).numpy().view(np.uint16)
    vc_b = vc.cpu().view(torch.int16).numpy().view(np.uint16)
    want_k, want_v = fx["kc"].copy(), fx["vc"].copy()
    for a in range(w["A"]):
        r, p = fx["rows"][a], fx["pos"][a]
        assert oracle.ulp_distance_bf16(kc_b[r, :, p], fx["k_rot"][a]).max() <= 1
        want_k[r, :, p] = kc_b[r, :, p]
        want_v[r, :, p] = fx["v"][a]
    assert np.array_equal(kc_b, want_k), "K cache bytes outside the new cells changed"
    assert np.array_equal(vc_b, want_v), "V cells or other V cache bytes differ"
    assert_attention_close(out.cpu(), fx["out"], f"tiny decode vs fixture ({call})")
