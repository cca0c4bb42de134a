"""The algorithmic work bench.py divides by its timings, counted again by
brute force on small workloads: every byte the decode step must move and
every multiply-add the causal prefills must do, enumerated one element at a
time from the definitions (microLLM-rocm ARCHITECTURE.md, "Tensor ownership
boundary": each token attends to its own row's prefix up to its position;
the prefill is causal within each prompt and sees a row's earlier prefix).
A wrong count would misstate every roofline fraction in the bench line."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402

BF16 = 2  # bytes per stored element


def brute_decode_bytes(A, H_q, H_kv, D, positions):
    attn = 0
    for a in range(A):
        for g in range(H_kv):
            for key in range(positions[a] + 1):      # keys 0..p inclusive
                attn += D * BF16 * 2                 # its K row and its V row
    attn += A * H_q * D * BF16                       # rotated queries read
    attn += A * H_q * D * BF16                       # output written
    store = 0
    for a in range(A):
        store += (H_q + 2 * H_kv) * D * BF16         # q, k, v read
        store += H_q * D * BF16                      # rotated q written
        store += 2 * H_kv * D * BF16                 # the new K and V cells written
    fused = attn + 2 * (2 * A * H_kv * D * BF16)     # new k, v read and their cells written, no q_rot round trip
    return attn, attn + store, fused


@pytest.mark.parametrize("positions", [[0], [5, 17], [0, 1, 127, 128, 4095], list(range(0, 300, 7))])
@pytest.mark.parametrize("heads", [(4, 2, 64), (32, 8, 128), (64, 8, 128)])
def test_decode_bytes(positions, heads):
    H_q, H_kv, D = heads
    wl = W.scaled_decode(W.LLAMA_DECODE, A=len(positions), H_q=H_q, H_kv=H_kv, D=D)
    got = bench.decode_bytes(wl, np.array(positions))
    assert got == brute_decode_bytes(len(positions), H_q, H_kv, D, positions)


def brute_causal_flops(D, H_q, spans):
    """spans: per prompt, (offset, length): query t sees keys 0 .. offset + t;
    each visible key costs D multiply-adds for q.k and D for p.v."""
    macs = 0
    for off, n in spans:
        for t in range(n):
            for _key in range(off + t + 1):
                macs += 2 * D
    return 2.0 * H_q * macs  # two FLOPs per multiply-add, every query head


def test_prefill_flops():
    wl = W.scaled_prefill(W.PREFILL, A=3, T=37, H_q=4, H_kv=2, D=16)
    assert bench.prefill_flops(wl) == brute_causal_flops(wl.D, wl.H_q, [(0, wl.T)] * wl.A)


@pytest.mark.parametrize("spans", [[(0, 37)], [(5, 3), (0, 1), (120, 40)], [(0, 0), (17, 9)]])
def test_varlen_flops(spans):
    wl = W.scaled_prefill(W.PREFILL, A=len(spans), T=64, H_q=4, H_kv=2, D=16)
    offs = [o for o, _ in spans]
    lens = [n for _, n in spans]
    assert bench.varlen_flops(wl, offs, lens) == brute_causal_flops(wl.D, wl.H_q, spans)


def test_varlen_with_zero_offsets_is_the_equal_length_prefill():
    wl = W.scaled_prefill(W.PREFILL, A=4, T=50, H_q=8, H_kv=2, D=32)
    assert bench.varlen_flops(wl, [0] * 4, [50] * 4) == bench.prefill_flops(wl)


def test_e2e_entry_prefers_the_checked_graph_and_keeps_the_plain_loop():
    import bench
    graph = {"value": 2.0, "unit": bench.UNIT, "h2d_bytes_per_step": 10, "d2h_bytes_per_step": 20,
             "spread": {"median_ms": 1.0}, "note": "one CUDA graph per step"}
    e = bench.e2e_line(1.0, {"median_ms": 2.0}, graph, 10, 20)
    assert e["value"] == 2.0 and e["mode"].startswith("cuda_graph")
    assert e["plain"]["value"] == 1.0 and e["plain"]["h2d_bytes_per_step"] == 10
    assert e["h2d_bytes_per_step"] == 10 and e["d2h_bytes_per_step"] == 20
    e = bench.e2e_line(1.0, {"median_ms": 2.0}, {"unavailable": "capture refused"}, 10, 20)
    assert e["value"] == 1.0 and e["mode"].startswith("plain") and e["graph"] == {"unavailable": "capture refused"}
