"""Writes tests/golden/tiny_decode.json, the fixture of the tiny decode step.

The step: 4 cache slots x 128 positions, two active tokens at cache rows
{0, 2} and positions {5, 17}, 4 query and 2 KV heads of width 64, split-half
RoPE with theta 1e4, scale 1/8.  The pages print no worked values for this
path (microLLM-rocm ARCHITECTURE.md, "Tensor ownership boundary", defines it
in words only), so the stored results are the FP64 oracle's, written by this
script from the seeded inputs it stores beside them: the fixture pins the
oracle against later changes to itself and gives the CUDA path a target that
needs neither the seeded generator nor the oracle at test time.

Stored: the inputs (q, k, v as BF16 bit patterns, the cached prefixes of the
two active rows, positions, rows; every other cache cell is 0x7F7F) and the
results (rotated q, rotated k, the attention output as FP64 and as BF16 bits).

    python tests/golden/make_golden.py      (from the repository root)
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads as W  # noqa: E402


def hexs(a) -> str:
    return np.asarray(a, dtype=np.uint16).astype(">u2").tobytes().hex()


def main():
    wl = W.TINY_DECODE
    inp = W.make_decode_inputs(wl)
    q, k, v = W.bf16_bits(inp.q), W.bf16_bits(inp.k), W.bf16_bits(inp.v)
    pos, rows = inp.positions.numpy(), inp.cache_rows.numpy()
    kc0, vc0 = inp.build_cache()
    kc0, vc0 = W.bf16_bits(kc0), W.bf16_bits(vc0)
    q_rot, kc1, vc1 = oracle.rope_kv_store(q, k, v, pos, rows, wl.theta, kc0, vc0)
    out = oracle.cached_gqa_attention(q_rot, kc1, vc1, pos, rows, wl.scale)
    k_rot = np.stack([kc1[rows[a], :, pos[a], :] for a in range(wl.A)])
    fx = {
        "what": "tiny decode step: FP64 oracle results on stored seeded inputs",
        "workload": {"slots": wl.slots, "max_seq": wl.max_seq, "A": wl.A, "H_q": wl.H_q, "H_kv": wl.H_kv,
                     "D": wl.D, "theta": wl.theta, "scale": wl.scale, "sentinel": W.SENTINEL_BITS},
        "positions": pos.tolist(),
        "cache_rows": rows.tolist(),
        "q": hexs(q), "k": hexs(k), "v": hexs(v),
        # cells [0, positions[a]) of every KV head of row cache_rows[a], [H_kv, p, D] each
        "k_prefix": [hexs(kc0[rows[a], :, : pos[a], :]) for a in range(wl.A)],
        "v_prefix": [hexs(vc0[rows[a], :, : pos[a], :]) for a in range(wl.A)],
        "q_rot": hexs(q_rot),
        "k_rot": hexs(k_rot),
        "out_f64": [float(x) for x in out.reshape(-1)],
        "out_bf16": hexs(oracle.f64_to_bf16(out)),
    }
    path = os.path.join(HERE, "tiny_decode.json")
    with open(path, "w") as f:
        json.dump(fx, f, indent=0)
        f.write("\n")
    print(path)


if __name__ == "__main__":
    main()
