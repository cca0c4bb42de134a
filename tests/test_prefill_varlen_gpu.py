"""GPU parity of the prefill of prompts of different lengths at their own
offsets (chunked prefill into rows that may hold a prefix) against the FP64
oracle, through the C ABI; plus its reductions to the equal-length prefill,
to the decode step and to itself in chunks."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_attention_close, bits

pytestmark = pytest.mark.gpu

FLAG_POSITION_RANGE, FLAG_ROW_RANGE = 0x1, 0x2


class VarlenRun:
    def __init__(self, inp: W.VarlenInputs, tail="nan"):
        import kv_cached_gqa_rope_gb300 as kv
        self.kv, self.inp, wl = kv, inp, inp.wl
        self.q, self.k, self.v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
        self.offsets, self.lengths, self.rows = inp.offsets.cuda(), inp.lengths.cuda(), inp.cache_rows.cuda()
        self.k_cache, self.v_cache = inp.build_cache("cuda", tail)
        self.k0, self.v0 = self.k_cache.clone(), self.v_cache.clone()
        self.out = W.sentinel_fill((wl.A, wl.T, wl.H_q, wl.D), "cuda")
        self.ws = kv.new_workspace(kv.prefill_gqa_cached_rows_workspace_size(wl.A, wl.T, wl.H_q, wl.H_kv, wl.D))

    def run(self):
        wl = self.inp.wl
        self.kv.prefill_varlen_gqa_cached_rows_out_(self.q, self.k, self.v, self.offsets, self.lengths, self.rows,
                                                    wl.theta, wl.scale, self.k_cache, self.v_cache, self.out,
                                                    self.ws)
        torch.cuda.synchronize()
        return self


def valid_prompts(inp: W.VarlenInputs):
    wl = inp.wl
    ok = []
    for a in range(wl.A):
        o, n, r = int(inp.offsets[a]), int(inp.lengths[a]), int(inp.cache_rows[a])
        if 0 <= n <= wl.T and o >= 0 and o + n <= wl.max_seq and 0 <= r < wl.slots:
            ok.append(a)
    return ok


def oracle_varlen(run: VarlenRun, prompts, select=None):
    """The oracle over the given prompts, on a compact cache holding only
    their rows as they were before the call (row i of it is slot rows[i])."""
    inp = run.inp
    rows = inp.cache_rows[prompts].long()
    kc = bits(run.k0[rows.cuda()])
    vc = bits(run.v0[rows.cuda()])
    sel = lambda t: W.bf16_bits(t[prompts])
    return oracle.prefill_varlen_gqa_cached_rows(sel(inp.q), sel(inp.k), sel(inp.v), inp.offsets[prompts].numpy(),
                                                 inp.lengths[prompts].numpy(), np.arange(len(prompts)),
                                                 inp.wl.theta, inp.wl.scale, kc, vc, select=select)


def check_caches(run: VarlenRun, prompts, kc_ref, vc_ref):
    """Cells [off, off+len) of each valid prompt's row hold rotated K (<= 1
    ulp of the oracle) and V (bit-exact); every other byte is unchanged."""
    inp = run.inp
    k_exp, v_exp = run.k0.clone(), run.v0.clone()
    for i, a in enumerate(prompts):
        r, o, n = int(inp.cache_rows[a]), int(inp.offsets[a]), int(inp.lengths[a])
        if n == 0:
            continue
        got_k = run.k_cache[r, :, o:o + n]
        d = oracle.ulp_distance_bf16(bits(got_k), kc_ref[i, :, o:o + n])
        assert d.max() <= 1, f"prompt {a}: K cells beyond 1 ulp: {int((d > 1).sum())}"
        assert np.array_equal(bits(run.v_cache[r, :, o:o + n]), vc_ref[i, :, o:o + n]), f"prompt {a}: V cells"
        k_exp[r, :, o:o + n] = got_k
        v_exp[r, :, o:o + n] = run.v_cache[r, :, o:o + n]
    assert torch.equal(k_exp.view(torch.int16), run.k_cache.view(torch.int16)), "K cache bytes outside the prompts changed"
    assert torch.equal(v_exp.view(torch.int16), run.v_cache.view(torch.int16)), "V cache bytes outside the prompts changed"


def check_outputs(run: VarlenRun, prompts, ref, what):
    """Rows t < len match the oracle; rows past a prompt's length and the
    outputs of skipped prompts are not written."""
    inp = run.inp
    out = run.out.cpu()
    mask = np.zeros(out.shape, dtype=bool)
    for i, a in enumerate(prompts):
        mask[a, : int(inp.lengths[a])] = True
    if mask.any():
        ref_full = np.zeros(out.shape)
        for i, a in enumerate(prompts):
            ref_full[a] = np.nan_to_num(ref[i])
        assert_attention_close(out, ref_full, what, mask=mask)
    untouched = bits(out)[~mask]
    assert np.all(untouched == W.SENTINEL_BITS), "out rows past a prompt's length were written"


CASES = [
    # ragged lengths, offsets off the 128-tile grid, a length-1 prompt
    dict(A=4, T=300, H_q=8, H_kv=2, D=128, slots=6, max_seq=1024, offsets=[0, 37, 500, 129], lengths=[300, 1, 77, 256]),
    # odd G (no head pairs), D = 64, a prompt ending at max_seq, an empty prompt
    dict(A=3, T=200, H_q=6, H_kv=2, D=64, slots=4, max_seq=600, offsets=[400, 255, 128], lengths=[200, 130, 0]),
    # G = 1, a prompt one tile long at offset one tile
    dict(A=2, T=128, H_q=4, H_kv=4, D=128, slots=3, max_seq=256, offsets=[128, 0], lengths=[128, 5]),
    # Llama-style heads, a prefix inside the first tile, a query tile split across two key tiles
    dict(A=3, T=160, H_q=32, H_kv=8, D=128, slots=5, max_seq=512, offsets=[100, 1, 300], lengths=[160, 127, 129]),
]


def _id(k):
    return f"A{k['A']}_T{k['T']}_G{k['H_q'] // k['H_kv']}_D{k['D']}"


def make(kw, index=30, salt=0, rows=None):
    kw = dict(kw)
    offsets, lengths = kw.pop("offsets"), kw.pop("lengths")
    wl = W.scaled_prefill(W.PREFILL, index=index, **kw)
    return W.make_varlen_inputs(wl, offsets, lengths, salt=salt, rows=rows)


@pytest.mark.parametrize("kw", CASES, ids=_id)
@pytest.mark.parametrize("tail", ["nan", "sentinel"])
def test_varlen_small_full(kw, tail):
    inp = make(kw)
    run = VarlenRun(inp, tail=tail).run()
    prompts = valid_prompts(inp)
    _, ref, kc, vc = oracle_varlen(run, prompts)
    check_caches(run, prompts, kc, vc)
    check_outputs(run, prompts, ref, f"varlen {kw} tail={tail}")
    assert run.kv.kvgqa_read_status(run.ws) == 0


@pytest.mark.parametrize("T", [256, 200])
def test_varlen_equal_lengths_is_prefill(T):
    """Offsets 0 and lengths T give the equal-length prefill: the same cache
    bytes; the same output bits when T is a multiple of the 128-key tile
    (otherwise the last key tile is read at another offset and the FP32 sums
    may round differently, so the outputs are compared with the tolerance)."""
    import kv_cached_gqa_rope_gb300 as kv
    wl = W.scaled_prefill(W.PREFILL, index=31, A=3, T=T, H_q=8, H_kv=2, D=128, slots=4, max_seq=512)
    inp = W.make_varlen_inputs(wl, [0] * 3, [T] * 3)
    run = VarlenRun(inp, tail="sentinel").run()
    kc, vc = run.k0.clone(), run.v0.clone()
    out = torch.empty_like(run.out)
    ws = kv.new_workspace(kv.prefill_gqa_cached_rows_workspace_size(wl.A, wl.T, wl.H_q, wl.H_kv, wl.D))
    kv.prefill_gqa_cached_rows_out_(run.q, run.k, run.v, run.rows, wl.theta, wl.scale, kc, vc, out, ws)
    torch.cuda.synchronize()
    assert torch.equal(kc.view(torch.int16), run.k_cache.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), run.v_cache.view(torch.int16))
    if T % 128 == 0:
        assert torch.equal(out.view(torch.int16), run.out.view(torch.int16))
    else:
        prompts = list(range(wl.A))
        _, ref, _, _ = oracle_varlen(run, prompts)
        check_outputs(run, prompts, ref, "varlen as equal-length")


def test_varlen_length_one_is_decode():
    """Prompts of one token at offsets p write the same cache cells as the
    decode store at positions p, and attend like the decode step."""
    import kv_cached_gqa_rope_gb300 as kv
    wl = W.scaled_prefill(W.PREFILL, index=32, A=5, T=1, H_q=32, H_kv=8, D=128, slots=8, max_seq=1024)
    offs = [0, 1, 127, 128, 1023]
    inp = W.make_varlen_inputs(wl, offs, [1] * 5)
    run = VarlenRun(inp, tail="sentinel").run()
    kc, vc = run.k0.clone(), run.v0.clone()
    q_out = torch.empty(wl.A, wl.H_q, wl.D, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q_out)
    pos = run.offsets
    ws1 = kv.new_workspace(kv.rope_kv_store_workspace_size())
    ws2 = kv.new_workspace(kv.cached_gqa_attention_workspace_size(wl.A, wl.H_q, wl.H_kv, wl.D))
    kv.rope_kv_store_out_(run.q[:, 0], run.k[:, 0], run.v[:, 0], pos, run.rows, wl.theta, q_out, kc, vc, ws1)
    kv.cached_gqa_attention_out_(q_out, kc, vc, pos, run.rows, wl.scale, out, ws2)
    torch.cuda.synchronize()
    assert torch.equal(kc.view(torch.int16), run.k_cache.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), run.v_cache.view(torch.int16))
    # two BF16-rounded results, each within the bar of the exact value: within
    # twice the bar of each other (one ulp at |x| >= 2 is already 1.6e-2)
    diff = (run.out[:, 0].float() - out.float()).abs().cpu().numpy()
    assert diff.max() <= 2 * 1e-2 and np.sqrt(np.mean(diff ** 2)) <= 2e-3, f"varlen vs decode: {diff.max():.3e}"
    _, ref, _, _ = oracle_varlen(run, list(range(wl.A)))
    check_outputs(run, list(range(wl.A)), ref, "length-one prompts")


def test_varlen_chunks_compose():
    """A prompt prefilled in three chunks leaves the same cache bytes as the
    whole prompt at once, and each chunk's outputs match the oracle of the
    whole prompt."""
    import kv_cached_gqa_rope_gb300 as kv
    L, cuts = 333, [0, 100, 228, 333]
    wl = W.scaled_prefill(W.PREFILL, index=33, A=2, T=L, H_q=8, H_kv=2, D=128, slots=3, max_seq=512)
    whole = W.make_varlen_inputs(wl, [0, 0], [L, L])
    run = VarlenRun(whole, tail="nan").run()
    kc, vc = run.k0.clone(), run.v0.clone()
    ws = kv.new_workspace(kv.prefill_gqa_cached_rows_workspace_size(wl.A, wl.T, wl.H_q, wl.H_kv, wl.D))
    pieces = []
    for c0, c1 in zip(cuts[:-1], cuts[1:]):
        n = c1 - c0
        offs = torch.full((wl.A,), c0, dtype=torch.int32, device="cuda")
        lens = torch.full((wl.A,), n, dtype=torch.int32, device="cuda")
        out = torch.empty(wl.A, n, wl.H_q, wl.D, dtype=torch.bfloat16, device="cuda")
        kv.prefill_varlen_gqa_cached_rows_out_(run.q[:, c0:c1].contiguous(), run.k[:, c0:c1].contiguous(),
                                               run.v[:, c0:c1].contiguous(), offs, lens, run.rows, wl.theta,
                                               wl.scale, kc, vc, out, ws)
        pieces.append(out)
    torch.cuda.synchronize()
    assert torch.equal(kc.view(torch.int16), run.k_cache.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), run.v_cache.view(torch.int16))
    chunked = torch.cat(pieces, dim=1)
    _, ref, _, _ = oracle_varlen(run, [0, 1])
    assert_attention_close(chunked.cpu(), ref, "chunked prefill")
    assert_attention_close(run.out.cpu(), ref, "whole prefill")
    assert kv.kvgqa_read_status(ws) == 0


def test_varlen_invalid_metadata_skipped_and_flagged():
    """Prompts whose offset/length leave [0, max_seq) or [0, T] are skipped
    and flag POSITION_RANGE; a row outside [0, S) flags ROW_RANGE; the valid
    prompts are unaffected."""
    kw = dict(A=5, T=96, H_q=8, H_kv=2, D=128, slots=6, max_seq=256,
              offsets=[10, 200, 0, -1, 5], lengths=[96, 57, 97, 3, 40])
    inp = make(kw, index=34)
    run = VarlenRun(inp, tail="nan").run()
    prompts = valid_prompts(inp)
    assert prompts == [0, 4]
    _, ref, kc, vc = oracle_varlen(run, prompts)
    check_caches(run, prompts, kc, vc)
    check_outputs(run, prompts, ref, "valid prompts beside invalid ones")
    assert run.kv.kvgqa_read_status(run.ws) == FLAG_POSITION_RANGE

    kw = dict(A=3, T=64, H_q=8, H_kv=2, D=128, slots=4, max_seq=256, offsets=[3, 0, 70], lengths=[64, 20, 33])
    inp = make(kw, index=35, rows=[2, 9, 0])
    run = VarlenRun(inp, tail="nan").run()
    prompts = valid_prompts(inp)
    assert prompts == [0, 2]
    _, ref, kc, vc = oracle_varlen(run, prompts)
    check_caches(run, prompts, kc, vc)
    check_outputs(run, prompts, ref, "valid prompts beside a bad row")
    assert run.kv.kvgqa_read_status(run.ws) == FLAG_ROW_RANGE


def test_varlen_full_size():
    """The 16 x 1024-token, 32/8-head prefill shapes with random chunk shapes
    (lengths 1..1024 at offsets anywhere in a 2048-position row, stale cells
    past each prompt filled with NaN): every cache cell and every output
    (a, t < len, h) against the oracle, element by element; rows past a
    prompt's length left unwritten."""
    wl = W.PREFILL
    offs, lens = W.random_offsets_lengths(wl)
    inp = W.make_varlen_inputs(wl, offs, lens)
    run = VarlenRun(inp, tail="nan").run()
    prompts = list(range(wl.A))
    _, ref, kc, vc = oracle_varlen(run, prompts)
    check_caches(run, prompts, kc, vc)
    check_outputs(run, prompts, ref, "chunked prefill, full size")
    assert run.kv.kvgqa_read_status(run.ws) == 0


def test_varlen_more_prompts_than_the_scan_holds():
    """2100 prompts (more than the 2048 whose lengths the store kernel scans
    in shared memory): the store walks the padded tokens instead; caches and
    outputs against the oracle as for the small cases, with empty prompts,
    prompts ending at max_seq and one with an out-of-range row among them."""
    rng = np.random.default_rng(11)
    A, T, max_seq = 2100, 3, 8
    lengths = rng.integers(0, T + 1, A)
    offsets = np.array([rng.integers(0, max_seq - n + 1) for n in lengths])
    kw = dict(A=A, T=T, H_q=2, H_kv=1, D=64, slots=A, max_seq=max_seq,
              offsets=[int(o) for o in offsets], lengths=[int(n) for n in lengths])
    inp = make(kw)
    inp.cache_rows[7] = A  # one prompt with a row out of range: skipped and flagged
    run = VarlenRun(inp).run()
    prompts = valid_prompts(inp)
    assert len(prompts) == A - 1
    _, ref, kc, vc = oracle_varlen(run, prompts)
    check_caches(run, prompts, kc, vc)
    check_outputs(run, prompts, ref, "varlen 2100 prompts")
    assert run.kv.kvgqa_read_status(run.ws) == FLAG_ROW_RANGE
