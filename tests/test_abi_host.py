"""Host-side contract of the C ABI, runnable without a GPU: the library loads,
exports every function include/kvgqa.h declares, and rejects malformed calls
with the documented status before touching CUDA."""
import ctypes
import os
import re

import pytest
import torch

import kv_cached_gqa_rope_gb300 as kv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvgqa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:kvgqa_status|int|const char\*)\s+(\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 9
    lib = kv.library()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(kv.EXPORTED_SYMBOLS)


def test_abi_version():
    assert kv.abi_version() == 1


def test_workspace_sizes():
    assert kv.rope_kv_store_workspace_size() == 256
    # status block + rotated queries + one int32 per (128-query tile, prompt) pair
    assert kv.prefill_gqa_cached_rows_workspace_size(16, 1024, 32, 8, 128) == 256 + 16 * 1024 * 32 * 128 * 2 + 16 * 8 * 4
    assert kv.prefill_gqa_cached_rows_workspace_size(0, 0, 4, 2, 64) == 256
    with pytest.raises(kv.KvgqaError) as e:
        kv.prefill_gqa_cached_rows_workspace_size(1, 1, 4, 2, 96)
    assert e.value.code == "EUNSUPPORTED"
    with pytest.raises(kv.KvgqaError) as e:
        kv.prefill_gqa_cached_rows_workspace_size(1, 1, 6, 4, 64)
    assert e.value.code == "EINVAL"


def aligned_bytes(n, align=256):
    """Host uint8 buffer of n bytes starting on an `align`-byte boundary."""
    raw = torch.zeros(n + align, dtype=torch.uint8)
    off = (-raw.data_ptr()) % align
    return raw[off:off + n]


def decode_args(A=2, H_q=4, H_kv=2, D=64, S=4, L=32):
    bf = torch.bfloat16
    return dict(q=torch.zeros(A, H_q, D, dtype=bf), k=torch.zeros(A, H_kv, D, dtype=bf),
                v=torch.zeros(A, H_kv, D, dtype=bf), positions=torch.zeros(A, dtype=torch.int32),
                cache_rows=torch.arange(A, dtype=torch.int32), theta=1e4,
                q_out=torch.zeros(A, H_q, D, dtype=bf), k_cache=torch.zeros(S, H_kv, L, D, dtype=bf),
                v_cache=torch.zeros(S, H_kv, L, D, dtype=bf), workspace=aligned_bytes(256))


def call_store(**kw):
    a = decode_args()
    a.update(kw)
    kv.rope_kv_store_out_(**a)


def code_of(fn, **kw):
    with pytest.raises(kv.KvgqaError) as e:
        fn(**kw)
    return e.value.code


def test_store_dtype_rejected():
    assert code_of(call_store, k=torch.zeros(2, 2, 64, dtype=torch.float32)) == "EDTYPE"
    assert code_of(call_store, positions=torch.zeros(2, dtype=torch.float32)) == "EDTYPE"
    assert code_of(call_store, cache_rows=torch.zeros(2, dtype=torch.uint8)) == "EDTYPE"
    with pytest.raises(TypeError):          # no C dtype for it at all
        call_store(q=torch.zeros(2, 4, 64, dtype=torch.float64))
    # FP16 storage is accepted only when every 16-bit operand is FP16
    assert code_of(call_store, q=torch.zeros(2, 4, 64, dtype=torch.float16)) == "EDTYPE"
    f16 = dict(q=torch.zeros(2, 4, 64, dtype=torch.float16), k=torch.zeros(2, 2, 64, dtype=torch.float16),
               v=torch.zeros(2, 2, 64, dtype=torch.float16), q_out=torch.zeros(2, 4, 64, dtype=torch.float16),
               k_cache=torch.zeros(4, 2, 16, 64, dtype=torch.float16))
    assert code_of(call_store, **f16) == "EDTYPE"                     # v_cache still bf16
    f16["v_cache"] = torch.zeros(4, 2, 16, 64, dtype=torch.float16)
    assert code_of(call_store, **f16) in ("ECUDA", "EDEVICE", "OK")    # past the dtype checks


def test_store_layout_rejected():
    q = torch.zeros(2, 64, 4, dtype=torch.bfloat16).transpose(1, 2)   # [A,H_q,D] view, not contiguous
    assert code_of(call_store, q=q) == "ELAYOUT"
    base = torch.zeros(2 * 4 * 64 + 1, dtype=torch.bfloat16)
    misaligned = base[1:].view(2, 4, 64)                               # 2-byte offset
    assert code_of(call_store, q=misaligned) == "ELAYOUT"


def test_store_shape_rejected():
    assert code_of(call_store, k=torch.zeros(3, 2, 64, dtype=torch.bfloat16)) == "EINVAL"
    assert code_of(call_store, q_out=torch.zeros(2, 4, 32, dtype=torch.bfloat16)) == "EINVAL"
    assert code_of(call_store, q=torch.zeros(2, 3, 64, dtype=torch.bfloat16),
                   q_out=torch.zeros(2, 3, 64, dtype=torch.bfloat16)) == "EINVAL"   # 3 % 2 != 0
    a = decode_args(D=96)
    assert code_of(kv.rope_kv_store_out_, **a) == "EUNSUPPORTED"
    a = decode_args(D=63)
    assert code_of(kv.rope_kv_store_out_, **a) == "EINVAL"


def test_store_scalars_rejected():
    assert code_of(call_store, theta=0.0) == "EINVAL"
    assert code_of(call_store, theta=float("inf")) == "EINVAL"
    assert code_of(call_store, theta=-5.0) == "EINVAL"


def test_store_alias_rejected():
    a = decode_args()
    a["q_out"] = a["q"]
    assert code_of(kv.rope_kv_store_out_, **a) == "EALIAS"
    a = decode_args()
    both = torch.zeros(2, 4, 2, 32, 64, dtype=torch.bfloat16)
    a["k_cache"], a["v_cache"] = both[0], both[0]
    assert code_of(kv.rope_kv_store_out_, **a) == "EALIAS"
    a = decode_args()
    vbuf = aligned_bytes(4 * 2 * 32 * 64 * 2)
    a["v_cache"] = vbuf.view(torch.bfloat16).view(4, 2, 32, 64)
    a["workspace"] = vbuf[:256]                     # aligned, and inside v_cache
    assert code_of(kv.rope_kv_store_out_, **a) == "EALIAS"


def test_store_workspace_rejected():
    assert code_of(call_store, workspace=aligned_bytes(100)) == "EWORKSPACE"
    assert code_of(call_store, workspace=aligned_bytes(300)[1:]) == "EWORKSPACE"   # misaligned
    assert code_of(call_store, workspace=torch.zeros(64, dtype=torch.int32)) == "EWORKSPACE"


def test_descriptor_bytes_enforced():
    a = decode_args()
    lib = kv.library()
    ds = {n: kv.describe(a[n]) for n in ("q", "k", "v", "positions", "cache_rows", "q_out", "k_cache", "v_cache", "workspace")}
    ds["k_cache"].bytes = 100      # claims less than the view needs
    import ctypes
    st = lib.rope_kv_store_out_(*(ctypes.byref(ds[n]) for n in ("q", "k", "v", "positions", "cache_rows")), 1e4,
                                *(ctypes.byref(ds[n]) for n in ("q_out", "k_cache", "v_cache", "workspace")), None)
    assert kv.STATUS_NAMES[st] == "EINVAL"
    assert b"bytes" in lib.kvgqa_last_error()


def test_null_descriptor_rejected():
    import ctypes
    lib = kv.library()
    a = decode_args()
    ds = [kv.describe(a[n]) for n in ("q", "k", "v", "positions", "cache_rows", "q_out", "k_cache", "v_cache")]
    st = lib.rope_kv_store_out_(*(ctypes.byref(d) for d in ds[:5]), 1e4, *(ctypes.byref(d) for d in ds[5:]),
                                None, None)
    assert kv.STATUS_NAMES[st] == "EINVAL"


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_valid_host_call_fails_cleanly_without_gpu():
    # All descriptor checks pass; the device lookup then fails with a status,
    # not a crash (host tensors can never be accepted as device memory).
    code = code_of(call_store)
    assert code in ("ECUDA", "EDEVICE")


def attention_args(A=2, H_q=4, H_kv=2, D=64, S=4, L=32):
    bf = torch.bfloat16
    return dict(q_rot=torch.zeros(A, H_q, D, dtype=bf), k_cache=torch.zeros(S, H_kv, L, D, dtype=bf),
                v_cache=torch.zeros(S, H_kv, L, D, dtype=bf), positions=torch.zeros(A, dtype=torch.int32),
                cache_rows=torch.arange(A, dtype=torch.int32), scale=0.125,
                out=torch.zeros(A, H_q, D, dtype=bf), workspace=aligned_bytes(256))


def test_attention_contract():
    a = attention_args()
    a["out"] = a["q_rot"]
    assert code_of(kv.cached_gqa_attention_out_, **a) == "EALIAS"
    a = attention_args()
    a["scale"] = float("nan")
    assert code_of(kv.cached_gqa_attention_out_, **a) == "EINVAL"
    a = attention_args(H_q=64, H_kv=2)          # G = 32 has no decode kernel
    assert code_of(kv.cached_gqa_attention_out_, **a) == "EUNSUPPORTED"
    a = attention_args()
    a["v_cache"] = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16)
    assert code_of(kv.cached_gqa_attention_out_, **a) == "EINVAL"
    a = attention_args(A=1100)
    assert code_of(kv.cached_gqa_attention_out_, **a) == "EUNSUPPORTED"


def prefill_args(A=2, T=8, H_q=4, H_kv=2, D=64, S=4, L=16):
    bf = torch.bfloat16
    return dict(q=torch.zeros(A, T, H_q, D, dtype=bf), k=torch.zeros(A, T, H_kv, D, dtype=bf),
                v=torch.zeros(A, T, H_kv, D, dtype=bf), cache_rows=torch.arange(A, dtype=torch.int32),
                theta=1e4, scale=0.125, k_cache=torch.zeros(S, H_kv, L, D, dtype=bf),
                v_cache=torch.zeros(S, H_kv, L, D, dtype=bf), out=torch.zeros(A, T, H_q, D, dtype=bf),
                workspace=aligned_bytes(256 + (A * T * H_q * D * 2 + 255) // 256 * 256 + A * ((T + 127) // 128) * 4))


def test_prefill_contract():
    a = prefill_args(T=20)                       # T > max_seq
    a["workspace"] = aligned_bytes(256 + 2 * 20 * 4 * 64 * 2)
    assert code_of(kv.prefill_gqa_cached_rows_out_, **a) == "EINVAL"
    a = prefill_args()
    a["workspace"] = aligned_bytes(1000)
    assert code_of(kv.prefill_gqa_cached_rows_out_, **a) == "EWORKSPACE"
    a = prefill_args()
    a["out"] = a["k_cache"].view(-1)[: 2 * 8 * 4 * 64].view(2, 8, 4, 64)
    assert code_of(kv.prefill_gqa_cached_rows_out_, **a) == "EALIAS"
    a = prefill_args()
    a["k"] = torch.zeros(2, 8, 4, 64, dtype=torch.bfloat16)
    assert code_of(kv.prefill_gqa_cached_rows_out_, **a) == "EINVAL"


def varlen_args(**kw):
    a = prefill_args(**kw)
    A = a["q"].shape[0]
    a["offsets"] = torch.zeros(A, dtype=torch.int32)
    a["lengths"] = torch.full((A,), a["q"].shape[1], dtype=torch.int32)
    return a


def test_prefill_varlen_contract():
    a = varlen_args()
    a["offsets"] = torch.zeros(3, dtype=torch.int32)      # not [A]
    assert code_of(kv.prefill_varlen_gqa_cached_rows_out_, **a) == "EINVAL"
    a = varlen_args()
    a["lengths"] = torch.zeros(2, dtype=torch.float32)    # not int32
    assert code_of(kv.prefill_varlen_gqa_cached_rows_out_, **a) == "EDTYPE"
    a = varlen_args()
    a["out"] = a["k_cache"].view(-1)[: 2 * 8 * 4 * 64].view(2, 8, 4, 64)
    assert code_of(kv.prefill_varlen_gqa_cached_rows_out_, **a) == "EALIAS"
    a = varlen_args(T=20)                                 # T > max_seq
    a["workspace"] = aligned_bytes(256 + 2 * 20 * 4 * 64 * 2)
    assert code_of(kv.prefill_varlen_gqa_cached_rows_out_, **a) == "EINVAL"
    lib = kv.library()
    # null offsets or lengths descriptors are rejected, not read as "equal length"
    ds = [kv.describe(t) for t in (a["q"], a["k"], a["v"])]
    null = ctypes.POINTER(kv.KvgqaTensor)()
    st = lib.prefill_varlen_gqa_cached_rows_out_(*[ctypes.byref(d) for d in ds], null, null,
                                                 ctypes.byref(kv.describe(a["cache_rows"])), 1e4, 0.125,
                                                 null, null, null, null, None)
    assert kv.STATUS_NAMES[st] == "EINVAL"


def step_args(A=2, H_q=4, H_kv=2, D=64, S=4, L=32):
    bf = torch.bfloat16
    return dict(q=torch.zeros(A, H_q, D, dtype=bf), k=torch.zeros(A, H_kv, D, dtype=bf),
                v=torch.zeros(A, H_kv, D, dtype=bf), positions=torch.zeros(A, dtype=torch.int32),
                cache_rows=torch.arange(A, dtype=torch.int32), theta=1e4, scale=0.125,
                k_cache=torch.zeros(S, H_kv, L, D, dtype=bf), v_cache=torch.zeros(S, H_kv, L, D, dtype=bf),
                out=torch.zeros(A, H_q, D, dtype=bf), workspace=aligned_bytes(256))


@pytest.mark.parametrize("call", [kv.decode_step_out_, kv.decode_step_single_launch_out_],
                         ids=["two_kernels", "single_launch"])
def test_decode_step_contract(call):
    """Both forms of the whole step share the host contract: every refusal
    below happens before anything is queued."""
    a = step_args()
    a["out"] = a["q"]
    assert code_of(call, **a) == "EALIAS"
    a = step_args()
    a["out"] = a["k_cache"].view(-1)[: 2 * 4 * 64].view(2, 4, 64)
    assert code_of(call, **a) == "EALIAS"
    a = step_args()
    a["theta"] = -1.0
    assert code_of(call, **a) == "EINVAL"
    a = step_args()
    a["scale"] = float("inf")
    assert code_of(call, **a) == "EINVAL"
    a = step_args(H_q=64, H_kv=2)               # G = 32 has no decode kernel
    assert code_of(call, **a) == "EUNSUPPORTED"
    a = step_args()
    a["v"] = torch.zeros(2, 3, 64, dtype=torch.bfloat16)
    assert code_of(call, **a) == "EINVAL"
    a = step_args()
    a["k"] = torch.zeros(2, 2, 64, dtype=torch.float32)
    assert code_of(call, **a) == "EDTYPE"
    a = step_args(A=1100)
    assert code_of(call, **a) == "EUNSUPPORTED"
    # every descriptor check passes: host tensors then fail the device check
    assert code_of(call, **step_args()) in ("ECUDA", "EDEVICE")


def test_overflowing_sizes_are_refused():
    """A descriptor whose sizes overflow a 64-bit byte count is refused with
    EINVAL before any byte range is computed from it (no wrap-around into a
    small, seemingly valid range)."""
    a = attention_args()
    lib = kv.library()
    ds = {name: kv.describe(t) for name, t in a.items() if isinstance(t, torch.Tensor)}
    ds["positions"].shape[0] = 1 << 62            # 2^62 int32 values: 2^64 bytes
    st = lib.cached_gqa_attention_out_(*[ctypes.byref(ds[n]) for n in ("q_rot", "k_cache", "v_cache", "positions",
                                                                        "cache_rows")],
                                       ctypes.c_float(0.125), ctypes.byref(ds["out"]), ctypes.byref(ds["workspace"]),
                                       None)
    assert kv.STATUS_NAMES[st] == "EINVAL"
    assert b"overflow" in lib.kvgqa_last_error()
