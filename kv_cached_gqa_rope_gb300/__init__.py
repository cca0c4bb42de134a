"""Python binding of libkvgqa, the GB300 cached GQA + RoPE decode/prefill path.

Argument marshalling only: torch tensors become non-owning C descriptors
(pointer, accessible bytes, shape, element strides, dtype, device) and the
current torch CUDA stream is passed explicitly.  Every step of the path runs
in the library's CUDA kernels; there is no fallback of any kind.  If the
library has not been built, importing this package raises.

Functions keep the names of the C entry points:

    rope_kv_store_out_(q, k, v, positions, cache_rows, theta, q_out, k_cache, v_cache, workspace)
    cached_gqa_attention_out_(q_rot, k_cache, v_cache, positions, cache_rows, scale, out, workspace)
    prefill_gqa_cached_rows_out_(q, k, v, cache_rows, theta, scale, k_cache, v_cache, out, workspace)
    prefill_varlen_gqa_cached_rows_out_(q, k, v, offsets, lengths, cache_rows, theta, scale,
                                        k_cache, v_cache, out, workspace)

plus the workspace-size queries and ``kvgqa_read_status``.  Shapes, layouts
and the meaning of every argument are documented in ``include/kvgqa.h``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libkvgqa.so")

KVGQA_BF16, KVGQA_I32, KVGQA_F32, KVGQA_U8, KVGQA_F16 = 1, 2, 3, 4, 5
STATUS_NAMES = {0: "OK", 1: "EINVAL", 2: "EDTYPE", 3: "ELAYOUT", 4: "EDEVICE", 5: "EALIAS",
                6: "EWORKSPACE", 7: "ECUDA", 8: "EUNSUPPORTED", 9: "EFULL"}
FLAG_POSITION_RANGE, FLAG_ROW_RANGE, FLAG_TIMEOUT = 0x1, 0x2, 0x4
STATUS_BYTES = 256
_DTYPES = {torch.bfloat16: KVGQA_BF16, torch.int32: KVGQA_I32, torch.float32: KVGQA_F32,
           torch.uint8: KVGQA_U8, torch.float16: KVGQA_F16}


class KvgqaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("bytes", ctypes.c_int64), ("ndim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("device", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 6), ("strides", ctypes.c_int64 * 6)]


class KvgqaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.code = STATUS_NAMES.get(status, str(status))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'` "
                          "or `python kv_cached_gqa_rope_gb300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(KvgqaTensor)
    st = ctypes.c_int
    lib.kvgqa_abi_version.restype = ctypes.c_int
    lib.kvgqa_last_error.restype = ctypes.c_char_p
    lib.rope_kv_store_workspace_size.argtypes = [ctypes.POINTER(ctypes.c_size_t)]
    lib.rope_kv_store_workspace_size.restype = st
    lib.rope_kv_store_out_.argtypes = [P, P, P, P, P, ctypes.c_double, P, P, P, P, ctypes.c_void_p]
    lib.rope_kv_store_out_.restype = st
    lib.cached_gqa_attention_workspace_size.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]
    lib.cached_gqa_attention_workspace_size.restype = st
    lib.cached_gqa_attention_out_.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, ctypes.c_void_p]
    lib.cached_gqa_attention_out_.restype = st
    lib.prefill_gqa_cached_rows_workspace_size.argtypes = [ctypes.c_int64] * 5 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.prefill_gqa_cached_rows_workspace_size.restype = st
    lib.prefill_gqa_cached_rows_out_.argtypes = [P, P, P, P, ctypes.c_double, ctypes.c_float, P, P, P, P, ctypes.c_void_p]
    lib.prefill_gqa_cached_rows_out_.restype = st
    lib.prefill_varlen_gqa_cached_rows_out_.argtypes = [P, P, P, P, P, P, ctypes.c_double, ctypes.c_float,
                                                        P, P, P, P, ctypes.c_void_p]
    lib.prefill_varlen_gqa_cached_rows_out_.restype = st
    lib.cached_gqa_attention_static_scratch_out_.argtypes = [P, P, P, P, P, ctypes.c_float, P, ctypes.c_void_p]
    lib.cached_gqa_attention_static_scratch_out_.restype = st
    lib.decode_step_workspace_size.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]
    lib.decode_step_workspace_size.restype = st
    lib.decode_step_out_.argtypes = [P, P, P, P, P, ctypes.c_double, ctypes.c_float, P, P, P, P, ctypes.c_void_p]
    lib.decode_step_out_.restype = st
    lib.decode_step_single_launch_out_.argtypes = lib.decode_step_out_.argtypes
    lib.decode_step_single_launch_out_.restype = st
    VP = ctypes.c_void_p
    lib.kvgqa_slots_create.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(VP)]
    lib.kvgqa_slots_destroy.argtypes = [VP]
    lib.kvgqa_slots_admit.argtypes = [VP, ctypes.c_int64, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
    lib.kvgqa_slots_release.argtypes = [VP, ctypes.c_int64, ctypes.c_int32]
    lib.kvgqa_slots_step.argtypes = [VP, VP, VP, ctypes.c_int32, VP, ctypes.c_int32, VP]
    lib.kvgqa_slots_query.argtypes = [VP, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                      ctypes.POINTER(ctypes.c_int64)]
    lib.kvgqa_metadata_upload.argtypes = [VP, ctypes.c_int32, P, VP]
    for name in ("kvgqa_slots_create", "kvgqa_slots_destroy", "kvgqa_slots_admit", "kvgqa_slots_release",
                 "kvgqa_slots_step", "kvgqa_slots_query", "kvgqa_metadata_upload"):
        getattr(lib, name).restype = st
    lib.kvgqa_read_status.argtypes = [P, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    lib.kvgqa_read_status.restype = st
    lib.kvgqa_check_bounded_wait.argtypes = [P, ctypes.c_void_p]
    lib.kvgqa_check_bounded_wait.restype = st
    return lib


_lib = _load()

EXPORTED_SYMBOLS = ("kvgqa_abi_version", "kvgqa_last_error", "rope_kv_store_workspace_size",
                    "rope_kv_store_out_", "cached_gqa_attention_workspace_size",
                    "cached_gqa_attention_out_", "prefill_gqa_cached_rows_workspace_size",
                    "prefill_gqa_cached_rows_out_", "kvgqa_read_status",
                    "cached_gqa_attention_static_scratch_out_", "decode_step_workspace_size",
                    "decode_step_out_", "kvgqa_slots_create", "kvgqa_slots_destroy", "kvgqa_slots_admit",
                    "kvgqa_slots_release", "kvgqa_slots_step", "kvgqa_slots_query", "kvgqa_metadata_upload",
                    "prefill_varlen_gqa_cached_rows_out_", "decode_step_single_launch_out_",
                    "kvgqa_check_bounded_wait")


def library() -> ctypes.CDLL:
    return _lib


def abi_version() -> int:
    return _lib.kvgqa_abi_version()


def describe(t: torch.Tensor) -> KvgqaTensor:
    """Non-owning descriptor of a torch tensor (no copy, no check)."""
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    d = KvgqaTensor()
    d.data = t.data_ptr() if t.numel() else None
    st = t.untyped_storage()
    d.bytes = st.nbytes() - t.storage_offset() * t.element_size()
    d.ndim = t.dim()
    d.dtype = _DTYPES[t.dtype]
    d.device = t.device.index if t.device.type == "cuda" else -1
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.strides[i] = t.stride(i)
    return d


def _stream(stream) -> int:
    if stream is None:
        # Without a usable CUDA device there is no current stream; pass the
        # default stream and let the library report the device error.
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else 0
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int):
    if status != 0:
        raise KvgqaError(status, _lib.kvgqa_last_error().decode())


def _ref(d: KvgqaTensor):
    return ctypes.byref(d)


def rope_kv_store_workspace_size() -> int:
    n = ctypes.c_size_t()
    _check(_lib.rope_kv_store_workspace_size(ctypes.byref(n)))
    return n.value


def cached_gqa_attention_workspace_size(A: int, H_q: int, H_kv: int, D: int, device: int = None) -> int:
    if device is None:
        device = torch.cuda.current_device()
    n = ctypes.c_size_t()
    _check(_lib.cached_gqa_attention_workspace_size(A, H_q, H_kv, D, device, ctypes.byref(n)))
    return n.value


def decode_step_workspace_size(A: int, H_q: int, H_kv: int, D: int, device: int = None) -> int:
    if device is None:
        device = torch.cuda.current_device()
    n = ctypes.c_size_t()
    _check(_lib.decode_step_workspace_size(A, H_q, H_kv, D, device, ctypes.byref(n)))
    return n.value


def prefill_gqa_cached_rows_workspace_size(A: int, T: int, H_q: int, H_kv: int, D: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.prefill_gqa_cached_rows_workspace_size(A, T, H_q, H_kv, D, ctypes.byref(n)))
    return n.value


def rope_kv_store_out_(q, k, v, positions, cache_rows, theta, q_out, k_cache, v_cache, workspace,
                       stream=None) -> None:
    ds = [describe(t) for t in (q, k, v, positions, cache_rows)]
    outs = [describe(t) for t in (q_out, k_cache, v_cache, workspace)]
    _check(_lib.rope_kv_store_out_(*map(_ref, ds), float(theta), *map(_ref, outs), _stream(stream)))


def cached_gqa_attention_out_(q_rot, k_cache, v_cache, positions, cache_rows, scale, out, workspace,
                              stream=None) -> None:
    ds = [describe(t) for t in (q_rot, k_cache, v_cache, positions, cache_rows)]
    o, w = describe(out), describe(workspace)
    _check(_lib.cached_gqa_attention_out_(*map(_ref, ds), float(scale), _ref(o), _ref(w), _stream(stream)))


def decode_step_out_(q, k, v, positions, cache_rows, theta, scale, k_cache, v_cache, out, workspace,
                     stream=None) -> None:
    """The whole decode step: the store of rope_kv_store_out_ and the
    attention of cached_gqa_attention_out_ (no q_out), the attention starting
    to stream the cache while the store runs."""
    ds = [describe(t) for t in (q, k, v, positions, cache_rows)]
    outs = [describe(t) for t in (k_cache, v_cache, out, workspace)]
    _check(_lib.decode_step_out_(*map(_ref, ds), float(theta), float(scale), *map(_ref, outs), _stream(stream)))


def decode_step_single_launch_out_(q, k, v, positions, cache_rows, theta, scale, k_cache, v_cache, out, workspace,
                                   stream=None) -> None:
    """decode_step_out_ in one kernel launch (same results, bit for bit)."""
    ds = [describe(t) for t in (q, k, v, positions, cache_rows)]
    outs = [describe(t) for t in (k_cache, v_cache, out, workspace)]
    _check(_lib.decode_step_single_launch_out_(*map(_ref, ds), float(theta), float(scale), *map(_ref, outs),
                                               _stream(stream)))


def cached_gqa_attention_static_scratch_out_(q_rot, k_cache, v_cache, positions, cache_rows, scale, out,
                                             stream=None) -> None:
    """Cached GQA attention without a workspace, for callers that cannot
    allocate device memory: the partials live in the library's own 4 MiB
    static device array, shared by every call (see include/kvgqa.h)."""
    ds = [describe(t) for t in (q_rot, k_cache, v_cache, positions, cache_rows)]
    o = describe(out)
    _check(_lib.cached_gqa_attention_static_scratch_out_(*map(_ref, ds), float(scale), _ref(o), _stream(stream)))


def prefill_gqa_cached_rows_out_(q, k, v, cache_rows, theta, scale, k_cache, v_cache, out, workspace,
                                 stream=None) -> None:
    ds = [describe(t) for t in (q, k, v, cache_rows)]
    outs = [describe(t) for t in (k_cache, v_cache, out, workspace)]
    _check(_lib.prefill_gqa_cached_rows_out_(*map(_ref, ds), float(theta), float(scale),
                                             *map(_ref, outs), _stream(stream)))


def prefill_varlen_gqa_cached_rows_out_(q, k, v, offsets, lengths, cache_rows, theta, scale, k_cache, v_cache,
                                        out, workspace, stream=None) -> None:
    """Prompts of lengths[a] tokens (padded to T) at positions offsets[a]..
    of rows that may already hold a prefix; the workspace is the one of
    prefill_gqa_cached_rows_workspace_size."""
    ds = [describe(t) for t in (q, k, v, offsets, lengths, cache_rows)]
    outs = [describe(t) for t in (k_cache, v_cache, out, workspace)]
    _check(_lib.prefill_varlen_gqa_cached_rows_out_(*map(_ref, ds), float(theta), float(scale),
                                                    *map(_ref, outs), _stream(stream)))


class Prepared:
    """One C-ABI call with its descriptors built once.

    Calling it crosses ctypes and runs the library's host checks and kernel
    launches; nothing is re-marshalled.  It keeps the tensors alive, so their
    addresses stay valid for as long as the object exists (the pattern a
    serving loop with fixed buffers, or a CUDA graph capture, wants)."""

    def __init__(self, fn, args, keep):
        self._fn, self._args, self._keep = fn, args, keep

    def __call__(self) -> None:
        _check(self._fn(*self._args))


def prepare_rope_kv_store_out_(q, k, v, positions, cache_rows, theta, q_out, k_cache, v_cache, workspace,
                               stream=None) -> Prepared:
    ds = [describe(t) for t in (q, k, v, positions, cache_rows, q_out, k_cache, v_cache, workspace)]
    args = (*map(_ref, ds[:5]), ctypes.c_double(theta), *map(_ref, ds[5:]), ctypes.c_void_p(_stream(stream)))
    return Prepared(_lib.rope_kv_store_out_, args,
                    (ds, q, k, v, positions, cache_rows, q_out, k_cache, v_cache, workspace))


def prepare_cached_gqa_attention_out_(q_rot, k_cache, v_cache, positions, cache_rows, scale, out, workspace,
                                      stream=None) -> Prepared:
    ds = [describe(t) for t in (q_rot, k_cache, v_cache, positions, cache_rows, out, workspace)]
    args = (*map(_ref, ds[:5]), ctypes.c_float(scale), *map(_ref, ds[5:]), ctypes.c_void_p(_stream(stream)))
    return Prepared(_lib.cached_gqa_attention_out_, args,
                    (ds, q_rot, k_cache, v_cache, positions, cache_rows, out, workspace))


def prepare_decode_step_out_(q, k, v, positions, cache_rows, theta, scale, k_cache, v_cache, out, workspace,
                             stream=None, single_launch=False) -> Prepared:
    ds = [describe(t) for t in (q, k, v, positions, cache_rows, k_cache, v_cache, out, workspace)]
    args = (*map(_ref, ds[:5]), ctypes.c_double(theta), ctypes.c_float(scale), *map(_ref, ds[5:]),
            ctypes.c_void_p(_stream(stream)))
    fn = _lib.decode_step_single_launch_out_ if single_launch else _lib.decode_step_out_
    return Prepared(fn, args, (ds, q, k, v, positions, cache_rows, k_cache, v_cache, out, workspace))


def prepare_prefill_gqa_cached_rows_out_(q, k, v, cache_rows, theta, scale, k_cache, v_cache, out, workspace,
                                         stream=None) -> Prepared:
    ds = [describe(t) for t in (q, k, v, cache_rows, k_cache, v_cache, out, workspace)]
    args = (*map(_ref, ds[:4]), ctypes.c_double(theta), ctypes.c_float(scale), *map(_ref, ds[4:]),
            ctypes.c_void_p(_stream(stream)))
    return Prepared(_lib.prefill_gqa_cached_rows_out_, args,
                    (ds, q, k, v, cache_rows, k_cache, v_cache, out, workspace))


def prepare_prefill_varlen_gqa_cached_rows_out_(q, k, v, offsets, lengths, cache_rows, theta, scale, k_cache,
                                                v_cache, out, workspace, stream=None) -> Prepared:
    ds = [describe(t) for t in (q, k, v, offsets, lengths, cache_rows, k_cache, v_cache, out, workspace)]
    args = (*map(_ref, ds[:6]), ctypes.c_double(theta), ctypes.c_float(scale), *map(_ref, ds[6:]),
            ctypes.c_void_p(_stream(stream)))
    return Prepared(_lib.prefill_varlen_gqa_cached_rows_out_, args,
                    (ds, q, k, v, offsets, lengths, cache_rows, k_cache, v_cache, out, workspace))


def kvgqa_read_status(workspace, stream=None) -> int:
    """Synchronise the stream, return and clear the workspace status word."""
    w = describe(workspace)
    flags = ctypes.c_int32()
    _check(_lib.kvgqa_read_status(_ref(w), _stream(stream), ctypes.byref(flags)))
    return flags.value


def kvgqa_check_bounded_wait(workspace, stream=None) -> None:
    """Queue the bounded-wait check (include/kvgqa.h); its result is the
    KVGQA_FLAG_TIMEOUT bit that kvgqa_read_status(workspace) then returns."""
    w = describe(workspace)
    _check(_lib.kvgqa_check_bounded_wait(_ref(w), _stream(stream)))


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled workspace (status word clear), 256-byte aligned."""
    return torch.zeros(max(int(nbytes), STATUS_BYTES), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


# ---------------------------------------------------------------------- slots
STOP, LENGTH, CANCEL = 0, 1, 2


class SlotTable:
    """The library's host slot table of the shared KV cache (which request owns
    which cache row, and how many tokens that row holds).  Lowest free row on
    admission, rows freed on stop / length / cancel, one decode step packs the
    [3, capacity] token/position/row metadata (see include/kvgqa.h)."""

    def __init__(self, num_slots: int, max_seq: int):
        h = ctypes.c_void_p()
        _check(_lib.kvgqa_slots_create(num_slots, max_seq, ctypes.byref(h)))
        self._h = h
        self.num_slots, self.max_seq = num_slots, max_seq

    def close(self):
        if self._h:
            _lib.kvgqa_slots_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def admit(self, request: int, prompt_len: int) -> int:
        row = ctypes.c_int32()
        _check(_lib.kvgqa_slots_admit(self._h, int(request), int(prompt_len), ctypes.byref(row)))
        return row.value

    def release(self, request: int, reason: int = STOP) -> None:
        _check(_lib.kvgqa_slots_release(self._h, int(request), int(reason)))

    def step(self, requests, tokens, meta: torch.Tensor):
        """Pack one decode step into the host int32 tensor `meta` [3, capacity];
        returns (A, finished) where finished[i] tells whether request i's row
        became full and was released."""
        import numpy as np
        if meta.dtype != torch.int32 or meta.dim() != 2 or meta.shape[0] != 3 or meta.device.type != "cpu" \
                or not meta.is_contiguous():
            raise ValueError("meta must be a contiguous host int32 tensor [3, capacity]")
        req = np.ascontiguousarray(np.asarray(requests, dtype=np.int64))
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        if tok.shape != req.shape:
            raise ValueError("one token per request")
        fin = np.zeros(len(req), dtype=np.uint8)
        _check(_lib.kvgqa_slots_step(self._h, req.ctypes.data, tok.ctypes.data, len(req), meta.data_ptr(),
                                     meta.shape[1], fin.ctypes.data))
        return len(req), fin.astype(bool)

    def query(self):
        active, free = ctypes.c_int32(), ctypes.c_int32()
        rel = (ctypes.c_int64 * 3)()
        _check(_lib.kvgqa_slots_query(self._h, ctypes.byref(active), ctypes.byref(free), rel))
        return {"active": active.value, "free": free.value,
                "released": {"stop": rel[0], "length": rel[1], "cancel": rel[2]}}


class StepMetadata:
    """Pinned host [3, capacity] int32 metadata and its device copy: one
    host-to-device copy per step, then zero-copy device views of the first A
    entries of each row (tokens, positions, cache_rows)."""

    def __init__(self, capacity: int, device=None):
        self.capacity = capacity
        self.host = torch.zeros(3, capacity, dtype=torch.int32).pin_memory()
        self.device = torch.zeros(3, capacity, dtype=torch.int32,
                                  device=device if device is not None else "cuda")
        self._desc = describe(self.device)

    def upload(self, A: int, stream=None):
        _check(_lib.kvgqa_metadata_upload(self.host.data_ptr(), self.capacity, _ref(self._desc), _stream(stream)))
        d = self.device
        return d[0, :A], d[1, :A], d[2, :A]

