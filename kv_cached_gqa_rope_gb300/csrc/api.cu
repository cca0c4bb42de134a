// C ABI of libkvgqa: descriptor validation and kernel dispatch.
//
// Boundary rules (microLLM-rocm ARCHITECTURE.md, sections "Tensor ownership
// boundary", "Tensor N0 invariants" and "Stable integration boundary";
// operator-development.md, "Public interfaces"): tensors arrive as non-owning
// descriptors; outputs, workspace, device and stream are explicit; zero-sized
// dimensions are valid; negative sizes are rejected; unsupported layouts are
// rejected rather than copied; alias, shape, dtype, device and contiguity
// errors are explicit.  Every check here reads host memory only, so a call
// never waits for the device (except kvgqa_read_status, which exists to wait).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "kvgqa.h"
#include "kvgqa_internal.h"
#include "slots.h"

namespace {

// Prefill workspace: the status block, the rotated queries (A*T*H_q*D 16-bit
// values, rounded up to 256 bytes), then the varlen item order (one int32 per
// (query tile, prompt) pair).
size_t prefill_qrot_bytes(int64_t A, int64_t T, int64_t H_q, int64_t D) {
  return (static_cast<size_t>(A) * T * H_q * D * 2 + 255) / 256 * 256;
}
size_t prefill_workspace_bytes(int64_t A, int64_t T, int64_t H_q, int64_t D) {
  return KVGQA_STATUS_BYTES + prefill_qrot_bytes(A, T, H_q, D) +
         static_cast<size_t>(kvgqa::prefill_order_entries(A, T)) * sizeof(int32_t);
}

thread_local std::string g_last_error;

struct Fail {
  kvgqa_status code;
};

[[noreturn]] void fail(kvgqa_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  throw Fail{code};
}

void check_cuda(cudaError_t e, const char* what) {
  if (e != cudaSuccess) fail(KVGQA_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

int64_t elem_size(int32_t dtype) {
  switch (dtype) {
    case KVGQA_BF16: return 2;
    case KVGQA_F16: return 2;
    case KVGQA_I32: return 4;
    case KVGQA_F32: return 4;
    case KVGQA_U8: return 1;
  }
  return 0;
}

const char* dtype_name(int32_t dtype) {
  switch (dtype) {
    case KVGQA_BF16: return "bf16";
    case KVGQA_F16: return "f16";
    case KVGQA_I32: return "int32";
    case KVGQA_F32: return "float32";
    case KVGQA_U8: return "uint8";
  }
  return "unknown";
}

// Whether the product of the sizes is below `limit`, computed without
// overflow (a product that overflows is not below any limit).  Negative sizes
// are refused later by check_tensor.
bool product_below(std::initializer_list<int64_t> sizes, int64_t limit) {
  int64_t p = 1;
  for (int64_t x : sizes)
    if (__builtin_mul_overflow(p, x, &p)) return false;
  return p < limit;
}

int64_t numel(const kvgqa_tensor& t) {
  int64_t n = 1;
  for (int i = 0; i < t.ndim; ++i) n *= t.shape[i];
  return n;
}

// A view: its name, descriptor and the byte range it touches.
struct View {
  const char* name;
  const kvgqa_tensor* t;
  uintptr_t lo = 0, hi = 0;  // [lo, hi) bytes used
};

// Checks common to every operand that read only the descriptor: rank, dtype,
// non-negative sizes, row-major contiguity, accessible bytes and alignment.
View check_tensor(const char* name, const kvgqa_tensor* t, int ndim, int32_t dtype, int64_t align) {
  if (!t) fail(KVGQA_EINVAL, "%s: null descriptor", name);
  if (t->ndim != ndim) fail(KVGQA_EINVAL, "%s: expected rank %d, got %d", name, ndim, t->ndim);
  if (t->dtype != dtype)
    fail(KVGQA_EDTYPE, "%s: expected %s, got %s", name, dtype_name(dtype), dtype_name(t->dtype));
  for (int i = ndim - 1; i >= 0; --i) {
    if (t->shape[i] < 0) fail(KVGQA_EINVAL, "%s: negative size in dim %d", name, i);
    if (t->strides[i] < 0) fail(KVGQA_ELAYOUT, "%s: negative stride in dim %d", name, i);
  }
  // the byte count, refused rather than wrapped when the sizes overflow 64
  // bits (so no element count below can overflow either)
  // (a tensor with a zero-sized dimension is empty whatever its other sizes)
  bool empty = false;
  for (int i = 0; i < ndim; ++i) empty |= t->shape[i] == 0;
  int64_t bytes = empty ? 0 : elem_size(dtype);
  for (int i = 0; i < ndim && !empty; ++i)
    if (__builtin_mul_overflow(bytes, t->shape[i], &bytes))
      fail(KVGQA_EINVAL, "%s: sizes overflow a 64-bit byte count", name);
  int64_t expect = 1;
  for (int i = ndim - 1; i >= 0; --i) {
    if (t->shape[i] > 1 && t->strides[i] != expect)
      fail(KVGQA_ELAYOUT, "%s: not contiguous row-major (dim %d stride %lld, expected %lld)", name,
           i, (long long)t->strides[i], (long long)expect);
    expect *= t->shape[i];
  }
  View v{name, t};
  if (bytes == 0) return v;
  if (!t->data) fail(KVGQA_EINVAL, "%s: null data with %lld elements", name, (long long)numel(*t));
  if (t->bytes < bytes)
    fail(KVGQA_EINVAL, "%s: view needs %lld bytes, descriptor allows %lld", name, (long long)bytes,
         (long long)t->bytes);
  if (reinterpret_cast<uintptr_t>(t->data) % align)
    fail(KVGQA_ELAYOUT, "%s: data pointer not %lld-byte aligned", name, (long long)align);
  v.lo = reinterpret_cast<uintptr_t>(t->data);
  v.hi = v.lo + static_cast<uintptr_t>(bytes);
  return v;
}

// Storage type of a call (BF16 or IEEE binary16), taken from its first 16-bit
// tensor; every other 16-bit tensor of the call must have the same type.
int32_t storage_type(const kvgqa_tensor* t, const char* name) {
  if (!t) fail(KVGQA_EINVAL, "%s: null descriptor", name);
  if (t->dtype != KVGQA_BF16 && t->dtype != KVGQA_F16)
    fail(KVGQA_EDTYPE, "%s: expected bf16 or f16, got %s", name, dtype_name(t->dtype));
  return t->dtype;
}

// The device checks: the declared device is the current one, and CUDA knows
// the pointer as device (or managed) memory of that device.
void check_device(std::initializer_list<const View*> views, int device) {
  for (const View* v : views) {
    if (v->lo == v->hi) continue;
    const kvgqa_tensor* t = v->t;
    if (t->device != device)
      fail(KVGQA_EDEVICE, "%s: on device %d, current device is %d", v->name, t->device, device);
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, t->data) != cudaSuccess) {
      cudaGetLastError();
      fail(KVGQA_EDEVICE, "%s: pointer not known to CUDA", v->name);
    }
    if ((attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) ||
        attr.device != device)
      fail(KVGQA_EDEVICE, "%s: not device memory of device %d", v->name, device);
  }
}

void require_shape(const View& v, std::initializer_list<int64_t> dims) {
  int i = 0;
  for (int64_t d : dims) {
    if (v.t->shape[i] != d)
      fail(KVGQA_EINVAL, "%s: dim %d is %lld, expected %lld", v.name, i, (long long)v.t->shape[i],
           (long long)d);
    ++i;
  }
}

bool overlap(const View& a, const View& b) {
  return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}

// A written view must not share a byte with any other operand.
void check_no_alias(std::initializer_list<const View*> written,
                    std::initializer_list<const View*> all) {
  for (const View* w : written)
    for (const View* o : all)
      if (w != o && overlap(*w, *o)) fail(KVGQA_EALIAS, "%s overlaps %s", w->name, o->name);
}

int current_device() {
  int dev = -1;
  check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
  return dev;
}

void check_head_dim(int64_t D) {
  if (D <= 0 || D % 2) fail(KVGQA_EINVAL, "head width D=%lld must be even and positive", (long long)D);
  if (D != 64 && D != 128) fail(KVGQA_EUNSUPPORTED, "head width D=%lld: kernels exist for 64 and 128", (long long)D);
}

void check_heads(int64_t H_q, int64_t H_kv) {
  if (H_q <= 0 || H_kv <= 0 || H_q % H_kv)
    fail(KVGQA_EINVAL, "H_q=%lld must be a positive multiple of H_kv=%lld", (long long)H_q, (long long)H_kv);
}

void check_theta(double theta) {
  if (!(theta > 0.0) || !std::isfinite(theta)) fail(KVGQA_EINVAL, "RoPE base theta must be finite and > 0");
}

// 2/pi to 256 bits: floor(2/pi * 2^256), least significant 64-bit word
// first (the binary expansion of 2/pi, evaluated with integer arithmetic
// from Machin's formula for pi).
constexpr uint64_t kTwoOverPi256[4] = {0xfe5163abdebbc561ull, 0xdb6295993c439041ull, 0xfc2757d1f534ddc0ull,
                                       0xa2f9836e4e441529ull};

// The RoPE frequencies f_i = theta^(-2i/D) (doubles) as quarter turns per
// position step, f_i * 2/pi: the exact product of f_i's 53-bit significand
// with the 256-bit constant, from which the 64 bits after the binary point
// (rounded down) and the two bits before it are taken.  The kernels reduce
// pos * f_i modulo pi/2 from these with integer arithmetic.
void fill_rope_freqs(kvgqa::RopeFreqs* out, int D, double theta) {
  for (int i = 0; i < D / 2; ++i) {
    const double f = std::pow(theta, -2.0 * i / D);
    if (!std::isfinite(f) || f < 0.0) fail(KVGQA_EINVAL, "RoPE base theta %g gives a frequency out of range", theta);
    int e = 0;
    const double m = std::frexp(f, &e);  // f = m * 2^e, m in [0.5, 1) (or f = 0)
    const uint64_t M = static_cast<uint64_t>(std::ldexp(m, 53));  // exact: f = M * 2^(e - 53)
    uint64_t P[5];  // M * kTwoOverPi256, so f * 2/pi = P * 2^(e - 53 - 256)
    unsigned __int128 c = 0;
    for (int w = 0; w < 4; ++w) {
      c += static_cast<unsigned __int128>(M) * kTwoOverPi256[w];
      P[w] = static_cast<uint64_t>(c);
      c >>= 64;
    }
    P[4] = static_cast<uint64_t>(c);
    // bits [lo, lo + 64) of P (zero outside it), i.e. floor(P / 2^lo) mod 2^64
    auto bits = [&](int lo) -> uint64_t {
      const int w = lo >= 0 ? lo / 64 : -((-lo + 63) / 64);
      const int sh = lo - 64 * w;
      auto word = [&](int k) -> uint64_t { return k >= 0 && k < 5 ? P[k] : 0; };
      uint64_t r = word(w) >> sh;
      if (sh) r |= word(w + 1) << (64 - sh);
      return r;
    };
    // f * 2/pi * 2^64 = P * 2^(e - 245)
    out->frac[i] = bits(245 - e);
    out->quad[i] = static_cast<uint8_t>(bits(245 - e + 64) & 3);
  }
}

View check_workspace(const kvgqa_tensor* ws, size_t need) {
  if (!ws) fail(KVGQA_EINVAL, "workspace: null descriptor");
  if (ws->ndim != 1 || ws->dtype != KVGQA_U8)
    fail(KVGQA_EWORKSPACE, "workspace: expected a rank-1 uint8 buffer");
  if (ws->shape[0] < static_cast<int64_t>(need))
    fail(KVGQA_EWORKSPACE, "workspace: %lld bytes, need %zu", (long long)ws->shape[0], need);
  if (reinterpret_cast<uintptr_t>(ws->data) % 256)
    fail(KVGQA_EWORKSPACE, "workspace: data pointer not 256-byte aligned");
  return check_tensor("workspace", ws, 1, KVGQA_U8, 256);
}

template <typename F>
kvgqa_status guarded(F&& f) {
  try {
    f();
    g_last_error.clear();
    return KVGQA_OK;
  } catch (const Fail& e) {
    return e.code;
  }
}

}  // namespace

extern "C" {

int kvgqa_abi_version(void) { return KVGQA_ABI_VERSION; }

const char* kvgqa_last_error(void) { return g_last_error.c_str(); }

kvgqa_status rope_kv_store_workspace_size(size_t* bytes) {
  return guarded([&] {
    if (!bytes) fail(KVGQA_EINVAL, "bytes: null");
    *bytes = KVGQA_STATUS_BYTES;
  });
}

kvgqa_status rope_kv_store_out_(const kvgqa_tensor* q, const kvgqa_tensor* k,
                                const kvgqa_tensor* v, const kvgqa_tensor* positions,
                                const kvgqa_tensor* cache_rows, double theta,
                                const kvgqa_tensor* q_out, const kvgqa_tensor* k_cache,
                                const kvgqa_tensor* v_cache, const kvgqa_tensor* workspace,
                                void* stream) {
  return guarded([&] {
    if (!q || !k_cache) fail(KVGQA_EINVAL, "null descriptor");
    if (q->ndim != 3 || k_cache->ndim != 4) fail(KVGQA_EINVAL, "q must be [A,H_q,D], caches [S,H_kv,max_seq,D]");
    const int64_t A = q->shape[0], H_q = q->shape[1], D = q->shape[2];
    const int64_t S = k_cache->shape[0], H_kv = k_cache->shape[1], max_seq = k_cache->shape[2];
    check_head_dim(D);
    check_heads(H_q, H_kv);
    check_theta(theta);
    const int32_t elem = storage_type(q, "q");
    View vq = check_tensor("q", q, 3, elem, 16);
    View vk = check_tensor("k", k, 3, elem, 16);
    View vv = check_tensor("v", v, 3, elem, 16);
    View vp = check_tensor("positions", positions, 1, KVGQA_I32, 4);
    View vr = check_tensor("cache_rows", cache_rows, 1, KVGQA_I32, 4);
    View vqo = check_tensor("q_out", q_out, 3, elem, 16);
    View vkc = check_tensor("k_cache", k_cache, 4, elem, 16);
    View vvc = check_tensor("v_cache", v_cache, 4, elem, 16);
    View vws = check_workspace(workspace, KVGQA_STATUS_BYTES);
    require_shape(vk, {A, H_kv, D});
    require_shape(vv, {A, H_kv, D});
    require_shape(vp, {A});
    require_shape(vr, {A});
    require_shape(vqo, {A, H_q, D});
    require_shape(vkc, {S, H_kv, max_seq, D});
    require_shape(vvc, {S, H_kv, max_seq, D});
    check_no_alias({&vqo, &vkc, &vvc, &vws}, {&vq, &vk, &vv, &vp, &vr, &vqo, &vkc, &vvc, &vws});
    const int dev = current_device();
    check_device({&vq, &vk, &vv, &vp, &vr, &vqo, &vkc, &vvc, &vws}, dev);
    if (A == 0) return;
    if (A > (1ll << 31) - 1) fail(KVGQA_EINVAL, "A too large");
    kvgqa::RopeStoreParams p{};
    p.q = static_cast<const uint16_t*>(q->data);
    p.k = static_cast<const uint16_t*>(k->data);
    p.v = static_cast<const uint16_t*>(v->data);
    p.positions = static_cast<const int32_t*>(positions->data);
    p.cache_rows = static_cast<const int32_t*>(cache_rows->data);
    p.q_out = static_cast<uint16_t*>(q_out->data);
    p.k_cache = static_cast<uint16_t*>(k_cache->data);
    p.v_cache = static_cast<uint16_t*>(v_cache->data);
    p.status = static_cast<int32_t*>(workspace->data);
    p.A = (int)A; p.T = 1; p.H_q = (int)H_q; p.H_kv = (int)H_kv; p.D = (int)D;
    p.S = (int)S; p.max_seq = (int)max_seq;
    p.f16 = elem == KVGQA_F16;
    fill_rope_freqs(&p.freqs, (int)D, theta);
    check_cuda(kvgqa::launch_rope_kv_store(p, 0, static_cast<cudaStream_t>(stream)),
               "rope_kv_store launch");
  });
}

kvgqa_status cached_gqa_attention_workspace_size(int64_t A, int64_t H_q, int64_t H_kv, int64_t D,
                                                 int32_t device, size_t* bytes) {
  return guarded([&] {
    if (!bytes) fail(KVGQA_EINVAL, "bytes: null");
    if (A < 0) fail(KVGQA_EINVAL, "A < 0");
    check_head_dim(D);
    check_heads(H_q, H_kv);
    const int G = (int)(H_q / H_kv);
    if (G > 16) fail(KVGQA_EUNSUPPORTED, "group size %d: decode kernels cover G <= 16", G);
    kvgqa::DecodeLayout lay;
    check_cuda(kvgqa::decode_layout(device, (int)D, kvgqa::decode_group_pad(G), A, H_kv, &lay),
               "decode kernel set-up");
    *bytes = KVGQA_STATUS_BYTES + lay.counter_bytes + lay.partial_bytes;
  });
}

kvgqa_status cached_gqa_attention_out_(const kvgqa_tensor* q_rot, const kvgqa_tensor* k_cache,
                                       const kvgqa_tensor* v_cache, const kvgqa_tensor* positions,
                                       const kvgqa_tensor* cache_rows, float scale,
                                       const kvgqa_tensor* out, const kvgqa_tensor* workspace,
                                       void* stream) {
  return guarded([&] {
    if (!q_rot || !k_cache) fail(KVGQA_EINVAL, "null descriptor");
    if (q_rot->ndim != 3 || k_cache->ndim != 4) fail(KVGQA_EINVAL, "q_rot must be [A,H_q,D], caches [S,H_kv,max_seq,D]");
    const int64_t A = q_rot->shape[0], H_q = q_rot->shape[1], D = q_rot->shape[2];
    const int64_t S = k_cache->shape[0], H_kv = k_cache->shape[1], max_seq = k_cache->shape[2];
    check_head_dim(D);
    check_heads(H_q, H_kv);
    if (!std::isfinite(scale)) fail(KVGQA_EINVAL, "scale must be finite");
    const int G = (int)(H_q / H_kv);
    if (G > 16) fail(KVGQA_EUNSUPPORTED, "group size %d: decode kernels cover G <= 16", G);
    if (A > kvgqa::kMaxActiveRows) fail(KVGQA_EUNSUPPORTED, "A=%lld exceeds %d active rows", (long long)A, kvgqa::kMaxActiveRows);
    if (!product_below({A, H_kv, max_seq}, 1ll << 31)) fail(KVGQA_EUNSUPPORTED, "A*H_kv*max_seq must stay below 2^31");
    const int32_t elem = storage_type(q_rot, "q_rot");
    View vq = check_tensor("q_rot", q_rot, 3, elem, 16);
    View vkc = check_tensor("k_cache", k_cache, 4, elem, 16);
    View vvc = check_tensor("v_cache", v_cache, 4, elem, 16);
    View vp = check_tensor("positions", positions, 1, KVGQA_I32, 4);
    View vr = check_tensor("cache_rows", cache_rows, 1, KVGQA_I32, 4);
    View vo = check_tensor("out", out, 3, elem, 16);
    require_shape(vvc, {S, H_kv, max_seq, D});
    require_shape(vp, {A});
    require_shape(vr, {A});
    require_shape(vo, {A, H_q, D});
    View vws0 = check_workspace(workspace, KVGQA_STATUS_BYTES);
    check_no_alias({&vo, &vws0}, {&vq, &vkc, &vvc, &vp, &vr, &vo, &vws0});
    const int dev = current_device();
    kvgqa::DecodeLayout lay;
    check_cuda(kvgqa::decode_layout(dev, (int)D, kvgqa::decode_group_pad(G), A, H_kv, &lay),
               "decode kernel set-up");
    View vws = check_workspace(workspace, KVGQA_STATUS_BYTES + lay.counter_bytes + lay.partial_bytes);
    check_device({&vq, &vkc, &vvc, &vp, &vr, &vo, &vws}, dev);
    if (A == 0) return;
    kvgqa::DecodeParams p{};
    p.q = static_cast<const uint16_t*>(q_rot->data);
    p.k_cache = static_cast<const uint16_t*>(k_cache->data);
    p.v_cache = static_cast<const uint16_t*>(v_cache->data);
    p.positions = static_cast<const int32_t*>(positions->data);
    p.cache_rows = static_cast<const int32_t*>(cache_rows->data);
    p.out = static_cast<uint16_t*>(out->data);
    unsigned char* ws = static_cast<unsigned char*>(workspace->data);
    p.status = reinterpret_cast<int32_t*>(ws);
    p.counters = reinterpret_cast<int32_t*>(ws + KVGQA_STATUS_BYTES);
    p.partials = reinterpret_cast<float*>(ws + KVGQA_STATUS_BYTES + lay.counter_bytes);
    p.A = (int)A; p.H_q = (int)H_q; p.H_kv = (int)H_kv; p.G = G; p.D = (int)D;
    p.S = (int)S; p.max_seq = (int)max_seq; p.num_ctas = lay.num_ctas;
    p.f16 = elem == KVGQA_F16;
    p.scale_log2 = scale * 1.4426950408889634f;
    check_cuda(kvgqa::launch_cached_gqa_attention(p, static_cast<cudaStream_t>(stream)),
               "cached_gqa_attention launch");
  });
}

namespace {
// Workspace of the whole decode step: the attention call's (status block,
// counters, partials), then the rotated queries [A, H_q, D] bf16.
size_t step_q_offset(const kvgqa::DecodeLayout& lay) {
  return (KVGQA_STATUS_BYTES + lay.counter_bytes + lay.partial_bytes + 255) / 256 * 256;
}
}  // namespace

kvgqa_status decode_step_workspace_size(int64_t A, int64_t H_q, int64_t H_kv, int64_t D, int32_t device,
                                        size_t* bytes) {
  return guarded([&] {
    if (!bytes) fail(KVGQA_EINVAL, "bytes: null");
    if (A < 0) fail(KVGQA_EINVAL, "A < 0");
    check_head_dim(D);
    check_heads(H_q, H_kv);
    const int G = (int)(H_q / H_kv);
    if (G > 16) fail(KVGQA_EUNSUPPORTED, "group size %d: decode kernels cover G <= 16", G);
    if (!product_below({A, H_q, D, 4}, 1ll << 62)) fail(KVGQA_EINVAL, "sizes overflow a 64-bit byte count");
    kvgqa::DecodeLayout lay;
    check_cuda(kvgqa::decode_layout(device, (int)D, kvgqa::decode_group_pad(G), A, H_kv, &lay),
               "decode kernel set-up");
    *bytes = step_q_offset(lay) + static_cast<size_t>(A) * H_q * D * 2;
  });
}

namespace {
// The whole decode step.  Two launches (default): the store kernel, then the
// attention with an early start.  Single launch: the attention kernel in its
// fused form rotates the queries and stores the new cells itself.
void decode_step_body(const kvgqa_tensor* q, const kvgqa_tensor* k, const kvgqa_tensor* v,
                      const kvgqa_tensor* positions, const kvgqa_tensor* cache_rows, double theta, float scale,
                      const kvgqa_tensor* k_cache, const kvgqa_tensor* v_cache, const kvgqa_tensor* out,
                      const kvgqa_tensor* workspace, void* stream, bool single_launch) {
    if (!q || !k_cache) fail(KVGQA_EINVAL, "null descriptor");
    if (q->ndim != 3 || k_cache->ndim != 4) fail(KVGQA_EINVAL, "q must be [A,H_q,D], caches [S,H_kv,max_seq,D]");
    const int64_t A = q->shape[0], H_q = q->shape[1], D = q->shape[2];
    const int64_t S = k_cache->shape[0], H_kv = k_cache->shape[1], max_seq = k_cache->shape[2];
    check_head_dim(D);
    check_heads(H_q, H_kv);
    check_theta(theta);
    if (!std::isfinite(scale)) fail(KVGQA_EINVAL, "scale must be finite");
    const int G = (int)(H_q / H_kv);
    if (G > 16) fail(KVGQA_EUNSUPPORTED, "group size %d: decode kernels cover G <= 16", G);
    if (A > kvgqa::kMaxActiveRows) fail(KVGQA_EUNSUPPORTED, "A=%lld exceeds %d active rows", (long long)A, kvgqa::kMaxActiveRows);
    if (!product_below({A, H_kv, max_seq}, 1ll << 31)) fail(KVGQA_EUNSUPPORTED, "A*H_kv*max_seq must stay below 2^31");
    const int32_t elem = storage_type(q, "q");
    View vq = check_tensor("q", q, 3, elem, 16);
    View vk = check_tensor("k", k, 3, elem, 16);
    View vv = check_tensor("v", v, 3, elem, 16);
    View vp = check_tensor("positions", positions, 1, KVGQA_I32, 4);
    View vr = check_tensor("cache_rows", cache_rows, 1, KVGQA_I32, 4);
    View vkc = check_tensor("k_cache", k_cache, 4, elem, 16);
    View vvc = check_tensor("v_cache", v_cache, 4, elem, 16);
    View vo = check_tensor("out", out, 3, elem, 16);
    require_shape(vk, {A, H_kv, D});
    require_shape(vv, {A, H_kv, D});
    require_shape(vp, {A});
    require_shape(vr, {A});
    require_shape(vvc, {S, H_kv, max_seq, D});
    require_shape(vo, {A, H_q, D});
    View vws0 = check_workspace(workspace, KVGQA_STATUS_BYTES);
    check_no_alias({&vkc, &vvc, &vo, &vws0}, {&vq, &vk, &vv, &vp, &vr, &vkc, &vvc, &vo, &vws0});
    const int dev = current_device();
    kvgqa::DecodeLayout lay;
    check_cuda(kvgqa::decode_layout(dev, (int)D, kvgqa::decode_group_pad(G), A, H_kv, &lay),
               "decode kernel set-up");
    const size_t q_off = step_q_offset(lay);
    View vws = check_workspace(workspace, q_off + static_cast<size_t>(A) * H_q * D * 2);
    check_device({&vq, &vk, &vv, &vp, &vr, &vkc, &vvc, &vo, &vws}, dev);
    if (A == 0) return;
    unsigned char* ws = static_cast<unsigned char*>(workspace->data);
    uint16_t* q_rot = reinterpret_cast<uint16_t*>(ws + q_off);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (single_launch) {
      kvgqa::DecodeParams p{};
      p.q = static_cast<const uint16_t*>(q->data);
      p.k_cache = static_cast<const uint16_t*>(k_cache->data);
      p.v_cache = static_cast<const uint16_t*>(v_cache->data);
      p.positions = static_cast<const int32_t*>(positions->data);
      p.cache_rows = static_cast<const int32_t*>(cache_rows->data);
      p.out = static_cast<uint16_t*>(out->data);
      p.status = reinterpret_cast<int32_t*>(ws);
      p.counters = reinterpret_cast<int32_t*>(ws + KVGQA_STATUS_BYTES);
      p.partials = reinterpret_cast<float*>(ws + KVGQA_STATUS_BYTES + lay.counter_bytes);
      p.A = (int)A; p.H_q = (int)H_q; p.H_kv = (int)H_kv; p.G = G; p.D = (int)D;
      p.S = (int)S; p.max_seq = (int)max_seq; p.num_ctas = lay.num_ctas;
      p.f16 = elem == KVGQA_F16;
      p.scale_log2 = scale * 1.4426950408889634f;
      p.fused = 1;
      p.k_new = static_cast<const uint16_t*>(k->data);
      p.v_new = static_cast<const uint16_t*>(v->data);
      p.k_cache_w = static_cast<uint16_t*>(k_cache->data);
      p.v_cache_w = static_cast<uint16_t*>(v_cache->data);
      fill_rope_freqs(&p.freqs, (int)D, theta);
      check_cuda(kvgqa::launch_cached_gqa_attention(p, st), "decode_step launch");
      return;
    }
    // 1. the store kernel: rotated queries into the workspace, new cells
    kvgqa::RopeStoreParams rp{};
    rp.q = static_cast<const uint16_t*>(q->data);
    rp.k = static_cast<const uint16_t*>(k->data);
    rp.v = static_cast<const uint16_t*>(v->data);
    rp.positions = static_cast<const int32_t*>(positions->data);
    rp.cache_rows = static_cast<const int32_t*>(cache_rows->data);
    rp.q_out = q_rot;
    rp.k_cache = static_cast<uint16_t*>(k_cache->data);
    rp.v_cache = static_cast<uint16_t*>(v_cache->data);
    rp.status = reinterpret_cast<int32_t*>(ws);
    rp.A = (int)A; rp.T = 1; rp.H_q = (int)H_q; rp.H_kv = (int)H_kv; rp.D = (int)D;
    rp.S = (int)S; rp.max_seq = (int)max_seq;
    rp.f16 = elem == KVGQA_F16;
    fill_rope_freqs(&rp.freqs, (int)D, theta);
    check_cuda(kvgqa::launch_rope_kv_store(rp, 0, st), "decode_step store launch");
    // 2. the attention, started while the store kernel runs: it streams the
    // cache tiles without a new cell before waiting for it
    kvgqa::DecodeParams p{};
    p.q = q_rot;
    p.k_cache = rp.k_cache;
    p.v_cache = rp.v_cache;
    p.positions = rp.positions;
    p.cache_rows = rp.cache_rows;
    p.out = static_cast<uint16_t*>(out->data);
    p.status = rp.status;
    p.counters = reinterpret_cast<int32_t*>(ws + KVGQA_STATUS_BYTES);
    p.partials = reinterpret_cast<float*>(ws + KVGQA_STATUS_BYTES + lay.counter_bytes);
    p.A = (int)A; p.H_q = (int)H_q; p.H_kv = (int)H_kv; p.G = G; p.D = (int)D;
    p.S = (int)S; p.max_seq = (int)max_seq; p.num_ctas = lay.num_ctas;
    p.f16 = elem == KVGQA_F16;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.early = 1;
    check_cuda(kvgqa::launch_cached_gqa_attention(p, st), "decode_step attention launch");
}
}  // namespace

kvgqa_status decode_step_out_(const kvgqa_tensor* q, const kvgqa_tensor* k, const kvgqa_tensor* v,
                              const kvgqa_tensor* positions, const kvgqa_tensor* cache_rows, double theta,
                              float scale, const kvgqa_tensor* k_cache, const kvgqa_tensor* v_cache,
                              const kvgqa_tensor* out, const kvgqa_tensor* workspace, void* stream) {
  return guarded([&] {
    decode_step_body(q, k, v, positions, cache_rows, theta, scale, k_cache, v_cache, out, workspace, stream, false);
  });
}

kvgqa_status decode_step_single_launch_out_(const kvgqa_tensor* q, const kvgqa_tensor* k, const kvgqa_tensor* v,
                                            const kvgqa_tensor* positions, const kvgqa_tensor* cache_rows,
                                            double theta, float scale, const kvgqa_tensor* k_cache,
                                            const kvgqa_tensor* v_cache, const kvgqa_tensor* out,
                                            const kvgqa_tensor* workspace, void* stream) {
  return guarded([&] {
    decode_step_body(q, k, v, positions, cache_rows, theta, scale, k_cache, v_cache, out, workspace, stream, true);
  });
}

kvgqa_status cached_gqa_attention_static_scratch_out_(const kvgqa_tensor* q_rot,
                                                      const kvgqa_tensor* k_cache,
                                                      const kvgqa_tensor* v_cache,
                                                      const kvgqa_tensor* positions,
                                                      const kvgqa_tensor* cache_rows, float scale,
                                                      const kvgqa_tensor* out, void* stream) {
  return guarded([&] {
    if (!q_rot || !k_cache) fail(KVGQA_EINVAL, "null descriptor");
    if (q_rot->ndim != 3 || k_cache->ndim != 4) fail(KVGQA_EINVAL, "q_rot must be [A,H_q,D], caches [S,H_kv,max_seq,D]");
    const int64_t A = q_rot->shape[0], H_q = q_rot->shape[1], D = q_rot->shape[2];
    const int64_t S = k_cache->shape[0], H_kv = k_cache->shape[1], max_seq = k_cache->shape[2];
    check_head_dim(D);
    check_heads(H_q, H_kv);
    if (!std::isfinite(scale)) fail(KVGQA_EINVAL, "scale must be finite");
    const int G = (int)(H_q / H_kv);
    if (G > 16) fail(KVGQA_EUNSUPPORTED, "group size %d: decode kernels cover G <= 16", G);
    if (A > kvgqa::kMaxActiveRows) fail(KVGQA_EUNSUPPORTED, "A=%lld exceeds %d active rows", (long long)A, kvgqa::kMaxActiveRows);
    if (!product_below({A, H_kv, max_seq}, 1ll << 31)) fail(KVGQA_EUNSUPPORTED, "A*H_kv*max_seq must stay below 2^31");
    const int32_t elem = storage_type(q_rot, "q_rot");
    View vq = check_tensor("q_rot", q_rot, 3, elem, 16);
    View vkc = check_tensor("k_cache", k_cache, 4, elem, 16);
    View vvc = check_tensor("v_cache", v_cache, 4, elem, 16);
    View vp = check_tensor("positions", positions, 1, KVGQA_I32, 4);
    View vr = check_tensor("cache_rows", cache_rows, 1, KVGQA_I32, 4);
    View vo = check_tensor("out", out, 3, elem, 16);
    require_shape(vvc, {S, H_kv, max_seq, D});
    require_shape(vp, {A});
    require_shape(vr, {A});
    require_shape(vo, {A, H_q, D});
    check_no_alias({&vo}, {&vq, &vkc, &vvc, &vp, &vr, &vo});
    const int dev = current_device();
    check_device({&vq, &vkc, &vvc, &vp, &vr, &vo}, dev);
    kvgqa::DecodeLayout lay;
    check_cuda(kvgqa::decode_layout(dev, (int)D, kvgqa::decode_group_pad(G), A, H_kv, &lay),
               "decode kernel set-up");
    const size_t need = KVGQA_STATUS_BYTES + lay.counter_bytes + lay.partial_bytes;
    if (need > kvgqa::kStaticScratchBytes)
      fail(KVGQA_EUNSUPPORTED, "needs %zu bytes of scratch; the library's static scratch holds %zu",
           need, kvgqa::kStaticScratchBytes);
    void* scratch = nullptr;
    check_cuda(kvgqa::static_scratch_address(dev, &scratch), "static scratch address");
    if (A == 0) return;
    // The status word and the per-(row, KV head) counters start every call at
    // zero: a call whose bounded wait gave up leaves counters it never
    // completed, and this variant has no status word for the caller to see it.
    check_cuda(cudaMemsetAsync(scratch, 0, KVGQA_STATUS_BYTES + lay.counter_bytes, static_cast<cudaStream_t>(stream)),
               "static scratch clear");
    kvgqa::DecodeParams p{};
    p.q = static_cast<const uint16_t*>(q_rot->data);
    p.k_cache = static_cast<const uint16_t*>(k_cache->data);
    p.v_cache = static_cast<const uint16_t*>(v_cache->data);
    p.positions = static_cast<const int32_t*>(positions->data);
    p.cache_rows = static_cast<const int32_t*>(cache_rows->data);
    p.out = static_cast<uint16_t*>(out->data);
    unsigned char* sc = static_cast<unsigned char*>(scratch);
    p.status = reinterpret_cast<int32_t*>(sc);
    p.counters = reinterpret_cast<int32_t*>(sc + KVGQA_STATUS_BYTES);
    p.partials = reinterpret_cast<float*>(sc + KVGQA_STATUS_BYTES + lay.counter_bytes);
    p.A = (int)A; p.H_q = (int)H_q; p.H_kv = (int)H_kv; p.G = G; p.D = (int)D;
    p.S = (int)S; p.max_seq = (int)max_seq; p.num_ctas = lay.num_ctas;
    p.f16 = elem == KVGQA_F16;
    p.scale_log2 = scale * 1.4426950408889634f;
    check_cuda(kvgqa::launch_cached_gqa_attention(p, static_cast<cudaStream_t>(stream)),
               "cached_gqa_attention launch");
  });
}

kvgqa_status prefill_gqa_cached_rows_workspace_size(int64_t A, int64_t T, int64_t H_q, int64_t H_kv,
                                                    int64_t D, size_t* bytes) {
  return guarded([&] {
    if (!bytes) fail(KVGQA_EINVAL, "bytes: null");
    if (A < 0 || T < 0) fail(KVGQA_EINVAL, "negative size");
    check_head_dim(D);
    check_heads(H_q, H_kv);
    if (!product_below({A, T, H_q, D, 4}, 1ll << 62)) fail(KVGQA_EINVAL, "sizes overflow a 64-bit byte count");
    *bytes = prefill_workspace_bytes(A, T, H_q, D);
  });
}

}  // extern "C"

namespace {

// The equal-length prefill (offsets = lengths = nullptr) and the prefill of
// prompts of different lengths at position offsets share this body.
void prefill_body(const kvgqa_tensor* q, const kvgqa_tensor* k, const kvgqa_tensor* v, const kvgqa_tensor* offsets,
                  const kvgqa_tensor* lengths, const kvgqa_tensor* cache_rows, double theta, float scale,
                  const kvgqa_tensor* k_cache, const kvgqa_tensor* v_cache, const kvgqa_tensor* out,
                  const kvgqa_tensor* workspace, void* stream) {
  if (!q || !k_cache) fail(KVGQA_EINVAL, "null descriptor");
  if (q->ndim != 4 || k_cache->ndim != 4) fail(KVGQA_EINVAL, "q must be [A,T,H_q,D], caches [S,H_kv,max_seq,D]");
  const bool varlen = offsets != nullptr || lengths != nullptr;
  const int64_t A = q->shape[0], T = q->shape[1], H_q = q->shape[2], D = q->shape[3];
  const int64_t S = k_cache->shape[0], H_kv = k_cache->shape[1], max_seq = k_cache->shape[2];
  check_head_dim(D);
  check_heads(H_q, H_kv);
  check_theta(theta);
  if (!std::isfinite(scale)) fail(KVGQA_EINVAL, "scale must be finite");
  if (T > max_seq) fail(KVGQA_EINVAL, "T=%lld exceeds max_seq=%lld", (long long)T, (long long)max_seq);
  if (!product_below({A, T}, 1ll << 31)) fail(KVGQA_EUNSUPPORTED, "A*T must stay below 2^31");
  const int32_t elem = storage_type(q, "q");
  View vq = check_tensor("q", q, 4, elem, 16);
  View vk = check_tensor("k", k, 4, elem, 16);
  View vv = check_tensor("v", v, 4, elem, 16);
  View vr = check_tensor("cache_rows", cache_rows, 1, KVGQA_I32, 4);
  View vkc = check_tensor("k_cache", k_cache, 4, elem, 16);
  View vvc = check_tensor("v_cache", v_cache, 4, elem, 16);
  View vo = check_tensor("out", out, 4, elem, 16);
  require_shape(vk, {A, T, H_kv, D});
  require_shape(vv, {A, T, H_kv, D});
  require_shape(vr, {A});
  require_shape(vvc, {S, H_kv, max_seq, D});
  require_shape(vo, {A, T, H_q, D});
  View voff{}, vlen{};
  if (varlen) {
    voff = check_tensor("offsets", offsets, 1, KVGQA_I32, 4);
    vlen = check_tensor("lengths", lengths, 1, KVGQA_I32, 4);
    require_shape(voff, {A});
    require_shape(vlen, {A});
  }
  View vws = check_workspace(workspace, prefill_workspace_bytes(A, T, H_q, D));
  if (varlen) {
    check_no_alias({&vkc, &vvc, &vo, &vws}, {&vq, &vk, &vv, &vr, &voff, &vlen, &vkc, &vvc, &vo, &vws});
  } else {
    check_no_alias({&vkc, &vvc, &vo, &vws}, {&vq, &vk, &vv, &vr, &vkc, &vvc, &vo, &vws});
  }
  const int dev = current_device();
  if (varlen) {
    check_device({&vq, &vk, &vv, &vr, &voff, &vlen, &vkc, &vvc, &vo, &vws}, dev);
  } else {
    check_device({&vq, &vk, &vv, &vr, &vkc, &vvc, &vo, &vws}, dev);
  }
  if (A == 0 || T == 0) return;
  kvgqa::RopeStoreParams rp{};
  unsigned char* ws = static_cast<unsigned char*>(workspace->data);
  uint16_t* q_rot = reinterpret_cast<uint16_t*>(ws + KVGQA_STATUS_BYTES);
  int32_t* order = reinterpret_cast<int32_t*>(ws + KVGQA_STATUS_BYTES + prefill_qrot_bytes(A, T, H_q, D));
  rp.q = static_cast<const uint16_t*>(q->data);
  rp.k = static_cast<const uint16_t*>(k->data);
  rp.v = static_cast<const uint16_t*>(v->data);
  rp.positions = nullptr;
  rp.cache_rows = static_cast<const int32_t*>(cache_rows->data);
  rp.offsets = varlen ? static_cast<const int32_t*>(offsets->data) : nullptr;
  rp.lengths = varlen ? static_cast<const int32_t*>(lengths->data) : nullptr;
  rp.q_out = q_rot;
  rp.item_order = varlen ? order : nullptr;
  rp.k_cache = static_cast<uint16_t*>(k_cache->data);
  rp.v_cache = static_cast<uint16_t*>(v_cache->data);
  rp.status = reinterpret_cast<int32_t*>(ws);
  rp.A = (int)A; rp.T = (int)T; rp.H_q = (int)H_q; rp.H_kv = (int)H_kv; rp.D = (int)D;
  rp.S = (int)S; rp.max_seq = (int)max_seq;
  rp.f16 = elem == KVGQA_F16;
  fill_rope_freqs(&rp.freqs, (int)D, theta);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  check_cuda(kvgqa::launch_rope_kv_store(rp, varlen ? 2 : 1, st), "prefill rope_kv_store launch");
  kvgqa::PrefillParams pp{};
  pp.q_rot = q_rot;
  pp.k_cache = rp.k_cache;
  pp.v_cache = rp.v_cache;
  pp.cache_rows = rp.cache_rows;
  pp.offsets = rp.offsets;
  pp.lengths = rp.lengths;
  pp.item_order = rp.item_order;
  pp.out = static_cast<uint16_t*>(out->data);
  pp.status = rp.status;
  pp.A = (int)A; pp.T = (int)T; pp.H_q = (int)H_q; pp.H_kv = (int)H_kv; pp.G = (int)(H_q / H_kv);
  pp.D = (int)D; pp.S = (int)S; pp.max_seq = (int)max_seq;
  pp.f16 = elem == KVGQA_F16;
  pp.scale_log2 = scale * 1.4426950408889634f;
  check_cuda(kvgqa::launch_prefill_attention(pp, st), "prefill attention launch");
}

}  // namespace

extern "C" {

kvgqa_status prefill_gqa_cached_rows_out_(const kvgqa_tensor* q, const kvgqa_tensor* k,
                                          const kvgqa_tensor* v, const kvgqa_tensor* cache_rows,
                                          double theta, float scale, const kvgqa_tensor* k_cache,
                                          const kvgqa_tensor* v_cache, const kvgqa_tensor* out,
                                          const kvgqa_tensor* workspace, void* stream) {
  return guarded([&] {
    prefill_body(q, k, v, nullptr, nullptr, cache_rows, theta, scale, k_cache, v_cache, out, workspace, stream);
  });
}

kvgqa_status prefill_varlen_gqa_cached_rows_out_(const kvgqa_tensor* q, const kvgqa_tensor* k,
                                                 const kvgqa_tensor* v, const kvgqa_tensor* offsets,
                                                 const kvgqa_tensor* lengths, const kvgqa_tensor* cache_rows,
                                                 double theta, float scale, const kvgqa_tensor* k_cache,
                                                 const kvgqa_tensor* v_cache, const kvgqa_tensor* out,
                                                 const kvgqa_tensor* workspace, void* stream) {
  return guarded([&] {
    if (!offsets || !lengths) fail(KVGQA_EINVAL, "offsets/lengths: null descriptor");
    prefill_body(q, k, v, offsets, lengths, cache_rows, theta, scale, k_cache, v_cache, out, workspace, stream);
  });
}

struct kvgqa_slots {
  kvgqa::SlotTable table;
};

kvgqa_status kvgqa_slots_create(int32_t num_slots, int32_t max_seq, kvgqa_slots** out) {
  return guarded([&] {
    if (!out) fail(KVGQA_EINVAL, "out: null");
    if (num_slots <= 0 || max_seq <= 0) fail(KVGQA_EINVAL, "num_slots and max_seq must be positive");
    *out = new kvgqa_slots{kvgqa::SlotTable(num_slots, max_seq)};
  });
}

kvgqa_status kvgqa_slots_destroy(kvgqa_slots* slots) {
  return guarded([&] { delete slots; });
}

kvgqa_status kvgqa_slots_admit(kvgqa_slots* slots, int64_t request, int32_t prompt_len, int32_t* row) {
  return guarded([&] {
    if (!slots || !row) fail(KVGQA_EINVAL, "null argument");
    if (prompt_len < 0 || prompt_len > slots->table.max_seq())
      fail(KVGQA_EINVAL, "prompt_len %d outside [0, max_seq=%d]", prompt_len, slots->table.max_seq());
    const int r = slots->table.admit(request, prompt_len);
    if (r < 0) fail(KVGQA_EFULL, "no free cache row (%d rows in use)", slots->table.active());
    *row = r;
  });
}

kvgqa_status kvgqa_slots_release(kvgqa_slots* slots, int64_t request, int32_t reason) {
  return guarded([&] {
    if (!slots) fail(KVGQA_EINVAL, "null argument");
    if (reason < 0 || reason > 2) fail(KVGQA_EINVAL, "reason must be 0 (stop), 1 (length) or 2 (cancel)");
    if (!slots->table.release(request, static_cast<kvgqa::SlotTable::Reason>(reason)))
      fail(KVGQA_EINVAL, "request %lld holds no row", (long long)request);
  });
}

kvgqa_status kvgqa_slots_step(kvgqa_slots* slots, const int64_t* requests, const int32_t* tokens, int32_t n,
                              int32_t* meta, int32_t capacity, uint8_t* finished) {
  return guarded([&] {
    if (!slots || !meta || (n > 0 && !requests)) fail(KVGQA_EINVAL, "null argument");
    if (n < 0 || n > capacity) fail(KVGQA_EINVAL, "n=%d must lie in [0, capacity=%d]", n, capacity);
    const int bad = slots->table.step(requests, tokens, n, meta, capacity, finished);
    if (bad >= 0)
      fail(KVGQA_EINVAL, "request %lld (entry %d) is not admitted, is repeated, or its row is full",
           (long long)requests[bad], bad);
  });
}

kvgqa_status kvgqa_slots_query(const kvgqa_slots* slots, int32_t* active, int32_t* free_rows, int64_t released[3]) {
  return guarded([&] {
    if (!slots) fail(KVGQA_EINVAL, "null argument");
    if (active) *active = slots->table.active();
    if (free_rows) *free_rows = slots->table.num_slots() - slots->table.active();
    if (released)
      for (int i = 0; i < 3; ++i) released[i] = slots->table.released(static_cast<kvgqa::SlotTable::Reason>(i));
  });
}

kvgqa_status kvgqa_metadata_upload(const int32_t* host_meta, int32_t capacity, const kvgqa_tensor* device_meta,
                                   void* stream) {
  return guarded([&] {
    if (!host_meta) fail(KVGQA_EINVAL, "host_meta: null");
    if (capacity <= 0) fail(KVGQA_EINVAL, "capacity must be positive");
    View vm = check_tensor("device_meta", device_meta, 2, KVGQA_I32, 4);
    require_shape(vm, {3, capacity});
    const int dev = current_device();
    check_device({&vm}, dev);
    check_cuda(cudaMemcpyAsync(device_meta->data, host_meta, sizeof(int32_t) * 3 * static_cast<size_t>(capacity),
                               cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)),
               "metadata copy");
  });
}

kvgqa_status kvgqa_check_bounded_wait(const kvgqa_tensor* workspace, void* stream) {
  return guarded([&] {
    View vws = check_workspace(workspace, KVGQA_STATUS_BYTES);
    check_device({&vws}, current_device());
    check_cuda(kvgqa::launch_bounded_wait_check(static_cast<int32_t*>(workspace->data),
                                                static_cast<cudaStream_t>(stream)),
               "bounded-wait check launch");
  });
}

kvgqa_status kvgqa_read_status(const kvgqa_tensor* workspace, void* stream, int32_t* flags) {
  return guarded([&] {
    if (!flags) fail(KVGQA_EINVAL, "flags: null");
    View vws = check_workspace(workspace, KVGQA_STATUS_BYTES);
    check_device({&vws}, current_device());
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t h = 0;
    check_cuda(cudaMemcpyAsync(&h, workspace->data, sizeof h, cudaMemcpyDeviceToHost, st), "status read");
    check_cuda(cudaMemsetAsync(workspace->data, 0, sizeof h, st), "status clear");
    check_cuda(cudaStreamSynchronize(st), "stream synchronize");
    if (h & KVGQA_FLAG_TIMEOUT) {
      // A call that gave up on a wait may have left split-K counters short of
      // their count; a zero-filled workspace is ready for any call again.
      check_cuda(cudaMemsetAsync(workspace->data, 0, static_cast<size_t>(workspace->shape[0]), st), "workspace clear");
      check_cuda(cudaStreamSynchronize(st), "stream synchronize");
    }
    *flags = h;
  });
}

}  // extern "C"
