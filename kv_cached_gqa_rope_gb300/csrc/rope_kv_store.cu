// K1: split-half RoPE of Q and K at each token's own position, fused with the
// K/V store into the token's cache cell.
//
// microLLM-rocm ARCHITECTURE.md, section "Tensor ownership boundary": device
// positions[A] and cache_rows[A] parameterise decode-only RoPE and the K/V
// store; inactive full-capacity rows stay untouched.  Section "Attention layout
// boundary": split-half RoPE needs an even head width, a nonnegative position
// and a positive base.  The same kernel serves the prefill into empty rows,
// where token (a, t) sits at position t of row cache_rows[a].
//
// Equal-length prefill: one CTA owns one position.  It evaluates the D/2
// cos/sin of pos * theta^(-2i/D) once (rope_cos_sin: integer reduction
// modulo pi/2, double-float series) and keeps them as FP32 hi+lo pairs in
// shared memory; the A tokens at that position then stream their heads
// through 16-byte vector loads and stores.  Decode: kTokenSplit CTAs share a
// token, each owning a quarter of the frequencies of every head (and a
// quarter of its V bytes), so that the angle work of a token is spread over
// four SMs; each CTA issues its loads before it evaluates its angles.  The
// prefill of prompts at offsets (one position per token): CTAs take groups of
// consecutive real tokens whole, like the equal-length kernel with per-token
// angles.  The rotation is evaluated with FP32 error-free products so that
// the BF16 result is within one rounding of the exact value even where
// x cos - y sin cancels.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "kvgqa_internal.h"
#include "ptx.cuh"
#include "elem.cuh"
#include "rope_math.cuh"

namespace kvgqa {
namespace {

// The cos/sin table is read eight consecutive entries at a time by lanes that
// differ in which group of eight they read; one 16-byte pad after every eight
// entries puts those lanes on different shared-memory banks.
__device__ __forceinline__ int cs_slot(int i) { return i + (i >> 3); }

// Rotate the 8 pairs (a[i], b[i]) held in two 16-byte chunks of the storage
// type; each result is rounded once (nearest even) back to it.
template <bool F16>
__device__ __forceinline__ void rotate8(const uint4& a, const uint4& b, const CosSin* cs,
                                        uint4& ya, uint4& yb) {
  using E = Elem<F16>;
  // cs points at the padded slot of pair 8c; the eight pairs follow contiguously
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
  uint32_t oa[4], ob[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float2 x1 = E::pair_to_f2(aw[w]);
    const float2 x2 = E::pair_to_f2(bw[w]);
    const CosSin c0 = cs[2 * w], c1 = cs[2 * w + 1];
    oa[w] = E::pack2(rot_first(x1.x, x2.x, c0), rot_first(x1.y, x2.y, c1));
    ob[w] = E::pack2(rot_second(x1.x, x2.x, c0), rot_second(x1.y, x2.y, c1));
  }
  ya = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  yb = make_uint4(ob[0], ob[1], ob[2], ob[3]);
}

template <int D, bool F16>
__global__ void __launch_bounds__(256, 4) rope_kv_store_kernel(const __grid_constant__ RopeStoreParams p) {
  constexpr int HALF = D / 2;
  constexpr int RU = D / 16;  // rotation units per head: 8 pairs each
  constexpr int VU = D / 8;   // copy units per head: 8 elements (16 bytes) each
  __shared__ CosSin cs[HALF + HALF / 8];

  // Inputs and outputs may belong to the previous kernel.  The prefill
  // attention kernel launched behind this one (programmatic dependent launch)
  // may start once every CTA here has exited: it needs every SM's whole
  // register file, so an earlier signal would only let it take SMs this
  // kernel's later CTAs still need.
  pdl_wait();
  const int pos = blockIdx.x;  // position t, shared by all A prompts
  const int ntok = p.A;

  for (int i = threadIdx.x; i < HALF; i += blockDim.x)
    cs[cs_slot(i)] = rope_cos_sin(pos, p.freqs.frac[i], p.freqs.quad[i]);
  __syncthreads();

  // The work of this position: every token's rotation units (8 pairs of Q or
  // K) and V copy units (16 bytes).  Each thread takes kBatch items at a time
  // and issues all their loads before using any, so several DRAM round trips
  // overlap (one at a time, the loop is bound by load latency, not bandwidth).
  // Prefill tokens whose cache row is out of range are skipped and flagged.
  constexpr int kBatch = 4;
  if (blockIdx.x == 0) {
    for (int a = threadIdx.x; a < ntok; a += blockDim.x) {
      const int row = p.cache_rows[a];
      if (row < 0 || row >= p.S) atomicOr(p.status, KVGQA_FLAG_ROW_RANGE);
    }
  }
  const int rot_units = (p.H_q + p.H_kv) * RU;
  const int n_rot = ntok * rot_units;
  for (int base = threadIdx.x; base < n_rot; base += kBatch * blockDim.x) {
    uint4 xa[kBatch], xb[kBatch];
    uint16_t* dst[kBatch];
    int cc[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int r = base + u * blockDim.x;
      dst[u] = nullptr;
      if (r >= n_rot) continue;
      const int ti = r / rot_units, rr = r % rot_units;
      const int a = ti;
      const int row = p.cache_rows[a];
      if (row < 0 || row >= p.S) continue;
      const size_t tok = static_cast<size_t>(a) * p.T + pos;
      const int h = rr / RU, c = rr % RU;
      const uint16_t* src;
      if (h < p.H_q) {
        src = p.q + (tok * p.H_q + h) * D;
        dst[u] = p.q_out + (tok * p.H_q + h) * D;
      } else {
        const int g = h - p.H_q;
        src = p.k + (tok * p.H_kv + g) * D;
        dst[u] = p.k_cache + ((static_cast<size_t>(row) * p.H_kv + g) * p.max_seq + pos) * D;
      }
      cc[u] = c;
      xa[u] = *reinterpret_cast<const uint4*>(src + c * 8);
      xb[u] = *reinterpret_cast<const uint4*>(src + HALF + c * 8);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (!dst[u]) continue;
      uint4 ya, yb;
      rotate8<F16>(xa[u], xb[u], cs + cs_slot(cc[u] * 8), ya, yb);
      *reinterpret_cast<uint4*>(dst[u] + cc[u] * 8) = ya;
      *reinterpret_cast<uint4*>(dst[u] + HALF + cc[u] * 8) = yb;
    }
  }
  const int copy_units = p.H_kv * VU;
  const int n_copy = ntok * copy_units;
  for (int base = threadIdx.x; base < n_copy; base += kBatch * blockDim.x) {
    uint4 x[kBatch];
    uint16_t* dst[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int r = base + u * blockDim.x;
      dst[u] = nullptr;
      if (r >= n_copy) continue;
      const int ti = r / copy_units, rr = r % copy_units;
      const int a = ti;
      const int row = p.cache_rows[a];
      if (row < 0 || row >= p.S) continue;
      const size_t tok = static_cast<size_t>(a) * p.T + pos;
      const int g = rr / VU, c = rr % VU;
      dst[u] = p.v_cache + ((static_cast<size_t>(row) * p.H_kv + g) * p.max_seq + pos) * D + c * 8;
      x[u] = *reinterpret_cast<const uint4*>(p.v + (tok * p.H_kv + g) * D + c * 8);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (dst[u]) *reinterpret_cast<uint4*>(dst[u]) = x[u];
  }
}

constexpr int kTokenSplit = 4;     // CTAs per token (decode, prompts at offsets)
constexpr int kTokenThreads = 128;
constexpr int kOrderBins = 512;    // key-tile counts told apart by the item order (larger ones share a bin)

// Prompts at offsets: the attention kernel deals its items (query tile qt of
// prompt a, all head pairs) round-robin over a persistent grid, so it wants
// them longest first, and with prefixes at offsets the query tile index no
// longer orders them.  One CTA (the caller's) counting-sorts the pairs
// c = qt * A + a by their key tiles (the tiles holding positions
// 0 .. off + min(len, qt*T + T) - 1; 0 for a pair with no work or invalid
// metadata, which the attention kernel skips) into p.item_order, most first.
// The order of pairs with equal counts is not fixed; no result depends on it.
__device__ void write_item_order(const RopeStoreParams& p) {
  __shared__ int bins[kOrderBins];
  const int nqt = (p.T + kPrefillTile - 1) / kPrefillTile;
  const int n = p.A * nqt;
  auto key = [&](int c) {
    const int qt = c / p.A, a = c % p.A;
    const int row = p.cache_rows[a], off = p.offsets[a], len = p.lengths[a];
    const bool ok = row >= 0 && row < p.S && len >= 0 && len <= p.T && off >= 0 && off <= p.max_seq - len;
    if (!ok || qt * kPrefillTile >= len) return 0;
    const int kend = off + min(len, qt * kPrefillTile + kPrefillTile);
    return min((kend + kPrefillTile - 1) / kPrefillTile, kOrderBins - 1);
  };
  for (int b = threadIdx.x; b < kOrderBins; b += blockDim.x) bins[b] = 0;
  __syncthreads();
  for (int c = threadIdx.x; c < n; c += blockDim.x) atomicAdd(&bins[key(c)], 1);
  __syncthreads();
  if (threadIdx.x == 0) {  // start of each bin, largest count first
    int run = 0;
    for (int b = kOrderBins - 1; b >= 0; --b) {
      const int cnt = bins[b];
      bins[b] = run;
      run += cnt;
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < n; c += blockDim.x) p.item_order[atomicAdd(&bins[key(c)], 1)] = c;
}

// One token at its own position: decode (token tk = a at positions[a],
// varlen = 0) or the prefill of prompts at offsets (token tk = a*T + t at
// offsets[a] + t, t < lengths[a], varlen = 1).  Part s of the token (one CTA)
// rotates the pairs of frequencies [s*F, s*F + F) of every Q and K head,
// F = D/2 / kTokenSplit, and copies part s of its V bytes.  Returns early,
// uniformly over the CTA, for a token with no work.
template <int D, bool F16>
__device__ __forceinline__ void token_body(const RopeStoreParams& p, int varlen, int tk, int part, CosSin* cs) {
  constexpr int HALF = D / 2;
  constexpr int F = HALF / kTokenSplit;  // frequencies of this CTA
  constexpr int UF = F / 8;              // rotation units (8 pairs) per head
  constexpr int VU = D / 8;              // V copy units (16 bytes) per head
  constexpr int kBatch = 2;
  static_assert(F % 8 == 0, "a CTA's frequencies are whole 16-byte units");
  const size_t tok = tk;  // index in the token-major inputs
  const int rot_items = (p.H_q + p.H_kv) * UF;
  const int copy_per_part = p.H_kv * VU / kTokenSplit;
  const int n_items = rot_items + copy_per_part;

  // Item j < rot_items: unit part*UF + j%UF of head j/UF (Q heads, then K
  // heads); otherwise V copy unit part*copy_per_part + (j - rot_items).  The
  // loads of the first round do not depend on the position or the row, so
  // they are issued before the metadata and the angles are known.
  auto load = [&](int j, uint4& xa, uint4& xb) {
    if (j < rot_items) {
      const int h = j / UF, c = part * UF + j % UF;
      const uint16_t* src = h < p.H_q ? p.q + (tok * p.H_q + h) * D : p.k + (tok * p.H_kv + (h - p.H_q)) * D;
      xa = *reinterpret_cast<const uint4*>(src + c * 8);
      xb = *reinterpret_cast<const uint4*>(src + HALF + c * 8);
    } else {
      const int u = part * copy_per_part + (j - rot_items);
      xa = *reinterpret_cast<const uint4*>(p.v + (tok * p.H_kv + u / VU) * D + (u % VU) * 8);
    }
  };
  // Prompts at offsets are padded to T: a token past its prompt's length
  // has no work, and its CTAs leave before loading anything.
  if (varlen) {
    const int off = p.offsets[tk / p.T], len = p.lengths[tk / p.T];
    const bool meta_ok = len >= 0 && len <= p.T && off >= 0 && off <= p.max_seq - len;
    if (meta_ok && tk % p.T >= len) return;  // (invalid metadata is flagged below)
  }
  uint4 xa[kBatch], xb[kBatch];
#pragma unroll
  for (int b = 0; b < kBatch; ++b) {
    const int j = threadIdx.x + b * kTokenThreads;
    if (j < n_items) load(j, xa[b], xb[b]);
  }

  int a, pos;
  if (!varlen) {
    a = tk;
    pos = p.positions[a];
  } else {
    a = tk / p.T;
    const int t = tk % p.T;
    const int off = p.offsets[a], len = p.lengths[a];
    const bool meta_ok = len >= 0 && len <= p.T && off >= 0 && off <= p.max_seq - len;
    if (meta_ok && t >= len) return;  // past this prompt's tokens
    if (!meta_ok) {
      if (threadIdx.x == 0 && t == 0 && part == 0) atomicOr(p.status, KVGQA_FLAG_POSITION_RANGE);
      return;
    }
    pos = off + t;
  }
  const int row = p.cache_rows[a];
  const bool pos_ok = pos >= 0 && pos < p.max_seq;
  const bool row_ok = row >= 0 && row < p.S;
  if (!pos_ok || !row_ok) {
    if (threadIdx.x == 0 && part == 0 && (!varlen || tk % p.T == 0))
      atomicOr(p.status, (pos_ok ? 0 : KVGQA_FLAG_POSITION_RANGE) | (row_ok ? 0 : KVGQA_FLAG_ROW_RANGE));
    return;
  }

  for (int i = threadIdx.x; i < F; i += kTokenThreads)
    cs[cs_slot(i)] = rope_cos_sin(pos, p.freqs.frac[part * F + i], p.freqs.quad[part * F + i]);
  __syncthreads();

  auto store = [&](int j, const uint4& va, const uint4& vb) {
    if (j < rot_items) {
      const int h = j / UF, cl = j % UF, c = part * UF + cl;
      uint16_t* dst = h < p.H_q ? p.q_out + (tok * p.H_q + h) * D
                                : p.k_cache + ((static_cast<size_t>(row) * p.H_kv + (h - p.H_q)) * p.max_seq + pos) * D;
      uint4 ya, yb;
      rotate8<F16>(va, vb, cs + cs_slot(cl * 8), ya, yb);
      *reinterpret_cast<uint4*>(dst + c * 8) = ya;
      *reinterpret_cast<uint4*>(dst + HALF + c * 8) = yb;
    } else {
      const int u = part * copy_per_part + (j - rot_items);
      *reinterpret_cast<uint4*>(p.v_cache + ((static_cast<size_t>(row) * p.H_kv + u / VU) * p.max_seq + pos) * D +
                                (u % VU) * 8) = va;
    }
  };
#pragma unroll
  for (int b = 0; b < kBatch; ++b) {
    const int j = threadIdx.x + b * kTokenThreads;
    if (j < n_items) store(j, xa[b], xb[b]);
  }
  // more heads than one round covers: the rest, loads first in each round
  for (int base = threadIdx.x + kBatch * kTokenThreads; base < n_items; base += kBatch * kTokenThreads) {
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int j = base + b * kTokenThreads;
      if (j < n_items) load(j, xa[b], xb[b]);
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int j = base + b * kTokenThreads;
      if (j < n_items) store(j, xa[b], xb[b]);
    }
  }
}

// Prompts at offsets with at most this many prompts run in the kernel below,
// which walks only their real tokens; with more prompts the per-token kernel
// walks the padded tokens.
constexpr int kScanPrompts = 2048;
constexpr int kVarlenGroup = 8;     // tokens per CTA and step (prompts at offsets)
constexpr int kVarlenThreads = 256;

// Decode: part s = blockIdx % 4 of token blockIdx / 4 (one token per CTA
// quartet).  Prompts at offsets (more than kScanPrompts of them): a grid sized
// to the GPU walks the padded tokens (stride gridDim / 4), so the tokens past
// a prompt's length cost a loop step, not a CTA launch.
template <int D, bool F16>
__global__ void __launch_bounds__(kTokenThreads) rope_kv_store_token_kernel(const __grid_constant__ RopeStoreParams p,
                                                                          int varlen) {
  constexpr int F = D / 2 / kTokenSplit;
  __shared__ CosSin cs[F + F / 8];
  pdl_wait();               // inputs and outputs may belong to the previous kernel
  if (!varlen) pdl_trigger();  // decode: the attention kernel may launch and set itself up meanwhile
  if (varlen && p.item_order && blockIdx.x == 0) write_item_order(p);
  const int part = blockIdx.x % kTokenSplit;
  const int n_tok = varlen ? p.A * p.T : p.A;
  const int step = gridDim.x / kTokenSplit;
  for (int tk = blockIdx.x / kTokenSplit; tk < n_tok; tk += step) {
    token_body<D, F16>(p, varlen, tk, part, cs);
    __syncthreads();  // cs is rewritten for the next token
  }
}

// Prompts at offsets (at most kScanPrompts of them), real tokens only.  Every
// CTA scans the valid prompts' lengths into shared memory (an invalid prompt
// counts zero tokens; CTA 0 flags it) with their offsets and rows.  The real
// tokens, in prompt order, form groups of kVarlenGroup; a CTA takes whole
// groups (grid stride), maps each token to (prompt, token) by binary search,
// evaluates the D/2 angles of each of the group's tokens into shared memory,
// then streams the group's rotation and copy units as the equal-length kernel
// does, kBatch loads in flight per thread.  A group's tokens are mostly
// consecutive positions of one prompt, so its cache writes are contiguous
// per head, and every head's units are read and written as whole rows.
template <int D, bool F16>
__global__ void __launch_bounds__(kVarlenThreads, 3) rope_kv_store_varlen_kernel(const __grid_constant__ RopeStoreParams p) {
  constexpr int HALF = D / 2;
  constexpr int CSN = HALF + HALF / 8;  // padded cos/sin entries per token
  constexpr int RU = D / 16;            // rotation units per head: 8 pairs each
  constexpr int VU = D / 8;             // copy units per head: 16 bytes each
  constexpr int NB = kVarlenGroup;
  constexpr int kBatch = 4;
  __shared__ CosSin cs[NB * CSN];
  __shared__ int tk_s[NB], pos_s[NB], row_s[NB];
  extern __shared__ int scan[];  // start[A + 1], then off[A], row[A]
  int* start = scan;
  int* off_s = scan + p.A + 1;
  int* rows_s = off_s + p.A;
  pdl_wait();  // (no early signal to the attention kernel behind it: see rope_kv_store_kernel)
  if (p.item_order && blockIdx.x == 0) write_item_order(p);
  for (int a = threadIdx.x; a < p.A; a += blockDim.x) {
    const int off = p.offsets[a], len = p.lengths[a], row = p.cache_rows[a];
    const bool meta_ok = len >= 0 && len <= p.T && off >= 0 && off <= p.max_seq - len;
    const bool row_ok = row >= 0 && row < p.S;
    start[a + 1] = meta_ok && row_ok ? len : 0;
    off_s[a] = off;
    rows_s[a] = row;
    if (blockIdx.x == 0 && !(meta_ok && row_ok))
      atomicOr(p.status, (meta_ok ? 0 : KVGQA_FLAG_POSITION_RANGE) | (row_ok ? 0 : KVGQA_FLAG_ROW_RANGE));
  }
  __syncthreads();
  if (threadIdx.x < 32) {  // exclusive scan by one warp, 32 prompts per step
    int carry = 0;
    for (int base = 0; base < p.A; base += 32) {
      const int a = base + threadIdx.x;
      int v = a < p.A ? start[a + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (threadIdx.x >= o) v += n;
      }
      if (a < p.A) start[a + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (threadIdx.x == 0) start[0] = 0;
  }
  __syncthreads();
  const int n_real = start[p.A];
  const int rot_units = (p.H_q + p.H_kv) * RU;
  const int copy_units = p.H_kv * VU;
  for (int g0 = blockIdx.x * NB; g0 < n_real; g0 += gridDim.x * NB) {
    if (threadIdx.x < NB) {
      const int idx = g0 + threadIdx.x;
      int t = -1, a = 0;
      if (idx < n_real) {
        int lo = 0, hi = p.A;  // the prompt a with start[a] <= idx < start[a + 1]
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (start[mid] <= idx) lo = mid;
          else hi = mid;
        }
        a = lo;
        t = idx - start[lo];
      }
      tk_s[threadIdx.x] = t < 0 ? -1 : a * p.T + t;
      pos_s[threadIdx.x] = t < 0 ? 0 : off_s[a] + t;
      row_s[threadIdx.x] = rows_s[a];
    }
    __syncthreads();
    const int nb = min(NB, n_real - g0);  // tokens of this group (the last group may be short)
    for (int i = threadIdx.x; i < nb * HALF; i += blockDim.x) {
      const int b = i / HALF, f = i % HALF;
      cs[b * CSN + cs_slot(f)] = rope_cos_sin(pos_s[b], p.freqs.frac[f], p.freqs.quad[f]);
    }
    __syncthreads();
    const int n_rot = nb * rot_units;
    for (int base = threadIdx.x; base < n_rot; base += kBatch * blockDim.x) {
      uint4 xa[kBatch], xb[kBatch];
      uint16_t* dst[kBatch];
      int cc[kBatch], bb[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int r = base + u * blockDim.x;
        dst[u] = nullptr;
        if (r >= n_rot) continue;
        const int b = r / rot_units, rr = r % rot_units;
        const size_t tok = tk_s[b];
        const int h = rr / RU, c = rr % RU;
        const uint16_t* src;
        if (h < p.H_q) {
          src = p.q + (tok * p.H_q + h) * D;
          dst[u] = p.q_out + (tok * p.H_q + h) * D;
        } else {
          const int g = h - p.H_q;
          src = p.k + (tok * p.H_kv + g) * D;
          dst[u] = p.k_cache + ((static_cast<size_t>(row_s[b]) * p.H_kv + g) * p.max_seq + pos_s[b]) * D;
        }
        cc[u] = c;
        bb[u] = b;
        xa[u] = *reinterpret_cast<const uint4*>(src + c * 8);
        xb[u] = *reinterpret_cast<const uint4*>(src + HALF + c * 8);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (!dst[u]) continue;
        uint4 ya, yb;
        rotate8<F16>(xa[u], xb[u], cs + bb[u] * CSN + cs_slot(cc[u] * 8), ya, yb);
        *reinterpret_cast<uint4*>(dst[u] + cc[u] * 8) = ya;
        *reinterpret_cast<uint4*>(dst[u] + HALF + cc[u] * 8) = yb;
      }
    }
    const int n_copy = nb * copy_units;
    for (int base = threadIdx.x; base < n_copy; base += kBatch * blockDim.x) {
      uint4 x[kBatch];
      uint16_t* dst[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int r = base + u * blockDim.x;
        dst[u] = nullptr;
        if (r >= n_copy) continue;
        const int b = r / copy_units, rr = r % copy_units;
        const size_t tok = tk_s[b];
        const int g = rr / VU, c = rr % VU;
        dst[u] = p.v_cache + ((static_cast<size_t>(row_s[b]) * p.H_kv + g) * p.max_seq + pos_s[b]) * D + c * 8;
        x[u] = *reinterpret_cast<const uint4*>(p.v + (tok * p.H_kv + g) * D + c * 8);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (dst[u]) *reinterpret_cast<uint4*>(dst[u]) = x[u];
    }
    __syncthreads();  // cs and the token slots are rewritten for the next group
  }
}

}  // namespace

cudaError_t launch_rope_kv_store(const RopeStoreParams& p, int mode, cudaStream_t stream) {
  // Prompts at offsets: four CTAs of 128 threads per token in flight, 16 CTAs
  // per SM (a grid-stride walk over the padded tokens).
  static int sm_count[64];
  static std::once_flag sm_once[64];
  int dev0 = 0;
  cudaError_t e0 = cudaGetDevice(&dev0);
  if (e0 != cudaSuccess) return e0;
  if (dev0 < 0 || dev0 >= 64) return cudaErrorInvalidDevice;
  std::call_once(sm_once[dev0], [dev0] {
    if (cudaDeviceGetAttribute(&sm_count[dev0], cudaDevAttrMultiProcessorCount, dev0) != cudaSuccess)
      sm_count[dev0] = 0;
  });
  // Prompts at offsets: as many CTAs as are resident at once (the walk over
  // the token groups is a grid-stride loop).
  static int varlen_ctas[64][4];  // per SM, for (D, storage) = (128|64, bf16|f16)
  static std::once_flag varlen_once[64];
  std::call_once(varlen_once[dev0], [dev0] {
    const void* fns[4] = {reinterpret_cast<const void*>(rope_kv_store_varlen_kernel<128, false>),
                          reinterpret_cast<const void*>(rope_kv_store_varlen_kernel<64, false>),
                          reinterpret_cast<const void*>(rope_kv_store_varlen_kernel<128, true>),
                          reinterpret_cast<const void*>(rope_kv_store_varlen_kernel<64, true>)};
    for (int i = 0; i < 4; ++i)
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&varlen_ctas[dev0][i], fns[i], kVarlenThreads,
                                                        (3 * kScanPrompts + 1) * sizeof(int)) != cudaSuccess ||
          varlen_ctas[dev0][i] <= 0)
        varlen_ctas[dev0][i] = 4;
  });
  const int vk = (p.D == 128 ? 0 : 1) + (p.f16 ? 2 : 0);
  const long long varlen_grid =
      std::max(1ll, static_cast<long long>(sm_count[dev0] > 0 ? sm_count[dev0] : 1) * varlen_ctas[dev0][vk]);
  const bool scan = mode == 2 && p.A <= kScanPrompts;  // real tokens only
  const long long varlen_cap = 4ll * (sm_count[dev0] > 0 ? sm_count[dev0] : 1) * kTokenSplit;  // padded walk
  const long long g = mode == 1 ? p.T
                    : mode == 0 ? static_cast<long long>(p.A) * kTokenSplit
                    : scan ? varlen_grid
                           : std::min(varlen_cap, static_cast<long long>(p.A) * p.T * kTokenSplit);
  if (g > 0x7fffffffll) return cudaErrorInvalidValue;
  const unsigned grid = static_cast<unsigned>(g);
  if (grid == 0) return cudaSuccess;
  if ((p.H_kv * (p.D / 8)) % kTokenSplit) return cudaErrorInvalidValue;  // V bytes split in whole units
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(mode == 1 ? 256 : scan ? kVarlenThreads : kTokenThreads);
  // the prompts' scan (prompts at offsets) in dynamic shared memory, so that
  // the decode store keeps its small footprint
  cfg.dynamicSmemBytes = scan ? static_cast<size_t>(3 * p.A + 1) * sizeof(int) : 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // The decode attention kernel that follows (programmatic launch) needs most
  // of an SM's shared memory; with the per-token store CTAs in the
  // shared-memory-heavy split it can start on their SMs while they run.  (The
  // prefill attention kernel cannot share an SM with store CTAs anyway: it
  // takes the whole register file.)
  static std::once_flag carveout_once[64];
  static cudaError_t carveout_err[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(carveout_once[dev], [dev] {
    const void* fns[4] = {reinterpret_cast<const void*>(rope_kv_store_token_kernel<128, false>),
                          reinterpret_cast<const void*>(rope_kv_store_token_kernel<64, false>),
                          reinterpret_cast<const void*>(rope_kv_store_token_kernel<128, true>),
                          reinterpret_cast<const void*>(rope_kv_store_token_kernel<64, true>)};
    carveout_err[dev] = cudaSuccess;
    for (const void* f : fns)
      if (carveout_err[dev] == cudaSuccess)
        carveout_err[dev] = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                 cudaSharedmemCarveoutMaxShared);
  });
  if (carveout_err[dev] != cudaSuccess) return carveout_err[dev];
  const int varlen = mode == 2;
  auto go = [&](auto d, auto f16) {
    constexpr int kD = decltype(d)::value;
    constexpr bool kF16 = decltype(f16)::value;
    if (mode == 1) return cudaLaunchKernelEx(&cfg, rope_kv_store_kernel<kD, kF16>, p);
    if (scan) return cudaLaunchKernelEx(&cfg, rope_kv_store_varlen_kernel<kD, kF16>, p);
    return cudaLaunchKernelEx(&cfg, rope_kv_store_token_kernel<kD, kF16>, p, varlen);
  };
  using T = std::true_type;
  using F = std::false_type;
  if (p.D == 128) return p.f16 ? go(std::integral_constant<int, 128>{}, T{}) : go(std::integral_constant<int, 128>{}, F{});
  if (p.D == 64) return p.f16 ? go(std::integral_constant<int, 64>{}, T{}) : go(std::integral_constant<int, 64>{}, F{});
  return cudaErrorInvalidValue;
}

}  // namespace kvgqa
