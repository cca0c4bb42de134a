// K2: split-K flash-decode over the shared slot KV cache, and K3: the combine.
//
// microLLM-rocm ARCHITECTURE.md, section "Tensor ownership boundary": each
// survivor token attends to its own row's cached prefix, with device
// positions[A] and cache_rows[A].  Section "Attention layout boundary": with
// GQA, one K/V head serves a group of query heads (the zero-stride idea: K/V
// are never expanded).  operator-development.md, "Public interfaces": low
// precision softmax keeps FP32 reductions and rounds only the caller output.
//
// Work split.  Segment (a, g) is the prefix of KV head g in row cache_rows[a]:
// n_a = positions[a] + 1 keys, contiguous in memory ((n_a * D * 2) bytes).  All
// segments, laid end to end, form one key range of K_tot keys; CTA b of the
// persistent grid takes keys [b*W, (b+1)*W) with W = ceil(K_tot / grid), so
// every SM streams the same number of bytes whatever the length mix.  A
// segment that lies inside one CTA is finished there (BF16 out written); a
// segment cut by a CTA boundary leaves FP32 partials (m, l, o) that K3 merges.
// Each CTA writes at most two partials (its first and its last segment).
//
// Inside a CTA: one producer warp streams 64-key K and V tiles (and, at a
// segment start, the G query rows) into a 4-stage shared-memory ring with
// bulk TMA copies completed on mbarriers; eight consumer warps take 8 keys of
// each tile.  In a consumer warp, D/8 lanes share one key: each lane owns a
// 16-byte chunk of D and holds that chunk of all G (padded to GP) query heads in
// registers.  Partial dot products are reduced with a transposing butterfly
// (shuffles) that leaves each lane with the full score of one head, so the
// FP32 online softmax needs no further exchange; probabilities go through a
// small per-warp shared buffer to the P.V accumulation, which uses packed
// FP32x2 FMAs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "kvgqa_internal.h"
#include "ptx.cuh"

namespace kvgqa {
namespace {

constexpr int NCW = 8;                  // consumer warps
constexpr int NT = 64;                  // keys per tile
constexpr int KPW = NT / NCW;           // keys of a tile per consumer warp
constexpr int NS = 4;                   // pipeline stages
constexpr int THREADS = (NCW + 1) * 32; // + one producer warp
constexpr int W_MIN = 256;              // fewest keys a CTA is given
constexpr unsigned FULL = 0xffffffffu;

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// One split-K partial result: o[GP][D], then m[GP], then l[GP] (each of the
// last two padded to at least 2 floats) so that every slot starts on a
// 16-byte boundary for the float4 accesses.
__host__ __device__ constexpr int slot_floats(int GP, int D) { return GP * D + 2 * (GP < 2 ? 2 : GP); }
__host__ __device__ constexpr int slot_l_offset(int GP, int D) { return GP * D + (GP < 2 ? 2 : GP); }
constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int D, int GP>
struct Cfg {
  static constexpr int L = D / 8;           // lanes sharing one key
  static constexpr int KPS = 32 / L;        // keys per warp step
  static constexpr int STEPS = KPW / KPS;   // warp steps per tile
  static constexpr int LOGL = ilog2(L);
  static constexpr int LOGG = ilog2(GP);
  static constexpr int KV_BYTES = NT * D * 2;
  static constexpr int Q_BYTES = GP * D * 2;
  static constexpr int STAGE = 2 * KV_BYTES + Q_BYTES;
  static constexpr int OFF_P = NS * STAGE;                     // [NCW][KPW][GP] f32
  static constexpr int OFF_ALPHA = OFF_P + NCW * KPW * GP * 4;  // [NCW][GP]
  static constexpr int OFF_CM = OFF_ALPHA + NCW * GP * 4;       // [NCW][GP]
  static constexpr int OFF_CL = OFF_CM + NCW * GP * 4;          // [NCW][GP]
  static constexpr int OFF_CO = OFF_CL + NCW * GP * 4;          // [NCW][GP][D]
  static constexpr int OFF_PREFIX = OFF_CO + NCW * GP * D * 4;  // [kMaxActiveRows + 1] int
  static constexpr int OFF_BAR = align_up(OFF_PREFIX + (kMaxActiveRows + 1) * 4, 16);
  static constexpr int OFF_FLAG = OFF_BAR + 2 * NS * 8;
  static constexpr int SMEM = OFF_FLAG + 16;
  static_assert(GP <= L, "group larger than the lanes of one key");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// Per-row key counts and their running sum (times H_kv): prefix[a] is the
// flattened start of row a's first segment.  Invalid metadata -> 0 keys.
__device__ void build_prefix(const DecodeParams& p, int* prefix, bool flag) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    int carry = 0, bad = 0;
    for (int base = 0; base < p.A; base += 32) {
      const int a = base + lane;
      int n = 0;
      if (a < p.A) {
        const int pos = p.positions[a];
        const int row = p.cache_rows[a];
        const bool pos_ok = pos >= 0 && pos < p.max_seq;
        const bool row_ok = row >= 0 && row < p.S;
        if (pos_ok && row_ok) n = (pos + 1) * p.H_kv;
        bad |= (pos_ok ? 0 : KVGQA_FLAG_POSITION_RANGE) | (row_ok ? 0 : KVGQA_FLAG_ROW_RANGE);
      }
      int incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(FULL, incl, off);
        if (lane >= off) incl += t;
      }
      if (a < p.A) prefix[a + 1] = carry + incl;
      carry += __shfl_sync(FULL, incl, 31);
    }
    if (lane == 0) prefix[0] = 0;
    for (int off = 16; off; off >>= 1) bad |= __shfl_xor_sync(FULL, bad, off);
    if (flag && lane == 0 && bad) atomicOr(p.status, bad);
  }
  __syncthreads();
}

__device__ __forceinline__ int keys_per_cta(int k_tot, int num_ctas) {
  const int w = (k_tot + num_ctas - 1) / num_ctas;
  return w < W_MIN ? W_MIN : w;
}

// Walks the tiles of one CTA's key range [x0, x1): segment by segment, NT keys
// at a time.  Producer and consumers run identical copies.
struct Cursor {
  const int* prefix;
  int H_kv, x0, x1;
  int x, a, g, n, seg_lo, seg_in;  // seg_in: where this CTA entered the segment

  __device__ __forceinline__ int row_keys(int r) const { return (prefix[r + 1] - prefix[r]) / H_kv; }

  __device__ void init(const int* pf, int h_kv, int A, int lo, int hi) {
    prefix = pf; H_kv = h_kv; x0 = lo; x1 = hi; x = lo;
    int l = 0, r = A - 1;  // last row with prefix[row] <= x0 and a nonempty range
    while (l < r) {
      const int mid = (l + r + 1) >> 1;
      if (prefix[mid] <= lo) l = mid; else r = mid - 1;
    }
    a = l;
    while (row_keys(a) == 0) ++a;
    n = row_keys(a);
    g = (lo - prefix[a]) / n;
    seg_lo = prefix[a] + g * n;
    seg_in = lo;
  }
  __device__ __forceinline__ bool more() const { return x < x1; }
  __device__ __forceinline__ int seg_end() const { return min(seg_lo + n, x1); }
  __device__ __forceinline__ int k0() const { return x - seg_lo; }
  __device__ __forceinline__ int nt() const { return min(NT, seg_end() - x); }
  __device__ __forceinline__ bool first() const { return x == seg_in; }
  __device__ __forceinline__ bool last() const { return x + nt() == seg_end(); }
  __device__ __forceinline__ bool whole() const { return seg_lo >= x0 && seg_lo + n <= x1; }
  __device__ __forceinline__ int slot() const { return seg_in == x0 ? 0 : 1; }
  __device__ void advance() {
    const bool was_last = last();
    x += nt();
    if (was_last && x < x1) {
      if (++g == H_kv) {
        g = 0;
        do { ++a; } while (row_keys(a) == 0);
        n = row_keys(a);
      }
      seg_lo = prefix[a] + g * n;
      seg_in = x;
    }
  }
};

template <int D, int GP>
__global__ void __launch_bounds__(THREADS, 1)
flash_decode_splitk_kernel(const __grid_constant__ DecodeParams p) {
  using C = Cfg<D, GP>;
  extern __shared__ __align__(128) unsigned char smem[];
  int* prefix = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + NS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  build_prefix(p, prefix, blockIdx.x == 0);  // ends with __syncthreads

  const int k_tot = prefix[p.A];
  const int W = keys_per_cta(k_tot, p.num_ctas);
  const int x0 = blockIdx.x * W;
  if (x0 >= k_tot) return;
  const int x1 = min(x0 + W, k_tot);

  Cursor cur;
  cur.init(prefix, p.H_kv, p.A, x0, x1);

  if (warp == NCW) {
    // ---------------------------------------------------------- producer
    if (lane != 0) return;
    const uint64_t pol_kv = l2_evict_first_policy();
    const uint64_t pol_q = l2_evict_last_policy();
    int it = 0;
    bool ok = true;
    for (; cur.more(); cur.advance(), ++it) {
      const int s = it % NS;
      if (it >= NS && !mbar_wait_bounded(&empty[s], ((it / NS) - 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      const int nt = cur.nt();
      const bool first = cur.first();
      const uint32_t kv_bytes = static_cast<uint32_t>(nt) * D * 2;
      const uint32_t q_bytes = first ? static_cast<uint32_t>(p.G) * D * 2 : 0u;
      unsigned char* st = smem + s * C::STAGE;
      const int row = p.cache_rows[cur.a];
      const size_t cell = (static_cast<size_t>(row) * p.H_kv + cur.g) * p.max_seq + cur.k0();
      mbar_arrive_expect_tx(&full[s], 2 * kv_bytes + q_bytes);
      bulk_g2s(st, p.k_cache + cell * D, kv_bytes, &full[s], pol_kv);
      bulk_g2s(st + C::KV_BYTES, p.v_cache + cell * D, kv_bytes, &full[s], pol_kv);
      if (first)
        bulk_g2s(st + 2 * C::KV_BYTES,
                 p.q + (static_cast<size_t>(cur.a) * p.H_q + static_cast<size_t>(cur.g) * p.G) * D,
                 q_bytes, &full[s], pol_q);
    }
    if (!ok) {
      // Drain: wait (bounded) for copies this warp may still have in flight.
      for (int t = it - NS < 0 ? 0 : it - NS; t < it; ++t) {
        volatile int no_abort = 0;
        mbar_wait_bounded(&full[t % NS], (t / NS) & 1, &no_abort, nullptr);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  constexpr int L = C::L, KPS = C::KPS, STEPS = C::STEPS, LOGL = C::LOGL, LOGG = C::LOGG;
  const int j = lane & (L - 1);                 // 16-byte chunk of D owned by this lane
  const int ks = lane >> LOGL;                  // key slot inside a warp step
  const int hsel = j >> (LOGL - LOGG);          // head whose score this lane ends with
  const bool head_rep = (j & ((L / GP) - 1)) == 0;  // one lane per (key slot, head)
  float* Pw = reinterpret_cast<float*>(smem + C::OFF_P) + warp * KPW * GP;
  float* alpha_w = reinterpret_cast<float*>(smem + C::OFF_ALPHA) + warp * GP;
  float* CM = reinterpret_cast<float*>(smem + C::OFF_CM);
  float* CL = reinterpret_cast<float*>(smem + C::OFF_CL);
  float* CO = reinterpret_cast<float*>(smem + C::OFF_CO);
  const uint32_t smem_base = smem_u32(smem);

  float2 qf[GP][4];
  float2 o[GP][4];
  float m_run = -INFINITY, l_run = 0.f;
#pragma unroll
  for (int i = 0; i < GP; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[i][c] = make_float2(0.f, 0.f);

  int it = 0;
  for (; cur.more(); cur.advance(), ++it) {
    const int s = it % NS;
    if (!mbar_wait_bounded(&full[s], (it / NS) & 1, abort_flag, p.status)) break;
    const uint32_t st = smem_base + s * C::STAGE;
    if (cur.first()) {
#pragma unroll
      for (int i = 0; i < GP; ++i) {
        const int h = i ^ hsel;  // heads permuted so the butterfly needs no selects
        if (h < p.G) {
          const uint4 w = lds128(st + 2 * C::KV_BYTES + h * D * 2 + j * 16);
          qf[i][0] = bf16x2_to_f2(w.x); qf[i][1] = bf16x2_to_f2(w.y);
          qf[i][2] = bf16x2_to_f2(w.z); qf[i][3] = bf16x2_to_f2(w.w);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) qf[i][c] = make_float2(0.f, 0.f);
        }
      }
    }
    const int nv = min(max(cur.nt() - warp * KPW, 0), KPW);  // valid keys of this warp
    if (nv > 0) {
      const uint32_t kbase = st + (warp * KPW) * D * 2 + j * 16;
      const uint32_t vbase = kbase + C::KV_BYTES;
      float sc[STEPS];
#pragma unroll
      for (int t = 0; t < STEPS; ++t) {
        const int key = t * KPS + ks;
        const uint4 w = lds128(kbase + key * D * 2);
        const float2 k0 = bf16x2_to_f2(w.x), k1 = bf16x2_to_f2(w.y);
        const float2 k2 = bf16x2_to_f2(w.z), k3 = bf16x2_to_f2(w.w);
        float part[GP];
#pragma unroll
        for (int i = 0; i < GP; ++i) {
          float2 acc = fmul2(qf[i][0], k0);
          acc = ffma2(qf[i][1], k1, acc);
          acc = ffma2(qf[i][2], k2, acc);
          acc = ffma2(qf[i][3], k3, acc);
          part[i] = acc.x + acc.y;
        }
        // Transposing butterfly: at level lv, exchange the upper half of the
        // live heads with the partner lane lane ^ 2^(LOGL-1-lv).
#pragma unroll
        for (int lv = 0; lv < LOGG; ++lv) {
          const int half = GP >> (lv + 1);
#pragma unroll
          for (int i = 0; i < half; ++i)
            part[i] += __shfl_xor_sync(FULL, part[i + half], 1 << (LOGL - 1 - lv));
        }
#pragma unroll
        for (int lv = LOGG; lv < LOGL; ++lv)
          part[0] += __shfl_xor_sync(FULL, part[0], 1 << (LOGL - 1 - lv));
        sc[t] = key < nv ? part[0] * p.scale_log2 : -INFINITY;
      }
      // Online softmax (base 2; scores already carry the log2(e) factor).
      float mb = sc[0];
#pragma unroll
      for (int t = 1; t < STEPS; ++t) mb = fmaxf(mb, sc[t]);
#pragma unroll
      for (int off = L; off < 32; off <<= 1) mb = fmaxf(mb, __shfl_xor_sync(FULL, mb, off));
      const float m_new = fmaxf(m_run, mb);
      const float alpha = exp2f(m_run - m_new);
      float psum = 0.f;
#pragma unroll
      for (int t = 0; t < STEPS; ++t) {
        const float pt = exp2f(sc[t] - m_new);
        psum += pt;
        if (head_rep) Pw[(t * KPS + ks) * GP + hsel] = pt;
      }
      l_run = l_run * alpha + psum;
      m_run = m_new;
      if (head_rep && ks == 0) alpha_w[hsel] = alpha;
      __syncwarp();
      if (__any_sync(FULL, alpha != 1.f)) {
#pragma unroll
        for (int i = 0; i < GP; ++i) {
          const float al = alpha_w[i];
#pragma unroll
          for (int c = 0; c < 4; ++c) o[i][c] = fmul2(o[i][c], make_float2(al, al));
        }
      }
#pragma unroll
      for (int t = 0; t < STEPS; ++t) {
        const int key = t * KPS + ks;
        if (key < nv) {
          const uint4 w = lds128(vbase + key * D * 2);
          const float2 v0 = bf16x2_to_f2(w.x), v1 = bf16x2_to_f2(w.y);
          const float2 v2 = bf16x2_to_f2(w.z), v3 = bf16x2_to_f2(w.w);
          float pv[GP];
          const uint32_t pa = smem_u32(Pw + key * GP);
          if constexpr (GP >= 4) {
#pragma unroll
            for (int i = 0; i < GP; i += 4) {
              const float4 q4 = lds128f(pa + i * 4);
              pv[i] = q4.x; pv[i + 1] = q4.y; pv[i + 2] = q4.z; pv[i + 3] = q4.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < GP; ++i) pv[i] = Pw[key * GP + i];
          }
#pragma unroll
          for (int i = 0; i < GP; ++i) {
            const float2 pp = make_float2(pv[i], pv[i]);
            o[i][0] = ffma2(pp, v0, o[i][0]);
            o[i][1] = ffma2(pp, v1, o[i][1]);
            o[i][2] = ffma2(pp, v2, o[i][2]);
            o[i][3] = ffma2(pp, v3, o[i][3]);
          }
        }
      }
      __syncwarp();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    if (cur.last()) {
      // ---------------------------------------------------- segment end
#pragma unroll
      for (int off = L; off < 32; off <<= 1) {
        l_run += __shfl_xor_sync(FULL, l_run, off);
#pragma unroll
        for (int i = 0; i < GP; ++i)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            o[i][c].x += __shfl_xor_sync(FULL, o[i][c].x, off);
            o[i][c].y += __shfl_xor_sync(FULL, o[i][c].y, off);
          }
      }
      if (ks == 0) {
#pragma unroll
        for (int i = 0; i < GP; ++i) {
          float4* dst = reinterpret_cast<float4*>(CO + (warp * GP + i) * D + j * 8);
          dst[0] = make_float4(o[i][0].x, o[i][0].y, o[i][1].x, o[i][1].y);
          dst[1] = make_float4(o[i][2].x, o[i][2].y, o[i][3].x, o[i][3].y);
        }
        if (head_rep) {
          CM[warp * GP + hsel] = m_run;
          CL[warp * GP + hsel] = l_run;
        }
      }
      named_bar_sync(1, NCW * 32);
      const bool whole = cur.whole();
      float* slotp = p.partials + static_cast<size_t>(blockIdx.x * 2 + cur.slot()) * slot_floats(GP, D);
      for (int item = threadIdx.x; item < p.G * (D / 8); item += NCW * 32) {
        const int h = item / (D / 8), c8 = item - h * (D / 8);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, CM[w * GP + h]);
        float lsum = 0.f, acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
          const float mw = CM[w * GP + h];
          const float sc = mw == -INFINITY ? 0.f : exp2f(mw - M);
          lsum += CL[w * GP + h] * sc;
          const float4* src = reinterpret_cast<const float4*>(CO + (w * GP + h) * D + c8 * 8);
          const float4 u0 = src[0], u1 = src[1];
          acc[0] += u0.x * sc; acc[1] += u0.y * sc; acc[2] += u0.z * sc; acc[3] += u0.w * sc;
          acc[4] += u1.x * sc; acc[5] += u1.y * sc; acc[6] += u1.z * sc; acc[7] += u1.w * sc;
        }
        if (whole) {
          const float inv = 1.f / lsum;
          uint4 pk;
          __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
          __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
          __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[4] * inv, acc[5] * inv);
          __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[6] * inv, acc[7] * inv);
          pk.x = *reinterpret_cast<uint32_t*>(&b0); pk.y = *reinterpret_cast<uint32_t*>(&b1);
          pk.z = *reinterpret_cast<uint32_t*>(&b2); pk.w = *reinterpret_cast<uint32_t*>(&b3);
          uint16_t* dst = p.out + (static_cast<size_t>(cur.a) * p.H_q + cur.g * p.G + h) * D + c8 * 8;
          *reinterpret_cast<uint4*>(dst) = pk;
        } else {
          float4* dst = reinterpret_cast<float4*>(slotp + h * D + c8 * 8);
          dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
          dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
          if (c8 == 0) {
            slotp[GP * D + h] = M;
            slotp[slot_l_offset(GP, D) + h] = lsum;
          }
        }
      }
      named_bar_sync(1, NCW * 32);
      m_run = -INFINITY;
      l_run = 0.f;
#pragma unroll
      for (int i = 0; i < GP; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[i][c] = make_float2(0.f, 0.f);
    }
  }
}

// K3: for every segment cut by a CTA boundary, merge the partials of the CTAs
// b0..b1 that cover it and write the BF16 output of its G query heads.
template <int D, int GP>
__global__ void __launch_bounds__(128) decode_combine_kernel(const __grid_constant__ DecodeParams p) {
  __shared__ int prefix[kMaxActiveRows + 1];
  build_prefix(p, prefix, false);
  const int a = blockIdx.x / p.H_kv, g = blockIdx.x - a * p.H_kv;
  const int n = (prefix[a + 1] - prefix[a]) / p.H_kv;
  if (n == 0) return;
  const int W = keys_per_cta(prefix[p.A], p.num_ctas);
  const int seg_lo = prefix[a] + g * n;
  const int b0 = seg_lo / W, b1 = (seg_lo + n - 1) / W;
  if (b0 == b1) return;  // finished by the split-K kernel
  const int slot0 = (b0 * W == seg_lo) ? 0 : 1;
  constexpr size_t SLOT = slot_floats(GP, D);
  for (int item = threadIdx.x; item < p.G * (D / 8); item += blockDim.x) {
    const int h = item / (D / 8), c8 = item - h * (D / 8);
    float M = -INFINITY;
    for (int b = b0; b <= b1; ++b) {
      const float* sp = p.partials + (static_cast<size_t>(b) * 2 + (b == b0 ? slot0 : 0)) * SLOT;
      M = fmaxf(M, sp[GP * D + h]);
    }
    float lsum = 0.f, acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int b = b0; b <= b1; ++b) {
      const float* sp = p.partials + (static_cast<size_t>(b) * 2 + (b == b0 ? slot0 : 0)) * SLOT;
      const float sc = exp2f(sp[GP * D + h] - M);
      lsum += sp[slot_l_offset(GP, D) + h] * sc;
      const float4 u0 = *reinterpret_cast<const float4*>(sp + h * D + c8 * 8);
      const float4 u1 = *reinterpret_cast<const float4*>(sp + h * D + c8 * 8 + 4);
      acc[0] += u0.x * sc; acc[1] += u0.y * sc; acc[2] += u0.z * sc; acc[3] += u0.w * sc;
      acc[4] += u1.x * sc; acc[5] += u1.y * sc; acc[6] += u1.z * sc; acc[7] += u1.w * sc;
    }
    const float inv = 1.f / lsum;
    uint4 pk;
    __nv_bfloat162 q0 = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
    __nv_bfloat162 q1 = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
    __nv_bfloat162 q2 = __floats2bfloat162_rn(acc[4] * inv, acc[5] * inv);
    __nv_bfloat162 q3 = __floats2bfloat162_rn(acc[6] * inv, acc[7] * inv);
    pk.x = *reinterpret_cast<uint32_t*>(&q0); pk.y = *reinterpret_cast<uint32_t*>(&q1);
    pk.z = *reinterpret_cast<uint32_t*>(&q2); pk.w = *reinterpret_cast<uint32_t*>(&q3);
    *reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(a) * p.H_q + g * p.G + h) * D + c8 * 8) = pk;
  }
}

template <int D, int GP>
struct Kernels {
  static void* splitk() { return reinterpret_cast<void*>(&flash_decode_splitk_kernel<D, GP>); }
  static cudaError_t prepare(int device, int* num_ctas) {
    // Opt in to the large dynamic shared memory once per device.
    static std::once_flag flags[64];
    static cudaError_t errs[64];
    static int ctas[64];
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::call_once(flags[device], [&]() {
      errs[device] = cudaFuncSetAttribute(flash_decode_splitk_kernel<D, GP>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, GP>::SMEM);
      int sms = 0, per_sm = 0;
      if (errs[device] == cudaSuccess)
        errs[device] = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
      if (errs[device] == cudaSuccess)
        errs[device] = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, flash_decode_splitk_kernel<D, GP>, THREADS, Cfg<D, GP>::SMEM);
      ctas[device] = sms * (per_sm > 0 ? per_sm : 1);
    });
    *num_ctas = ctas[device];
    return errs[device];
  }
  static cudaError_t launch(const DecodeParams& p, cudaStream_t stream) {
    flash_decode_splitk_kernel<D, GP><<<p.num_ctas, THREADS, Cfg<D, GP>::SMEM, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_combine_kernel<D, GP><<<p.A * p.H_kv, 128, 0, stream>>>(p);
    return cudaGetLastError();
  }
};

template <typename F>
cudaError_t dispatch(int D, int GP, F&& f) {
  if (D == 128) {
    switch (GP) {
      case 1: return f(Kernels<128, 1>{});
      case 2: return f(Kernels<128, 2>{});
      case 4: return f(Kernels<128, 4>{});
      case 8: return f(Kernels<128, 8>{});
    }
  } else if (D == 64) {
    switch (GP) {
      case 1: return f(Kernels<64, 1>{});
      case 2: return f(Kernels<64, 2>{});
      case 4: return f(Kernels<64, 4>{});
      case 8: return f(Kernels<64, 8>{});
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int decode_group_pad(int G) {
  int gp = 1;
  while (gp < G) gp <<= 1;
  return gp;
}

cudaError_t decode_launch_shape(int device, int D, int GP, int* num_ctas, size_t* partial_bytes) {
  int n = 0;
  const cudaError_t e = dispatch(D, GP, [&](auto k) { return decltype(k)::prepare(device, &n); });
  if (e != cudaSuccess) return e;
  *num_ctas = n;
  *partial_bytes = static_cast<size_t>(n) * 2 * slot_floats(GP, D) * sizeof(float);
  return cudaSuccess;
}

// Scratch for callers that cannot allocate device memory themselves: the
// split-K partials (and the status word in front of them) live in this
// file-scope device array instead of a caller workspace.  Every GPU that
// loads the library holds it until the process exits; all calls share it.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

cudaError_t static_scratch_address(int device, void** ptr) {
  static std::once_flag flags[64];
  static void* addr[64];
  static cudaError_t errs[64];
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  // Runs once per device, with that device current (the caller's current device).
  std::call_once(flags[device], [&] { errs[device] = cudaGetSymbolAddress(&addr[device], g_static_scratch); });
  *ptr = addr[device];
  return errs[device];
}

cudaError_t launch_cached_gqa_attention(const DecodeParams& p, cudaStream_t stream) {
  if (p.A == 0) return cudaSuccess;
  const int GP = decode_group_pad(p.G);
  return dispatch(p.D, GP, [&](auto k) { return decltype(k)::launch(p, stream); });
}

}  // namespace kvgqa
