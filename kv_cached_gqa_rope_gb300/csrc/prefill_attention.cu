// K4: causal GQA attention of the equal-length prefill, on tcgen05 tensor
// cores with the accumulators in tensor memory.
//
// microLLM-rocm ARCHITECTURE.md, section "Tensor ownership boundary": equal-
// length pending prompts run as one batch and each prefix is mapped into its
// target empty shared-cache row; section "Attention layout boundary": Q/K/V
// leave the projection token-major (BTHD) and context is written back
// token-major; with GQA one K/V head serves G query heads without expansion.
// The rotated K and V have already been stored into the target cache rows
// (K1), so this kernel reads them straight from the cache.
//
// A persistent grid (one CTA per SM) walks (128-query tile, prompt a, query
// head h) items, longest first, dealt round-robin; per item:
//   warp 4      TMA producer: the Q tile once, then 128-key K and V tiles of
//               the row's cached prefix into a 2-stage ring (128B swizzle);
//   warp 5      one thread issues tcgen05.mma: S = Q K^T into one of two TMEM
//               buffers (the next tile's S overlaps this tile's softmax), and
//               O += P V into a TMEM accumulator;
//   warps 0-3   softmax, one thread per query row: S row from TMEM, scale,
//               causal mask on the diagonal tile, FP32 online softmax, P as
//               BF16 into shared memory (the A operand of P V), O rescaled in
//               TMEM only when the row maximum grew by more than 2^8 (the
//               exponent base is otherwise kept, which leaves O / l exact);
//               at the end O / l is rounded to BF16 and stored token-major.
// Key tiles past the diagonal are never visited.  Tensor maps bound the key
// and query ranges by T, so tile rows past the prompt read as zeros.
// Tiles are scheduled longest first (the last query tiles have the most keys).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "kvgqa_internal.h"
#include "tcgen05.cuh"

namespace kvgqa {
namespace {

constexpr int BM = 128;        // query rows per tile
constexpr int BN = 128;        // keys per tile
constexpr int SUB = 16384;     // one [128 rows x 64 bf16] swizzled sub-tile
constexpr int THREADS = 224;   // 4 softmax warps + Q/K producer + MMA + V producer
constexpr int TMEM_COLS = 512; // S x2 (128 cols each), O (128), P x2 (64 each)
constexpr int P_COL = 3 * BN;  // P buffers: BF16 pairs packed in 32-bit columns
constexpr unsigned FULLMASK = 0xffffffffu;

template <int D>
struct PCfg {
  static constexpr int NSUB = D / 64;               // 64-wide sub-tiles per row
  static constexpr int NK = D == 128 ? 3 : 4;       // K stages
  static constexpr int NV = NK;                     // V stages
  static constexpr int TILE = NSUB * SUB;           // one K or V tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = TILE;
  static constexpr int V_OFF = K_OFF + NK * TILE;
  static constexpr int BAR_OFF = V_OFF + NV * TILE;
  // q_full, q_empty, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], s_full[2], p_full[2], o_done[2], drain
  static constexpr int NBAR = 2 + 2 * NK + 2 * NV + 7;
  static constexpr int SLOT_OFF = BAR_OFF + NBAR * 8;
  static constexpr int FLAG_OFF = SLOT_OFF + 8;
  static constexpr int SMEM = FLAG_OFF + 16 + 1024;  // + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct PrefillMaps {
  CUtensorMap q;  // [A][T][H_q][D] rotated queries
  CUtensorMap k;  // cache [S*H_kv][T(bounded)][D]
  CUtensorMap v;
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 2^x on the special-function unit (flushes results below 2^-126 to zero,
// which no BF16 probability needs).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The work of the persistent grid: items (query tile qt, prompt a, head h),
// longest first (tile qt visits qt + 1 key tiles), dealt round-robin to the
// CTAs; every role of a CTA walks the same sequence, tile by tile.
struct TileWalk {
  int i, stride, n_items, nqt, heads, H_q, H_kv, G, S;
  const int32_t* rows;
  int qt, a, h, kv_row;  // current item
  int j;                 // key tile within the item
  bool ok;               // false past the last item

  __device__ bool load_item() {
    while (i < n_items) {
      qt = nqt - 1 - i / heads;
      const int rem = i % heads;
      a = rem / H_q;
      h = rem % H_q;
      const int r = rows[a];
      if (r >= 0 && r < S) {
        kv_row = r * H_kv + h / G;
        j = 0;
        return true;
      }
      i += stride;  // prompts with an invalid row are skipped (and flagged by the producer)
    }
    return false;
  }
  __device__ void init(const PrefillParams& p, int first, int step) {
    nqt = (p.T + BM - 1) / BM;
    heads = p.A * p.H_q;
    n_items = nqt * heads;
    H_q = p.H_q; H_kv = p.H_kv; G = p.G; S = p.S; rows = p.cache_rows;
    i = first;
    stride = step;
    ok = load_item();
  }
  __device__ __forceinline__ bool first_tile() const { return j == 0; }
  __device__ __forceinline__ bool last_tile() const { return j == qt; }
  __device__ void advance() {
    if (j < qt) { ++j; return; }
    i += stride;
    ok = load_item();
  }
};

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
prefill_attention_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v) {
  using C = PCfg<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = k_full + C::NK;
  uint64_t* v_full = k_empty + C::NK;
  uint64_t* v_empty = v_full + C::NV;
  uint64_t* s_full = v_empty + C::NV;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SLOT_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::FLAG_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  TileWalk walk;
  walk.init(p, blockIdx.x, gridDim.x);
  if (!walk.ok) {  // uniform: this CTA has no valid item
    if (threadIdx.x == 0) {
      for (int i = blockIdx.x; i < walk.n_items; i += gridDim.x) {
        const int r = p.cache_rows[(i % walk.heads) / p.H_q];
        if (r < 0 || r >= p.S) { atomicOr(p.status, KVGQA_FLAG_ROW_RANGE); break; }
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], BM);
      mbar_init(&o_done[b], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(smem);

  if (warp == 4) {
    // ------------------------------------------------------------ Q and K producer
    if (lane == 0) {
      const uint64_t pol_q = l2_evict_first_policy();
      const uint64_t pol_kv = l2_evict_last_policy();  // K/V tiles are re-read by the group's heads
      // prompts whose cache row is invalid are skipped by every role; flag them here
      for (int i = blockIdx.x; i < walk.n_items; i += gridDim.x) {
        const int r = p.cache_rows[(i % walk.heads) / p.H_q];
        if (r < 0 || r >= p.S) { atomicOr(p.status, KVGQA_FLAG_ROW_RANGE); break; }
      }
      int it = 0, qi = 0;
      for (; walk.ok; walk.advance()) {
        if (walk.first_tile()) {
          if (qi >= 1 && !mbar_wait_bounded(q_empty, (qi - 1) & 1, abort_flag, p.status)) break;
          mbar_arrive_expect_tx(q_full, BM * D * 2);
          for (int sub = 0; sub < C::NSUB; ++sub)
            tma_load_4d(smem + C::Q_OFF + sub * SUB, &map_q, sub * 64, walk.h, walk.qt * BM, walk.a, q_full, pol_q);
          ++qi;
        }
        const int s = it % C::NK;
        if (it >= C::NK && !mbar_wait_bounded(&k_empty[s], ((it / C::NK) - 1) & 1, abort_flag, p.status)) break;
        unsigned char* st = smem + C::K_OFF + s * C::TILE;
        mbar_arrive_expect_tx(&k_full[s], BN * D * 2);
        for (int sub = 0; sub < C::NSUB; ++sub)
          tma_load_3d(st + sub * SUB, &map_k, sub * 64, walk.j * BN, walk.kv_row, &k_full[s], pol_kv);
        ++it;
      }
      if (*abort_flag) {
        volatile int none = 0;
        if (qi >= 1) mbar_wait_bounded(q_full, (qi - 1) & 1, &none, nullptr);
        for (int t = it - C::NK < 0 ? 0 : it - C::NK; t < it; ++t)
          mbar_wait_bounded(&k_full[t % C::NK], (t / C::NK) & 1, &none, nullptr);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ V producer
    if (lane == 0) {
      const uint64_t pol_kv = l2_evict_last_policy();
      int it = 0;
      for (; walk.ok; walk.advance()) {
        const int s = it % C::NV;
        if (it >= C::NV && !mbar_wait_bounded(&v_empty[s], ((it / C::NV) - 1) & 1, abort_flag, p.status)) break;
        unsigned char* st = smem + C::V_OFF + s * C::TILE;
        mbar_arrive_expect_tx(&v_full[s], BN * D * 2);
        for (int sub = 0; sub < C::NSUB; ++sub)
          tma_load_3d(st + sub * SUB, &map_v, sub * 64, walk.j * BN, walk.kv_row, &v_full[s], pol_kv);
        ++it;
      }
      if (*abort_flag) {
        volatile int none = 0;
        for (int t = it - C::NV < 0 ? 0 : it - C::NV; t < it; ++t)
          mbar_wait_bounded(&v_full[t % C::NV], (t / C::NV) & 1, &none, nullptr);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, 1);
      const uint32_t q_addr = sbase + C::Q_OFF;
      bool issued = false;
      int qi_next = 0;  // Q loads consumed so far by the look-ahead walk
      TileWalk ahead = walk;
      // S = Q K^T of look-ahead tile t; K stage and (after an item's last tile) Q are freed on completion
      auto issue_qk = [&](int t) -> bool {
        if (ahead.first_tile()) {
          if (!mbar_wait_bounded(q_full, qi_next & 1, abort_flag, p.status)) return false;
          ++qi_next;
        }
        if (!mbar_wait_bounded(&k_full[t % C::NK], (t / C::NK) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t k_addr = sbase + C::K_OFF + (t % C::NK) * C::TILE;
        const uint32_t d_tmem = tmem + (t & 1) * BN;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks / 4) * SUB + (ks % 4) * 32;
          umma_f16_ss(d_tmem, smem_desc_sw128(q_addr + off, 16, 1024), smem_desc_sw128(k_addr + off, 16, 1024),
                      IDESC_QK, ks > 0);
        }
        umma_commit(&s_full[t & 1]);
        umma_commit(&k_empty[t % C::NK]);
        if (ahead.last_tile()) umma_commit(q_empty);
        issued = true;
        ahead.advance();
        return true;
      };
      bool ok = issue_qk(0);
      for (int t = 0; ok && walk.ok; ++t, walk.advance()) {
        if (ahead.ok && !issue_qk(t + 1)) break;
        if (!mbar_wait_bounded(&p_full[t & 1], (t >> 1) & 1, abort_flag, p.status)) break;
        if (!mbar_wait_bounded(&v_full[t % C::NV], (t / C::NV) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t v_addr = sbase + C::V_OFF + (t % C::NV) * C::TILE;
        const uint32_t p_tmem = tmem + P_COL + (t & 1) * (BN / 2);
        const uint32_t acc0 = walk.first_tile() ? 0u : 1u;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          umma_f16_ts(tmem + 2 * BN, p_tmem + ks * 8, smem_desc_sw128(v_addr + ks * 2048, SUB, 1024), IDESC_PV,
                      ks > 0 ? 1u : acc0);
        umma_commit(&o_done[t & 1]);
        umma_commit(&v_empty[t % C::NV]);
      }
      if (*abort_flag && issued) {
        // let every MMA issued so far finish before TMEM is released
        umma_commit(drain);
        volatile int none = 0;
        mbar_wait_bounded(drain, 0, &none, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-3)
    const int r = threadIdx.x;  // query row in the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float c = p.scale_log2;
    const float ce = c > 0.f ? c : 1.f;
    float m_ref = -INFINITY, l = 0.f;
    for (int t = 0; walk.ok; ++t, walk.advance()) {
      const bool first = walk.first_tile(), diag = walk.last_tile();
      if (!__all_sync(FULLMASK, mbar_wait_bounded(&s_full[t & 1], (t >> 1) & 1, abort_flag, p.status))) break;
      tc_fence_after();
      // the four 32-column loads are issued back to back, then waited for once
      uint32_t u0[32], u1[32], u2[32], u3[32];
      tmem_ld32(tmem + lane_base + (t & 1) * BN + 0, u0);
      tmem_ld32(tmem + lane_base + (t & 1) * BN + 32, u1);
      tmem_ld32(tmem + lane_base + (t & 1) * BN + 64, u2);
      tmem_ld32(tmem + lane_base + (t & 1) * BN + 96, u3);
      tmem_wait_ld();
      float sv[BN];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        sv[i] = __uint_as_float(u0[i]);
        sv[32 + i] = __uint_as_float(u1[i]);
        sv[64 + i] = __uint_as_float(u2[i]);
        sv[96 + i] = __uint_as_float(u3[i]);
      }
      // Scores enter the softmax as s * ce with ce > 0 (a non-positive scale is
      // folded into the scores first, a path no usual caller takes).  On the
      // diagonal tile, keys after the query become -inf, so they weigh zero.
      if (c <= 0.f) {
#pragma unroll
        for (int i = 0; i < BN; ++i) sv[i] *= c;
      }
      if (diag) {
#pragma unroll
        for (int i = 0; i < BN; ++i) sv[i] = i <= r ? sv[i] : -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = sv[k];
#pragma unroll
      for (int i = 8; i < BN; ++i) mx[i & 7] = fmaxf(mx[i & 7], sv[i]);
      const float mraw = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float mt = mraw * ce;                    // tile maximum of the scaled scores
      const bool grow = first || mt > m_ref + 8.f;   // keep the old base unless it grew by 2^8
      float alpha = 1.f;
      if (grow) {
        alpha = first ? 0.f : ex2(m_ref - mt);
        m_ref = mt;
        l *= alpha;
      }
      // P buffer t&1 in TMEM was last read by the P.V of tile t-2; an O rescale
      // needs the P.V of tile t-1 complete.
      if (t >= 2 && !__all_sync(FULLMASK, mbar_wait_bounded(&o_done[t & 1], ((t - 2) >> 1) & 1, abort_flag, p.status)))
        break;
      const bool rescale = __any_sync(FULLMASK, grow && !first);
      if (rescale && !__all_sync(FULLMASK, mbar_wait_bounded(&o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, abort_flag,
                                                          p.status)))
        break;
      tc_fence_after();
      if (rescale) {
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t u[32];
          tmem_ld32(tmem + lane_base + 2 * BN + q * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
          tmem_st32(tmem + lane_base + 2 * BN + q * 32, u);
        }
        tmem_wait_st();
      }
      // P as BF16 pairs into TMEM buffer t&1 (the A operand of P.V): row r, key
      // pair j in 32-bit column j.
      float2 ls = make_float2(0.f, 0.f);
      const float2 c2 = make_float2(ce, ce), nm2 = make_float2(-m_ref, -m_ref);
      const uint32_t p_tmem = tmem + lane_base + P_COL + (t & 1) * (BN / 2);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int i0 = half * 64 + 2 * e;
          const float2 x = ffma2(make_float2(sv[i0], sv[i0 + 1]), c2, nm2);
          const float2 pr = make_float2(ex2(x.x), ex2(x.y));
          ls = fadd2(ls, pr);
          w[e] = pack2(pr.x, pr.y);
        }
        tmem_st32(p_tmem + half * 32, w);
      }
      tmem_wait_st();
      l += ls.x + ls.y;
      tc_fence_before();
      mbar_arrive(&p_full[t & 1]);

      if (diag) {
        // ---------------------------------------------------- item epilogue
        if (!__all_sync(FULLMASK, mbar_wait_bounded(&o_done[t & 1], (t >> 1) & 1, abort_flag, p.status))) break;
        tc_fence_after();
        const int tq = walk.qt * BM + r;
        const float inv = 1.f / l;
        uint16_t* dst = p.out + ((static_cast<size_t>(walk.a) * p.T + tq) * p.H_q + walk.h) * D;
        uint32_t u[D];
#pragma unroll
        for (int q = 0; q < D / 32; ++q) tmem_ld32(tmem + lane_base + 2 * BN + q * 32, *reinterpret_cast<uint32_t(*)[32]>(u + q * 32));
        tmem_wait_ld();
        if (tq < p.T) {
#pragma unroll
          for (int q8 = 0; q8 < D / 8; ++q8) {
            uint4 o;
            o.x = pack2(__uint_as_float(u[q8 * 8 + 0]) * inv, __uint_as_float(u[q8 * 8 + 1]) * inv);
            o.y = pack2(__uint_as_float(u[q8 * 8 + 2]) * inv, __uint_as_float(u[q8 * 8 + 3]) * inv);
            o.z = pack2(__uint_as_float(u[q8 * 8 + 4]) * inv, __uint_as_float(u[q8 * 8 + 5]) * inv);
            o.w = pack2(__uint_as_float(u[q8 * 8 + 6]) * inv, __uint_as_float(u[q8 * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + q8 * 8) = o;
          }
        }
      }
    }
  }

  __syncwarp();  // the role warps reconverge (their lane 0 worked alone)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, TMEM_COLS);
}

cudaError_t make_maps(const PrefillParams& p, PrefillMaps* m) {
  auto enc = tma_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t D = p.D;
  {
    cuuint64_t dims[4] = {D, static_cast<cuuint64_t>(p.H_q), static_cast<cuuint64_t>(p.T),
                          static_cast<cuuint64_t>(p.A)};
    cuuint64_t strides[3] = {D * 2, D * 2 * p.H_q, D * 2 * p.H_q * p.T};
    cuuint32_t box[4] = {64, 1, BM, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&m->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(p.q_rot), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // Keys: positions [0, T) of each (slot, kv head); positions >= T are
  // outside the map and read as zeros.
  cuuint64_t dims[3] = {D, static_cast<cuuint64_t>(p.T), static_cast<cuuint64_t>(p.S) * p.H_kv};
  cuuint64_t strides[2] = {D * 2, D * 2 * static_cast<cuuint64_t>(p.max_seq)};
  cuuint32_t box[3] = {64, BN, 1};
  cuuint32_t es[3] = {1, 1, 1};
  if (enc(&m->k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(p.k_cache), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (enc(&m->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(p.v_cache), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

template <int D>
cudaError_t launch_d(const PrefillParams& p, const PrefillMaps& m, cudaStream_t stream) {
  static std::once_flag flags[64];
  static cudaError_t errs[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(flags[dev], [&] {
    errs[dev] = cudaFuncSetAttribute(prefill_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     PCfg<D>::SMEM);
  });
  if (errs[dev] != cudaSuccess) return errs[dev];
  static int sms[64];
  static std::once_flag sm_flags[64];
  std::call_once(sm_flags[dev], [&] {
    if (cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms[dev] = 0;
  });
  if (sms[dev] <= 0) return cudaErrorInvalidDevice;
  const long long items = static_cast<long long>((p.T + BM - 1) / BM) * p.A * p.H_q;
  const unsigned grid = static_cast<unsigned>(items < sms[dev] ? items : sms[dev]);  // one CTA per SM
  prefill_attention_kernel<D><<<grid, THREADS, PCfg<D>::SMEM, stream>>>(p, m.q, m.k, m.v);
  return cudaGetLastError();
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tma_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

cudaError_t launch_prefill_attention(const PrefillParams& p, cudaStream_t stream) {
  if (p.A == 0 || p.T == 0) return cudaSuccess;
  PrefillMaps m;
  cudaError_t e = make_maps(p, &m);
  if (e != cudaSuccess) return e;
  if (p.D == 128) return launch_d<128>(p, m, stream);
  if (p.D == 64) return launch_d<64>(p, m, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvgqa
