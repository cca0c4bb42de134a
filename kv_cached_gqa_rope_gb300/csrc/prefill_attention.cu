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
// One CTA computes a 128-query tile of one (prompt a, query head h):
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
constexpr int THREADS = 192;   // 4 softmax warps + producer + MMA
constexpr int TMEM_COLS = 512;
constexpr unsigned FULLMASK = 0xffffffffu;

template <int D>
struct PCfg {
  static constexpr int NSUB = D / 64;               // 64-wide sub-tiles per row
  static constexpr int NS = D == 128 ? 2 : 3;       // K/V stages
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = NSUB * SUB;
  static constexpr int STAGE = 2 * NSUB * SUB;      // K then V
  static constexpr int P_OFF = KV_OFF + NS * STAGE;
  static constexpr int BAR_OFF = P_OFF + 2 * SUB;
  // barriers: q_full, kv_full[NS], kv_empty[NS], s_full[2], p_full, o_done, drain
  static constexpr int NBAR = 1 + 2 * NS + 2 + 3;
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
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 1 + C::NS;
  uint64_t* s_full = bars + 1 + 2 * C::NS;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SLOT_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::FLAG_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqt = (p.T + BM - 1) / BM;
  const int heads = p.A * p.H_q;
  const int qt = nqt - 1 - static_cast<int>(blockIdx.x) / heads;  // longest tiles first
  const int rem = static_cast<int>(blockIdx.x) % heads;
  const int a = rem / p.H_q, h = rem % p.H_q, g = h / p.G;
  const int row = p.cache_rows[a];
  if (row < 0 || row >= p.S) {
    if (threadIdx.x == 0 && qt == nqt - 1 && h == 0) atomicOr(p.status, KVGQA_FLAG_ROW_RANGE);
    return;
  }
  const int nkt = qt + 1;  // key tiles 0..qt (the last one on the diagonal)

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, BM);
    mbar_init(o_done, 1);
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_q = l2_evict_first_policy();
      const uint64_t pol_kv = l2_evict_last_policy();  // K/V tiles are re-read by the group's heads
      mbar_arrive_expect_tx(q_full, BM * D * 2);
      for (int sub = 0; sub < C::NSUB; ++sub)
        tma_load_4d(smem + C::Q_OFF + sub * SUB, &map_q, sub * 64, h, qt * BM, a, q_full, pol_q);
      const int kv_row = row * p.H_kv + g;
      int j = 0;
      for (; j < nkt; ++j) {
        const int s = j % C::NS;
        if (j >= C::NS && !mbar_wait_bounded(&kv_empty[s], ((j / C::NS) - 1) & 1, abort_flag, p.status)) break;
        unsigned char* st = smem + C::KV_OFF + s * C::STAGE;
        mbar_arrive_expect_tx(&kv_full[s], 2 * BN * D * 2);
        for (int sub = 0; sub < C::NSUB; ++sub) {
          tma_load_3d(st + sub * SUB, &map_k, sub * 64, j * BN, kv_row, &kv_full[s], pol_kv);
          tma_load_3d(st + (C::NSUB + sub) * SUB, &map_v, sub * 64, j * BN, kv_row, &kv_full[s], pol_kv);
        }
      }
      if (*abort_flag) {
        // drain: wait (bounded) for the copies that may still be landing
        volatile int none = 0;
        mbar_wait_bounded(q_full, 0, &none, nullptr);
        for (int t = j - C::NS < 0 ? 0 : j - C::NS; t < j; ++t)
          mbar_wait_bounded(&kv_full[t % C::NS], (t / C::NS) & 1, &none, nullptr);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, 1);
      const uint32_t q_addr = sbase + C::Q_OFF, p_addr = sbase + C::P_OFF;
      bool issued = false;
      auto issue_qk = [&](int j) {
        const uint32_t k_addr = sbase + C::KV_OFF + (j % C::NS) * C::STAGE;
        const uint32_t d_tmem = tmem + (j & 1) * BN;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks / 4) * SUB + (ks % 4) * 32;
          umma_f16_ss(d_tmem, smem_desc_sw128(q_addr + off, 16, 1024), smem_desc_sw128(k_addr + off, 16, 1024),
                      IDESC_QK, ks > 0);
        }
        umma_commit(&s_full[j & 1]);
        issued = true;
      };
      bool ok = mbar_wait_bounded(q_full, 0, abort_flag, p.status) &&
                mbar_wait_bounded(&kv_full[0], 0, abort_flag, p.status);
      if (ok) {
        tc_fence_after();
        issue_qk(0);
      }
      for (int j = 0; ok && j < nkt; ++j) {
        if (j + 1 < nkt) {
          if (!mbar_wait_bounded(&kv_full[(j + 1) % C::NS], ((j + 1) / C::NS) & 1, abort_flag, p.status)) break;
          tc_fence_after();
          issue_qk(j + 1);
        }
        if (!mbar_wait_bounded(p_full, j & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t v_addr = sbase + C::KV_OFF + (j % C::NS) * C::STAGE + C::NSUB * SUB;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint32_t poff = (ks / 4) * SUB + (ks % 4) * 32;
          umma_f16_ss(tmem + 2 * BN, smem_desc_sw128(p_addr + poff, 16, 1024),
                      smem_desc_sw128(v_addr + ks * 2048, SUB, 1024), IDESC_PV, (j > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(o_done);
        umma_commit(&kv_empty[j % C::NS]);
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
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    unsigned char* prow0 = smem + C::P_OFF + r * 128;
    for (int j = 0; j < nkt; ++j) {
      // wait outcomes are made warp-uniform: tcgen05.ld/st need the whole warp
      if (!__all_sync(FULLMASK, mbar_wait_bounded(&s_full[j & 1], (j >> 1) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_base + (j & 1) * BN + c * 32, u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(u[i]) * p.scale_log2;
      }
      if (j == qt) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c > r) x[c] = -INFINITY;
      }
      float mt = x[0];
#pragma unroll
      for (int c = 1; c < BN; ++c) mt = fmaxf(mt, x[c]);
      // PV of the previous tile must be done before O is rescaled or P rewritten.
      if (j > 0 && !__all_sync(FULLMASK, mbar_wait_bounded(o_done, (j - 1) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool grow = mt > m_ref + 8.f;  // always true for the first tile
      float alpha = 1.f;
      if (grow) {
        alpha = exp2f(m_ref - mt);          // 0 for the first tile
        m_ref = mt;
        l *= alpha;
      }
      if (j > 0 && __any_sync(FULLMASK, grow)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t u[32];
          tmem_ld32(tmem + lane_base + 2 * BN + c * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
          tmem_st32(tmem + lane_base + 2 * BN + c * 32, u);
        }
        tmem_wait_st();
      }
      float lsum = 0.f;
#pragma unroll
      for (int ch = 0; ch < BN / 8; ++ch) {  // 16 chunks of 8 keys
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = exp2f(x[ch * 8 + 2 * e] - m_ref);
          const float p1 = exp2f(x[ch * 8 + 2 * e + 1] - m_ref);
          w[e] = pack2(p0, p1);
          // accumulate the rounded weights: O / l is then a convex combination of V
          lsum += __uint_as_float(w[e] << 16) + __uint_as_float(w[e] & 0xffff0000u);
        }
        const int sub = ch / 8, cc = ch % 8;
        uint4* dst = reinterpret_cast<uint4*>(prow0 + sub * SUB + ((cc ^ (r & 7)) << 4));
        *dst = make_uint4(w[0], w[1], w[2], w[3]);
      }
      l += lsum;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok && __all_sync(FULLMASK, mbar_wait_bounded(o_done, (nkt - 1) & 1, abort_flag, p.status))) {
      tc_fence_after();
      const int t = qt * BM + r;
      const float inv = 1.f / l;
      uint16_t* dst = p.out + ((static_cast<size_t>(a) * p.T + t) * p.H_q + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_base + 2 * BN + c * 32, u);
        tmem_wait_ld();
        if (t < p.T) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 o;
            o.x = pack2(__uint_as_float(u[q4 * 8 + 0]) * inv, __uint_as_float(u[q4 * 8 + 1]) * inv);
            o.y = pack2(__uint_as_float(u[q4 * 8 + 2]) * inv, __uint_as_float(u[q4 * 8 + 3]) * inv);
            o.z = pack2(__uint_as_float(u[q4 * 8 + 4]) * inv, __uint_as_float(u[q4 * 8 + 5]) * inv);
            o.w = pack2(__uint_as_float(u[q4 * 8 + 6]) * inv, __uint_as_float(u[q4 * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + c * 32 + q4 * 8) = o;
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
  const int nqt = (p.T + BM - 1) / BM;
  const unsigned grid = static_cast<unsigned>(nqt) * p.A * p.H_q;
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
