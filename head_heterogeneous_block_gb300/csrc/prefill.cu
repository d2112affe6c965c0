// Block-sparse causal prefill attention on sm_103a.
//
// One persistent CTA per schedule worker walks that worker's (head,
// query-block) items.  For every item it loads the 128-row query tile once
// and then, for each selected key block j, computes S = Q K_j^T and
// O += softmax(S) V_j with flash-style online softmax:
//
//   warp 0      TMA producer: Q tiles and the selected K / V blocks, each a
//               128-byte-swizzled box of the [heads*S, d] view, into rings of
//               shared-memory stages.
//   warp 1      MMA issuer (one thread): tcgen05.mma kind::f16, bf16 inputs,
//               fp32 accumulators in tensor memory.  S_j goes to one of two
//               TMEM buffers so QK^T of block j+1 overlaps the softmax of
//               block j; P_j is written back over S_j (bf16) and used as the
//               TMEM A operand of P V.  O accumulates in TMEM.
//   warps 2-5   softmax (one query row per thread): read S_j from TMEM, mask
//               the diagonal block causally, keep the running max and sum,
//               write P_j; rescale O in TMEM only when the max grew by more
//               than 2^8 (otherwise the stale max is kept and cancels in the
//               final division); epilogue O / l -> bf16, and the log-sum-exp.
//
// The work items and their order come from the plan's LPT schedule (S-HPLB,
// "Algoritmo Greedy"), with workers = CTAs instead of GPUs.
// Every index read from idx / cnt / the schedule is range-checked; bad values
// are clamped and flagged in the device status word, never dereferenced.
// Every wait is bounded; on a timeout the CTA flags SA_DEV_TIMEOUT, lets its
// copies and MMAs drain, frees its tensor memory and exits.

#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "sparse_attn.h"

namespace {

using namespace sa_dev;

template <int D, int BK>
struct Cfg {
  static constexpr int kM = 128;                  // query rows per tile
  static constexpr int kPanels = D / 64;          // 128-byte column panels
  static constexpr int kQPanel = kM * 128;        // bytes of one Q panel
  static constexpr int kKVPanel = BK * 128;       // bytes of one K/V panel
  static constexpr int kQBytes = kM * D * 2;
  static constexpr int kKVBytes = BK * D * 2;
  static constexpr int kNQ = 2;                   // Q stages
  static constexpr int kNK = 3;                   // K stages
  static constexpr int kNV = 2;                   // V stages
  static constexpr uint32_t kS0 = 0, kS1 = BK, kO = 2 * BK;   // TMEM columns
  static constexpr uint32_t kTmemCols = (2 * BK + D <= 256) ? 256 : 512;
  static constexpr int kData = kNQ * kQBytes + kNK * kKVBytes + kNV * kKVBytes;
  static constexpr int kThreads = 192;
  static constexpr int kSmem = kData + 256 + 1024;  // + barriers + alignment slack
};

struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[3], k_empty[3];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done;   // one phase per P.V (waited only before an O rescale)
  uint64_t o_last;   // one phase per item, after its last P.V (epilogue)
  uint64_t o_free, drain;
  uint32_t tmem_base;
  int abort;
};

struct Params {
  const int32_t* idx;
  const int32_t* cnt;
  const int32_t* wptr;
  const int32_t* items;
  int32_t kmax, num_items, num_workers, nb, S, B, G;
  float scale_log2;
  void* o;
  int32_t out_f32;
  float* lse;
  int32_t* dev_status;
};

struct Item {
  int32_t h, i, n;
  const int32_t* list;
};

// Item at schedule position `pos`; n == 0 means "skip" (flagged).
__device__ __forceinline__ Item load_item(const Params& p, int pos, bool report) {
  Item r{0, 0, 0, nullptr};
  const int32_t item = p.items[pos];
  if (item < 0 || item >= p.num_items) {
    if (report) atomicOr(p.dev_status, SA_DEV_BAD_ITEM);
    return r;
  }
  r.h = item / p.nb;
  r.i = item - r.h * p.nb;
  const int32_t lim = min(p.kmax, r.i + 1);
  int32_t n = p.cnt[item];
  if (n < 1 || n > lim) {
    if (report) atomicOr(p.dev_status, SA_DEV_BAD_COUNT);
    n = max(1, min(n, lim));
  }
  r.n = n;
  r.list = p.idx + size_t(item) * size_t(p.kmax);
  return r;
}

__device__ __forceinline__ int32_t load_block(const Item& it, int t, const Params& p,
                                              bool report) {
  int32_t j = it.list[t];
  if (j < 0 || j > it.i) {
    if (report) atomicOr(p.dev_status, SA_DEV_BAD_INDEX);
    j = 0;
  }
  return j;
}

__device__ __forceinline__ void raise_abort(Bars* bars, const Params& p) {
  atomicOr(p.dev_status, SA_DEV_TIMEOUT);
  *(volatile int*)&bars->abort = 1;
}

// Wait for the last `min(issued, stages)` loads of a ring to land.
__device__ __forceinline__ void drain_ring(uint64_t* full, uint32_t issued, int stages) {
  const uint32_t first = issued > uint32_t(stages) ? issued - stages : 0;
  for (uint32_t x = first; x < issued; ++x)
    mbar_wait(&full[x % stages], (x / stages) & 1, nullptr);
}

template <int D, int BK>
__global__ void __launch_bounds__(192, 1)
    prefill_attention_kernel(const __grid_constant__ CUtensorMap tq,
                             const __grid_constant__ CUtensorMap tk,
                             const __grid_constant__ CUtensorMap tv, const Params p) {
  using C = Cfg<D, BK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::kNQ * C::kQBytes;
  uint8_t* sV = sK + C::kNK * C::kKVBytes;
  Bars* bars = reinterpret_cast<Bars*>(sV + C::kNV * C::kKVBytes);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // This worker's slice of the schedule.
  int32_t begin = p.wptr[blockIdx.x], end = p.wptr[blockIdx.x + 1];
  if (begin < 0 || end > p.num_items || begin > end) {
    if (threadIdx.x == 0) atomicOr(p.dev_status, SA_DEV_BAD_ITEM);
    begin = end = 0;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 128);
    }
    for (int s = 0; s < 3; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->o_last, 1);
    mbar_init(&bars->o_free, 128);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      const uint64_t pol_kv = l2_policy_evict_last();
      const uint64_t pol_q = l2_policy_evict_first();
      uint32_t qi = 0, kissued = 0, vissued = 0;
      bool ok = true;
      for (int pos = begin; pos < end && ok; ++pos) {
        const Item it = load_item(p, pos, true);
        if (it.n == 0) continue;
        const int g = it.h / p.G;
        const int qs = qi % C::kNQ;
        if (qi >= uint32_t(C::kNQ) &&
            !mbar_wait(&bars->q_empty[qs], ((qi / C::kNQ) - 1) & 1, abort)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars->q_full[qs], C::kQBytes);
#pragma unroll
        for (int s = 0; s < C::kPanels; ++s)
          tma_load_2d(sQ + qs * C::kQBytes + s * C::kQPanel, &tq, &bars->q_full[qs], s * 64,
                      it.h * p.S + it.i * p.B, pol_q);
        ++qi;
        for (int t = 0; t < it.n; ++t) {
          const int32_t j = load_block(it, t, p, true);
          const int ks = kissued % C::kNK;
          if (kissued >= uint32_t(C::kNK) &&
              !mbar_wait(&bars->k_empty[ks], ((kissued / C::kNK) - 1) & 1, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->k_full[ks], C::kKVBytes);
#pragma unroll
          for (int s = 0; s < C::kPanels; ++s)
            tma_load_2d(sK + ks * C::kKVBytes + s * C::kKVPanel, &tk, &bars->k_full[ks], s * 64,
                        g * p.S + j * BK, pol_kv);
          ++kissued;
          const int vs = vissued % C::kNV;
          if (vissued >= uint32_t(C::kNV) &&
              !mbar_wait(&bars->v_empty[vs], ((vissued / C::kNV) - 1) & 1, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->v_full[vs], C::kKVBytes);
#pragma unroll
          for (int s = 0; s < C::kPanels; ++s)
            tma_load_2d(sV + vs * C::kKVBytes + s * C::kKVPanel, &tv, &bars->v_full[vs], s * 64,
                        g * p.S + j * BK, pol_kv);
          ++vissued;
        }
      }
      if (!ok) raise_abort(bars, p);
      // Copies still in flight must land before this CTA's shared memory goes.
      drain_ring(bars->q_full, qi, C::kNQ);
      drain_ring(bars->k_full, kissued, C::kNK);
      drain_ring(bars->v_full, vissued, C::kNV);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, BK, 0, 0);  // Q, K both K-major
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, 0, 1);   // P (TMEM), V MN-major
      uint32_t qi = 0, kb = 0, items_done = 0;
      bool ok = true;

      auto issue_pv = [&](uint32_t b, bool first) -> bool {
        const int pb = b & 1;
        if (!mbar_wait(&bars->p_full[pb], (b >> 1) & 1, abort)) return false;
        const int vs = b % C::kNV;
        if (!mbar_wait(&bars->v_full[vs], (b / C::kNV) & 1, abort)) return false;
        if (first && items_done > 0 && !mbar_wait(&bars->o_free, (items_done - 1) & 1, abort))
          return false;
        tc_fence_after();
        const uint32_t v_base = smem_u32(sV + vs * C::kKVBytes);
        const uint32_t p_tmem = tmem + (pb ? C::kS1 : C::kS0);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // 16 keys per step: 16 rows of 128 bytes in every d panel
          const uint64_t bd = smem_desc_sw128(v_base + kk * 16 * 128, C::kKVPanel, 1024);
          mma_ts(tmem + C::kO, p_tmem + kk * 8, bd, idesc_pv, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(&bars->v_empty[vs]);
        mma_commit(&bars->o_done);
        return true;
      };

      for (int pos = begin; pos < end && ok; ++pos) {
        const Item it = load_item(p, pos, false);
        if (it.n == 0) continue;
        const int qs = qi % C::kNQ;
        if (!mbar_wait(&bars->q_full[qs], (qi / C::kNQ) & 1, abort)) {
          ok = false;
          break;
        }
        const uint32_t q_base = smem_u32(sQ + qs * C::kQBytes);
        for (int t = 0; t < it.n; ++t) {
          const int ks = kb % C::kNK;
          if (!mbar_wait(&bars->k_full[ks], (kb / C::kNK) & 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k_base = smem_u32(sK + ks * C::kKVBytes);
          const uint32_t s_tmem = tmem + ((kb & 1) ? C::kS1 : C::kS0);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // 16 dims per step: panel kk/4, 32-byte column offset inside the
            // swizzle atom (the hardware applies the XOR on the full address)
            const uint32_t off = (kk % 4) * 32;
            const uint64_t ad =
                smem_desc_sw128(q_base + (kk / 4) * C::kQPanel + off, 16, 1024);
            const uint64_t bd =
                smem_desc_sw128(k_base + (kk / 4) * C::kKVPanel + off, 16, 1024);
            mma_ss(s_tmem, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[kb & 1]);
          mma_commit(&bars->k_empty[ks]);
          if (t == it.n - 1) mma_commit(&bars->q_empty[qs]);
          if (t > 0 && !issue_pv(kb - 1, t == 1)) {
            ok = false;
            break;
          }
          ++kb;
        }
        if (!ok) break;
        if (!issue_pv(kb - 1, it.n == 1)) {
          ok = false;
          break;
        }
        mma_commit(&bars->o_last);
        ++qi;
        ++items_done;
      }
      if (!ok) raise_abort(bars, p);
      // Every MMA must be complete before the tensor memory is freed.
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------ softmax warps
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;          // query row within the tile
    const uint32_t lanes = tmem + (uint32_t(quarter * 32) << 16);
    const float c = p.scale_log2;
    uint32_t kb = 0, items_done = 0;
    bool ok = true;
    for (int pos = begin; pos < end && ok; ++pos) {
      const Item it = load_item(p, pos, false);
      if (it.n == 0) continue;
      float m_used = -INFINITY, l = 0.f;
      for (int t = 0; t < it.n; ++t) {
        const int32_t j = load_block(it, t, p, false);
        const int sb = kb & 1;
        if (!mbar_wait(&bars->s_full[sb], (kb >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t scol = sb ? C::kS1 : C::kS0;
        uint32_t sr[BK / 32][32];
#pragma unroll
        for (int q = 0; q < BK / 32; ++q) tmem_ld32(lanes + scol + q * 32, sr[q]);
        tmem_ld_wait(sr[0]);
#pragma unroll
        for (int q = 1; q < BK / 32; ++q) reg_fence(sr[q]);
        float s[BK];
#pragma unroll
        for (int q = 0; q < BK / 32; ++q)
#pragma unroll
          for (int x = 0; x < 32; ++x) s[q * 32 + x] = __uint_as_float(sr[q][x]);
        if (j == it.i) {
#pragma unroll
          for (int x = 0; x < BK; ++x)
            if (x > row) s[x] = -INFINITY;
        }
        float mx = s[0];
#pragma unroll
        for (int x = 1; x < BK; ++x) mx = fmaxf(mx, s[x]);
        const float m_blk = mx * c;
        if (t == 0) {
          m_used = m_blk;
        } else {
          const bool need = m_blk > m_used + 8.0f;
          if (__any_sync(0xffffffffu, need)) {
            // O still receives P V of the previous block: let it finish first.
            // The parity wait is unambiguous: S of this block was committed
            // after P V of block kb-2, so at least kb-1 phases are complete,
            // and P V of this block is not issued yet.
            if (!mbar_wait(&bars->o_done, (kb - 1) & 1, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            float alpha = 1.f;
            if (need) {
              alpha = ex2(m_used - m_blk);
              m_used = m_blk;
              l *= alpha;
            }
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
              uint32_t r[32];
              tmem_ld32(lanes + C::kO + q * 32, r);
              tmem_ld_wait(r);
#pragma unroll
              for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * alpha);
              tmem_st32(lanes + C::kO + q * 32, r);
            }
            tmem_st_wait();
          }
        }
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < BK / 64; ++q) {
          uint32_t pk[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const float p0 = ex2(fmaf(s[q * 64 + 2 * x], c, -m_used));
            const float p1 = ex2(fmaf(s[q * 64 + 2 * x + 1], c, -m_used));
            pk[x] = pack_bf16x2(p0, p1);
            // normalise by the same rounded weights the P.V product uses
            sum += __uint_as_float(pk[x] << 16) + __uint_as_float(pk[x] & 0xFFFF0000u);
          }
          tmem_st32(lanes + scol + q * 32, pk);
        }
        tmem_st_wait();
        l += sum;
        tc_fence_before();
        mbar_arrive(&bars->p_full[sb]);
        ++kb;
      }
      if (!ok) break;
      // ---- epilogue: O / l.  o_last has exactly one phase per item and
      // this warp waits on every one of them.
      if (!mbar_wait(&bars->o_last, items_done & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv_l = 1.f / l;
      const bool store = row < p.B;
      const size_t orow = size_t(it.h) * p.S + size_t(it.i) * p.B + size_t(row);
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t r[32];
        tmem_ld32(lanes + C::kO + q * 32, r);
        tmem_ld_wait(r);
        if (!store) continue;
        if (p.out_f32) {
          uint4* d4 = reinterpret_cast<uint4*>(static_cast<float*>(p.o) + orow * D + q * 32);
#pragma unroll
          for (int x = 0; x < 8; ++x)
            d4[x] = make_uint4(__float_as_uint(__uint_as_float(r[4 * x]) * inv_l),
                               __float_as_uint(__uint_as_float(r[4 * x + 1]) * inv_l),
                               __float_as_uint(__uint_as_float(r[4 * x + 2]) * inv_l),
                               __float_as_uint(__uint_as_float(r[4 * x + 3]) * inv_l));
        } else {
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x)
            pk[x] = pack_bf16x2(__uint_as_float(r[2 * x]) * inv_l,
                                __uint_as_float(r[2 * x + 1]) * inv_l);
          uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow * D +
                                               q * 32);
#pragma unroll
          for (int x = 0; x < 4; ++x)
            d4[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
        }
      }
      if (p.lse && store)
        p.lse[size_t(it.h) * p.S + size_t(it.i) * p.B + row] =
            (m_used + log2f(l)) * 0.6931471805599453f;
      tc_fence_before();
      mbar_arrive(&bars->o_free);
      ++items_done;
    }
    if (!ok) raise_abort(bars, p);
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  }
  return fn;
}

// [rows, d] bf16 view, boxes of 64 columns x box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, int d, int box_rows) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cuuint64_t(d), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(d) * 2};
  const cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int BK>
cudaError_t launch(const sa_k::PrefillArgs& a, cudaStream_t st, bool* encode_failed) {
  using C = Cfg<D, BK>;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, a.q, uint64_t(a.Hq) * a.S, D, C::kM) ||
      !make_map(&tk, a.k, uint64_t(a.Hkv) * a.S, D, BK) ||
      !make_map(&tv, a.v, uint64_t(a.Hkv) * a.S, D, BK)) {
    *encode_failed = true;
    return cudaErrorInvalidValue;
  }
  Params p;
  p.idx = a.idx;
  p.cnt = a.cnt;
  p.wptr = a.wptr;
  p.items = a.items;
  p.kmax = a.kmax;
  p.num_items = a.num_items;
  p.num_workers = a.num_workers;
  p.nb = a.S / a.B;
  p.S = a.S;
  p.B = a.B;
  p.G = a.Hq / a.Hkv;
  p.scale_log2 = float(1.4426950408889634 / std::sqrt(double(D)));
  p.o = a.o;
  p.out_f32 = a.out_f32;
  p.lse = a.lse;
  p.dev_status = a.dev_status;
  auto kern = prefill_attention_kernel<D, BK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  if (a.num_workers == 0) return cudaSuccess;
  kern<<<a.num_workers, C::kThreads, C::kSmem, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

namespace sa_k {

cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t st, bool* encode_failed) {
  *encode_failed = false;
  if (a.d == 128 && a.B == 128) return launch<128, 128>(a, st, encode_failed);
  if (a.d == 64 && a.B == 64) return launch<64, 64>(a, st, encode_failed);
  return cudaErrorInvalidValue;
}

}  // namespace sa_k
