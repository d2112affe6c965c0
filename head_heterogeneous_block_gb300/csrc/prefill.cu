// Block-sparse causal prefill attention on sm_103a.
//
// One persistent CTA per schedule worker walks that worker's (head,
// query-block) items.  For every item it loads the 128-row query tile once
// and then, for each selected key block j, computes S = Q K_j^T and
// O += softmax(S) V_j with flash-style online softmax:
//
//   warp 0      producer: reads the schedule, the block counts and the block
//               lists (32 indices per load), publishes each item's metadata
//               through a small shared-memory ring, and issues TMA loads of
//               the Q tile and the selected K / V blocks (128-byte-swizzled
//               boxes of the [heads*S, d] view) into rings of stages.
//   warp 1      MMA issuer (one thread): tcgen05.mma kind::f16, bf16 inputs,
//               fp32 accumulators in tensor memory.  S_j alternates between
//               two TMEM buffers so Q K_{j+1}^T overlaps the softmax of block
//               j; P_j is written back into S_j's columns (bf16) and is the
//               TMEM A operand of P V.  O accumulates in TMEM.
//   warps 2-9   softmax, two warpgroups: each row of the tile has one thread
//               in each group, which take the left and right halves of the
//               S columns (and of O).  The halves exchange their partial row
//               maxima through shared memory, so both keep the same running
//               max; O is rescaled in TMEM only when the max grew by more
//               than 2^8 (the stale max cancels in the final division).  The
//               normaliser sums the same bf16-rounded weights that enter P V.
//               Epilogue: O / l in fp32 or bf16, and the log-sum-exp.
//
// The work items and their order come from the plan's LPT schedule (S-HPLB,
// "Algoritmo Greedy"), with workers = CTAs instead of GPUs.
// Every index read from idx / cnt / the schedule is range-checked; bad values
// are clamped and flagged in the device status word, never dereferenced.
// Every wait (including the exchanges between the two softmax groups) is a
// bounded mbarrier wait; on a timeout the CTA flags SA_DEV_TIMEOUT, lets its
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
  static constexpr int kNK = 2;                   // K stages
  static constexpr int kNV = 2;                   // V stages
  static constexpr int kHalfS = BK / 2;           // S columns per softmax group
  static constexpr int kHalfO = D / 2;            // O columns per softmax group
  static constexpr uint32_t kS0 = 0, kS1 = BK, kO = 2 * BK;   // TMEM columns
  static constexpr uint32_t kTmemCols = (2 * BK + D <= 256) ? 256 : 512;
  static constexpr int kData = kNQ * kQBytes + kNK * kKVBytes + kNV * kKVBytes;
  static constexpr int kThreads = 320;
};

constexpr int kNI = 4;        // item-metadata ring slots
constexpr int kSoftmaxThreads = 256;

struct ItemInfo {
  int32_t h, i, n, diag_last;   // n == 0: end of this worker's list
};

struct Shared {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done;        // one phase per P.V (waited only before an O rescale)
  uint64_t o_last;        // one phase per item, after its last P.V (epilogue)
  uint64_t o_free;        // one phase per item: the epilogue has read O
  uint64_t drain;
  uint64_t info_full[kNI], info_empty[kNI];
  uint64_t xmax_bar[2];   // per block: both groups posted their partial maxima
  uint64_t xsum_bar[2];   // per item: both groups posted their partial sums
  ItemInfo info[kNI];
  float xmax[2][2][128];  // [block parity][group][row]
  float xsum[2][2][128];  // [item parity][group][row]
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

__device__ __forceinline__ void raise_abort(Shared* sh, const Params& p) {
  atomicOr(p.dev_status, SA_DEV_TIMEOUT);
  *(volatile int*)&sh->abort = 1;
}

// Wait for the last `min(issued, stages)` loads of a ring to land.
__device__ __forceinline__ void drain_ring(uint64_t* full, uint32_t issued, int stages) {
  const uint32_t first = issued > uint32_t(stages) ? issued - stages : 0;
  for (uint32_t x = first; x < issued; ++x)
    mbar_wait(&full[x % stages], (x / stages) & 1, nullptr);
}

template <int D, int BK>
__global__ void __launch_bounds__(320, 1)
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
  Shared* sh = reinterpret_cast<Shared*>(sV + C::kNV * C::kKVBytes);
  volatile int* abort = &sh->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh->q_full[s], 1);
      mbar_init(&sh->q_empty[s], 1);
      mbar_init(&sh->k_full[s], 1);
      mbar_init(&sh->k_empty[s], 1);
      mbar_init(&sh->v_full[s], 1);
      mbar_init(&sh->v_empty[s], 1);
      mbar_init(&sh->s_full[s], 1);
      mbar_init(&sh->p_full[s], kSoftmaxThreads);
      mbar_init(&sh->xmax_bar[s], kSoftmaxThreads);
      mbar_init(&sh->xsum_bar[s], kSoftmaxThreads);
    }
    for (int s = 0; s < kNI; ++s) {
      mbar_init(&sh->info_full[s], 1);
      mbar_init(&sh->info_empty[s], 1 + kSoftmaxThreads / 32);
    }
    mbar_init(&sh->o_done, 1);
    mbar_init(&sh->o_last, 1);
    mbar_init(&sh->o_free, kSoftmaxThreads);
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ producer warp
    int32_t begin = p.wptr[blockIdx.x], end = p.wptr[blockIdx.x + 1];
    if (begin < 0 || end > p.num_items || begin > end) {
      if (lane == 0) atomicOr(p.dev_status, SA_DEV_BAD_ITEM);
      begin = end = 0;
    }
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
    }
    const uint64_t pol_kv = l2_policy_evict_last();
    const uint64_t pol_q = l2_policy_evict_first();
    uint32_t qi = 0, kiss = 0, viss = 0;
    bool ok = true;
    // the schedule entry is read one item ahead of its use
    int32_t item_next = (begin < end) ? p.items[begin] : -1;
    for (int pos = begin; pos < end && ok; ++pos) {
      const int32_t item = item_next;
      if (pos + 1 < end) item_next = p.items[pos + 1];
      if (item < 0 || item >= p.num_items) {
        if (lane == 0) atomicOr(p.dev_status, SA_DEV_BAD_ITEM);
        continue;
      }
      const int32_t h = item / p.nb, i = item - h * p.nb;
      const int32_t lim = min(p.kmax, i + 1);
      int32_t n = p.cnt[item];
      if (n < 1 || n > lim) {
        if (lane == 0) atomicOr(p.dev_status, SA_DEV_BAD_COUNT);
        n = max(1, min(n, lim));
      }
      const int32_t* list = p.idx + size_t(item) * size_t(p.kmax);
      int32_t jl = (lane < n) ? list[lane] : 0;
      const int32_t jlast = list[n - 1];
      const int g = h / p.G;
      if (lane == 0) {
        // publish the item's metadata for the MMA and softmax warps
        const int slot = qi % kNI;
        if (qi >= uint32_t(kNI) &&
            !mbar_wait(&sh->info_empty[slot], ((qi / kNI) - 1) & 1, abort))
          ok = false;
        if (ok) {
          sh->info[slot] = ItemInfo{h, i, n, jlast == i ? 1 : 0};
          mbar_arrive(&sh->info_full[slot]);
          const int qs = qi % C::kNQ;
          if (qi >= uint32_t(C::kNQ) &&
              !mbar_wait(&sh->q_empty[qs], ((qi / C::kNQ) - 1) & 1, abort))
            ok = false;
          if (ok) {
            mbar_arrive_expect_tx(&sh->q_full[qs], C::kQBytes);
#pragma unroll
            for (int s = 0; s < C::kPanels; ++s)
              tma_load_2d(sQ + qs * C::kQBytes + s * C::kQPanel, &tq, &sh->q_full[qs], s * 64,
                          h * p.S + i * p.B, pol_q);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++qi;
      int32_t jprev = -1;
      for (int t = 0; t < n; ++t) {
        if ((t & 31) == 0 && t > 0) jl = (t + lane < n) ? list[t + lane] : 0;
        int32_t j = __shfl_sync(0xffffffffu, jl, t & 31);
        if (j < 0 || j > i || j <= jprev) {   // out of range or not ascending
          if (lane == 0) atomicOr(p.dev_status, SA_DEV_BAD_INDEX);
          if (j < 0 || j > i) j = 0;
        }
        jprev = j;
        if (lane == 0) {
          const int ks = kiss % C::kNK;
          if (kiss >= uint32_t(C::kNK) &&
              !mbar_wait(&sh->k_empty[ks], ((kiss / C::kNK) - 1) & 1, abort))
            ok = false;
          if (ok) {
            mbar_arrive_expect_tx(&sh->k_full[ks], C::kKVBytes);
#pragma unroll
            for (int s = 0; s < C::kPanels; ++s)
              tma_load_2d(sK + ks * C::kKVBytes + s * C::kKVPanel, &tk, &sh->k_full[ks],
                          s * 64, g * p.S + j * BK, pol_kv);
            ++kiss;
            const int vs = viss % C::kNV;
            if (viss >= uint32_t(C::kNV) &&
                !mbar_wait(&sh->v_empty[vs], ((viss / C::kNV) - 1) & 1, abort))
              ok = false;
            if (ok) {
              mbar_arrive_expect_tx(&sh->v_full[vs], C::kKVBytes);
#pragma unroll
              for (int s = 0; s < C::kPanels; ++s)
                tma_load_2d(sV + vs * C::kKVBytes + s * C::kKVPanel, &tv, &sh->v_full[vs],
                            s * 64, g * p.S + j * BK, pol_kv);
              ++viss;
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    if (lane == 0) {
      if (ok) {
        // end marker for the consumers
        const int slot = qi % kNI;
        if (qi >= uint32_t(kNI) &&
            !mbar_wait(&sh->info_empty[slot], ((qi / kNI) - 1) & 1, abort))
          ok = false;
        if (ok) {
          sh->info[slot] = ItemInfo{0, 0, 0, 0};
          mbar_arrive(&sh->info_full[slot]);
        }
      }
      if (!ok) raise_abort(sh, p);
      // copies still in flight must land before this CTA's shared memory goes
      drain_ring(sh->q_full, qi, C::kNQ);
      drain_ring(sh->k_full, kiss, C::kNK);
      drain_ring(sh->v_full, viss, C::kNV);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, BK, 0, 0);  // Q, K both K-major
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, 0, 1);   // P (TMEM), V MN-major
      uint32_t qi = 0, kb = 0;
      bool ok = true;

      auto issue_pv = [&](uint32_t b, bool first) -> bool {
        const int pb = b & 1;
        if (!mbar_wait(&sh->p_full[pb], (b >> 1) & 1, abort)) return false;
        const int vs = b % C::kNV;
        if (!mbar_wait(&sh->v_full[vs], (b / C::kNV) & 1, abort)) return false;
        if (first && qi > 0 && !mbar_wait(&sh->o_free, (qi - 1) & 1, abort)) return false;
        tc_fence_after();
        const uint32_t v_base = smem_u32(sV + vs * C::kKVBytes);
        const uint32_t s_col = pb ? C::kS1 : C::kS0;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // keys [16kk, 16kk+16) sit in the P half of the group that owns them
          const int half = (kk * 16) / C::kHalfS;
          const uint32_t a_col = s_col + half * C::kHalfS + (kk * 16 - half * C::kHalfS) / 2;
          // 16 keys per step: 16 rows of 128 bytes in every d panel
          const uint64_t bd = smem_desc_sw128(v_base + kk * 16 * 128, C::kKVPanel, 1024);
          mma_ts(tmem + C::kO, tmem + a_col, bd, idesc_pv, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(&sh->v_empty[vs]);
        mma_commit(&sh->o_done);
        return true;
      };

      for (;;) {
        const int slot = qi % kNI;
        if (!mbar_wait(&sh->info_full[slot], (qi / kNI) & 1, abort)) {
          ok = false;
          break;
        }
        const int n = sh->info[slot].n;
        mbar_arrive(&sh->info_empty[slot]);
        if (n == 0) break;
        const int qs = qi % C::kNQ;
        if (!mbar_wait(&sh->q_full[qs], (qi / C::kNQ) & 1, abort)) {
          ok = false;
          break;
        }
        const uint32_t q_base = smem_u32(sQ + qs * C::kQBytes);
        for (int t = 0; t < n; ++t) {
          const int ks = kb % C::kNK;
          if (!mbar_wait(&sh->k_full[ks], (kb / C::kNK) & 1, abort)) {
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
            const uint64_t ad = smem_desc_sw128(q_base + (kk / 4) * C::kQPanel + off, 16, 1024);
            const uint64_t bd =
                smem_desc_sw128(k_base + (kk / 4) * C::kKVPanel + off, 16, 1024);
            mma_ss(s_tmem, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(&sh->s_full[kb & 1]);
          mma_commit(&sh->k_empty[ks]);
          if (t == n - 1) mma_commit(&sh->q_empty[qs]);
          if (t > 0 && !issue_pv(kb - 1, t == 1)) {
            ok = false;
            break;
          }
          ++kb;
        }
        if (!ok) break;
        if (!issue_pv(kb - 1, n == 1)) {
          ok = false;
          break;
        }
        mma_commit(&sh->o_last);
        ++qi;
      }
      if (!ok) raise_abort(sh, p);
      // every MMA must be complete before the tensor memory is freed
      mma_commit(&sh->drain);
      mbar_wait(&sh->drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------ softmax groups
    const int grp = (warp - 2) >> 2;              // 0: left half, 1: right half
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;          // query row within the tile
    const uint32_t lanes = tmem + (uint32_t(quarter * 32) << 16);
    const float c = p.scale_log2;
    const uint32_t o_col = C::kO + grp * C::kHalfO;
    uint32_t kb = 0, qi = 0;
    bool ok = true;
    for (;;) {
      const int slot = qi % kNI;
      if (!mbar_wait(&sh->info_full[slot], (qi / kNI) & 1, abort)) {
        ok = false;
        break;
      }
      const ItemInfo it = sh->info[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->info_empty[slot]);
      if (it.n == 0) break;
      float m_used = -INFINITY, l = 0.f;
      for (int t = 0; t < it.n; ++t) {
        const int sb = kb & 1;
        if (!mbar_wait(&sh->s_full[sb], (kb >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t scol = (sb ? C::kS1 : C::kS0) + grp * C::kHalfS;
        uint32_t sr[C::kHalfS / 32][32];
#pragma unroll
        for (int q = 0; q < C::kHalfS / 32; ++q) tmem_ld32(lanes + scol + q * 32, sr[q]);
        tmem_ld_wait(sr[0]);
#pragma unroll
        for (int q = 1; q < C::kHalfS / 32; ++q) reg_fence(sr[q]);
        float s[C::kHalfS];
#pragma unroll
        for (int q = 0; q < C::kHalfS / 32; ++q)
#pragma unroll
          for (int x = 0; x < 32; ++x) s[q * 32 + x] = __uint_as_float(sr[q][x]);
        if (it.diag_last && t == it.n - 1) {
          // key column grp*kHalfS + x is visible to row `row` when <= row
#pragma unroll
          for (int x = 0; x < C::kHalfS; ++x)
            if (grp * C::kHalfS + x > row) s[x] = -INFINITY;
        }
        // partial row maximum over eight independent chains
        float mx[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx[a] = s[a];
#pragma unroll
        for (int x = 8; x + 16 <= C::kHalfS; x += 16)
#pragma unroll
          for (int a = 0; a < 8; ++a) mx[a] = max3(mx[a], s[x + a], s[x + 8 + a]);
        if constexpr ((C::kHalfS - 8) % 16 != 0) {
#pragma unroll
          for (int a = 0; a < 8; ++a) mx[a] = fmaxf(mx[a], s[C::kHalfS - 8 + a]);
        }
        const float mine = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]),
                                fmaxf(mx[6], mx[7]));
        // exchange with the other group (same row, other half of the columns)
        sh->xmax[sb][grp][row] = mine;
        mbar_arrive(&sh->xmax_bar[sb]);
        if (!mbar_wait(&sh->xmax_bar[sb], (kb >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        const float m_blk = fmaxf(mine, sh->xmax[sb][grp ^ 1][row]) * c;
        if (t == 0) {
          m_used = m_blk;
        } else {
          const bool need = m_blk > m_used + 8.0f;
          if (__any_sync(0xffffffffu, need)) {
            // O still receives P V of the previous block: let it finish first.
            // The parity wait is unambiguous: S of this block was committed
            // after P V of block kb-2, so at least kb-1 phases are complete,
            // and P V of this block is not issued yet.
            if (!mbar_wait(&sh->o_done, (kb - 1) & 1, abort)) {
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
            for (int q = 0; q < C::kHalfO / 32; ++q) {
              uint32_t r[32];
              tmem_ld32(lanes + o_col + q * 32, r);
              tmem_ld_wait(r);
#pragma unroll
              for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * alpha);
              tmem_st32(lanes + o_col + q * 32, r);
            }
            tmem_st_wait();
          }
        }
        // P = 2^(s*c - m) in bf16, written over this group's S columns; the
        // normaliser sums the rounded values
        float sum0 = 0.f, sum1 = 0.f, sum2 = 0.f, sum3 = 0.f;
        const float nm = -m_used;
        uint32_t pk[C::kHalfS / 2];
#pragma unroll
        for (int x = 0; x < C::kHalfS / 2; ++x) {
          float a0, a1;
          fma2(a0, a1, s[2 * x], s[2 * x + 1], c, c, nm, nm);
          pk[x] = pack_bf16x2(ex2(a0), ex2(a1));
          if (x & 1)
            add2(sum2, sum3, __uint_as_float(pk[x] << 16), __uint_as_float(pk[x] & 0xFFFF0000u));
          else
            add2(sum0, sum1, __uint_as_float(pk[x] << 16), __uint_as_float(pk[x] & 0xFFFF0000u));
        }
        if constexpr (C::kHalfS / 2 == 32) {
          tmem_st32(lanes + scol, pk);
        } else {
          tmem_st16(lanes + scol, pk);
        }
        tmem_st_wait();
        l += (sum0 + sum1) + (sum2 + sum3);
        tc_fence_before();
        mbar_arrive(&sh->p_full[sb]);
        ++kb;
      }
      if (!ok) break;
      // ---- epilogue: exchange the partial sums, then O / l for this half.
      // o_last has exactly one phase per item and this warp waits on every one.
      sh->xsum[qi & 1][grp][row] = l;
      mbar_arrive(&sh->xsum_bar[qi & 1]);
      if (!mbar_wait(&sh->o_last, qi & 1, abort) ||
          !mbar_wait(&sh->xsum_bar[qi & 1], (qi >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float lt = l + sh->xsum[qi & 1][grp ^ 1][row];
      const float inv_l = 1.f / lt;
      const bool store = row < p.B;
      const size_t orow = size_t(it.h) * p.S + size_t(it.i) * p.B + size_t(row);
#pragma unroll
      for (int q = 0; q < C::kHalfO / 32; ++q) {
        uint32_t r[32];
        tmem_ld32(lanes + o_col + q * 32, r);
        tmem_ld_wait(r);
        if (!store) continue;
        const int col = grp * C::kHalfO + q * 32;
        if (p.out_f32) {
          uint4* d4 = reinterpret_cast<uint4*>(static_cast<float*>(p.o) + orow * D + col);
#pragma unroll
          for (int x = 0; x < 8; ++x)
            d4[x] = make_uint4(__float_as_uint(__uint_as_float(r[4 * x]) * inv_l),
                               __float_as_uint(__uint_as_float(r[4 * x + 1]) * inv_l),
                               __float_as_uint(__uint_as_float(r[4 * x + 2]) * inv_l),
                               __float_as_uint(__uint_as_float(r[4 * x + 3]) * inv_l));
        } else {
          uint32_t ob[16];
#pragma unroll
          for (int x = 0; x < 16; ++x)
            ob[x] = pack_bf16x2(__uint_as_float(r[2 * x]) * inv_l,
                                __uint_as_float(r[2 * x + 1]) * inv_l);
          uint4* d4 =
              reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow * D + col);
#pragma unroll
          for (int x = 0; x < 4; ++x)
            d4[x] = make_uint4(ob[4 * x], ob[4 * x + 1], ob[4 * x + 2], ob[4 * x + 3]);
        }
      }
      if (p.lse && store && grp == 0)
        p.lse[orow] = (m_used + log2f(lt)) * 0.6931471805599453f;
      tc_fence_before();
      mbar_arrive(&sh->o_free);
      ++qi;
    }
    if (!ok) raise_abort(sh, p);
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
  constexpr int kSmem = C::kData + int(sizeof(Shared)) + 1024;
  static_assert(kSmem <= 232448, "shared memory budget");
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
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  if (a.num_workers == 0) return cudaSuccess;
  kern<<<a.num_workers, C::kThreads, kSmem, st>>>(tq, tk, tv, p);
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
