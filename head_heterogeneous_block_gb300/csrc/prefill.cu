// Block-sparse causal prefill attention on sm_103a.
//
// One persistent CTA per schedule worker walks that worker's (head,
// query-block) items.  For every item it loads the 128-row query tile once
// and then, for each selected key block j, computes S = Q K_j^T and
// O += softmax(S) V_j with flash-style online softmax.  Twenty warps:
//
//   warp 0      producer: reads the schedule, the block counts and the block
//               lists (32 indices per load), publishes each item's metadata
//               through a small shared-memory ring, and issues TMA loads of
//               the Q tile and the selected K blocks (128-byte-swizzled boxes
//               of the [heads*S, d] view) into a ring of stages.
//   warp 2      producer of the V blocks (its own ring).
//   warp 1      Q K^T issuer: tcgen05.mma kind::f16 (bf16 in, fp32 out), both
//               operands from shared memory, into one of three S buffers in
//               tensor memory; it runs up to three blocks ahead of P V.
//   warp 3      P V issuer: P (bf16, written over its S buffer) is the
//               tensor-memory A operand, V the shared-memory B operand, O
//               accumulates in tensor memory.  The four control warps sit on
//               the four schedulers.
//   warps 4-19  softmax, four column groups of four warps: each thread owns
//               one row of the tile and a quarter of its S columns (and of
//               O's).  The first block of every item is the sink block 0; its
//               row maximum, exchanged once between the four groups, is the
//               reference maximum m of the row for the whole item.  Every
//               block's weights are 2^(s*c - m), so a later block may give
//               weights above 1; m cancels in O / l, so there is no per-block
//               exchange and no rescale of O.  The normaliser sums the same
//               bf16-rounded weights that enter P V.  A row whose normaliser
//               passes 2^126, or whose O is not finite, is marked and, after
//               the worker's last item, recomputed exactly in fp32 on the CUDA
//               cores.  Epilogue (after the next item's first block): O / l
//               and the log-sum-exp; fp32 output is stored directly, bf16
//               output is staged, 128-byte swizzled, in the finished item's Q
//               stage and written by TMA stores.
//
// The work items and their order come from the plan's LPT schedule (S-HPLB,
// "Algoritmo Greedy"), with workers = CTAs instead of GPUs.
// Every index read from idx / cnt / the schedule is range-checked; bad values
// are clamped and flagged in the device status word, never dereferenced.
// Every wait is a bounded mbarrier wait; on a timeout the CTA flags
// SA_DEV_TIMEOUT, lets its copies and MMAs drain, frees its tensor memory and
// exits.

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
  static constexpr int kNQ = 2;                   // Q stages (the next item's loads early)
  static constexpr int kNK = 2;                   // K stages
  static constexpr int kNV = 2;                   // V stages (a V load has ~2 block periods)
  static constexpr int kNS = 3;                   // S buffers in tensor memory
  static constexpr int kGroups = 4;               // softmax column groups
  static constexpr int kCols = BK / kGroups;      // S columns per group
  static constexpr int kOCols = D / kGroups;      // O columns per group
  static constexpr uint32_t kO = kNS * BK;        // TMEM column of O
  static constexpr uint32_t kTmemCols = (kNS * BK + D <= 256) ? 256 : 512;
  static constexpr int kData = kNQ * kQBytes + kNK * kKVBytes + kNV * kKVBytes;
  static_assert(kNS * BK + D <= 512, "tensor memory budget");
  static_assert(kCols == 16 || kCols == 32, "group width");
  static_assert(kOCols == 16 || kOCols == 32, "group width");
};

constexpr int kNI = 4;                 // item-metadata ring slots
constexpr int kSoftmaxWarps = 16;      // warps 4..19
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
// warp 0: producer (items, Q, K); 1: Q.K^T issuer; 2: producer (V);
// 3: P.V issuer -- one per scheduler -- then the softmax warps
constexpr int kThreads = 128 + kSoftmaxThreads;

struct ItemInfo {
  int32_t h, i, n, diag_last;   // n == 0: end of this worker's list
  int32_t pos;                  // position in this worker's list
};

// Items of a worker's list whose rows the exact pass recomputes, one bit per
// list position (lists longer than this report SA_DEV_RANGE instead).
constexpr int kRedoWords = 1024;

struct Shared {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[3], k_empty[3];
  uint64_t v_full[3], v_empty[3];
  uint64_t s_full[3];     // S of block b is in TMEM buffer b % 3
  uint64_t p_full[3];     // P of block b written (every softmax group)
  uint64_t pv_done[3];    // P.V of block b complete (its S buffer may be rewritten)
  uint64_t o_last;        // one phase per item, after its last P.V (epilogue)
  uint64_t o_free;        // one phase per item: every group finished the epilogue
  uint64_t xch_bar;       // exchange between the softmax groups
  uint64_t stage_bar;     // one phase per item: the output tile is staged
  uint64_t store_done;    // the P.V issuer's output stores have all completed
  uint64_t drain_qk, drain_pv;
  uint64_t info_full[kNI], info_empty[kNI];
  ItemInfo info[kNI];
  uint32_t redo[kRedoWords];
  float xch[2][4][128];   // [use parity][group][row]: partial row max per block, or
                          // partial sum per item; use u goes to buffer u & 1
  int32_t stage_row[2];   // first output row of the tile staged in Q stage x
  uint32_t tmem_base;
  int abort;
};

struct Params {
  const __nv_bfloat16* q;   // [Hq*S][D], [Hkv*S][D], [Hkv*S][D]: read only by exact_row
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
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
  uint64_t wait_ns;   // limit of every operational wait; drains keep kWaitLimitNs
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

// A block index as both producers use it: out-of-range entries become block 0.
__device__ __forceinline__ int32_t clamp_block(int32_t j, int32_t i) {
  return (j < 0 || j > i) ? 0 : j;
}

// Exact attention of one query row of item (h, i) over the item's selected
// blocks, for output columns [col0, col0 + NC): two passes in fp32 on the
// CUDA cores, the row's maximum first, then the weights, their sum and the
// weighted values.  It serves only rows whose sum left the range of the
// tensor-core pass (a later block scoring far above the item's first block,
// or values so large that O overflowed), so it favours plainness over speed.
template <int D, int BK, int NC>
__device__ __noinline__ void exact_row(const Params& p, int32_t h, int32_t i, int32_t n,
                                       int row, int col0, bool write_lse) {
  const size_t orow = size_t(h) * p.S + size_t(i) * p.B + size_t(row);
  const __nv_bfloat16* q = p.q + orow * D;
  const size_t kv0 = size_t(h / p.G) * p.S;
  const int32_t* list = p.idx + (size_t(h) * p.nb + i) * size_t(p.kmax);
  const float c = p.scale_log2;
  float m = -INFINITY;
  for (int t = 0; t < n; ++t) {
    const int32_t j = clamp_block(list[t], i);
    const int keys = j == i ? row + 1 : BK;   // causal inside the diagonal block
    for (int u = 0; u < keys; ++u) {
      const __nv_bfloat16* kr = p.k + (kv0 + size_t(j) * BK + u) * D;
      float sc = 0.f;
#pragma unroll 8
      for (int x = 0; x < D; ++x) sc = fmaf(__bfloat162float(q[x]), __bfloat162float(kr[x]), sc);
      m = fmaxf(m, sc * c);
    }
  }
  float l = 0.f, acc[NC];
#pragma unroll
  for (int x = 0; x < NC; ++x) acc[x] = 0.f;
  for (int t = 0; t < n; ++t) {
    const int32_t j = clamp_block(list[t], i);
    const int keys = j == i ? row + 1 : BK;
    for (int u = 0; u < keys; ++u) {
      const size_t key = kv0 + size_t(j) * BK + u;
      const __nv_bfloat16* kr = p.k + key * D;
      float sc = 0.f;
#pragma unroll 8
      for (int x = 0; x < D; ++x) sc = fmaf(__bfloat162float(q[x]), __bfloat162float(kr[x]), sc);
      const float w = ex2(sc * c - m);
      l += w;
      const __nv_bfloat16* vr = p.v + key * D + col0;
#pragma unroll
      for (int x = 0; x < NC; ++x) acc[x] = fmaf(w, __bfloat162float(vr[x]), acc[x]);
    }
  }
  const float inv_l = 1.f / l;
  if (p.out_f32) {
    float* o = static_cast<float*>(p.o) + orow * D + col0;
    for (int x = 0; x < NC; ++x) o[x] = acc[x] * inv_l;
  } else {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o) + orow * D + col0;
    for (int x = 0; x < NC; ++x) o[x] = __float2bfloat16_rn(acc[x] * inv_l);
  }
  if (write_lse && p.lse) p.lse[orow] = (m + log2f(l)) * 0.6931471805599453f;
}

template <int D, int BK>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_attention_kernel(const __grid_constant__ CUtensorMap tq,
                             const __grid_constant__ CUtensorMap tk,
                             const __grid_constant__ CUtensorMap tv,
                             const __grid_constant__ CUtensorMap to, const Params p) {
  using C = Cfg<D, BK>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The data stages need 1024-byte alignment; the launch reserves no slack
  // for it, so a misaligned window is reported instead of used.
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.dev_status, SA_DEV_BAD_LAUNCH);
    return;
  }
  uint8_t* sQ = smem_raw;
  uint8_t* sK = sQ + C::kNQ * C::kQBytes;
  uint8_t* sV = sK + C::kNK * C::kKVBytes;
  Shared* sh = reinterpret_cast<Shared*>(sV + C::kNV * C::kKVBytes);
  volatile int* abort = &sh->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh->q_full[s], 1);
      // the item's last Q.K^T (commit) and its output tile leaving the stage
      mbar_init(&sh->q_empty[s], 2);
    }
    for (int s = 0; s < 3; ++s) {
      mbar_init(&sh->k_full[s], 1);
      mbar_init(&sh->k_empty[s], 1);
      mbar_init(&sh->v_full[s], 1);
      mbar_init(&sh->v_empty[s], 1);
      mbar_init(&sh->s_full[s], 1);
      mbar_init(&sh->p_full[s], kSoftmaxThreads);
      mbar_init(&sh->pv_done[s], 1);
    }
    for (int s = 0; s < kNI; ++s) {
      mbar_init(&sh->info_full[s], 1);
      mbar_init(&sh->info_empty[s], 3 + kSoftmaxWarps);
    }
    mbar_init(&sh->o_last, 1);
    mbar_init(&sh->o_free, kSoftmaxThreads);
    mbar_init(&sh->xch_bar, kSoftmaxThreads);
    mbar_init(&sh->stage_bar, kSoftmaxThreads);
    mbar_init(&sh->store_done, 1);
    mbar_init(&sh->drain_qk, 1);
    mbar_init(&sh->drain_pv, 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  for (int x = threadIdx.x; x < kRedoWords; x += kThreads) sh->redo[x] = 0;
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------- producer: items, Q, K
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
    uint32_t qi = 0, kiss = 0;
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
        // publish the item's metadata for the MMA, V-producer and softmax warps
        const int slot = qi % kNI;
        if (qi >= uint32_t(kNI) &&
            !mbar_wait(&sh->info_empty[slot], ((qi / kNI) - 1) & 1, abort, p.wait_ns))
          ok = false;
        if (ok) {
          sh->info[slot] = ItemInfo{h, i, n, jlast == i ? 1 : 0, pos - begin};
          mbar_arrive(&sh->info_full[slot]);
          const int qs = qi % C::kNQ;
          if (qi >= uint32_t(C::kNQ) &&
              !mbar_wait(&sh->q_empty[qs], ((qi / C::kNQ) - 1) & 1, abort, p.wait_ns))
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
        const int32_t jraw = __shfl_sync(0xffffffffu, jl, t & 31);
        if (jraw < 0 || jraw > i || jraw <= jprev) {   // out of range or not ascending
          if (lane == 0) atomicOr(p.dev_status, SA_DEV_BAD_INDEX);
        }
        const int32_t j = clamp_block(jraw, i);
        jprev = jraw;
        if (lane == 0) {
          const int ks = kiss % C::kNK;
          if (kiss >= uint32_t(C::kNK) &&
              !mbar_wait(&sh->k_empty[ks], ((kiss / C::kNK) - 1) & 1, abort, p.wait_ns))
            ok = false;
          if (ok) {
            mbar_arrive_expect_tx(&sh->k_full[ks], C::kKVBytes);
#pragma unroll
            for (int s = 0; s < C::kPanels; ++s)
              tma_load_2d(sK + ks * C::kKVBytes + s * C::kKVPanel, &tk, &sh->k_full[ks],
                          s * 64, g * p.S + j * BK, pol_kv);
            ++kiss;
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
            !mbar_wait(&sh->info_empty[slot], ((qi / kNI) - 1) & 1, abort, p.wait_ns))
          ok = false;
        if (ok) {
          sh->info[slot] = ItemInfo{0, 0, 0, 0, 0};
          mbar_arrive(&sh->info_full[slot]);
        }
      }
      if (!ok) raise_abort(sh, p);
      // copies still in flight must land before this CTA's shared memory goes
      drain_ring(sh->q_full, qi, C::kNQ);
      drain_ring(sh->k_full, kiss, C::kNK);
    }
  } else if (warp == 2) {
    // ------------------------------------------------- producer: V
    // Runs apart from the K stream so K loads are never held up by V stages,
    // which free two blocks later.
    const uint64_t pol_kv = l2_policy_evict_last();
    uint32_t qi = 0, viss = 0;
    bool ok = true;
    for (;;) {
      const int slot = qi % kNI;
      if (!warp_wait(&sh->info_full[slot], (qi / kNI) & 1, abort, p.wait_ns)) {
        ok = false;
        break;
      }
      const ItemInfo it = sh->info[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->info_empty[slot]);
      if (it.n == 0) break;
      const int32_t* list = p.idx + (size_t(it.h) * p.nb + it.i) * size_t(p.kmax);
      const int g = it.h / p.G;
      int32_t jl = (lane < it.n) ? list[lane] : 0;
      for (int t = 0; t < it.n; ++t) {
        if ((t & 31) == 0 && t > 0) jl = (t + lane < it.n) ? list[t + lane] : 0;
        const int32_t j = clamp_block(__shfl_sync(0xffffffffu, jl, t & 31), it.i);
        if (lane == 0) {
          const int vs = viss % C::kNV;
          if (viss >= uint32_t(C::kNV) &&
              !mbar_wait(&sh->v_empty[vs], ((viss / C::kNV) - 1) & 1, abort, p.wait_ns))
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
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      if (!ok) break;
      ++qi;
    }
    if (lane == 0) {
      if (!ok) raise_abort(sh, p);
      drain_ring(sh->v_full, viss, C::kNV);
    }
  } else if (warp == 1) {
    // ------------------------------------------------- Q.K^T issuer
    // The whole warp runs the loop; one elected lane issues and commits.
    // S buffer b % 3 is reused once P.V of block b-3 has completed.  The
    // barrier phases a step needs are tested together (one non-blocking test
    // per lane, one ballot) and only the missing ones are waited on.
    constexpr uint32_t idesc_qk = idesc_bf16(128, BK, 0, 0);  // Q, K both K-major
    static_assert(C::kNS == 3, "S ring indexing");
    uint32_t qi = 0, kb = 0, stage = 0, phase = 0;   // S ring
    uint32_t kst = 0, kph = 0;                       // K ring
    bool ok = true;
    for (;;) {
      const int slot = qi % kNI;
      if (!warp_wait(&sh->info_full[slot], (qi / kNI) & 1, abort, p.wait_ns)) {
        ok = false;
        break;
      }
      const int n = sh->info[slot].n;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->info_empty[slot]);
      if (n == 0) break;
      const int qs = qi % C::kNQ;
      if (!warp_wait(&sh->q_full[qs], (qi / C::kNQ) & 1, abort, p.wait_ns)) {
        ok = false;
        break;
      }
      const uint64_t qdesc = smem_desc_sw128(smem_u32(sQ + qs * C::kQBytes), 16, 1024);
      for (int t = 0; t < n; ++t) {
        // lane 0: K of this block; lane 1: P.V of block kb-3 (same S buffer)
        const bool reuse = kb >= 3;
        uint64_t* bar = &sh->k_full[kst];
        uint32_t par = kph;
        if (lane == 1 && reuse) {
          bar = &sh->pv_done[stage];
          par = phase ^ 1u;
        }
        const uint32_t have = __ballot_sync(0xffffffffu, mbar_test(bar, par));
        if (!(have & 1u) && !warp_wait(&sh->k_full[kst], kph, abort, p.wait_ns)) {
          ok = false;
          break;
        }
        if (reuse && !(have & 2u) && !warp_wait(&sh->pv_done[stage], phase ^ 1u, abort, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t kdesc = smem_desc_sw128(smem_u32(sK + kst * C::kKVBytes), 16, 1024);
        const uint32_t s_tmem = tmem + stage * BK;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // 16 dims per step: panel kk/4, 32-byte column offset inside the
            // swizzle atom (the hardware applies the XOR on the full address)
            const uint32_t qoff = (kk / 4) * C::kQPanel + (kk % 4) * 32;
            const uint32_t koff = (kk / 4) * C::kKVPanel + (kk % 4) * 32;
            mma_ss(s_tmem, qdesc + uint64_t(qoff >> 4), kdesc + uint64_t(koff >> 4), idesc_qk,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(&sh->s_full[stage]);
          mma_commit(&sh->k_empty[kst]);
          if (t == n - 1) mma_commit(&sh->q_empty[qs]);
        }
        __syncwarp();
        ++kb;
        if (++stage == 3) {
          stage = 0;
          phase ^= 1u;
        }
        if (++kst == C::kNK) {
          kst = 0;
          kph ^= 1u;
        }
      }
      if (!ok) break;
      ++qi;
    }
    if (lane == 0) {
      if (!ok) raise_abort(sh, p);
      // every MMA must be complete before the tensor memory is freed
      mma_commit(&sh->drain_qk);
      mbar_wait(&sh->drain_qk, 0, nullptr);
    }
  } else if (warp == 3) {
    // ------------------------------------------------- P.V issuer
    constexpr uint32_t idesc_pv = idesc_bf16(128, D, 0, 1);   // P (TMEM), V MN-major
    static_assert(C::kNS == 3, "S ring indexing");
    uint32_t qi = 0, stage = 0, phase = 0;   // S / P buffers
    uint32_t vstage = 0, vphase = 0;         // V ring
    bool ok = true;
    // bf16 output: this warp also writes the staged output tiles (one TMA
    // store per 64-column panel) and releases their Q stages, in the time it
    // otherwise spends waiting for P, so no softmax warp waits for a store.
    // Item x is staged after the first block of item x+1, so it is stored
    // before this warp waits for block 1 of item x+1 (or, when that item has
    // one block, for the first block of item x+2), by which time its staging
    // has finished anyway.
    uint32_t spq = 0;                        // next item whose tile is stored
    auto store_upto = [&](uint32_t upto) -> bool {
      for (; spq < upto; ++spq) {
        if (!warp_wait(&sh->stage_bar, spq & 1, abort, p.wait_ns)) return false;
        if (lane == 0) {
          const uint8_t* stg = sQ + (spq % C::kNQ) * C::kQBytes;
          const int32_t r0 = sh->stage_row[spq & 1];
          // evict-first: the output is not read again, and its lines would
          // otherwise push K/V blocks that later items reuse out of L2
#pragma unroll
          for (int s = 0; s < C::kPanels; ++s)
            tma_store_2d_hint(&to, stg + s * C::kQPanel, s * 64, r0, l2_policy_evict_first());
          bulk_commit_group();
          bulk_wait_read_all();
          mbar_arrive(&sh->q_empty[spq % C::kNQ]);
        }
        __syncwarp();
      }
      return true;
    };
    for (;;) {
      const int slot = qi % kNI;
      if (!warp_wait(&sh->info_full[slot], (qi / kNI) & 1, abort, p.wait_ns)) {
        ok = false;
        break;
      }
      const int n = sh->info[slot].n;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->info_empty[slot]);
      if (n == 0) break;
      for (int t = 0; t < n; ++t) {
        const bool first = t == 0;
        if (!p.out_f32 && !store_upto(first ? (qi > 0 ? qi - 1 : 0) : qi)) {
          ok = false;
          break;
        }
        const bool need_o = first && qi > 0;   // previous item's epilogue must read O first
        // lane 0: P, lane 1: V, lane 2: O
        uint64_t* bar = &sh->p_full[stage];
        uint32_t par = phase;
        if (lane == 1) {
          bar = &sh->v_full[vstage];
          par = vphase;
        }
        if (lane == 2 && need_o) {
          bar = &sh->o_free;
          par = (qi - 1) & 1;
        }
        const uint32_t have = __ballot_sync(0xffffffffu, mbar_test(bar, par));
        if (!(have & 1u) && !warp_wait(&sh->p_full[stage], phase, abort, p.wait_ns)) {
          ok = false;
          break;
        }
        if (!(have & 2u) && !warp_wait(&sh->v_full[vstage], vphase, abort, p.wait_ns)) {
          ok = false;
          break;
        }
        if (need_o && !(have & 4u) && !warp_wait(&sh->o_free, (qi - 1) & 1, abort, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // 16 keys per step: 16 rows of 128 bytes in every d panel
        const uint64_t vdesc =
            smem_desc_sw128(smem_u32(sV + vstage * C::kKVBytes), C::kKVPanel, 1024);
        const uint32_t s_col = tmem + stage * BK;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // keys [16kk, 16kk+16) belong to group 16kk / kCols, whose P starts
            // at that group's first S column
            constexpr int kW = C::kCols;
            const int grp = (kk * 16) / kW;
            const uint32_t a_col = s_col + grp * kW + (kk * 16 - grp * kW) / 2;
            mma_ts(tmem + C::kO, a_col, vdesc + uint64_t((kk * 16 * 128) >> 4), idesc_pv,
                   (first && kk == 0) ? 0u : 1u);
          }
          mma_commit(&sh->v_empty[vstage]);
          mma_commit(&sh->pv_done[stage]);
          if (t == n - 1) mma_commit(&sh->o_last);
        }
        __syncwarp();
        if (++stage == 3) {
          stage = 0;
          phase ^= 1u;
        }
        if (++vstage == C::kNV) {
          vstage = 0;
          vphase ^= 1u;
        }
      }
      if (!ok) break;
      ++qi;
    }
    // the last items' tiles (the final one is staged after the list)
    if (ok && !p.out_f32) ok = store_upto(qi);
    if (lane == 0) {
      if (!ok) raise_abort(sh, p);
      // the stores complete before the exact pass may rewrite rows and
      // before the CTA's shared memory goes
      bulk_wait_all();
      mbar_arrive(&sh->store_done);
      mma_commit(&sh->drain_pv);
      mbar_wait(&sh->drain_pv, 0, nullptr);
    }
  } else {
    // ------------------------------------------------- softmax groups
    const int grp = (warp - 4) >> 2;              // column group 0..3
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;          // query row within the tile
    const uint32_t lanes = tmem + (uint32_t(quarter * 32) << 16);
    const float c = p.scale_log2;
    const uint32_t o_col = C::kO + grp * C::kOCols;
    uint32_t kb = 0, qi = 0, xn = 0;   // xn: uses of the exchange buffer so far
    uint32_t sst = 0, sph = 0;         // S ring stage and phase of block kb
    bool ok = true;
    // The epilogue of an item (O / l out to memory, O released) runs after the
    // next item's first block: by then that item's last P.V has finished, so
    // the wait on it costs nothing, and the next item's first P.V waits for
    // the release as before.  The last item's epilogue runs after the loop.
    bool pend = false;
    ItemInfo pit{};
    float pl = 0.f, pm = 0.f;
    uint32_t pq = 0;
    auto epilogue = [&]() -> bool {
      // exchange the partial sums (the same double buffer), then O / l for
      // this group's columns.  O is read and released before the sums are
      // collected, so the next item's first P.V does not wait for the
      // exchange.  o_last has exactly one phase per item, waited on every time.
      float* xb = &sh->xch[xn & 1][0][0];
      xb[grp * 128 + row] = pl;
      mbar_arrive(&sh->xch_bar);
      if (!wait_all(&sh->o_last, pq & 1, abort, p.wait_ns)) return false;
      tc_fence_after();
      uint32_t r[C::kOCols];
      if constexpr (C::kOCols == 32) {
        tmem_ld32(lanes + o_col, r);
        tmem_ld_wait(r);
      } else {
        tmem_ld16(lanes + o_col, r);
        tmem_ld_wait(r);
      }
      // O is in registers: the next item's first P.V may overwrite it
      tc_fence_before();
      mbar_arrive(&sh->o_free);
      if (!wait_all(&sh->xch_bar, xn & 1, abort, p.wait_ns)) return false;
      ++xn;
      const float lt = (xb[row] + xb[128 + row]) + (xb[256 + row] + xb[384 + row]);
      const float inv_l = 1.f / lt;
      const bool store = row < p.B;
      const size_t orow = size_t(pit.h) * p.S + size_t(pit.i) * p.B + size_t(row);
      const int col = grp * C::kOCols;
      // the range the tensor-core pass keeps: the sum below 2^126 (so
      // neither P nor l overflows) and O finite; beyond it the row's
      // columns are recomputed exactly
      float osum = 0.f;
#pragma unroll
      for (int x = 0; x < C::kOCols; ++x) osum += __uint_as_float(r[x]);
      const bool in_range = lt <= 0x1p126f && fabsf(osum) <= 3.0e38f;
      if (store && !in_range) {
        // the whole item is recomputed after the list (the bit is set by
        // every thread that finds a row out of range; one is enough)
        if (pit.pos < 32 * kRedoWords)
          atomicOr(&sh->redo[pit.pos >> 5], 1u << (pit.pos & 31));
        else
          atomicOr(p.dev_status, SA_DEV_RANGE);
      }
      if (store && in_range && p.lse && grp == 0)
        p.lse[orow] = (pm + log2f(lt)) * 0.6931471805599453f;
      if (p.out_f32) {
        if (store && in_range) {
          uint4* d4 = reinterpret_cast<uint4*>(static_cast<float*>(p.o) + orow * D + col);
#pragma unroll
          for (int x = 0; x < C::kOCols / 4; ++x)
            d4[x] = make_uint4(__float_as_uint(__uint_as_float(r[4 * x]) * inv_l),
                               __float_as_uint(__uint_as_float(r[4 * x + 1]) * inv_l),
                               __float_as_uint(__uint_as_float(r[4 * x + 2]) * inv_l),
                               __float_as_uint(__uint_as_float(r[4 * x + 3]) * inv_l));
        }
        // the item's Q stage needs no staging: release it at once
        if (warp == 4 && lane == 0) mbar_arrive(&sh->q_empty[pq % C::kNQ]);
        return true;
      }
      // bf16: the tile is staged in the finished item's Q stage (its last
      // Q.K^T is complete, and the producer reloads it only after the store
      // below has read it), laid out as the 128-byte-swizzled boxes a TMA
      // store reads, then written with one store per 64-column panel: rows
      // reach memory whole instead of as 32 scattered pieces per warp store
      uint8_t* stg = sQ + (pq % C::kNQ) * C::kQBytes;
      if (store) {
        uint32_t ob[C::kOCols / 2];
#pragma unroll
        for (int x = 0; x < C::kOCols / 2; ++x)
          ob[x] = in_range ? pack_bf16x2(__uint_as_float(r[2 * x]) * inv_l,
                                         __uint_as_float(r[2 * x + 1]) * inv_l)
                           : 0u;   // rewritten by the exact pass
#pragma unroll
        for (int x = 0; x < C::kOCols / 8; ++x) {
          const int c16 = (col + 8 * x) / 8;           // 16-byte chunk of the row
          const int panel = c16 / 8, chunk = c16 % 8;
          uint4* dst = reinterpret_cast<uint4*>(stg + panel * C::kQPanel + row * 128 +
                                                ((chunk ^ (row & 7)) << 4));
          *dst = make_uint4(ob[4 * x], ob[4 * x + 1], ob[4 * x + 2], ob[4 * x + 3]);
        }
      }
      fence_proxy_async_smem();
      if (warp == 4 && lane == 0) sh->stage_row[pq & 1] = pit.h * p.S + pit.i * p.B;
      // the P.V issuer stores the tile once every thread has staged its part
      mbar_arrive(&sh->stage_bar);
      return true;
    };
    for (;;) {
      const int slot = qi % kNI;
      if (!wait_all(&sh->info_full[slot], (qi / kNI) & 1, abort, p.wait_ns)) {
        ok = false;
        break;
      }
      const ItemInfo it = sh->info[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->info_empty[slot]);
      if (it.n == 0) break;
      float m_used = -INFINITY;
      // the item's normaliser, in four partial sums combined at its end
      float sum0 = 0.f, sum1 = 0.f, sum2 = 0.f, sum3 = 0.f;
      for (int t = 0; t < it.n; ++t) {
        const int sb = int(sst);
        if (!wait_all(&sh->s_full[sb], sph, abort, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t scol = sb * BK + grp * C::kCols;
        float s[C::kCols];
        if constexpr (C::kCols == 32) {
          uint32_t sr[32];
          tmem_ld32(lanes + scol, sr);
          tmem_ld_wait(sr);
#pragma unroll
          for (int x = 0; x < 32; ++x) s[x] = __uint_as_float(sr[x]);
        } else {
          uint32_t sr[16];
          tmem_ld16(lanes + scol, sr);
          tmem_ld_wait(sr);
#pragma unroll
          for (int x = 0; x < 16; ++x) s[x] = __uint_as_float(sr[x]);
        }
        if (it.diag_last && t == it.n - 1) {
          // key column grp*kCols + x is visible to row `row` when <= row
#pragma unroll
          for (int x = 0; x < C::kCols; ++x)
            if (grp * C::kCols + x > row) s[x] = -INFINITY;
        }
        if (t == 0) {
          // first block of the item: its row maximum, exchanged between the
          // groups, is the reference every block of the item uses.  Use xn
          // writes buffer xn & 1: every thread read use xn-2 before it posted
          // use xn-1, and this thread saw use xn-1 complete, so that buffer
          // is free.
          float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
          for (int x = 4; x + 8 <= C::kCols; x += 8)
#pragma unroll
            for (int a = 0; a < 4; ++a) mx[a] = max3(mx[a], s[x + a], s[x + 4 + a]);
#pragma unroll
          for (int a = 0; a < 4; ++a) mx[a] = fmaxf(mx[a], s[C::kCols - 4 + a]);
          float* xb = &sh->xch[xn & 1][0][0];
          xb[grp * 128 + row] = fmaxf(max3(mx[0], mx[1], mx[2]), mx[3]);
          mbar_arrive(&sh->xch_bar);
          if (!wait_all(&sh->xch_bar, xn & 1, abort, p.wait_ns)) {
            ok = false;
            break;
          }
          m_used = max3(fmaxf(xb[row], xb[128 + row]), xb[256 + row], xb[384 + row]) * c;
          ++xn;
        }
        // P = 2^(s*c - m) in bf16 with the item's reference maximum m_used,
        // written over this group's S columns.  Later blocks may score above
        // it: their weights exceed 1 but stay exact in bf16 and fp32, the
        // reference cancels in O / l, and no group has to wait for another.
        // A row whose sum leaves the range checked at the end of the item is
        // recomputed exactly.
        {
          uint32_t pk[C::kCols / 2];
          const float nm = -m_used;
#pragma unroll
          for (int x = 0; x < C::kCols / 2; ++x) {
            float a0, a1;
            fma2(a0, a1, s[2 * x], s[2 * x + 1], c, c, nm, nm);
            pk[x] = pack_bf16x2(ex2(a0), ex2(a1));
            // the normaliser sums the rounded values
            if (x & 1)
              add_bf16x2(sum2, sum3, pk[x]);
            else
              add_bf16x2(sum0, sum1, pk[x]);
          }
          if constexpr (C::kCols == 32) {
            tmem_st16(lanes + scol, pk);
          } else {
            tmem_st8(lanes + scol, pk);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sh->p_full[sb]);
        ++kb;
        if (++sst == uint32_t(C::kNS)) {
          sst = 0;
          sph ^= 1u;
        }
        if (t == 0 && pend) {
          if (!epilogue()) {
            ok = false;
            break;
          }
          pend = false;
        }
      }
      if (!ok) break;
      pend = true;
      pit = it;
      pl = (sum0 + sum1) + (sum2 + sum3);
      pm = m_used;
      pq = qi;
      ++qi;
    }
    if (ok && pend) ok = epilogue();
    if (!ok) raise_abort(sh, p);
    // the output tiles' stores complete before any exact rewrite
    if (!p.out_f32 && !wait_all(&sh->store_done, 0, nullptr)) ok = false;
    // every epilogue of the list has set its bits: recompute the marked items,
    // one (row, column group) per thread
    asm volatile("bar.sync 1, %0;" ::"r"(kSoftmaxThreads) : "memory");
    if (ok && row < p.B) {
      const int32_t begin = p.wptr[blockIdx.x];
      for (int w = 0; w < kRedoWords; ++w) {
        uint32_t bits = sh->redo[w];
        while (bits) {
          const int32_t pos = begin + 32 * w + __ffs(bits) - 1;
          bits &= bits - 1;
          const int32_t item = p.items[pos];
          const int32_t h = item / p.nb, i = item - h * p.nb;
          const int32_t n = max(1, min(p.cnt[item], min(p.kmax, i + 1)));
          exact_row<D, BK, C::kOCols>(p, h, i, n, row, grp * C::kOCols, grp == 0);
        }
      }
    }
    // a role that gave up may have left a tensor-memory access in flight; all
    // of them end before the allocation is freed below
    tmem_ld_wait();
    tmem_st_wait();
    tc_fence_before();
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
  // data stages + the small shared block; the kernel checks the alignment
  constexpr int kSmem = C::kData + int(sizeof(Shared));
  static_assert(kSmem <= 232448, "shared memory budget");
  CUtensorMap tq, tk, tv, to;
  // the bf16 output is written by TMA in boxes of one query block; fp32 output
  // is stored directly (the map is then unused)
  if (!make_map(&tq, a.q, uint64_t(a.Hq) * a.S, D, C::kM) ||
      !make_map(&tk, a.k, uint64_t(a.Hkv) * a.S, D, BK) ||
      !make_map(&tv, a.v, uint64_t(a.Hkv) * a.S, D, BK) ||
      !make_map(&to, a.out_f32 ? a.q : a.o, uint64_t(a.Hq) * a.S, D, a.B)) {
    *encode_failed = true;
    return cudaErrorInvalidValue;
  }
  Params p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k);
  p.v = static_cast<const __nv_bfloat16*>(a.v);
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
  p.wait_ns = a.wait_ns ? a.wait_ns : kWaitLimitNs;
  auto kern = prefill_attention_kernel<D, BK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  if (a.num_workers == 0) return cudaSuccess;
  kern<<<a.num_workers, kThreads, kSmem, st>>>(tq, tk, tv, to, p);
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
