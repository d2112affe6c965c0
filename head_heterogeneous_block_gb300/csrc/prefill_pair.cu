// Block-sparse causal prefill attention for group-shared block lists: one K/V
// tile feeds two query heads.
//
// With one block list per KV group, the two heads of a head pair (2p, 2p+1)
// at query block i attend the same key blocks (Fluxion models access at the
// level of the GQA group: "Riepilogo Tecnico: Fluxion", "Componenti di
// Sistema").  A persistent CTA walks its worker's pair items (p, i); for each
// selected key block it loads K and V once and runs both heads' query tiles
// against them:
//
//   S_A = Q_A K^T,  S_B = Q_B K^T,  O_A += P_A V,  O_B += P_B V,
//
// with S_A, S_B, O_A and O_B filling the 512 tensor-memory columns.  The
// softmax warps take the tiles in turn (A of block j, B of block j, A of
// block j+1, ...), so while they work on one tile the tensor cores compute
// the other's products.  Twenty warps, as in the per-head kernel:
//
//   warp 0      producer: schedule, counts and block lists; both heads' Q
//               tiles per item (two item stages, so the next item's load early)
//               and the K blocks, once per block for both heads.
//   warp 1      Q K^T issuer: per block, S_A then S_B (tcgen05.mma kind::f16,
//               operands in shared memory); a tile's S buffer is rewritten once
//               P V of that tile's previous block has completed.
//   warp 2      producer of the V blocks.
//   warp 3      P V issuer: O_A += P_A V, then O_B += P_B V, P from tensor
//               memory over its S buffer.
//   warps 4-19  softmax, four column groups of four warps, each thread one
//               row and a quarter of the columns of the tile in hand.  Each
//               tile's first block of an item sets that tile's reference row
//               maximum (exchanged once between the groups); later blocks use
//               it as is: weights above 1 stay exact and the reference cancels
//               in O / l.  A row whose sum leaves the range (2^126, or O not
//               finite) is recomputed exactly after the list.  Epilogue: O / l
//               for both heads, in fp32 by direct stores or in bf16 through
//               the finished item's Q stages and a TMA store.
//
// Work items and their order come from the plan's LPT schedule over head
// pairs (S-HPLB, "Algoritmo Greedy", workers = CTAs).  Every index read from
// idx / cnt / the schedule is range-checked; bad values are clamped and
// flagged, never dereferenced.  Every wait is bounded; on a timeout the CTA
// flags SA_DEV_TIMEOUT, drains its copies and MMAs, frees its tensor memory
// and exits.

#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "sparse_attn.h"

namespace {

using namespace sa_dev;

template <int D, int BK>
struct PCfg {
  static constexpr int kM = 128;                  // query rows per tile
  static constexpr int kPanels = D / 64;          // 128-byte column panels
  static constexpr int kQPanel = kM * 128;        // bytes of one Q panel
  static constexpr int kKVPanel = BK * 128;       // bytes of one K/V panel
  static constexpr int kQBytes = kM * D * 2;      // one head's Q tile
  static constexpr int kKVBytes = BK * D * 2;
  static constexpr int kNQ = 2;                   // item stages, each both heads' Q
  static constexpr int kNK = 2;                   // K stages
  static constexpr int kNV = 1;                   // V stages
  static constexpr int kGroups = 4;               // softmax column groups
  static constexpr int kCols = BK / kGroups;      // S columns per group
  static constexpr int kOCols = D / kGroups;      // O columns per group
  static constexpr uint32_t kO = 2 * BK;          // TMEM column of O_A (O_B follows)
  static constexpr uint32_t kTmemCols = (2 * BK + 2 * D <= 256) ? 256 : 512;
  static constexpr int kData = 2 * kNQ * kQBytes + (kNK + kNV) * kKVBytes;
  static_assert(2 * BK + 2 * D <= 512, "tensor memory budget");
  static_assert(kCols == 16 || kCols == 32, "group width");
  static_assert(kOCols == 16 || kOCols == 32, "group width");
};

constexpr int kNI = 4;                 // item-metadata ring slots
constexpr int kSoftmaxWarps = 16;      // warps 4..19
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kThreads = 128 + kSoftmaxThreads;
// Pair items of a worker's list whose rows the exact pass recomputes, one bit
// per list position (longer lists report SA_DEV_RANGE instead).
constexpr int kRedoWords = 64;

struct PairInfo {
  int32_t p, i, n, diag_last;   // n == 0: end of this worker's list
  int32_t pos;                  // position in this worker's list
};

struct Shared {
  uint64_t q_full[2], q_empty[2];   // per item stage: both heads' Q tiles
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full[1], v_empty[1];
  uint64_t s_full[2];     // per tile: its S is ready
  uint64_t p_full[2];     // per tile: every softmax thread wrote its P
  uint64_t pv_done[2];    // per tile: its P.V is complete (its S may be rewritten)
  uint64_t o_last;        // one phase per item: both tiles' last P.V complete
  uint64_t o_free;        // one phase per item: the epilogue read O_A and O_B
  uint64_t xch_bar;       // one phase per exchange: every group posted
  uint64_t xch_free;      // one phase per exchange: every group read
  uint64_t stage_bar;     // one phase per item: both output tiles staged
  uint64_t drain_qk, drain_pv;
  uint64_t info_full[kNI], info_empty[kNI];
  PairInfo info[kNI];
  uint32_t redo[kRedoWords];
  float xch[4][128];      // [group][row]: a partial row maximum or sum
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
  const int32_t* items;     // pair items p*nb + i
  int32_t kmax, num_items, num_workers, nb, S, B, G;
  float scale_log2;
  void* o;
  int32_t out_f32;
  float* lse;
  int32_t* dev_status;
  uint64_t wait_ns;
};

__device__ __forceinline__ void raise_abort(Shared* sh, const Params& p) {
  atomicOr(p.dev_status, SA_DEV_TIMEOUT);
  *(volatile int*)&sh->abort = 1;
}

__device__ __forceinline__ void drain_ring(uint64_t* full, uint32_t issued, int stages) {
  const uint32_t first = issued > uint32_t(stages) ? issued - stages : 0;
  for (uint32_t x = first; x < issued; ++x)
    mbar_wait(&full[x % stages], (x / stages) & 1, nullptr);
}

__device__ __forceinline__ int32_t clamp_block(int32_t j, int32_t i) {
  return (j < 0 || j > i) ? 0 : j;
}

// Exact attention of one query row of item (h, i) over the item's selected
// blocks for output columns [col0, col0 + NC): two fp32 passes on the CUDA
// cores (the row maximum, then weights, their sum and the weighted values),
// for rows the tensor-core pass could not keep in range.
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
    const int keys = j == i ? row + 1 : BK;
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
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tq,
                        const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv,
                        const __grid_constant__ CUtensorMap to, const Params p) {
  using C = PCfg<D, BK>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.dev_status, SA_DEV_BAD_LAUNCH);
    return;
  }
  // Q stage of (item stage s, tile x): sQ + (2 s + x) * kQBytes
  uint8_t* sQ = smem_raw;
  uint8_t* sK = sQ + 2 * C::kNQ * C::kQBytes;
  uint8_t* sV = sK + C::kNK * C::kKVBytes;
  Shared* sh = reinterpret_cast<Shared*>(sV + C::kNV * C::kKVBytes);
  volatile int* abort = &sh->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh->q_full[s], 1);
      mbar_init(&sh->q_empty[s], 2);   // the item's last Q.K^T, its output leaving the stage
      mbar_init(&sh->k_full[s], 1);
      mbar_init(&sh->k_empty[s], 1);
      mbar_init(&sh->s_full[s], 1);
      mbar_init(&sh->p_full[s], kSoftmaxThreads);
      mbar_init(&sh->pv_done[s], 1);
    }
    mbar_init(&sh->v_full[0], 1);
    mbar_init(&sh->v_empty[0], 1);
    for (int s = 0; s < kNI; ++s) {
      mbar_init(&sh->info_full[s], 1);
      mbar_init(&sh->info_empty[s], 3 + kSoftmaxWarps);
    }
    mbar_init(&sh->o_last, 1);
    mbar_init(&sh->o_free, kSoftmaxThreads);
    mbar_init(&sh->xch_bar, kSoftmaxThreads);
    mbar_init(&sh->xch_free, kSoftmaxThreads);
    mbar_init(&sh->stage_bar, kSoftmaxThreads);
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
    int32_t item_next = (begin < end) ? p.items[begin] : -1;
    for (int pos = begin; pos < end && ok; ++pos) {
      const int32_t item = item_next;
      if (pos + 1 < end) item_next = p.items[pos + 1];
      if (item < 0 || item >= p.num_items) {
        if (lane == 0) atomicOr(p.dev_status, SA_DEV_BAD_ITEM);
        continue;
      }
      const int32_t pr = item / p.nb, i = item - pr * p.nb;
      const int32_t h0 = 2 * pr;                 // the pair's heads: h0, h0 + 1
      const int32_t row_id = h0 * p.nb + i;      // both heads hold the same list
      const int32_t lim = min(p.kmax, i + 1);
      int32_t n = p.cnt[row_id];
      if (n < 1 || n > lim) {
        if (lane == 0) atomicOr(p.dev_status, SA_DEV_BAD_COUNT);
        n = max(1, min(n, lim));
      }
      const int32_t* list = p.idx + size_t(row_id) * size_t(p.kmax);
      int32_t jl = (lane < n) ? list[lane] : 0;
      const int32_t jlast = list[n - 1];
      const int g = h0 / p.G;
      if (lane == 0) {
        const int slot = qi % kNI;
        if (qi >= uint32_t(kNI) &&
            !mbar_wait(&sh->info_empty[slot], ((qi / kNI) - 1) & 1, abort, p.wait_ns))
          ok = false;
        if (ok) {
          sh->info[slot] = PairInfo{pr, i, n, jlast == i ? 1 : 0, pos - begin};
          mbar_arrive(&sh->info_full[slot]);
          const int qs = qi % C::kNQ;
          if (qi >= uint32_t(C::kNQ) &&
              !mbar_wait(&sh->q_empty[qs], ((qi / C::kNQ) - 1) & 1, abort, p.wait_ns))
            ok = false;
          if (ok) {
            mbar_arrive_expect_tx(&sh->q_full[qs], 2 * C::kQBytes);
#pragma unroll
            for (int x = 0; x < 2; ++x)
#pragma unroll
              for (int s = 0; s < C::kPanels; ++s)
                tma_load_2d(sQ + (2 * qs + x) * C::kQBytes + s * C::kQPanel, &tq,
                            &sh->q_full[qs], s * 64, (h0 + x) * p.S + i * p.B, pol_q);
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
        if (jraw < 0 || jraw > i || jraw <= jprev) {
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
        const int slot = qi % kNI;
        if (qi >= uint32_t(kNI) &&
            !mbar_wait(&sh->info_empty[slot], ((qi / kNI) - 1) & 1, abort, p.wait_ns))
          ok = false;
        if (ok) {
          sh->info[slot] = PairInfo{0, 0, 0, 0, 0};
          mbar_arrive(&sh->info_full[slot]);
        }
      }
      if (!ok) raise_abort(sh, p);
      drain_ring(sh->q_full, qi, C::kNQ);
      drain_ring(sh->k_full, kiss, C::kNK);
    }
  } else if (warp == 2) {
    // ------------------------------------------------- producer: V
    const uint64_t pol_kv = l2_policy_evict_last();
    uint32_t qi = 0, viss = 0;
    bool ok = true;
    for (;;) {
      const int slot = qi % kNI;
      if (!warp_wait(&sh->info_full[slot], (qi / kNI) & 1, abort, p.wait_ns)) {
        ok = false;
        break;
      }
      const PairInfo it = sh->info[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->info_empty[slot]);
      if (it.n == 0) break;
      const int32_t h0 = 2 * it.p;
      const int32_t* list = p.idx + (size_t(h0) * p.nb + it.i) * size_t(p.kmax);
      const int g = h0 / p.G;
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
    constexpr uint32_t idesc_qk = idesc_bf16(128, BK, 0, 0);  // Q, K both K-major
    uint32_t qi = 0, kst = 0, kph = 0;
    uint32_t nq[2] = {0, 0};   // Q.K^T issued per tile (registers: indexed by constants)
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
      for (int t = 0; t < n && ok; ++t) {
        if (!warp_wait(&sh->k_full[kst], kph, abort, p.wait_ns)) {
          ok = false;
          break;
        }
        const uint64_t kdesc = smem_desc_sw128(smem_u32(sK + kst * C::kKVBytes), 16, 1024);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          // S_x is rewritten once P.V of tile x's previous block has completed
          if (nq[x] >= 1 && !warp_wait(&sh->pv_done[x], (nq[x] - 1) & 1, abort, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t qdesc =
              smem_desc_sw128(smem_u32(sQ + (2 * qs + x) * C::kQBytes), 16, 1024);
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t qoff = (kk / 4) * C::kQPanel + (kk % 4) * 32;
              const uint32_t koff = (kk / 4) * C::kKVPanel + (kk % 4) * 32;
              mma_ss(tmem + x * BK, qdesc + uint64_t(qoff >> 4), kdesc + uint64_t(koff >> 4),
                     idesc_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit(&sh->s_full[x]);
            if (x == 1) {
              mma_commit(&sh->k_empty[kst]);
              if (t == n - 1) mma_commit(&sh->q_empty[qs]);
            }
          }
          __syncwarp();
          ++nq[x];
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
      mma_commit(&sh->drain_qk);
      mbar_wait(&sh->drain_qk, 0, nullptr);
    }
  } else if (warp == 3) {
    // ------------------------------------------------- P.V issuer
    constexpr uint32_t idesc_pv = idesc_bf16(128, D, 0, 1);   // P (TMEM), V MN-major
    uint32_t qi = 0, vst = 0, vph = 0;
    uint32_t np[2] = {0, 0};   // P.V issued per tile
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
      for (int t = 0; t < n && ok; ++t) {
        if (!warp_wait(&sh->v_full[vst], vph, abort, p.wait_ns)) {
          ok = false;
          break;
        }
        const uint64_t vdesc =
            smem_desc_sw128(smem_u32(sV + vst * C::kKVBytes), C::kKVPanel, 1024);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!warp_wait(&sh->p_full[x], np[x] & 1, abort, p.wait_ns) ||
              (t == 0 && x == 0 && qi > 0 &&
               !warp_wait(&sh->o_free, (qi - 1) & 1, abort, p.wait_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t s_col = tmem + x * BK;
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              constexpr int kW = C::kCols;
              const int grp = (kk * 16) / kW;
              const uint32_t a_col = s_col + grp * kW + (kk * 16 - grp * kW) / 2;
              mma_ts(tmem + C::kO + x * D, a_col, vdesc + uint64_t((kk * 16 * 128) >> 4),
                     idesc_pv, (t == 0 && kk == 0) ? 0u : 1u);
            }
            mma_commit(&sh->pv_done[x]);
            if (x == 1) {
              mma_commit(&sh->v_empty[vst]);
              if (t == n - 1) mma_commit(&sh->o_last);
            }
          }
          __syncwarp();
          ++np[x];
        }
        if (++vst == C::kNV) {
          vst = 0;
          vph ^= 1u;
        }
      }
      if (!ok) break;
      ++qi;
    }
    if (lane == 0) {
      if (!ok) raise_abort(sh, p);
      mma_commit(&sh->drain_pv);
      mbar_wait(&sh->drain_pv, 0, nullptr);
    }
  } else {
    // ------------------------------------------------- softmax groups
    const int grp = (warp - 4) >> 2;              // column group 0..3
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;          // query row within the tiles
    const uint32_t lanes = tmem + (uint32_t(quarter * 32) << 16);
    const float c = p.scale_log2;
    uint32_t qi = 0, xn = 0;                      // xn: exchanges so far
    uint32_t ns[2] = {0, 0};                      // blocks per tile so far
    bool ok = true;
    // One exchange between the four column groups of a row: post v, collect
    // the four posts.  The array has one buffer: a use waits until every
    // group read the previous one.
    auto exchange = [&](float v, float (&out)[4]) -> bool {
      if (xn > 0 && !wait_all(&sh->xch_free, (xn - 1) & 1, abort, p.wait_ns)) return false;
      sh->xch[grp][row] = v;
      mbar_arrive(&sh->xch_bar);
      if (!wait_all(&sh->xch_bar, xn & 1, abort, p.wait_ns)) return false;
#pragma unroll
      for (int x = 0; x < 4; ++x) out[x] = sh->xch[x][row];
      mbar_arrive(&sh->xch_free);
      ++xn;
      return true;
    };
    bool pend = false;
    PairInfo pit{};
    float pl[2] = {0.f, 0.f}, pm[2] = {0.f, 0.f};
    uint32_t pq = 0;
    auto epilogue = [&]() -> bool {
      float lt[2];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        float part[4];
        if (!exchange(pl[x], part)) return false;
        lt[x] = (part[0] + part[1]) + (part[2] + part[3]);
      }
      if (!wait_all(&sh->o_last, pq & 1, abort, p.wait_ns)) return false;
      tc_fence_after();
      const bool store = row < p.B;
      const int col = grp * C::kOCols;
      const int qs = pq % C::kNQ;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        uint32_t r[C::kOCols];
        if constexpr (C::kOCols == 32) {
          tmem_ld32(lanes + C::kO + x * D + grp * C::kOCols, r);
        } else {
          tmem_ld16(lanes + C::kO + x * D + grp * C::kOCols, r);
        }
        tmem_ld_wait(r);
        if (x == 1) {
          // both O tiles read: the next item's first P.V may overwrite them
          tc_fence_before();
          mbar_arrive(&sh->o_free);
        }
        const int32_t h = 2 * pit.p + x;
        const size_t orow = size_t(h) * p.S + size_t(pit.i) * p.B + size_t(row);
        const float inv_l = 1.f / lt[x];
        float osum = 0.f;
#pragma unroll
        for (int e = 0; e < C::kOCols; ++e) osum += __uint_as_float(r[e]);
        const bool in_range = lt[x] <= 0x1p126f && fabsf(osum) <= 3.0e38f;
        if (store && !in_range) {
          if (pit.pos < 32 * kRedoWords)
            atomicOr(&sh->redo[pit.pos >> 5], 1u << (pit.pos & 31));
          else
            atomicOr(p.dev_status, SA_DEV_RANGE);
        }
        if (store && in_range && p.lse && grp == 0)
          p.lse[orow] = (pm[x] + log2f(lt[x])) * 0.6931471805599453f;
        if (p.out_f32) {
          if (store && in_range) {
            uint4* d4 = reinterpret_cast<uint4*>(static_cast<float*>(p.o) + orow * D + col);
#pragma unroll
            for (int e = 0; e < C::kOCols / 4; ++e)
              d4[e] = make_uint4(__float_as_uint(__uint_as_float(r[4 * e]) * inv_l),
                                 __float_as_uint(__uint_as_float(r[4 * e + 1]) * inv_l),
                                 __float_as_uint(__uint_as_float(r[4 * e + 2]) * inv_l),
                                 __float_as_uint(__uint_as_float(r[4 * e + 3]) * inv_l));
          }
        } else if (store) {
          // bf16: staged in the finished item's Q stage of this head,
          // 128-byte swizzled as the TMA store reads it
          uint8_t* stg = sQ + (2 * qs + x) * C::kQBytes;
          uint32_t ob[C::kOCols / 2];
#pragma unroll
          for (int e = 0; e < C::kOCols / 2; ++e)
            ob[e] = in_range ? pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l,
                                           __uint_as_float(r[2 * e + 1]) * inv_l)
                             : 0u;   // rewritten by the exact pass
#pragma unroll
          for (int e = 0; e < C::kOCols / 8; ++e) {
            const int c16 = (col + 8 * e) / 8;
            const int panel = c16 / 8, chunk = c16 % 8;
            uint4* dst = reinterpret_cast<uint4*>(stg + panel * C::kQPanel + row * 128 +
                                                  ((chunk ^ (row & 7)) << 4));
            *dst = make_uint4(ob[4 * e], ob[4 * e + 1], ob[4 * e + 2], ob[4 * e + 3]);
          }
        }
      }
      if (p.out_f32) {
        if (warp == 4 && lane == 0) mbar_arrive(&sh->q_empty[qs]);
        return true;
      }
      fence_proxy_async_smem();
      mbar_arrive(&sh->stage_bar);
      bool sent = true;
      if (warp == 4 && lane == 0) {
        sent = mbar_wait(&sh->stage_bar, pq & 1, abort, p.wait_ns);
        if (sent) {
#pragma unroll
          for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int s = 0; s < C::kPanels; ++s)
              tma_store_2d_hint(&to, sQ + (2 * qs + x) * C::kQBytes + s * C::kQPanel, s * 64,
                                (2 * pit.p + x) * p.S + pit.i * p.B, l2_policy_evict_first());
          bulk_commit_group();
          bulk_wait_read_all();
          mbar_arrive(&sh->q_empty[qs]);
        }
      }
      return __all_sync(0xffffffffu, sent);
    };
    for (;;) {
      const int slot = qi % kNI;
      if (!wait_all(&sh->info_full[slot], (qi / kNI) & 1, abort, p.wait_ns)) {
        ok = false;
        break;
      }
      const PairInfo it = sh->info[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->info_empty[slot]);
      if (it.n == 0) break;
      float m_used[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
      for (int t = 0; t < it.n && ok; ++t) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!wait_all(&sh->s_full[x], ns[x] & 1, abort, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t scol = x * BK + grp * C::kCols;
          float s[C::kCols];
          if constexpr (C::kCols == 32) {
            uint32_t sr[32];
            tmem_ld32(lanes + scol, sr);
            tmem_ld_wait(sr);
#pragma unroll
            for (int e = 0; e < 32; ++e) s[e] = __uint_as_float(sr[e]);
          } else {
            uint32_t sr[16];
            tmem_ld16(lanes + scol, sr);
            tmem_ld_wait(sr);
#pragma unroll
            for (int e = 0; e < 16; ++e) s[e] = __uint_as_float(sr[e]);
          }
          if (it.diag_last && t == it.n - 1) {
#pragma unroll
            for (int e = 0; e < C::kCols; ++e)
              if (grp * C::kCols + e > row) s[e] = -INFINITY;
          }
          if (t == 0) {
            // the tile's first block of the item: its row maximum is the
            // reference every block of the item uses for this tile
            float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
            for (int e = 4; e + 8 <= C::kCols; e += 8)
#pragma unroll
              for (int a = 0; a < 4; ++a) mx[a] = max3(mx[a], s[e + a], s[e + 4 + a]);
#pragma unroll
            for (int a = 0; a < 4; ++a) mx[a] = fmaxf(mx[a], s[C::kCols - 4 + a]);
            float part[4];
            if (!exchange(fmaxf(max3(mx[0], mx[1], mx[2]), mx[3]), part)) {
              ok = false;
              break;
            }
            m_used[x] = max3(fmaxf(part[0], part[1]), part[2], part[3]) * c;
          }
          float sum0 = 0.f, sum1 = 0.f, sum2 = 0.f, sum3 = 0.f;
          {
            uint32_t pk[C::kCols / 2];
            const float nm = -m_used[x];
#pragma unroll
            for (int e = 0; e < C::kCols / 2; ++e) {
              float a0, a1;
              fma2(a0, a1, s[2 * e], s[2 * e + 1], c, c, nm, nm);
              pk[e] = pack_bf16x2(ex2(a0), ex2(a1));
              if (e & 1)
                add_bf16x2(sum2, sum3, pk[e]);
              else
                add_bf16x2(sum0, sum1, pk[e]);
            }
            if constexpr (C::kCols == 32) {
              tmem_st16(lanes + scol, pk);
            } else {
              tmem_st8(lanes + scol, pk);
            }
          }
          tmem_st_wait();
          l[x] += (sum0 + sum1) + (sum2 + sum3);
          tc_fence_before();
          mbar_arrive(&sh->p_full[x]);
          ++ns[x];
          if (t == 0 && x == 0 && pend) {
            if (!epilogue()) {
              ok = false;
              break;
            }
            pend = false;
          }
        }
      }
      if (!ok) break;
      pend = true;
      pit = it;
      pl[0] = l[0];
      pl[1] = l[1];
      pm[0] = m_used[0];
      pm[1] = m_used[1];
      pq = qi;
      ++qi;
    }
    if (ok && pend) ok = epilogue();
    if (!ok) raise_abort(sh, p);
    if (warp == 4 && lane == 0) bulk_wait_all();
    // recompute the marked items' rows of both heads, one (row, group) per thread
    asm volatile("bar.sync 1, %0;" ::"r"(kSoftmaxThreads) : "memory");
    if (ok && row < p.B) {
      const int32_t begin = p.wptr[blockIdx.x];
      for (int w = 0; w < kRedoWords; ++w) {
        uint32_t bits = sh->redo[w];
        while (bits) {
          const int32_t pos = begin + 32 * w + __ffs(bits) - 1;
          bits &= bits - 1;
          const int32_t item = p.items[pos];
          const int32_t pr = item / p.nb, i = item - pr * p.nb;
          const int32_t n = max(1, min(p.cnt[2 * pr * p.nb + i], min(p.kmax, i + 1)));
          for (int x = 0; x < 2; ++x)
            exact_row<D, BK, C::kOCols>(p, 2 * pr + x, i, n, row, grp * C::kOCols, grp == 0);
        }
      }
    }
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
  using C = PCfg<D, BK>;
  constexpr int kSmem = C::kData + int(sizeof(Shared));
  static_assert(kSmem <= 232448, "shared memory budget");
  CUtensorMap tq, tk, tv, to;
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
  auto kern = prefill_pair_kernel<D, BK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  if (a.num_workers == 0) return cudaSuccess;
  kern<<<a.num_workers, kThreads, kSmem, st>>>(tq, tk, tv, to, p);
  return cudaGetLastError();
}

}  // namespace

namespace sa_k {

cudaError_t launch_prefill_attention_pairs(const PrefillArgs& a, cudaStream_t st,
                                           bool* encode_failed) {
  *encode_failed = false;
  if (a.Hq % 2 != 0 || (a.Hq / a.Hkv) % 2 != 0) return cudaErrorInvalidValue;
  if (a.d == 128 && a.B == 128) return launch<128, 128>(a, st, encode_failed);
  if (a.d == 64 && a.B == 64) return launch<64, 64>(a, st, encode_failed);
  return cudaErrorInvalidValue;
}

}  // namespace sa_k
