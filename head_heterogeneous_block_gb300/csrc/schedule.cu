// LPT schedule rebuilt on the device from per-item block counts.
//
// When the selection decides how many blocks each (head, query-block) item
// keeps (top-p), the costs are known only on the device.  This kernel runs the
// same greedy longest-first multiway partition as the host plan (S-HPLB,
// "Algoritmo Greedy"): items by cost descending, ties to the lower item id,
// each given to the least-loaded worker, ties to the lowest worker id.  The
// result is the CSR schedule the forward kernel reads (wptr [W+1], items [N]),
// each worker's items listed in item order: items are head-major, so the
// CTAs, walking their lists at a similar pace, tend to read the same KV head
// at the same time (with costs that vary per row, assignment order would mix
// all heads at every moment).
//
// One CTA of 16 warps:
//   1. stable counting sort by cost, descending (all warps): per-warp chunk
//      histograms, per-cost chunk offsets, then each warp scatters its chunk
//      in item-id order (lanes with equal cost ranked by lane);
//   2. the greedy (warp 0), placed one run of equal-cost items at a time (see
//      below): the same assignment as walking the items one by one, without a
//      sequential step per item;
//   3. CSR (all warps): worker offsets, then a stable scatter of the items by
//      worker, in item order (per-warp chunk histograms, as in 1).
// Scratch (sorted items, the worker of each sorted position, the worker of
// each item: 3 x N int32) is caller memory; num_items <= 2^19 keeps every
// load in 32 bits.

#include <cstdint>

#include "kernels.h"

namespace {

constexpr int kMaxCost = 2048;          // costs are block counts: 1..nb <= 2048
constexpr int kMaxWorkers = 256;
constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxItems = 1 << 19;

struct RebuildSmem {
  int32_t tab[kWarps][kMaxCost + 1];    // chunk counts per cost, then chunk offsets
  int32_t first[kMaxCost + 1];          // items of cost > c: the run of cost c starts here
  int16_t runs[kMaxCost + 1];           // the costs that occur, descending
  int32_t wbase[kMaxWorkers];
  // the workers taking pairs in a run, compacted in id order: sort key
  // (L mod c, compacted index), then L / c, pair count and id
  uint32_t key[kMaxWorkers];
  uint32_t sq[kMaxWorkers], sn[kMaxWorkers];
  int32_t sw[kMaxWorkers];
};

__device__ __forceinline__ int clamp_cost(int c) {
  return c < 0 ? 0 : (c > kMaxCost ? kMaxCost : c);
}

__global__ void __launch_bounds__(kThreads, 1) lpt_rebuild_kernel(sa_k::RebuildArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RebuildSmem& sh = *reinterpret_cast<RebuildSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lt = (1u << lane) - 1u;
  const int N = a.num_items, W = a.num_workers;
  int32_t* sorted = a.scratch;             // [N] item ids, cost descending
  int32_t* where = a.scratch + N;          // [N] worker of sorted[s]
  int32_t* owner = a.scratch + 2 * N;      // [N] worker of item x

  // ---- 1. stable counting sort by cost, descending
  for (int i = tid; i < kWarps * (kMaxCost + 1); i += kThreads) (&sh.tab[0][0])[i] = 0;
  __syncthreads();
  const int chunk = ((N + kWarps - 1) / kWarps + 31) & ~31;
  const int x0 = min(N, warp * chunk), x1 = min(N, x0 + chunk);
  for (int x = x0 + lane; x < x1; x += 32) atomicAdd(&sh.tab[warp][clamp_cost(a.cnt[x])], 1);
  __syncthreads();
  for (int c = tid; c <= kMaxCost; c += kThreads) {
    int32_t run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int32_t t = sh.tab[w][c];
      sh.tab[w][c] = run;
      run += t;
    }
    sh.first[c] = run;                    // the count of cost c, for now
  }
  __syncthreads();
  if (warp == 0) {
    // first[c] := items of cost > c; lane l scans costs j = kMaxCost - c in
    // [l*S, l*S + S), then an exclusive scan of the lanes' sums
    constexpr int S = (kMaxCost + 1 + 31) / 32;
    int32_t sum = 0;
    for (int j = lane * S; j < min(kMaxCost + 1, lane * S + S); ++j) sum += sh.first[kMaxCost - j];
    int32_t inc = sum;
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    int32_t run = inc - sum;
    for (int j = lane * S; j < min(kMaxCost + 1, lane * S + S); ++j) {
      const int32_t n = sh.first[kMaxCost - j];
      sh.first[kMaxCost - j] = run;
      run += n;
    }
  }
  __syncthreads();
  for (int base = x0; base < x1; base += 32) {
    const int x = base + lane;
    const int c = x < x1 ? clamp_cost(a.cnt[x]) : -1;
    const uint32_t same = __match_any_sync(0xffffffffu, c);
    if (x < x1) sorted[sh.first[c] + sh.tab[warp][c] + __popc(same & lt)] = x;
    __syncwarp();
    if (x < x1 && lane == __ffs(same) - 1) sh.tab[warp][c] += __popc(same);
    __syncwarp();
  }

  // ---- 2. the greedy (warp 0), one run of equal-cost items at a time.  With
  // r items of cost c left to place, the greedy's choices are the r smallest
  // pairs (value, worker) among the sequences L_w + m*c (m >= 0): every step
  // takes the smallest head of those sequences (the least-loaded worker, ties
  // to the lowest id) and moves that worker's head up by c.  So a run is
  // placed at once: a binary search finds the value V of the r-th pair, worker
  // w takes n_w = #(its pairs below V), plus one pair at V if it is among the
  // first workers (by id) with a pair at V.  A pair of w has the value
  // q*c + (L_w mod c) at level q = L_w / c + m, so the pairs in (value,
  // worker) order are the levels in turn, each over the workers taking pairs
  // sorted by (L_w mod c, w): the k-th item of the run goes to the worker of
  // the k-th pair.  Lane l keeps the load and list length of workers
  // l + 32 j in registers.
  if (warp == 0) {
    constexpr int kSlots = kMaxWorkers / 32;
    int nruns = 0;
    for (int c0 = kMaxCost; c0 >= 0; c0 -= 32) {
      const int c = c0 - lane;
      const bool occ = c >= 0 && (c ? sh.first[c - 1] : N) > sh.first[c];
      const uint32_t m = __ballot_sync(0xffffffffu, occ);
      if (occ) sh.runs[nruns + __popc(m & lt)] = int16_t(c);
      nruns += __popc(m);
    }
    uint32_t Ld[kSlots];
    int32_t Cn[kSlots];
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      Ld[j] = 0;
      Cn[j] = 0;
    }
    uint32_t total = 0;
    __syncwarp();
    for (int ir = 0; ir < nruns; ++ir) {
      const int c = sh.runs[ir];
      const int start = sh.first[c], end = c ? sh.first[c - 1] : N;
      const int r = end - start;
      // the least-loaded worker, ties to the lowest id
      uint32_t v = 0xFFFFFFFFu, wmin = 0xFFFFFFFFu;
#pragma unroll
      for (int j = kSlots - 1; j >= 0; --j)
        if (lane + 32 * j < W && Ld[j] <= v) {
          v = Ld[j];
          wmin = uint32_t(lane + 32 * j);
        }
      const uint32_t mn = __reduce_min_sync(0xffffffffu, v);
      if (c == 0) {
        // zero cost: every item goes to the least-loaded worker, loads unchanged
        const int w0 = int(__reduce_min_sync(0xffffffffu, v == mn ? wmin : 0xFFFFFFFFu));
        for (int k = lane; k < r; k += 32) where[start + k] = w0;
#pragma unroll
        for (int j = 0; j < kSlots; ++j)
          if (lane + 32 * j == w0) Cn[j] += r;
        continue;
      }
      const uint32_t cc = uint32_t(c);
      uint32_t Lq[kSlots], Lr[kSlots];
#pragma unroll
      for (int j = 0; j < kSlots; ++j) {
        Lq[j] = Ld[j] / cc;
        Lr[j] = Ld[j] - Lq[j] * cc;
      }
      // pairs of worker w below V = Vq*c + Vr: max(0, Vq - Lq + [Vr > Lr])
      auto below = [&](uint32_t V) -> uint32_t {
        const uint32_t Vq = V / cc, Vr = V - Vq * cc;
        int32_t n = 0;
#pragma unroll
        for (int j = 0; j < kSlots; ++j)
          if (lane + 32 * j < W) n += max(0, int32_t(Vq - Lq[j]) + (Vr > Lr[j] ? 1 : 0));
        return __reduce_add_sync(0xffffffffu, uint32_t(n));
      };
      // below(lo) = 0 < r <= below(hi): the second bound holds since
      // below(V) >= sum_w (V - L_w) / c
      const uint32_t rc = uint32_t(r) * cc;
      uint32_t lo = mn, hi = min(mn + rc, (total + rc + uint32_t(W) - 1) / uint32_t(W));
      while (hi - lo > 1) {
        const uint32_t mid = lo + (hi - lo) / 2;
        if (below(mid) < uint32_t(r)) lo = mid;
        else hi = mid;
      }
      const uint32_t V = lo;                          // value of the r-th pair
      const uint32_t extra = uint32_t(r) - below(V);  // pairs taken at exactly V
      const uint32_t Vq = V / cc, Vr = V - Vq * cc;
      // the workers taking pairs, compacted in id order
      uint32_t Nn[kSlots];
      uint32_t at_before = 0;
      int A = 0;
#pragma unroll
      for (int j = 0; j < kSlots; ++j) {
        Nn[j] = 0;
        if (32 * j < W) {
          const int w = lane + 32 * j;
          bool at = false;
          if (w < W) {
            Nn[j] = uint32_t(max(0, int32_t(Vq - Lq[j]) + (Vr > Lr[j] ? 1 : 0)));
            at = Vr == Lr[j] && Vq >= Lq[j];
          }
          const uint32_t m = __ballot_sync(0xffffffffu, at);
          if (at && at_before + __popc(m & lt) < extra) ++Nn[j];
          at_before += __popc(m);
          const uint32_t act = __ballot_sync(0xffffffffu, Nn[j] > 0);
          if (Nn[j] > 0) {
            const int k = A + __popc(act & lt);
            sh.key[k] = (Lr[j] << 8) | uint32_t(k);      // c <= 2048, k < 256
            sh.sq[k] = Lq[j];
            sh.sn[k] = Nn[j];
            sh.sw[k] = w;
          }
          A += __popc(act);
        }
      }
      __syncwarp();
      // order them by (L mod c, id): a stable radix sort on the bits of
      // L mod c, the list being in id order already; element i = lane + 32 t
      const int T = (A + 31) / 32;
      uint32_t kk[kSlots];
#pragma unroll
      for (int t = 0; t < kSlots; ++t) kk[t] = lane + 32 * t < A ? sh.key[lane + 32 * t] : 0u;
      const int nbits = cc > 1 ? 32 - __clz(int(cc - 1)) : 0;
      for (int bit = 8; bit < 8 + nbits; ++bit) {
        uint32_t Z[kSlots], nz = 0;
#pragma unroll
        for (int t = 0; t < kSlots; ++t) {
          Z[t] = __ballot_sync(0xffffffffu, lane + 32 * t < A && ((kk[t] >> bit) & 1u) == 0);
          nz += __popc(Z[t]);
        }
        if (nz == 0 || nz == uint32_t(A)) continue;   // every key has the same bit
        __syncwarp();
        uint32_t zb = 0;
#pragma unroll
        for (int t = 0; t < kSlots; ++t) {
          const uint32_t i = lane + 32 * t;
          const uint32_t z = zb + __popc(Z[t] & lt);   // zeros before element i
          if (i < uint32_t(A)) sh.key[((kk[t] >> bit) & 1u) ? nz + (i - z) : z] = kk[t];
          zb += __popc(Z[t]);
        }
        __syncwarp();
#pragma unroll
        for (int t = 0; t < kSlots; ++t)
          if (lane + 32 * t < A) kk[t] = sh.key[lane + 32 * t];
      }
      uint32_t tq[kSlots], tn[kSlots], tw[kSlots];
      uint32_t qlo = 0xFFFFFFFFu, qhi = 0;
#pragma unroll
      for (int t = 0; t < kSlots; ++t) {
        tq[t] = tn[t] = tw[t] = 0;
        if (lane + 32 * t < A) {
          const int k = int(kk[t] & 0xFFu);
          tq[t] = sh.sq[k];
          tn[t] = sh.sn[k];
          tw[t] = uint32_t(sh.sw[k]);
          qlo = min(qlo, tq[t]);
          qhi = max(qhi, tq[t] + tn[t] - 1);
        }
      }
      qlo = __reduce_min_sync(0xffffffffu, qlo);
      qhi = __reduce_max_sync(0xffffffffu, qhi);
      // at most r + 1 levels: the least-loaded worker alone has (V - mn) / c
      // pairs below V, fewer than r
      int pos = 0;
      for (uint32_t qv = qlo; qv <= qhi && pos < r; ++qv) {
#pragma unroll
        for (int t = 0; t < kSlots; ++t) {
          if (t < T) {
            const bool on = tq[t] <= qv && qv < tq[t] + tn[t];
            const uint32_t m = __ballot_sync(0xffffffffu, on);
            const int at = start + pos + __popc(m & lt);
            if (on && at < end) where[at] = int32_t(tw[t]);
            pos += __popc(m);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kSlots; ++j) {
        Ld[j] += Nn[j] * cc;
        Cn[j] += int32_t(Nn[j]);
      }
      total += rc;
      __syncwarp();
    }
    // ---- 3a. worker offsets: an exclusive scan of the list lengths in
    // worker order, slot by slot
    int32_t carry = 0;
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      const int w = lane + 32 * j;
      const int32_t x = w < W ? Cn[j] : 0;
      int32_t inc = x;
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      if (w < W) {
        sh.wbase[w] = carry + inc - x;
        a.wptr[w] = carry + inc - x;
      }
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) a.wptr[W] = carry;
  }
  __syncthreads();

  // ---- 3b. the worker of every item, then a stable scatter by worker in
  // item order: chunk counts per worker, their offsets from the worker
  // offsets, and each warp's chunk in order (lanes with equal worker ranked
  // by lane)
  for (int s = tid; s < N; s += kThreads) owner[sorted[s]] = where[s];
  for (int i = tid; i < kWarps * kMaxWorkers; i += kThreads) sh.tab[i / kMaxWorkers][i % kMaxWorkers] = 0;
  __syncthreads();
  for (int x = x0 + lane; x < x1; x += 32) {
    const int w = owner[x];
    if (w >= 0 && w < W) atomicAdd(&sh.tab[warp][w], 1);
  }
  __syncthreads();
  for (int w = tid; w < W; w += kThreads) {
    int32_t run = sh.wbase[w];
    for (int k = 0; k < kWarps; ++k) {
      const int32_t t = sh.tab[k][w];
      sh.tab[k][w] = run;
      run += t;
    }
  }
  __syncthreads();
  for (int base = x0; base < x1; base += 32) {
    const int x = base + lane;
    int w = x < x1 ? owner[x] : -1;
    if (w >= W) w = -1;
    const uint32_t same = __match_any_sync(0xffffffffu, w);
    if (w >= 0) {
      const int slot = sh.tab[warp][w] + __popc(same & lt);
      if (slot < N) a.items[slot] = x;
    }
    __syncwarp();
    if (w >= 0 && lane == __ffs(same) - 1) sh.tab[warp][w] += __popc(same);
    __syncwarp();
  }
}

}  // namespace

namespace sa_k {

cudaError_t launch_lpt_rebuild(const RebuildArgs& a, cudaStream_t st) {
  if (a.num_workers < 1 || a.num_workers > kMaxWorkers || a.num_items < 0 ||
      a.num_items > kMaxItems)
    return cudaErrorInvalidValue;
  const int smem = int(sizeof(RebuildSmem));
  cudaError_t e = cudaFuncSetAttribute(lpt_rebuild_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  lpt_rebuild_kernel<<<1, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sa_k
