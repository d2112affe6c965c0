// Select step: per-row top-k_h block selection (one CTA per row).  With a
// group-shared plan a row is (KV group, query block): the candidates are
// ranked by the sum of the group's heads' scores (the order of their mean)
// and the list is written for every head of the group.
//
// A prefill row (h, i) keeps min(k_h, i+1) blocks: the sink block 0 ("Riepilogo
// Tecnico: Fluxion", "Intuizioni Chiave" 1), the diagonal block i, and the
// highest-scoring blocks of 1..i-1, ties to the lower index.  A decode
// retrieval head is the row i = nb-1; a decode streaming head keeps block 0
// and the last window_blocks blocks ("Intuizioni Chiave" 2).
//
// The threshold is the exact k-th largest score, found by radix selection
// over the order-preserving bit pattern of the scores (sa_topk::mark_top);
// kept blocks are marked in a bitmap and written in ascending order with
// warp ballots (sa_topk::emit_ascending).

#include <algorithm>
#include <cstdint>

#include "kernels.h"
#include "sparse_attn.h"
#include "topk.cuh"

namespace {

constexpr int kThreads = 128;
constexpr int kPerThread = 16;            // candidates per thread: nb <= 2048

using sa_topk::order_bits;

// One row per CTA of kT threads with kPer candidates each: rows of up to
// kPer * kT blocks.
template <int kT, int kPer>
__device__ __forceinline__ void select_row(const sa_k::SelectArgs& a) {
  __shared__ uint32_t bits[kPer * kT / 32];
  __shared__ sa_topk::Scratch scr;
  const int tid = threadIdx.x;
  // decode rows may be restricted to a list of heads (one kind of head)
  const int row = a.heads ? (int(blockIdx.x) / a.nh) * a.Hq + a.heads[blockIdx.x % a.nh]
                          : int(blockIdx.x);

  int h, i, G = 1;
  const float* srow;
  if (a.decode) {
    // a retrieval head's row has L / g_h blocks of its own size g_h
    h = row % a.Hq;
    const int gsz = a.gran ? a.gran[h] : 0;
    const int nbh = (gsz > 0 && a.kinds[h] != SA_HEAD_STREAMING) ? a.L / gsz : a.nb;
    i = min(nbh, kPer * kT) - 1;
    srow = a.scores + size_t(row) * (a.stride > 0 ? a.stride : a.nb);
  } else if (a.group_shared) {
    G = a.group;
    const int g = row / a.nb;
    i = row - g * a.nb;
    h = g * G;                                  // the group's first head
    srow = a.scores + (size_t(h) * a.nb + i) * a.nb;
  } else {
    h = row / a.nb;
    i = row - h * a.nb;
    srow = a.scores + (size_t(h) * a.nb + i) * a.nb;
  }
  const size_t head_stride = size_t(a.nb) * a.nb;   // between heads' score rows
  const bool streaming = a.decode && a.kinds[h] == SA_HEAD_STREAMING;
  const int nwords = (i + 1 + 31) / 32;
  for (int w = tid; w < nwords; w += kT) bits[w] = 0u;
  __syncthreads();

  if (streaming) {
    const int lo = max(1, a.nb - a.window_blocks);
    for (int j = tid; j <= i; j += kT)
      if (j == 0 || j >= lo) atomicOr(&bits[j >> 5], 1u << (j & 31));
  } else {
    const int keep = min(a.budgets[h], i + 1);
    const int rest = keep - ((i == 0) ? 1 : 2);
    const int ncand = max(0, i - 1);          // blocks 1..i-1
    if (rest >= ncand) {
      for (int j = tid; j <= i; j += kT) atomicOr(&bits[j >> 5], 1u << (j & 31));
    } else {
      if (tid == 0) {
        atomicOr(&bits[0], 1u);
        atomicOr(&bits[i >> 5], 1u << (i & 31));
      }
      if (rest > 0) {
        uint32_t u[kPer];
        if (G == 1) {
          // all of a thread's candidate loads in flight together
#pragma unroll
          for (int r = 0; r < kPer; ++r) {
            const int j = 1 + tid + r * kT;
            u[r] = (j <= i - 1) ? order_bits(srow[j]) : 0u;
          }
        } else {
          // group-shared rows rank by the sum of the group's heads' scores
#pragma unroll
          for (int r = 0; r < kPer; ++r) {
            const int j = 1 + tid + r * kT;
            float sc = 0.f;
            if (j <= i - 1)
              for (int x = 0; x < G; ++x) sc += srow[x * head_stride + j];
            u[r] = (j <= i - 1) ? order_bits(sc) : 0u;
          }
        }
        sa_topk::mark_top<kT, kPer, (kT > 128)>(u, i - 1, uint32_t(rest), bits, scr, tid, 0);
      }
    }
  }
  __syncthreads();

  // ascending block indices, padded with -1, into the row of every head
  // that shares the list
  {
    const size_t orow = a.decode ? size_t(row) : size_t(h) * a.nb + i;
    int32_t* out = a.idx + orow * a.kmax;
    const int total = sa_topk::emit_ascending<kT>(bits, i, out, a.kmax, scr, tid, 0);
    if (tid == 0) a.cnt[orow] = min(total, a.kmax);
    if (G > 1) {
      // the other heads of a group-shared row get copies of the list
      __syncthreads();
      for (int x = 1; x < G; ++x) {
        int32_t* dst = a.idx + (orow + size_t(x) * a.nb) * a.kmax;
        for (int t = tid; t < a.kmax; t += kT) dst[t] = out[t];
        if (tid == 0) a.cnt[orow + size_t(x) * a.nb] = min(total, a.kmax);
      }
    }
  }
}

// Prefill launches tens of thousands of short rows: nine 128-thread CTAs per
// SM (at most 56 registers) keep more of them in flight, and a row takes only
// as many candidates per thread as its length needs.  Decode rows take a
// 512-thread CTA each.
template <int kPer>
__global__ void __launch_bounds__(128, 9) select_kernel(sa_k::SelectArgs a) {
  // (prefill rows only) a row i has i - 1 candidates: shorter rows take
  // fewer per thread
  const int i = int(blockIdx.x) % a.nb;
  if (kPer > 4 && i < 4 * 128)
    select_row<128, 4>(a);
  else if (kPer > 8 && i < 8 * 128)
    select_row<128, 8>(a);
  else
    select_row<128, kPer>(a);
}
template <int kPer>
__global__ void __launch_bounds__(512) select_kernel_wide(sa_k::SelectArgs a) {
  select_row<512, kPer>(a);
}

// Top-p selection of prefill row (h, i): block probabilities are the
// softmax of the row's pooled scores over j <= i; the row keeps blocks 0 and
// i, then blocks of 1..i-1 by score (ties to the lower index) until the kept
// probability reaches p.  Probabilities are summed in 64-bit fixed point (units
// of 2^-32 of the row's total), so the result does not depend on the order of
// the additions.  The threshold is found as in select_kernel, with histograms
// of probability mass next to the counts.
// The rows i in [i0, i0 + span) of every head, kPer candidates per thread
// (rows of up to kPer * kThreads blocks).
template <int kPer>
__global__ void __launch_bounds__(kThreads) select_topp_kernel(sa_k::TopPArgs a, int i0,
                                                                int span) {
  __shared__ uint32_t bits[kPer * kThreads / 32];
  __shared__ unsigned long long hmass[kThreads / 32][256];   // one histogram per warp
  __shared__ uint32_t hcount[kThreads / 32][256];
  __shared__ float redf[kThreads / 32];
  __shared__ unsigned long long ctl_m[2];
  __shared__ uint32_t ctl[3];
  __shared__ uint32_t wsum[kThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = int(blockIdx.x) / span, i = i0 + int(blockIdx.x) % span;
  const int row = h * a.nb + i;
  const float* srow = a.scores + (size_t(h) * a.nb + i) * a.nb;
  const int nwords = (i + 1 + 31) / 32;
  for (int w = tid; w < nwords; w += kThreads) bits[w] = 0u;

  // scores of blocks j = tid + r*kThreads (all j <= i, mandatory ones included)
  float sv[kPer];
  float mx = -INFINITY;
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int j = tid + r * kThreads;
    sv[r] = (j <= i) ? srow[j] : -INFINITY;
    mx = fmaxf(mx, sv[r]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) redf[warp] = mx;
  __syncthreads();
  mx = redf[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) mx = fmaxf(mx, redf[w]);
  __syncthreads();
  float e[kPer], tot = 0.f;
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int j = tid + r * kThreads;
    e[r] = (j <= i) ? exp2f((sv[r] - mx) * 1.4426950408889634f) : 0.f;
    tot += e[r];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  if (lane == 0) redf[warp] = tot;
  __syncthreads();
  tot = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) tot += redf[w];   // same order in every thread
  const float scale = 4294967296.0f / tot;                  // 2^32 / total
  // fixed-point masses (a block's share is at most 2^32, kept as 2^32 - 1);
  // the mandatory blocks' mass is taken first
  uint32_t q[kPer];
  unsigned long long mand = 0;
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int j = tid + r * kThreads;
    const float x = e[r] * scale;
    q[r] = (j <= i) ? (x >= 4294967296.0f ? 0xFFFFFFFFu : uint32_t(x)) : 0u;
    if (j == 0 || j == i) mand += q[r];
  }
  if (tid == 0) ctl_m[0] = 0ull;
  __syncthreads();
  if (mand) atomicAdd(&ctl_m[0], mand);
  if (tid == 0) {
    atomicOr(&bits[0], 1u);
    atomicOr(&bits[i >> 5], 1u << (i & 31));
  }
  __syncthreads();
  const double pd = double(a.p) * 4294967296.0;
  const unsigned long long goal = pd >= 1.8e19 ? ~0ull : (unsigned long long)ceil(pd);
  const unsigned long long have = ctl_m[0];
  __syncthreads();
  if (i >= 2 && goal > have) {
    unsigned long long need = goal - have;           // mass wanted from blocks 1..i-1
    uint32_t u[kPer];
    unsigned long long cand = 0;
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int j = tid + r * kThreads;
      const bool c = j >= 1 && j <= i - 1;
      u[r] = c ? order_bits(sv[r]) : 0u;
      if (c) cand += q[r];
    }
    if (tid == 0) ctl_m[1] = 0ull;
    __syncthreads();
    atomicAdd(&ctl_m[1], cand);
    __syncthreads();
    if (ctl_m[1] <= need) {
      // even every candidate does not reach p: keep them all
      for (int j = 1 + tid; j <= i - 1; j += kThreads) atomicOr(&bits[j >> 5], 1u << (j & 31));
    } else {
      uint32_t prefix = 0, mask = 0, eq_count = 0;
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = tid; b < (kThreads / 32) * 256; b += kThreads) {
          (&hmass[0][0])[b] = 0ull;
          (&hcount[0][0])[b] = 0u;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
          const int j = tid + r * kThreads;
          if (j >= 1 && j <= i - 1 && (u[r] & mask) == prefix) {
            const uint32_t b = (u[r] >> shift) & 255u;
            atomicAdd(&hmass[warp][b], (unsigned long long)q[r]);
            atomicAdd(&hcount[warp][b], 1u);
          }
        }
        __syncthreads();
        if (warp == 0) {
          // lane l holds bins 255-8l .. 248-8l (descending), summed over warps
          unsigned long long mb[8], local = 0;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            mb[k] = 0ull;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) mb[k] += hmass[w][255 - 8 * lane - k];
            local += mb[k];
          }
          unsigned long long incl = local;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
          }
          const unsigned long long excl = incl - local;
          if (excl < need && need <= incl) {
            unsigned long long acc = excl;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (acc + mb[k] >= need) {
                uint32_t n = 0;
#pragma unroll
                for (int w = 0; w < kThreads / 32; ++w) n += hcount[w][255 - 8 * lane - k];
                ctl[0] = uint32_t(255 - 8 * lane - k);
                ctl[1] = n;
                ctl_m[0] = acc;                          // mass of the higher bins
                break;
              }
              acc += mb[k];
            }
          }
        }
        __syncthreads();
        const uint32_t b = ctl[0];
        need -= ctl_m[0];
        eq_count = ctl[1];
        prefix |= b << shift;
        mask |= 0xFFu << shift;
        __syncthreads();
        if (eq_count == 1 && shift > 0) {
          // one candidate left in the bin: it is the threshold
#pragma unroll
          for (int r = 0; r < kPer; ++r) {
            const int j = tid + r * kThreads;
            if (j >= 1 && j <= i - 1 && (u[r] & mask) == prefix) ctl[2] = u[r];
          }
          __syncthreads();
          prefix = ctl[2];
          __syncthreads();
          break;
        }
      }
      const uint32_t T = prefix;
      // candidates above T are all kept; of those equal to T (equal masses),
      // the lowest indices, as many as the remaining mass needs
      unsigned long long qT = 0;
#pragma unroll
      for (int r = 0; r < kPer; ++r) {
        const int j = tid + r * kThreads;
        if (j >= 1 && j <= i - 1 && u[r] == T) qT = q[r];
      }
      if (tid == 0) ctl_m[1] = 0ull;
      __syncthreads();
      if (qT) atomicMax(&ctl_m[1], qT);
      __syncthreads();
      qT = ctl_m[1];
      uint32_t take = qT ? uint32_t((need + qT - 1) / qT) : eq_count;
      take = max(1u, min(take, eq_count));
      if (take == eq_count) {
        // every candidate at T is kept: no order among them is needed
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
          const int j = tid + r * kThreads;
          if (j >= 1 && j <= i - 1 && u[r] >= T) atomicOr(&bits[j >> 5], 1u << (j & 31));
        }
      } else {
      uint32_t taken = 0;
      for (int r = 0; r < kPer; ++r) {
        const int j = tid + r * kThreads;
        const bool valid = j >= 1 && j <= i - 1;
        const bool eq = valid && u[r] == T;
        const uint32_t m = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) wsum[warp] = __popc(m);
        __syncthreads();
        uint32_t before = taken;
        for (int w = 0; w < warp; ++w) before += wsum[w];
        before += __popc(m & ((1u << lane) - 1u));
        if (valid && (u[r] > T || (eq && before < take))) atomicOr(&bits[j >> 5], 1u << (j & 31));
        for (int w = 0; w < kThreads / 32; ++w) taken += wsum[w];
        __syncthreads();
      }
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    int32_t* out = a.idx + size_t(row) * a.kmax;
    int written = 0;
    for (int base = 0; base <= i; base += 32) {
      const int j = base + lane;
      const bool on = (j <= i) && ((bits[j >> 5] >> (j & 31)) & 1u);
      const uint32_t m = __ballot_sync(0xffffffffu, on);
      const int pos = written + __popc(m & ((1u << lane) - 1u));
      if (on && pos < a.kmax) out[pos] = j;
      written += __popc(m);
    }
    for (int t = written + lane; t < a.kmax; t += 32) out[t] = -1;
    if (lane == 0) a.cnt[row] = min(written, a.kmax);
  }
}

}  // namespace

namespace sa_k {

cudaError_t launch_select_topp(const TopPArgs& a, cudaStream_t st) {
  if (a.rows == 0) return cudaSuccess;
  if (a.nb > kPerThread * kThreads) return cudaErrorInvalidValue;
  // a row i holds i + 1 blocks: rows below 512 and 1024 blocks take 4 and 8
  // candidates per thread (three launches, each with its own registers)
  const int heads = a.rows / a.nb;
  const int bounds[4] = {0, 4 * kThreads, 8 * kThreads, kPerThread * kThreads};
  for (int r = 0; r < 3; ++r) {
    const int lo = bounds[r], hi = std::min(bounds[r + 1], a.nb);
    if (hi <= lo) continue;
    const unsigned grid = unsigned(heads) * unsigned(hi - lo);
    if (r == 0)
      select_topp_kernel<4><<<grid, kThreads, 0, st>>>(a, lo, hi - lo);
    else if (r == 1)
      select_topp_kernel<8><<<grid, kThreads, 0, st>>>(a, lo, hi - lo);
    else
      select_topp_kernel<kPerThread><<<grid, kThreads, 0, st>>>(a, lo, hi - lo);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t st) {
  if (a.rows == 0) return cudaSuccess;
  if (a.heads && (!a.decode || a.nh <= 0)) return cudaErrorInvalidValue;
  // decode launches few rows (sequences x heads): wider CTAs per row
  const int row = std::max(a.nb, a.max_row);
  if (!a.decode && row <= 16 * kThreads)
    select_kernel<16><<<unsigned(a.rows), kThreads, 0, st>>>(a);
  else if (a.decode && row <= 4 * 512)
    select_kernel_wide<4><<<unsigned(a.rows), 512, 0, st>>>(a);
  else if (a.decode && row <= 8 * 512)
    select_kernel_wide<8><<<unsigned(a.rows), 512, 0, st>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace sa_k
