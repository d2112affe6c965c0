// Decode attention of one (sequence, query head) row by four warps.
//
// Shared by the decode attention kernel (one CTA per row) and the one-launch
// decode step (one warpgroup per row, after the row's selection).  A head's
// selected blocks are split into 16-token units (a block of g tokens is g/16
// units); warp w of the four takes units w, w+4, w+8, ...  Each warp streams
// its units through kStages shared-memory stages of its own: a unit's 16 key
// rows and 16 value rows (4 KB each, contiguous in the cache) arrive by two
// bulk asynchronous copies on the stage's mbarrier, and the copies of the
// warp's next units are in flight while it works on the current one.  Lane l
// owns dimensions [4l, 4l+4) of every row: it forms 16 partial dot products
// over its four dimensions, a reduce-scatter over the warp (16 shuffles)
// leaves the score of row r in lanes r and r + 16, the warp keeps an online
// softmax and accumulates P V in the same dimension layout.  The four partial
// states are merged by their log-sum-exp ("Riepilogo Tecnico: Fluxion",
// "Intuizioni Chiave" 2: streaming and retrieval heads differ only in their
// block lists).  The arithmetic does not depend on kStages, so both callers
// give the same bits.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"
#include "sparse_attn.h"

namespace sa_da {

constexpr int kD = 128;
constexpr int kB = 32;                        // the default block size
constexpr int kWarps = 4;                     // warps per row
constexpr int kU = 16;                        // tokens per unit
constexpr uint32_t kUnitBytes = kU * kD * 2;  // one unit of K (or of V)
static_assert(kD == 4 * 32, "lane l <-> dims [4l, 4l+4)");

// The row's inputs, as one warp sees them.
struct Row {
  const __nv_bfloat16* K;                     // the KV head's keys [L][d] of this sequence
  const __nv_bfloat16* V;
  const int32_t* list;                        // the row's block list
  int n;                                      // its length (already checked)
  int gsz, per, nb;                           // block size, units per block, blocks
  uint64_t limit;                             // limit of each wait for a copy
  int32_t* dev_status;
};

// One warp's share of the row: units w, w + 4, ... through its stages
// sk/sv[kStages] and barriers full[kStages].  `base` counts the units this
// warp has taken through these stages before (their mbarrier phases); it is
// advanced past this row's units.  Returns false if a wait ran out; the
// copies then in flight have landed (or the drain gave up too) and the state
// is not to be merged.
template <int kStages>
__device__ __forceinline__ bool attend_warp(const Row& r, const float (&q4)[4],
                                            uint2 (*sk)[kU][32], uint2 (*sv)[kU][32],
                                            uint64_t* full, uint32_t& base, int warp, int lane,
                                            float scale_log2, float& m_out, float& l_out,
                                            float (&o)[4]) {
  float m = -INFINITY, l = 0.f;
  o[0] = o[1] = o[2] = o[3] = 0.f;
  const int units = r.n * r.per;
  // first token of unit x: unit x % per of block list[x / per]
  auto unit_start = [&](int x) -> size_t {
    int j = r.list[x / r.per];
    if (j < 0 || j >= r.nb) {
      if (lane == 0) atomicOr(r.dev_status, SA_DEV_BAD_INDEX);
      j = 0;
    }
    return size_t(j) * r.gsz + size_t(x % r.per) * kU;
  };
  // the warp's c-th unit of the row goes to stage (base + c) % kStages
  auto issue = [&](int x, int c) {
    const size_t t0 = unit_start(x);
    const int s = int((base + uint32_t(c)) % kStages);
    if (lane == 0) {
      sa_dev::mbar_arrive_expect_tx(&full[s], 2 * kUnitBytes);
      sa_dev::bulk_load(&sk[s][0][0], r.K + t0 * kD, kUnitBytes, &full[s]);
      sa_dev::bulk_load(&sv[s][0][0], r.V + t0 * kD, kUnitBytes, &full[s]);
    }
  };
  int issued = 0, used = 0;                   // this row's units issued and consumed
  for (; issued < kStages && warp + issued * kWarps < units; ++issued)
    issue(warp + issued * kWarps, issued);
  bool ok = true;
  for (int x = warp; x < units; x += kWarps) {
    const uint32_t c = base + uint32_t(used);
    const int s = int(c % kStages);
    if (!sa_dev::wait_all(&full[s], (c / kStages) & 1u, nullptr, r.limit)) {
      ok = false;
      break;
    }
    uint2 kv[kU], vv[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) kv[u] = sk[s][u][lane];
#pragma unroll
    for (int u = 0; u < kU; ++u) vv[u] = sv[s][u][lane];
    ++used;
    // every lane has its rows in registers: the stage takes the warp's next
    // unit (the async proxy writes it after these generic reads)
    __syncwarp();
    if (warp + issued * kWarps < units) {
      sa_dev::fence_proxy_async_smem();
      issue(warp + issued * kWarps, issued);
      ++issued;
    }
    // partial dot products of row u over this lane's four dimensions
    float part[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      float d = __uint_as_float(kv[u].x << 16) * q4[0];
      d = fmaf(__uint_as_float(kv[u].x & 0xFFFF0000u), q4[1], d);
      d = fmaf(__uint_as_float(kv[u].y << 16), q4[2], d);
      part[u] = fmaf(__uint_as_float(kv[u].y & 0xFFFF0000u), q4[3], d);
    }
    // reduce-scatter inside each half-warp: at width w a lane keeps the half
    // of the rows whose bit w matches its own and adds the partner's copy;
    // after four rounds lane t holds row t & 15 over its half's dimensions,
    // and one more exchange adds the other half's
#pragma unroll
    for (int w = kU / 2; w >= 1; w >>= 1) {
      const bool upper = (lane & w) != 0;
#pragma unroll
      for (int i = 0; i < w; ++i) {
        const float send = upper ? part[i] : part[i + w];
        const float keep = upper ? part[i + w] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
      }
    }
    const float s_row = (part[0] + __shfl_xor_sync(0xffffffffu, part[0], 16)) * scale_log2;
    float mb = s_row;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
    const float mn = fmaxf(m, mb);
    const float alpha = sa_dev::ex2(m - mn);
    const float p = sa_dev::ex2(s_row - mn);
    float ps = p;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] *= alpha;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const float pu = __shfl_sync(0xffffffffu, p, u);
      o[0] = fmaf(pu, __uint_as_float(vv[u].x << 16), o[0]);
      o[1] = fmaf(pu, __uint_as_float(vv[u].x & 0xFFFF0000u), o[1]);
      o[2] = fmaf(pu, __uint_as_float(vv[u].y << 16), o[2]);
      o[3] = fmaf(pu, __uint_as_float(vv[u].y & 0xFFFF0000u), o[3]);
    }
    m = mn;
  }
  if (!ok) {
    if (lane == 0) atomicOr(r.dev_status, SA_DEV_TIMEOUT);
    // copies still in flight land before the stages are reused or the CTA's
    // shared memory goes
    if (lane == 0)
      for (int c = used; c < issued; ++c) {
        const uint32_t cc = base + uint32_t(c);
        sa_dev::mbar_wait(&full[cc % kStages], (cc / kStages) & 1u, nullptr);
      }
    __syncwarp();
    m = -INFINITY;                            // this warp's part is not merged
  }
  base += uint32_t(issued);
  m_out = m;
  l_out = l;
  return ok;
}

// The four warps' states of a row, merged by one warp.
struct Merge {
  float m[kWarps], l[kWarps];
  float o[kWarps][kD];
};

__device__ __forceinline__ void post_state(Merge& x, int warp, int lane, float m, float l,
                                           const float (&o)[4]) {
  if (lane == 0) {
    x.m[warp] = m;
    x.l[warp] = l;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) x.o[warp][lane * 4 + e] = o[e];
}

// Called by one warp after the four have posted (and a barrier): o[row] and
// lse[row].
__device__ __forceinline__ void merge_store(const Merge& x, int lane, size_t row, void* out,
                                            bool out_f32, float* lse) {
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, x.m[w]);
  float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (x.m[w] == -INFINITY) continue;        // a warp that had no block
    const float f = sa_dev::ex2(x.m[w] - M);
    L += x.l[w] * f;
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] += x.o[w][lane * 4 + e] * f;
  }
  const float inv = 1.f / L;
  if (out_f32) {
    float* dst = static_cast<float*>(out) + row * kD + lane * 4;
    *reinterpret_cast<float4*>(dst) =
        make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
  } else {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(out) + row * kD + lane * 4;
    uint2 pk;
    pk.x = sa_dev::pack_bf16x2(acc[0] * inv, acc[1] * inv);
    pk.y = sa_dev::pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
  }
  if (lse && lane == 0) lse[row] = (M + log2f(L)) * 0.6931471805599453f;
}

// log2(e) / sqrt(128): scores enter the exponentials in base 2
constexpr float kScaleLog2 = float(1.4426950408889634 / 11.313708498984761);

}  // namespace sa_da
