// Decode attention over the selected KV blocks (HBM-bound).
//
// One CTA per (sequence, query head), four warps.  A head's selected blocks
// are split into 16-token units (a block of g tokens is g/16 units; the
// default B = 32 is two), and a step takes 32 rows: the 16 tokens of two
// consecutive units.  Each warp takes every fourth step.  Lane l owns
// dimensions [4l, 4l+4) of every key and value row, so each row is one
// coalesced 256-byte load across the warp; key and value rows are loaded
// together before any arithmetic (16 KB in flight per warp and step).  Every
// lane forms 32 partial dot products over its four dimensions; a
// reduce-scatter over the warp (31 shuffles) leaves the score of row t in
// lane t, the warp keeps an online softmax, and then accumulates P V in the
// same dimension layout.  The four partial states are merged by their
// log-sum-exp.  Streaming and retrieval heads differ only in their block
// lists, and retrieval heads may select at their own block size ("Riepilogo
// Tecnico: Fluxion", "Intuizioni Chiave" 2).

#include <cuda_bf16.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "sparse_attn.h"

namespace {

constexpr int kD = 128;
constexpr int kB = 32;
constexpr int kWarps = 4;
constexpr int kU = 16;       // tokens per unit; a step is two units
static_assert(kB == 32 && kD == 4 * 32, "lane t <-> row t, lane l <-> dims [4l, 4l+4)");

__global__ void __launch_bounds__(kWarps * 32, 4) decode_attention_kernel(sa_k::DecodeArgs a,
                                                                       float scale_log2) {
  __shared__ float sq[kD];
  __shared__ float sm[kWarps], sl[kWarps];
  __shared__ float so[kWarps][kD];
  // rows may be restricted to a list of heads (one kind of head)
  const int row = a.heads ? (int(blockIdx.x) / a.nh) * a.Hq + a.heads[blockIdx.x % a.nh]
                          : int(blockIdx.x);
  const int b = row / a.Hq, h = row % a.Hq;
  const int g = h / (a.Hq / a.Hkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this head's block size (a multiple of 16) and block count
  int gsz = a.gran ? a.gran[h] : kB;
  if (gsz < kU || (gsz % kU) != 0 || a.L % gsz != 0) gsz = kB;
  const int per = gsz / kU;                   // units per block
  const int nb = a.L / gsz;

  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + size_t(row) * kD;
  for (int c = threadIdx.x; c < kD; c += kWarps * 32) sq[c] = __bfloat162float(q[c]);
  __syncthreads();

  int n = a.cnt[row];
  if (n < 1 || n > a.kmax) {
    if (threadIdx.x == 0) atomicOr(a.dev_status, SA_DEV_BAD_COUNT);
    n = max(1, min(n, a.kmax));
  }
  const int32_t* list = a.idx + size_t(row) * a.kmax;
  const size_t head_off = (size_t(b) * a.Hkv + g) * size_t(a.L) * kD;
  const __nv_bfloat16* K = static_cast<const __nv_bfloat16*>(a.k) + head_off;
  const __nv_bfloat16* V = static_cast<const __nv_bfloat16*>(a.v) + head_off;

  float m = -INFINITY, l = 0.f;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  const float q4[4] = {sq[4 * lane], sq[4 * lane + 1], sq[4 * lane + 2], sq[4 * lane + 3]};
  const int units = n * per;
  // first token of unit x: unit x % per of block list[x / per]
  auto unit_start = [&](int x) -> size_t {
    int j = list[x / per];
    if (j < 0 || j >= nb) {
      if (lane == 0) atomicOr(a.dev_status, SA_DEV_BAD_INDEX);
      j = 0;
    }
    return size_t(j) * gsz + size_t(x % per) * kU;
  };
  for (int t = warp; 2 * t < units; t += kWarps) {
    const size_t t0 = unit_start(2 * t);
    const bool two = 2 * t + 1 < units;       // else rows 16..31 are masked
    const size_t t1 = two ? unit_start(2 * t + 1) : t0;
    const uint2* kc0 = reinterpret_cast<const uint2*>(K + t0 * kD) + lane;
    const uint2* kc1 = reinterpret_cast<const uint2*>(K + t1 * kD) + lane;
    const uint2* vc0 = reinterpret_cast<const uint2*>(V + t0 * kD) + lane;
    const uint2* vc1 = reinterpret_cast<const uint2*>(V + t1 * kD) + lane;
    uint2 kv[kB], vv[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) kv[u] = __ldg(u < kU ? kc0 + u * (kD / 4) : kc1 + (u - kU) * (kD / 4));
#pragma unroll
    for (int u = 0; u < kB; ++u) vv[u] = __ldg(u < kU ? vc0 + u * (kD / 4) : vc1 + (u - kU) * (kD / 4));
    // partial dot products of row u over this lane's four dimensions
    float part[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      float a = __uint_as_float(kv[u].x << 16) * q4[0];
      a = fmaf(__uint_as_float(kv[u].x & 0xFFFF0000u), q4[1], a);
      a = fmaf(__uint_as_float(kv[u].y << 16), q4[2], a);
      part[u] = fmaf(__uint_as_float(kv[u].y & 0xFFFF0000u), q4[3], a);
    }
    // reduce-scatter: at width w each lane keeps the half of the rows whose
    // bit w matches its own and adds the partner's copy of that half; after
    // five rounds lane t holds the full dot product of row t
#pragma unroll
    for (int w = kB / 2; w >= 1; w >>= 1) {
      const bool upper = (lane & w) != 0;
#pragma unroll
      for (int i = 0; i < w; ++i) {
        const float send = upper ? part[i] : part[i + w];
        const float keep = upper ? part[i + w] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
      }
    }
    const float s = (two || lane < kU) ? part[0] * scale_log2 : -INFINITY;
    float mb = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
    const float mn = fmaxf(m, mb);
    const float alpha = sa_dev::ex2(m - mn);
    const float p = sa_dev::ex2(s - mn);
    float ps = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] *= alpha;
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const float pu = __shfl_sync(0xffffffffu, p, u);
      o[0] = fmaf(pu, __uint_as_float(vv[u].x << 16), o[0]);
      o[1] = fmaf(pu, __uint_as_float(vv[u].x & 0xFFFF0000u), o[1]);
      o[2] = fmaf(pu, __uint_as_float(vv[u].y << 16), o[2]);
      o[3] = fmaf(pu, __uint_as_float(vv[u].y & 0xFFFF0000u), o[3]);
    }
    m = mn;
  }
  if (lane == 0) {
    sm[warp] = m;
    sl[warp] = l;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) so[warp][lane * 4 + e] = o[e];
  __syncthreads();
  if (warp == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm[w]);
    float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      if (sm[w] == -INFINITY) continue;     // a warp that had no block
      const float f = sa_dev::ex2(sm[w] - M);
      L += sl[w] * f;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] += so[w][lane * 4 + e] * f;
    }
    const float inv = 1.f / L;
    if (a.out_f32) {
      float* dst = static_cast<float*>(a.o) + size_t(row) * kD + lane * 4;
      *reinterpret_cast<float4*>(dst) =
          make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    } else {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.o) + size_t(row) * kD + lane * 4;
      uint2 pk;
      pk.x = sa_dev::pack_bf16x2(acc[0] * inv, acc[1] * inv);
      pk.y = sa_dev::pack_bf16x2(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2*>(dst) = pk;
    }
    if (a.lse && lane == 0) a.lse[row] = (M + log2f(L)) * 0.6931471805599453f;
  }
}

}  // namespace

namespace sa_k {

cudaError_t launch_decode_attention(const DecodeArgs& a, cudaStream_t st) {
  if (a.d != kD || a.B != kB) return cudaErrorInvalidValue;
  if (a.heads && a.nh <= 0) return cudaErrorInvalidValue;
  const int rows = a.Bt * (a.heads ? a.nh : a.Hq);
  if (rows == 0) return cudaSuccess;
  const float scale_log2 = float(1.4426950408889634 / 11.313708498984761);  // log2(e)/sqrt(128)
  decode_attention_kernel<<<rows, kWarps * 32, 0, st>>>(a, scale_log2);
  return cudaGetLastError();
}

}  // namespace sa_k
