// Decode attention over the selected KV blocks (HBM-bound).
//
// One CTA per (sequence, query head), four warps.  Each warp takes every
// fourth selected block: lane t scores token t of the 32-token block against
// the query (16-byte loads of the key row), the warp keeps an online softmax,
// and then accumulates P V with lane l owning dimensions [4l, 4l+4) (each
// value row is one coalesced 256-byte load across the warp).  Key and value
// rows of a block are loaded together before any arithmetic, so a warp has
// 16 KB in flight per block.  The four partial states are merged by their
// log-sum-exp.  Streaming and retrieval heads differ only in their block
// lists ("Riepilogo Tecnico: Fluxion", "Intuizioni Chiave" 2).

#include <cuda_bf16.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "sparse_attn.h"

namespace {

constexpr int kD = 128;
constexpr int kB = 32;
constexpr int kWarps = 4;

__global__ void __launch_bounds__(kWarps * 32) decode_attention_kernel(sa_k::DecodeArgs a,
                                                                       float scale_log2) {
  __shared__ float sq[kD];
  __shared__ float sm[kWarps], sl[kWarps];
  __shared__ float so[kWarps][kD];
  const int row = blockIdx.x;
  const int b = row / a.Hq, h = row % a.Hq;
  const int g = h / (a.Hq / a.Hkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = a.L / kB;

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
  for (int t = warp; t < n; t += kWarps) {
    int j = list[t];
    if (j < 0 || j >= nb) {
      if (lane == 0) atomicOr(a.dev_status, SA_DEV_BAD_INDEX);
      j = 0;
    }
    const uint4* krow = reinterpret_cast<const uint4*>(K + (size_t(j) * kB + lane) * kD);
    const uint2* vcol = reinterpret_cast<const uint2*>(V + size_t(j) * kB * kD) + lane;
    uint4 kv[kD / 8];
    uint2 vv[kB];
#pragma unroll
    for (int c = 0; c < kD / 8; ++c) kv[c] = __ldg(krow + c);
#pragma unroll
    for (int u = 0; u < kB; ++u) vv[u] = __ldg(vcol + u * (kD / 4));
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kD / 8; ++c) {
      const uint32_t w[4] = {kv[c].x, kv[c].y, kv[c].z, kv[c].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s = fmaf(__uint_as_float(w[e] << 16), sq[8 * c + 2 * e], s);
        s = fmaf(__uint_as_float(w[e] & 0xFFFF0000u), sq[8 * c + 2 * e + 1], s);
      }
    }
    s *= scale_log2;
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
  const int rows = a.Bt * a.Hq;
  if (rows == 0) return cudaSuccess;
  const float scale_log2 = float(1.4426950408889634 / 11.313708498984761);  // log2(e)/sqrt(128)
  decode_attention_kernel<<<rows, kWarps * 32, 0, st>>>(a, scale_log2);
  return cudaGetLastError();
}

}  // namespace sa_k
