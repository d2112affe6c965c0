// Index step: block mean-pooling and pooled block scores.
//
// Block granularity follows "Riepilogo Tecnico: Fluxion" ("Accoppiamento
// Granularità-Budget") and the Index operation of Spin ("Abstracción de
// Partición Unificada"); the block summary (the mean) is a reading.
//
// pool_kernel      HBM-bound: every block of B rows x d bf16 is read once with
//                  16-byte loads, summed in fp32 and scaled by 1/B.
// prefill_scores   S[h,i,j] = qbar[h,i] . kbar[g,j] * scale for j <= i; a
//                  64x64 fp32 SIMT tile per CTA over the lower triangle (the
//                  contraction is small -- d = 128 -- and selection needs fp32
//                  accuracy, so no reduced-precision tensor path).
// decode_scores    scores[b,h,j] = q[b,h] . kbar[b,g,j] * scale; a warp takes
//                  16 pooled key rows (coalesced, all in flight) for all G
//                  query heads of the group and reduces with a reduce-scatter.

#include <cuda_bf16.h>

#include <cstdint>

#include "kernels.h"

namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

// One CTA per pooled row: x rows [r*B, (r+1)*B) of width d -> out[r][0..d).
template <int D>
__global__ void __launch_bounds__(256) pool_kernel(const uint4* __restrict__ x,
                                                   float* __restrict__ out, int block) {
  constexpr int kVec = D / 8;                 // 16-byte vectors per row
  constexpr int kGroups = 256 / kVec;         // rows handled in parallel
  __shared__ float part[kGroups][D];
  const int v = threadIdx.x % kVec;
  const int g = threadIdx.x / kVec;
  const size_t base = size_t(blockIdx.x) * block * kVec;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int r = g; r < block; r += kGroups) {
    float f[8];
    bf16x8_to_f32(__ldg(&x[base + size_t(r) * kVec + v]), f);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] += f[k];
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) part[g][v * 8 + k] = acc[k];
  __syncthreads();
  const float inv = 1.f / float(block);
  for (int c = threadIdx.x; c < D; c += 256) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < kGroups; ++q) s += part[q][c];
    out[size_t(blockIdx.x) * D + c] = s * inv;
  }
}

// 64x64 output tile per CTA, 256 threads, each 4x4 outputs; d in chunks of 32.
constexpr int kT = 64, kKc = 32;

__global__ void __launch_bounds__(256) prefill_scores_kernel(const float* __restrict__ qbar,
                                                             const float* __restrict__ kbar,
                                                             float* __restrict__ scores, int nb,
                                                             int d, int group, float scale,
                                                             int tiles) {
  // blockIdx.x enumerates lower-triangle tile pairs (ti >= tj); blockIdx.y = head
  int t = blockIdx.x, ti = 0;
  while (t > ti) {
    t -= ti + 1;
    ++ti;
  }
  const int tj = t;
  const int h = blockIdx.y;
  const float* qh = qbar + size_t(h) * nb * d;
  const float* kg = kbar + size_t(h / group) * nb * d;
  __shared__ float sq[kKc][kT + 4];
  __shared__ float sk[kKc][kT + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int c0 = 0; c0 < d; c0 += kKc) {
    for (int e = threadIdx.x; e < kT * kKc; e += 256) {
      const int r = e / kKc, c = e % kKc;
      const int qi = ti * kT + r, kj = tj * kT + r;
      sq[c][r] = (qi < nb) ? qh[size_t(qi) * d + c0 + c] : 0.f;
      sk[c][r] = (kj < nb) ? kg[size_t(kj) * d + c0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < kKc; ++c) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a[u] = sq[c][ty * 4 + u];
        b[u] = sk[c][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int w = 0; w < 4; ++w) acc[u][w] = fmaf(a[u], b[w], acc[u][w]);
    }
    __syncthreads();
  }
  (void)tiles;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = ti * kT + ty * 4 + u;
    if (i >= nb) continue;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int j = tj * kT + tx * 4 + w;
      if (j <= i) scores[(size_t(h) * nb + i) * nb + j] = acc[u][w] * scale;
    }
  }
}

// CTA = (128 pooled rows, kv head g, sequence b); 8 warps of 16 rows.  D = 128.
constexpr int kMaxGroup = 16;

__global__ void __launch_bounds__(256) decode_scores_kernel(const __nv_bfloat16* __restrict__ q,
                                                            const float* __restrict__ kbar,
                                                            float* __restrict__ scores, int Hq,
                                                            int Hkv, int group, int nb,
                                                            float scale) {
  // Each warp scores 16 pooled key rows against every query head of the KV
  // group.  Lane l holds dimensions [4(l%32).. ) of each row -- one coalesced
  // 512-byte load per row, 16 rows in flight -- and forms partial dot products;
  // a reduce-scatter over the 16 lanes of each half-warp (15 shuffles) and one
  // exchange between the halves leave row r's score in lanes r and r + 16.
  constexpr int D = 128, R = 16;
  __shared__ float sq[kMaxGroup][D];
  const int b = blockIdx.z, g = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < group * D; e += 256) {
    const int hh = e / D, c = e % D;
    sq[hh][c] = __bfloat162float(q[(size_t(b) * Hq + g * group + hh) * D + c]);
  }
  __syncthreads();
  const float4* kb = reinterpret_cast<const float4*>(kbar + (size_t(b) * Hkv + g) * nb * D);
  const int j0 = (blockIdx.x * 8 + warp) * R;
  if (j0 >= nb) return;
  float4 kv[R];
#pragma unroll
  for (int u = 0; u < R; ++u) {
    const int j = min(j0 + u, nb - 1);        // rows past nb are read (in range) and not stored
    kv[u] = __ldg(&kb[size_t(j) * (D / 4) + lane]);
  }
  for (int hh = 0; hh < group; ++hh) {
    const float4 q4 = *reinterpret_cast<const float4*>(&sq[hh][lane * 4]);
    float part[R];
#pragma unroll
    for (int u = 0; u < R; ++u)
      part[u] = fmaf(kv[u].x, q4.x, fmaf(kv[u].y, q4.y, fmaf(kv[u].z, q4.z, kv[u].w * q4.w)));
#pragma unroll
    for (int w = R / 2; w >= 1; w >>= 1) {
      const bool upper = (lane & w) != 0;
#pragma unroll
      for (int i = 0; i < w; ++i) {
        const float send = upper ? part[i] : part[i + w];
        const float keep = upper ? part[i + w] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
      }
    }
    const float sc = part[0] + __shfl_xor_sync(0xffffffffu, part[0], 16);
    const int j = j0 + (lane & (R - 1));
    if (lane < R && j < nb) scores[(size_t(b) * Hq + g * group + hh) * nb + j] = sc * scale;
  }
}

}  // namespace

namespace sa_k {

cudaError_t launch_pool(const void* x, float* out, int64_t rows, int block, int d,
                        cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const uint4* xv = static_cast<const uint4*>(x);
  if (d == 128)
    pool_kernel<128><<<unsigned(rows), 256, 0, st>>>(xv, out, block);
  else if (d == 64)
    pool_kernel<64><<<unsigned(rows), 256, 0, st>>>(xv, out, block);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_prefill_scores(const float* qbar, const float* kbar, float* scores, int Hq,
                                  int group, int nb, int d, float scale, cudaStream_t st) {
  const int tiles = (nb + kT - 1) / kT;
  const dim3 grid(unsigned(tiles * (tiles + 1) / 2), unsigned(Hq));
  prefill_scores_kernel<<<grid, 256, 0, st>>>(qbar, kbar, scores, nb, d, group, scale, tiles);
  return cudaGetLastError();
}

cudaError_t launch_decode_scores(const void* q, const float* kbar, float* scores, int Bt, int Hq,
                                 int group, int nb, int d, float scale, cudaStream_t st) {
  if (d != 128 || group > kMaxGroup) return cudaErrorInvalidValue;
  // 8 warps x 16 rows per CTA
  const dim3 grid(unsigned((nb + 127) / 128), unsigned(Hq / group), unsigned(Bt));
  decode_scores_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(q), kbar, scores,
                                             Hq, Hq / group, group, nb, scale);
  return cudaGetLastError();
}

}  // namespace sa_k
