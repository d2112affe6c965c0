// Index step: block mean-pooling and pooled block scores.
//
// Block granularity follows "Riepilogo Tecnico: Fluxion" ("Accoppiamento
// Granularità-Budget") and the Index operation of Spin ("Abstracción de
// Partición Unificada"); the block summary (the mean) is a reading.
//
// pool_kernel      HBM-bound: every block of B rows x d bf16 is read once with
//                  16-byte loads, summed in fp32 and scaled by 1/B.
// prefill_scores   S[h,i,j] = qbar[h,i] . kbar[g,j] * scale for j <= i; a
//                  64x64 tile per CTA over the lower triangle on the tensor
//                  cores (tf32 MMAs on both operands split in two, products
//                  hi*hi + hi*lo + lo*hi: selection needs fp32-level scores).
// decode_scores    scores[b,h,j] = q[b,h] . kbar[b,g,j] * scale; persistent
//                  CTAs stream 32 KB chunks of pooled keys through a
//                  three-stage cp.async ring while scoring earlier chunks; a
//                  warp scores 16 rows for all G query heads of the group
//                  with tf32 tensor-core MMAs (split in two for fp32-level
//                  accuracy).  With per-head block sizes, one pass per
//                  size scores the retrieval heads of that size; a group with
//                  none of them is skipped without reading its cache.

#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "index.cuh"
#include "kernels.h"
#include "sparse_attn.h"

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

using namespace sa_ix;

// Prefill scores on the tensor cores: one 64x64 tile of (query block i, key
// block j), j <= i, per CTA over the lower triangle.  The tile's pooled query
// and key rows (fp32) are copied into XOR-swizzled shared memory with
// cp.async; warp w takes tile rows 16(w%4) .. +16 and columns 32(w/4) .. +32
// as four m16n8k8 tf32 MMA tiles.  Both operands are fp32: each is split into
// a tf32 part and the rest, and the products hi*hi + hi*lo + lo*hi keep
// fp32-level scores (selection needs them; a single tf32 or bf16 product
// would not).  The k order inside an MMA is permuted as in the decode kernel.
constexpr int kT = 64;

template <int D>
__global__ void __launch_bounds__(256) prefill_scores_kernel(const float* __restrict__ qbar,
                                                             const float* __restrict__ kbar,
                                                             float* __restrict__ scores, int nb,
                                                             int group, float scale) {
  constexpr int kC = D / 4;                   // 16-byte chunks per row
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float4 (*sa)[kC] = reinterpret_cast<float4 (*)[kC]>(smem_raw);
  float4 (*sb)[kC] = reinterpret_cast<float4 (*)[kC]>(smem_raw + kT * kC * sizeof(float4));
  // blockIdx.x enumerates lower-triangle tile pairs (ti >= tj); blockIdx.y = head
  int t = blockIdx.x, ti = 0;
  while (t > ti) {
    t -= ti + 1;
    ++ti;
  }
  const int tj = t, h = blockIdx.y;
  const int i0 = ti * kT, j0 = tj * kT;
  const float4* qh = reinterpret_cast<const float4*>(qbar + size_t(h) * nb * D);
  const float4* kg = reinterpret_cast<const float4*>(kbar + size_t(h / group) * nb * D);
  for (int e = threadIdx.x; e < kT * kC; e += 256) {
    const int r = e / kC, c = e - r * kC;
    if (i0 + r < nb) cp_async16(&sa[r][swz<kC>(r, c)], qh + size_t(i0 + r) * kC + c);
    if (j0 + r < nb) cp_async16(&sb[r][swz<kC>(r, c)], kg + size_t(j0 + r) * kC + c);
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  // rows past nb hold stale data; they only reach outputs that are not stored
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, tq = lane & 3;
  const int ra = 16 * (warp & 3) + gq;        // this lane's tile rows: ra, ra + 8
  const int cb = 32 * (warp >> 2);            // the warp's tile columns: cb .. cb + 32
  float acc[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
#pragma unroll
  for (int m = 0; m < D / 16; ++m) {          // dimensions 16m .. 16m + 16: two k-steps
    const float4 xa = sa[ra][swz<kC>(ra, 4 * m + tq)];
    const float4 xb = sa[ra + 8][swz<kC>(ra + 8, 4 * m + tq)];
    uint32_t ah0[4], al0[4], ah1[4], al1[4];
    split_tf32(xa.x, ah0[0], al0[0]);
    split_tf32(xb.x, ah0[1], al0[1]);
    split_tf32(xa.y, ah0[2], al0[2]);
    split_tf32(xb.y, ah0[3], al0[3]);
    split_tf32(xa.z, ah1[0], al1[0]);
    split_tf32(xb.z, ah1[1], al1[1]);
    split_tf32(xa.w, ah1[2], al1[2]);
    split_tf32(xb.w, ah1[3], al1[3]);
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const int rn = cb + 8 * n + gq;         // the key block of this lane's B column
      const float4 y = sb[rn][swz<kC>(rn, 4 * m + tq)];
      uint32_t bh0, bl0, bh1, bl1, bh2, bl2, bh3, bl3;
      split_tf32(y.x, bh0, bl0);
      split_tf32(y.y, bh1, bl1);
      split_tf32(y.z, bh2, bl2);
      split_tf32(y.w, bh3, bl3);
      mma_tf32(acc[n], ah0, bh0, bh1);
      mma_tf32(acc[n], ah0, bl0, bl1);
      mma_tf32(acc[n], al0, bh0, bh1);
      mma_tf32(acc[n], ah1, bh2, bh3);
      mma_tf32(acc[n], ah1, bl2, bl3);
      mma_tf32(acc[n], al1, bh2, bh3);
    }
  }
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = i0 + ra + ((e & 2) ? 8 : 0);
      const int j = j0 + cb + 8 * n + 2 * tq + (e & 1);
      if (i < nb && j <= i) scores[(size_t(h) * nb + i) * nb + j] = acc[n][e] * scale;
    }
}

// Decode scores, persistent: two CTAs per SM walk chunks of 64 pooled key
// rows of one (sequence, KV head), c = blockIdx.x, + gridDim.x, ...  Each
// chunk (32 KB of pooled keys and the group's query rows) is copied into a
// three-stage shared-memory ring with cp.async while the previous chunks are
// scored, so the loads of one chunk overlap the arithmetic of the others.
// The scores of a chunk are a small dense product, [64 rows x 128] x
// [128 x G heads], on the tf32 tensor cores at fp32-level accuracy
// (sa_ix::score_chunk).  D = 128.
constexpr int kMaxGroup = 16;
constexpr int kRows = 64;                     // pooled rows per chunk
constexpr int kStages = 3;
constexpr int kScoreThreads = 128;
constexpr int kScoreCtasPerSm = 2;
constexpr int kMaxKvHeads = 256;              // per-group head masks kept in shared memory

struct ScoreStage {
  float4 k[kRows][32];                        // 64 rows x 128 floats, chunks swizzled
  uint2 q[kMaxGroup][32];                     // the group's queries, bf16
};

__global__ void __launch_bounds__(kScoreThreads, kScoreCtasPerSm)
    decode_scores_kernel(const __nv_bfloat16* __restrict__ q, const float* __restrict__ kbar,
                         float* __restrict__ scores, int Bt, int Hq, int Hkv, int group, int nb,
                         int stride, float scale, const uint8_t* __restrict__ kinds,
                         const int32_t* __restrict__ gran, int size) {
  constexpr int D = 128;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ScoreStage* st = reinterpret_cast<ScoreStage*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (nb + kRows - 1) / kRows;   // chunks per (sequence, KV head)
  const int total = Bt * Hkv * per;
  // each group's heads this pass scores: all, or the retrieval heads of `size`
  __shared__ uint32_t gmask[kMaxKvHeads];
  for (int g = tid; g < Hkv; g += kScoreThreads) {
    uint32_t m = 0;
    for (int hh = 0; hh < group; ++hh) {
      const int h = g * group + hh;
      if (!gran || (kinds[h] != SA_HEAD_STREAMING && gran[h] == size)) m |= 1u << hh;
    }
    gmask[g] = m;
  }
  __syncthreads();
  // the CTA's chunks in order, those of groups with no head to score skipped
  auto next_chunk = [&](int c) -> int {
    if (c >= total) return total;
    for (c += gridDim.x; c < total; c += gridDim.x)
      if (gmask[(c / per) % Hkv]) return c;
    return total;
  };
  auto issue = [&](int c, int s) {
    if (c < total) {
      const int bg = c / per, r0 = (c - bg * per) * kRows;
      const int rows = min(kRows, nb - r0);
      const float4* src = reinterpret_cast<const float4*>(kbar + (size_t(bg) * nb + r0) * D);
      for (int e = tid; e < rows * 32; e += kScoreThreads) {
        const int r = e >> 5;
        cp_async16(&st[s].k[r][swz<32>(r, e & 31)], src + e);
      }
      const int b = bg / Hkv, g = bg - b * Hkv;
      const uint2* qs = reinterpret_cast<const uint2*>(q + (size_t(b) * Hq + g * group) * D);
      for (int e = tid; e < group * 32; e += kScoreThreads)
        cp_async8(&st[s].q[e >> 5][e & 31], qs + e);
    }
    cp_async_commit();                        // empty groups keep the count uniform
  };
  // chunk k of this CTA's sequence goes to stage k % kStages; ahead[x] is
  // chunk k + x (issued, x < kStages - 1), and chunk k + kStages - 1 is
  // issued into the stage chunk k - 1 left
  int ahead[kStages - 1];
  ahead[0] = next_chunk(int(blockIdx.x) - int(gridDim.x));
  issue(ahead[0], 0);
#pragma unroll
  for (int x = 1; x < kStages - 1; ++x) {
    ahead[x] = next_chunk(ahead[x - 1]);
    issue(ahead[x], x);
  }
  for (int k = 0; ahead[0] < total; ++k) {
    const int cur = ahead[0];
    const int nxt = next_chunk(ahead[kStages - 2]);
    issue(nxt, (k + kStages - 1) % kStages);
    cp_async_wait_group<kStages - 1>();       // this thread's copies of chunk k landed
    __syncthreads();                          // ... and every thread's
    const ScoreStage& sg = st[k % kStages];
    const int bg = cur / per, r0 = (cur - bg * per) * kRows;
    const int b = bg / Hkv, g = bg - b * Hkv;
    const uint32_t hmask = gmask[g];
    if (r0 + 16 * warp < nb) {
      score_chunk(sg.k, sg.q, group, warp, lane, [&](int hh, int r, float v) {
        const int j = r0 + r;
        if (((hmask >> hh) & 1u) && j < nb)
          scores[(size_t(b) * Hq + g * group + hh) * stride + j] = v * scale;
      });
    }
    __syncthreads();                          // stage k % kStages is free again
#pragma unroll
    for (int x = 0; x < kStages - 2; ++x) ahead[x] = ahead[x + 1];
    ahead[kStages - 2] = nxt;
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
  const int smem = 2 * kT * d * int(sizeof(float));
  cudaError_t e;
  if (d == 128) {
    e = cudaFuncSetAttribute(prefill_scores_kernel<128>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      prefill_scores_kernel<128><<<grid, 256, smem, st>>>(qbar, kbar, scores, nb, group, scale);
  } else if (d == 64) {
    e = cudaFuncSetAttribute(prefill_scores_kernel<64>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      prefill_scores_kernel<64><<<grid, 256, smem, st>>>(qbar, kbar, scores, nb, group, scale);
  } else {
    return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_prefill_index(const void* q, const void* k, float* scores, float* ws, int Hq,
                                 int Hkv, int nb, int block, int d, cudaStream_t st) {
  float* qbar = ws;
  float* kbar = qbar + size_t(Hq) * nb * d;
  cudaError_t e = launch_pool(q, qbar, int64_t(Hq) * nb, block, d, st);
  if (e == cudaSuccess) e = launch_pool(k, kbar, int64_t(Hkv) * nb, block, d, st);
  if (e == cudaSuccess)
    e = launch_prefill_scores(qbar, kbar, scores, Hq, Hq / Hkv, nb, d,
                              float(1.0 / std::sqrt(double(d))), st);
  return e;
}

cudaError_t launch_decode_scores(const void* q, const float* kbar, float* scores, int Bt, int Hq,
                                 int group, int nb, int d, float scale, cudaStream_t st,
                                 int stride, const uint8_t* kinds, const int32_t* gran,
                                 int size) {
  if (d != 128 || group > kMaxGroup) return cudaErrorInvalidValue;
  if (gran && !kinds) return cudaErrorInvalidValue;
  const int Hkv = Hq / group;
  if (Hkv > kMaxKvHeads) return cudaErrorInvalidValue;
  const long long chunks = (long long)Bt * Hkv * ((nb + kRows - 1) / kRows);
  if (chunks == 0) return cudaSuccess;
  if (chunks >= (1ll << 30)) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int smem = int(kStages * sizeof(ScoreStage));
  e = cudaFuncSetAttribute(decode_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long slots = (long long)sms * kScoreCtasPerSm;
  const int grid = int(chunks < slots ? chunks : slots);
  decode_scores_kernel<<<grid, kScoreThreads, smem, st>>>(
      static_cast<const __nv_bfloat16*>(q), kbar, scores, Bt, Hq, Hkv, group, nb,
      stride > 0 ? stride : nb, scale, kinds, gran, size);
  return cudaGetLastError();
}

}  // namespace sa_k
