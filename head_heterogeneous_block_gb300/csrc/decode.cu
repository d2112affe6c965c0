// Decode attention over the selected KV blocks (HBM-bound).
//
// One CTA per (sequence, query head), four warps, each warp with two
// shared-memory stages of its own (three CTAs per SM: 96 KB in flight per
// SM).  The row's work is sa_da::attend_warp (decode_attn.cuh): 16-token
// units streamed by bulk copies, scores by a warp reduce-scatter, an online
// softmax per warp, and the four warps' states merged by their log-sum-exp.
// Streaming and retrieval heads differ only in their block lists, and
// retrieval heads may select at their own block size ("Riepilogo Tecnico:
// Fluxion", "Intuizioni Chiave" 2).

#include <cuda_bf16.h>

#include <cstdint>

#include "decode_attn.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "sparse_attn.h"

namespace {

using sa_da::kB;
using sa_da::kD;
using sa_da::kU;
using sa_da::kWarps;
constexpr int kStages = 2;                   // per warp

struct DecodeSmem {
  uint2 k[kWarps * kStages][kU][32];         // warp w's stages are 2w and 2w + 1
  uint2 v[kWarps * kStages][kU][32];
  uint64_t full[kWarps * kStages];
};

__global__ void __launch_bounds__(kWarps * 32, 3) decode_attention_kernel(sa_k::DecodeArgs a,
                                                                       float scale_log2) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem& sh = *reinterpret_cast<DecodeSmem*>(smem_raw);
  __shared__ float sq[kD];
  __shared__ sa_da::Merge mg;
  // rows may be restricted to a list of heads (one kind of head)
  const int row = a.heads ? (int(blockIdx.x) / a.nh) * a.Hq + a.heads[blockIdx.x % a.nh]
                          : int(blockIdx.x);
  const int b = row / a.Hq, h = row % a.Hq;
  const int g = h / (a.Hq / a.Hkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this head's block size (a multiple of 16) and block count
  int gsz = a.gran ? a.gran[h] : kB;
  if (gsz < kU || (gsz % kU) != 0 || a.L % gsz != 0) gsz = kB;

  if (threadIdx.x < kWarps * kStages) sa_dev::mbar_init(&sh.full[threadIdx.x], 1);
  sa_dev::fence_mbar_init();
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + size_t(row) * kD;
  for (int c = threadIdx.x; c < kD; c += kWarps * 32) sq[c] = __bfloat162float(q[c]);
  __syncthreads();

  int n = a.cnt[row];
  if (n < 1 || n > a.kmax) {
    if (threadIdx.x == 0) atomicOr(a.dev_status, SA_DEV_BAD_COUNT);
    n = max(1, min(n, a.kmax));
  }
  const size_t head_off = (size_t(b) * a.Hkv + g) * size_t(a.L) * kD;
  sa_da::Row r;
  r.K = static_cast<const __nv_bfloat16*>(a.k) + head_off;
  r.V = static_cast<const __nv_bfloat16*>(a.v) + head_off;
  r.list = a.idx + size_t(row) * a.kmax;
  r.n = n;
  r.gsz = gsz;
  r.per = gsz / kU;                           // units per block
  r.nb = a.L / gsz;
  r.limit = a.wait_ns ? a.wait_ns : sa_dev::kWaitLimitNs;
  r.dev_status = a.dev_status;
  const float q4[4] = {sq[4 * lane], sq[4 * lane + 1], sq[4 * lane + 2], sq[4 * lane + 3]};
  float m, l, o[4];
  uint32_t base = 0;
  sa_da::attend_warp<kStages>(r, q4, &sh.k[kStages * warp], &sh.v[kStages * warp],
                              &sh.full[kStages * warp], base, warp, lane, scale_log2, m, l, o);
  sa_da::post_state(mg, warp, lane, m, l, o);
  __syncthreads();
  if (warp == 0) sa_da::merge_store(mg, lane, size_t(row), a.o, a.out_f32 != 0, a.lse);
}

}  // namespace

namespace sa_k {

cudaError_t launch_decode_attention(const DecodeArgs& a, cudaStream_t st) {
  if (a.d != kD || a.B != kB) return cudaErrorInvalidValue;
  if (a.heads && a.nh <= 0) return cudaErrorInvalidValue;
  const int rows = a.Bt * (a.heads ? a.nh : a.Hq);
  if (rows == 0) return cudaSuccess;
  const float scale_log2 = sa_da::kScaleLog2;
  constexpr int kSmem = int(sizeof(DecodeSmem));
  cudaError_t e = cudaFuncSetAttribute(decode_attention_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  decode_attention_kernel<<<rows, kWarps * 32, kSmem, st>>>(a, scale_log2);
  return cudaGetLastError();
}

}  // namespace sa_k
