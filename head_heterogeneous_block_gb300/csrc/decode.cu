// Decode attention over the selected KV blocks (HBM-bound).
//
// One CTA per (sequence, query head), four warps.  A head's selected blocks
// are split into 16-token units (a block of g tokens is g/16 units; the
// default B = 32 is two); warp w takes units w, w+4, w+8, ...  Each warp
// streams its units through two shared-memory stages of its own: a unit's
// 16 key rows and 16 value rows (4 KB each, contiguous in the cache) arrive
// by two bulk asynchronous copies on the stage's mbarrier, and the copies of
// the warp's next unit are in flight while it works on the current one, so
// every warp keeps loads outstanding all the time (three CTAs per SM: 96 KB
// in flight per SM).  Lane l owns dimensions [4l, 4l+4) of every row: it
// forms 16 partial dot products over its four dimensions, a reduce-scatter
// over the warp (16 shuffles) leaves the score of row r in lanes r and
// r + 16, the warp keeps an online softmax and accumulates P V in the same
// dimension layout.  The four partial states are merged by their
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
constexpr int kU = 16;                       // tokens per unit
constexpr int kStages = 2;                   // per warp
constexpr uint32_t kUnitBytes = kU * kD * 2; // one unit of K (or of V)
static_assert(kD == 4 * 32, "lane l <-> dims [4l, 4l+4)");

struct DecodeSmem {
  uint2 k[kWarps * kStages][kU][32];         // stage s = 2 * warp + (unit count & 1)
  uint2 v[kWarps * kStages][kU][32];
  uint64_t full[kWarps * kStages];
};

__global__ void __launch_bounds__(kWarps * 32, 3) decode_attention_kernel(sa_k::DecodeArgs a,
                                                                       float scale_log2) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem& sh = *reinterpret_cast<DecodeSmem*>(smem_raw);
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
  const uint64_t limit = a.wait_ns ? a.wait_ns : sa_dev::kWaitLimitNs;

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
  // the warp's c-th unit (x = warp + c * kWarps) goes to stage 2 * warp + (c & 1)
  auto issue = [&](int x, int c) {
    const size_t t0 = unit_start(x);
    const int s = kStages * warp + (c & 1);
    if (lane == 0) {
      sa_dev::mbar_arrive_expect_tx(&sh.full[s], 2 * kUnitBytes);
      sa_dev::bulk_load(&sh.k[s][0][0], K + t0 * kD, kUnitBytes, &sh.full[s]);
      sa_dev::bulk_load(&sh.v[s][0][0], V + t0 * kD, kUnitBytes, &sh.full[s]);
    }
  };
  int issued = 0, used = 0;                   // this warp's units issued and consumed
  for (; issued < kStages && warp + issued * kWarps < units; ++issued)
    issue(warp + issued * kWarps, issued);
  bool ok = true;
  for (int x = warp; x < units; x += kWarps) {
    const int s = kStages * warp + (used & 1);
    if (!sa_dev::wait_all(&sh.full[s], (used >> 1) & 1, nullptr, limit)) {
      ok = false;
      break;
    }
    uint2 kv[kU], vv[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) kv[u] = sh.k[s][u][lane];
#pragma unroll
    for (int u = 0; u < kU; ++u) vv[u] = sh.v[s][u][lane];
    ++used;
    // every lane has its rows in registers: the stage takes the warp's unit
    // after next (the async proxy writes it after these generic reads)
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
    if (lane == 0) atomicOr(a.dev_status, SA_DEV_TIMEOUT);
    // copies still in flight land before the CTA's shared memory goes
    if (lane == 0)
      for (int c = used; c < issued; ++c)
        sa_dev::mbar_wait(&sh.full[kStages * warp + (c & 1)], (c >> 1) & 1, nullptr);
    __syncwarp();
    m = -INFINITY;                            // this warp's part is not merged
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
  constexpr int kSmem = int(sizeof(DecodeSmem));
  cudaError_t e = cudaFuncSetAttribute(decode_attention_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  decode_attention_kernel<<<rows, kWarps * 32, kSmem, st>>>(a, scale_log2);
  return cudaGetLastError();
}

}  // namespace sa_k
