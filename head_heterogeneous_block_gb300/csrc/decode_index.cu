// Decode Index and Select of the retrieval heads in one launch.
//
// A decode step's retrieval heads score every pooled key block of their
// sequence (Index) and keep the top-k_h of them with the sink block and the
// last block (Select): "Riepilogo Tecnico: Fluxion", "Intuizioni Chiave" 1
// and 2; the Index / Select split is Spin's ("Abstracción de Partición
// Unificada").  The two steps as separate launches leave the GPU nearly idle
// between them: the scores go out to memory, and the selection starts only
// when the last score is written.  Here one thread-block cluster per
// (sequence, KV group) does both:
//
//   1. Each of the cluster's kCP CTAs streams its share of the group's pooled
//      keys (rows [rank*R, rank*R + R)) through a three-stage cp.async ring and
//      scores them for the group's retrieval heads on the tf32 tensor cores
//      (sa_ix::score_chunk, the routine of the separate score kernel, so the
//      scores are bit-identical).  Scores stay in the CTA's shared memory
//      (and go to global memory only when the caller asks for them).
//   2. A cluster barrier; then each retrieval head of the group is taken by
//      one warpgroup of one CTA, which gathers the head's score row from the
//      cluster's CTAs (16-byte distributed shared memory loads) into its own
//      shared memory, finds the row's threshold as the select kernel does
//      (sa_topk::find_threshold) and writes the list straight from it
//      (sa_topk::emit_top).
//   3. A second cluster barrier, so no CTA exits while another reads its
//      scores.
//
// The one-launch decode step (kAttend) goes on where the separate calls would
// launch the attention: the warpgroup that selected a retrieval head attends
// it at once (sa_da::attend_warp, the decode attention kernel's routine, with
// one stage per warp in the chunk ring), and the group's streaming heads, whose
// lists are block 0 and the last window_blocks blocks, are dealt to the other
// warpgroups.  No head waits for the others' selection or for a launch, so
// the heads that attend keep HBM busy while others still select.
//
// Every wait is a hardware barrier of the CTA or the cluster, whose CTAs the
// cluster launch schedules together, or a cp.async group wait; no CTA spins
// on memory another writes.  d = 128, G <= 16, nb <= 4096.

#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "decode_attn.cuh"
#include "index.cuh"
#include "kernels.h"
#include "sparse_attn.h"
#include "topk.cuh"

namespace {

namespace cg = cooperative_groups;
using namespace sa_ix;

constexpr int kThreads = 256;       // all copy; warps 0-3 score; two warpgroups select
constexpr int kRows = 64;           // pooled rows per chunk (32 KB)
constexpr int kStages = 3;          // two chunks in flight
constexpr int kStageBytes = kRows * 32 * 16;
constexpr int kMaxGroup = 16;
constexpr int kAttnStage = 2 * int(sa_da::kUnitBytes);   // one unit of K and V per warp

// Dynamic shared memory: region 0, the group's queries [G][32] uint2, the
// scores [max_retrieval][R] fp32 (a row per retrieval head of the group, by
// its slot).  Region 0 holds the kStages chunk buffers while scoring; then
// the two warpgroups' gathered score rows and selection scratch, and (with
// kAttend) from attn_base on the eight warps' attention stages and the two
// warpgroups' merge areas.
__host__ __device__ constexpr int select_bytes(int per) {
  return 2 * per * 128 * 4 + 2 * int(sizeof(sa_topk::Scratch));
}
__host__ __device__ constexpr int attn_base(int per) { return (select_bytes(per) + 127) / 128 * 128; }
__host__ __device__ constexpr int region0_bytes(int per, bool attend) {
  const int ring = kStages * kStageBytes;
  const int att = attn_base(per) + 8 * kAttnStage + 2 * int(sizeof(sa_da::Merge));
  return ((attend && att > ring ? att : ring) + 127) / 128 * 128;
}
size_t smem_bytes(int group, int max_retrieval, int rows_per_cta, int per, bool attend) {
  return size_t(region0_bytes(per, attend)) + size_t(group) * 256 +
         size_t(max_retrieval) * size_t(rows_per_cta) * 4;
}

// The attention of decode row `row` by one warpgroup (warps wi = 0..3 of
// warpgroup wg), once its list and count are written and the warpgroup has
// passed its barrier: warp wg*4 + wi streams its units through its own stage
// at `att` + (wg*4 + wi) * kAttnStage, and the four states are merged in the
// warpgroup's merge area.
__device__ __forceinline__ void attend_row(const sa_k::IndexSelectArgs& a, size_t row,
                                           const uint2 (&qrow)[32], unsigned char* att,
                                           uint64_t* afull, uint32_t& abase, int wg, int wi,
                                           int lane, int gt, int bar) {
  const int w8 = wg * 4 + wi;
  int n = a.cnt[row];
  if (n < 1 || n > a.kmax) {
    if (gt == 0) atomicOr(a.dev_status, SA_DEV_BAD_COUNT);
    n = max(1, min(n, a.kmax));
  }
  const int b = int(row / size_t(a.Hq)), h = int(row % size_t(a.Hq));
  const size_t head_off = (size_t(b) * a.Hkv + h / a.group) * size_t(a.L) * sa_da::kD;
  sa_da::Row r;
  r.K = static_cast<const __nv_bfloat16*>(a.k) + head_off;
  r.V = static_cast<const __nv_bfloat16*>(a.v) + head_off;
  r.list = a.idx + row * a.kmax;
  r.n = n;
  r.gsz = sa_da::kB;
  r.per = sa_da::kB / sa_da::kU;
  r.nb = a.L / sa_da::kB;
  r.limit = a.wait_ns ? a.wait_ns : sa_dev::kWaitLimitNs;
  r.dev_status = a.dev_status;
  // the query in fp32, exactly as bf16 widens
  const uint2 qv = qrow[lane];
  const float q4[4] = {__uint_as_float(qv.x << 16), __uint_as_float(qv.x & 0xFFFF0000u),
                       __uint_as_float(qv.y << 16), __uint_as_float(qv.y & 0xFFFF0000u)};
  auto sk = reinterpret_cast<uint2 (*)[sa_da::kU][32]>(att + w8 * kAttnStage);
  auto sv = reinterpret_cast<uint2 (*)[sa_da::kU][32]>(att + w8 * kAttnStage + sa_da::kUnitBytes);
  // the stage was last written or read by ordinary loads and stores (the
  // chunk ring, or this warp's previous row)
  sa_dev::fence_proxy_async_smem();
  float m, l, o[4];
  sa_da::attend_warp<1>(r, q4, sk, sv, &afull[w8], abase, wi, lane, sa_da::kScaleLog2, m, l, o);
  sa_da::Merge& mg = reinterpret_cast<sa_da::Merge*>(att + 8 * kAttnStage)[wg];
  sa_da::post_state(mg, wi, lane, m, l, o);
  sa_topk::group_sync<128>(bar);
  if (wi == 0) sa_da::merge_store(mg, lane, row, a.o, a.out_f32 != 0, a.lse);
  sa_topk::group_sync<128>(bar);                // the merge area is reused by the next row
}

template <int kCP, int kPer, bool kAttend>
__global__ void __launch_bounds__(kThreads, 2)
    decode_index_select_kernel(sa_k::IndexSelectArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = int(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.group, nb = a.nb, R = a.rows_per_cta;
  const int pair = int(blockIdx.x) / kCP;       // (sequence b, KV group g)
  const int b = pair / a.Hkv, g = pair - b * a.Hkv;
  // the group's retrieval heads; a group without any has nothing to do (the
  // same for every CTA of the cluster, so none waits at a barrier for it)
  uint32_t rmask = 0;
  for (int hh = 0; hh < G; ++hh)
    if (a.kinds[g * G + hh] != SA_HEAD_STREAMING) rmask |= 1u << hh;
  if (!kAttend && rmask == 0) return;

  // the heads' budgets, read while the scores stream in; retrieval head
  // number x of the group (in head order) has slot x, and (kAttend) the
  // streaming heads follow in head order.  Slot x is taken by CTA x % kCP,
  // warpgroup (x / kCP) % 2.
  __shared__ int32_t s_budget[kMaxGroup];
  __shared__ int32_t s_slot[kMaxGroup];
  __shared__ uint64_t s_afull[8];               // (kAttend) a warp's attention stage
  if (tid < G) {
    const uint32_t below = (1u << tid) - 1u;
    s_budget[tid] = a.budgets[g * G + tid];
    s_slot[tid] = ((rmask >> tid) & 1u)
                      ? __popc(rmask & below)
                      : (kAttend ? __popc(rmask) + __popc(~rmask & below) : -1);
  }

  constexpr int kRegion0 = region0_bytes(kPer, kAttend);
  float4 (*stage)[kRows][32] = reinterpret_cast<float4 (*)[kRows][32]>(smem_raw);
  uint2 (*qs)[32] = reinterpret_cast<uint2 (*)[32]>(smem_raw + kRegion0);
  float* sc = reinterpret_cast<float*>(smem_raw + kRegion0 + G * 256);
  const uint2* qg = reinterpret_cast<const uint2*>(a.q) + (size_t(b) * a.Hq + g * G) * 32;
  if constexpr (kAttend) {
    // every CTA attends with the group's queries, whether or not it scores
    if (tid < 8) sa_dev::mbar_init(&s_afull[tid], 1);
    sa_dev::fence_mbar_init();
    for (int e = tid; e < G * 32; e += kThreads) qs[e >> 5][e & 31] = qg[e];
    __syncthreads();
  }

  // ---- 1. scores of rows [r0, r0 + rows) for the retrieval heads
  const int r0 = rank * R;
  const int rows = max(0, min(nb - r0, R));
  const int nch = rmask ? (rows + kRows - 1) / kRows : 0;
  const float4* kb = reinterpret_cast<const float4*>(a.kbar) + (size_t(pair) * nb + r0) * 32;
  if (!kAttend && nch > 0) {
    // the queries join the first chunk's copy group
    for (int e = tid; e < G * 32; e += kThreads) cp_async8(&qs[e >> 5][e & 31], qg + e);
  }
  auto issue = [&](int c) {
    if (c < nch) {
      const int n = min(kRows, rows - c * kRows);
      const float4* src = kb + size_t(c) * kRows * 32;
      float4 (*dst)[32] = stage[c % kStages];
      for (int e = tid; e < n * 32; e += kThreads) {
        const int r = e >> 5;
        cp_async16(&dst[r][swz<32>(r, e & 31)], src + e);
      }
    }
    cp_async_commit();                          // empty groups keep the count uniform
  };
#pragma unroll
  for (int c = 0; c < kStages - 1; ++c) issue(c);
  for (int c = 0; c < nch; ++c) {
    issue(c + kStages - 1);                     // into the buffer chunk c - 1 left
    cp_async_wait_group<kStages - 1>();         // this thread's copies of chunk c landed
    __syncthreads();                            // ... and every thread's
    const int base = c * kRows;
    if (warp < kRows / 16 && base + 16 * warp < rows) {
      score_chunk(stage[c % kStages], qs, G, warp, lane, [&](int hh, int r, float v) {
        const int j = base + r;
        if (((rmask >> hh) & 1u) && j < rows) {
          const float s = v * a.scale;
          sc[__popc(rmask & ((1u << hh) - 1u)) * R + j] = s;   // the head's slot
          if (a.scores) a.scores[(size_t(b) * a.Hq + g * G + hh) * nb + r0 + j] = s;
        }
      });
    }
    __syncthreads();                            // chunk c's buffer is free again
  }
  cp_async_wait_all();

  // ---- 2. every CTA's scores are in its shared memory; up to 2 * kCP heads
  // are selected at once, each by 128 threads on the warpgroup's own named
  // barrier (a group without retrieval heads, which only attends, has no
  // scores to share: the same for every CTA of the cluster)
  if (rmask) cluster.sync();
  const int wg = warp >> 2, gt = tid & 127, bar = 1 + wg;
  float* srow = reinterpret_cast<float*>(smem_raw) + wg * (kPer * 128);
  sa_topk::Scratch& scr =
      reinterpret_cast<sa_topk::Scratch*>(smem_raw + 2 * kPer * 128 * 4)[wg];
  const int i = nb - 1;                         // a decode row is the last block's
  uint32_t abase = 0;                           // this warp's units through its stage
  for (int hh = 0; hh < G; ++hh) {
    const int slot = s_slot[hh];
    if (slot < 0 || slot % kCP != rank || (slot / kCP) % 2 != wg) continue;
    const size_t row = size_t(b) * a.Hq + g * G + hh;
    int32_t* out = a.idx + row * a.kmax;
    if (kAttend && !((rmask >> hh) & 1u)) {
      // a streaming head: block 0 and blocks lo..i, ascending, padded with -1
      const int lo = max(1, nb - a.window_blocks);
      const int total = 1 + max(0, i - lo + 1);
      for (int j = gt; j < a.kmax; j += 128) out[j] = j >= total ? -1 : (j == 0 ? 0 : lo + j - 1);
      if (gt == 0) a.cnt[row] = min(total, a.kmax);
      sa_topk::group_sync<128>(bar);
      if constexpr (kAttend) attend_row(a, row, qs[hh], smem_raw + attn_base(kPer), s_afull,
                                        abase, wg, warp & 3, lane, gt, bar);
      continue;
    }
    const int keep = min(s_budget[hh], i + 1);
    const int rest = keep - ((i == 0) ? 1 : 2);
    const int ncand = max(0, i - 1);            // blocks 1..i-1
    int total;
    if (rest >= ncand) {                        // every block
      for (int j = gt; j < a.kmax; j += 128) out[j] = j <= i ? j : -1;
      total = i + 1;
    } else if (rest == 0) {                     // blocks 0 and i
      for (int j = gt; j < a.kmax; j += 128) out[j] = j == 0 ? 0 : (j == 1 ? i : -1);
      total = 2;
    } else {
      // the head's scores, four blocks per 16-byte load (R is a multiple of
      // 64, so the four lie in one CTA)
      for (int j0 = 4 * gt; j0 < nb; j0 += 4 * 128) {
        const int owner = j0 / R;
        const float* src = cluster.map_shared_rank(sc, owner) + slot * R + (j0 - owner * R);
        *reinterpret_cast<float4*>(srow + j0) = *reinterpret_cast<const float4*>(src);
      }
      sa_topk::group_sync<128>(bar);
      uint32_t u[kPer];
#pragma unroll
      for (int r = 0; r < kPer; ++r) {
        const int j = 1 + gt + r * 128;
        u[r] = j <= i - 1 ? sa_topk::order_bits(srow[j]) : 0u;
      }
      const sa_topk::Threshold th =
          sa_topk::find_threshold<128, kPer, false>(u, i - 1, uint32_t(rest), scr, gt, bar);
      total = sa_topk::emit_top<128, kPer>(u, i - 1, th, out, a.kmax, scr, gt, bar);
    }
    if (gt == 0) a.cnt[row] = min(total, a.kmax);
    sa_topk::group_sync<128>(bar);              // the row buffer is reused by the next head
    if constexpr (kAttend) attend_row(a, row, qs[hh], smem_raw + attn_base(kPer), s_afull, abase,
                                      wg, warp & 3, lane, gt, bar);
  }

  // ---- 3. no CTA leaves while another may still read its scores
  if (rmask) cluster.sync();
}

template <int kCP, int kPer, bool kAttend>
cudaError_t launch_with(const sa_k::IndexSelectArgs& a, int grid, size_t smem, cudaStream_t st) {
  auto kern = decode_index_select_kernel<kCP, kPer, kAttend>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCP;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Cluster size and rows per CTA, then the launch: four CTAs per group when
// that fills the GPU, else eight; a warpgroup selects a row with 16
// candidates per thread up to 2048 blocks, else 32.
template <bool kAttend>
cudaError_t launch_clusters(const sa_k::IndexSelectArgs& args, cudaStream_t st) {
  if (args.group < 1 || args.group > kMaxGroup || args.nb < 1 || args.nb > 4096)
    return cudaErrorInvalidValue;
  const long long pairs = (long long)args.Bt * args.Hkv;
  if (pairs == 0) return cudaSuccess;
  if (pairs > (1ll << 26)) return cudaErrorInvalidValue;
  if (args.max_retrieval < (kAttend ? 0 : 1) || args.max_retrieval > args.group)
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int cp = pairs * 4 >= sms ? 4 : 8;
  sa_k::IndexSelectArgs a = args;
  const int per = (a.nb + cp - 1) / cp;
  a.rows_per_cta = (per + kRows - 1) / kRows * kRows;
  const int grid = int(pairs * cp);
  if (a.nb <= 16 * 128) {
    const size_t smem = smem_bytes(a.group, a.max_retrieval, a.rows_per_cta, 16, kAttend);
    return cp == 4 ? launch_with<4, 16, kAttend>(a, grid, smem, st)
                   : launch_with<8, 16, kAttend>(a, grid, smem, st);
  }
  const size_t smem = smem_bytes(a.group, a.max_retrieval, a.rows_per_cta, 32, kAttend);
  return cp == 4 ? launch_with<4, 32, kAttend>(a, grid, smem, st)
                 : launch_with<8, 32, kAttend>(a, grid, smem, st);
}

}  // namespace

namespace sa_k {

cudaError_t launch_decode_index_select(const IndexSelectArgs& args, cudaStream_t st) {
  return launch_clusters<false>(args, st);
}

cudaError_t launch_decode_step(const IndexSelectArgs& args, cudaStream_t st) {
  if (args.L != args.nb * sa_da::kB || !args.k || !args.v || !args.o || !args.dev_status)
    return cudaErrorInvalidValue;
  return launch_clusters<true>(args, st);
}

}  // namespace sa_k
