// Select step: per-row top-k_h block selection (one warp per row).
//
// A prefill row (h, i) keeps min(k_h, i+1) blocks: the sink block 0 ("Riepilogo
// Tecnico: Fluxion", "Intuizioni Chiave" 1), the diagonal block i, and the
// highest-scoring blocks of 1..i-1, ties to the lower index.  A decode
// retrieval head is the row i = nb-1; a decode streaming head keeps block 0
// and the last window_blocks blocks ("Intuizioni Chiave" 2).
//
// The candidates are packed into 64-bit keys (order-preserving bits of the
// fp32 score, then the complement of the block index, so larger keys win and
// equal scores prefer the lower index) and sorted descending with a warp
// bitonic sort in shared memory; the kept blocks are marked in a bitmap and
// written out in ascending order with warp ballots.

#include <cstdint>

#include "kernels.h"
#include "sparse_attn.h"

namespace {

constexpr int kWarps = 4;

__device__ __forceinline__ uint64_t score_key(float s, int j) {
  uint32_t u = __float_as_uint(s);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (uint64_t(u) << 32) | uint64_t(0xFFFFFFFFu - uint32_t(j));
}

__global__ void __launch_bounds__(kWarps * 32) select_kernel(sa_k::SelectArgs a, int n2) {
  extern __shared__ uint64_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* keys = sh + size_t(warp) * n2;
  uint32_t* bits = reinterpret_cast<uint32_t*>(sh + size_t(kWarps) * n2) + warp * (n2 / 32 + 1);
  const int row = blockIdx.x * kWarps + warp;
  if (row >= a.rows) return;

  int h, i;
  const float* srow;
  if (a.decode) {
    h = row % a.Hq;
    i = a.nb - 1;
    srow = a.scores + size_t(row) * a.nb;
  } else {
    h = row / a.nb;
    i = row - h * a.nb;
    srow = a.scores + (size_t(h) * a.nb + i) * a.nb;
  }
  const bool streaming = a.decode && a.kinds[h] == SA_HEAD_STREAMING;
  int32_t* out = a.idx + size_t(row) * a.kmax;

  // Membership of block j: mandatory, window, or chosen by score.
  const int nwords = (i + 1 + 31) / 32;
  for (int w = lane; w < nwords; w += 32) bits[w] = 0u;
  __syncwarp();

  int keep;
  if (streaming) {
    const int lo = max(1, a.nb - a.window_blocks);
    keep = 1 + (a.nb - lo);
    for (int j = lane; j <= i; j += 32)
      if (j == 0 || j >= lo) atomicOr(&bits[j >> 5], 1u << (j & 31));
  } else {
    keep = min(a.budgets[h], i + 1);
    const int mandatory = (i == 0) ? 1 : 2;
    const int rest = keep - mandatory;
    const int ncand = max(0, i - 1);        // blocks 1..i-1
    if (rest >= ncand) {
      for (int j = lane; j <= i; j += 32) atomicOr(&bits[j >> 5], 1u << (j & 31));
    } else {
      if (lane == 0) {
        atomicOr(&bits[0], 1u);
        atomicOr(&bits[i >> 5], 1u << (i & 31));
      }
      if (rest > 0) {
        int n = 1;
        while (n < ncand) n <<= 1;
        for (int t = lane; t < n; t += 32) keys[t] = (t < ncand) ? score_key(srow[t + 1], t + 1) : 0ull;
        __syncwarp();
        // bitonic sort, descending
        for (int k = 2; k <= n; k <<= 1) {
          for (int jj = k >> 1; jj > 0; jj >>= 1) {
            for (int t = lane; t < n; t += 32) {
              const int x = t ^ jj;
              if (x > t) {
                const uint64_t u = keys[t], v = keys[x];
                const bool down = (t & k) == 0;   // this pair's run sorts descending
                if (down ? (u < v) : (u > v)) {
                  keys[t] = v;
                  keys[x] = u;
                }
              }
            }
            __syncwarp();
          }
        }
        for (int t = lane; t < rest; t += 32) {
          const int j = int(0xFFFFFFFFu - uint32_t(keys[t] & 0xFFFFFFFFull));
          atomicOr(&bits[j >> 5], 1u << (j & 31));
        }
      }
    }
  }
  __syncwarp();

  // Emit ascending block indices, then pad with -1.
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
  (void)keep;
}

}  // namespace

namespace sa_k {

cudaError_t launch_select(const SelectArgs& a, cudaStream_t st) {
  if (a.rows == 0) return cudaSuccess;
  int n2 = 32;
  while (n2 < a.nb) n2 <<= 1;
  const size_t smem = size_t(kWarps) * n2 * sizeof(uint64_t) +
                      size_t(kWarps) * (n2 / 32 + 1) * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(smem));
  if (e != cudaSuccess) return e;
  const unsigned grid = unsigned((a.rows + kWarps - 1) / kWarps);
  select_kernel<<<grid, kWarps * 32, smem, st>>>(a, n2);
  return cudaGetLastError();
}

}  // namespace sa_k
