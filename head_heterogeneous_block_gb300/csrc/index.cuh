// Index step building blocks shared by the score kernels: cp.async copies,
// the shared-memory swizzle, and fp32-level dot products on the tf32 tensor
// cores (each fp32 operand split into a tf32 part and the rest).
//
// score_chunk is the decode scoring of one staged chunk of pooled keys; the
// score kernel and the fused score-and-select kernel both call it, so the two
// compute bit-identical scores.
#pragma once

#include <cstdint>

namespace sa_ix {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
// 16-byte chunk c of a row of kC chunks sits at c ^ 4(r mod kC/4): the rows
// a quarter-warp reads together land on different banks
template <int kC>
__device__ __forceinline__ int swz(int r, int c) { return c ^ ((r & (kC / 4 - 1)) << 2); }

// x = hi + lo with hi a tf32 value (the 10 leading mantissa bits of x)
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = __float_as_uint(x) & 0xFFFFE000u;
  lo = __float_as_uint(x - __uint_as_float(hi));
}

// D += A . B for one m16n8k8 tile (A 16x8 row-major, B 8x8 column-major, tf32)
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Decode scores of one staged chunk of 64 pooled key rows (d = 128):
// k[r][c] holds row r's 16-byte chunk c at swz<32>(r, c); q[x] is query head
// x of the group (bf16, 32 x 8 bytes).  Warp w (0..3) takes rows 16w .. 16w+16
// as m16n8k8 tf32 MMAs, 8 heads per tile, fp32 accumulation.  A pooled key x
// is split into x_hi (tf32) and x_lo = x - x_hi (exact in fp32; the MMA reads
// its top tf32 bits), both multiplied by the query (bf16, exact in tf32) into
// separate accumulators that are added at the end, so the products keep
// about 20 bits of x.  The k order inside an MMA is permuted (lane t of a quad
// takes dimensions 16m + 4t .. +4, two k-steps), so every shared-memory read is
// conflict-free.  emit(x, r, s) receives the unscaled score of head x < group
// and row r for every row of the warp's 16 (rows past the staged ones hold
// stale data: the caller drops them).
template <typename Emit>
__device__ __forceinline__ void score_chunk(const float4 (*k)[32], const uint2 (*q)[32], int group,
                                            int warp, int lane, Emit&& emit) {
  const int gq = lane >> 2, tq = lane & 3;    // MMA fragment coordinates
  const int ra = 16 * warp + gq;              // this lane's rows: ra and ra + 8
  for (int n0 = 0; n0 < group; n0 += 8) {     // 8 heads per tile
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acl[4] = {0.f, 0.f, 0.f, 0.f};
    const int hn = n0 + gq;                   // the head of this lane's B column
#pragma unroll
    for (int m = 0; m < 8; ++m) {             // dimensions 16m .. 16m + 16: two k-steps
      const float4 xa = k[ra][swz<32>(ra, 4 * m + tq)];
      const float4 xb = k[ra + 8][swz<32>(ra + 8, 4 * m + tq)];
      uint2 qb = make_uint2(0u, 0u);
      if (hn < group) qb = q[hn][4 * m + tq];
      const uint32_t q0 = qb.x << 16, q1 = qb.x & 0xFFFF0000u;
      const uint32_t q2 = qb.y << 16, q3 = qb.y & 0xFFFF0000u;
      uint32_t hi[4], lo[4];
      // k-step 2m: dimensions +0 (k = t) and +1 (k = t + 4)
      split_tf32(xa.x, hi[0], lo[0]);
      split_tf32(xb.x, hi[1], lo[1]);
      split_tf32(xa.y, hi[2], lo[2]);
      split_tf32(xb.y, hi[3], lo[3]);
      mma_tf32(acc, hi, q0, q1);
      mma_tf32(acl, lo, q0, q1);
      // k-step 2m + 1: dimensions +2 and +3
      split_tf32(xa.z, hi[0], lo[0]);
      split_tf32(xb.z, hi[1], lo[1]);
      split_tf32(xa.w, hi[2], lo[2]);
      split_tf32(xb.w, hi[3], lo[3]);
      mma_tf32(acc, hi, q2, q3);
      mma_tf32(acl, lo, q2, q3);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] += acl[e];
    // acc: rows ra (0, 1) and ra + 8 (2, 3), heads n0 + 2t and n0 + 2t + 1
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int hh = n0 + 2 * tq + (e & 1);
      if (hh < group) emit(hh, ra + ((e & 2) ? 8 : 0), acc[e]);
    }
  }
}

}  // namespace sa_ix
