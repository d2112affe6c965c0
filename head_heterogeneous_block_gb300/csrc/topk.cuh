// Exact top-k of one row of fp32 block scores, for the select kernels.
//
// The rule is the Select step's ("Riepilogo Tecnico: Fluxion", "Intuizioni
// Chiave" 1 and 2): of the candidate blocks 1..last keep the `need` with the
// highest scores, ties to the lower index.  The threshold is found by radix
// selection over the order-preserving bit pattern of the scores: at most four
// passes, each a 256-bin shared-memory histogram of the next 8 bits among the
// candidates that still match the prefix.  The result is the exact need-th
// largest score T: every candidate above T is kept, and of those equal to T
// the lowest indices.  mark_top marks the kept blocks in a shared-memory
// bitmap, which emit_ascending writes out in ascending order; emit_top writes
// a row's list straight from the threshold.
//
// A row is handled by a group of kT threads (a whole CTA, or one warpgroup of
// it) that synchronise on their own named barrier, so several rows can be
// selected at once in one CTA.  In each pass one warp scans the histogram and
// hands the bin on through shared memory.
//
// Candidate layout: thread t of the group holds the candidates
// j = 1 + t + r*kT, r < kPer, as order bits u[r] (entries with j > last are
// ignored).  Every thread of the group calls these functions with its index
// t in the group and the group's barrier (bar.sync id, kT threads, id 0, 1
// or 2; id 0 with kT = the CTA's size is __syncthreads).
#pragma once

#include <cstdint>

namespace sa_topk {

// Monotone map of fp32 to uint32: a > b as floats iff bits(a) > bits(b).
__device__ __forceinline__ uint32_t order_bits(float s) {
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// bar.sync on barrier `bar` (0, 1 or 2) for kT threads; the ids are
// immediates so that a kernel reserves only the barriers it names
template <int kT>
__device__ __forceinline__ void group_sync(int bar) {
  if (bar == 0)
    asm volatile("bar.sync 0, %0;" ::"n"(kT) : "memory");
  else if (bar == 1)
    asm volatile("bar.sync 1, %0;" ::"n"(kT) : "memory");
  else
    asm volatile("bar.sync 2, %0;" ::"n"(kT) : "memory");
}

struct Scratch {
  uint32_t hist[256];
  uint32_t cnt[256];       // per (candidate column r, warp): counts of a class of candidates
  uint32_t ctl[4];         // the threshold bin of a pass
};

// The threshold of a row: candidates with order bits above T (or, when
// !ties, at least T) are kept, and when ties, the `need` lowest-indexed of
// those equal to T.
struct Threshold {
  uint32_t T;
  uint32_t need;
  bool ties;
};

// Adds to hist the next 8 bits (at `shift`) of the candidates of 1..last
// whose higher bits equal prefix.
template <int kT, int kPer, bool kMatch>
__device__ __forceinline__ void count_pass(const uint32_t (&u)[kPer], int last, uint32_t prefix,
                                           uint32_t mask, int shift, uint32_t* hist, int tid) {
  const int lane = tid & 31;
  if (kMatch && shift == 24) {
    // the top byte (sign and high exponent bits) puts most scores in a few
    // bins: one atomic per bin and warp instead of per lane
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int j = 1 + tid + r * kT;
      const uint32_t bin = j <= last ? (u[r] >> 24) : 256u;
      const uint32_t same = __match_any_sync(0xffffffffu, bin);
      if (bin < 256u && lane == __ffs(same) - 1) atomicAdd(&hist[bin], __popc(same));
    }
  } else {
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int j = 1 + tid + r * kT;
      if (j <= last && (u[r] & mask) == prefix) atomicAdd(&hist[(u[r] >> shift) & 255u], 1u);
    }
  }
}

// One warp finds the bin holding the need-th largest: lane l holds bins
// 255-8l .. 248-8l (descending), a scan over the lanes, then the lane whose
// range holds it picks the bin.  Every lane gets the bin, the count above it
// and the count in it.
__device__ __forceinline__ void scan_bins(const uint32_t* hist, uint32_t need, int lane,
                                          uint32_t& bin, uint32_t& above, uint32_t& in_bin) {
  uint32_t c[8], local = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    c[k] = hist[255 - 8 * lane - k];
    local += c[k];
  }
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const uint32_t excl = incl - local;
  const bool here = excl < need && need <= incl;
  bin = above = in_bin = 0;
  if (here) {
    uint32_t acc = excl;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (acc + c[k] >= need) {
        bin = uint32_t(255 - 8 * lane - k);
        above = acc;
        in_bin = c[k];
        break;
      }
      acc += c[k];
    }
  }
  const int src = __ffs(__ballot_sync(0xffffffffu, here)) - 1;
  bin = __shfl_sync(0xffffffffu, bin, src);
  above = __shfl_sync(0xffffffffu, above, src);
  in_bin = __shfl_sync(0xffffffffu, in_bin, src);
}

// Finds the threshold that keeps the `need` (>= 1, < number of candidates)
// highest candidates of 1..last, ties to the lower index.  kPer * kT <= 4096.
template <int kT, int kPer, bool kMatch>
__device__ __forceinline__ Threshold find_threshold(const uint32_t (&u)[kPer], int last,
                                                    uint32_t need, Scratch& s, int tid, int bar) {
  const int lane = tid & 31;
  uint32_t prefix = 0, mask = 0, eq_total = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += kT) s.hist[b] = 0u;
    group_sync<kT>(bar);
    count_pass<kT, kPer, kMatch>(u, last, prefix, mask, shift, s.hist, tid);
    group_sync<kT>(bar);
    if (tid < 32) {
      uint32_t bin, above, in_bin;
      scan_bins(s.hist, need, lane, bin, above, in_bin);
      if (lane == 0) {
        s.ctl[0] = bin;
        s.ctl[1] = above;
        s.ctl[2] = in_bin;
      }
    }
    group_sync<kT>(bar);
    need -= s.ctl[1];
    eq_total = s.ctl[2];
    prefix |= s.ctl[0] << shift;
    mask |= 0xFFu << shift;
    group_sync<kT>(bar);
    // the bin holds exactly the candidates still needed: all of them, and
    // everything above, are kept (u >= prefix, lower bits zero)
    if (eq_total == need) break;
  }
  return Threshold{prefix, need, eq_total != need};
}

// Marks in `bits` the `need` (>= 1, < number of candidates) highest
// candidates of 1..last, ties to the lower index.  Ends without a barrier:
// synchronise the group before reading `bits`.  kPer * kT <= 4096.
template <int kT, int kPer, bool kMatch>
__device__ __forceinline__ void mark_top(const uint32_t (&u)[kPer], int last, uint32_t need_in,
                                         uint32_t* bits, Scratch& s, int tid, int bar) {
  static_assert(kPer * (kT / 32) <= 128, "tie counts");
  constexpr int kWarps = kT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  const Threshold th = find_threshold<kT, kPer, kMatch>(u, last, need_in, s, tid, bar);
  const uint32_t T = th.T, need = th.need;
  if (!th.ties) {
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int j = 1 + tid + r * kT;
      if (j <= last && u[r] >= T) atomicOr(&bits[j >> 5], 1u << (j & 31));
    }
    return;
  }
  // ties straddle the threshold: every candidate above T, and the `need`
  // lowest-indexed ones equal to T.  Candidate (t, r) has index 1 + t + r*kT,
  // so the equal ones before it are those of the columns r' < r and those of
  // column r at lower t: column by column, two barriers each (the fewest
  // registers; ties at the threshold are rare)
  uint32_t taken = 0;
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int j = 1 + tid + r * kT;
    const bool valid = j <= last;
    const bool eq = valid && u[r] == T;
    const uint32_t m = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) s.cnt[warp] = __popc(m);
    group_sync<kT>(bar);
    uint32_t before = taken;
    for (int w = 0; w < warp; ++w) before += s.cnt[w];
    before += __popc(m & ((1u << lane) - 1u));
    if (valid && (u[r] > T || (eq && before < need))) atomicOr(&bits[j >> 5], 1u << (j & 31));
    for (int w = 0; w < kWarps; ++w) taken += s.cnt[w];
    group_sync<kT>(bar);
  }
}

// Writes the blocks marked in bits (blocks 0..i; bits past i are zero) in
// ascending order to out[0 .. kmax) and pads with -1.  Returns the number of
// marked blocks (to every thread of the group).  Warp w takes a contiguous
// range of the bitmap's words: counts, one barrier, a prefix over the warps,
// then ballots per word.  The caller synchronises the group before reusing
// `bits` or `s`.
template <int kT>
__device__ __forceinline__ int emit_ascending(const uint32_t* bits, int i, int32_t* out, int kmax,
                                              Scratch& s, int tid, int bar) {
  constexpr int kWarps = kT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  const int nw = (i + 32) / 32;             // words holding blocks 0..i
  const int wper = (nw + kWarps - 1) / kWarps;
  const int w0 = min(nw, warp * wper), w1 = min(nw, w0 + wper);
  uint32_t mine = 0;
  for (int x = w0 + lane; x < w1; x += 32) mine += __popc(bits[x]);
  mine = __reduce_add_sync(0xffffffffu, mine);
  if (lane == 0) s.cnt[warp] = mine;
  group_sync<kT>(bar);
  int written = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int n = int(s.cnt[w]);
    if (w < warp) written += n;
    total += n;
  }
  for (int x = w0; x < w1; ++x) {
    const bool on = ((bits[x] >> lane) & 1u) != 0;
    const uint32_t m = __ballot_sync(0xffffffffu, on);
    const int pos = written + __popc(m & ((1u << lane) - 1u));
    if (on && pos < kmax) out[pos] = 32 * x + lane;
    written += __popc(m);
  }
  for (int t = total + tid; t < kmax; t += kT) out[t] = -1;
  return total;
}

// Writes row i = last + 1's list straight from its threshold: block 0, the
// kept candidates of 1..last in ascending order, block i; pads with -1 to
// kmax and returns the list's length (to every thread of the group).  A
// kept candidate's position is 1 + the kept candidates before it in index
// order: those of the columns r' < r, then those of column r at lower t,
// counted per (column, warp) with ballots, with one barrier.  The caller
// synchronises the group before reusing `s`.
template <int kT, int kPer>
__device__ __forceinline__ int emit_top(const uint32_t (&u)[kPer], int last, Threshold th,
                                        int32_t* out, int kmax, Scratch& s, int tid, int bar) {
  static_assert(2 * kPer * (kT / 32) <= 256, "column counts");
  constexpr int kWarps = kT / 32;
  constexpr int kEq = kPer * kWarps;        // equal-to-T counts follow the above-T ones
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t lt = (1u << lane) - 1u;
  auto above = [&](int r) {
    return 1 + tid + r * kT <= last && (th.ties ? u[r] > th.T : u[r] >= th.T);
  };
  auto equal = [&](int r) { return 1 + tid + r * kT <= last && th.ties && u[r] == th.T; };
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const uint32_t am = __ballot_sync(0xffffffffu, above(r));
    const uint32_t em = __ballot_sync(0xffffffffu, equal(r));
    if (lane == 0) {
      s.cnt[r * kWarps + warp] = __popc(am);
      s.cnt[kEq + r * kWarps + warp] = __popc(em);
    }
  }
  group_sync<kT>(bar);
  uint32_t a_before = 0, e_before = 0;
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    uint32_t a_col = 0, e_col = 0, a_mine = a_before, e_mine = e_before;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t na = s.cnt[r * kWarps + w], ne = s.cnt[kEq + r * kWarps + w];
      a_col += na;
      e_col += ne;
      if (w < warp) {
        a_mine += na;
        e_mine += ne;
      }
    }
    // the ballots again rather than kept (registers are the scarcer)
    const bool ab = above(r), eq = equal(r);
    a_mine += __popc(__ballot_sync(0xffffffffu, ab) & lt);
    e_mine += __popc(__ballot_sync(0xffffffffu, eq) & lt);
    if (ab || (eq && e_mine < th.need)) {
      const uint32_t pos = 1 + a_mine + min(e_mine, th.need);
      if (pos < uint32_t(kmax)) out[pos] = 1 + tid + r * kT;
    }
    a_before += a_col;
    e_before += e_col;
  }
  const int total = 2 + int(a_before + min(e_before, th.need));
  if (tid == 0) {
    out[0] = 0;
    if (total - 1 < kmax) out[total - 1] = last + 1;
  }
  for (int t = total + tid; t < kmax; t += kT) out[t] = -1;
  return total;
}

}  // namespace sa_topk
