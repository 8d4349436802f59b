// Lagrangian multiple-choice-knapsack bit allocation on one thread-block
// cluster: the same solution as allocate_kernel (alloc.cuh), for pools whose
// thresholds fit in the cluster's shared memory.
//   [RDKV §2.1 objective; §2.2 reverse water-filling over {0,2,4,8,16}]
//
// Every upgrade item (u, k) has the multiplier theta = c_k key_u, an exact
// fp64 bit pattern (theta_bits).  Each CTA owns a contiguous range of units
// and keeps the TOP 32 BITS of every item's theta in shared memory (positive
// doubles order like their bit patterns).  lambda* is selected exactly:
//   1. two radix passes (11 + 11 bits) over the cached top halves; the
//      cost-weighted histograms are merged across the cluster through
//      distributed shared memory (reduce-scatter: CTA r sums bin slice r of
//      every CTA's histogram, then every CTA reads the slice that holds the
//      crossing);
//   2. the items sharing the selected top 22 bits (a band 2^-10 wide, a
//      handful in practice) are gathered, with their full 64-bit thetas, into
//      every CTA, which finishes the selection locally (four passes over the
//      remaining 42 bits) without further cluster traffic.  If there are more
//      of them than the gather buffer holds, the cluster passes continue over
//      the remaining bits instead.
// Ties at lambda* are resolved in unit order by a cluster-wide scan, then the
// budget-fix rounds take, one at a time, the best next step that still fits
// (theta descending, lowest unit first).  Synchronisation is the hardware
// cluster barrier only (no global-memory spin waits); every CTA executes the
// same sequence of barriers, and a last one keeps every CTA's shared memory
// alive until all remote reads are done.
#pragma once

#include <cooperative_groups.h>

#include "alloc.cuh"

namespace kvs {

namespace cg = cooperative_groups;

constexpr int kCAThreads = 512;
constexpr int kCAWarps = kCAThreads / 32;
constexpr int kCAMaxCluster = 16;
constexpr int kCATieList = 64;   // ties at lambda* settled from a list (more: block scans)

struct CACand {
  unsigned long long theta;  // full bit pattern
  long long uk;              // unit * 4 + step
};

// dynamic shared memory bytes for `per` units of K steps on a cluster of CL
// CTAs, with room for `cand_cap` gathered candidates
__host__ __device__ inline size_t ca_smem_bytes(long long per, int K, int CL, int cand_cap) {
  size_t b = static_cast<size_t>(per) * K * 4;  // top halves
  b = (b + 15) & ~static_cast<size_t>(15);
  b += kRadixBins * 4;                          // histogram
  b += (kRadixBins / CL) * 4;                   // merged slice
  b = (b + 15) & ~static_cast<size_t>(15);
  b += static_cast<size_t>(cand_cap) * sizeof(CACand);
  b += static_cast<size_t>(per);                // levels
  return (b + 15) & ~static_cast<size_t>(15);
}

template <class T>
__device__ __forceinline__ T ca_block_sum(T v, T* sbuf) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sbuf[threadIdx.x >> 5] = v;
  __syncthreads();
  T s = 0;
#pragma unroll
  for (int i = 0; i < kCAWarps; ++i) s += static_cast<T>(sbuf[i]);
  return s;
}

// exclusive scan over the block in thread order; *total = block sum.
// sbuf needs kCAWarps + 1 entries.
__device__ __forceinline__ unsigned long long ca_block_exscan(unsigned long long v, unsigned long long* sbuf,
                                                              unsigned long long* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) sbuf[warp] = x;
  __syncthreads();
  if (warp == 0) {  // exclusive offsets of the warps, and the total
    const unsigned long long t = lane < kCAWarps ? sbuf[lane] : 0ull;
    unsigned long long z = t;
#pragma unroll
    for (int o = 1; o < kCAWarps; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, z, o);
      if (lane >= o) z += y;
    }
    if (lane < kCAWarps) sbuf[lane] = z - t;
    if (lane == kCAWarps - 1) sbuf[kCAWarps] = z;
  }
  __syncthreads();
  *total = sbuf[kCAWarps];
  return sbuf[warp] + x - v;
}

struct CABest {
  unsigned long long theta;  // full fp64 bit pattern, 0 = none
  long long u;
  int cost;
  int pad_;
};

__device__ __forceinline__ bool ca_better(const CABest& a, const CABest& b) {
  if (a.theta == 0ull) return false;
  if (b.theta == 0ull) return true;
  if (a.theta != b.theta) return a.theta > b.theta;
  return a.u < b.u;
}

// Digit selection over a local histogram `loc` of S bins (bin j = digit
// base_bin + j): the digit in which the running cost, highest digits first,
// starting from `base`, passes B.  Thread t owns the m bins just below
// S-1-t*m; a block scan gives the cost of all higher bins.  Returns the digit
// and sets *above_out to the cost strictly above it.
__device__ __forceinline__ unsigned ca_block_select(const uint32_t* loc, int S, int base_bin, unsigned long long base,
                                                    unsigned long long B, unsigned long long* sred, unsigned* s_sel,
                                                    unsigned long long* s_above, unsigned long long* above_out) {
  const int tid = threadIdx.x;
  const int m = (S + kCAThreads - 1) / kCAThreads;
  unsigned long long mine = 0;
  for (int e = 0; e < m; ++e) {
    const int j = S - 1 - (tid * m + e);
    if (j >= 0) mine += loc[j];
  }
  unsigned long long blk;
  const unsigned long long ex = ca_block_exscan(mine, sred, &blk);
  const bool over = base + ex + mine > B;
  const int first = __syncthreads_count(!over);  // `over` is monotone in tid
  if (tid == min(first, kCAThreads - 1)) {
    if (first >= kCAThreads) record_error(KVS_ERR_RANGE);  // invariant broken; keep indices in range
    unsigned long long a = base + ex;
    int sel = base_bin;
    for (int e = 0; e < m; ++e) {
      const int j = S - 1 - (tid * m + e);
      if (j < 0) break;
      if (a + loc[j] > B) {
        sel = base_bin + j;
        break;
      }
      a += loc[j];
    }
    *s_sel = static_cast<unsigned>(sel);
    *s_above = a;
  }
  __syncthreads();
  *above_out = *s_above;
  return *s_sel;
}

// grid (CL * pools): cluster q solves pool q, whose units are q*U .. q*U + U-1
// of w, sigma and bits (every pool has the same size and budget).
template <int CL>
__global__ void __launch_bounds__(kCAThreads, 1) allocate_cluster_kernel(const AllocParams p, const int cand_cap) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  cg::cluster_group cluster = cg::this_cluster();
  const long long pool_base = static_cast<long long>(blockIdx.x / CL) * p.U;
  const float* __restrict__ pw = p.w + pool_base;
  const float* __restrict__ psig = p.sigma + pool_base;
  uint8_t* __restrict__ pbits = p.bits + pool_base;
  const int rank = CL > 1 ? static_cast<int>(cluster.block_rank()) : 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.K;
  const long long per = p.per;
  const long long u_begin = static_cast<long long>(rank) * per;
  const int n_mine = static_cast<int>(max(0ll, min(p.U, u_begin + per) - u_begin));
  constexpr int S = kRadixBins / CL;  // bins per merged slice
  auto csync = [&]() {
    if (CL > 1)
      cluster.sync();
    else
      __syncthreads();
  };
  auto remote = [&](auto* ptr, int r) { return CL > 1 ? cluster.map_shared_rank(ptr, r) : ptr; };

  extern __shared__ __align__(16) unsigned char ca_raw[];
  uint32_t* th = reinterpret_cast<uint32_t*>(ca_raw);  // [K][per]
  size_t off = (static_cast<size_t>(per) * K * 4 + 15) & ~static_cast<size_t>(15);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ca_raw + off);
  off += kRadixBins * 4;
  uint32_t* merged = reinterpret_cast<uint32_t*>(ca_raw + off);
  off += S * 4;
  off = (off + 15) & ~static_cast<size_t>(15);
  CACand* cand = reinterpret_cast<CACand*>(ca_raw + off);
  off += static_cast<size_t>(cand_cap) * sizeof(CACand);
  uint8_t* lvl = ca_raw + off;

  __shared__ unsigned long long s_red[kCAWarps + 1];
  __shared__ unsigned long long s_pub[2];  // values other CTAs read after a cluster barrier
  __shared__ int s_pub_bad;
  __shared__ unsigned long long s_slice_tot;
  __shared__ unsigned long long s_gather[kCAMaxCluster];
  __shared__ unsigned long long s_goff[kCAMaxCluster + 1];
  __shared__ CABest s_best[2];
  __shared__ CABest s_wbest[kCAWarps];
  __shared__ unsigned s_sel;
  __shared__ unsigned long long s_above;
  __shared__ unsigned s_fill;
  __shared__ unsigned long long s_pub_lam;
  __shared__ unsigned s_ntie;
  __shared__ int s_tie_i[kCATieList], s_tie_c[kCATieList];

  // ---- phase 0: validate, cache top halves, total cost of positive items ----
  // (loads batched 8 units per thread so their latencies overlap)
  const int full_cost = p.width[K];
  unsigned long long my_total = 0;
  int my_bad = 0;
  for (int i0 = 0; i0 < n_mine; i0 += 8 * kCAThreads) {
    float wv[8], sv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j * kCAThreads + tid;
      wv[j] = i < n_mine ? pw[u_begin + i] : 0.f;
      sv[j] = i < n_mine ? psig[u_begin + i] : 0.f;
    }
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {  // not unrolled: keeps the executed code small
      const int i = i0 + j * kCAThreads + tid;
      if (i >= n_mine) break;
      const bool ok = isfinite(wv[j]) && isfinite(sv[j]) && wv[j] >= 0.f && sv[j] >= 0.f;
      if (!ok) my_bad = 1;
      const KeyParts kp = key_parts(ok ? wv[j] : 0.f, ok ? sv[j] : 0.f);
      for (int k = 0; k < K; ++k) {
        const unsigned long long t =
            p.dyadic ? theta_from_parts(p, kp, k) : (ok ? theta_bits(p, wv[j], sv[j], k) : 0ull);
        th[k * per + i] = static_cast<uint32_t>(t >> 32);
      }
      if (th[i] != 0u) my_total += static_cast<unsigned long long>(full_cost);
    }
  }
  const unsigned long long blk_total = ca_block_sum(my_total, s_red);
  const int blk_bad = __syncthreads_or(my_bad);
  if (tid == 0) {
    s_pub[0] = blk_total;
    s_pub_bad = blk_bad;
  }
  csync();
  if (tid < CL)
    s_gather[tid] = *remote(&s_pub[0], tid) | (static_cast<unsigned long long>(*remote(&s_pub_bad, tid) != 0) << 63);
  __syncthreads();
  unsigned long long total = 0;
  int bad = 0;
  for (int q = 0; q < CL; ++q) {
    total += s_gather[q] & ~(1ull << 63);
    bad |= static_cast<int>(s_gather[q] >> 63);
  }
  __syncthreads();
  if (bad || total <= p.B) {  // uniform over the cluster
    if (bad && rank == 0 && tid == 0) record_error(KVS_ERR_RANGE);
    for (int i = tid; i < n_mine; i += kCAThreads)
      pbits[u_begin + i] = (!bad && th[i] != 0u) ? static_cast<uint8_t>(full_cost) : 0;
    csync();
    return;
  }

  // ---- phase 1: exact lambda* -------------------------------------------------
  // One cluster pass: cost-weighted histogram of digit (v >> shift) & dmask of
  // the values each_value() yields, merged across the cluster; returns the
  // digit in which the running cost passes B and advances `above`.
  unsigned long long above = 0;
  auto cluster_pass = [&](auto&& each_value, int shift, int width) -> unsigned {
    const unsigned dmask = (1u << width) - 1u;
    for (int b = tid; b < kRadixBins; b += kCAThreads) hist[b] = 0u;
    __syncthreads();
    each_value([&](uint32_t v, int cost) { atomicAdd(&hist[(v >> shift) & dmask], static_cast<unsigned>(cost)); });
    __syncthreads();
    if (CL == 1) return ca_block_select(hist, kRadixBins, 0, above, p.B, s_red, &s_sel, &s_above, &above);
    csync();  // every CTA's histogram is complete
    unsigned long long part = 0;
    for (int j = tid; j < S; j += kCAThreads) {
      uint32_t v[CL];
#pragma unroll
      for (int q = 0; q < CL; ++q) v[q] = remote(hist, q)[rank * S + j];
      uint32_t sum = 0;
#pragma unroll
      for (int q = 0; q < CL; ++q) sum += v[q];
      merged[j] = sum;
      part += sum;
    }
    const unsigned long long st = ca_block_sum(part, s_red);
    if (tid == 0) s_slice_tot = st;
    csync();  // every merged slice and its total are complete; hist is free again
    if (tid < CL) s_gather[tid] = *remote(&s_slice_tot, tid);
    __syncthreads();
    int q = -1;
    unsigned long long base = above;
    for (int r = CL - 1; r >= 0; --r) {
      if (base + s_gather[r] > p.B) {
        q = r;
        break;
      }
      base += s_gather[r];
    }
    if (q < 0) {  // cannot happen (the matched items' cost passes B); keeps indices in range
      q = 0;
      base = above;
      if (tid == 0) record_error(KVS_ERR_RANGE);
    }
    const uint32_t* rm = remote(merged, q);
    for (int j = tid; j < S; j += kCAThreads) hist[j] = rm[j];
    __syncthreads();
    return ca_block_select(hist, S, q * S, base, p.B, s_red, &s_sel, &s_above, &above);
  };
  // items whose cached top half matches `pre` under `msk`
  auto each_top = [&](uint32_t pre, uint32_t msk) {
    return [&, pre, msk](auto&& f) {
      for (int k = 0; k < K; ++k) {
        const int cost = p.cost[k];
        const uint32_t* tk = th + k * per;
        for (int i = tid; i < n_mine; i += kCAThreads) {
          const uint32_t v = tk[i];
          if (v != 0u && (v & msk) == pre) f(v, cost);
        }
      }
    };
  };

  uint32_t P = 0, M = 0;  // selected top bits so far
#pragma unroll 1
  for (int ps = 0; ps < 2; ++ps) {  // bits 31..21, then 20..10
    const int sh = ps == 0 ? 21 : 10;
    const unsigned d = cluster_pass(each_top(P, M), sh, 11);
    P |= d << sh;
    M |= 0x7FFu << sh;
  }

  // the items sharing the top 22 bits, gathered into every CTA when they fit
  unsigned cnt = 0;
  for (int k = 0; k < K; ++k)
    for (int i = tid; i < n_mine; i += kCAThreads) cnt += (th[k * per + i] & M) == P ? 1u : 0u;
  const unsigned long long blk_cnt = ca_block_sum(static_cast<unsigned long long>(cnt), s_red);
  if (tid == 0) s_pub[1] = blk_cnt;
  csync();
  if (tid < CL) s_gather[tid] = *remote(&s_pub[1], tid);
  __syncthreads();
  if (tid == 0) {
    unsigned long long o = 0;
    for (int q = 0; q < CL; ++q) {
      s_goff[q] = o;
      o += s_gather[q];
    }
    s_goff[CL] = o;
    s_fill = 0;
  }
  __syncthreads();
  const unsigned long long n_cand = s_goff[CL];
  unsigned long long lam;
  if (n_cand <= static_cast<unsigned long long>(cand_cap)) {  // uniform
    const unsigned long long my_off = s_goff[rank];
    for (int k = 0; k < K; ++k)
      for (int i = tid; i < n_mine; i += kCAThreads)
        if ((th[k * per + i] & M) == P) {
          const long long u = u_begin + i;
          const unsigned slot = atomicAdd(&s_fill, 1u);
          cand[my_off + slot] = {theta_bits(p, pw[u], psig[u], k), u * 4 + k};
        }
    __syncthreads();
    csync();  // every CTA's segment is written
    for (unsigned long long j = tid; j < n_cand; j += kCAThreads) {
      int q = 0;
      while (q + 1 < CL && j >= s_goff[q + 1]) ++q;
      if (q != rank) cand[j] = remote(cand, q)[j];
    }
    __syncthreads();
    unsigned long long pre = static_cast<unsigned long long>(P) << 32;
    if (n_cand <= 32) {
      // one warp: lambda* is the theta whose cost strictly above stays within
      // B while the cost at or above it does not
      if (warp == 0) {
        const bool has = static_cast<unsigned long long>(lane) < n_cand;
        const unsigned long long t = has ? cand[lane].theta : 0ull;
        const unsigned c = has ? static_cast<unsigned>(p.cost[cand[lane].uk & 3]) : 0u;
        unsigned long long gt = 0, ge = 0;
        for (int m = 0; m < 32; ++m) {
          const unsigned long long tm = __shfl_sync(0xFFFFFFFFu, t, m);
          const unsigned cm = __shfl_sync(0xFFFFFFFFu, c, m);
          if (tm > t) gt += cm;
          if (tm >= t) ge += cm;
        }
        const bool hit = has && above + gt <= p.B && above + ge > p.B;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, hit);
        const int src = bal ? __ffs(bal) - 1 : 0;
        if (bal == 0u && lane == 0) record_error(KVS_ERR_RANGE);
        const unsigned long long lt = __shfl_sync(0xFFFFFFFFu, t, src);
        const unsigned long long lg = __shfl_sync(0xFFFFFFFFu, gt, src);
        if (lane == 0) {
          s_above = above + lg;
          s_pub_lam = lt;
        }
      }
      __syncthreads();
      above = s_above;
      pre = s_pub_lam;
    } else if (n_cand <= 128) {
      // one candidate per thread: lambda* is a theta whose cost strictly
      // above stays within B while the cost at or above it does not (every
      // candidate with that theta qualifies; the lowest index is taken)
      const bool has = static_cast<unsigned long long>(tid) < n_cand;
      const unsigned long long t = has ? cand[tid].theta : 0ull;
      unsigned long long gt = 0, ge = 0;
      if (has) {
        for (unsigned long long m = 0; m < n_cand; ++m) {
          const CACand cm = cand[m];
          const unsigned c = static_cast<unsigned>(p.cost[cm.uk & 3]);
          if (cm.theta > t) gt += c;
          if (cm.theta >= t) ge += c;
        }
      }
      const bool hit = has && above + gt <= p.B && above + ge > p.B;
      if (tid == 0) s_sel = 0xFFFFFFFFu;
      __syncthreads();
      if (hit) atomicMin(&s_sel, static_cast<unsigned>(tid));
      __syncthreads();
      const unsigned src = s_sel;
      if (src == 0xFFFFFFFFu) {                    // cannot happen; keeps the result defined
        if (tid == 0) record_error(KVS_ERR_RANGE);
      } else if (tid == static_cast<int>(src)) {
        s_above = above + gt;
        s_pub_lam = t;
      }
      __syncthreads();
      if (src != 0xFFFFFFFFu) {
        above = s_above;
        pre = s_pub_lam;
      }
    } else {
      // local passes over bits 41..0 of the full thetas (the top 22 are P)
      unsigned long long msk = static_cast<unsigned long long>(M) << 32;
      const int shifts[4] = {31, 20, 9, 0}, widths[4] = {11, 11, 11, 9};
#pragma unroll 1
      for (int ps = 0; ps < 4; ++ps) {
        const int sh = shifts[ps];
        const unsigned long long dmask = (1ull << widths[ps]) - 1ull;
        for (int b = tid; b < kRadixBins; b += kCAThreads) hist[b] = 0u;
        __syncthreads();
        for (unsigned long long j = tid; j < n_cand; j += kCAThreads) {
          const CACand c = cand[j];
          if ((c.theta & msk) == pre)
            atomicAdd(&hist[(c.theta >> sh) & dmask], static_cast<unsigned>(p.cost[c.uk & 3]));
        }
        __syncthreads();
        const unsigned d = ca_block_select(hist, 1 << widths[ps], 0, above, p.B, s_red, &s_sel, &s_above, &above);
        pre |= static_cast<unsigned long long>(d) << sh;
        msk |= dmask << sh;
      }
    }
    lam = pre;
    csync();  // nobody reads this CTA's candidates any more
  } else {
    // too many near-equal items: finish with cluster passes, low halves recomputed
    const unsigned d2 = cluster_pass(each_top(P, M), 0, 10);
    P |= d2;
    uint32_t PL = 0, ML = 0;
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
#pragma unroll 1
    for (int ps = 0; ps < 3; ++ps) {
      const uint32_t pre = PL, msk = ML, top = P;
      auto each_low = [&](auto&& f) {
        for (int k = 0; k < K; ++k) {
          const int cost = p.cost[k];
          for (int i = tid; i < n_mine; i += kCAThreads) {
            if (th[k * per + i] != top) continue;
            const long long u = u_begin + i;
            const uint32_t v = static_cast<uint32_t>(theta_bits(p, pw[u], psig[u], k));
            if ((v & msk) == pre) f(v, cost);
          }
        }
      };
      const unsigned d = cluster_pass(each_low, shifts[ps], widths[ps]);
      PL |= d << shifts[ps];
      ML |= ((1u << widths[ps]) - 1u) << shifts[ps];
    }
    lam = (static_cast<unsigned long long>(P) << 32) | PL;
  }
  const uint32_t lam_top = static_cast<uint32_t>(lam >> 32);

  // ---- phase 2: levels of the Lagrangian prefix; ties at lambda* in unit order
  // level of unit i = #{k : theta > lam}; tie cost if some theta == lam
  // (thetas fall with k, so the first theta not above lam ends the count)
  auto unit_level = [&](int i, int* tie_cost) {
    int l = 0;
    *tie_cost = 0;
    for (int k = 0; k < K; ++k) {
      const uint32_t t = th[k * per + i];
      if (t > lam_top) {
        ++l;
        continue;
      }
      if (t == lam_top && t != 0u) {
        const long long u = u_begin + i;
        const unsigned long long f = theta_bits(p, pw[u], psig[u], k);
        if (f > lam) {
          ++l;
          continue;
        }
        if (f == lam) *tie_cost = p.cost[k];
      }
      break;
    }
    return l;
  };
  // levels first; ties at lambda* (the theta of lambda* itself, and any equal
  // ones: a handful) are listed and settled below
  unsigned long long my_tie = 0;
  if (tid == 0) s_ntie = 0;
  __syncthreads();
  for (int i = tid; i < n_mine; i += kCAThreads) {
    int tc;
    lvl[i] = static_cast<uint8_t>(unit_level(i, &tc));
    my_tie += static_cast<unsigned long long>(tc);
    if (tc) {
      const unsigned slot = atomicAdd(&s_ntie, 1u);
      if (slot < kCATieList) {
        s_tie_i[slot] = i;
        s_tie_c[slot] = tc;
      }
    }
  }
  const int cta_has_tie = __syncthreads_or(my_tie != 0ull);
  const unsigned long long blk_tie = cta_has_tie ? ca_block_sum(my_tie, s_red) : 0ull;
  if (tid == 0) s_pub[1] = blk_tie;
  csync();
  if (tid < CL) s_gather[tid] = *remote(&s_pub[1], tid);
  __syncthreads();
  unsigned long long carry = above, all_ties = 0;
  for (int q = 0; q < CL; ++q) {
    if (q < rank) carry += s_gather[q];
    all_ties += s_gather[q];
  }
  __syncthreads();
  unsigned long long my_used = 0;  // cumulative cost through the last tie taken here
  if (cta_has_tie && s_ntie <= kCATieList) {  // uniform: the list holds every tie of this CTA
    // warp 0 orders the listed ties by unit and takes them while the running cost fits B
    if (warp == 0) {
      const int nt = static_cast<int>(s_ntie);
      int ia = lane < nt ? s_tie_i[lane] : 0x7FFFFFFF, ib = lane + 32 < nt ? s_tie_i[lane + 32] : 0x7FFFFFFF;
      const int ca = lane < nt ? s_tie_c[lane] : 0, cb = lane + 32 < nt ? s_tie_c[lane + 32] : 0;
      // rank of each entry in unit order, then the cost of the entries before it
      unsigned long long before_a = 0, before_b = 0;
      for (int m = 0; m < nt; ++m) {
        const int im = __shfl_sync(0xFFFFFFFFu, m < 32 ? ia : ib, m & 31);
        const int cm = __shfl_sync(0xFFFFFFFFu, m < 32 ? ca : cb, m & 31);
        if (im < ia) before_a += static_cast<unsigned long long>(cm);
        if (im < ib) before_b += static_cast<unsigned long long>(cm);
      }
      unsigned long long mu = 0;
      if (lane < nt) {
        const unsigned long long cum = carry + before_a + static_cast<unsigned long long>(ca);
        if (cum <= p.B) {
          lvl[ia] = static_cast<uint8_t>(lvl[ia] + 1);
          mu = cum;
        }
      }
      if (lane + 32 < nt) {
        const unsigned long long cum = carry + before_b + static_cast<unsigned long long>(cb);
        if (cum <= p.B) {
          lvl[ib] = static_cast<uint8_t>(lvl[ib] + 1);
          mu = max(mu, cum);
        }
      }
      my_used = mu;                                // folded over the block below
    }
    __syncthreads();
  } else if (cta_has_tie) {  // many ties: take them in unit order, block scan by block scan
    for (int base = 0; base < n_mine; base += kCAThreads) {
      const int i = base + tid;
      int tc = 0;
      if (i < n_mine) (void)unit_level(i, &tc);
      unsigned long long chunk_total;
      const unsigned long long ex = ca_block_exscan(static_cast<unsigned long long>(tc), s_red, &chunk_total);
      if (i < n_mine && tc != 0) {
        const unsigned long long cum = carry + ex + static_cast<unsigned long long>(tc);
        if (cum <= p.B) {
          lvl[i] = static_cast<uint8_t>(lvl[i] + 1);
          my_used = max(my_used, cum);
        }
      }
      carry += chunk_total;
    }
  }
  for (int i = tid; i < n_mine; i += kCAThreads) pbits[u_begin + i] = static_cast<uint8_t>(p.width[lvl[i]]);
  // cost of the prefix = the largest cumulative cost of a tie taken, or `above`
  unsigned long long used = above;
  if (all_ties != 0ull) {  // uniform over the cluster
    unsigned long long m = my_used;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    __syncthreads();
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    if (tid == 0) {
      unsigned long long b = 0;
      for (int i = 0; i < kCAWarps; ++i) b = max(b, s_red[i]);
      s_pub[0] = b;
    }
    csync();
    if (tid < CL) s_gather[tid] = *remote(&s_pub[0], tid);
    __syncthreads();
    for (int q = 0; q < CL; ++q) used = max(used, s_gather[q]);
  }

  // ---- phase 3: budget-fix rounds -------------------------------------------
  long long R = static_cast<long long>(p.B) - static_cast<long long>(used);
  for (int round = 0; round < kMaxFixRounds && R >= p.min_cost; ++round) {
    CABest best = {0ull, 0ll, 0, 0};
    uint32_t best_top = 0;
    for (int i = tid; i < n_mine; i += kCAThreads) {
      const int k = lvl[i];
      if (k >= K || p.cost[k] > R) continue;
      const uint32_t t = th[k * per + i];
      if (t == 0u || t < best_top) continue;
      const long long u = u_begin + i;
      const CABest c = {theta_bits(p, pw[u], psig[u], k), u, p.cost[k], 0};
      if (t > best_top || ca_better(c, best)) {
        best = c;
        best_top = t;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      CABest oc;
      oc.theta = __shfl_xor_sync(0xFFFFFFFFu, best.theta, o);
      oc.u = __shfl_xor_sync(0xFFFFFFFFu, best.u, o);
      oc.cost = __shfl_xor_sync(0xFFFFFFFFu, best.cost, o);
      oc.pad_ = 0;
      if (ca_better(oc, best)) best = oc;
    }
    if (lane == 0) s_wbest[warp] = best;
    __syncthreads();
    if (tid == 0) {
      CABest bb = s_wbest[0];
      for (int i = 1; i < kCAWarps; ++i)
        if (ca_better(s_wbest[i], bb)) bb = s_wbest[i];
      s_best[round & 1] = bb;
    }
    csync();
    if (tid < CL) s_wbest[tid] = *remote(&s_best[round & 1], tid);
    __syncthreads();
    CABest g = s_wbest[0];
    for (int q = 1; q < CL; ++q)
      if (ca_better(s_wbest[q], g)) g = s_wbest[q];
    if (g.theta == 0ull) break;  // uniform: every CTA sees the same g
    if (g.u >= u_begin && g.u < u_begin + n_mine && tid == 0) {
      const int i = static_cast<int>(g.u - u_begin);
      const int l = lvl[i] + 1;
      lvl[i] = static_cast<uint8_t>(l);
      pbits[g.u] = static_cast<uint8_t>(p.width[l]);
    }
    R -= g.cost;
    __syncthreads();
  }
  csync();  // no CTA leaves while another may still read its shared memory
}

}  // namespace kvs
