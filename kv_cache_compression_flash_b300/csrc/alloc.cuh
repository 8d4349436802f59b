// Lagrangian (reverse water-filling) multiple-choice-knapsack bit allocation.
//   min sum_u w_u sigma_u 2^-b_u  s.t.  sum_u b_u <= B,  b_u in a width set
//   [RDKV §2.1 objective; §2.2 discrete widths {0,2,4,8,16}, Lagrangian relaxation]
//
// D_u(b) = key_u 2^-b is strictly convex in b, so the Lagrangian argmin of
// D_u(b) + lambda b climbs the widths in order: unit u leaves width b_k when
// lambda drops below theta_{u,k} = c_k key_u (c_k = chord slope of 2^-b,
// key_u = w_u sigma_u exactly in fp64).  Sorting every "upgrade item" (u, k)
// by theta descending (ties: u, then k ascending) and taking the longest
// prefix that fits B is the Lagrangian solution at the critical multiplier
// lambda* = theta of the first item that does not fit.  A budget-fix scan then
// keeps taking later items that still fit and whose previous step was taken.
//
// B300 design: one cooperative launch, all blocks resident, grid barriers with
// bounded waits (several pools side by side: a block row per pool).  Each
// block computes its units' thetas once (fp64) into shared memory.  lambda*
// is found exactly by a 6-pass radix select (11-bit digits) on the fp64 bit
// patterns of theta (positive doubles order like their bit patterns), each
// pass a cost-weighted 2048-bin histogram; every block then decides the digit
// redundantly so one barrier per pass suffices.  Ties at lambda* are resolved
// in unit order by a grid-wide scan; the fix scan is an arg-max
// (theta, then lowest unit) over each unit's next upgrade, repeated while the
// leftover budget buys something (at most max_step/min_step rounds).
#pragma once

#include "common.cuh"

namespace kvs {

constexpr int kAllocThreads = 256;
constexpr int kMaxFixRounds = 16;

constexpr int kRadixBits = 11;                 // digit width of the radix select
constexpr int kRadixBins = 1 << kRadixBits;    // 2048
constexpr int kRadixPasses = 6;                // 11+11+11+11+11+9 = 64 bits
constexpr int kBinsPerThread = kRadixBins / kAllocThreads;

__host__ __device__ constexpr int radix_shift(int pass) { return pass < 5 ? 53 - 11 * pass : 0; }
__host__ __device__ constexpr int radix_width(int pass) { return pass < 5 ? 11 : 9; }

struct AllocHeader {
  GridSync sync;
  unsigned long long total;  // cost of every positive upgrade item
  int bad;                   // a weight or sigma was negative or not finite
  int pad_;
  unsigned long long first_cut;  // cost taken before the first item that did not fit
};

struct FixCand {
  unsigned long long theta;  // fp64 bit pattern, 0 = no candidate
  long long u;
  int cost;
  int pad_;
};

struct AllocParams {
  const float* w;
  const float* sigma;
  uint8_t* bits;
  long long U;
  long long per;    // units per block
  unsigned long long B;
  int K;            // upgrade steps = allowed widths - 1
  int min_cost;     // smallest step
  double c[4];      // chord slopes, descending
  int cost[4];      // step sizes b_{k+1} - b_k
  int width[5];     // allowed widths, ascending, width[0] = 0
  int dyadic;       // every c_k = n_k 2^-e_k exactly (n_k < 2^16): thetas from integer arithmetic
  unsigned n[4];
  int e[4];
  AllocHeader* hdr;
  unsigned long long* hist;       // [kRadixPasses][kRadixBins] cost-weighted counts
  unsigned long long* tie_block;  // [gridDim.x]
  FixCand* cand;                  // [kMaxFixRounds][gridDim.x]
};

// key = (double)w * (double)sigma is exact: its significand is the product of
// the two 24-bit significands.  KeyParts holds that product M (< 2^48) and the
// exponent E of its lowest bit; M == 0 when the key is 0.
struct KeyParts {
  unsigned long long M;
  int E;
};

__device__ __forceinline__ KeyParts key_parts(float w, float s) {
  const uint32_t wb = __float_as_uint(w), sb = __float_as_uint(s);
  uint32_t ew = (wb >> 23) & 0xFFu, es = (sb >> 23) & 0xFFu;
  uint32_t mw = wb & 0x7FFFFFu, ms = sb & 0x7FFFFFu;
  if (ew) mw |= 0x800000u; else ew = 1u;  // subnormal: no implicit bit, exponent of 1
  if (es) ms |= 0x800000u; else es = 1u;
  KeyParts kp;
  kp.M = static_cast<unsigned long long>(mw) * ms;
  kp.E = static_cast<int>(ew + es) - 300;
  return kp;
}

// Bit pattern of theta = fl64(c_k * key) for finite w, sigma >= 0 (0 when the
// key is 0).  With dyadic slopes c_k = n_k 2^-e_k the product n_k M (< 2^64)
// is formed exactly in integers and rounded once to 53 bits, half to even:
// the same double the fp64 multiply gives, without the fp64 pipe (slow on this
// part).
__device__ __forceinline__ unsigned long long theta_from_parts(const AllocParams& p, const KeyParts& kp, int k) {
  if (kp.M == 0ull) return 0ull;
  const unsigned long long P = kp.M * p.n[k];
  const int lz = __clzll(static_cast<long long>(P));
  const unsigned long long Pn = P << lz;  // leading one at bit 63
  unsigned long long mant = Pn >> 11;     // 53 bits
  const unsigned rest = static_cast<unsigned>(Pn & 0x7FFull);
  int ex = 63 - lz + kp.E - p.e[k];       // value = 1.f * 2^ex
  if (rest > 0x400u || (rest == 0x400u && (mant & 1ull))) {
    ++mant;
    if (mant == (1ull << 53)) {
      mant >>= 1;
      ++ex;
    }
  }
  return (static_cast<unsigned long long>(ex + 1023) << 52) | (mant & ((1ull << 52) - 1ull));
}

__device__ __forceinline__ unsigned long long theta_bits(const AllocParams& p, float w, float s, int k) {
  if (!p.dyadic) {
    const double key = static_cast<double>(w) * static_cast<double>(s);
    return key > 0.0 ? static_cast<unsigned long long>(__double_as_longlong(p.c[k] * key)) : 0ull;
  }
  return theta_from_parts(p, key_parts(w, s), k);
}

__device__ __forceinline__ unsigned long long ld_vol(const unsigned long long* p) {
  return *reinterpret_cast<const volatile unsigned long long*>(p);
}

template <class T>
__device__ __forceinline__ T block_sum(T v, T* sbuf) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) sbuf[warp] = v;
  __syncthreads();
  T s = 0;
  for (int i = 0; i < (kAllocThreads >> 5); ++i) s += sbuf[i];
  return s;
}

// exclusive scan of v over the block in thread order; returns the block total in *total
__device__ __forceinline__ unsigned long long block_exscan(unsigned long long v, unsigned long long* sbuf,
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
  unsigned long long before = 0, tot = 0;
  for (int i = 0; i < (kAllocThreads >> 5); ++i) {
    if (i < warp) before += sbuf[i];
    tot += sbuf[i];
  }
  *total = tot;
  return before + x - v;
}

__device__ __forceinline__ bool cand_better(const FixCand& a, const FixCand& b) {  // a before b in item order
  if (a.theta != b.theta) return a.theta > b.theta;
  return a.u < b.u;
}

// first candidate in item order over the block (result valid in every thread)
__device__ __forceinline__ FixCand block_best(FixCand best, FixCand* s_cand) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FixCand o_c;
    o_c.theta = __shfl_xor_sync(0xFFFFFFFFu, best.theta, o);
    o_c.u = __shfl_xor_sync(0xFFFFFFFFu, best.u, o);
    o_c.cost = __shfl_xor_sync(0xFFFFFFFFu, best.cost, o);
    o_c.pad_ = 0;
    if (o_c.theta != 0ull && (best.theta == 0ull || cand_better(o_c, best))) best = o_c;
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s_cand[threadIdx.x >> 5] = best;
  __syncthreads();
  FixCand bb = s_cand[0];
  for (int i = 1; i < (kAllocThreads >> 5); ++i)
    if (s_cand[i].theta != 0ull && (bb.theta == 0ull || cand_better(s_cand[i], bb))) bb = s_cand[i];
  return bb;
}

// theta bit pattern of item (u, k): from the block's shared-memory cache when
// CACHE, else recomputed (fp64 is slow on this part, so the cache is the fast
// path).  0 when the unit's key is not positive.
template <bool CACHE>
struct ThetaSource {
  const AllocParams& p;
  const float* w;                   // the pool's weights and sigmas
  const float* sigma;
  const unsigned long long* cache;  // [K][per]
  long long u_begin;
  __device__ __forceinline__ unsigned long long operator()(long long u, int k) const {
    if (CACHE) return cache[static_cast<long long>(k) * p.per + (u - u_begin)];
    return theta_bits(p, w[u], sigma[u], k);
  }
};

// grid (blocks per pool, pools): block row q solves pool q (units q*U ..) on
// its own slice of the workspace: header q, histograms q, and the per-block
// tie and candidate arrays of row q; its grid barriers count that row only.
template <bool CACHE>
__global__ void __launch_bounds__(kAllocThreads) allocate_kernel(const AllocParams p) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  // the block row's pool (pointers only: the parameters stay in parameter space)
  const long long q = blockIdx.y;
  const float* const pw = p.w + q * p.U;
  const float* const psig = p.sigma + q * p.U;
  uint8_t* const pbits = p.bits + q * p.U;
  unsigned long long* const phist = p.hist + q * kRadixPasses * kRadixBins;
  unsigned long long* const ptie = p.tie_block + q * gridDim.x;
  FixCand* const pcand = p.cand + q * kMaxFixRounds * gridDim.x;
  extern __shared__ unsigned long long s_theta[];  // [K][per] when CACHE
  __shared__ unsigned s_hist[kRadixBins];          // per-block cost per bin (< 2^32: units per block x 16)
  __shared__ unsigned long long s_red[kAllocThreads / 32];
  __shared__ unsigned long long s_sel_above;
  __shared__ int s_sel;
  __shared__ int s_lvl_of_width[17];
  __shared__ FixCand s_cand[kAllocThreads / 32];
  __shared__ FixCand s_best;
  __shared__ int s_flag;

  const int nb = gridDim.x, b = blockIdx.x, tid = threadIdx.x;
  const long long u_begin = static_cast<long long>(b) * p.per;
  const long long u_end = min(p.U, u_begin + p.per);
  AllocHeader* H = p.hdr + q;
  const ThetaSource<CACHE> theta{p, pw, psig, s_theta, u_begin};

  if (tid < 17) s_lvl_of_width[tid] = -1;
  __syncthreads();
  if (tid <= p.K) s_lvl_of_width[p.width[tid]] = tid;
  // the first pass's global histogram starts at zero (later ones are cleared
  // one pass ahead, see below)
  if (b == 0)
    for (int i = tid; i < kRadixBins; i += kAllocThreads) phist[i] = 0ull;

  // ---- phase 0: validate, cache thetas, total cost of positive items ------
  unsigned long long my_total = 0;
  int my_bad = 0;
  const int full_cost = p.width[p.K];
  for (long long u = u_begin + tid; u < u_end; u += kAllocThreads) {
    const float wf = pw[u], sf = psig[u];
    if (!(isfinite(wf) && isfinite(sf) && wf >= 0.f && sf >= 0.f)) my_bad = 1;
    const double key = static_cast<double>(wf) * static_cast<double>(sf);
    if (key > 0.0) my_total += static_cast<unsigned long long>(full_cost);
    if (CACHE)
      for (int k = 0; k < p.K; ++k)
        s_theta[static_cast<long long>(k) * p.per + (u - u_begin)] = key > 0.0 ? theta_bits(p, wf, sf, k) : 0ull;
  }
  const unsigned long long blk_total = block_sum(my_total, s_red);
  const int blk_bad = __syncthreads_or(my_bad);
  unsigned long long total = blk_total;
  int bad = blk_bad;
  if (nb > 1) {
    if (tid == 0) {
      if (blk_total) atomicAdd(&H->total, blk_total);
      if (blk_bad) atomicOr(&H->bad, 1);
    }
    if (!grid_barrier(&H->sync, nb)) return;
    total = ld_vol(&H->total);
    bad = *reinterpret_cast<volatile int*>(&H->bad);
  }
  if (bad) {
    if (b == 0 && tid == 0) record_error(KVS_ERR_RANGE);
    for (long long u = u_begin + tid; u < u_end; u += kAllocThreads) pbits[u] = 0;
    return;
  }
  if (total <= p.B) {  // every upgrade fits
    for (long long u = u_begin + tid; u < u_end; u += kAllocThreads)
      pbits[u] = theta(u, 0) != 0ull ? static_cast<uint8_t>(full_cost) : 0;
    return;
  }

  // ---- phase 1: radix select of lambda* on theta bit patterns ------------
  unsigned long long prefix = 0, pmask = 0, above = 0;
  for (int pass = 0; pass < kRadixPasses; ++pass) {
    const int shift = radix_shift(pass);
    const unsigned long long dmask = (1ull << radix_width(pass)) - 1ull;
    for (int i = tid; i < kRadixBins; i += kAllocThreads) s_hist[i] = 0;
    // the next pass's global histogram is idle until the barrier below
    if (b == nb - 1 && pass + 1 < kRadixPasses)
      for (int i = tid; i < kRadixBins; i += kAllocThreads) phist[(pass + 1) * kRadixBins + i] = 0ull;
    __syncthreads();
    // Early passes see the exponent bits, which nearly all thetas share: the
    // lanes of a warp that fall in one bin are merged first (match_any), so a
    // bin takes one atomic per warp and step instead of one per item.
    for (long long base = u_begin; base < u_end; base += kAllocThreads) {
      const long long u = base + tid;
      for (int k = 0; k < p.K; ++k) {
        const unsigned long long v = u < u_end ? theta(u, k) : 0ull;
        const unsigned bin = (v != 0ull && (v & pmask) == prefix) ? static_cast<unsigned>((v >> shift) & dmask)
                                                                   : static_cast<unsigned>(kRadixBins);
        const unsigned grp = __match_any_sync(0xFFFFFFFFu, bin);
        if (bin != static_cast<unsigned>(kRadixBins) && (tid & 31) == __ffs(grp) - 1)
          atomicAdd(&s_hist[bin], static_cast<unsigned>(__popc(grp) * p.cost[k]));
      }
    }
    __syncthreads();
    const bool single = nb == 1;  // one block: its histogram is the whole histogram
    if (!single) {
      for (int i = tid; i < kRadixBins; i += kAllocThreads)
        if (s_hist[i]) atomicAdd(&phist[pass * kRadixBins + i], static_cast<unsigned long long>(s_hist[i]));
      if (!grid_barrier(&H->sync, nb)) return;
    }
    {
      // thread t owns the kBinsPerThread digits just below 2047 - t*kBinsPerThread
      // (descending); a scan over threads gives the cost of all higher digits, and
      // the first thread whose range pushes the running cost past B holds lambda*
      unsigned long long h[kBinsPerThread], mine = 0;
      const unsigned long long* hp = phist + pass * kRadixBins;
#pragma unroll
      for (int j = 0; j < kBinsPerThread; ++j) {
        const int bin = kRadixBins - 1 - (tid * kBinsPerThread + j);
        h[j] = single ? static_cast<unsigned long long>(s_hist[bin]) : ld_vol(&hp[bin]);
        mine += h[j];
      }
      unsigned long long block_total;
      const unsigned long long ex = block_exscan(mine, s_red, &block_total);
      const bool over = above + ex + mine > p.B;
      const int first = __syncthreads_count(!over);  // over is monotone in tid
      if (tid == first) {
        unsigned long long a = above + ex;
        int sel = 0;
        for (int j = 0; j < kBinsPerThread; ++j) {
          if (a + h[j] > p.B) {
            sel = kRadixBins - 1 - (tid * kBinsPerThread + j);
            break;
          }
          a += h[j];
        }
        s_sel = sel;
        s_sel_above = a;
      }
    }
    __syncthreads();
    prefix |= static_cast<unsigned long long>(s_sel) << shift;
    pmask |= dmask << shift;
    above = s_sel_above;
    __syncthreads();
  }
  const unsigned long long lam = prefix;  // theta bits of the first item that does not fit

  // ---- phase 2: prefix levels; ties at lambda* resolved in unit order -----
  unsigned long long my_tie = 0;
  for (long long u = u_begin + tid; u < u_end; u += kAllocThreads)
    for (int k = 0; k < p.K; ++k)
      if (theta(u, k) == lam) my_tie += p.cost[k];
  unsigned long long carry = above;
  if (nb > 1) {
    const unsigned long long blk_tie = block_sum(my_tie, s_red);
    if (tid == 0) ptie[b] = blk_tie;
    if (!grid_barrier(&H->sync, nb)) return;
    unsigned long long e = 0;
    for (int i = tid; i < b; i += kAllocThreads) e += ld_vol(&ptie[i]);
    carry += block_sum(e, s_red);
  }
  for (long long base = u_begin; base < u_end; base += kAllocThreads) {
    const long long u = base + tid;
    int lvl = 0;
    unsigned long long tie = 0;
    if (u < u_end) {
      for (int k = 0; k < p.K; ++k) {
        const unsigned long long v = theta(u, k);
        if (v > lam) ++lvl;
        else if (v == lam) tie = p.cost[k];
      }
    }
    unsigned long long chunk_total;
    const unsigned long long ex = block_exscan(tie, s_red, &chunk_total);
    if (u < u_end) {
      const unsigned long long cum = carry + ex + tie;  // cost through this item
      if (tie) {
        if (cum <= p.B) ++lvl;
        else if (cum - tie <= p.B) H->first_cut = cum - tie;  // exactly one item: the first misfit
      }
      pbits[u] = static_cast<uint8_t>(p.width[lvl]);
    }
    carry += chunk_total;
  }
  if (nb > 1) {
    if (!grid_barrier(&H->sync, nb)) return;
  } else {
    __syncthreads();
  }

  // ---- phase 3: budget-fix rounds ------------------------------------------
  long long R = static_cast<long long>(p.B) - static_cast<long long>(ld_vol(&H->first_cut));
  for (int it = 0; it < kMaxFixRounds; ++it) {
    if (R < p.min_cost) break;
    FixCand best = {0ull, 0ll, 0, 0};
    for (long long u = u_begin + tid; u < u_end; u += kAllocThreads) {
      const int lvl = s_lvl_of_width[pbits[u]];
      if (lvl < 0 || lvl >= p.K || p.cost[lvl] > R) continue;
      const unsigned long long th = theta(u, lvl);
      if (th == 0ull) continue;
      FixCand c = {th, u, p.cost[lvl], 0};
      if (best.theta == 0ull || cand_better(c, best)) best = c;
    }
    best = block_best(best, s_cand);
    if (nb == 1) {  // the block's best is the global best
      if (tid == 0) {
        s_best = best;
        s_flag = best.theta != 0ull;
      }
    } else {
      if (tid == 0) pcand[it * nb + b] = best;
      if (!grid_barrier(&H->sync, nb)) return;
      FixCand bb = {0ull, 0ll, 0, 0};
      for (int i = tid; i < nb; i += kAllocThreads) {
        const volatile FixCand* vc = &pcand[it * nb + i];
        FixCand c2 = {vc->theta, vc->u, vc->cost, 0};
        if (c2.theta != 0ull && (bb.theta == 0ull || cand_better(c2, bb))) bb = c2;
      }
      bb = block_best(bb, s_cand);
      if (tid == 0) {
        s_best = bb;
        s_flag = bb.theta != 0ull;
      }
    }
    __syncthreads();
    if (!s_flag) break;
    const long long ub = s_best.u;
    if (ub >= u_begin && ub < u_end && tid == static_cast<int>((ub - u_begin) % kAllocThreads)) {
      const int lvl = s_lvl_of_width[pbits[ub]];
      pbits[ub] = static_cast<uint8_t>(p.width[lvl + 1]);
    }
    R -= s_best.cost;
    __syncthreads();
  }
}

}  // namespace kvs
