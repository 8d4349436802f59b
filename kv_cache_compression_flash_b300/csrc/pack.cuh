// Quantise / pack a KV cache into width-grouped streams and back.
//   [RDKV §2.2 stage 2 (V tokens) and stage 3 (K channels over kept tokens);
//    §2.3 TriZone: packed rows grouped by width {2,4,8}, 16-bit rows kept raw]
//
// Code (a reading of the summary, which names widths but no quantiser):
// groups of 64 elements; widths 2/4/8 use a symmetric uniform code with
// qmax = 2^(w-1)-1, scale s = fp16 rounded up from absmax/qmax, and
// q = round-half-even(x/s) (correctly rounded fp32 division: for bf16 x and
// fp16 s it picks the same integer as exact division); width 16 keeps the raw
// bf16 bits.  One half-warp owns one group: lane i holds elements 4i..4i+3,
// whose 4w code bits are contiguous in the group's 8w-byte block, so each lane
// issues one aligned store of w/2 bytes and a half-warp writes its block in one
// coalesced transaction.
//
// Stream order (ascending unit id within a width) comes from a plan computed
// on one thread-block cluster (exclusive scans of the per-width unit and
// group counts, exchanged through distributed shared memory); the pack and
// dequantise kernels then run over the whole GPU.
#pragma once

#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace kvs {

constexpr int kPlanThreads = 512;

// A stream set may hold several pools (independent (layer, sequence) caches
// of the same shape) back to back: pool q's arrays start at q * cap_units[s]
// (ids, group offsets) and q * cap_groups[s] (codes in 8w-byte groups,
// scales), its counts at counts[8 q].  Group offsets and unit ids stay local
// to the pool, so each pool's streams read like a one-pool set.
struct StreamPtrs {
  uint8_t* codes[4];
  uint16_t* scales[4];
  int32_t* ids[4];
  int64_t* goff[4];
  long long cap_units[4];
  long long cap_groups[4];
  int64_t* counts;  // [8]
};

__device__ __forceinline__ int width_slot(uint32_t w) {
  return w == 2 ? 0 : w == 4 ? 1 : w == 8 ? 2 : w == 16 ? 3 : -1;
}

__device__ __forceinline__ unsigned half_mask() { return 0xFFFFu << (threadIdx.x & 16); }

// round-half-even(x / s) for bf16 x and fp16 s > 0 with |x / s| <= 128, from
// one reciprocal r ~ 1/s: floor(x r) is within one of the nearest integer
// (|x r - x/s| <= 2^-16), and the choice between n0 = floor(x r) and n0 + 1
// is the sign of x - (n0 + 1/2) s.  One FMA gives that sign exactly: the
// product (n0 + 1/2) s has at most 20 significant bits, and a single rounding
// never changes the sign of a difference nor makes a nonzero one zero.  A zero
// difference is a tie, which goes to the even neighbour.
__device__ __forceinline__ int round_div_even(const float x, const float s, const float r) {
  const float n0 = floorf(x * r);
  const float e = fmaf(-(n0 + 0.5f), s, x);
  int n = static_cast<int>(n0);
  if (e > 0.f || (e == 0.f && (n & 1))) ++n;
  return n;
}

// round-half-even(x / s): x * (1/s) is within 2^-16 of x / s, so its rint is
// the answer unless it sits near a half-integer; there the exact test decides
__device__ __forceinline__ int q_round(const float x, const float s, const float r) {
  const float t = x * r;
  const float q = rintf(t);
  if (fabsf(t - q) < 0.49993896484375f) return static_cast<int>(q);  // 1/2 - 2^-14
  return round_div_even(x, s, r);
}

// Quantise this lane's 4 elements of a 64-element group (the half-warp holds
// the group).  Returns the 4w code bits; *scale_bits gets the fp16 scale.
__device__ __forceinline__ uint32_t quantize_lane4(const float (&x)[4], const int w, uint16_t* scale_bits,
                                                   bool* overflow) {
  float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  const unsigned m = half_mask();
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(m, a, o));
  const float qmax = static_cast<float>((1 << (w - 1)) - 1);
  const __half sh = __float2half_ru(__fdiv_rn(a, qmax));
  const float s = __half2float(sh);
  *overflow = isinf(s);
  *scale_bits = __half_as_ushort(sh);
  uint32_t packed = 0;
  const uint32_t cmask = (1u << w) - 1u;
  if (s > 0.f && !isinf(s)) {
    const float r = __frcp_rn(s);
#pragma unroll
    for (int e = 0; e < 4; ++e) packed |= (static_cast<uint32_t>(q_round(x[e], s, r)) & cmask) << (w * e);
  }
  return packed;
}

__device__ __forceinline__ void store_lane_codes(uint8_t* group_base, const int w, const int l16,
                                                 const uint32_t packed, const uint2 raw) {
  switch (w) {
    case 2: group_base[l16] = static_cast<uint8_t>(packed); break;
    case 4: reinterpret_cast<uint16_t*>(group_base)[l16] = static_cast<uint16_t>(packed); break;
    case 8: reinterpret_cast<uint32_t*>(group_base)[l16] = packed; break;
    default: reinterpret_cast<uint2*>(group_base)[l16] = raw; break;
  }
}

// Decode this lane's 4 elements of a group.
__device__ __forceinline__ void dequant_lane4(const uint8_t* group_base, const int w, const int l16,
                                              const uint16_t* scale_ptr, float (&y)[4]) {
  if (w == 16) {
    const uint2 raw = reinterpret_cast<const uint2*>(group_base)[l16];
    y[0] = __uint_as_float(raw.x << 16);
    y[1] = __uint_as_float(raw.x & 0xFFFF0000u);
    y[2] = __uint_as_float(raw.y << 16);
    y[3] = __uint_as_float(raw.y & 0xFFFF0000u);
    return;
  }
  uint32_t packed;
  if (w == 2)
    packed = group_base[l16];
  else if (w == 4)
    packed = reinterpret_cast<const uint16_t*>(group_base)[l16];
  else
    packed = reinterpret_cast<const uint32_t*>(group_base)[l16];
  const float s = __half2float(__ushort_as_half(*scale_ptr));
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int code = static_cast<int>((packed >> (w * e)) & ((1u << w) - 1u));
    const int q = code >= (1 << (w - 1)) ? code - (1 << w) : code;
    y[e] = static_cast<float>(q) * s;
  }
}

__device__ __forceinline__ void lane_bf16x4(const uint16_t* src, float (&x)[4], uint2* raw) {
  const uint2 r = *reinterpret_cast<const uint2*>(src);
  *raw = r;
  x[0] = __uint_as_float(r.x << 16);
  x[1] = __uint_as_float(r.x & 0xFFFF0000u);
  x[2] = __uint_as_float(r.y << 16);
  x[3] = __uint_as_float(r.y & 0xFFFF0000u);
}

__device__ __forceinline__ float bf16_lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// plan for token units (axis 0): ids and group offsets of every stored unit
// ---------------------------------------------------------------------------
// Packs the four per-width counters of a thread into two u64 (32 bits each).
__device__ __forceinline__ void plan_pack2(const unsigned (&c)[4], unsigned long long* lo, unsigned long long* hi) {
  *lo = static_cast<unsigned long long>(c[0]) | (static_cast<unsigned long long>(c[1]) << 32);
  *hi = static_cast<unsigned long long>(c[2]) | (static_cast<unsigned long long>(c[3]) << 32);
}

// exclusive scan over the block in thread order (kPlanThreads threads);
// sbuf holds kPlanThreads/32 + 1 entries; *total = block sum.  Sums must stay
// below 2^32 per 32-bit field.
__device__ __forceinline__ unsigned long long plan_block_exscan(unsigned long long v, unsigned long long* sbuf,
                                                                unsigned long long* total) {
  constexpr int NW = kPlanThreads / 32;
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
  if (warp == 0) {
    const unsigned long long t = lane < NW ? sbuf[lane] : 0ull;
    unsigned long long z = t;
#pragma unroll
    for (int o = 1; o < NW; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, z, o);
      if (lane >= o) z += y;
    }
    if (lane < NW) sbuf[lane] = z - t;
    if (lane == NW - 1) sbuf[NW] = z;
  }
  __syncthreads();
  *total = sbuf[NW];
  return sbuf[warp] + x - v;
}

// 16 width bytes starting at unit u (zero past `end`): one 16-byte load
// when aligned and in range, else byte loads
__device__ __forceinline__ uint4 load_bits16(const uint8_t* __restrict__ bits, const long long u, const long long end) {
  if (u + 16 <= end && (reinterpret_cast<uintptr_t>(bits + u) & 15u) == 0)
    return __ldg(reinterpret_cast<const uint4*>(bits + u));
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int e = 0; e < 16; ++e)
    if (u + e < end) w[e >> 2] |= static_cast<uint32_t>(bits[u + e]) << (8 * (e & 3));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ int bits16_at(const uint4& v, int e) {
  const uint32_t w = e < 4 ? v.x : e < 8 ? v.y : e < 12 ? v.z : v.w;
  return static_cast<int>((w >> (8 * (e & 3))) & 0xFFu);
}

// One cluster of CL CTAs; CTA r plans units [r*per, r*per + per) in steps of
// kPlanThreads * 16 units, thread t taking 16 contiguous ones per step.
// Writes ids[s][k] = unit and group_offsets[s][k] = k * groups_per_unit for
// the k-th stored unit of width slot s, and counts.  Each step's ids are
// staged in shared memory by width and then written out contiguously.
// grid (CL * pools): cluster q plans pool q (units q*U .. q*U + U-1 of bits).
template <int CL>
__global__ void __launch_bounds__(kPlanThreads, 1) rows_plan_kernel(const uint8_t* __restrict__ bits,
                                                                    const long long U, const long long per,
                                                                    const int groups_per_unit, const StreamPtrs sp) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  const long long pool = blockIdx.x / CL;
  bits += pool * U;
  namespace cgp = cooperative_groups;
  cgp::cluster_group cluster = cgp::this_cluster();
  const int rank = CL > 1 ? static_cast<int>(cluster.block_rank()) : 0;
  constexpr int kStep = kPlanThreads * 16;
  __shared__ unsigned long long sbuf[kPlanThreads / 32 + 1];
  __shared__ unsigned long long s_tot[2];
  __shared__ unsigned long long s_all[CL][2];
  __shared__ int32_t stage[kStep];
  __shared__ int s_seg[5];
  const long long begin = static_cast<long long>(rank) * per;
  const long long end = min(U, begin + per);
  auto count16 = [&](const uint4& v, unsigned (&c)[4]) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int sl = width_slot(bits16_at(v, e));
      if (sl >= 0) ++c[sl];
    }
  };
  // totals of this CTA's range, then every CTA's, for the running prefix
  unsigned long long tlo = 0, thi = 0;
  for (long long b = begin; b < end; b += kStep) {
    unsigned c[4] = {0u, 0u, 0u, 0u};
    count16(load_bits16(bits, b + threadIdx.x * 16, end), c);
    tlo += static_cast<unsigned long long>(c[0]) | (static_cast<unsigned long long>(c[1]) << 32);
    thi += static_cast<unsigned long long>(c[2]) | (static_cast<unsigned long long>(c[3]) << 32);
  }
  {
    unsigned long long a, bb;
    (void)plan_block_exscan(tlo, sbuf, &a);
    (void)plan_block_exscan(thi, sbuf, &bb);
    if (threadIdx.x == 0) {
      s_tot[0] = a;
      s_tot[1] = bb;
    }
  }
  if (CL > 1) cluster.sync();
  else __syncthreads();
  if (threadIdx.x < CL) {
    const unsigned long long* rt = CL > 1 ? cluster.map_shared_rank(s_tot, static_cast<int>(threadIdx.x)) : s_tot;
    s_all[threadIdx.x][0] = rt[0];
    s_all[threadIdx.x][1] = rt[1];
  }
  __syncthreads();
  unsigned long long plo = 0, phi = 0, glo = 0, ghi = 0;
  for (int q = 0; q < CL; ++q) {
    if (q < rank) {
      plo += s_all[q][0];
      phi += s_all[q][1];
    }
    glo += s_all[q][0];
    ghi += s_all[q][1];
  }
  for (long long b = begin; b < end; b += kStep) {
    const long long u0 = b + threadIdx.x * 16;
    const uint4 v = load_bits16(bits, u0, end);
    unsigned c[4] = {0u, 0u, 0u, 0u};
    count16(v, c);
    unsigned long long slo, shi;
    const unsigned long long elo = plan_block_exscan(
        static_cast<unsigned long long>(c[0]) | (static_cast<unsigned long long>(c[1]) << 32), sbuf, &slo);
    const unsigned long long ehi = plan_block_exscan(
        static_cast<unsigned long long>(c[2]) | (static_cast<unsigned long long>(c[3]) << 32), sbuf, &shi);
    const int st[4] = {static_cast<int>(slo & 0xFFFFFFFFull), static_cast<int>(slo >> 32),
                       static_cast<int>(shi & 0xFFFFFFFFull), static_cast<int>(shi >> 32)};
    const int seg[5] = {0, st[0], st[0] + st[1], st[0] + st[1] + st[2], st[0] + st[1] + st[2] + st[3]};
    int lr[4] = {seg[0] + static_cast<int>(elo & 0xFFFFFFFFull), seg[1] + static_cast<int>(elo >> 32),
                 seg[2] + static_cast<int>(ehi & 0xFFFFFFFFull), seg[3] + static_cast<int>(ehi >> 32)};
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int sl = width_slot(bits16_at(v, e));
      if (sl >= 0 && u0 + e < end) stage[lr[sl]++] = static_cast<int32_t>(u0 + e);
    }
    if (threadIdx.x < 5) s_seg[threadIdx.x] = seg[threadIdx.x];
    __syncthreads();
    const long long base[4] = {static_cast<long long>(plo & 0xFFFFFFFFull), static_cast<long long>(plo >> 32),
                               static_cast<long long>(phi & 0xFFFFFFFFull), static_cast<long long>(phi >> 32)};
    for (int j = threadIdx.x; j < s_seg[4]; j += kPlanThreads) {
      int sl = 0;
      while (sl < 3 && j >= s_seg[sl + 1]) ++sl;
      const long long k = base[sl] + (j - s_seg[sl]);
      if (k < sp.cap_units[sl]) {
        sp.ids[sl][pool * sp.cap_units[sl] + k] = stage[j];
        sp.goff[sl][pool * sp.cap_units[sl] + k] = k * groups_per_unit;
      }
    }
    __syncthreads();  // the stage is reused by the next step
    plo += slo;
    phi += shi;
  }
  if (rank == CL - 1 && threadIdx.x < 4) {
    const int sl = threadIdx.x;
    const unsigned long long tot = sl == 0   ? (glo & 0xFFFFFFFFull)
                                   : sl == 1 ? (glo >> 32)
                                   : sl == 2 ? (ghi & 0xFFFFFFFFull)
                                             : (ghi >> 32);
    const long long units = static_cast<long long>(tot), groups = units * groups_per_unit;
    if (sp.counts) {
      sp.counts[8 * pool + sl] = units;
      sp.counts[8 * pool + 4 + sl] = groups;
    }
    if (units > sp.cap_units[sl] || groups > sp.cap_groups[sl]) record_error(KVS_ERR_RANGE);
  }
  if (CL > 1) cluster.sync();  // keep shared memory alive until every CTA has read the totals
}

// entry offsets (in groups) of the four widths from the device counts
__device__ __forceinline__ void entry_offsets(const StreamPtrs& sp, const int gpu, const long long pool,
                                              long long* s_off) {
  if (threadIdx.x == 0) {
    long long run = 0;
    for (int s = 0; s < 4; ++s) {
      s_off[s] = run;
      run += min(static_cast<long long>(sp.counts[8 * pool + s]), sp.cap_units[s]) * gpu;
    }
    s_off[4] = run;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// token units (axis 0, V cache): one lane per 64-element group, over the
// stream entries the plan wrote (consecutive lanes write consecutive blocks)
// ---------------------------------------------------------------------------
__device__ __forceinline__ int entry_slot(const long long* s_off, const long long gidx) {
  int s = 0;
  while (s < 3 && gidx >= s_off[s + 1]) ++s;
  return s;
}

// grid (blocks, pools): blockIdx.y is the pool (U units of X each)
template <int DH>
__global__ void __launch_bounds__(256) pack_rows_kernel(const uint16_t* __restrict__ X, const StreamPtrs sp,
                                                        const long long U) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  constexpr int GPU = DH / 64;
  __shared__ long long s_off[5];
  const long long pool = blockIdx.y;
  X += pool * U * DH;
  entry_offsets(sp, GPU, pool, s_off);
  const int l16 = threadIdx.x & 15;
  const int total = static_cast<int>(s_off[4]);  // groups < 2^31 (units < 2^31, two groups each)
  const int stride = gridDim.x * (blockDim.x / 16);
  for (int gidx = blockIdx.x * (blockDim.x / 16) + (threadIdx.x >> 4); gidx < total; gidx += stride) {
    const int s = entry_slot(s_off, gidx);
    const int grp = gidx - static_cast<int>(s_off[s]);  // == entry * GPU + gi
    if (grp >= sp.cap_groups[s]) continue;
    const long long u = sp.ids[s][pool * sp.cap_units[s] + grp / GPU];
    const long long gb = pool * sp.cap_groups[s];
    float x[4];
    uint2 raw;
    lane_bf16x4(X + u * DH + (grp % GPU) * 64 + l16 * 4, x, &raw);
    const int w = s == 3 ? 16 : (2 << s);
    uint32_t packed = 0;
    if (w != 16) {
      uint16_t sb;
      bool ovf;
      packed = quantize_lane4(x, w, &sb, &ovf);
      if (l16 == 0) {
        sp.scales[s][gb + grp] = sb;
        if (ovf) record_error(KVS_ERR_RANGE);
      }
    }
    store_lane_codes(sp.codes[s] + (gb + grp) * (8 * w), w, l16, packed, raw);
  }
}

// Token units decoded from the stream entries (entry j of width slot s is
// unit ids[s][j] with groups goff[s][j] ..), one half-warp per group; rows of
// evicted units (bits == 0) are zeroed in the same launch, one warp per row.
// grid (blocks, pools): blockIdx.y is the pool (U units of bits and out each)
template <int DH>
__global__ void __launch_bounds__(256) dequant_rows_kernel(const StreamPtrs sp, const uint8_t* __restrict__ bits,
                                                           const long long U, float* __restrict__ out) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  constexpr int GPU = DH / 64;
  __shared__ long long s_off[5];
  const long long pool = blockIdx.y;
  bits += pool * U;
  out += pool * U * DH;
  entry_offsets(sp, GPU, pool, s_off);
  const int l16 = threadIdx.x & 15;
  const int total = static_cast<int>(s_off[4]);
  const int stride = gridDim.x * (blockDim.x / 16);
  for (int gidx = blockIdx.x * (blockDim.x / 16) + (threadIdx.x >> 4); gidx < total; gidx += stride) {
    const int s = entry_slot(s_off, gidx);
    const int local = gidx - static_cast<int>(s_off[s]);
    const int jj = local / GPU, gi = local % GPU;
    const long long u = sp.ids[s][pool * sp.cap_units[s] + jj];
    const long long grp = sp.goff[s][pool * sp.cap_units[s] + jj] + gi;
    if (grp >= sp.cap_groups[s]) continue;
    const long long gg = pool * sp.cap_groups[s] + grp;
    const int w = s == 3 ? 16 : (2 << s);
    float y[4];
    dequant_lane4(sp.codes[s] + gg * (8 * w), w, l16, sp.scales[s] + gg, y);
    *reinterpret_cast<float4*>(out + u * DH + gi * 64 + l16 * 4) = make_float4(y[0], y[1], y[2], y[3]);
  }
  // evicted rows: a warp takes 32 rows, then zeroes the ones with width 0
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  for (long long r0 = (static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5)) * 32; r0 < U;
       r0 += nwarps * 32) {
    const bool zero = r0 + lane < U && bits[r0 + lane] == 0;
    unsigned m = __ballot_sync(0xFFFFFFFFu, zero);
    while (m) {
      const int i = __ffs(m) - 1;
      m &= m - 1;
      float4* o4 = reinterpret_cast<float4*>(out + (r0 + i) * DH);
      for (int c4 = lane; c4 < DH / 4; c4 += 32) o4[c4] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// ---------------------------------------------------------------------------
// channel units (axis 1, K cache) over the tokens each head keeps
// ---------------------------------------------------------------------------
// One cluster of CL CTAs; CTA r handles heads r, r + CL, ...:
//   kept[g][0 .. n_kept) = the kept tokens of head g, ascending;
//   kept[g][n_kept .. N) = its dropped tokens (descending from the end); n_kept[g].
// Then CTA 0 plans the channel units u = g*DH + c in unit order:
//   chan_base[u] = first stream group of unit u (-1: not stored), and, with
//   write_streams, ids / group offsets / counts (a unit of head g has
//   ceil(n_kept[g] / 64) groups).
template <int DH>
__global__ void __launch_bounds__(kPlanThreads, 1) channels_plan_kernel(
    const uint8_t* __restrict__ keep, const int N, const int Hkv, const uint8_t* __restrict__ bits,
    int* __restrict__ kept, int* __restrict__ n_kept, long long* __restrict__ chan_base, const StreamPtrs sp,
    const int write_streams) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  namespace cgp = cooperative_groups;
  cgp::cluster_group cluster = cgp::this_cluster();
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  // cluster q plans pool q: its Hkv heads of keep / kept / n_kept and Hkv*DH units
  const long long pool = blockIdx.x / CL;
  keep += pool * Hkv * N;
  kept += pool * Hkv * N;
  n_kept += pool * Hkv;
  bits += pool * Hkv * DH;
  chan_base += pool * Hkv * DH;
  __shared__ unsigned long long sbuf[kPlanThreads / 32 + 1];
  constexpr int kStep = kPlanThreads * 16;
  for (int g = rank; g < Hkv; g += CL) {
    const uint8_t* kb = keep + static_cast<size_t>(g) * N;
    int* kg = kept + static_cast<size_t>(g) * N;
    unsigned long long carry = 0;  // kept tokens before this step
    for (int b = 0; b < N; b += kStep) {
      const int t0 = b + threadIdx.x * 16;
      const uint4 v = load_bits16(kb, t0, N);
      unsigned mask = 0;
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (bits16_at(v, e) != 0) mask |= 1u << e;
      unsigned long long step_tot;
      const unsigned long long ex = plan_block_exscan(__popc(mask), sbuf, &step_tot);
      int pk = static_cast<int>(carry + ex);       // next kept slot
      int pd = N - 1 - (t0 - pk);                  // next dropped slot, from the end
      const int valid = max(0, min(16, N - t0));
      for (int e = 0; e < valid; ++e) {
        if (mask & (1u << e))
          kg[pk++] = t0 + e;
        else
          kg[pd--] = t0 + e;
      }
      carry += step_tot;
    }
    if (threadIdx.x == 0) n_kept[g] = static_cast<int>(carry);
  }
  cluster.sync();  // every head's kept count is written (cluster scope orders global memory)
  if (rank != 0) return;
  // channel plan: thread t takes units [t*m, t*m + m); per-width unit counts
  // (16-bit fields) and group counts (32-bit fields) scanned over the block
  const int U = Hkv * DH;
  const int m = (U + kPlanThreads - 1) / kPlanThreads;
  const int u0 = threadIdx.x * m, u1 = min(U, u0 + m);
  unsigned long long cu = 0, cg01 = 0, cg23 = 0;
  for (int u = u0; u < u1; ++u) {
    const int sl = width_slot(bits[u]);
    if (sl < 0) continue;
    const unsigned long long ng = static_cast<unsigned long long>((__ldcg(n_kept + u / DH) + 63) / 64);
    cu += 1ull << (16 * sl);
    if (sl < 2) cg01 += ng << (32 * sl);
    else cg23 += ng << (32 * (sl - 2));
  }
  unsigned long long tu, t01, t23;
  const unsigned long long eu = plan_block_exscan(cu, sbuf, &tu);
  const unsigned long long e01 = plan_block_exscan(cg01, sbuf, &t01);
  const unsigned long long e23 = plan_block_exscan(cg23, sbuf, &t23);
  long long ru[4], rg[4];
  for (int sl = 0; sl < 4; ++sl) {
    ru[sl] = static_cast<long long>((eu >> (16 * sl)) & 0xFFFFull);
    rg[sl] = static_cast<long long>(sl < 2 ? (e01 >> (32 * sl)) & 0xFFFFFFFFull : (e23 >> (32 * (sl - 2))) & 0xFFFFFFFFull);
  }
  for (int u = u0; u < u1; ++u) {
    const int sl = width_slot(bits[u]);
    if (sl < 0) {
      chan_base[u] = -1;
      continue;
    }
    const long long ng = (__ldcg(n_kept + u / DH) + 63) / 64;
    const bool fits = ru[sl] < sp.cap_units[sl] && rg[sl] + ng <= sp.cap_groups[sl];
    chan_base[u] = fits ? rg[sl] : -1;
    if (write_streams && fits) {
      sp.ids[sl][pool * sp.cap_units[sl] + ru[sl]] = u;
      sp.goff[sl][pool * sp.cap_units[sl] + ru[sl]] = rg[sl];
    }
    ++ru[sl];
    rg[sl] += ng;
  }
  if (threadIdx.x < 4 && write_streams) {
    const int sl = threadIdx.x;
    const long long units = static_cast<long long>((tu >> (16 * sl)) & 0xFFFFull);
    const long long groups =
        static_cast<long long>(sl < 2 ? (t01 >> (32 * sl)) & 0xFFFFFFFFull : (t23 >> (32 * (sl - 2))) & 0xFFFFFFFFull);
    if (sp.counts) {
      sp.counts[8 * pool + sl] = units;
      sp.counts[8 * pool + 4 + sl] = groups;
    }
    if (units > sp.cap_units[sl] || groups > sp.cap_groups[sl]) record_error(KVS_ERR_RANGE);
  }
}

// grid (ceil(N/64), Hkv), 256 threads: kept-token group j of head g for every
// channel; one half-warp per channel (lane i: tokens 4i..4i+3)
// (blockIdx.y runs over the heads of every pool: pool blockIdx.y / Hkv)
template <int DH>
__global__ void __launch_bounds__(256) pack_channels_kernel(const uint16_t* __restrict__ X, const int N,
                                                            const uint8_t* __restrict__ bits,
                                                            const long long* __restrict__ chan_base,
                                                            const int* __restrict__ kept,
                                                            const int* __restrict__ n_kept, const StreamPtrs sp,
                                                            const int Hkv) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  // odd word stride: the column reads below (lane i takes rows 4i..4i+3)
  // spread over the banks instead of piling onto two
  constexpr int LDW = DH / 2 + 1;  // 32-bit words per row
  __shared__ uint32_t tile[64][LDW];
  __shared__ int s_w[DH];
  __shared__ long long s_base[DH];
  const int j = blockIdx.x, g = blockIdx.y;
  const int n = n_kept[g];
  if (j * 64 >= n) return;
  const int rows = min(64, n - j * 64);
  for (int c = threadIdx.x; c < DH; c += blockDim.x) {
    const long long b = chan_base[g * DH + c];
    s_w[c] = bits[g * DH + c];
    s_base[c] = b >= 0 ? b + j : -1;
  }
  for (int e = threadIdx.x; e < 64 * (DH / 8); e += 256) {
    const int i = e / (DH / 8), c8 = (e % (DH / 8)) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (i < rows) {
      const int t = kept[static_cast<size_t>(g) * N + j * 64 + i];
      v = __ldg(reinterpret_cast<const uint4*>(X + (static_cast<size_t>(g) * N + t) * DH + c8));
    }
    uint32_t* row = &tile[i][c8 / 2];
    row[0] = v.x;
    row[1] = v.y;
    row[2] = v.z;
    row[3] = v.w;
  }
  __syncthreads();
  const int l16 = threadIdx.x & 15, hw = threadIdx.x >> 4;
  for (int c = hw; c < DH; c += 16) {
    const long long grp = s_base[c];
    if (grp < 0) continue;
    const int w = s_w[c];
    const int s = width_slot(w);
    const long long gg = static_cast<long long>(g / Hkv) * sp.cap_groups[s] + grp;
    float x[4];
    uint32_t rw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      rw[e] = (tile[4 * l16 + e][c >> 1] >> ((c & 1) * 16)) & 0xFFFFu;
      x[e] = __uint_as_float(rw[e] << 16);
    }
    const uint2 raw = make_uint2(rw[0] | (rw[1] << 16), rw[2] | (rw[3] << 16));
    uint32_t packed = 0;
    if (w != 16) {
      uint16_t sb;
      bool ovf;
      packed = quantize_lane4(x, w, &sb, &ovf);
      if (l16 == 0) {
        sp.scales[s][gg] = sb;
        if (ovf) record_error(KVS_ERR_RANGE);
      }
    }
    store_lane_codes(sp.codes[s] + gg * (8 * w), w, l16, packed, raw);
  }
}

// grid (ceil(N/64) + 1, Hkv), 256 threads.  CTA (j, g) with j below the head's
// kept-group count decodes kept-token group j of every channel (one
// half-warp per channel) through a shared-memory tile and writes the tokens'
// rows; the CTAs after those zero the head's dropped tokens, 64 per CTA.
// (blockIdx.y runs over the heads of every pool: pool blockIdx.y / Hkv)
template <int DH>
__global__ void __launch_bounds__(256) dequant_channels_kernel(const StreamPtrs sp, const int N,
                                                               const uint8_t* __restrict__ bits,
                                                               const long long* __restrict__ chan_base,
                                                               const int* __restrict__ kept,
                                                               const int* __restrict__ n_kept,
                                                               float* __restrict__ out, const int Hkv) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  constexpr int LD = DH + 1;  // odd stride: conflict-light column writes
  __shared__ float tile[64][LD];
  __shared__ int s_w[DH];
  __shared__ long long s_base[DH];
  const int j = blockIdx.x, g = blockIdx.y;
  const int n = n_kept[g];
  const int ngk = (n + 63) / 64;
  if (j >= ngk) {  // zero dropped tokens kept[g][n + 64 jz ..]
    const int d0 = n + (j - ngk) * 64;
    if (d0 >= N) return;
    const int cnt = min(64, N - d0);
    for (int e = threadIdx.x; e < cnt * (DH / 4); e += 256) {
      const int i = e / (DH / 4), c4 = (e % (DH / 4)) * 4;
      const int t = kept[static_cast<size_t>(g) * N + d0 + i];
      *reinterpret_cast<float4*>(out + (static_cast<size_t>(g) * N + t) * DH + c4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  const int rows = min(64, n - j * 64);
  for (int c = threadIdx.x; c < DH; c += blockDim.x) {
    const long long b = chan_base[g * DH + c];
    s_w[c] = bits[g * DH + c];
    s_base[c] = b >= 0 ? b + j : -1;
  }
  __syncthreads();
  const int l16 = threadIdx.x & 15, hw = threadIdx.x >> 4;
  for (int c = hw; c < DH; c += 16) {
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    const long long grp = s_base[c];
    if (grp >= 0) {
      const int w = s_w[c];
      const int s = width_slot(w);
      const long long gg = static_cast<long long>(g / Hkv) * sp.cap_groups[s] + grp;
      dequant_lane4(sp.codes[s] + gg * (8 * w), w, l16, sp.scales[s] + gg, y);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) tile[4 * l16 + e][c] = y[e];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < rows * (DH / 4); e += 256) {
    const int i = e / (DH / 4), c4 = (e % (DH / 4)) * 4;
    const int t = kept[static_cast<size_t>(g) * N + j * 64 + i];
    *reinterpret_cast<float4*>(out + (static_cast<size_t>(g) * N + t) * DH + c4) =
        make_float4(tile[i][c4], tile[i][c4 + 1], tile[i][c4 + 2], tile[i][c4 + 3]);
  }
}

// ---------------------------------------------------------------------------
// dequantise the channel streams without a plan kernel (N <= kDirectMaxN)
// ---------------------------------------------------------------------------
// grid (ceil(N/64) + 1, Hkv), 256 threads.  Each CTA works out for its own
// head what the plan kernel would give: the kept tokens in order (a block scan
// of the head's keep bytes) and each channel's first stream group (the entry
// of unit g*DH + c in its width stream is the number of earlier units of that
// width; the group offset is read back from the stream).  CTA j < ngk decodes
// kept-token group j; the CTAs after those zero the head's dropped tokens.
constexpr int kDirectMaxN = 16384;

__device__ __forceinline__ unsigned long long direct_exscan256(unsigned long long v, unsigned long long* sbuf,
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
  if (warp == 0) {
    const unsigned long long t = lane < 8 ? sbuf[lane] : 0ull;
    unsigned long long z = t;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, z, o);
      if (lane >= o) z += y;
    }
    if (lane < 8) sbuf[lane] = z - t;
    if (lane == 7) sbuf[8] = z;
  }
  __syncthreads();
  *total = sbuf[8];
  return sbuf[warp] + x - v;
}

// (blockIdx.y runs over the heads of every pool: pool blockIdx.y / Hkv)
template <int DH>
__global__ void __launch_bounds__(256) dequant_channels_direct_kernel(const StreamPtrs sp, const int N,
                                                                      const uint8_t* __restrict__ bits,
                                                                      const uint8_t* __restrict__ keep,
                                                                      float* __restrict__ out, const int Hkv) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  constexpr int LD = DH + 1;
  __shared__ float tile[64][LD];
  __shared__ int s_w[DH];
  __shared__ long long s_base[DH];
  __shared__ int s_tok[64];
  __shared__ unsigned long long sbuf[9];
  const int j = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
  // ---- the head's kept tokens: thread tid takes bytes [t0, t0 + per) ----
  const int per = ((N + 255) / 256 + 15) / 16 * 16;
  const int t0 = tid * per;
  const uint8_t* kb = keep + static_cast<size_t>(g) * N;
  int cnt = 0;
  for (int e = 0; e < per; e += 16) {
    if (t0 + e >= N) break;
    const uint4 v = load_bits16(kb, t0 + e, N);
#pragma unroll
    for (int k = 0; k < 16; ++k) cnt += (t0 + e + k < N && bits16_at(v, k) != 0) ? 1 : 0;
  }
  unsigned long long tot;
  const int ex = static_cast<int>(direct_exscan256(static_cast<unsigned long long>(cnt), sbuf, &tot));
  const int n = static_cast<int>(tot);
  const int ngk = (n + 63) / 64;
  const bool kept_cta = j < ngk;
  // this CTA's 64 list entries: kept ranks [64j, 64j + 64), or dropped ranks after the kept groups
  const int lo = kept_cta ? 64 * j : 64 * (j - ngk);
  const int hi = lo + 64;
  const int my_lo = kept_cta ? ex : t0 - ex;                       // first kept / dropped rank of my bytes
  const int my_n = kept_cta ? cnt : max(0, min(per, N - t0)) - cnt;
  if (my_lo < hi && my_lo + my_n > lo) {
    int r = my_lo;
    for (int e = 0; e < per && t0 + e < N; ++e) {
      const bool kept = kb[t0 + e] != 0;
      if (kept == kept_cta) {
        if (r >= lo && r < hi) s_tok[r - lo] = t0 + e;
        ++r;
      }
    }
  }
  const int rows = kept_cta ? min(64, n - lo) : max(0, min(64, (N - n) - lo));
  if (!kept_cta) {
    __syncthreads();
    for (int e = tid; e < rows * (DH / 4); e += 256) {
      const int i = e / (DH / 4), c4 = (e % (DH / 4)) * 4;
      *reinterpret_cast<float4*>(out + (static_cast<size_t>(g) * N + s_tok[i]) * DH + c4) =
          make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  // ---- each channel's entry in its width stream, then its first group ----
  unsigned long long before = 0;                   // units of each width before this head, 16-bit fields
  const long long pool = g / Hkv;
  const uint8_t* pbits = bits + pool * Hkv * DH;   // the pool's unit widths
  for (int u = tid; u < (g % Hkv) * DH; u += 256) {
    const int sl = width_slot(pbits[u]);
    if (sl >= 0) before += 1ull << (16 * sl);
  }
  unsigned long long base_all;
  (void)direct_exscan256(before, sbuf, &base_all);
  const int sl_me = tid < DH ? width_slot(bits[g * DH + tid]) : -1;
  const unsigned long long mine = sl_me >= 0 ? 1ull << (16 * sl_me) : 0ull;
  unsigned long long head_tot;
  const unsigned long long exh = direct_exscan256(mine, sbuf, &head_tot);
  if (tid < DH) {
    long long b = -1;
    if (sl_me >= 0) {
      const long long entry = static_cast<long long>(((base_all + exh) >> (16 * sl_me)) & 0xFFFFull);
      if (entry < sp.cap_units[sl_me]) b = sp.goff[sl_me][pool * sp.cap_units[sl_me] + entry] + j;
      if (b >= sp.cap_groups[sl_me]) b = -1;
    }
    s_w[tid] = sl_me >= 0 ? static_cast<int>(bits[g * DH + tid]) : 0;
    s_base[tid] = b;
  }
  __syncthreads();
  const int l16 = threadIdx.x & 15, hw = threadIdx.x >> 4;
  for (int c = hw; c < DH; c += 16) {
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    const long long grp = s_base[c];
    if (grp >= 0) {
      const int w = s_w[c];
      const int s = width_slot(w);
      const long long gg = pool * sp.cap_groups[s] + grp;
      dequant_lane4(sp.codes[s] + gg * (8 * w), w, l16, sp.scales[s] + gg, y);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) tile[4 * l16 + e][c] = y[e];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < rows * (DH / 4); e += 256) {
    const int i = e / (DH / 4), c4 = (e % (DH / 4)) * 4;
    *reinterpret_cast<float4*>(out + (static_cast<size_t>(g) * N + s_tok[i]) * DH + c4) =
        make_float4(tile[i][c4], tile[i][c4 + 1], tile[i][c4 + 2], tile[i][c4 + 3]);
  }
}

}  // namespace kvs
