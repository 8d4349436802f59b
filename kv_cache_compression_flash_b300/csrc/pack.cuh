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

// the w-bit two's-complement code in the low bits of c, as a float (exact:
// the integer is added to 1.5 * 2^23 in the mantissa, no conversion unit)
__device__ __forceinline__ float code_to_float(const uint32_t c, const int w) {
  const int q = static_cast<int>(c << (32 - w)) >> (32 - w);
  return __fsub_rn(__int_as_float(0x4B400000 + q), 12582912.f);
}

// max of two packed bf16 pairs
__device__ __forceinline__ uint32_t bf16x2_max(const uint32_t a, const uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Round-half-even of t = x r on the FMA pipe, two elements per instruction:
// adding 1.5 * 2^23 rounds |t| < 2^22 to the nearest integer (ties to even),
// which lands in the low mantissa bits, so the low w bits of y's pattern are
// the w-bit two's-complement code.  d = t - (y - 1.5 * 2^23) is exact; an
// element with |d| within 2^-14 of 1/2 may round differently from x / s, and
// q_round settles those exactly.
//
// How far x / s can be from a half integer h: with x = m_x 2^(e_x - 7) (bf16)
// and s = m_s 2^(e_s - 10) (fp16), x - h s is a multiple of 2^(e_s - 11)
// whenever |x / s| >= 1/8, so x / s is either exactly h or at least 2^-12
// away from it; x r is within 2^-16 of x / s, so only exact ties can round
// the wrong way.  At width 2 (|x / s| <= 1) the only half integers are
// +-1/2, whose even neighbour is 0: with r = 1/s rounded toward zero, |x r|
// <= |x / s|, so a tie lands on or below 1/2 and rounds to 0, and every other
// quotient rounds as x / s does.  Width 2 therefore needs no check at all;
// there ties are common (s is the group maximum itself, so an element equal
// to half of it is one), at widths 4 and 8 they are rare.
constexpr float kRoundMagic = 12582912.f;                             // 1.5 * 2^23
constexpr float kNearHalfSq = 0.49993896484375f * 0.49993896484375f;  // (1/2 - 2^-14)^2
constexpr float kNoCheck = 4.f;                                       // above every d^2: never near

// the reciprocal the quantisers use at width w (see above)
__device__ __forceinline__ float quant_recip(const float s, const int w) {
  return w == 2 ? __frcp_rz(s) : __frcp_rn(s);
}


__device__ __forceinline__ float bf16_lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }

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

// exclusive scan over a block of NT threads in thread order; sbuf holds
// NT/32 + 1 entries; *total = block sum.  Fields packed into the 64 bits
// must not carry into each other.
template <int NT>
__device__ __forceinline__ unsigned long long block_exscan_u64(unsigned long long v, unsigned long long* sbuf,
                                                               unsigned long long* total) {
  constexpr int NW = NT / 32;
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

// ---------------------------------------------------------------------------
// token units (axis 0, V cache), in unit order
// ---------------------------------------------------------------------------
// A pool's units are cut into chunks of kRowChunk.  rows_count_kernel counts
// each chunk's units per stored width; the pack and dequantise kernels take
// one chunk per CTA: the counts of the earlier chunks give the chunk's first
// entry in every width stream, a block scan of its widths the entry of each
// unit (the k-th stored unit of width w is entry k of stream w, so the
// streams stay in ascending unit order).  Rows are then read or written in
// unit order, 16 bytes a lane and eight lanes per 64-element group, with no
// indirection between the loads.
constexpr int kRowChunk = 1024;
constexpr int kRowThreads = 256;
static_assert(kRowChunk == 4 * kRowThreads, "four units per thread");

// cnt[(pool * n_chunks + chunk) * 4 + slot] = units of the chunk stored in width slot `slot`
__global__ void __launch_bounds__(kRowThreads) rows_count_kernel(const uint8_t* __restrict__ bits, const long long U,
                                                                 const int n_chunks, uint32_t* __restrict__ cnt) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  const long long pool = blockIdx.y;
  const long long u0 = static_cast<long long>(blockIdx.x) * kRowChunk;
  bits += pool * U;
  unsigned long long c = 0;  // four 16-bit counters
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const long long u = u0 + threadIdx.x * 4 + e;
    const int sl = u < U ? width_slot(bits[u]) : -1;
    if (sl >= 0) c += 1ull << (16 * sl);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
  __shared__ unsigned long long s[kRowThreads / 32];
  if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x < 4) {
    unsigned long long t = 0;
#pragma unroll
    for (int i = 0; i < kRowThreads / 32; ++i) t += s[i];
    cnt[(pool * n_chunks + blockIdx.x) * 4 + threadIdx.x] = static_cast<uint32_t>((t >> (16 * threadIdx.x)) & 0xFFFFull);
  }
}

// The chunk blockIdx.x of pool `pool`: s_w[i] = width of unit u0 + i, s_ent[i]
// = its entry in its width stream (-1: width 0, or past the capacity).  With
// write_streams, also the unit ids and group offsets of the chunk's entries
// and, from the pool's last chunk, the counts.  With s_list, the chunk's
// stored units grouped by width slot, ascending within a slot (slot q's
// units at s_list[lists[q] .. lists[q + 1])), and *slot_units = the units
// per slot in four 16-bit fields.  Returns the chunk's units.
__device__ __forceinline__ int rows_chunk_plan(const uint8_t* __restrict__ bits, const long long U, const int n_chunks,
                                               const uint32_t* __restrict__ cnt, const long long pool, const int gpu,
                                               const StreamPtrs& sp, const bool write_streams, int* s_ent,
                                               uint8_t* s_w, long long* s_base, unsigned long long* sbuf,
                                               uint16_t* s_list = nullptr, unsigned long long* slot_units = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = blockIdx.x;
  const long long u0 = static_cast<long long>(chunk) * kRowChunk;
  const int n = static_cast<int>(min(static_cast<long long>(kRowChunk), U - u0));
  if (warp < 4) {  // the chunk's first entry per width: the earlier chunks' counts
    long long a = 0;
    const uint32_t* cp = cnt + pool * n_chunks * 4 + warp;
    for (int c = lane; c < chunk; c += 32) a += cp[static_cast<long long>(c) * 4];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
    if (lane == 0) s_base[warp] = a;
  }
  uint32_t wv = 0;
  unsigned long long c = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int i = tid * 4 + e;
    const uint32_t b = i < n ? bits[u0 + i] : 0u;
    wv |= b << (8 * e);
    const int sl = width_slot(b);
    if (sl >= 0) c += 1ull << (16 * sl);
  }
  unsigned long long tot;
  unsigned long long ex = block_exscan_u64<kRowThreads>(c, sbuf, &tot);  // its barriers also publish s_base
  // start of each slot's list: the chunk totals of the slots below it (16-bit fields)
  const unsigned long long list0 = (tot << 16) + (tot << 32) + (tot << 48);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int i = tid * 4 + e;
    const uint32_t b = (wv >> (8 * e)) & 0xFFu;
    const int sl = width_slot(b);
    int ent = -1;
    if (sl >= 0 && i < n) {
      if (s_list) s_list[((list0 + ex) >> (16 * sl)) & 0xFFFFull] = static_cast<uint16_t>(i);
      const long long k = s_base[sl] + static_cast<long long>((ex >> (16 * sl)) & 0xFFFFull);
      ex += 1ull << (16 * sl);
      if (k < sp.cap_units[sl]) {
        ent = static_cast<int>(k);
        if (write_streams) {
          sp.ids[sl][pool * sp.cap_units[sl] + k] = static_cast<int32_t>(u0 + i);
          sp.goff[sl][pool * sp.cap_units[sl] + k] = k * gpu;
        }
      }
    }
    s_ent[i] = ent;
    s_w[i] = static_cast<uint8_t>(b);
  }
  if (write_streams && chunk == n_chunks - 1 && tid < 4) {
    const long long units = s_base[tid] + static_cast<long long>((tot >> (16 * tid)) & 0xFFFFull);
    const long long groups = units * gpu;
    if (sp.counts) {
      sp.counts[8 * pool + tid] = units;
      sp.counts[8 * pool + 4 + tid] = groups;
    }
    if (units > sp.cap_units[tid] || groups > sp.cap_groups[tid]) record_error(KVS_ERR_RANGE);
  }
  if (slot_units) *slot_units = tot;
  __syncthreads();
  return n;
}

__device__ __forceinline__ void bf16x8(const uint4 u, float (&x)[8]) {
  const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(v[k] << 16);
    x[2 * k + 1] = __uint_as_float(v[k] & 0xFFFF0000u);
  }
}

// Offset-binary rounding at width W (2, 4 or 8): adding M = 1.5 * 2^23 +
// 2^(W-1) to t = x r in one FMA rounds t to the nearest integer q (ties to
// even: M is even) and leaves c = q + 2^(W-1), which lies in [1, 2^W - 1], in
// the low bits of the result's pattern, above the pattern of 1.5 * 2^23.  The
// W-bit two's-complement code of q is c with its top bit flipped.  So the
// codes of 8 elements at bits [W e, W e + W) are the sum of the patterns
// shifted by W e (one shift-add each), minus the same sum over 1.5 * 2^23's
// pattern, with every code's top bit flipped; each c fits its field, so the
// fields never carry into each other.
template <int W>
struct OffsetCode {
  static constexpr float kMagic = 12582912.f + static_cast<float>(1 << (W - 1));
  static constexpr uint32_t kBase = 0x4B400000u;  // the pattern of 1.5 * 2^23
  static constexpr int kPerWord = 32 / W;  // codes per 32-bit word
  // sum of kBase << (W e) over the word's codes, mod 2^32
  static constexpr uint32_t kBaseSum = [] {
    uint32_t v = 0u;
    for (int e = 0; e < kPerWord; ++e) v += kBase << (W * e);
    return v;
  }();
  // every code's top bit
  static constexpr uint32_t kTopBits = [] {
    uint32_t v = 0u;
    for (int e = 0; e < kPerWord; ++e) v |= (1u << (W - 1)) << (W * e);
    return v;
  }();
};

// The codes of NE elements of one group (scale s > 0, r = quant_recip(s, W))
// at width W: element e at bits [W e, W e + W) of words[], NE W / 32 words.
// At widths 4 and 8, elements whose x r lies within 2^-14 of a half integer
// are settled by q_round.
template <int W, int NE>
__device__ __forceinline__ void quantize_w(const float (&x)[NE], const float s, const float r,
                                           uint32_t (&words)[NE * W / 32]) {
  using OC = OffsetCode<W>;
  const unsigned long long r2 = f2_pack(r, r), m2 = f2_pack(OC::kMagic, OC::kMagic), neg1 = f2_pack(-1.f, -1.f);
  uint32_t yb[NE];
  float dd[NE];
#pragma unroll
  for (int k = 0; k < NE / 2; ++k) {
    const unsigned long long xp = f2_pack(x[2 * k], x[2 * k + 1]);
    const unsigned long long y = f2_fma(xp, r2, m2);  // M + round(x r)
    float y0, y1;
    f2_unpack(y, &y0, &y1);
    yb[2 * k] = __float_as_uint(y0);
    yb[2 * k + 1] = __float_as_uint(y1);
    if constexpr (W != 2) {  // width 2 (r rounded toward zero) is exact as it stands
      const unsigned long long nq = f2_fma(y, neg1, m2);  // -round(x r), exact
      const unsigned long long d = f2_fma(xp, r2, nq);    // x r - round(x r)
      f2_unpack(f2_mul(d, d), &dd[2 * k], &dd[2 * k + 1]);
    }
  }
  if constexpr (W != 2) {
    float m = dd[0];
#pragma unroll
    for (int e = 1; e + 1 < NE; e += 2) m = fmax3(m, dd[e], dd[e + 1]);
    if (NE % 2 == 0) m = fmaxf(m, dd[NE - 1]);
    if (m >= kNearHalfSq) {
#pragma unroll
      for (int e = 0; e < NE; ++e)
        yb[e] = OC::kBase + (1u << (W - 1)) + static_cast<uint32_t>(q_round(x[e], s, r));  // the exact test
    }
  }
#pragma unroll
  for (int h = 0; h < NE * W / 32; ++h) {
    uint32_t acc = 0u;
#pragma unroll
    for (int f = 0; f < OC::kPerWord; ++f) acc += yb[h * OC::kPerWord + f] << (W * f);
    words[h] = (acc - OC::kBaseSum) ^ OC::kTopBits;
  }
}

// The offset code of quantize_w with the width w (2, 4 or 8) in
// registers instead of the instruction stream, so lanes of one warp that hold
// channels of different widths run the same instructions: the codes of 8
// elements are a = sum over e < 4 and b = sum over e >= 4 of the patterns
// times 2^(w (e mod 4)); the low word is a + b 2^(4w) (w <= 4) or a (w = 8),
// the high word 0 or b, each minus the same sums over 1.5 * 2^23's pattern
// and with the codes' top bits flipped.
struct DynCode {
  float magic;                 // 1.5 * 2^23 + 2^(w-1)
  float near_sq;               // kNearHalfSq, or kNoCheck at width 2
  uint32_t half;               // 2^(w-1)
  uint32_t m1, m2, m3;         // 2^w, 2^2w, 2^3w
  uint32_t mhi, hsel;          // 2^4w and 0 (w <= 4); 0 and 1 (w = 8)
  uint32_t sub_lo, xor_lo, sub_hi, xor_hi;
};

__device__ __forceinline__ DynCode dyn_code(const int w) {
  DynCode c;
  c.half = 1u << (w - 1);
  c.magic = 12582912.f + static_cast<float>(c.half);
  c.near_sq = w == 2 ? kNoCheck : kNearHalfSq;
  c.m1 = 1u << w;
  c.m2 = c.m1 * c.m1;
  c.m3 = c.m2 * c.m1;
  const uint32_t sum4 = 1u + c.m1 + c.m2 + c.m3;  // 2^(w e) over e < 4
  const uint32_t s4 = OffsetCode<2>::kBase * sum4, t4 = c.half * sum4;
  if (w == 8) {
    c.mhi = 0u, c.hsel = 1u, c.sub_lo = s4, c.xor_lo = t4, c.sub_hi = s4, c.xor_hi = t4;
  } else {
    const uint32_t m4 = c.m2 * c.m2;
    c.mhi = m4, c.hsel = 0u, c.sub_lo = s4 + s4 * m4, c.xor_lo = t4 + t4 * m4, c.sub_hi = 0u, c.xor_hi = 0u;
  }
  return c;
}

// the 8w code bits of x[0..7] (scale s > 0, r = quant_recip(s, w)) at the width of c
__device__ __forceinline__ unsigned long long quantize_octet_dyn(const float (&x)[8], const float s, const float r,
                                                                 const DynCode& c) {
  const unsigned long long r2 = f2_pack(r, r), m2 = f2_pack(c.magic, c.magic), neg1 = f2_pack(-1.f, -1.f);
  uint32_t yb[8];
  float dd[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const unsigned long long xp = f2_pack(x[2 * k], x[2 * k + 1]);
    const unsigned long long y = f2_fma(xp, r2, m2);
    const unsigned long long nq = f2_fma(y, neg1, m2);
    const unsigned long long d = f2_fma(xp, r2, nq);
    float y0, y1;
    f2_unpack(y, &y0, &y1);
    yb[2 * k] = __float_as_uint(y0);
    yb[2 * k + 1] = __float_as_uint(y1);
    f2_unpack(f2_mul(d, d), &dd[2 * k], &dd[2 * k + 1]);
  }
  if (fmax3(fmax3(dd[0], dd[1], dd[2]), fmax3(dd[3], dd[4], dd[5]), fmaxf(dd[6], dd[7])) >= c.near_sq) {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      yb[e] = OffsetCode<2>::kBase + c.half + static_cast<uint32_t>(q_round(x[e], s, r));  // the exact test
  }
  const uint32_t a = yb[0] + yb[1] * c.m1 + yb[2] * c.m2 + yb[3] * c.m3;
  const uint32_t b = yb[4] + yb[5] * c.m1 + yb[6] * c.m2 + yb[7] * c.m3;
  const uint32_t lo = (a + b * c.mhi - c.sub_lo) ^ c.xor_lo;
  const uint32_t hi = (b * c.hsel - c.sub_hi) ^ c.xor_hi;
  return static_cast<unsigned long long>(lo) | (static_cast<unsigned long long>(hi) << 32);
}

// Pack this lane's 16 elements of the groups of kRowSteps warp steps at
// width W (warp-uniform).  Lanes 4j .. 4j + 3 hold one group; ent[k] < 0: no
// group.
constexpr int kRowSteps = 2;

template <int W, int GPU>
__device__ __forceinline__ void pack_rows_steps(const StreamPtrs& sp, const long long pool, const int slot,
                                                const int l4, const int gi, const uint4 (&raw)[kRowSteps][2],
                                                const int (&ent)[kRowSteps]) {
#pragma unroll
  for (int k = 0; k < kRowSteps; ++k) {
    const long long gg = pool * sp.cap_groups[slot] + static_cast<long long>(ent[k]) * GPU + gi;
    // the group's stores (not its shuffles, which every lane joins) are skipped when out of bounds
    const bool store = ent[k] >= 0 && KVS_IN_BOUNDS(static_cast<long long>(ent[k]) * GPU + gi < sp.cap_groups[slot]);
    if constexpr (W == 16) {
      if (store) {
        uint4* dst = reinterpret_cast<uint4*>(sp.codes[3] + gg * 128) + 2 * l4;
        dst[0] = raw[k][0];
        dst[1] = raw[k][1];
      }
    } else {
      float x[16];
      const uint32_t v[8] = {raw[k][0].x, raw[k][0].y, raw[k][0].z, raw[k][0].w,
                             raw[k][1].x, raw[k][1].y, raw[k][1].z, raw[k][1].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        x[2 * e] = bf16_lo(v[e]);
        x[2 * e + 1] = bf16_hi(v[e]);
      }
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) a = fmaxf(a, fabsf(x[e]));
#pragma unroll
      for (int o = 2; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
      const __half sh = W == 2 ? __float2half_ru(a) : __float2half_ru(__fdiv_rn(a, static_cast<float>((1 << (W - 1)) - 1)));
      const float sc = __half2float(sh);
      uint32_t words[W / 2];
#pragma unroll
      for (int h = 0; h < W / 2; ++h) words[h] = 0u;
      if (sc > 0.f && !isinf(sc)) quantize_w<W, 16>(x, sc, quant_recip(sc, W), words);
      if (store) {
        if (l4 == 0) {
          sp.scales[slot][gg] = __half_as_ushort(sh);
          if (isinf(sc)) record_error(KVS_ERR_RANGE);
        }
        uint8_t* dst = sp.codes[slot] + gg * (8 * W) + l4 * (2 * W);
        if constexpr (W == 2)
          *reinterpret_cast<uint32_t*>(dst) = words[0];
        else if constexpr (W == 4)
          *reinterpret_cast<uint2*>(dst) = make_uint2(words[0], words[1]);
        else
          *reinterpret_cast<uint4*>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
      }
    }
  }
}

// grid (chunks, pools): pack the stored units of one chunk.  The plan groups
// the chunk's units by width, so every warp works at one width (a template
// parameter) on the units of one list: a warp takes 8 groups per step (4
// lanes, 32 bytes a lane, per 64-element group), kRowSteps steps' loads in
// flight.
template <int DH>
__global__ void __launch_bounds__(kRowThreads) pack_rows_kernel(const uint16_t* __restrict__ X,
                                                                const uint8_t* __restrict__ bits, const long long U,
                                                                const int n_chunks, const uint32_t* __restrict__ cnt,
                                                                const StreamPtrs sp) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  constexpr int GPU = DH / 64;
  constexpr int kWarps = kRowThreads / 32;
  constexpr int kStepUnits = 8 / GPU;            // units of one warp step
  constexpr int kItemUnits = kRowSteps * kStepUnits;  // units of one work item
  __shared__ int s_ent[kRowChunk];
  __shared__ uint8_t s_w[kRowChunk];
  __shared__ uint16_t s_list[kRowChunk];
  __shared__ long long s_base[4];
  __shared__ unsigned long long sbuf[kWarps + 1];
  const long long pool = blockIdx.y;
  unsigned long long per_slot;
  rows_chunk_plan(bits + pool * U, U, n_chunks, cnt, pool, GPU, sp, true, s_ent, s_w, s_base, sbuf, s_list, &per_slot);
  const uint16_t* Xc = X + (pool * U + static_cast<long long>(blockIdx.x) * kRowChunk) * DH;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, sub = lane >> 2, l4 = lane & 3;
  // per slot: its units, first list entry and first work item
  int n_sl[4], list0[4], item0[5];
  list0[0] = 0;
  item0[0] = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    n_sl[q] = static_cast<int>((per_slot >> (16 * q)) & 0xFFFFull);
    if (q < 3) list0[q + 1] = list0[q] + n_sl[q];
    item0[q + 1] = item0[q] + (n_sl[q] + kItemUnits - 1) / kItemUnits;
  }
  for (int it = warp; it < item0[4]; it += kWarps) {
    const int slot = (it >= item0[1]) + (it >= item0[2]) + (it >= item0[3]);
    int ns = 0, l0 = 0, i0 = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q == slot) ns = n_sl[q], l0 = list0[q], i0 = item0[q];
    uint4 raw[kRowSteps][2];
    int ent[kRowSteps];
#pragma unroll
    for (int k = 0; k < kRowSteps; ++k) {
      const int j = (it - i0) * kItemUnits + k * kStepUnits + sub / GPU;  // place in the slot's list
      const int ui = j < ns ? s_list[l0 + j] : -1;
      ent[k] = ui >= 0 ? s_ent[ui] : -1;
      raw[k][0] = raw[k][1] = make_uint4(0u, 0u, 0u, 0u);
      if (ent[k] >= 0) {
        const uint4* src = reinterpret_cast<const uint4*>(Xc + static_cast<long long>(ui) * DH + (sub % GPU) * 64 + l4 * 16);
        raw[k][0] = __ldg(src);
        raw[k][1] = __ldg(src + 1);
      }
    }
    switch (slot) {
      case 0: pack_rows_steps<2, GPU>(sp, pool, 0, l4, sub % GPU, raw, ent); break;
      case 1: pack_rows_steps<4, GPU>(sp, pool, 1, l4, sub % GPU, raw, ent); break;
      case 2: pack_rows_steps<8, GPU>(sp, pool, 2, l4, sub % GPU, raw, ent); break;
      default: pack_rows_steps<16, GPU>(sp, pool, 3, l4, sub % GPU, raw, ent); break;
    }
  }
}

// Decode this lane's 8 elements of a group.
__device__ __forceinline__ void dequant_lane8(const uint8_t* group_base, const int w, const int l8,
                                              const uint16_t* scale_ptr, float (&y)[8]) {
  if (w == 16) {
    const uint2* p = reinterpret_cast<const uint2*>(group_base) + 2 * l8;
    const uint2 a = p[0], b = p[1];
    bf16x8(make_uint4(a.x, a.y, b.x, b.y), y);
    return;
  }
  unsigned long long packed;
  if (w == 2)
    packed = reinterpret_cast<const uint16_t*>(group_base)[l8];
  else if (w == 4)
    packed = reinterpret_cast<const uint32_t*>(group_base)[l8];
  else
    packed = reinterpret_cast<const unsigned long long*>(group_base)[l8];
  const float s = __half2float(__ushort_as_half(*scale_ptr));
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] = code_to_float(static_cast<uint32_t>(packed >> (w * e)), w) * s;
}

// grid (chunks, pools): every row of one chunk, in unit order (width 0 -> zeros)
template <int DH>
__global__ void __launch_bounds__(kRowThreads) dequant_rows_kernel(const StreamPtrs sp, const uint8_t* __restrict__ bits,
                                                                   const long long U, const int n_chunks,
                                                                   const uint32_t* __restrict__ cnt,
                                                                   float* __restrict__ out) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  constexpr int GPU = DH / 64;
  constexpr int kWarps = kRowThreads / 32;
  __shared__ int s_ent[kRowChunk];
  __shared__ uint8_t s_w[kRowChunk];
  __shared__ long long s_base[4];
  __shared__ unsigned long long sbuf[kWarps + 1];
  const long long pool = blockIdx.y;
  const int n = rows_chunk_plan(bits + pool * U, U, n_chunks, cnt, pool, GPU, sp, false, s_ent, s_w, s_base, sbuf);
  float* oc = out + (pool * U + static_cast<long long>(blockIdx.x) * kRowChunk) * DH;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, sub = lane >> 3, l8 = lane & 7;
  const int ng = n * GPU;
  for (int gl = warp * 4 + sub; gl - sub < ng; gl += kWarps * 4) {
    if (gl >= ng) continue;
    const int ui = gl / GPU;
    const int w = s_w[ui], ent = s_ent[ui], s = width_slot(w);
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = 0.f;
    if (s >= 0 && ent >= 0 && KVS_IN_BOUNDS(static_cast<long long>(ent) * GPU + gl % GPU < sp.cap_groups[s])) {
      const long long gg = pool * sp.cap_groups[s] + static_cast<long long>(ent) * GPU + gl % GPU;
      dequant_lane8(sp.codes[s] + gg * (8 * w), w, l8, sp.scales[s] + gg, y);
    }
    float4* o = reinterpret_cast<float4*>(oc + static_cast<long long>(gl) * 64 + l8 * 8);
    o[0] = make_float4(y[0], y[1], y[2], y[3]);
    o[1] = make_float4(y[4], y[5], y[6], y[7]);
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
        if (mask & (1u << e)) {
          if (KVS_IN_BOUNDS(pk >= 0 && pk < N)) kg[pk] = t0 + e;
          ++pk;
        } else {
          if (KVS_IN_BOUNDS(pd >= 0 && pd < N)) kg[pd] = t0 + e;
          --pd;
        }
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

// Channel kernels: a CTA takes the kept tokens of TG = 512 / DH consecutive
// 64-token groups of one head; warp w takes group w / (DH / 64) and 64
// channels, two per lane (one 4-byte word of a row), so every row load and
// every row store of a warp is one contiguous 128-byte (256-byte) segment and
// needs no shared-memory transpose.  A lane holds its two channels' 64 values
// of the group in registers (64 loads in flight), takes each channel's
// absolute maximum with packed bf16 maxima, and writes the group's codes
// eight elements (w bytes) at a time.
constexpr int kChanThreads = 256;

template <int DH>
__host__ __device__ constexpr int chan_groups_per_cta() { return 8 / (DH / 64); }

// grid (ceil(ceil(N/64) / TG), pools * Hkv).  The codes of a warp's 64
// channel blocks are staged in shared memory and then written block by block,
// eight lanes per block (16 bytes a lane), so each store instruction writes
// four contiguous blocks instead of 32 scattered pieces.  In the stage, the
// 16-byte chunk j of channel slot cl's 128-byte block sits at chunk
// j ^ ((cl / 2) mod 8): the lanes' stores of one octet (channel slots 2 apart)
// then spread over eight bank groups instead of one.
template <int DH>
__host__ __device__ constexpr size_t chan_pack_smem() { return static_cast<size_t>(kChanThreads / 32) * 64 * 128; }

// byte b of channel slot cl's block in a warp's stage
__device__ __forceinline__ int stage_off(const int cl, const int b) {
  return cl * 128 + ((((b >> 4) ^ (cl >> 1)) & 7) << 4) + (b & 15);
}

template <int DH>
__global__ void __launch_bounds__(kChanThreads) pack_channels_kernel(const uint16_t* __restrict__ X, const int N,
                                                                     const uint8_t* __restrict__ bits,
                                                                     const long long* __restrict__ chan_base,
                                                                     const int* __restrict__ kept,
                                                                     const int* __restrict__ n_kept, const StreamPtrs sp,
                                                                     const int Hkv) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  constexpr int CB = DH / 64;                       // warps per group: 64 channels each
  constexpr int TG = chan_groups_per_cta<DH>();
  extern __shared__ __align__(16) uint8_t cstage[];  // per warp: 64 channel blocks of up to 128 bytes
  __shared__ int s_tok[64 * TG];
  __shared__ uint8_t* s_dst[kChanThreads / 32][64];
  __shared__ int s_wd[kChanThreads / 32][64];
  const int jb = blockIdx.x, g = blockIdx.y;
  const long long pool = g / Hkv;
  const int n = n_kept[g];
  const int k0 = jb * 64 * TG;
  if (k0 >= n) return;
  const int rows = min(64 * TG, n - k0);
  for (int i = threadIdx.x; i < 64 * TG; i += kChanThreads)
    s_tok[i] = i < rows ? kept[static_cast<long long>(g) * N + k0 + i] : 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int jg = warp / CB, r0 = jg * 64;
  if (r0 >= rows) return;
  const int nr = min(64, rows - r0);
  const int c0 = (warp % CB) * 64 + 2 * lane;
  const uint16_t* Xg = X + static_cast<long long>(g) * N * DH + c0;
  uint32_t v[64];  // channels c0 (low half) and c0 + 1 (high half) of the group's tokens; zeros past the kept ones
#pragma unroll
  for (int e = 0; e < 64; ++e)
    v[e] = (e < nr && KVS_IN_BOUNDS(s_tok[r0 + e] >= 0 && s_tok[r0 + e] < N))
               ? __ldg(reinterpret_cast<const uint32_t*>(Xg + static_cast<long long>(s_tok[r0 + e]) * DH))
               : 0u;
  uint32_t amax = 0u;
#pragma unroll
  for (int e = 0; e < 64; ++e) amax = bf16x2_max(amax, v[e] & 0x7FFF7FFFu);
  uint8_t* stage = cstage + warp * (64 * 128);
  // the two channels' widths, destinations and scales
  int wd[2];
  float sc[2], rc[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int cl = 2 * lane + h;  // the channel's slot in the warp's stage
    const long long u = static_cast<long long>(g) * DH + c0 + h;
    const int w = bits[u], s = width_slot(w);
    const long long b = chan_base[u];
    wd[h] = (s >= 0 && b >= 0 && KVS_IN_BOUNDS(b + jb * TG + jg < sp.cap_groups[s])) ? w : 0;
    s_wd[warp][cl] = wd[h];
    sc[h] = 0.f;
    rc[h] = 0.f;
    if (!wd[h]) continue;
    const long long gg = pool * sp.cap_groups[s] + b + jb * TG + jg;
    s_dst[warp][cl] = sp.codes[s] + gg * (8 * w);
    if (w == 16) continue;
    const float a = __uint_as_float(((amax >> (16 * h)) & 0xFFFFu) << 16);
    const float qmax = static_cast<float>((1 << (w - 1)) - 1);
    const __half shalf = __float2half_ru(__fdiv_rn(a, qmax));
    sc[h] = __half2float(shalf);
    sp.scales[s][gg] = __half_as_ushort(shalf);
    if (isinf(sc[h])) record_error(KVS_ERR_RANGE);
    if (sc[h] > 0.f && !isinf(sc[h])) rc[h] = quant_recip(sc[h], w);
  }
  // each channel of the pair in turn: widths 2 / 4 / 8 share one instruction
  // stream (constants in registers), width 16 copies the raw values
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int cl = 2 * lane + h;
    const int w = wd[h];
    if (w == 16) {
#pragma unroll
      for (int o = 0; o < 8; ++o) {
        uint32_t r4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)  // the channel's halves of two tokens
          r4[k] = h ? __byte_perm(v[8 * o + 2 * k], v[8 * o + 2 * k + 1], 0x7632)
                    : __byte_perm(v[8 * o + 2 * k], v[8 * o + 2 * k + 1], 0x5410);
        *reinterpret_cast<uint4*>(stage + stage_off(cl, 16 * o)) = make_uint4(r4[0], r4[1], r4[2], r4[3]);
      }
    } else if (w != 0) {
      const DynCode c = dyn_code(w);
      const float scl = sc[h], rcp = rc[h];
      // the octets' codes (8w bits each) gather in a 64-bit word, stored as
      // it fills: no branch on the width, one 8-byte store per 64 code bits
      unsigned long long word = 0ull;
      int fill = 0, k = 0;
#pragma unroll
      for (int o = 0; o < 8; ++o) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = h ? bf16_hi(v[8 * o + e]) : bf16_lo(v[8 * o + e]);
        const unsigned long long packed = rcp != 0.f ? quantize_octet_dyn(x, scl, rcp, c) : 0ull;
        word |= packed << fill;
        fill += 8 * w;
        if (fill == 64) {
          *reinterpret_cast<unsigned long long*>(stage + stage_off(cl, 8 * k)) = word;
          ++k;
          word = 0ull;
          fill = 0;
        }
      }
    }
  }
  __syncwarp();
  // the staged blocks, four channels per step, eight lanes per block
  const int sub = lane >> 3, l8 = lane & 7;
#pragma unroll 4
  for (int c4 = 0; c4 < 64; c4 += 4) {
    const int cl = c4 + sub;
    const int w = s_wd[warp][cl];
    if (2 * l8 < w)  // a block is 8w bytes: w/2 chunks of 16
      *reinterpret_cast<uint4*>(s_dst[warp][cl] + 16 * l8) = *reinterpret_cast<const uint4*>(stage + stage_off(cl, 16 * l8));
  }
}

// 8 decoded values of one channel's octet o of a group
__device__ __forceinline__ void dequant_octet(const uint8_t* group_base, const int w, const int o, const float s,
                                              float (&y)[8]) {
  if (w == 16) {
    const uint2* p = reinterpret_cast<const uint2*>(group_base) + 2 * o;
    const uint2 a = p[0], b = p[1];
    bf16x8(make_uint4(a.x, a.y, b.x, b.y), y);
    return;
  }
  unsigned long long packed;
  if (w == 2)
    packed = reinterpret_cast<const uint16_t*>(group_base)[o];
  else if (w == 4)
    packed = reinterpret_cast<const uint32_t*>(group_base)[o];
  else
    packed = reinterpret_cast<const unsigned long long*>(group_base)[o];
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] = code_to_float(static_cast<uint32_t>(packed >> (w * e)), w) * s;
}

// grid (ceil(N / (64 TG)) + 1, pools * Hkv).  CTA jb below the head's count of
// kept blocks decodes kept-token groups [TG jb, ..) of every channel and
// writes those tokens' rows (a lane's two channels: one 8-byte store per
// token); the CTAs after those zero the head's dropped tokens, 64 TG per CTA.
template <int DH>
__global__ void __launch_bounds__(kChanThreads) dequant_channels_kernel(const StreamPtrs sp, const int N,
                                                                        const uint8_t* __restrict__ bits,
                                                                        const long long* __restrict__ chan_base,
                                                                        const int* __restrict__ kept,
                                                                        const int* __restrict__ n_kept,
                                                                        float* __restrict__ out, const int Hkv) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  constexpr int CB = DH / 64;
  constexpr int TG = chan_groups_per_cta<DH>();
  constexpr int TOK = 64 * TG;
  __shared__ int s_tok[TOK];
  const int jb = blockIdx.x, g = blockIdx.y;
  const long long pool = g / Hkv;
  const int n = n_kept[g];
  const int nkb = (n + TOK - 1) / TOK;
  const int* kg = kept + static_cast<long long>(g) * N;
  float* og = out + static_cast<long long>(g) * N * DH;
  if (jb >= nkb) {  // zero dropped tokens kept[g][n + TOK (jb - nkb) ..]
    const int d0 = n + (jb - nkb) * TOK;
    if (d0 >= N) return;
    const int cnt = min(TOK, N - d0);
    for (int e = threadIdx.x; e < cnt * (DH / 4); e += kChanThreads) {
      const int i = e / (DH / 4), c4 = (e % (DH / 4)) * 4;
      const int tok = kg[d0 + i];
      if (KVS_IN_BOUNDS(tok >= 0 && tok < N))
        *reinterpret_cast<float4*>(og + static_cast<long long>(tok) * DH + c4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  const int k0 = jb * TOK;
  const int rows = min(TOK, n - k0);
  for (int i = threadIdx.x; i < TOK; i += kChanThreads) s_tok[i] = i < rows ? kg[k0 + i] : 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int jg = warp / CB, r0 = jg * 64;
  if (r0 >= rows) return;
  const int nr = min(64, rows - r0);
  const int c0 = (warp % CB) * 64 + 2 * lane;
  const uint8_t* blk[2];
  int wd[2];
  float sc[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const long long u = static_cast<long long>(g) * DH + c0 + h;
    const int w = bits[u], s = width_slot(w);
    const long long b = chan_base[u];
    wd[h] = (s >= 0 && b >= 0 && KVS_IN_BOUNDS(b + jb * TG + jg < sp.cap_groups[s])) ? w : 0;
    blk[h] = nullptr;
    sc[h] = 0.f;
    if (wd[h]) {
      const long long gg = pool * sp.cap_groups[s] + b + jb * TG + jg;
      blk[h] = sp.codes[s] + gg * (8 * w);
      sc[h] = w == 16 ? 1.f : __half2float(__ushort_as_half(sp.scales[s][gg]));
    }
  }
  float* orow = og + c0;
#pragma unroll 2
  for (int o = 0; o < 8; ++o) {
    float y0[8], y1[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y0[e] = y1[e] = 0.f;
    if (wd[0]) dequant_octet(blk[0], wd[0], o, sc[0], y0);
    if (wd[1]) dequant_octet(blk[1], wd[1], o, sc[1], y1);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = 8 * o + e;
      if (i < nr && KVS_IN_BOUNDS(s_tok[r0 + i] >= 0 && s_tok[r0 + i] < N))
        *reinterpret_cast<float2*>(orow + static_cast<long long>(s_tok[r0 + i]) * DH) = make_float2(y0[e], y1[e]);
    }
  }
}

}  // namespace kvs
