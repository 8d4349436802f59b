// TriZone decode attention: one decode step over a compressed pool, with the
// dequantisation fused into both products   [RDKV §2.3, TriZone].
//
//   zone A: the K channels (widths 2/4/8) and V rows (widths 2/4/8) of the
//           packed old cache;
//   zone B: the width-16 streams, read as raw bf16;
//   zone C: k_new / v_new, bf16 rows of the tokens generated since compression.
//
// Evicted tokens (V width 0) take no part in the softmax; K channels of width 0
// add nothing to the logits.  Query head hd reads KV head hd / G.
//
// Kernels:
//   trizone_index_kernel   once per compressed pool, per KV head: the number of
//                          kept tokens, the K entry range of each width, the
//                          width slot of every kept token (in ascending order)
//                          and, per 64-token group, the first V entry of each
//                          width.
//   trizone_decode_kernel  CTAs x < n_split: the packed zones.  Each warp takes
//                          64-token groups (the K group of 64 kept tokens) and
//                          keeps a running max and sum over them (flash
//                          decoding).  Both products run on the tensor cores
//                          (mma.sync m16n8k16, bf16 in, fp32 out): the codes go
//                          from registers straight into the B operand, so no
//                          dequantised copy exists anywhere.
//                          CTAs x >= n_split: zone C, bf16 rows, fp32 FMA.
//   trizone_combine_kernel per query head: merges the CTA partials in order.
//
// The K product.  A = q' (rows 0-3: bf16 high part of the 4 heads, rows 4-7:
// the bf16 low part, q' - hi, rows 8-15 zero), q'_c = q_c * s_{c,j} * log2(e)
// / sqrt(d) for channel c and group j; B = the codes of 16 channels of one
// width (the channel list is sorted by width and padded to blocks of 16) for
// 8 tokens.  Column n of tile t is token 8n + t of the group, so a lane's B
// values for all 8 tiles sit in one w-byte word of the channel's group block.
// The split q' = hi + lo keeps 16 significant bits of the product operand.
//
// The V product.  Rows as above with p'_t = p_t * s_{t,gr} (gr: the 64-channel
// group of the row), B = the codes of 16 rows of one width (the group's rows
// taken width by width, in the V stream's order, padded to 16) for 8 channels;
// column n of n-tile jn is channel 8n + jn of the channel group.
//
// Codes become bf16 exactly: for w <= 4 the bit pattern 0x4300 | (x ^ 2^(w-1))
// is the bf16 value 128 + x + 2^(w-1), and one bf16x2 FMA subtracts the bias;
// for w = 8 the same construction in fp32 (0x4B000000 | (x ^ 128)) gives x as
// a float whose high half is its bf16 pattern.  Width-16 values are bf16
// already.
#pragma once

#include "common.cuh"
#include "pack.cuh"

namespace kvs {

constexpr int kTzThreads = 256;   // 8 warps
constexpr int kTzD = 128;         // head dimension of the decode kernels
constexpr int kTzHdr = 16;        // int64 header words per KV head in the index
constexpr int kTzSlots = 192;     // K channel slots: 128 channels, each width padded to a multiple of 16
constexpr int kTzChunkC = 128;    // zone C tokens per step of a CTA

// header words of one KV head
enum { TZ_NKEPT = 0, TZ_KELO = 1, TZ_KN = 5, TZ_KGLO = 9, TZ_NG = 13 };

// byte offsets of the index parts
struct TzLayout {
  long long vstart, vslot, total;
};
__host__ __device__ inline long long tz_round256(long long x) { return (x + 255) / 256 * 256; }
__host__ __device__ inline TzLayout tz_layout(long long Hkv, long long N) {
  const long long ng = (N + 63) / 64;
  TzLayout L;
  L.vstart = tz_round256(Hkv * kTzHdr * 8);
  L.vslot = L.vstart + tz_round256(Hkv * (ng + 1) * 4 * 4);
  L.total = L.vslot + tz_round256(Hkv * N);
  return L;
}

__device__ __forceinline__ long long tz_count(const StreamPtrs& s, int i) {
  const long long c = s.counts[i];
  return c < s.cap_units[i] ? c : s.cap_units[i];
}

// first entry e in [0, n) with ids[e] >= key (ids ascending)
__device__ __forceinline__ long long tz_lower_bound(const int32_t* ids, long long n, long long key) {
  long long lo = 0, hi = n;
  while (lo < hi) {
    const long long mid = (lo + hi) >> 1;
    if (static_cast<long long>(ids[mid]) < key) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// index: one CTA of 1024 threads per KV head
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) trizone_index_kernel(StreamPtrs ks, StreamPtrs vs, const uint8_t* bits_v,
                                                             int N, int d, long long* hdr, int* vstart,
                                                             uint8_t* vslot) {
  pdl_wait();
  const int g = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long ngmax = (N + 63) / 64;
  int* VS = vstart + static_cast<long long>(g) * (ngmax + 1) * 4;
  __shared__ long long s_vlo[4], s_base[4], s_klo[4], s_kn[4], s_kglo[4];
  __shared__ unsigned long long s_wsum[32];
  if (tid < 4) {
    s_vlo[tid] = tz_lower_bound(vs.ids[tid], tz_count(vs, tid), static_cast<long long>(g) * N);
    s_base[tid] = 0;
  }
  __syncthreads();
  const uint8_t* b = bits_v + static_cast<long long>(g) * N;
  for (int t0 = 0; t0 < N; t0 += 1024) {
    const int t = t0 + tid;
    const uint32_t w = t < N ? b[t] : 0u;
    const int slot = width_slot(w);
    if (w != 0 && slot < 0) record_error(KVS_ERR_RANGE);
    // four per-width counts packed in 16-bit fields (a chunk holds <= 1024)
    const unsigned long long mine = slot >= 0 ? (1ull << (16 * slot)) : 0ull;
    unsigned long long x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      unsigned long long v = s_wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      s_wsum[lane] = v;
    }
    __syncthreads();
    if (slot >= 0) {
      const unsigned long long excl = (warp ? s_wsum[warp - 1] : 0ull) + x - mine;
      long long before[4], rank = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        before[k] = s_base[k] + static_cast<long long>((excl >> (16 * k)) & 0xffffull);
        rank += before[k];
      }
      long long e = s_vlo[0] + before[0];
#pragma unroll
      for (int k = 1; k < 4; ++k)
        if (slot == k) e = s_vlo[k] + before[k];
      const long long want = static_cast<long long>(g) * N + t;
      // a V unit (one token row of d = 128) holds two groups, so entry e starts at group 2e
      if (!(e < tz_count(vs, slot) && static_cast<long long>(vs.ids[slot][e]) == want &&
            vs.goff[slot][e] == 2 * e && 2 * e + 2 <= vs.cap_groups[slot]))
        record_error(KVS_ERR_RANGE);   // the V streams do not match bits_v
      vslot[static_cast<long long>(g) * N + rank] = static_cast<uint8_t>(slot);
      if ((rank & 63) == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) VS[(rank >> 6) * 4 + k] = static_cast<int>(s_vlo[k] + before[k]);
      }
    }
    __syncthreads();
    if (tid < 4) s_base[tid] += static_cast<long long>((s_wsum[31] >> (16 * tid)) & 0xffffull);
    __syncthreads();
  }
  const long long nkept = s_base[0] + s_base[1] + s_base[2] + s_base[3];
  const long long nG = (nkept + 63) / 64;
  if (tid < 4) {
    VS[nG * 4 + tid] = static_cast<int>(s_vlo[tid] + s_base[tid]);
    const long long n = tz_count(ks, tid);
    const long long lo = tz_lower_bound(ks.ids[tid], n, static_cast<long long>(g) * d);
    const long long hi = tz_lower_bound(ks.ids[tid], n, static_cast<long long>(g) * d + d);
    s_klo[tid] = lo;
    s_kn[tid] = hi - lo;
    s_kglo[tid] = hi > lo ? ks.goff[tid][lo] : 0;
    long long* H = hdr + static_cast<long long>(g) * kTzHdr;
    H[TZ_KELO + tid] = lo;
    H[TZ_KN + tid] = hi - lo;
    H[TZ_KGLO + tid] = s_kglo[tid];
    if (tid == 0) {
      H[TZ_NKEPT] = nkept;
      H[TZ_NG] = nG;
    }
  }
  __syncthreads();
  // the decode kernel addresses channel k of a width at first group + k * nG
  for (int s = 0; s < 4; ++s) {
    for (long long k = tid; k < s_kn[s]; k += 1024) {
      const long long e = s_klo[s] + k;
      if (ks.goff[s][e] != s_kglo[s] + k * nG || s_kglo[s] + (k + 1) * nG > ks.cap_groups[s])
        record_error(KVS_ERR_RANGE);
    }
  }
}

// ---------------------------------------------------------------------------
// operands
// ---------------------------------------------------------------------------
// one m16n8k16 bf16 MMA on rows 0-7 (rows 8-15 of A are zero; their outputs are dropped)
__device__ __forceinline__ void tz_mma(float& d0, float& d1, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  [[maybe_unused]] float x0, x1;  // rows 8-15 of the product: not needed
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%5}, {%7,%8}, {%0,%1,%9,%9};"
      : "+f"(d0), "+f"(d1), "=f"(x0), "=f"(x1)
      : "r"(a0), "r"(0u), "r"(a2), "r"(b0), "r"(b1), "f"(0.f));
}

// bf16x2 of (lo, hi), round to nearest
__device__ __forceinline__ uint32_t tz_bf2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// the high and low bf16 parts of two values: x = hi + lo to 16 significant bits
__device__ __forceinline__ void tz_split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = tz_bf2(x0, x1);
  lo = tz_bf2(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
}

__device__ __forceinline__ uint32_t tz_bsub(uint32_t x, uint32_t negbias) {   // x - bias on both bf16 halves
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(0x3F803F80u), "r"(negbias));
  return r;
}

__device__ __forceinline__ uint32_t tz_word(const uint4& r, int i) {
  return i == 0 ? r.x : (i == 1 ? r.y : (i == 2 ? r.z : r.w));
}

// The 8 bf16x2 B values of a word pair: value i of word a (low half) and of
// word b (high half).  ra and rb are the aligned 16 bytes holding the lane's
// w-byte words, which start at byte o of them.
template <int W>
__device__ __forceinline__ void tz_pairs8(const uint4& ra, const uint4& rb, int o, uint32_t (&v)[8]) {
  if constexpr (W == 2) {
    const uint32_t a = tz_word(ra, o >> 2) >> ((o & 3) * 8), b = tz_word(rb, o >> 2) >> ((o & 3) * 8);
    const uint32_t ab = __byte_perm(a, b, 0x5410);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = tz_bsub(((ab >> (2 * i)) & 0x00030003u) ^ 0x43024302u, 0xC302C302u);
  } else if constexpr (W == 4) {
    const uint32_t a = tz_word(ra, o >> 2), b = tz_word(rb, o >> 2);
    const uint32_t lo = __byte_perm(a, b, 0x5410), hi = __byte_perm(a, b, 0x7632);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] = tz_bsub(((lo >> (4 * i)) & 0x000F000Fu) ^ 0x43084308u, 0xC308C308u);
      v[4 + i] = tz_bsub(((hi >> (4 * i)) & 0x000F000Fu) ^ 0x43084308u, 0xC308C308u);
    }
  } else if constexpr (W == 8) {
    const int i0 = o >> 2;
    const uint32_t a0 = tz_word(ra, i0) ^ 0x80808080u, a1 = tz_word(ra, i0 + 1) ^ 0x80808080u;
    const uint32_t b0 = tz_word(rb, i0) ^ 0x80808080u, b1 = tz_word(rb, i0 + 1) ^ 0x80808080u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t sel = 0x7650u | static_cast<uint32_t>(i & 3);
      const float fa = __uint_as_float(__byte_perm(i < 4 ? a0 : a1, 0x4B000000u, sel)) - 8388736.0f;
      const float fb = __uint_as_float(__byte_perm(i < 4 ? b0 : b1, 0x4B000000u, sel)) - 8388736.0f;
      v[i] = __byte_perm(__float_as_uint(fa), __float_as_uint(fb), 0x7632);
    }
  } else {
    const uint32_t av[4] = {ra.x, ra.y, ra.z, ra.w}, bv[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __byte_perm(av[i >> 1], bv[i >> 1], (i & 1) ? 0x7632 : 0x5410);
  }
}

__device__ __forceinline__ void tz_prefetch(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint4 tz_ld16(const uint8_t* p) {   // the aligned 16 bytes holding p
  return __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<uintptr_t>(p) & ~static_cast<uintptr_t>(15)));
}

// ---------------------------------------------------------------------------
// shared memory
// ---------------------------------------------------------------------------
struct TzWarpBuf {
  uint32_t qhl[2][4][kTzSlots / 2];        // A of the K product: bf16 pairs [part][head][slot pair]
  float pw[64][4];                         // the group's softmax numerators [local rank][head]
  uint8_t lr[4][64];                       // local ranks of the group's rows, width by width
};
struct TzPackedShared {
  float qs[kTzD][4];                       // scaled query [channel][head]
  int ch_id[kTzSlots];                     // channel of a slot; -1: padding
  int blk_w[kTzSlots / 16];                // width of each block of 16 slots
  const uint8_t* ch_code[kTzSlots];        // code block of the slot's channel, group 0
  const uint16_t* ch_scale[kTzSlots];      // its scales (widths 2/4/8)
  const uint8_t* v_code[4];
  const uint16_t* v_scale[4];
  long long v_cap_units[4], v_cap_groups[4];
  union {
    TzWarpBuf w[8];
    struct {
      float m[8][4], l[8][4];
      float o[8][4][kTzD];
    } merge;
  } u;
};
struct TzZoneCShared {
  float qs[kTzD][4];
  float red[8][4][kTzChunkC];
  float p[kTzChunkC][4];
  float hm[8][4], hs[8][4];
};
union TzShared {
  TzPackedShared a;
  TzZoneCShared c;
};

// ---------------------------------------------------------------------------
// the packed zones
// ---------------------------------------------------------------------------
template <int HG>
__device__ __forceinline__ void tz_packed(TzPackedShared& sh, const uint16_t* __restrict__ q, const StreamPtrs& ks,
                                          const StreamPtrs& vs, const long long* __restrict__ H,
                                          const int* __restrict__ VS, const uint8_t* __restrict__ vslot_g,
                                          long long nkept, int hd0, int part_idx, int nparts, float qscale,
                                          float* __restrict__ pm, float* __restrict__ pl, float* __restrict__ po,
                                          int slots) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y;
  const long long nG = (nkept + 63) / 64;
  const long long j0 = part_idx * nG / nparts, j1 = (part_idx + 1) * nG / nparts;

  for (int i = tid; i < 4 * kTzD; i += kTzThreads) {
    const int h = i / kTzD, c = i % kTzD;
    sh.qs[c][h] = h < HG ? bf16_lo(q[static_cast<long long>(hd0 + h) * kTzD + c]) * qscale : 0.f;
  }
  // channel slots: width class by width class, each padded to a multiple of 16
  long long n_s[4];
  int nblk = 0, nch = 0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    long long n = H[TZ_KN + s];
    n = n < 0 ? 0 : (n > kTzD - nch ? kTzD - nch : n);
    n_s[s] = n;
    nch += static_cast<int>(n);
    nblk += static_cast<int>((n + 15) / 16);
  }
  if (tid < kTzSlots) {
    int p = tid, s = 0, k = -1;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int padded = static_cast<int>((n_s[c] + 15) / 16 * 16);
      if (k < 0 && s == c) {
        if (p < padded) k = p; else { p -= padded; s = c + 1; }
      }
    }
    int id = -1;
    const uint8_t* code = nullptr;
    const uint16_t* scale = nullptr;
    if (k >= 0 && s < 4 && k < n_s[s]) {
      const long long e = H[TZ_KELO + s] + k;
      const long long grp = H[TZ_KGLO + s] + static_cast<long long>(k) * nG;
      const int c = e >= 0 && e < ks.cap_units[s] ? ks.ids[s][e] - g * kTzD : -1;
      if (c < 0 || c >= kTzD || grp < 0 || grp + nG > ks.cap_groups[s]) {
        record_error(KVS_ERR_RANGE);          // index and streams disagree: the channel is skipped
      } else {
        id = c;
        code = ks.codes[s] + grp * (16 << s);
        scale = s < 3 ? ks.scales[s] + grp : nullptr;
      }
    }
    sh.ch_id[tid] = id;
    sh.ch_code[tid] = code;
    sh.ch_scale[tid] = scale;
    if ((tid & 15) == 0) sh.blk_w[tid >> 4] = (s < 4 && k >= 0) ? (2 << s) : 0;
  }
  if (tid < 4) {
    sh.v_code[tid] = vs.codes[tid];
    sh.v_scale[tid] = vs.scales[tid];
    sh.v_cap_units[tid] = vs.cap_units[tid];
    sh.v_cap_groups[tid] = vs.cap_groups[tid];
  }
  __syncthreads();

  // Bring a group's K blocks, its width bytes and its V rows into L2 ahead of
  // use: every load of the group then waits on L2 rather than on DRAM.
  auto prefetch_group = [&](long long jp) {
    for (int p = lane; p < nblk * 16; p += 32) {
      if (sh.ch_id[p] < 0) continue;
      const int w = sh.blk_w[p >> 4];
      tz_prefetch(sh.ch_code[p] + jp * (8 * w));
      if (sh.ch_scale[p]) tz_prefetch(sh.ch_scale[p] + jp);
    }
    if (lane == 0) tz_prefetch(vslot_g + 64 * jp);
    const int e_a = lane < 4 ? VS[jp * 4 + lane] : 0;
    const int e_b = lane < 4 ? VS[jp * 4 + 4 + lane] : 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const long long ea = __shfl_sync(0xffffffffu, e_a, s), eb = __shfl_sync(0xffffffffu, e_b, s);
      if (ea < 0 || eb > sh.v_cap_units[s] || eb <= ea) continue;
      const long long b0 = 2 * ea * (16 << s), b1 = 2 * eb * (16 << s);   // V row bytes of the group
      for (long long off = (b0 & ~127ll) + 128ll * lane; off < b1; off += 128ll * 32) tz_prefetch(sh.v_code[s] + off);
      if (s < 3 && lane == 31) tz_prefetch(sh.v_scale[s] + 2 * ea);
    }
  };

  TzWarpBuf& wb = sh.u.w[warp];
  const int gq = lane >> 2, t4 = lane & 3;          // fragment row / column group
  const int hrow = gq & 3, part = gq >> 2;          // the lane's A row: head, high (0) or low (1) part
  float m_run = -INFINITY, l_run = 0.f;             // of head hrow
  float oacc[2][8][2];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) oacc[a][b][0] = oacc[a][b][1] = 0.f;

  if (j0 + warp < j1) prefetch_group(j0 + warp);
  for (long long j = j0 + warp; j < j1; j += 8) {
    const int cnt = static_cast<int>(nkept - 64 * j < 64 ? nkept - 64 * j : 64);
    // the group's small loads first; the next group's data towards L2
    const int s0 = 2 * lane < cnt ? vslot_g[64 * j + 2 * lane] : 4;
    const int s1 = 2 * lane + 1 < cnt ? vslot_g[64 * j + 2 * lane + 1] : 4;
    const int ebase_l = lane < 4 ? VS[j * 4 + lane] : 0;
    if (j + 8 < j1) prefetch_group(j + 8);

    // ---- A of the K product: q' = q * s_{c,j}, split into bf16 high and low parts ----
    for (int pp = lane; pp < nblk * 8; pp += 32) {
      float x[2][4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int p = 2 * pp + e;
        const int c = sh.ch_id[p];
        float sc = 0.f;
        if (c >= 0) sc = sh.ch_scale[p] ? __half2float(__ushort_as_half(__ldg(sh.ch_scale[p] + j))) : 1.f;
#pragma unroll
        for (int h = 0; h < 4; ++h) x[e][h] = c >= 0 ? sh.qs[c][h] * sc : 0.f;
      }
#pragma unroll
      for (int h = 0; h < 4; ++h) tz_split2(x[0][h], x[1][h], wb.qhl[0][h][pp], wb.qhl[1][h][pp]);
    }
    __syncwarp();

    // ---- logits: the K product, block by block ----
    float dk[8][2];
#pragma unroll
    for (int t = 0; t < 8; ++t) dk[t][0] = dk[t][1] = 0.f;
    for (int b = 0; b < nblk; ++b) {
      const int w = sh.blk_w[b];
      const int p0 = 16 * b + 2 * t4;
      uint4 r[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int p = p0 + (e & 1) + 8 * (e >> 1);
        r[e] = sh.ch_id[p] >= 0 ? tz_ld16(sh.ch_code[p] + j * (8 * w) + gq * w) : make_uint4(0u, 0u, 0u, 0u);
      }
      const uint32_t a0 = wb.qhl[part][hrow][p0 >> 1], a2 = wb.qhl[part][hrow][(p0 + 8) >> 1];
      const int o = (gq * w) & 15;
      uint32_t v0[8], v1[8];
      if (w == 2) {
        tz_pairs8<2>(r[0], r[1], o, v0);
        tz_pairs8<2>(r[2], r[3], o, v1);
      } else if (w == 4) {
        tz_pairs8<4>(r[0], r[1], o, v0);
        tz_pairs8<4>(r[2], r[3], o, v1);
      } else if (w == 8) {
        tz_pairs8<8>(r[0], r[1], o, v0);
        tz_pairs8<8>(r[2], r[3], o, v1);
      } else {
        tz_pairs8<16>(r[0], r[1], o, v0);
        tz_pairs8<16>(r[2], r[3], o, v1);
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) tz_mma(dk[t][0], dk[t][1], a0, a2, v0[t], v1[t]);
    }
    // rows hrow (high part) and hrow + 4 (low part) sit 16 lanes apart: add them.
    // Lane (gq, t4) then holds head hrow's logits of tokens 16*t4 + t (dk[t][0])
    // and 16*t4 + 8 + t (dk[t][1]).
    float mg = -INFINITY;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        float v = dk[t][u] + __shfl_xor_sync(0xffffffffu, dk[t][u], 16);
        if (16 * t4 + 8 * u + t >= cnt) v = -INFINITY;
        dk[t][u] = v;
        mg = fmaxf(mg, v);
      }
    }
    mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, 1));
    mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, 2));
    const float mn = fmaxf(m_run, mg);                // finite: the group holds a token
    const float alpha = ex2_approx(m_run - mn);       // 0 on the first group
    m_run = mn;
    float ls = 0.f;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float p = ex2_approx(dk[t][u] - mn);    // 0 for the masked tokens
        ls += p;
        if (lane < 16) wb.pw[16 * t4 + 8 * u + t][hrow] = p;
      }
    }
    ls += __shfl_xor_sync(0xffffffffu, ls, 1);
    ls += __shfl_xor_sync(0xffffffffu, ls, 2);
    l_run = l_run * alpha + ls;
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        oacc[a][b][0] *= alpha;
        oacc[a][b][1] *= alpha;
      }

    // ---- the group's rows, width by width (ranks ascending within a width) ----
    int n_w[4];
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const unsigned m0 = __ballot_sync(0xffffffffu, s0 == s), m1 = __ballot_sync(0xffffffffu, s1 == s);
      const int before = __popc(m0 & lt) + __popc(m1 & lt);
      if (s0 == s) wb.lr[s][before] = static_cast<uint8_t>(2 * lane);
      if (s1 == s) wb.lr[s][before + (s0 == s ? 1 : 0)] = static_cast<uint8_t>(2 * lane + 1);
      n_w[s] = __popc(m0) + __popc(m1);
    }
    __syncwarp();

    // ---- the V product ----
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int w = 2 << s;
      const long long ebase = __shfl_sync(0xffffffffu, ebase_l, s);
      for (int bb = 0; bb < n_w[s]; bb += 16) {
        // the lane's 4 rows of the block: 2*t4, 2*t4+1, 2*t4+8, 2*t4+9
        uint4 r[2][4];
        float pv[2][4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int idx = bb + 2 * t4 + (e & 1) + 8 * (e >> 1);
          r[0][e] = r[1][e] = make_uint4(0u, 0u, 0u, 0u);
          pv[0][e] = pv[1][e] = 0.f;
          if (idx < n_w[s]) {
            const long long ent = ebase + idx;
            if (ent >= 0 && ent < sh.v_cap_units[s] && 2 * ent + 2 <= sh.v_cap_groups[s]) {
              const float p = wb.pw[wb.lr[s][idx]][hrow];
              const uint8_t* row = sh.v_code[s] + 2 * ent * (8 * w) + gq * w;
              r[0][e] = tz_ld16(row);
              r[1][e] = tz_ld16(row + 8 * w);
              if (s < 3) {
                const uint32_t sc2 = __ldg(reinterpret_cast<const uint32_t*>(sh.v_scale[s] + 2 * ent));
                pv[0][e] = p * __half2float(__ushort_as_half(static_cast<unsigned short>(sc2 & 0xffffu)));
                pv[1][e] = p * __half2float(__ushort_as_half(static_cast<unsigned short>(sc2 >> 16)));
              } else {
                pv[0][e] = pv[1][e] = p;
              }
            } else {
              record_error(KVS_ERR_RANGE);    // index and streams disagree: the row is skipped
            }
          }
        }
        const int o = (gq * w) & 15;
#pragma unroll
        for (int gr = 0; gr < 2; ++gr) {
          uint32_t a0h, a0l, a2h, a2l;
          tz_split2(pv[gr][0], pv[gr][1], a0h, a0l);
          tz_split2(pv[gr][2], pv[gr][3], a2h, a2l);
          const uint32_t a0 = part ? a0l : a0h, a2 = part ? a2l : a2h;
          uint32_t v0[8], v1[8];
          if (s == 0) {
            tz_pairs8<2>(r[gr][0], r[gr][1], o, v0);
            tz_pairs8<2>(r[gr][2], r[gr][3], o, v1);
          } else if (s == 1) {
            tz_pairs8<4>(r[gr][0], r[gr][1], o, v0);
            tz_pairs8<4>(r[gr][2], r[gr][3], o, v1);
          } else if (s == 2) {
            tz_pairs8<8>(r[gr][0], r[gr][1], o, v0);
            tz_pairs8<8>(r[gr][2], r[gr][3], o, v1);
          } else {
            tz_pairs8<16>(r[gr][0], r[gr][1], o, v0);
            tz_pairs8<16>(r[gr][2], r[gr][3], o, v1);
          }
#pragma unroll
          for (int jn = 0; jn < 8; ++jn) tz_mma(oacc[gr][jn][0], oacc[gr][jn][1], a0, a2, v0[jn], v1[jn]);
        }
      }
    }
    __syncwarp();
  }

  // ---- merge the warps' states, then the CTA's partial ----
  // high and low rows: add the lane 16 apart; lane (gq < 4, t4) then holds head
  // gq's output for channels 64*gr + 8*(2*t4) + jn and 64*gr + 8*(2*t4 + 1) + jn
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      oacc[a][b][0] += __shfl_xor_sync(0xffffffffu, oacc[a][b][0], 16);
      oacc[a][b][1] += __shfl_xor_sync(0xffffffffu, oacc[a][b][1], 16);
    }
  __syncthreads();                                 // every warp is done with its buffers
  if (lane < 16) {
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        sh.u.merge.o[warp][hrow][64 * a + 16 * t4 + b] = oacc[a][b][0];
        sh.u.merge.o[warp][hrow][64 * a + 16 * t4 + 8 + b] = oacc[a][b][1];
      }
    if (t4 == 0) {
      sh.u.merge.m[warp][hrow] = m_run;
      sh.u.merge.l[warp][hrow] = l_run;
    }
  }
  __syncthreads();
  pdl_trigger();
  for (int i = tid; i < HG * kTzD; i += kTzThreads) {
    const int h = i / kTzD, c = i % kTzD;
    float M = -INFINITY;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) M = fmaxf(M, sh.u.merge.m[w8][h]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w8 = 0; w8 < 8; ++w8) {
        const float mw = sh.u.merge.m[w8][h];
        if (mw == -INFINITY) continue;
        const float f = ex2_approx(mw - M);
        L = fmaf(sh.u.merge.l[w8][h], f, L);
        O = fmaf(sh.u.merge.o[w8][h][c], f, O);
      }
    }
    const long long rr = static_cast<long long>(hd0 + h) * slots + blockIdx.x;
    po[rr * kTzD + c] = O;
    if (c == 0) {
      pm[rr] = M;
      pl[rr] = L;
    }
  }
}

// ---------------------------------------------------------------------------
// zone C: bf16 rows, 128 tokens per step, one token per thread for the logits
// and one row per warp step (lane: 4 channels) for the output
// ---------------------------------------------------------------------------
template <int HG>
__device__ __forceinline__ void tz_block_reduce(float (&v)[HG], float (&buf)[8][4], bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    float x = v[h];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float y = __shfl_xor_sync(0xffffffffu, x, o);
      x = is_max ? fmaxf(x, y) : x + y;
    }
    if (lane == 0) buf[warp][h] = x;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    float x = buf[0][h];
#pragma unroll
    for (int w8 = 1; w8 < 8; ++w8) x = is_max ? fmaxf(x, buf[w8][h]) : x + buf[w8][h];
    v[h] = x;
  }
}

template <int HG>
__device__ __forceinline__ void tz_zone_c(TzZoneCShared& sh, const uint16_t* __restrict__ q,
                                          const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                                          int nc, int nc_cap, int hd0, int part_idx, int nparts, float qscale,
                                          float* __restrict__ pm, float* __restrict__ pl, float* __restrict__ po,
                                          int slots) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y;
  const long long nchunks = (nc + kTzChunkC - 1) / kTzChunkC;
  const long long c0 = part_idx * nchunks / nparts, c1 = (part_idx + 1) * nchunks / nparts;
  for (int i = tid; i < HG * kTzD; i += kTzThreads) {
    const int h = i / kTzD, c = i % kTzD;
    sh.qs[c][h] = bf16_lo(q[static_cast<long long>(hd0 + h) * kTzD + c]) * qscale;
  }
  float m_run[HG], l_run[HG], oacc[HG][4];
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[h][e] = 0.f;
  }
  for (long long ck = c0; ck < c1; ++ck) {
    const long long i0 = ck * kTzChunkC;
    const int cnt = static_cast<int>(nc - i0 < kTzChunkC ? nc - i0 : kTzChunkC);
    __syncthreads();                                  // sh.p of the previous step is consumed
    float logit[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) logit[h] = -INFINITY;
    if (tid < cnt) {
      float a[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) a[h] = 0.f;
      const uint4* kr = reinterpret_cast<const uint4*>(k_new + (static_cast<long long>(g) * nc_cap + i0 + tid) * kTzD);
      for (int c8 = 0; c8 < kTzD / 8; ++c8) {
        const uint4 r = __ldg(kr + c8);
        const float f[8] = {bf16_lo(r.x), bf16_hi(r.x), bf16_lo(r.y), bf16_hi(r.y),
                            bf16_lo(r.z), bf16_hi(r.z), bf16_lo(r.w), bf16_hi(r.w)};
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
          for (int h = 0; h < HG; ++h) a[h] = fmaf(f[e], sh.qs[c8 * 8 + e][h], a[h]);
      }
#pragma unroll
      for (int h = 0; h < HG; ++h) logit[h] = a[h];
    }
    float mc[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) mc[h] = logit[h];
    tz_block_reduce<HG>(mc, sh.hm, true);
    float ps[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      const float mn = fmaxf(m_run[h], mc[h]);
      const float alpha = ex2_approx(m_run[h] - mn);
      m_run[h] = mn;
      l_run[h] *= alpha;
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[h][e] *= alpha;
      const float pr = tid < cnt ? ex2_approx(logit[h] - mn) : 0.f;
      if (tid < kTzChunkC) sh.p[tid][h] = pr;
      ps[h] = pr;
    }
    tz_block_reduce<HG>(ps, sh.hs, false);            // its barrier also publishes sh.p
#pragma unroll
    for (int h = 0; h < HG; ++h) l_run[h] += ps[h];
    for (int t = warp; t < cnt; t += 8) {
      const uint2 r = __ldg(reinterpret_cast<const uint2*>(
          v_new + (static_cast<long long>(g) * nc_cap + i0 + t) * kTzD + 4 * lane));
      const float f[4] = {bf16_lo(r.x), bf16_hi(r.x), bf16_lo(r.y), bf16_hi(r.y)};
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float p = sh.p[t][h];
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[h][e] = fmaf(p, f[e], oacc[h][e]);
      }
    }
  }
  __syncthreads();
  pdl_trigger();
#pragma unroll
  for (int h = 0; h < HG; ++h)
    *reinterpret_cast<float4*>(&sh.red[warp][h][4 * lane]) = make_float4(oacc[h][0], oacc[h][1], oacc[h][2], oacc[h][3]);
  __syncthreads();
  const bool empty = c0 >= c1;
  for (int i = tid; i < HG * kTzD; i += kTzThreads) {
    const int h = i / kTzD, c = i % kTzD;
    float s = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) s += sh.red[w8][h][c];
    const long long rr = static_cast<long long>(hd0 + h) * slots + blockIdx.x;
    po[rr * kTzD + c] = s;
    if (c == 0) {
      pm[rr] = empty ? -INFINITY : m_run[h];
      pl[rr] = empty ? 0.f : l_run[h];
    }
  }
}

// ---------------------------------------------------------------------------
// decode: grid (n_split + n_csplit, Hkv, G / HG), 256 threads
// ---------------------------------------------------------------------------
template <int HG>
__global__ void __launch_bounds__(kTzThreads, 2) trizone_decode_kernel(
    const uint16_t* __restrict__ q, int G, int N, StreamPtrs ks, StreamPtrs vs, const long long* __restrict__ hdr,
    const int* __restrict__ vstart, const uint8_t* __restrict__ vslot, const uint16_t* __restrict__ k_new,
    const uint16_t* __restrict__ v_new, const int* __restrict__ n_new, int nc_cap, int n_split, float qscale,
    float* __restrict__ pm, float* __restrict__ pl, float* __restrict__ po) {
  __shared__ __align__(16) TzShared sh;
  const int g = blockIdx.y;
  const int hd0 = g * G + blockIdx.z * HG;          // first query head of this CTA
  const int slots = gridDim.x;
  const int x = blockIdx.x;
  pdl_wait();
  if (x < n_split) {
    const long long* H = hdr + static_cast<long long>(g) * kTzHdr;
    long long nkept = H[TZ_NKEPT];
    nkept = nkept < 0 ? 0 : (nkept > N ? N : nkept);   // an index not built for this pool reads nothing outside it
    const long long ngmax = (N + 63) / 64;
    tz_packed<HG>(sh.a, q, ks, vs, H, vstart + static_cast<long long>(g) * (ngmax + 1) * 4,
                  vslot + static_cast<long long>(g) * N, nkept, hd0, x, n_split, qscale, pm, pl, po, slots);
  } else {
    int nc = n_new ? *n_new : 0;
    if (nc < 0 || nc > nc_cap) {
      if (x == n_split && g == 0 && blockIdx.z == 0 && threadIdx.x == 0) record_error(KVS_ERR_RANGE);
      nc = nc < 0 ? 0 : nc_cap;
    }
    tz_zone_c<HG>(sh.c, q, k_new, v_new, nc, nc_cap, hd0, x - n_split, slots - n_split, qscale, pm, pl, po, slots);
  }
}

// ---------------------------------------------------------------------------
// combine: one CTA of 1024 threads per query head; thread (r, c) adds the
// partials r, r + 8, ... of channel c, then the 8 sums are added in order.
// Empty partials (max = -inf) get weight 0; their outputs are written as 0.
// ---------------------------------------------------------------------------
constexpr int kTzCombineThreads = 8 * kTzD;

__global__ void __launch_bounds__(kTzCombineThreads) trizone_combine_kernel(int slots, const float* __restrict__ pm,
                                                                            const float* __restrict__ pl,
                                                                            const float* __restrict__ po,
                                                                            float* __restrict__ out,
                                                                            float* __restrict__ lse) {
  pdl_wait();
  __shared__ float s_f[1024], s_o[8][kTzD], s_red[32], s_M;
  const int hd = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long r0 = static_cast<long long>(hd) * slots;
  const int n = slots < 1024 ? slots : 1024;        // the host keeps slots <= 1024
  float m = tid < n ? pm[r0 + tid] : -INFINITY;
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) s_red[warp] = M;
  __syncthreads();
  if (tid == 0) {
    float x = s_red[0];
    for (int w = 1; w < 32; ++w) x = fmaxf(x, s_red[w]);
    s_M = x;
  }
  __syncthreads();
  M = s_M;
  const float f = (tid < n && M != -INFINITY && m != -INFINITY) ? exp2f(m - M) : 0.f;
  if (tid < n) s_f[tid] = f;
  float L = tid < n ? pl[r0 + tid] * f : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  __syncthreads();
  if (lane == 0) s_red[warp] = L;
  __syncthreads();
  const int c = tid & (kTzD - 1), r = tid >> 7;
  float O = 0.f;
  for (int x = r; x < n; x += 8) O = fmaf(po[(r0 + x) * kTzD + c], s_f[x], O);
  s_o[r][c] = O;
  __syncthreads();
  if (tid < kTzD) {
    float Ls = 0.f;
    for (int w = 0; w < 32; ++w) Ls += s_red[w];
    float Os = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) Os += s_o[k][tid];
    out[static_cast<long long>(hd) * kTzD + tid] = Ls > 0.f ? Os / Ls : 0.f;
    if (tid == 0) lse[hd] = Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
  }
}

}  // namespace kvs
