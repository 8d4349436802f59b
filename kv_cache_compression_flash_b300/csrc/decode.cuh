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
// Three kernels:
//   trizone_index_kernel   once per compressed pool: per KV head the number of
//                          kept tokens, the K entry range of each width and,
//                          for every kept token in ascending order, where its V
//                          row sits (width slot << 30 | first group).
//   trizone_decode_kernel  per (chunk of 256 kept or new tokens, KV head, head
//                          slice): logits from the channel-major K codes, the
//                          chunk's softmax numerators, and the V products;
//                          writes (max, sum, unnormalised output) per head.
//   trizone_combine_kernel per query head: merges the chunk partials in chunk
//                          order (log-sum-exp merge), writes out and lse.
//
// Arithmetic: fp32 throughout; logits in the log2 domain (q is pre-multiplied
// by log2(e)/sqrt(d)); the scale of a K group is folded into the query
// (q'_c = q_c * s_{c,j}) and the scale of a V group into the probability
// (p'_t = p_t * s_{t,j}).  A w-bit two's-complement code x becomes a float
// exactly: the bit pattern 0x4B000000 | (x ^ 2^(w-1)) is the float
// 2^23 + x + 2^(w-1), from which one subtraction leaves x.
#pragma once

#include "common.cuh"
#include "pack.cuh"

namespace kvs {

constexpr int kTzChunk = 128;     // tokens per decode step of a CTA (2 groups of 64)
constexpr int kTzThreads = 256;   // 8 warps
constexpr int kTzD = 128;         // head dimension of the decode kernels
constexpr int kTzHdr = 16;        // int64 header words per KV head in the index
constexpr uint32_t kTzLocMask = (1u << 30) - 1;

// header words of one KV head
enum { TZ_NKEPT = 0, TZ_KELO = 1, TZ_KN = 5, TZ_KGLO = 9, TZ_NG = 13 };

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
                                                             int N, int d, long long* hdr, uint32_t* vloc) {
  pdl_wait();
  const int g = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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
      long long rank = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) rank += s_base[k] + static_cast<long long>((excl >> (16 * k)) & 0xffffull);
      const long long e = s_vlo[slot] + s_base[slot] + static_cast<long long>((excl >> (16 * slot)) & 0xffffull);
      const long long want = static_cast<long long>(g) * N + t;
      if (e < tz_count(vs, slot) && static_cast<long long>(vs.ids[slot][e]) == want) {
        const long long fg = vs.goff[slot][e];
        if (fg >= 0 && fg <= static_cast<long long>(kTzLocMask))
          vloc[static_cast<long long>(g) * N + rank] = (static_cast<uint32_t>(slot) << 30) | static_cast<uint32_t>(fg);
        else
          record_error(KVS_ERR_RANGE);
      } else {
        record_error(KVS_ERR_RANGE);   // the V streams do not match bits_v
      }
    }
    __syncthreads();
    if (tid < 4) s_base[tid] += static_cast<long long>((s_wsum[31] >> (16 * tid)) & 0xffffull);
    __syncthreads();
  }
  const long long nkept = s_base[0] + s_base[1] + s_base[2] + s_base[3];
  const long long nG = (nkept + 63) / 64;
  if (tid < 4) {
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
// code decoding
// ---------------------------------------------------------------------------
template <int W>
__device__ __forceinline__ float tz_code(uint32_t word, int sh) {
  constexpr uint32_t kMask = (1u << W) - 1u;
  constexpr uint32_t kMagic = 0x4B000000u | (1u << (W - 1));
  constexpr float kBias = 8388608.0f + static_cast<float>(1u << (W - 1));
  return __uint_as_float(((word >> sh) & kMask) ^ kMagic) - kBias;
}


constexpr int kTzKU = kTzD / 8;   // K channels per warp (8 warps split the channels)
constexpr int kTzVU = kTzChunk / 8;   // V rows per warp

struct TzShared {
  float qs[kTzD][4];                       // scaled query, [channel][head]
  float qp[kTzD][2][4];                    // q times the scale of the chunk's group, [channel slot][group][head]
  int ch_id[kTzD];
  int ch_w[kTzD];                          // 0: skip the channel
  const uint8_t* ch_code[kTzD];            // code block of the channel's first group
  const uint16_t* ch_scale[kTzD];          // its scale (widths 2/4/8)
  const uint8_t* v_code[4];
  const uint16_t* v_scale[4];
  long long v_cap[4];
  float red[8][4][kTzChunk];               // cross-warp partial logits / outputs
  float p[kTzChunk][4];                    // softmax numerators, [token][head]
  float pp[kTzChunk][2][4];                // p times the scale of the row's group, [token][group][head]
  float hm[8][4], hs[8][4];                // per-warp max and sum
};

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

// four w-bit codes (or four bf16 values when w = 16) from the low bits of r, as floats
__device__ __forceinline__ void tz_decode4(unsigned long long r, int w, float (&f)[4]) {
  const uint32_t lo = static_cast<uint32_t>(r), hi = static_cast<uint32_t>(r >> 32);
  if (w == 2) {
#pragma unroll
    for (int e = 0; e < 4; ++e) f[e] = tz_code<2>(lo, 2 * e);
  } else if (w == 4) {
#pragma unroll
    for (int e = 0; e < 4; ++e) f[e] = tz_code<4>(lo, 4 * e);
  } else if (w == 8) {
#pragma unroll
    for (int e = 0; e < 4; ++e) f[e] = tz_code<8>(lo, 8 * e);
  } else {
    f[0] = bf16_lo(lo); f[1] = bf16_hi(lo); f[2] = bf16_lo(hi); f[3] = bf16_hi(hi);
  }
}

// acc[h][pair] += f * v[h] over 4 values
template <int HG>
__device__ __forceinline__ void tz_fma4v(unsigned long long (&acc)[HG][2], const float (&f)[4], const float4& v) {
  const unsigned long long f01 = f2_pack(f[0], f[1]), f23 = f2_pack(f[2], f[3]);
  const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    const unsigned long long pp = f2_pack(vv[h], vv[h]);
    acc[h][0] = f2_fma(f01, pp, acc[h][0]);
    acc[h][1] = f2_fma(f23, pp, acc[h][1]);
  }
}

// ---------------------------------------------------------------------------
// decode: grid (n_split + n_csplit, Hkv, G / HG), 256 threads.  CTA x < n_split
// walks its share of the old zone's 128-token chunks, CTA x >= n_split its
// share of zone C's, keeping a running max and sum over the chunks (flash
// decoding); each writes one partial per head.
//
// Per chunk every load is issued before any is used: lane l of warp w holds
// the codes of K channel slots w, w+8, ... for tokens 4l..4l+3 and the V
// codes of rows 16w..16w+15 for channels 4(l%16)..+3 of group l/16; thread t
// fetches one K scale (slot t/2, group t%2) and one V scale (row t/2, group
// t%2); the V row locations of the next chunk are fetched one chunk ahead.
// ---------------------------------------------------------------------------
template <int HG>
__global__ void __launch_bounds__(kTzThreads, 2) trizone_decode_kernel(
    const uint16_t* __restrict__ q, int G, int N, StreamPtrs ks, StreamPtrs vs, const long long* __restrict__ hdr,
    const uint32_t* __restrict__ vloc, const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
    const int* __restrict__ n_new, int nc_cap, int n_split, float qscale, float* __restrict__ pm,
    float* __restrict__ pl, float* __restrict__ po) {
  __shared__ __align__(16) TzShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y;
  const int hd0 = g * G + blockIdx.z * HG;          // first query head of this CTA
  const int slots = gridDim.x;
  const int x = blockIdx.x;
  const bool old_zone = x < n_split;

  pdl_wait();
  const long long* H = hdr + static_cast<long long>(g) * kTzHdr;
  long long nkept = H[TZ_NKEPT];
  nkept = nkept < 0 ? 0 : (nkept > N ? N : nkept);   // an index not built for this pool reads nothing outside it
  long long nvalid = nkept;
  if (!old_zone) {
    int nc = n_new ? *n_new : 0;
    if (nc < 0 || nc > nc_cap) {
      if (x == n_split && g == 0 && blockIdx.z == 0 && tid == 0) record_error(KVS_ERR_RANGE);
      nc = nc < 0 ? 0 : nc_cap;
    }
    nvalid = nc;
  }
  const long long nchunks = (nvalid + kTzChunk - 1) / kTzChunk;
  const long long nparts = old_zone ? n_split : slots - n_split;
  const long long part = old_zone ? x : x - n_split;
  const long long c0 = part * nchunks / nparts, c1 = (part + 1) * nchunks / nparts;

  for (int i = tid; i < HG * kTzD; i += kTzThreads) {
    const int h = i / kTzD, c = i % kTzD;
    sh.qs[c][h] = bf16_lo(q[static_cast<long long>(hd0 + h) * kTzD + c]) * qscale;
  }
  const long long nG = (nkept + 63) / 64;
  int nch = 0;
  if (old_zone) {
    // channel list of this KV head, width by width
    long long n_s[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      long long n = H[TZ_KN + s];
      n = n < 0 ? 0 : (n > kTzD - nch ? kTzD - nch : n);
      n_s[s] = n;
      nch += static_cast<int>(n);
    }
    if (tid < kTzD) {
      sh.ch_id[tid] = 0;
      sh.ch_w[tid] = 0;
      sh.ch_code[tid] = nullptr;
      sh.ch_scale[tid] = nullptr;
    }
    if (tid < nch) {
      int k = tid, s = 0;
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        if (s == i && k >= n_s[i]) {
          k -= static_cast<int>(n_s[i]);
          s = i + 1;
        }
      }
      const long long e = H[TZ_KELO + s] + k;
      const long long grp = H[TZ_KGLO + s] + static_cast<long long>(k) * nG;
      const int c = e >= 0 && e < ks.cap_units[s] ? ks.ids[s][e] - g * kTzD : -1;
      if (c < 0 || c >= kTzD || grp < 0 || grp + nG > ks.cap_groups[s]) {
        record_error(KVS_ERR_RANGE);          // index and streams disagree: the channel is skipped
      } else {
        const int w = 2 << s;
        sh.ch_id[tid] = c;
        sh.ch_w[tid] = w;
        sh.ch_code[tid] = ks.codes[s] + grp * (8 * w);
        sh.ch_scale[tid] = s < 3 ? ks.scales[s] + grp : nullptr;
      }
    }
    if (tid < 4) {
      sh.v_code[tid] = vs.codes[tid];
      sh.v_scale[tid] = vs.scales[tid];
      sh.v_cap[tid] = vs.cap_groups[tid];
    }
  }

  float m_run[HG], l_run[HG];
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
  }
  unsigned long long oacc[HG][2];
#pragma unroll
  for (int h = 0; h < HG; ++h) oacc[h][0] = oacc[h][1] = 0ull;
  const int sg = lane >> 4, spos = lane & 15;        // group (0/1) and position of the lane's 4 values
  const long long vrow0 = static_cast<long long>(g) * N;

  // V row locations of the first chunk: vlw (lane < 16: row 16*warp + lane), vls (row tid/2)
  uint32_t vlw = 0u, vls = 0u;
  if (old_zone && c0 < c1) {
    const long long i0 = c0 * kTzChunk;
    if (lane < 16 && i0 + kTzVU * warp + lane < nvalid) vlw = __ldg(vloc + vrow0 + i0 + kTzVU * warp + lane);
    if (i0 + (tid >> 1) < nvalid) vls = __ldg(vloc + vrow0 + i0 + (tid >> 1));
  }

  for (long long ck = c0; ck < c1; ++ck) {
    const long long i0 = ck * kTzChunk;
    const int cnt = static_cast<int>(nvalid - i0 < kTzChunk ? nvalid - i0 : kTzChunk);
    __syncthreads();                                  // the previous chunk is done with the shared arrays

    // ---- every load of the chunk ----
    unsigned long long kraw[kTzKU], vraw[kTzVU];
    float ksc = 0.f, vsc = 1.f;
    uint32_t vlw_next = 0u, vls_next = 0u;
    if (old_zone) {
      const long long gj = 2 * ck + sg;               // the lane's K group within each channel
#pragma unroll
      for (int u = 0; u < kTzKU; ++u) {
        const int k = warp + 8 * u;
        const int w = (k < nch && gj < nG) ? sh.ch_w[k] : 0;
        kraw[u] = 0ull;
        if (w) {
          const uint8_t* pc = sh.ch_code[k] + gj * (8 * w) + spos * (w >> 1);
          kraw[u] = __ldg(reinterpret_cast<const unsigned long long*>(reinterpret_cast<uintptr_t>(pc) & ~static_cast<uintptr_t>(7)));
        }
      }
      {
        const int k = tid >> 1;
        const long long gk = 2 * ck + (tid & 1);
        const int w = (k < nch && gk < nG) ? sh.ch_w[k] : 0;
        if (w) ksc = w < 16 ? __half2float(__ushort_as_half(__ldg(sh.ch_scale[k] + gk))) : 1.f;
      }
#pragma unroll
      for (int u = 0; u < kTzVU; ++u) {
        const uint32_t vl = __shfl_sync(0xffffffffu, vlw, u);
        vraw[u] = 0ull;
        if (kTzVU * warp + u < cnt) {
          const int s = static_cast<int>(vl >> 30);
          const long long grp = static_cast<long long>(vl & kTzLocMask) + sg;
          if (grp < sh.v_cap[s]) {
            const int w = 2 << s;
            const uint8_t* pv = sh.v_code[s] + grp * (8 * w) + spos * (w >> 1);
            vraw[u] = __ldg(reinterpret_cast<const unsigned long long*>(reinterpret_cast<uintptr_t>(pv) & ~static_cast<uintptr_t>(7)));
          } else {
            record_error(KVS_ERR_RANGE);      // index and streams disagree: the row is skipped
          }
        }
      }
      if ((tid >> 1) < cnt) {
        const int s = static_cast<int>(vls >> 30);
        const long long grp = static_cast<long long>(vls & kTzLocMask) + (tid & 1);
        if (s < 3 && grp < sh.v_cap[s]) vsc = __half2float(__ushort_as_half(__ldg(sh.v_scale[s] + grp)));
      }
      if (ck + 1 < c1) {
        const long long i1 = i0 + kTzChunk;
        if (lane < 16 && i1 + kTzVU * warp + lane < nvalid) vlw_next = __ldg(vloc + vrow0 + i1 + kTzVU * warp + lane);
        if (i1 + (tid >> 1) < nvalid) vls_next = __ldg(vloc + vrow0 + i1 + (tid >> 1));
      }
    } else {
#pragma unroll
      for (int u = 0; u < kTzVU; ++u) {
        const int j = kTzVU * warp + u;
        vraw[u] = j < cnt ? __ldg(reinterpret_cast<const unsigned long long*>(
                                v_new + (static_cast<long long>(g) * nc_cap + i0 + j) * kTzD + 4 * lane))
                          : 0ull;
      }
    }

    // ---- logits ----
    float logit[HG];
    if (old_zone) {
      {
        const int k = tid >> 1, gsel = tid & 1;
        const int c = sh.ch_id[k];
#pragma unroll
        for (int h = 0; h < 4; ++h) sh.qp[k][gsel][h] = h < HG ? sh.qs[c][h] * ksc : 0.f;
      }
      __syncthreads();
      unsigned long long acc[HG][2];
#pragma unroll
      for (int h = 0; h < HG; ++h) acc[h][0] = acc[h][1] = 0ull;
#pragma unroll
      for (int u = 0; u < kTzKU; ++u) {
        const int k = warp + 8 * u;
        const int w = k < nch ? sh.ch_w[k] : 0;
        if (!w) continue;
        float f[4];
        tz_decode4(kraw[u] >> (((spos * (w >> 1)) & 7) * 8), w, f);
        tz_fma4v<HG>(acc, f, *reinterpret_cast<const float4*>(sh.qp[k][sg]));
      }
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        float a0, a1, a2, a3;
        f2_unpack(acc[h][0], &a0, &a1);
        f2_unpack(acc[h][1], &a2, &a3);
        *reinterpret_cast<float4*>(&sh.red[warp][h][4 * lane]) = make_float4(a0, a1, a2, a3);
      }
      __syncthreads();
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        float sacc = 0.f;
        if (tid < kTzChunk) {
#pragma unroll
          for (int w8 = 0; w8 < 8; ++w8) sacc += sh.red[w8][h][tid];
        }
        logit[h] = tid < cnt ? sacc : -INFINITY;
      }
    } else {
      // zone C: bf16 rows, one token per thread
      float a[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) a[h] = 0.f;
      if (tid < cnt) {
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
      }
#pragma unroll
      for (int h = 0; h < HG; ++h) logit[h] = tid < cnt ? a[h] : -INFINITY;
    }

    // ---- running max and sum over the chunks ----
    float mc[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) mc[h] = logit[h];
    tz_block_reduce<HG>(mc, sh.hm, true);
    float ps[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      const float mn = fmaxf(m_run[h], mc[h]);        // finite: the chunk holds a token
      const float alpha = ex2_approx(m_run[h] - mn);   // 0 on the first chunk
      m_run[h] = mn;
      l_run[h] *= alpha;
      const unsigned long long aa = f2_pack(alpha, alpha);
      oacc[h][0] = f2_fma(oacc[h][0], aa, 0ull);
      oacc[h][1] = f2_fma(oacc[h][1], aa, 0ull);
      const float pr = tid < cnt ? ex2_approx(logit[h] - mn) : 0.f;
      if (tid < kTzChunk) sh.p[tid][h] = pr;
      ps[h] = pr;
    }
    tz_block_reduce<HG>(ps, sh.hs, false);            // its barrier also publishes sh.p
#pragma unroll
    for (int h = 0; h < HG; ++h) l_run[h] += ps[h];
    {
      const int j = tid >> 1, gsel = tid & 1;
#pragma unroll
      for (int h = 0; h < 4; ++h) sh.pp[j][gsel][h] = (h < HG && j < cnt) ? sh.p[j][h] * vsc : 0.f;
    }
    __syncthreads();

    // ---- V products ----
#pragma unroll
    for (int u = 0; u < kTzVU; ++u) {
      const int j = kTzVU * warp + u;
      if (j >= cnt) break;
      int w = 16;
      if (old_zone) w = 2 << static_cast<int>(__shfl_sync(0xffffffffu, vlw, u) >> 30);
      float f[4];
      tz_decode4(old_zone ? vraw[u] >> (((spos * (w >> 1)) & 7) * 8) : vraw[u], w, f);
      tz_fma4v<HG>(oacc, f, *reinterpret_cast<const float4*>(sh.pp[j][old_zone ? sg : 0]));
    }
    vlw = vlw_next;
    vls = vls_next;
  }

  // ---- the CTA's partial: (running max, sum, unnormalised output) per head ----
  __syncthreads();
  pdl_trigger();
  const bool empty = c0 >= c1;
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    float a0, a1, a2, a3;
    f2_unpack(oacc[h][0], &a0, &a1);
    f2_unpack(oacc[h][1], &a2, &a3);
    *reinterpret_cast<float4*>(&sh.red[warp][h][4 * lane]) = make_float4(a0, a1, a2, a3);
  }
  __syncthreads();
  if (!empty) {
    for (int i = tid; i < HG * kTzD; i += kTzThreads) {
      const int h = i / kTzD, c = i % kTzD;
      float sacc = 0.f;
#pragma unroll
      for (int w8 = 0; w8 < 8; ++w8) sacc += sh.red[w8][h][c];
      po[(static_cast<long long>(hd0 + h) * slots + x) * kTzD + c] = sacc;
    }
  }
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    if (tid == h) {
      const long long r = static_cast<long long>(hd0 + h) * slots + x;
      pm[r] = empty ? -INFINITY : m_run[h];
      pl[r] = empty ? 0.f : l_run[h];
    }
  }
}

// ---------------------------------------------------------------------------
// combine: one CTA of 128 threads per query head; merges the partials in
// order, skipping the empty ones (max = -inf)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTzD) trizone_combine_kernel(int slots, const float* __restrict__ pm,
                                                               const float* __restrict__ pl,
                                                               const float* __restrict__ po, float* __restrict__ out,
                                                               float* __restrict__ lse) {
  pdl_wait();
  const int hd = blockIdx.x, c = threadIdx.x;
  const long long r0 = static_cast<long long>(hd) * slots;
  float M = -INFINITY;
  for (int x = 0; x < slots; ++x) M = fmaxf(M, pm[r0 + x]);
  float L = 0.f, O = 0.f;
  if (M != -INFINITY) {
#pragma unroll 4
    for (int x = 0; x < slots; ++x) {
      const float m = pm[r0 + x];
      if (m == -INFINITY) continue;
      const float f = exp2f(m - M);
      L = fmaf(pl[r0 + x], f, L);
      O = fmaf(po[(r0 + x) * kTzD + c], f, O);
    }
  }
  out[static_cast<long long>(hd) * kTzD + c] = L > 0.f ? O / L : 0.f;
  if (c == 0) lse[hd] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace kvs
