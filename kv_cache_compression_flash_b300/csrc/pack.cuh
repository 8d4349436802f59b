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
// Stream order (ascending unit id within a width) comes from a three-kernel
// plan: per-chunk counts, one exclusive scan over the chunks, per-unit ranks.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace kvs {

constexpr int kPlanThreads = 256;
constexpr int kPlanChunk = kPlanThreads * 4;

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
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float q = s > 0.f ? rintf(__fdiv_rn(x[e], s)) : 0.f;
    packed |= (static_cast<uint32_t>(static_cast<int>(q)) & cmask) << (w * e);
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

// ---------------------------------------------------------------------------
// plan for token units (axis 0): rank of each unit within its width
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPlanThreads) plan_count_kernel(const uint8_t* __restrict__ bits,
                                                                  const long long U,
                                                                  int* __restrict__ chunk_counts) {
  __shared__ int s_c[kPlanThreads / 32][4];
  const long long base = static_cast<long long>(blockIdx.x) * kPlanChunk + threadIdx.x * 4;
  int c[4] = {0, 0, 0, 0};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const long long u = base + e;
    if (u < U) {
      const int s = width_slot(bits[u]);
      if (s >= 0) ++c[s];
    }
  }
#pragma unroll
  for (int s = 0; s < 4; ++s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c[s] += __shfl_xor_sync(0xFFFFFFFFu, c[s], o);
  }
  if ((threadIdx.x & 31) == 0)
    for (int s = 0; s < 4; ++s) s_c[threadIdx.x >> 5][s] = c[s];
  __syncthreads();
  if (threadIdx.x < 4) {
    int t = 0;
    for (int i = 0; i < kPlanThreads / 32; ++i) t += s_c[i][threadIdx.x];
    chunk_counts[blockIdx.x * 4 + threadIdx.x] = t;
  }
}

// single block: chunk counts -> exclusive offsets (in place); totals -> counts
__global__ void __launch_bounds__(1024) plan_scan_kernel(int* __restrict__ chunk_counts, const int nchunk,
                                                         const int groups_per_unit, const StreamPtrs sp) {
  __shared__ long long s_tot[4];
  if (threadIdx.x < 4) {
    const int s = threadIdx.x;
    long long run = 0;
    for (int i = 0; i < nchunk; ++i) {
      const int v = chunk_counts[i * 4 + s];
      chunk_counts[i * 4 + s] = static_cast<int>(run);
      run += v;
    }
    s_tot[s] = run;
  }
  __syncthreads();
  if (threadIdx.x < 4) {
    const int s = threadIdx.x;
    const long long units = s_tot[s], groups = units * groups_per_unit;
    if (sp.counts) {
      sp.counts[s] = units;
      sp.counts[4 + s] = groups;
    }
    if (units > sp.cap_units[s] || groups > sp.cap_groups[s]) record_error(KVS_ERR_RANGE);
  }
}

// per-unit ranks; with `sp` non-null also writes ids and group offsets
__global__ void __launch_bounds__(kPlanThreads) plan_rank_kernel(const uint8_t* __restrict__ bits,
                                                                 const long long U,
                                                                 const int* __restrict__ chunk_off,
                                                                 const int groups_per_unit, int* __restrict__ rank,
                                                                 const StreamPtrs sp, const int write_streams) {
  __shared__ int s_w[kPlanThreads / 32][4];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long base = static_cast<long long>(blockIdx.x) * kPlanChunk + threadIdx.x * 4;
  int slot[4];
  int c[4] = {0, 0, 0, 0};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const long long u = base + e;
    slot[e] = u < U ? width_slot(bits[u]) : -1;
    if (slot[e] >= 0) ++c[slot[e]];
  }
  int ex[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    int x = c[s];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    ex[s] = x - c[s];
    if (lane == 31) s_w[warp][s] = x;
  }
  __syncthreads();
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    int before = chunk_off[blockIdx.x * 4 + s];
    for (int i = 0; i < warp; ++i) before += s_w[i][s];
    ex[s] += before;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const long long u = base + e;
    if (u >= U) break;
    const int s = slot[e];
    int r = -1;
    if (s >= 0) {
      r = ex[s]++;
      if (write_streams && r < sp.cap_units[s]) {
        sp.ids[s][r] = static_cast<int32_t>(u);
        sp.goff[s][r] = static_cast<int64_t>(r) * groups_per_unit;
      }
    }
    rank[u] = r;
  }
}

// ---------------------------------------------------------------------------
// token units (axis 0, V cache): one half-warp per 64-element group
// ---------------------------------------------------------------------------
template <int DH>
__global__ void __launch_bounds__(256) pack_rows_kernel(const uint16_t* __restrict__ X,
                                                        const uint8_t* __restrict__ bits,
                                                        const int* __restrict__ rank, const long long U,
                                                        const StreamPtrs sp) {
  constexpr int GPU = DH / 64;
  const int l16 = threadIdx.x & 15;
  const long long n_groups = U * GPU;
  const long long stride = static_cast<long long>(gridDim.x) * (blockDim.x / 16);
  for (long long gidx = static_cast<long long>(blockIdx.x) * (blockDim.x / 16) + (threadIdx.x >> 4);
       gidx < n_groups; gidx += stride) {
    const long long u = gidx / GPU;
    const int gi = static_cast<int>(gidx % GPU);
    const int w = bits[u];
    const int s = width_slot(w);
    if (s < 0) continue;
    const int r = rank[u];
    if (r < 0 || r >= sp.cap_units[s]) continue;
    const long long grp = static_cast<long long>(r) * GPU + gi;
    if (grp >= sp.cap_groups[s]) continue;
    float x[4];
    uint2 raw;
    lane_bf16x4(X + u * DH + gi * 64 + l16 * 4, x, &raw);
    uint32_t packed = 0;
    if (w != 16) {
      uint16_t sb;
      bool ovf;
      packed = quantize_lane4(x, w, &sb, &ovf);
      if (l16 == 0) {
        sp.scales[s][grp] = sb;
        if (ovf) record_error(KVS_ERR_RANGE);
      }
    }
    store_lane_codes(sp.codes[s] + grp * (8 * w), w, l16, packed, raw);
  }
}

// Token units decoded from the streams themselves: entry j of width slot s is
// unit ids[s][j] with groups goff[s][j] ..; counts[] (written by the packer)
// says how many entries each slot holds.  One half-warp per group.
template <int DH>
__global__ void __launch_bounds__(256) dequant_entries_rows_kernel(const StreamPtrs sp, float* __restrict__ out) {
  constexpr int GPU = DH / 64;
  __shared__ long long s_off[5];
  if (threadIdx.x == 0) {
    long long run = 0;
    for (int s = 0; s < 4; ++s) {
      s_off[s] = run;
      run += min(static_cast<long long>(sp.counts[s]), sp.cap_units[s]) * GPU;
    }
    s_off[4] = run;
  }
  __syncthreads();
  const int l16 = threadIdx.x & 15;
  const long long total = s_off[4];
  const long long stride = static_cast<long long>(gridDim.x) * (blockDim.x / 16);
  for (long long gidx = static_cast<long long>(blockIdx.x) * (blockDim.x / 16) + (threadIdx.x >> 4); gidx < total;
       gidx += stride) {
    int s = 0;
    while (s < 3 && gidx >= s_off[s + 1]) ++s;
    const long long local = gidx - s_off[s];
    const long long jj = local / GPU;
    const int gi = static_cast<int>(local % GPU);
    const long long u = sp.ids[s][jj];
    const long long grp = sp.goff[s][jj] + gi;
    if (grp >= sp.cap_groups[s]) continue;
    const int w = s == 3 ? 16 : (2 << s);
    float y[4];
    dequant_lane4(sp.codes[s] + grp * (8 * w), w, l16, sp.scales[s] + grp, y);
    *reinterpret_cast<float4*>(out + u * DH + gi * 64 + l16 * 4) = make_float4(y[0], y[1], y[2], y[3]);
  }
}

// ---------------------------------------------------------------------------
// channel units (axis 1, K cache) over the tokens each head keeps
// ---------------------------------------------------------------------------
// kept[g][j] = j-th kept token of head g (ascending); n_kept[g].  One block
// per head, 4 consecutive tokens per thread per step.
__global__ void __launch_bounds__(1024) kept_index_kernel(const uint8_t* __restrict__ keep_bits, const int N,
                                                          int* __restrict__ kept, int* __restrict__ n_kept) {
  __shared__ int s_w[32];
  __shared__ int s_carry;
  const int g = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  const uint8_t* kb = keep_bits + static_cast<size_t>(g) * N;
  for (int base = 0; base < N; base += 4096) {
    const int t0 = base + threadIdx.x * 4;
    int k[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) k[e] = (t0 + e < N && kb[t0 + e] != 0) ? 1 : 0;
    const int mine = k[0] + k[1] + k[2] + k[3];
    int x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    int before = s_carry;
    for (int i = 0; i < warp; ++i) before += s_w[i];
    int pos = before + x - mine;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (k[e]) kept[static_cast<size_t>(g) * N + pos++] = t0 + e;
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int i = 0; i < 32; ++i) tot += s_w[i];
      s_carry += tot;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) n_kept[g] = s_carry;
}

// single block plan over channel units u = g*DH + c: rank, ids, group offsets
// (a unit of head g has ceil(n_kept[g]/64) groups), counts and capacity check
constexpr int kPlanChannelThreads = 1024;
__global__ void __launch_bounds__(kPlanChannelThreads) plan_channels_kernel(const uint8_t* __restrict__ bits,
                                                                     const int U, const int DH,
                                                                     const int* __restrict__ n_kept,
                                                                     int* __restrict__ rank, const StreamPtrs sp,
                                                                     const int write_streams) {
  __shared__ long long s_u[kPlanChannelThreads / 32][4], s_g[kPlanChannelThreads / 32][4];
  __shared__ long long s_cu[4], s_cg[4];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < 4) s_cu[threadIdx.x] = s_cg[threadIdx.x] = 0;
  __syncthreads();
  for (int base = 0; base < U; base += kPlanChannelThreads) {
    const int u = base + threadIdx.x;
    const int s = u < U ? width_slot(bits[u]) : -1;
    const long long ng = u < U ? (n_kept[u / DH] + 63) / 64 : 0;
    long long exu[4], exg[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      long long xu = (s == q) ? 1 : 0, xg = (s == q) ? ng : 0;
      const long long cu0 = xu, cg0 = xg;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long yu = __shfl_up_sync(0xFFFFFFFFu, xu, o), yg = __shfl_up_sync(0xFFFFFFFFu, xg, o);
        if (lane >= o) {
          xu += yu;
          xg += yg;
        }
      }
      exu[q] = xu - cu0;
      exg[q] = xg - cg0;
      if (lane == 31) {
        s_u[warp][q] = xu;
        s_g[warp][q] = xg;
      }
    }
    __syncthreads();
    if (s >= 0) {
      long long ru = s_cu[s] + exu[s], rg = s_cg[s] + exg[s];
      for (int i = 0; i < warp; ++i) {
        ru += s_u[i][s];
        rg += s_g[i][s];
      }
      rank[u] = static_cast<int>(ru);
      if (write_streams && ru < sp.cap_units[s]) {
        sp.ids[s][ru] = u;
        sp.goff[s][ru] = rg;
      }
    } else if (u < U) {
      rank[u] = -1;
    }
    __syncthreads();
    if (threadIdx.x < 4) {
      for (int i = 0; i < kPlanChannelThreads / 32; ++i) {
        s_cu[threadIdx.x] += s_u[i][threadIdx.x];
        s_cg[threadIdx.x] += s_g[i][threadIdx.x];
      }
    }
    __syncthreads();
  }
  if (threadIdx.x < 4 && write_streams) {
    const int s = threadIdx.x;
    if (sp.counts) {
      sp.counts[s] = s_cu[s];
      sp.counts[4 + s] = s_cg[s];
    }
    if (s_cu[s] > sp.cap_units[s] || s_cg[s] > sp.cap_groups[s]) record_error(KVS_ERR_RANGE);
  }
}

// Width and first stream group of every channel of head g, staged once per CTA
// (so the per-channel loops below issue no dependent global loads).  base = -1
// for channels that are not stored.
template <int DH>
__device__ __forceinline__ void stage_channel_meta(const StreamPtrs& sp, const uint8_t* __restrict__ bits,
                                                   const int* __restrict__ rank, const int g, const int j,
                                                   int* s_w, long long* s_base) {
  for (int c = threadIdx.x; c < DH; c += blockDim.x) {
    const int u = g * DH + c;
    const int w = bits[u];
    const int s = width_slot(w);
    long long base = -1;
    if (s >= 0) {
      const int r = rank[u];
      if (r >= 0 && r < sp.cap_units[s]) {
        const long long grp = sp.goff[s][r] + j;
        if (grp < sp.cap_groups[s]) base = grp;
      }
    }
    s_w[c] = w;
    s_base[c] = base;
  }
}

// grid (ceil(N/64), Hkv), 256 threads: token group j of head g for every channel
template <int DH>
__global__ void __launch_bounds__(256) pack_channels_kernel(const uint16_t* __restrict__ X, const int N,
                                                            const uint8_t* __restrict__ bits,
                                                            const int* __restrict__ rank,
                                                            const int* __restrict__ kept,
                                                            const int* __restrict__ n_kept, const StreamPtrs sp) {
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
  stage_channel_meta<DH>(sp, bits, rank, g, j, s_w, s_base);
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
        sp.scales[s][grp] = sb;
        if (ovf) record_error(KVS_ERR_RANGE);
      }
    }
    store_lane_codes(sp.codes[s] + grp * (8 * w), w, l16, packed, raw);
  }
}

template <int DH>
__global__ void __launch_bounds__(256) dequant_channels_kernel(const StreamPtrs sp, const int N,
                                                               const uint8_t* __restrict__ bits,
                                                               const int* __restrict__ rank,
                                                               const int* __restrict__ kept,
                                                               const int* __restrict__ n_kept,
                                                               float* __restrict__ out) {
  constexpr int LD = DH + 1;  // odd stride: conflict-light column writes
  __shared__ float tile[64][LD];
  __shared__ int s_w[DH];
  __shared__ long long s_base[DH];
  const int j = blockIdx.x, g = blockIdx.y;
  const int n = n_kept[g];
  if (j * 64 >= n) return;
  const int rows = min(64, n - j * 64);
  stage_channel_meta<DH>(sp, bits, rank, g, j, s_w, s_base);
  __syncthreads();
  const int l16 = threadIdx.x & 15, hw = threadIdx.x >> 4;
  for (int c = hw; c < DH; c += 16) {
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    const long long grp = s_base[c];
    if (grp >= 0) {
      const int w = s_w[c];
      const int s = width_slot(w);
      dequant_lane4(sp.codes[s] + grp * (8 * w), w, l16, sp.scales[s] + grp, y);
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

// zero the rows of tokens that are not kept (bits == 0)
template <int DH>
__global__ void __launch_bounds__(256) zero_dropped_rows_kernel(const uint8_t* __restrict__ keep_bits,
                                                                const long long rows, float* __restrict__ out) {
  constexpr int TPR = DH / 4;
  const long long total = rows * TPR;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = e / TPR;
    if (keep_bits[r] == 0)
      *reinterpret_cast<float4*>(out + r * DH + (e % TPR) * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

}  // namespace kvs
