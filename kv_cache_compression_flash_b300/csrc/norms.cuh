// Column and row norms for the RD weights and unit scales.
//   channel weight  w_c = |Q_{:,c}| |K_{:,c}| / sqrt(d)       [RDKV §2.1, w_c]
//   unit scale      sigma = RMS of a unit's values (token row of V, or channel
//                   of K over the tokens kept by stage 2)       [RDKV §2.1-2.2]
// HBM-bound streaming kernels: 16-byte loads, fp32 accumulation, fixed-order
// reductions (so results are deterministic).
#pragma once

#include "common.cuh"

namespace kvs {

constexpr int kNormThreads = 256;
constexpr int kColChunkRows = 64;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

// part[(g * nchunk + chunk) * DH + c] = sum over the chunk's rows r (kept ones
// when keep != null) of X[g][r][c]^2;  cnt[g * nchunk + chunk] = kept rows.
// X viewed as [groups, rows, DH]; grid (nchunk, groups).
template <int DH>
__global__ void __launch_bounds__(kNormThreads) colsumsq_kernel(const uint16_t* __restrict__ X, const int rows,
                                                                const uint8_t* __restrict__ keep,
                                                                float* __restrict__ part, int* __restrict__ cnt) {
  constexpr int TPR = DH / 8;              // threads per row
  constexpr int RPI = kNormThreads / TPR;  // rows per iteration
  __shared__ float red[RPI][DH];
  __shared__ int red_cnt[RPI];
  const int chunk = blockIdx.x, g = blockIdx.y, nchunk = gridDim.x;
  const int rsub = threadIdx.x / TPR, cseg = (threadIdx.x % TPR) * 8;
  const int r_begin = chunk * kColChunkRows, r_end = min(rows, r_begin + kColChunkRows);
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.f;
  int n = 0;
  const size_t gbase = static_cast<size_t>(g) * rows;
  for (int base = r_begin + rsub; base < r_end; base += 4 * RPI) {
    uint4 u[4];
    bool ok[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // four independent loads in flight
      const int r = base + j * RPI;
      ok[j] = r < r_end && (keep == nullptr || keep[gbase + r] != 0);
      u[j] = ok[j] ? __ldg(reinterpret_cast<const uint4*>(X + (gbase + r) * DH + cseg)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float f[8];
      bf16x8_to_f32(u[j], f);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = fmaf(f[k], f[k], acc[k]);
      n += ok[j] ? 1 : 0;
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) red[rsub][cseg + k] = acc[k];
  if (threadIdx.x % TPR == 0) red_cnt[rsub] = n;
  __syncthreads();
  for (int c = threadIdx.x; c < DH; c += kNormThreads) {
    float s = 0.f;
    for (int i = 0; i < RPI; ++i) s += red[i][c];
    part[(static_cast<size_t>(g) * nchunk + chunk) * DH + c] = s;
  }
  if (threadIdx.x == 0 && cnt) {
    int s = 0;
    for (int i = 0; i < RPI; ++i) s += red_cnt[i];
    cnt[g * nchunk + chunk] = s;
  }
}

// sum of the chunk partials of column (g, c): one warp, lane-strided, then a
// fixed xor tree (deterministic)
__device__ __forceinline__ float warp_sum_partials(const float* __restrict__ part, const int nchunk, const int g,
                                                   const int c, const int d) {
  float s = 0.f;
  for (int i = threadIdx.x & 31; i < nchunk; i += 32) s += part[(static_cast<size_t>(g) * nchunk + i) * d + c];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  return s;
}

// w_c[g][c] = sqrt(sum_q) * sqrt(sum_k) * inv_sqrt_d; one warp per output
__global__ void channel_weight_finalize_kernel(const float* __restrict__ qpart, const int nq,
                                               const float* __restrict__ kpart, const int nk, const int Hkv,
                                               const int d, const float inv_sqrt_d, float* __restrict__ w_c) {
  const int idx = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (idx >= Hkv * d) return;
  const int g = idx / d, c = idx % d;
  const float sq = warp_sum_partials(qpart, nq, g, c, d);
  const float sk = warp_sum_partials(kpart, nk, g, c, d);
  if ((threadIdx.x & 31) == 0) w_c[idx] = sqrtf(sq) * sqrtf(sk) * inv_sqrt_d;
}

// sigma[g][c] = sqrt(sum / kept), 0 when no token is kept; one warp per output
__global__ void masked_rms_finalize_kernel(const float* __restrict__ part, const int* __restrict__ cnt,
                                           const int nchunk, const int Hkv, const int d,
                                           float* __restrict__ sigma) {
  const int idx = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (idx >= Hkv * d) return;
  const int g = idx / d, c = idx % d;
  const float s = warp_sum_partials(part, nchunk, g, c, d);
  int n = 0;
  for (int i = threadIdx.x & 31; i < nchunk; i += 32) n += cnt[g * nchunk + i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xFFFFFFFFu, n, o);
  if ((threadIdx.x & 31) == 0) sigma[idx] = n > 0 ? sqrtf(s / static_cast<float>(n)) : 0.f;
}

// sigma[row] = sqrt(mean_c X[row][c]^2); DH/8 threads per row
template <int DH>
__global__ void __launch_bounds__(kNormThreads) row_rms_kernel(const uint16_t* __restrict__ X, const int rows,
                                                               float* __restrict__ sigma) {
  constexpr int TPR = DH / 8;
  constexpr int RPB = kNormThreads / TPR;
  const int sub = threadIdx.x % TPR;
  for (int base = blockIdx.x * RPB; base < rows; base += gridDim.x * RPB) {
    const int r = base + static_cast<int>(threadIdx.x / TPR);
    float acc = 0.f;
    if (r < rows) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(X + static_cast<size_t>(r) * DH + sub * 8));
      float f[8];
      bf16x8_to_f32(u, f);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc = fmaf(f[k], f[k], acc);
    }
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (sub == 0 && r < rows) sigma[r] = sqrtf(acc / static_cast<float>(DH));
  }
}

}  // namespace kvs
