// KVSculpt: the attention targets of the compression zone and the closed-form
// values for fixed compressed keys   [KVSculpt §2: the compressed pairs are
// fitted to the block's attention output and LSE; with the keys fixed, the
// values are a ridge least-squares solution].
//
//   block_attention_kernel<DH>  grid (ceil(G*W / 8), Hkv), 256 threads: one
//       warp per query row of the group (the G heads' W rows are contiguous in
//       Q).  Keys in chunks of 32, lane l scores key c0 + l; an online softmax
//       (running max and sum) rescales the output, of which lane l owns
//       channels [l*DH/32, (l+1)*DH/32); the chunk's value rows are read
//       coalesced, one row per step, its weight broadcast by a shuffle.
//       Row r sees keys t < n_block with t <= q_pos0 + r.
//   ridge_softmax_kernel<DH>    grid (ceil(R/8), Hkv), 256 threads: one warp
//       per training query, lane l holds the logits of keys l, l+32, ...;
//       A = softmax over all k compressed keys (no mask: every training query
//       sees the whole compressed block).
//   ridge_atb_kernel            C = P^T Q (+ lam I), 32 x 32 output tiles over
//       32-row slices of P [R, m] and Q [R, n]: gives A^T A + lam I and A^T Y.
//   ridge_solve_kernel          one CTA per head: right-looking Cholesky of
//       A^T A + lam I in place, column j broadcast from shared memory, then a
//       forward and a backward substitution per right-hand side (thread c owns
//       channel c).
// fp32 throughout, on the FMA pipes.
#pragma once

#include "common.cuh"

namespace kvs {

constexpr int kRidgeMaxK = 512;
constexpr int kRidgeSolveThreads = 1024;
constexpr int kSculptRowsPerCta = 8;

__device__ __forceinline__ float sculpt_bf16(uint16_t v) { return __uint_as_float(static_cast<uint32_t>(v) << 16); }

// q . k for one bf16 key row of DH channels, q pre-scaled in shared memory
template <int DH>
__device__ __forceinline__ float sculpt_dot(const uint16_t* __restrict__ krow, const float* q) {
  const uint4* kr = reinterpret_cast<const uint4*>(krow);
  float acc = 0.f;
#pragma unroll 4
  for (int c8 = 0; c8 < DH / 8; ++c8) {
    const uint4 v = __ldg(kr + c8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(w[e] << 16), q[8 * c8 + 2 * e], acc);
      acc = fmaf(__uint_as_float(w[e] & 0xffff0000u), q[8 * c8 + 2 * e + 1], acc);
    }
  }
  return acc;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Y[hd, r, :] and lse[hd, r] over the visible keys of [0, n_block)
template <int DH>
__global__ void __launch_bounds__(256) block_attention_kernel(const uint16_t* __restrict__ Q,
                                                              const uint16_t* __restrict__ K,
                                                              const uint16_t* __restrict__ V, int G, int W, int N,
                                                              int q_pos0, int n_block, float scale,
                                                              float* __restrict__ Y, float* __restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  constexpr int E = DH / 32;  // output channels per lane
  __shared__ float qs[kSculptRowsPerCta][DH];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const int rho = blockIdx.x * kSculptRowsPerCta + warp;  // rho = j * W + r within group g
  if (rho >= G * W) return;                                // whole warps leave; no block barrier follows
  const int r = rho % W;
  const long long qrow = static_cast<long long>(g) * G * W + rho;  // = (g * G + j) * W + r
  const uint16_t* q = Q + qrow * DH;
  for (int c = lane; c < DH; c += 32) qs[warp][c] = sculpt_bf16(q[c]) * scale;
  __syncwarp();
  const int n_vis = min(n_block, q_pos0 + r + 1);  // >= 1: q_pos0 >= 0 and n_block >= 1
  const uint16_t* Kg = K + static_cast<long long>(g) * N * DH;
  const uint16_t* Vg = V + static_cast<long long>(g) * N * DH;
  float o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int c0 = 0; c0 < n_vis; c0 += 32) {
    const int t = c0 + lane;
    const float s = t < n_vis ? sculpt_dot<DH>(Kg + static_cast<long long>(t) * DH, qs[warp]) : -INFINITY;
    const float m_new = fmaxf(m, warp_max_f(s));  // finite: key c0 is visible
    const float alpha = expf(m - m_new);          // 0 on the first chunk
    const float p = t < n_vis ? expf(s - m_new) : 0.f;
    l = l * alpha + warp_sum_f(p);
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] *= alpha;
    const int jn = min(32, n_vis - c0);
    for (int jj = 0; jj < jn; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const uint16_t* vr = Vg + static_cast<long long>(c0 + jj) * DH + lane * E;
      if constexpr (E == 4) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(vr));
        o[0] = fmaf(pj, __uint_as_float(v.x << 16), o[0]);
        o[1] = fmaf(pj, __uint_as_float(v.x & 0xffff0000u), o[1]);
        o[2] = fmaf(pj, __uint_as_float(v.y << 16), o[2]);
        o[3] = fmaf(pj, __uint_as_float(v.y & 0xffff0000u), o[3]);
      } else {
        const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(vr));
        o[0] = fmaf(pj, __uint_as_float(v << 16), o[0]);
        o[1] = fmaf(pj, __uint_as_float(v & 0xffff0000u), o[1]);
      }
    }
    m = m_new;
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int e = 0; e < E; ++e) Y[qrow * DH + lane * E + e] = o[e] * inv;
  if (lse != nullptr && lane == 0) lse[qrow] = m + logf(l);
}

// A[g][r][i] = softmax_i(Qt[g][r] . Kc[g][i] * scale), one warp per row r
template <int DH>
__global__ void __launch_bounds__(256) ridge_softmax_kernel(const uint16_t* __restrict__ Qt,
                                                            const uint16_t* __restrict__ Kc, int R, int k,
                                                            float scale, float* __restrict__ A) {
  pdl_wait();
  pdl_trigger();
  __shared__ float qs[kSculptRowsPerCta][DH];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const int r = blockIdx.x * kSculptRowsPerCta + warp;
  if (r >= R) return;  // whole warps leave; no block barrier follows
  const uint16_t* q = Qt + (static_cast<long long>(g) * R + r) * DH;
  for (int c = lane; c < DH; c += 32) qs[warp][c] = sculpt_bf16(q[c]) * scale;
  __syncwarp();
  constexpr int kPer = kRidgeMaxK / 32;
  float s[kPer];
  float m = -INFINITY;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = lane + 32 * u;
    s[u] = -INFINITY;
    if (i < k) {
      s[u] = sculpt_dot<DH>(Kc + (static_cast<long long>(g) * k + i) * DH, qs[warp]);
      m = fmaxf(m, s[u]);
    }
  }
  m = warp_max_f(m);
  float sum = 0.f;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    s[u] = lane + 32 * u < k ? expf(s[u] - m) : 0.f;
    sum += s[u];
  }
  const float inv = 1.f / warp_sum_f(sum);  // the row maximum contributes 1
  float* a = A + (static_cast<long long>(g) * R + r) * k;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = lane + 32 * u;
    if (i < k) a[i] = s[u] * inv;
  }
}

// C[g][i][j] = sum_r P[g][r][i] Q[g][r][j]  (+ lam on the diagonal when add_diag)
// grid (ceil(n/32), ceil(m/32), Hkv), 256 threads: thread (ty, tx) owns rows
// ty, ty+8, ty+16, ty+24 of column tx of the 32 x 32 tile
__global__ void __launch_bounds__(256) ridge_atb_kernel(const float* __restrict__ P, const float* __restrict__ Q,
                                                        int R, int m, int n, float lam, int add_diag,
                                                        float* __restrict__ C) {
  pdl_wait();
  pdl_trigger();
  __shared__ float ps[32][33], qs[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int g = blockIdx.z;
  const int i0 = blockIdx.y * 32, j0 = blockIdx.x * 32;
  const float* Pg = P + static_cast<long long>(g) * R * m;
  const float* Qg = Q + static_cast<long long>(g) * R * n;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int r0 = 0; r0 < R; r0 += 32) {
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * 32; e += 256) {
      const int rr = e >> 5, cc = e & 31;
      const int r = r0 + rr;
      ps[rr][cc] = (r < R && i0 + cc < m) ? Pg[static_cast<long long>(r) * m + i0 + cc] : 0.f;
      qs[rr][cc] = (r < R && j0 + cc < n) ? Qg[static_cast<long long>(r) * n + j0 + cc] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int rr = 0; rr < 32; ++rr) {
      const float qv = qs[rr][tx];
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[u] = fmaf(ps[rr][ty + 8 * u], qv, acc[u]);
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = i0 + ty + 8 * u, j = j0 + tx;
    if (i < m && j < n)
      C[(static_cast<long long>(g) * m + i) * n + j] = acc[u] + ((add_diag != 0 && i == j) ? lam : 0.f);
  }
}

// In place: the lower triangle of M[g] (k x k) becomes its Cholesky factor L;
// B[g] (k x d) holds L^-1 A^T Y afterwards and Vc[g] = L^-T L^-1 A^T Y.  A
// pivot that is not positive records KVS_ERR_RANGE and the head's values are 0.
__global__ void __launch_bounds__(kRidgeSolveThreads) ridge_solve_kernel(float* __restrict__ M, float* __restrict__ B,
                                                                         int k, int d, float* __restrict__ Vc) {
  pdl_wait();
  __shared__ float s_col[kRidgeMaxK];
  __shared__ float s_piv;
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int kWarps = kRidgeSolveThreads / 32;
  const int g = blockIdx.x;
  float* Mg = M + static_cast<long long>(g) * k * k;
  float* Bg = B + static_cast<long long>(g) * k * d;
  float* Vg = Vc + static_cast<long long>(g) * k * d;
  if (tid == 0) s_bad = 0;
  for (int j = 0; j < k; ++j) {
    __syncthreads();  // column j's trailing updates are done
    if (tid == 0) {
      const float p = Mg[static_cast<long long>(j) * k + j];
      if (p > 0.f) {
        s_piv = sqrtf(p);
        Mg[static_cast<long long>(j) * k + j] = s_piv;
      } else {
        s_bad = 1;
      }
    }
    __syncthreads();
    if (s_bad) break;  // the same value in every thread after the barrier
    const float inv = 1.f / s_piv;
    for (int i = j + 1 + tid; i < k; i += kRidgeSolveThreads) {
      const float v = Mg[static_cast<long long>(i) * k + j] * inv;
      Mg[static_cast<long long>(i) * k + j] = v;
      s_col[i] = v;
    }
    __syncthreads();
    // trailing lower triangle: M[i][c] -= L[i][j] L[c][j] for j < c <= i
    for (int i = j + 1 + warp; i < k; i += kWarps) {
      const float lij = s_col[i];
      float* row = Mg + static_cast<long long>(i) * k;
      for (int c = j + 1 + lane; c <= i; c += 32) row[c] = fmaf(-lij, s_col[c], row[c]);
    }
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) record_error(KVS_ERR_RANGE);
    for (long long e = tid; e < static_cast<long long>(k) * d; e += kRidgeSolveThreads) Vg[e] = 0.f;
    return;
  }
  if (tid < d) {
    const int c = tid;
    for (int j = 0; j < k; ++j) {  // L y = A^T Y
      const float* row = Mg + static_cast<long long>(j) * k;
      float acc = Bg[static_cast<long long>(j) * d + c];
      for (int p = 0; p < j; ++p) acc = fmaf(-row[p], Bg[static_cast<long long>(p) * d + c], acc);
      Bg[static_cast<long long>(j) * d + c] = acc / row[j];
    }
    for (int j = k - 1; j >= 0; --j) {  // L^T x = y
      float acc = Bg[static_cast<long long>(j) * d + c];
      for (int p = j + 1; p < k; ++p)
        acc = fmaf(-Mg[static_cast<long long>(p) * k + j], Vg[static_cast<long long>(p) * d + c], acc);
      Vg[static_cast<long long>(j) * d + c] = acc / Mg[static_cast<long long>(j) * k + j];
    }
  }
}

}  // namespace kvs
