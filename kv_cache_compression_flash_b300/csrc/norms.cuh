// Column and row norms for the RD weights and unit scales.
//   channel weight  w_c = |Q_{:,c}| |K_{:,c}| / sqrt(d)       [RDKV §2.1, w_c]
//   unit scale      sigma = RMS of a unit's values (token row of V, or channel
//                   of K over the tokens kept by stage 2)       [RDKV §2.1-2.2]
// HBM-bound streaming kernels: 16-byte loads, fp32 accumulation, fixed-order
// reductions (so results are deterministic).
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace kvs {

constexpr int kNormThreads = 256;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

// sigma[row] = sqrt(mean_c X[row][c]^2); DH/8 threads per row, four rows per
// thread in flight
template <int DH>
__global__ void __launch_bounds__(kNormThreads) row_rms_kernel(const uint16_t* __restrict__ X, const int rows,
                                                               float* __restrict__ sigma) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  constexpr int TPR = DH / 8;
  constexpr int RPB = kNormThreads / TPR;
  const int sub = threadIdx.x % TPR;
  for (int base = blockIdx.x * RPB * 4; base < rows; base += gridDim.x * RPB * 4) {
    uint4 u[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = base + j * RPB + static_cast<int>(threadIdx.x / TPR);
      u[j] = r < rows ? __ldg(reinterpret_cast<const uint4*>(X + static_cast<size_t>(r) * DH + sub * 8))
                      : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = base + j * RPB + static_cast<int>(threadIdx.x / TPR);
      float f[8];
      bf16x8_to_f32(u[j], f);
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) acc = fmaf(f[k], f[k], acc);
#pragma unroll
      for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
      if (sub == 0 && r < rows) sigma[r] = sqrtf(acc / static_cast<float>(DH));
    }
  }
}

// ---------------------------------------------------------------------------
// Column sums of squares on one thread-block cluster per group: CTA r of the
// cluster reduces rows [r*R, r*R + R) of group g (and of a second tensor B
// when given), the cluster's CTA 0 adds the CTAs' partials in rank order
// through distributed shared memory and writes the result, so no workspace
// and no second launch is needed (and the sum order is fixed).
//   mode kColChannelWeight: out[g][c] = sqrt(sum_A) sqrt(sum_B) * scale  (w_c)
//   mode kColMaskedRms:     out[g][c] = sqrt(sum_A over kept rows / kept), 0 if none
// grid (CL, groups), cluster (CL, 1, 1), kColThreads threads.
// ---------------------------------------------------------------------------
constexpr int kColThreads = 256;  // three CTAs per SM, each with its own copy ring
constexpr int kColChannelWeight = 0;
constexpr int kColMaskedRms = 1;
constexpr int kColChannelStats = 2;  // both from one read of the keys (A = K with keep, B = Q):
                                     // out = the masked RMS of A, out2 = sqrt(sum_A all rows) sqrt(sum_B) * scale

// The CTA's rows reach shared memory through a ring of kColStages stages,
// 16 KB each, filled by 1-D bulk copies (a CTA's rows of one group are
// contiguous), so the loads in flight are not bounded by registers: three
// CTAs per SM keep 192 KB moving.  Thread 0 issues the copies; every warp
// releases a stage after reading it.
constexpr int kColStages = 4;
constexpr int kColStageBytes = 16384;

template <int DH>
struct ColRing {
  static constexpr int kRows = kColStageBytes / (DH * 2);  // rows per stage
  uint16_t rows[kColStages][kRows * DH];
  uint64_t full[kColStages], empty[kColStages];
};

template <int DH>
__host__ __device__ constexpr size_t col_ring_bytes() { return sizeof(ColRing<DH>); }

// Chunk g (counted over the CTA's whole life) into stage g mod kColStages,
// after the warps have released chunk g - kColStages from it.
template <int DH>
__device__ __forceinline__ bool col_issue(ColRing<DH>& R, const long long g, const uint16_t* src, const int rows,
                                          volatile int* abort_flag) {
  const int s = static_cast<int>(g % kColStages);
  if (g >= kColStages && !mbar_wait(&R.empty[s], static_cast<uint32_t>((g / kColStages - 1) & 1), abort_flag))
    return false;
  const uint32_t bytes = static_cast<uint32_t>(rows) * DH * 2;
  mbar_arrive_expect_tx(&R.full[s], bytes);
  bulk_load(R.rows[s], src, bytes, &R.full[s]);
  return true;
}

// acc: sums of squares over the kept rows of [r_begin, r_end); with ALL,
// acc_all: over every row.  *chunk counts the chunks through the ring (it
// continues across calls); *issued the chunks thread 0 has issued.  Returns
// false after a timed-out wait (the flag is then set for the whole CTA).
template <int DH, bool ALL = false>
__device__ __forceinline__ bool colsq_rows(const uint16_t* __restrict__ X, const uint8_t* __restrict__ keep,
                                           const int r_begin, const int r_end, ColRing<DH>& R, long long* chunk,
                                           long long* issued, float (&acc)[8], float (&acc_all)[8], int* n_kept,
                                           volatile int* abort_flag) {
  constexpr int TPR = DH / 8;                // threads per row, 8 channels each
  constexpr int RPI = kColThreads / TPR;     // rows per step
  constexpr int CR = ColRing<DH>::kRows;
  constexpr int RPT = CR / RPI;              // rows per thread and chunk
  const int rsub = threadIdx.x / TPR, cseg = (threadIdx.x % TPR) * 8;
  const int n = max(0, r_end - r_begin);
  const int nch = (n + CR - 1) / CR;
  const long long g0 = *chunk;
  int kept = 0;
  bool ok = true;
  // the keep bytes of this thread's rows, one chunk ahead of the rows
  auto keep_bytes = [&](const int c, uint8_t (&kb)[RPT]) {
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      const int rr = rsub + k * RPI, row = c * CR + rr;
      kb[k] = (keep == nullptr || c >= nch || row >= n) ? 1 : __ldg(keep + r_begin + row);
    }
  };
  uint8_t kb_next[RPT];
  keep_bytes(0, kb_next);
  if (threadIdx.x == 0)
    for (int c = 0; c < min(nch, kColStages) && ok; ++c) {
      ok = col_issue(R, g0 + c, X + static_cast<size_t>(r_begin + c * CR) * DH, min(CR, n - c * CR), abort_flag);
      if (ok) ++*issued;
    }
  for (int c = 0; c < nch && ok; ++c) {
    const long long g = g0 + c;
    const int s = static_cast<int>(g % kColStages);
    if (!mbar_wait(&R.full[s], static_cast<uint32_t>((g / kColStages) & 1), abort_flag)) {
      ok = false;
      break;
    }
    const int m = min(CR, n - c * CR);
    const int rb = r_begin + c * CR;
    uint8_t kb[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) kb[k] = kb_next[k];
    keep_bytes(c + 1, kb_next);
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      const int rr = rsub + k * RPI;
      if (rr >= m) break;
      const uint4 u = *reinterpret_cast<const uint4*>(&R.rows[s][rr * DH + cseg]);
      float f[8];
      bf16x8_to_f32(u, f);
      if (ALL) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc_all[e] = fmaf(f[e], f[e], acc_all[e]);
      }
      if (kb[k] == 0) continue;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(f[e], f[e], acc[e]);
      ++kept;
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&R.empty[s]);
    if (threadIdx.x == 0 && c + kColStages < nch) {
      ok = col_issue(R, g + kColStages, X + static_cast<size_t>(rb + kColStages * CR) * DH,
                     min(CR, n - (c + kColStages) * CR), abort_flag);
      if (ok) ++*issued;
    }
  }
  *chunk = g0 + nch;
  *n_kept = kept;
  return ok;
}

// per-CTA column partials: red[c] = sum over the CTA's rows (fixed order)
template <int DH>
__device__ __forceinline__ void colsq_block_reduce(const float (&acc)[8], float* red_rows /*[RPI][DH]*/,
                                                   float* out /*[DH]*/) {
  constexpr int TPR = DH / 8;
  constexpr int RPI = kColThreads / TPR;
  const int rsub = threadIdx.x / TPR, cseg = (threadIdx.x % TPR) * 8;
#pragma unroll
  for (int k = 0; k < 8; ++k) red_rows[rsub * DH + cseg + k] = acc[k];
  __syncthreads();
  for (int c = threadIdx.x; c < DH; c += kColThreads) {
    float s = 0.f;
    for (int i = 0; i < RPI; ++i) s += red_rows[i * DH + c];
    out[c] = s;
  }
}

template <int DH, bool STATS>
__global__ void __launch_bounds__(kColThreads, 3) colsq_cluster_kernel(
    const uint16_t* __restrict__ A, const int rows_a, const uint8_t* __restrict__ keep_a,
    const uint16_t* __restrict__ B, const int rows_b, const int mode, const float scale, float* __restrict__ out,
    float* __restrict__ out2) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  namespace cgn = cooperative_groups;
  cgn::cluster_group cluster = cgn::this_cluster();
  constexpr int TPR = DH / 8;
  constexpr int RPI = kColThreads / TPR;
  extern __shared__ __align__(128) uint8_t col_smem[];
  ColRing<DH>& R = *reinterpret_cast<ColRing<DH>*>(col_smem);
  __shared__ float red_rows[RPI * DH];
  __shared__ float part_a[DH], part_b[DH], part_all[STATS ? DH : 1];
  __shared__ int red_n[kColThreads / 32];
  __shared__ int s_n;
  __shared__ int s_abort;
  const int CL = static_cast<int>(cluster.num_blocks());
  const int r = static_cast<int>(cluster.block_rank());
  const int g = blockIdx.y;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kColStages; ++i) {
      mbar_init(&R.full[i], 1);
      mbar_init(&R.empty[i], kColThreads / 32);
    }
    s_abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  volatile int* abort_flag = &s_abort;
  long long chunk = 0, issued = 0;
  float acc[8], acc_all[8];
  int n = 0;
  {
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = acc_all[k] = 0.f;
    const int per = (rows_a + CL - 1) / CL;
    const int r0 = min(rows_a, r * per), r1 = min(rows_a, r0 + per);
    colsq_rows<DH, STATS>(A + static_cast<size_t>(g) * rows_a * DH,
                          keep_a ? keep_a + static_cast<size_t>(g) * rows_a : nullptr, r0, r1, R, &chunk, &issued,
                          acc, acc_all, &n, abort_flag);
    colsq_block_reduce<DH>(acc, red_rows, part_a);
    if (STATS) {
      __syncthreads();
      colsq_block_reduce<DH>(acc_all, red_rows, part_all);
    }
  }
  if (threadIdx.x % TPR != 0) n = 0;  // one count per row slot
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xFFFFFFFFu, n, o);
  if ((threadIdx.x & 31) == 0) red_n[threadIdx.x >> 5] = n;
  if (B != nullptr && !*abort_flag) {
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
    const int per = (rows_b + CL - 1) / CL;
    const int r0 = min(rows_b, r * per), r1 = min(rows_b, r0 + per);
    int nb;
    colsq_rows<DH>(B + static_cast<size_t>(g) * rows_b * DH, nullptr, r0, r1, R, &chunk, &issued, acc, acc_all, &nb,
                   abort_flag);
    colsq_block_reduce<DH>(acc, red_rows, part_b);
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    // a wait ran out: let the copies already issued land before the CTA's
    // shared memory goes away (each wait bounded again)
    volatile int no_abort = 0;
    for (long long q = 0; q < issued; ++q)
      (void)mbar_wait(&R.full[q % kColStages], static_cast<uint32_t>((q / kColStages) & 1), &no_abort);
  }
  if (threadIdx.x == 0) {
    int t = 0;
    for (int i = 0; i < kColThreads / 32; ++i) t += red_n[i];
    s_n = t;
  }
  cluster.sync();  // every CTA's partials are complete
  bool any_abort = false;
  if (r == 0)
    for (int q = 0; q < CL; ++q) any_abort |= *cluster.map_shared_rank(&s_abort, q) != 0;
  if (r == 0 && !any_abort) {  // after a timed-out wait the outputs are left as they were
    for (int c = threadIdx.x; c < DH; c += kColThreads) {
      float sa = 0.f, sb = 0.f, sall = 0.f;
      int nn = 0;
      for (int q = 0; q < CL; ++q) {
        sa += cluster.map_shared_rank(part_a, q)[c];
        if (B != nullptr) sb += cluster.map_shared_rank(part_b, q)[c];
        if (STATS) sall += cluster.map_shared_rank(part_all, q)[c];
        nn += *cluster.map_shared_rank(&s_n, q);
      }
      float v;
      if (mode == kColChannelWeight)
        v = sqrtf(sa) * sqrtf(sb) * scale;
      else
        v = nn > 0 ? sqrtf(sa / static_cast<float>(nn)) : 0.f;
      out[static_cast<size_t>(g) * DH + c] = v;
      if (STATS) out2[static_cast<size_t>(g) * DH + c] = sqrtf(sall) * sqrtf(sb) * scale;
    }
  }
  cluster.sync();  // keep every CTA's shared memory until CTA 0 has read it
}

// ---------------------------------------------------------------------------
// threshold pruning with a sliding window   [KVzap §2.3]
// bits[g][t] = keep_width if score >= tau or t >= N - window, else 0; four
// scores per thread (16-byte loads when the row allows)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) threshold_keep_kernel(const float* __restrict__ score, const long long total,
                                                             const int N, const float tau, const int window,
                                                             const uint8_t keep_width, uint8_t* __restrict__ bits) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  const bool vec = (N % 4) == 0;
  for (long long i4 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * 4; i4 < total;
       i4 += static_cast<long long>(gridDim.x) * blockDim.x * 4) {
    float v[4];
    if (vec) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(score + i4));
      v[0] = f.x, v[1] = f.y, v[2] = f.z, v[3] = f.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = i4 + e < total ? score[i4 + e] : 0.f;
    }
    uint32_t out = 0;
    bool bad = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const long long i = i4 + e;
      const int t = static_cast<int>(i % N);
      if (!isfinite(v[e])) bad = true;
      const bool keep = t >= N - window || (isfinite(v[e]) && v[e] >= tau);
      out |= static_cast<uint32_t>(keep ? keep_width : 0) << (8 * e);
    }
    if (bad && i4 < total) record_error(KVS_ERR_RANGE);
    if (vec) {
      *reinterpret_cast<uint32_t*>(bits + i4) = out;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (i4 + e < total) bits[i4 + e] = static_cast<uint8_t>(out >> (8 * e));
    }
  }
}

}  // namespace kvs
