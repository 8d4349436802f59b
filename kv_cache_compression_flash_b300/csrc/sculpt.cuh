// KVSculpt: the attention targets of the compression zone and the closed-form
// values for fixed compressed keys   [KVSculpt §2: the compressed pairs are
// fitted to the block's attention output and LSE; with the keys fixed, the
// values are a ridge least-squares solution].
//
//   block_attention_kernel<DH>  flash-style on the tensor cores (mma.sync
//       m16n8k16 bf16, fp32 accumulation): 64 query rows of one KV group per
//       CTA, keys in chunks of 64 staged by cp.async, an online softmax, and
//       the P V product with P split into bf16 hi + lo so that the weights
//       keep 16 significant bits.  Row r sees keys t < n_block, t <= q_pos0 + r.
//   ridge_softmax_kernel<DH>    A = softmax over all k compressed keys (no
//       mask: every training query sees the whole compressed block), the
//       logits on the tensor cores as in the block attention, in two sweeps
//       over the keys (row max and sum, then the weights).
//   ridge_atb_kernel            C = P^T Q (+ lam I), 64 x 64 output tiles with
//       4 x 4 per thread over 16-row slices of P [R, m] and Q [R, n]: gives
//       A^T A + lam I (lower triangle) and A^T Y.
//   ridge_solve_kernel          one CTA per head: Cholesky of A^T A + lam I in
//       place by panels of 32 columns, then the forward and backward
//       substitutions for the d right-hand sides, also by blocks of 32 rows.
// A^T A, A^T Y and the solve are fp32 on the FMA pipes.
#pragma once

#include "common.cuh"

namespace kvs {

constexpr int kRidgeMaxK = 512;
constexpr int kRidgeMaxD = 128;
constexpr int kRidgeSolveThreads = 1024;

// ---- block attention on the tensor cores (mma.sync m16n8k16, bf16 -> fp32) ----
constexpr int kBaThreads = 128;  // 4 warps x 16 query rows
constexpr int kBaKeys = 64;      // keys per chunk

template <int DH>
struct BaCfg {
  static constexpr int kLd = DH + 8;                          // smem row stride (elements): 16 B of padding
  static constexpr int kTileElems = kBaKeys * kLd;            // one K or V chunk
  static constexpr size_t kSmem = 4ull * kTileElems * 2 + 128;  // K and V, two buffers each, + alignment
};

__device__ __forceinline__ void ba_cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void ba_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void ba_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ba_ldsm4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ba_ldsm4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// d += a b, a 16 x 16 row-major (a0: rows 0-7 k 0-7, a1: rows 8-15 k 0-7, a2: rows 0-7 k 8-15, a3: rows 8-15
// k 8-15), b 16 x 8 column-major (b0: k 0-7, b1: k 8-15), d 16 x 8 (d0 d1: row lane/4, d2 d3: row lane/4 + 8)
__device__ __forceinline__ void ba_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// bf16x2 (first value in the low half), round to nearest
__device__ __forceinline__ uint32_t ba_bf2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// x0, x1 = hi + lo to 16 significant bits (hi and lo bf16x2)
__device__ __forceinline__ void ba_split(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = ba_bf2(x0, x1);
  lo = ba_bf2(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
}

// Y[hd, r, :] and lse[hd, r] over the visible keys t < min(n_block, q_pos0 + r + 1).
// grid (ceil(W / PP), Hkv * G / Gt), 128 threads; PP = 64 / Gt positions of Gt
// heads of one KV group per CTA, so every key chunk serves all 64 rows.  Warp w
// takes 16 rows: head w / (4 / Gt), positions p0 + (w % (4 / Gt)) * 16 + 0..15.
// Per chunk of 64 keys (cp.async, double-buffered, rows past the block clamped
// to its last key and masked): S = Q K^T by 64 MMAs (K through ldmatrix), the
// online max and sum in the log2 domain (each row's values sit in the 4 lanes
// of a quad), then O += P V with P split into bf16 hi + lo (two MMAs, 16
// significant bits) and V through ldmatrix.trans.
template <int DH>
__global__ void __launch_bounds__(kBaThreads) block_attention_kernel(
    const uint16_t* __restrict__ Q, const uint16_t* __restrict__ K, const uint16_t* __restrict__ V, int G, int Gt,
    int W, int N, int q_pos0, int n_block, float c_log2, float* __restrict__ Y, float* __restrict__ lse) {
  constexpr int kLd = BaCfg<DH>::kLd, kTile = BaCfg<DH>::kTileElems;
  constexpr int KS = DH / 16;  // k-steps of S
  constexpr int NT = DH / 8;   // channel n-tiles of O
  constexpr int kChunks16 = DH / 8;  // 16-byte pieces per key row
  extern __shared__ uint8_t ba_raw[];
  uint16_t* sm = reinterpret_cast<uint16_t*>((reinterpret_cast<uintptr_t>(ba_raw) + 127) & ~uintptr_t(127));
  // sm: K buffer 0, K buffer 1, V buffer 0, V buffer 1
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = lane >> 2, qi = lane & 3;
  const int wph = 4 / Gt, PP = 64 / Gt;
  const int n_hc = G / Gt;
  const int g = blockIdx.y / n_hc, hc = blockIdx.y % n_hc;
  const int p0 = blockIdx.x * PP;
  const int hd = g * G + hc * Gt + warp / wph;
  const int pw = p0 + (warp % wph) * 16;  // the warp's first position (relative to the window)
  const int r_lo = min(pw + quad, W - 1), r_hi = min(pw + quad + 8, W - 1);
  const int nv_lo = min(n_block, q_pos0 + r_lo + 1), nv_hi = min(n_block, q_pos0 + r_hi + 1);
  const int p_last = min(p0 + PP - 1, W - 1);
  const int n_keys = min(n_block, q_pos0 + p_last + 1);  // keys any row of the CTA sees
  const int n_chunks = (n_keys + kBaKeys - 1) / kBaKeys;
  const uint16_t* Kg = K + static_cast<long long>(g) * N * DH;
  const uint16_t* Vg = V + static_cast<long long>(g) * N * DH;

  pdl_wait();
  pdl_trigger();
  auto load_chunk = [&](int ch, int buf) {
    const int t0 = ch * kBaKeys;
    for (int e = tid; e < kBaKeys * kChunks16; e += kBaThreads) {
      const int row = e / kChunks16, piece = e % kChunks16;
      const long long src = static_cast<long long>(min(t0 + row, n_block - 1)) * DH + piece * 8;
      const int dst = row * kLd + piece * 8;
      ba_cp16(smem_u32(sm + buf * kTile + dst), Kg + src);
      ba_cp16(smem_u32(sm + (2 + buf) * kTile + dst), Vg + src);
    }
    ba_commit();
  };
  load_chunk(0, 0);

  // Q fragments, loaded once (rows past the window repeat the last row; not stored)
  uint32_t qf[KS][4];
  {
    const uint16_t* q_lo = Q + (static_cast<long long>(hd) * W + r_lo) * DH + 2 * qi;
    const uint16_t* q_hi = Q + (static_cast<long long>(hd) * W + r_hi) * DH + 2 * qi;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qf[ks][0] = __ldg(reinterpret_cast<const uint32_t*>(q_lo + 16 * ks));
      qf[ks][1] = __ldg(reinterpret_cast<const uint32_t*>(q_hi + 16 * ks));
      qf[ks][2] = __ldg(reinterpret_cast<const uint32_t*>(q_lo + 16 * ks + 8));
      qf[ks][3] = __ldg(reinterpret_cast<const uint32_t*>(q_hi + 16 * ks + 8));
    }
  }
  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;  // l: this lane's part of the row sum

  // ldmatrix row addresses: lane l feeds row l % 8 of matrix l / 8
  const int mi = lane >> 3, mr = lane & 7;
  const int k_row = (mi >> 1) * 8 + mr, k_col = (mi & 1) * 8;  // K: keys (+8 for matrices 2, 3), channels
  const int v_row = (mi & 1) * 8 + mr, v_col = (mi >> 1) * 8;  // V: keys (+8 for matrices 1, 3), channels

  for (int ch = 0; ch < n_chunks; ++ch) {
    const int buf = ch & 1;
    if (ch + 1 < n_chunks) {
      load_chunk(ch + 1, buf ^ 1);
      ba_wait<1>();
    } else {
      ba_wait<0>();
    }
    __syncthreads();
    const uint32_t kbase = smem_u32(sm + buf * kTile), vbase = smem_u32(sm + (2 + buf) * kTile);
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int n2 = 0; n2 < 4; ++n2) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t b0, b1, b2, b3;
        ba_ldsm4(kbase + ((16 * n2 + k_row) * kLd + 16 * ks + k_col) * 2, b0, b1, b2, b3);
        ba_mma(s[2 * n2], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
        ba_mma(s[2 * n2 + 1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
      }
    }
    // mask, scale to the log2 domain, chunk maxima
    const int t0 = ch * kBaKeys;
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = t0 + 8 * j + 2 * qi;
      s[j][0] = t < nv_lo ? s[j][0] * c_log2 : -INFINITY;
      s[j][1] = t + 1 < nv_lo ? s[j][1] * c_log2 : -INFINITY;
      s[j][2] = t < nv_hi ? s[j][2] * c_log2 : -INFINITY;
      s[j][3] = t + 1 < nv_hi ? s[j][3] * c_log2 : -INFINITY;
      mx_lo = fmaxf(mx_lo, fmaxf(s[j][0], s[j][1]));
      mx_hi = fmaxf(mx_hi, fmaxf(s[j][2], s[j][3]));
    }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);  // finite: key 0 is in chunk 0
    const float a_lo = exp2f(m_lo - mn_lo), a_hi = exp2f(m_hi - mn_hi);  // 0 on the first chunk
    m_lo = mn_lo;
    m_hi = mn_hi;
    float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      s[j][0] = exp2f(s[j][0] - mn_lo);
      s[j][1] = exp2f(s[j][1] - mn_lo);
      s[j][2] = exp2f(s[j][2] - mn_hi);
      s[j][3] = exp2f(s[j][3] - mn_hi);
      ps_lo += s[j][0] + s[j][1];
      ps_hi += s[j][2] + s[j][3];
    }
    l_lo = l_lo * a_lo + ps_lo;
    l_hi = l_hi * a_hi + ps_hi;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      o[j][0] *= a_lo;
      o[j][1] *= a_lo;
      o[j][2] *= a_hi;
      o[j][3] *= a_hi;
    }
    // O += P V: k-step kk covers keys 16 kk .. 16 kk + 15 of the chunk (n-tiles 2 kk, 2 kk + 1 of S)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t h0, h1, h2, h3, w0, w1, w2, w3;
      ba_split(s[2 * kk][0], s[2 * kk][1], h0, w0);
      ba_split(s[2 * kk][2], s[2 * kk][3], h1, w1);
      ba_split(s[2 * kk + 1][0], s[2 * kk + 1][1], h2, w2);
      ba_split(s[2 * kk + 1][2], s[2 * kk + 1][3], h3, w3);
#pragma unroll
      for (int n2 = 0; n2 < NT / 2; ++n2) {
        uint32_t b0, b1, b2, b3;
        ba_ldsm4_t(vbase + ((16 * kk + v_row) * kLd + 16 * n2 + v_col) * 2, b0, b1, b2, b3);
        ba_mma(o[2 * n2], h0, h1, h2, h3, b0, b1);
        ba_mma(o[2 * n2], w0, w1, w2, w3, b0, b1);
        ba_mma(o[2 * n2 + 1], h0, h1, h2, h3, b2, b3);
        ba_mma(o[2 * n2 + 1], w0, w1, w2, w3, b2, b3);
      }
    }
    __syncthreads();  // every warp is done with this buffer before it is refilled
  }
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
  const float i_lo = 1.f / l_lo, i_hi = 1.f / l_hi;
  const bool st_lo = pw + quad < W, st_hi = pw + quad + 8 < W;
  float* y_lo = Y + (static_cast<long long>(hd) * W + r_lo) * DH + 2 * qi;
  float* y_hi = Y + (static_cast<long long>(hd) * W + r_hi) * DH + 2 * qi;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    if (st_lo) *reinterpret_cast<float2*>(y_lo + 8 * j) = make_float2(o[j][0] * i_lo, o[j][1] * i_lo);
    if (st_hi) *reinterpret_cast<float2*>(y_hi + 8 * j) = make_float2(o[j][2] * i_hi, o[j][3] * i_hi);
  }
  if (lse != nullptr && qi == 0) {
    if (st_lo) lse[static_cast<long long>(hd) * W + r_lo] = (m_lo + log2f(l_lo)) * 0.69314718055994530942f;
    if (st_hi) lse[static_cast<long long>(hd) * W + r_hi] = (m_hi + log2f(l_hi)) * 0.69314718055994530942f;
  }
}

// A[g][r][i] = softmax_i(Qt[g][r] . Kc[g][i] / sqrt(d)) over the k compressed keys.
// grid (ceil(R / 64), Hkv), 128 threads, 16 rows a warp; the logits come from
// mma.sync as in the block attention, over chunks of 64 keys (cp.async,
// double-buffered, rows past k clamped and masked), in two sweeps: the row max
// and sum, then the normalised weights written to A.
template <int DH>
struct RsCfg {
  static constexpr int kLd = DH + 8;
  static constexpr int kTileElems = kBaKeys * kLd;
  static constexpr size_t kSmem = 2ull * kTileElems * 2 + 128;
};

template <int DH>
__global__ void __launch_bounds__(kBaThreads) ridge_softmax_kernel(const uint16_t* __restrict__ Qt,
                                                                   const uint16_t* __restrict__ Kc, int R, int k,
                                                                   float c_log2, float* __restrict__ A) {
  constexpr int kLd = RsCfg<DH>::kLd, kTile = RsCfg<DH>::kTileElems;
  constexpr int KS = DH / 16;
  constexpr int kChunks16 = DH / 8;
  extern __shared__ uint8_t rs_raw[];
  uint16_t* sm = reinterpret_cast<uint16_t*>((reinterpret_cast<uintptr_t>(rs_raw) + 127) & ~uintptr_t(127));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = lane >> 2, qi = lane & 3;
  const int g = blockIdx.y;
  const int rw = blockIdx.x * 64 + warp * 16;  // the warp's first row
  const int r_lo = min(rw + quad, R - 1), r_hi = min(rw + quad + 8, R - 1);
  const bool st_lo = rw + quad < R, st_hi = rw + quad + 8 < R;
  const int n_chunks = (k + kBaKeys - 1) / kBaKeys;
  const uint16_t* Kg = Kc + static_cast<long long>(g) * k * DH;

  pdl_wait();
  pdl_trigger();
  auto load_chunk = [&](int ch, int buf) {
    const int t0 = ch * kBaKeys;
    for (int e = tid; e < kBaKeys * kChunks16; e += kBaThreads) {
      const int row = e / kChunks16, piece = e % kChunks16;
      ba_cp16(smem_u32(sm + buf * kTile + row * kLd + piece * 8),
              Kg + static_cast<long long>(min(t0 + row, k - 1)) * DH + piece * 8);
    }
    ba_commit();
  };
  load_chunk(0, 0);
  uint32_t qf[KS][4];
  {
    const uint16_t* q_lo = Qt + (static_cast<long long>(g) * R + r_lo) * DH + 2 * qi;
    const uint16_t* q_hi = Qt + (static_cast<long long>(g) * R + r_hi) * DH + 2 * qi;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qf[ks][0] = __ldg(reinterpret_cast<const uint32_t*>(q_lo + 16 * ks));
      qf[ks][1] = __ldg(reinterpret_cast<const uint32_t*>(q_hi + 16 * ks));
      qf[ks][2] = __ldg(reinterpret_cast<const uint32_t*>(q_lo + 16 * ks + 8));
      qf[ks][3] = __ldg(reinterpret_cast<const uint32_t*>(q_hi + 16 * ks + 8));
    }
  }
  const int mi = lane >> 3, mr = lane & 7;
  const int k_row = (mi >> 1) * 8 + mr, k_col = (mi & 1) * 8;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float* a_lo = A + (static_cast<long long>(g) * R + r_lo) * k;
  float* a_hi = A + (static_cast<long long>(g) * R + r_hi) * k;
  const int n_it = 2 * n_chunks;
  for (int it = 0; it < n_it; ++it) {
    const int buf = it & 1, ch = it % n_chunks;
    if (it + 1 < n_it) {
      load_chunk((it + 1) % n_chunks, buf ^ 1);
      ba_wait<1>();
    } else {
      ba_wait<0>();
    }
    __syncthreads();
    const uint32_t kbase = smem_u32(sm + buf * kTile);
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int n2 = 0; n2 < 4; ++n2) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t b0, b1, b2, b3;
        ba_ldsm4(kbase + ((16 * n2 + k_row) * kLd + 16 * ks + k_col) * 2, b0, b1, b2, b3);
        ba_mma(s[2 * n2], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
        ba_mma(s[2 * n2 + 1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
      }
    }
    const int t0 = ch * kBaKeys;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = t0 + 8 * j + 2 * qi;
      s[j][0] = t < k ? s[j][0] * c_log2 : -INFINITY;
      s[j][1] = t + 1 < k ? s[j][1] * c_log2 : -INFINITY;
      s[j][2] = t < k ? s[j][2] * c_log2 : -INFINITY;
      s[j][3] = t + 1 < k ? s[j][3] * c_log2 : -INFINITY;
    }
    if (it < n_chunks) {  // sweep 1: the row max and sum
      float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        mx_lo = fmaxf(mx_lo, fmaxf(s[j][0], s[j][1]));
        mx_hi = fmaxf(mx_hi, fmaxf(s[j][2], s[j][3]));
      }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);  // finite: key 0 is in chunk 0
      float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        ps_lo += exp2f(s[j][0] - mn_lo) + exp2f(s[j][1] - mn_lo);
        ps_hi += exp2f(s[j][2] - mn_hi) + exp2f(s[j][3] - mn_hi);
      }
      l_lo = l_lo * exp2f(m_lo - mn_lo) + ps_lo;
      l_hi = l_hi * exp2f(m_hi - mn_hi) + ps_hi;
      m_lo = mn_lo;
      m_hi = mn_hi;
      if (it == n_chunks - 1) {  // the full row sums, then their reciprocals
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
        l_lo = 1.f / l_lo;
        l_hi = 1.f / l_hi;
      }
    } else {  // sweep 2: the weights
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int t = t0 + 8 * j + 2 * qi;
        if (st_lo && t < k) a_lo[t] = exp2f(s[j][0] - m_lo) * l_lo;
        if (st_lo && t + 1 < k) a_lo[t + 1] = exp2f(s[j][1] - m_lo) * l_lo;
        if (st_hi && t < k) a_hi[t] = exp2f(s[j][2] - m_hi) * l_hi;
        if (st_hi && t + 1 < k) a_hi[t + 1] = exp2f(s[j][3] - m_hi) * l_hi;
      }
    }
    __syncthreads();  // every warp is done with this buffer before it is refilled
  }
}

// C[g][i][j] = sum_r P[g][r][i] Q[g][r][j]  (+ lam on the diagonal when add_diag)
// grid (ceil(n/64), ceil(m/64), Hkv), 256 threads: a 64 x 64 output tile,
// thread (ty, tx) = (tid / 16, tid % 16) owns rows 4 ty .. 4 ty + 3 and columns
// 4 tx .. 4 tx + 3; slices of 16 rows of P and Q pass through shared memory,
// the next slice's loads in flight while the current one is multiplied.  With
// lower_only, tiles wholly above the diagonal are skipped: the solve reads only
// the lower triangle of A^T A + lam I.
constexpr int kAtbTile = 64, kAtbSlice = 16;

__global__ void __launch_bounds__(256) ridge_atb_kernel(const float* __restrict__ P, const float* __restrict__ Q,
                                                        int R, int m, int n, float lam, int add_diag, int lower_only,
                                                        float* __restrict__ C) {
  pdl_wait();
  pdl_trigger();
  const int i0 = blockIdx.y * kAtbTile, j0 = blockIdx.x * kAtbTile;
  if (lower_only != 0 && j0 > i0 + kAtbTile - 1) return;  // the whole CTA, before any barrier
  __shared__ __align__(16) float ps[kAtbSlice][kAtbTile];
  __shared__ __align__(16) float qs[kAtbSlice][kAtbTile];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int g = blockIdx.z;
  const float* Pg = P + static_cast<long long>(g) * R * m;
  const float* Qg = Q + static_cast<long long>(g) * R * n;
  // this thread's four loads per slice: element e = tid + 256 u -> row e / 64, column e % 64
  float pv[4], qv[4];
  auto fetch = [&](int r0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = tid + 256 * u, rr = e >> 6, cc = e & 63, r = r0 + rr;
      pv[u] = (r < R && i0 + cc < m) ? Pg[static_cast<long long>(r) * m + i0 + cc] : 0.f;
      qv[u] = (r < R && j0 + cc < n) ? Qg[static_cast<long long>(r) * n + j0 + cc] : 0.f;
    }
  };
  float acc[4][4];
#pragma unroll
  for (int u = 0; u < 4; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
  fetch(0);
  for (int r0 = 0; r0 < R; r0 += kAtbSlice) {
    __syncthreads();  // the previous slice is consumed
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = tid + 256 * u;
      ps[e >> 6][e & 63] = pv[u];
      qs[e >> 6][e & 63] = qv[u];
    }
    __syncthreads();
    if (r0 + kAtbSlice < R) fetch(r0 + kAtbSlice);
#pragma unroll
    for (int rr = 0; rr < kAtbSlice; ++rr) {
      const float4 a = *reinterpret_cast<const float4*>(&ps[rr][4 * ty]);
      const float4 b = *reinterpret_cast<const float4*>(&qs[rr][4 * tx]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int i = i0 + 4 * ty + u, j = j0 + 4 * tx + v;
      if (i < m && j < n)
        C[(static_cast<long long>(g) * m + i) * n + j] = acc[u][v] + ((add_diag != 0 && i == j) ? lam : 0.f);
    }
}

// In place: the lower triangle of M[g] (k x k) becomes its Cholesky factor L,
// B[g] (k x d) becomes L^-1 A^T Y and Vc[g] = L^-T L^-1 A^T Y.  Blocked by
// panels of kCholNb columns: the panel's diagonal block is factored by one warp
// in shared memory, the rows below it are solved against it (one thread per
// row, the row in registers) and kept in shared memory, and the trailing lower
// triangle takes the panel's rank-32 update (one warp per row, one lane per
// column).  The two triangular solves go panel by panel too: the block of 32
// rows first takes the product with every solved row (thread = row x channel),
// then its 32 x 32 triangle is solved in registers (one thread per channel).
// A pivot that is not positive records KVS_ERR_RANGE and the head's values
// are 0.
constexpr int kCholNb = 32;
constexpr int kCholLd = kCholNb + 1;  // panel row stride in shared memory (no bank conflicts)

inline size_t ridge_solve_smem(int k) { return static_cast<size_t>(k) * kCholLd * sizeof(float); }

__global__ void __launch_bounds__(kRidgeSolveThreads) ridge_solve_kernel(float* __restrict__ M, float* __restrict__ B,
                                                                         int k, int d, float* __restrict__ Vc) {
  pdl_wait();
  extern __shared__ float s_panel[];  // [k][kCholLd]: the panel's rows below its diagonal block
  __shared__ float s_diag[kCholNb][kCholLd];
  __shared__ float s_y[kCholNb * kRidgeMaxD];  // a block of 32 solution rows, [row][channel]
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int kWarps = kRidgeSolveThreads / 32;
  const int g = blockIdx.x;
  float* Mg = M + static_cast<long long>(g) * k * k;
  float* Bg = B + static_cast<long long>(g) * k * d;
  float* Vg = Vc + static_cast<long long>(g) * k * d;
  const int nd = d >> 5;  // channels per lane in the row-block products: 2 or 4
  if (tid == 0) s_bad = 0;
  __syncthreads();

  // ---- factorisation ----
  for (int J = 0; J < k; J += kCholNb) {
    const int nb = min(kCholNb, k - J);
    for (int e = tid; e < kCholNb * kCholNb; e += kRidgeSolveThreads) {
      const int r = e / kCholNb, c = e % kCholNb;
      s_diag[r][c] = (r < nb && c <= r) ? Mg[static_cast<long long>(J + r) * k + J + c] : 0.f;
    }
    __syncthreads();
    if (warp == 0) {  // lane r owns row r of the diagonal block
      for (int c = 0; c < nb; ++c) {
        const float p = s_diag[c][c];
        if (!(p > 0.f)) {  // the same value in every lane
          if (lane == 0) s_bad = 1;
          break;
        }
        const float piv = sqrtf(p);
        __syncwarp();
        if (lane == c) s_diag[c][c] = piv;
        if (lane > c && lane < nb) s_diag[lane][c] /= piv;
        __syncwarp();
        if (lane > c && lane < nb) {
          const float lrc = s_diag[lane][c];
          for (int c2 = c + 1; c2 <= lane; ++c2) s_diag[lane][c2] = fmaf(-lrc, s_diag[c2][c], s_diag[lane][c2]);
        }
        __syncwarp();
      }
      if (lane < nb)
        for (int c = 0; c <= lane; ++c) Mg[static_cast<long long>(J + lane) * k + J + c] = s_diag[lane][c];
    }
    __syncthreads();
    if (s_bad) break;  // the same value in every thread after the barrier
    const int t = k - J - nb;  // rows below the diagonal block (nb = kCholNb whenever t > 0)
    for (int ii = tid; ii < t; ii += kRidgeSolveThreads) {  // x L_JJ^T = M[i, J:J+32], x kept in the panel
      float* row = Mg + static_cast<long long>(J + nb + ii) * k + J;
      float* x = s_panel + ii * kCholLd;
      for (int c = 0; c < kCholNb; ++c) {
        float v = row[c];
        for (int c2 = 0; c2 < c; ++c2) v = fmaf(-x[c2], s_diag[c][c2], v);
        v /= s_diag[c][c];
        x[c] = v;
        row[c] = v;
      }
    }
    __syncthreads();
    for (int ii = warp; ii < t; ii += kWarps) {  // trailing lower triangle
      const float* pi = s_panel + ii * kCholLd;
      float* row = Mg + static_cast<long long>(J + nb + ii) * k + J + nb;
      for (int cc = lane; cc <= ii; cc += 32) {
        const float* pc = s_panel + cc * kCholLd;
        float acc = 0.f;
#pragma unroll 8
        for (int q = 0; q < kCholNb; ++q) acc = fmaf(pi[q], pc[q], acc);
        row[cc] -= acc;
      }
    }
    __syncthreads();
  }
  if (s_bad) {
    if (tid == 0) record_error(KVS_ERR_RANGE);
    for (long long e = tid; e < static_cast<long long>(k) * d; e += kRidgeSolveThreads) Vg[e] = 0.f;
    return;
  }

  // ---- L y = A^T Y (in B), then L^T x = y (into Vc) ----
  for (int pass = 0; pass < 2; ++pass) {
    const bool fwd = pass == 0;
    const float* src = Bg;
    float* dst = fwd ? Bg : Vg;
    for (int jb = 0; jb < k; jb += kCholNb) {
      const int J = fwd ? jb : ((k - 1) / kCholNb) * kCholNb - jb;
      const int nb = min(kCholNb, k - J);
      for (int e = tid; e < kCholNb * kCholNb; e += kRidgeSolveThreads) {
        const int r = e / kCholNb, c = e % kCholNb;
        s_diag[r][c] = (r < nb && c <= r) ? Mg[static_cast<long long>(J + r) * k + J + c] : (r == c ? 1.f : 0.f);
      }
      for (int r = warp; r < nb; r += kWarps) {  // row J + r minus its product with the solved rows
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int p0 = fwd ? 0 : J + nb, p1 = fwd ? J : k;
        for (int p = p0; p < p1; ++p) {
          const float l = fwd ? Mg[static_cast<long long>(J + r) * k + p] : Mg[static_cast<long long>(p) * k + J + r];
          const float* xp = dst + static_cast<long long>(p) * d + lane;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (u < nd) acc[u] = fmaf(l, xp[32 * u], acc[u]);
        }
        float* out = dst + static_cast<long long>(J + r) * d + lane;
        const float* in = src + static_cast<long long>(J + r) * d + lane;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (u < nd) out[32 * u] = in[32 * u] - acc[u];
      }
      __syncthreads();
      if (tid < d) {  // the 32 x 32 triangle for channel tid, through shared memory
        float* y = s_y + tid;  // y[r * kRidgeMaxD]
        for (int r = 0; r < nb; ++r) y[r * kRidgeMaxD] = dst[static_cast<long long>(J + r) * d + tid];
        if (fwd) {
          for (int r = 0; r < nb; ++r) {
            float v = y[r * kRidgeMaxD];
            for (int r2 = 0; r2 < r; ++r2) v = fmaf(-s_diag[r][r2], y[r2 * kRidgeMaxD], v);
            y[r * kRidgeMaxD] = v / s_diag[r][r];
          }
        } else {
          for (int r = nb - 1; r >= 0; --r) {
            float v = y[r * kRidgeMaxD];
            for (int r2 = r + 1; r2 < nb; ++r2) v = fmaf(-s_diag[r2][r], y[r2 * kRidgeMaxD], v);
            y[r * kRidgeMaxD] = v / s_diag[r][r];
          }
        }
        for (int r = 0; r < nb; ++r) dst[static_cast<long long>(J + r) * d + tid] = y[r * kRidgeMaxD];
      }
      __syncthreads();
    }
  }
}

}  // namespace kvs
