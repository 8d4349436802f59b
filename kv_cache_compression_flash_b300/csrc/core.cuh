// KV-CoRE: the data-dependent low-rank compressibility of a KV cache
// [KV-CoRE §2].  Per KV head, the covariance (Gram) matrix G = sum_t x_t x_t^T
// is accumulated over the tokens, its eigenvalues give the singular values of
// the cache (sigma_i = sqrt(lambda_i)), and the normalised effective rank
// (NER) summarises how few of them dominate.
//
//   gram_partial_kernel  grid (n_split, Hkv), 256 threads: each CTA owns a
//                        token range.  A 128-token tile of X [tokens x 128
//                        channels] is read with 16-byte loads, transposed in
//                        registers (8 x 8 bf16 blocks) and stored as X^T in the
//                        K-major 128-byte-swizzle layout; both MMA operands are
//                        that one tile, so tcgen05.mma (M = N = 128, K = 16,
//                        bf16 products exact in fp32) accumulates X^T X in TMEM
//                        (even and odd tiles in two accumulators, added at the
//                        end: half the sequential fp32 additions).
//                        Two tile buffers: the next tile is transposed while
//                        the tensor core consumes the previous one.
//   gram_reduce_kernel   adds the per-range partials in range order
//                        (deterministic) into G, optionally onto its contents
//                        (incremental accumulation over token blocks).
//   spectrum_kernel      one CTA per head: cyclic Jacobi on the symmetric
//                        128 x 128 G in fp32 (the circle method pairs all 128
//                        indices each round; 64 disjoint rotations per round),
//                        then sigma sorted descending, the numerical rank and
//                        the NER.
#pragma once

#include "common.cuh"

namespace kvs {

constexpr int kGramThreads = 256;
constexpr int kGramD = 128;
constexpr int kGramTile = 128;                   // tokens per tile (two 64-token K panels)
constexpr int kGramTileBytes = 2 * 16384;        // X^T tile: 128 rows x 128 tokens bf16
// two tile buffers, alignment slack and the control block, padded so that at
// most two CTAs share an SM: two CTAs take all 512 TMEM columns
constexpr int kGramSmem = 80 * 1024;
static_assert(2 * kGramTileBytes + 1024 + 64 <= kGramSmem, "gram shared memory");

struct GramCtl {
  uint64_t mma_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// byte offset of (row r, 16-byte chunk c) in a K-major 128-byte-swizzle panel
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Rows t of head g are X + g * head_stride + t * ld (ld = 128 and head_stride
// = N * 128 for a [heads, N, 128] cache; for the output projection W_O [D,
// Hq * 128], head h's column slice has ld = Hq * 128 and head_stride = 128).
__global__ void __launch_bounds__(kGramThreads) gram_partial_kernel(const uint16_t* __restrict__ X, int N,
                                                                    const long long ld, const long long head_stride,
                                                                    const uint8_t* __restrict__ keep,
                                                                    int tokens_per_cta, float* __restrict__ part) {
  extern __shared__ uint8_t gsm_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  GramCtl& S = *reinterpret_cast<GramCtl*>(base + 2 * kGramTileBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x, g = blockIdx.y, Hkv = gridDim.y;
  const long long t_lo = static_cast<long long>(s) * tokens_per_cta;
  const long long t_hi = t_lo + tokens_per_cta < N ? t_lo + tokens_per_cta : N;
  const int ntiles = t_hi > t_lo ? static_cast<int>((t_hi - t_lo + kGramTile - 1) / kGramTile) : 0;
  float* P = part + (static_cast<long long>(s) * Hkv + g) * kGramD * kGramD;

  if (tid == 0) {
    mbar_init(&S.mma_done[0], 1);
    mbar_init(&S.mma_done[1], 1);
    mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, 256);                 // two accumulators: even and odd tiles
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;
  const uint32_t sbase = smem_u32(base);
  const int to = tid >> 4, co = tid & 15;          // this thread's 8 x 8 block: tokens 8*to.., channels 8*co..
  const uint16_t* Xg = X + static_cast<long long>(g) * head_stride;
  const uint8_t* kg = keep ? keep + static_cast<long long>(g) * N : nullptr;

  // this thread's 8 rows of tile i (16 bytes each); zeros past the range and for dropped tokens
  auto load_tile = [&](int i, uint4 (&row)[8]) {
    const long long t0 = t_lo + static_cast<long long>(i) * kGramTile + 8 * to;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const long long t = t0 + r;
      const bool live = t < t_hi && (!kg || kg[t] != 0);
      row[r] = live ? __ldg(reinterpret_cast<const uint4*>(Xg + t * ld + 8 * co)) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  uint4 nxt[8];
  if (ntiles > 0) load_tile(0, nxt);
  bool ok = true;
  for (int i = 0; i < ntiles && ok; ++i) {
    const int b = i & 1;
    // tile i is in registers; the loads of tile i + 1 go out before it is used
    uint4 row[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) row[r] = nxt[r];
    if (i + 1 < ntiles) load_tile(i + 1, nxt);
    const bool free_ok = i < 2 || mbar_wait(&S.mma_done[b], ((i >> 1) - 1) & 1, abort_flag);
    if (!__syncthreads_and(free_ok)) {            // a bounded wait ran out: every thread stops here
      ok = false;
      break;
    }
    tc_fence_after();
    // transpose: output row j (channel 8*co + j) holds tokens 8*to .. 8*to+7
    const uint32_t w[8][4] = {{row[0].x, row[0].y, row[0].z, row[0].w}, {row[1].x, row[1].y, row[1].z, row[1].w},
                              {row[2].x, row[2].y, row[2].z, row[2].w}, {row[3].x, row[3].y, row[3].z, row[3].w},
                              {row[4].x, row[4].y, row[4].z, row[4].w}, {row[5].x, row[5].y, row[5].z, row[5].w},
                              {row[6].x, row[6].y, row[6].z, row[6].w}, {row[7].x, row[7].y, row[7].z, row[7].w}};
    uint8_t* buf = base + b * kGramTileBytes + (to >> 3) * 16384;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
      uint4 o;
      o.x = __byte_perm(w[0][j >> 1], w[1][j >> 1], sel);
      o.y = __byte_perm(w[2][j >> 1], w[3][j >> 1], sel);
      o.z = __byte_perm(w[4][j >> 1], w[5][j >> 1], sel);
      o.w = __byte_perm(w[6][j >> 1], w[7][j >> 1], sel);
      *reinterpret_cast<uint4*>(buf + sw128_off(8 * co + j, to & 7)) = o;
    }
    fence_async_shared();                          // the stores above become visible to the tensor core
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      const uint32_t a = sbase + b * kGramTileBytes;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * 16384u + (kk & 3) * 32u;
        umma_bf16(tmem + 128u * b, sdesc_kmajor_sw128(a + off), sdesc_kmajor_sw128(a + off), idesc,
                  (i > 1 || kk > 0) ? 1u : 0u);
      }
      umma_commit(&S.mma_done[b]);
    }
  }
  // every MMA this CTA issued has finished before TMEM is read or freed
  if (tid == 0 && ntiles > 0) umma_commit(&S.drain);
  __syncthreads();
  if (ntiles > 0) mbar_wait(&S.drain, 0, abort_flag);
  __syncthreads();
  const bool have = ntiles > 0 && ok && !S.abort_flag;
  tc_fence_after();
  if (warp < 4) {
    const int rrow = 32 * warp + lane;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v[32], v2[32];
      if (have) {
        tmem_load32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 32 * c, v);
        if (ntiles > 1) {
          tmem_load32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 128 + 32 * c, v2);
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] += v2[k];
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = 0.f;
      }
      float4* dst = reinterpret_cast<float4*>(P + rrow * kGramD + 32 * c);
#pragma unroll
      for (int k = 0; k < 8; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    }
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// G (+)= sum over ranges of the partials, in range order
__global__ void __launch_bounds__(256) gram_reduce_kernel(const float* __restrict__ part, int n_split,
                                                          long long per_split, int accumulate, float* __restrict__ G) {
  pdl_wait();
  const long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (i >= per_split) return;
  float acc = accumulate ? G[i] : 0.f;
  for (int s = 0; s < n_split; ++s) acc += part[s * per_split + i];
  G[i] = acc;
}

// ---------------------------------------------------------------------------
// spectrum: one CTA of 256 threads per head, G in shared memory (row pitch 129)
// ---------------------------------------------------------------------------
constexpr int kSpecThreads = 1024;
constexpr int kSpecPitch = kGramD + 1;
constexpr int kSpecMaxSweeps = 24;
constexpr size_t kSpecSmem = static_cast<size_t>(kGramD) * kSpecPitch * 4 + 64 * 4 * 4 + 32 * 4 + 64;

__global__ void __launch_bounds__(kSpecThreads) spectrum_kernel(const float* __restrict__ G, float rtol,
                                                                float* __restrict__ sigma, float* __restrict__ ner,
                                                                int* __restrict__ rank) {
  extern __shared__ float ssm[];
  float* A = ssm;                                    // [128][129]
  float* cs = A + kGramD * kSpecPitch;               // c[64], s[64]
  int* pq = reinterpret_cast<int*>(cs + 128);        // p[64], q[64]
  float* red = cs + 256;                             // [32]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.x;
  const float* Gg = G + static_cast<long long>(g) * kGramD * kGramD;
  pdl_wait();
  for (int i = tid; i < kGramD * kGramD; i += kSpecThreads) {
    const int r = i / kGramD, c = i % kGramD;
    A[r * kSpecPitch + c] = 0.5f * (Gg[r * kGramD + c] + Gg[c * kGramD + r]);   // exact symmetry
  }
  __syncthreads();
  auto block_sum = [&](float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kSpecThreads / 32; ++w) t += red[w];
    return t;
  };
  float fro = 0.f;
  for (int i = tid; i < kGramD * kGramD; i += kSpecThreads) {
    const float a = A[(i / kGramD) * kSpecPitch + i % kGramD];
    fro += a * a;
  }
  fro = block_sum(fro);
  float prev_off = INFINITY;
  for (int sweep = 0; sweep < kSpecMaxSweeps; ++sweep) {
    float off = 0.f;
    for (int i = tid; i < kGramD * kGramD; i += kSpecThreads) {
      const int r = i / kGramD, c = i % kGramD;
      if (r != c) off += A[r * kSpecPitch + c] * A[r * kSpecPitch + c];
    }
    off = block_sum(off);
    // converged (off-diagonal norm below 1e-5 |G|_F), an all-zero matrix, or,
    // after the first sweeps, no longer halving (the fp32 rounding floor)
    if (!(off > 1e-10f * fro) || (sweep >= 4 && !(off < 0.5f * prev_off))) break;
    prev_off = off;
    for (int round = 0; round < kGramD - 1; ++round) {
      if (tid < 64) {
        // circle method: index 127 is fixed, the others turn one place per round
        int p, q;
        if (tid == 0) {
          p = round;
          q = kGramD - 1;
        } else {
          p = (round + tid) % (kGramD - 1);
          q = (round - tid + (kGramD - 1)) % (kGramD - 1);
        }
        if (p > q) {
          const int t = p;
          p = q;
          q = t;
        }
        const float app = A[p * kSpecPitch + p], aqq = A[q * kSpecPitch + q], apq = A[p * kSpecPitch + q];
        float c = 1.f, sn = 0.f;
        if (fabsf(apq) > 1e-30f) {
          const float theta = (aqq - app) / (2.f * apq);
          const float t = copysignf(1.f, theta) / (fabsf(theta) + sqrtf(theta * theta + 1.f));
          c = rsqrtf(t * t + 1.f);
          sn = t * c;
        }
        cs[tid] = c;
        cs[64 + tid] = sn;
        pq[tid] = p;
        pq[64 + tid] = q;
      }
      __syncthreads();
      // rows: A <- P^T A
      for (int i = tid; i < 64 * kGramD; i += kSpecThreads) {
        const int k = i / kGramD, col = i % kGramD;
        const int p = pq[k], q = pq[64 + k];
        const float c = cs[k], sn = cs[64 + k];
        const float ap = A[p * kSpecPitch + col], aq = A[q * kSpecPitch + col];
        A[p * kSpecPitch + col] = c * ap - sn * aq;
        A[q * kSpecPitch + col] = sn * ap + c * aq;
      }
      __syncthreads();
      // columns: A <- A P
      for (int i = tid; i < 64 * kGramD; i += kSpecThreads) {
        const int k = i % 64, rr = i / 64;
        const int p = pq[k], q = pq[64 + k];
        const float c = cs[k], sn = cs[64 + k];
        const float ap = A[rr * kSpecPitch + p], aq = A[rr * kSpecPitch + q];
        A[rr * kSpecPitch + p] = c * ap - sn * aq;
        A[rr * kSpecPitch + q] = sn * ap + c * aq;
      }
      __syncthreads();
    }
  }
  // sigma = sqrt(max(lambda, 0)), sorted descending (bitonic sort of 128 values)
  float* sv = cs;                                    // reuse: 128 floats
  if (tid < kGramD) sv[tid] = sqrtf(fmaxf(A[tid * kSpecPitch + tid], 0.f));
  __syncthreads();
  for (int k = 2; k <= kGramD; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (tid < kGramD) {
        const int ixj = tid ^ j;
        if (ixj > tid) {
          const float a = sv[tid], b = sv[ixj];
          const bool desc = (tid & k) == 0;
          if (desc ? (a < b) : (a > b)) {
            sv[tid] = b;
            sv[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  const float smax = sv[0];
  const float x = tid < kGramD ? sv[tid] : 0.f;
  const bool in_rank = tid < kGramD && smax > 0.f && x > rtol * smax;
  const float r = block_sum(in_rank ? 1.f : 0.f);
  const float ssum = block_sum(in_rank ? x : 0.f);
  float h = 0.f;
  if (in_rank) {
    const float p = x / ssum;
    h = -p * logf(p);
  }
  h = block_sum(h);
  if (tid < kGramD) sigma[static_cast<long long>(g) * kGramD + tid] = x;
  if (tid == 0) {
    const int ri = static_cast<int>(r + 0.5f);
    rank[g] = ri;
    ner[g] = ri > 0 ? expf(h) / static_cast<float>(ri) : 0.f;
  }
}

}  // namespace kvs
