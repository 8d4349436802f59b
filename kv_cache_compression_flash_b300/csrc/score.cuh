// Attention-derived importance scores of a prefilled KV cache.
//
//   pass 1 (lse_pass_kernel):  lse_r = ln sum_{t<=p_r} exp(s_{r,t})
//       [KVSculpt: KV Cache Compression as Distillation, §2 loss, LSE term]
//   pass 2 (colreduce_pass_kernel), probabilities recomputed as a = exp(s - lse):
//       sum mode:  w_t = sum over the group's heads and rows of a_{r,t}
//                  [RDKV, §2.1, token distortion weight w_t = sum_tau a_{tau,t}]
//       max mode:  s_t = max_heads max_r a_{r,t} |h_r| / |W_O^h v_t|
//                  [KVzap, §2.1, KVzip and KVzip+ scores]
//
// Both passes are flash-style: 128x128 logit tiles S = Q K^T are produced by
// tcgen05.mma into tensor memory (fp32) from 128-byte-swizzled bf16 tiles that
// TMA streams into shared memory; the N x N matrix never exists in HBM.
// Reducer warp w reads TMEM lanes 32(w%4)..+31 (one tile row per thread), all
// 128 columns of a tile in four 32-column chunks whose loads overlap the
// previous chunk's arithmetic (packed fp32x2 FMA/ADD, ex2 on the
// special-function unit).  The reducer warps form two groups that take
// alternate tiles (ping-pong), so one group's TMEM loads and barrier waits
// overlap the other's arithmetic, and two TMEM buffers let the MMA of the next
// tile run meanwhile.  Both passes run one persistent CTA per SM: 16 reducer
// warps, TMA warp 16, MMA warp 17.
//
// GQA packing: a 128-row query tile holds P = 128/Gt consecutive window rows
// of Gt heads of one KV group (row j = head (j / P), position pmin + j % P), so
// every K tile that TMA brings in serves Gt heads at once.
//
// Pass 1 is Q-stationary (one tile of query rows per CTA, looping over key
// tiles, online max / sum in the log2 domain).  Pass 2 is K-stationary
// (S^T = K Q^T: one tile of keys per CTA looping over query tiles) so the
// per-key reduction over queries is a per-thread reduction along the TMEM
// row: no shuffles or atomics.  Long loops are split across CTAs and merged in
// a fixed order by small finalize kernels, so results are deterministic.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace kvs {

constexpr int kScoreThreads1 = 576;  // pass 1: 16 reducer warps (two row tiles), 1 TMA warp, 1 MMA warp
constexpr int kTmaWarp1 = 16, kMmaWarp1 = 17;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

struct ScoreGeom {
  int Hq, Hkv, G, Gt, P, W, N, q_pos0;
  int pos_cap;  // N - 1: a query at a later position sees every key (a block of keys before the queries)
  int n_hc;   // G / Gt head chunks per group
  int n_pb;   // ceil(W / P) position blocks
  int n_rt;   // Hkv * n_hc * n_pb query-row tiles
  int n_kt;   // ceil(N / 128) key tiles
  float c_log2;  // log2(e) / sqrt(d)
};

__host__ __device__ inline int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

// last position of position block pb, and the key tiles it needs
__host__ __device__ inline int pb_pmax(const ScoreGeom& g, int pb) {
  int r1 = (pb + 1) * g.P;
  if (r1 > g.W) r1 = g.W;
  const int p = g.q_pos0 + r1 - 1;
  return p < g.pos_cap ? p : g.pos_cap;
}
__host__ __device__ inline int pb_nkt(const ScoreGeom& g, int pb) { return pb_pmax(g, pb) / 128 + 1; }

// first position block that any key of key tile kt is visible to
__host__ __device__ inline int kt_pb_lo(const ScoreGeom& g, int kt) {
  const int t0 = kt * 128;
  const int num = t0 - g.q_pos0 - g.P + 1;
  return num <= 0 ? 0 : ceil_div_i(num, g.P);
}
__host__ __device__ inline int kt_nvis(const ScoreGeom& g, int kt) {
  const int t0 = kt * 128;
  if (t0 > g.q_pos0 + g.W - 1) return 0;
  const int lo = kt_pb_lo(g, kt);
  return lo < g.n_pb ? g.n_pb - lo : 0;
}

template <int DH>
struct TileCfg {
  static constexpr int kPanels = DH / 64;           // 64-column (128-byte) panels per row
  static constexpr int kTileBytes = kPanels * 16384;  // 128 rows x DH bf16
  static constexpr int kKSteps = DH / 16;           // MMA K=16 steps
};

template <int DH>
__device__ __forceinline__ void issue_tile_mma(uint32_t d_tmem, uint32_t a_base, uint32_t b_base) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
#pragma unroll
  for (int kk = 0; kk < TileCfg<DH>::kKSteps; ++kk) {
    const uint32_t off = (kk >> 2) * 16384u + (kk & 3) * 32u;
    umma_bf16(d_tmem, sdesc_kmajor_sw128(a_base + off), sdesc_kmajor_sw128(b_base + off), idesc,
              kk > 0 ? 1u : 0u);
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// ---------------------------------------------------------------------------
// pass 1: row log-sum-exp
// ---------------------------------------------------------------------------
template <int DH, int NS>
struct LseSmem {
  uint8_t q[2][2][TileCfg<DH>::kTileBytes];  // [item parity][row tile]
  uint8_t k[NS][TileCfg<DH>::kTileBytes];
  uint64_t q_full[2], q_empty[2], k_full[NS], k_empty[NS], s_full[2], s_empty[2], drain;
  uint32_t tmem_base;
  int abort_flag;
};

// partial[((rt * n_split + split) * 2 + group) * 128 + row] = (running max m,
// sum l), log2 domain: the row's 2^(x - m) summed over the split's key tiles
// that reducer group `group` took (even or odd ones), x = s * log2(e)/sqrt(d).

// one 32-column chunk of a pass-1 row: mask (diagonal tiles), running max and
// rescaled sum
__device__ __forceinline__ void lse_chunk(uint32_t (&r)[32], const int t0, const int pos, const bool diag,
                                          const float c, float& m, float& l) {
  float* v = reinterpret_cast<float*>(r);
  if (diag) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (t0 + j > pos) v[j] = -INFINITY;
  }
  float x[11];
#pragma unroll
  for (int k = 0; k < 10; ++k) x[k] = fmax3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
  x[10] = fmaxf(v[30], v[31]);
  const float y0 = fmax3(x[0], x[1], x[2]), y1 = fmax3(x[3], x[4], x[5]), y2 = fmax3(x[6], x[7], x[8]);
  const float z = fmax3(fmax3(y0, y1, y2), x[9], x[10]);
  const float m_new = fmaxf(m, z * c);
  if (m_new == -INFINITY) return;  // every element so far masked
  const unsigned long long c2 = f2_pack(c, c), nm2 = f2_pack(-m_new, -m_new);
  unsigned long long acc0 = 0ull, acc1 = 0ull;  // two packed pairs of partial sums
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    float e0, e1, e2, e3;
    f2_unpack(f2_fma(f2_pack(v[j], v[j + 1]), c2, nm2), &e0, &e1);
    f2_unpack(f2_fma(f2_pack(v[j + 2], v[j + 3]), c2, nm2), &e2, &e3);
    acc0 = f2_add(acc0, f2_pack(ex2_approx(e0), ex2_approx(e1)));
    acc1 = f2_add(acc1, f2_pack(ex2_approx(e2), ex2_approx(e3)));
  }
  float s0, s1;
  f2_unpack(f2_add(acc0, acc1), &s0, &s1);
  l = l * ex2_approx(m - m_new) + (s0 + s1);
  m = m_new;
}

// Persistent CTAs (one per SM) walk work items it = blockIdx.x, + gridDim.x, ...;
// item (pair, split) = TWO row tiles (position blocks 2pp, 2pp+1 of a head
// chunk) over key tiles [split * kt_chunk, ..).  Every K tile TMA brings in
// feeds two MMAs (M = 256 in effect), halving the L2 -> shared-memory traffic
// per flop; the pipeline (TMA ring, two double-buffered TMEM accumulator
// pairs, the next item's row tiles) runs on across items.  Reducer warps 0-7
// take the even K tiles and warps 8-15 the odd ones (ping-pong: one group's
// TMEM loads overlap the other's arithmetic); within a group, warps 0-3 and
// 4-7 take row tiles 0 and 1, one tile row (all 128 columns) per thread.
// Warp 16 issues TMA, warp 17 the MMAs.
struct LseItem {
  int pb0, g, hc, gh, kt0, kt1, split;
  bool two;
};

// it = split * (pairs * heads) + jy: the split index varies slowest, so the
// persistent CTAs' strided item sequences do not line up with the short last
// chunks
__device__ __forceinline__ bool lse_item(const ScoreGeom& geo, const int kt_chunk, const int n_split, const int it,
                                         LseItem* x) {
  const int n_pp = (geo.n_pb + 1) / 2;
  const int n_jy = n_pp * geo.Hkv * geo.n_hc;
  const int jy = it % n_jy, split = it / n_jy;
  x->split = split;
  const int pp = n_pp - 1 - (jy % n_pp);  // longest rows first
  x->gh = jy / n_pp;
  x->g = x->gh / geo.n_hc;
  x->hc = x->gh % geo.n_hc;
  x->pb0 = 2 * pp;
  x->two = 2 * pp + 1 < geo.n_pb;
  x->kt0 = split * kt_chunk;
  x->kt1 = min(pb_nkt(geo, x->two ? x->pb0 + 1 : x->pb0), x->kt0 + kt_chunk);
  return x->kt0 < x->kt1;
}

template <int DH, int NS>
__global__ void __launch_bounds__(kScoreThreads1, 1)
    lse_pass_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                    const ScoreGeom geo, const int kt_chunk, const int n_split, const int n_items,
                    float2* __restrict__ partial) {
  extern __shared__ uint8_t smem_raw[];
  LseSmem<DH, NS>& S = *reinterpret_cast<LseSmem<DH, NS>*>(align1024(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (timeout_recorded()) return;  // uniform over the CTA, before any barrier

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.q_full[b], 1);
      mbar_init(&S.q_empty[b], 1);
      mbar_init(&S.s_full[b], 1);
      mbar_init(&S.s_empty[b], 8);  // the 8 warps of the group that owns buffer b
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&S.k_full[s], 1);
      mbar_init(&S.k_empty[s], 1);
    }
    mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // Q, K and the offsets may come from the previous kernel on the stream
  pdl_trigger();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;

  if (warp == kTmaWarp1) {
    if (lane == 0) {  // TMA producer
      prefetch_tensormap(&mapQ);
      prefetch_tensormap(&mapK);
      constexpr uint32_t kBytes = TileCfg<DH>::kTileBytes;
      int n_it = 0, kc = 0, issued = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        LseItem x;
        if (!lse_item(geo, kt_chunk, n_split, it, &x)) continue;
        const int qb = n_it & 1;
        if (!mbar_wait(&S.q_empty[qb], ((n_it >> 1) & 1) ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(&S.q_full[qb], 2 * kBytes);
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int p = 0; p < TileCfg<DH>::kPanels; ++p)  // a missing second tile reads as zeros
            tma_load_3d(S.q[qb][t] + p * 16384, &mapQ, &S.q_full[qb], p * 64, (x.pb0 + t) * geo.P,
                        x.g * geo.G + x.hc * geo.Gt);
        ++n_it;
        for (int kt = x.kt0; kt < x.kt1; ++kt, ++kc) {
          const int s = kc % NS;
          if (!mbar_wait(&S.k_empty[s], ((kc / NS) & 1) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&S.k_full[s], kBytes);
#pragma unroll
          for (int p = 0; p < TileCfg<DH>::kPanels; ++p)
            tma_load_3d(S.k[s] + p * 16384, &mapK, &S.k_full[s], p * 64, kt * 128, x.g);
          issued = kc + 1;
        }
      }
      if (*abort_flag) {  // let our copies land before the CTA goes away
        volatile int never = 0;
        for (int i = max(0, n_it - 2); i < n_it; ++i) mbar_wait(&S.q_full[i & 1], (i >> 1) & 1, &never);
        for (int i = max(0, issued - NS); i < issued; ++i) mbar_wait(&S.k_full[i % NS], (i / NS) & 1, &never);
      }
    }
  } else if (warp == kMmaWarp1) {
    if (lane == 0) {  // MMA issuer: two row tiles against each K tile
      int n_it = 0, kc = 0;
      bool ok = true;
      // test hook: withhold the first tile's arrive, so the reducers' bounded wait runs out
      const bool withhold = *reinterpret_cast<volatile int*>(&g_debug_fault) == KVS_DEBUG_WITHHOLD_LSE_ARRIVE;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        LseItem x;
        if (!lse_item(geo, kt_chunk, n_split, it, &x)) continue;
        const int qb = n_it & 1;
        if (!mbar_wait(&S.q_full[qb], (n_it >> 1) & 1, abort_flag)) break;
        ++n_it;
        for (int kt = x.kt0; kt < x.kt1; ++kt, ++kc) {
          const int s = kc % NS, b = kc & 1;
          if (!mbar_wait(&S.k_full[s], (kc / NS) & 1, abort_flag) ||
              !mbar_wait(&S.s_empty[b], ((kc >> 1) & 1) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_tile_mma<DH>(tmem + (2 * b) * 128, smem_u32(S.q[qb][0]), smem_u32(S.k[s]));
          if (x.two) issue_tile_mma<DH>(tmem + (2 * b + 1) * 128, smem_u32(S.q[qb][1]), smem_u32(S.k[s]));
          umma_commit(&S.k_empty[s]);
          if (!(withhold && kc == 0)) umma_commit(&S.s_full[b]);
        }
        if (ok) umma_commit(&S.q_empty[qb]);  // the item's row tiles are free once its MMAs finish
      }
      if (*abort_flag) {
        volatile int never = 0;
        umma_commit(&S.drain);
        mbar_wait(&S.drain, 0, &never);
      }
    }
  } else {  // warps 0-15: group warp / 8 takes the tiles of its parity (ping-pong), row tile (warp / 4) % 2
    const int grp = warp >> 3, t = (warp >> 2) & 1, q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const float c = geo.c_log2;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + t * 128;
    uint32_t va[32], vb[32];
    int kc = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      LseItem x;
      if (!lse_item(geo, kt_chunk, n_split, it, &x)) continue;
      const int p0 = geo.q_pos0 + (x.pb0 + t) * geo.P;
      const int pmin = min(p0, geo.pos_cap);
      const int pos = min(p0 + row % geo.P, geo.pos_cap);
      const bool active = t == 0 || x.two;
      float m = -INFINITY, l = 0.f;
      for (int kt = x.kt0; kt < x.kt1; ++kt, ++kc) {
        if ((kc & 1) != grp) continue;  // the other group's tile
        const int b = kc & 1;
        if (!mbar_wait(&S.s_full[b], (kc >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (active) {
          const int t0 = kt * 128;
          const bool diag = t0 + 127 > pmin;
          const uint32_t base = lane_base + b * 256;
          // four 32-column chunks; each chunk's load overlaps the previous chunk's arithmetic
          tmem_issue32(base, va);
          tmem_wait32(va);
          tmem_issue32(base + 32, vb);
          lse_chunk(va, t0, pos, diag, c, m, l);
          tmem_wait32(vb);
          tmem_issue32(base + 64, va);
          lse_chunk(vb, t0 + 32, pos, diag, c, m, l);
          tmem_wait32(va);
          tmem_issue32(base + 96, vb);
          lse_chunk(va, t0 + 64, pos, diag, c, m, l);
          tmem_wait32(vb);
          tc_fence_before();  // this warp is done with the TMEM buffer
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.s_empty[b]);
          lse_chunk(vb, t0 + 96, pos, diag, c, m, l);
        } else {  // no second row tile: only release the buffer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.s_empty[b]);
        }
      }
      if (ok && active) {
        const int rt = x.gh * geo.n_pb + x.pb0 + t;
        partial[((static_cast<size_t>(rt) * n_split + x.split) * 2 + grp) * 128 + row] = make_float2(m, l);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merges pass-1 partials in split order.  Writes lse (natural log) for the
// valid rows and, per query tile, the pass-2 offsets
//     b[rt][row] = lse2 - log2|h_r|   (|h_r| = 1 when hn is null; +inf for padding rows)
// so that pass 2 computes a_{r,t} |h_r| = 2^(s c - b).
__global__ void lse_finalize_kernel(const ScoreGeom geo, const int kt_chunk, const int n_split,
                                    const float2* __restrict__ partial, const float* __restrict__ hn,
                                    float* __restrict__ lse, float* __restrict__ b_plain,
                                    float* __restrict__ b_scaled) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  if (timeout_recorded()) return;  // the partials were never written: leave the outputs untouched
  const int rt = blockIdx.x, row = threadIdx.x;
  const int pb = rt % geo.n_pb;
  const int gh = rt / geo.n_pb;
  const int g = gh / geo.n_hc, hc = gh % geo.n_hc;
  const int ns = ceil_div_i(pb_nkt(geo, pb), kt_chunk);
  const float2* p = partial + static_cast<size_t>(rt) * n_split * 256 + row;
  float M = -INFINITY;
  for (int s = 0; s < 2 * ns; ++s) M = fmaxf(M, p[s * 128].x);
  float L = 0.f;
  for (int s = 0; s < 2 * ns; ++s) {
    const float2 v = p[s * 128];
    if (v.x != -INFINITY) L += v.y * ex2_approx(v.x - M);
  }
  const float l2 = M + lg2_approx(L);
  const int hl = row / geo.P, r = pb * geo.P + row % geo.P;
  const bool valid = r < geo.W && hl < geo.Gt;
  if (valid) lse[static_cast<size_t>(g * geo.G + hc * geo.Gt + hl) * geo.W + r] = l2 * kLn2;
  if (b_plain) b_plain[static_cast<size_t>(rt) * 128 + row] = valid ? l2 : INFINITY;
  if (b_scaled) b_scaled[static_cast<size_t>(rt) * 128 + row] = valid ? l2 - lg2_approx(hn[r]) : INFINITY;
}

// Pass-2 offsets from a given lse (natural log, [Hq, W]), same layout as above.
__global__ void lse_offsets_kernel(const ScoreGeom geo, const float* __restrict__ lse, const float* __restrict__ hn,
                                   float* __restrict__ b_plain, float* __restrict__ b_scaled) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  const int rt = blockIdx.x, row = threadIdx.x;
  const int pb = rt % geo.n_pb;
  const int gh = rt / geo.n_pb;
  const int g = gh / geo.n_hc, hc = gh % geo.n_hc;
  const int hl = row / geo.P, r = pb * geo.P + row % geo.P;
  const bool valid = r < geo.W && hl < geo.Gt;
  const float l2 = valid ? lse[static_cast<size_t>(g * geo.G + hc * geo.Gt + hl) * geo.W + r] * kLog2e : 0.f;
  if (b_plain) b_plain[static_cast<size_t>(rt) * 128 + row] = valid ? l2 : INFINITY;
  if (b_scaled) b_scaled[static_cast<size_t>(rt) * 128 + row] = valid ? l2 - lg2_approx(hn[r]) : INFINITY;
}

// ---------------------------------------------------------------------------
// pass 2: per-key reductions over queries (K-stationary, persistent)
// ---------------------------------------------------------------------------
// Persistent CTAs (one per SM, all 512 TMEM columns) walk work items
// it = blockIdx.x, + gridDim.x, ...; an item is a PAIR of key tiles (kt0,
// kt0 + 1) of KV head g and a range of the query tiles that see key tile kt0
// (head chunk major, position block minor).  Every query tile TMA brings in
// feeds two MMAs, S^T_j = K_j Q^T for both key tiles (M = 256 keys in
// effect), which halves the L2 -> shared-memory traffic per flop against one
// key tile per CTA: one 128x128 tile per 128x128x128 MMA would ask the L2 for
// more bytes per clock than it delivers.  Query tiles entirely before key tile
// kt0 + 1 skip its MMA.
// Reducer warp w: group hh = w / 8 takes the query tiles of its parity
// (ping-pong over the two TMEM buffer pairs), key tile j = (w / 4) % 2, TMEM
// lane quarter w % 4; each thread owns one key and reduces along its TMEM
// row.  At the end of an item the two groups' values of a key are combined in
// a fixed order (group 1 hands its value to group 0 through shared memory,
// ordered by an mbarrier pair: no named barrier, so a wait that gives up can
// never leave a warp stranded).  Warp 16 issues TMA, warp 17 the MMAs.
constexpr int kScoreThreads2 = 576;
constexpr int kTmaWarp2 = 16, kMmaWarp2 = 17;

template <int DH, int NS>
struct ColSmem {
  uint8_t k[2][TileCfg<DH>::kTileBytes];   // the item's two key tiles
  uint8_t q[NS][TileCfg<DH>::kTileBytes];  // query-tile ring
  float bv[NS][128];                       // the offsets that came with each query tile
  float comb[2][128];                      // group 1 -> group 0 hand-off, per key tile
  uint64_t k_full, k_empty, q_full[NS], q_empty[NS], s_full[2], s_empty[2], c_full, c_empty, drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct ColItem {
  int g, kt0, q0, q1, nvis, pb_lo, pb_lo1, split;
  bool two;
};

__host__ __device__ inline int col_pairs(const ScoreGeom& geo) { return (geo.n_kt + 1) / 2; }

// item it = split * (pairs * Hkv) + pair * Hkv + g: early pairs (the longest
// query lists) first within each split.  The split index varies slowest: the
// persistent CTAs take items it, it + gridDim.x, ..., and with the split
// fastest an even grid would hand every even CTA the long first chunks and
// every odd CTA the short last ones.
__device__ __forceinline__ bool col_item(const ScoreGeom& geo, const int qt_chunk, const int n_split, const int it,
                                         ColItem* x) {
  const int per_split = col_pairs(geo) * geo.Hkv;
  x->split = it / per_split;
  const int r = it % per_split;
  x->g = r % geo.Hkv;
  x->kt0 = 2 * (r / geo.Hkv);
  x->two = x->kt0 + 1 < geo.n_kt;
  x->nvis = kt_nvis(geo, x->kt0);
  x->pb_lo = geo.n_pb - x->nvis;
  x->pb_lo1 = x->two ? geo.n_pb - kt_nvis(geo, x->kt0 + 1) : geo.n_pb;  // first block key tile kt0+1 sees
  const int nq = x->nvis * geo.n_hc;
  x->q0 = x->split * qt_chunk;
  x->q1 = min(nq, x->q0 + qt_chunk);
  return x->q0 < x->q1;
}

// MAXMODE = false: out = sum_j 2^(s_j c - b_j)                            (w_t)
// MAXMODE = true : out = max_heads 2^(max_j (s_j c - b_j)) / vn[head][t]   (vn null: / 1)
// Output goes to out_direct (n_split == 1) or out_partial[split][g*N + t].
template <int DH, int NS, int GT, bool MAXMODE>
__global__ void __launch_bounds__(kScoreThreads2, 1)
    colreduce_pass_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                          const ScoreGeom geo, const int qt_chunk, const int n_split, const int n_items,
                          const float* __restrict__ bvals, const float* __restrict__ vn,
                          float* __restrict__ out_direct, float* __restrict__ out_partial) {
  constexpr int P = 128 / GT;
  extern __shared__ uint8_t smem_raw[];
  ColSmem<DH, NS>& S = *reinterpret_cast<ColSmem<DH, NS>*>(align1024(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (timeout_recorded()) return;  // uniform over the CTA, before any barrier

  if (threadIdx.x == 0) {
    mbar_init(&S.k_full, 1);
    mbar_init(&S.k_empty, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&S.q_full[s], 1);
      mbar_init(&S.q_empty[s], 1 + 8);  // the MMAs, and the 8 warps that read the staged offsets
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.s_full[b], 1);
      mbar_init(&S.s_empty[b], 8);      // the 8 warps of the group that owns buffer pair b
    }
    mbar_init(&S.c_full, 8);
    mbar_init(&S.c_empty, 8);
    mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // Q, K and the offsets may come from the previous kernel on the stream
  pdl_trigger();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;

  if (warp == kTmaWarp2) {
    if (lane == 0) {  // TMA producer
      prefetch_tensormap(&mapQ);
      prefetch_tensormap(&mapK);
      constexpr uint32_t kBytes = TileCfg<DH>::kTileBytes;
      int n_it = 0, qc = 0, issued = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        ColItem x;
        if (!col_item(geo, qt_chunk, n_split, it, &x)) continue;
        // the key tiles: one buffer, free once the previous item's MMAs are done
        if (!mbar_wait(&S.k_empty, (n_it & 1) ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(&S.k_full, 2 * kBytes);
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int p = 0; p < TileCfg<DH>::kPanels; ++p)  // a tile past the last key reads as zeros
            tma_load_3d(S.k[t] + p * 16384, &mapK, &S.k_full, p * 64, (x.kt0 + t) * 128, x.g);
        ++n_it;
        for (int q = x.q0; q < x.q1; ++q, ++qc) {
          const int s = qc % NS;
          if (!mbar_wait(&S.q_empty[s], ((qc / NS) & 1) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const int hc = q / x.nvis, pb = x.pb_lo + q % x.nvis;
          const int rt = (x.g * geo.n_hc + hc) * geo.n_pb + pb;
          mbar_arrive_expect_tx(&S.q_full[s], kBytes + 512u);
#pragma unroll
          for (int p = 0; p < TileCfg<DH>::kPanels; ++p)
            tma_load_3d(S.q[s] + p * 16384, &mapQ, &S.q_full[s], p * 64, pb * P, x.g * geo.G + hc * GT);
          bulk_load(S.bv[s], bvals + static_cast<size_t>(rt) * 128, 512u, &S.q_full[s]);
          issued = qc + 1;
        }
      }
      if (*abort_flag) {  // let our copies land before the CTA goes away
        volatile int never = 0;
        if (n_it > 0) mbar_wait(&S.k_full, (n_it - 1) & 1, &never);
        for (int i = max(0, issued - NS); i < issued; ++i) mbar_wait(&S.q_full[i % NS], (i / NS) & 1, &never);
      }
    }
  } else if (warp == kMmaWarp2) {
    if (lane == 0) {  // MMA issuer: S^T_j = K_j (M = 128 keys) x Q_tile^T (N = 128 rows), j = 0, 1
      int n_it = 0, qc = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        ColItem x;
        if (!col_item(geo, qt_chunk, n_split, it, &x)) continue;
        if (!mbar_wait(&S.k_full, n_it & 1, abort_flag)) break;
        ++n_it;
        for (int q = x.q0; q < x.q1; ++q, ++qc) {
          const int s = qc % NS, b = qc & 1;
          if (!mbar_wait(&S.q_full[s], (qc / NS) & 1, abort_flag) ||
              !mbar_wait(&S.s_empty[b], ((qc >> 1) & 1) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int pb = x.pb_lo + q % x.nvis;
          issue_tile_mma<DH>(tmem + (2 * b) * 128, smem_u32(S.k[0]), smem_u32(S.q[s]));
          if (x.two && pb >= x.pb_lo1) issue_tile_mma<DH>(tmem + (2 * b + 1) * 128, smem_u32(S.k[1]), smem_u32(S.q[s]));
          umma_commit(&S.q_empty[s]);
          umma_commit(&S.s_full[b]);
        }
        if (ok) umma_commit(&S.k_empty);  // the key tiles are free once the item's MMAs finish
      }
      if (*abort_flag) {
        volatile int never = 0;
        umma_commit(&S.drain);
        mbar_wait(&S.drain, 0, &never);
      }
    }
  } else {  // warps 0-15: one key per thread (TMEM lane of key tile j); group hh takes the query tiles of its parity
    const int hh = warp >> 3, j = (warp >> 2) & 1, q4 = warp & 3;
    const int krow = q4 * 32 + lane;
    const float c = geo.c_log2;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + j * 128;
    uint32_t va[32], vb[32];
    int qc = 0, n_it = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      ColItem x;
      if (!col_item(geo, qt_chunk, n_split, it, &x)) continue;
      const int t0 = (x.kt0 + j) * 128;
      const int t = t0 + krow;
      float acc = 0.f, best = 0.f;
      float mx[GT];
#pragma unroll
      for (int h = 0; h < GT; ++h) mx[h] = -INFINITY;
      int cur_hc = -1;
      auto flush = [&](int hc) {
#pragma unroll
        for (int h = 0; h < GT; ++h) {
          if (mx[h] != -INFINITY && t < geo.N) {
            float r = ex2_approx(mx[h]);
            if (vn) r = r / vn[static_cast<size_t>(x.g * geo.G + hc * GT + h) * geo.N + t];
            best = fmaxf(best, r);
          }
          mx[h] = -INFINITY;
        }
      };
      // one 32-column chunk: x = s c - b_col, masked where the query precedes the key
      auto chunk = [&](uint32_t (&r)[32], const float* bcol, const int col0, const int pmin, const bool diag) {
        float* v = reinterpret_cast<float*>(r);
        const unsigned long long c2 = f2_pack(c, c);
        const float4* b4 = reinterpret_cast<const float4*>(bcol);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 bb = b4[j4];
          f2_unpack(f2_fma(f2_pack(v[4 * j4], v[4 * j4 + 1]), c2, f2_pack(-bb.x, -bb.y)), &v[4 * j4],
                    &v[4 * j4 + 1]);
          f2_unpack(f2_fma(f2_pack(v[4 * j4 + 2], v[4 * j4 + 3]), c2, f2_pack(-bb.z, -bb.w)), &v[4 * j4 + 2],
                    &v[4 * j4 + 3]);
        }
        if (diag) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (pmin + ((col0 + e) % P) < t) v[e] = -INFINITY;
        }
        if (MAXMODE) {
          float y[11];
#pragma unroll
          for (int k = 0; k < 10; ++k) y[k] = fmax3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
          y[10] = fmaxf(v[30], v[31]);
          const float z = fmax3(fmax3(fmax3(y[0], y[1], y[2]), fmax3(y[3], y[4], y[5]), fmax3(y[6], y[7], y[8])),
                                y[9], y[10]);
          const int hl = col0 / P;  // P >= 32: the chunk lies in one head
#pragma unroll
          for (int h = 0; h < GT; ++h)
            if (h == hl) mx[h] = fmaxf(mx[h], z);
        } else {
          unsigned long long a0 = 0ull, a1 = 0ull;
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            a0 = f2_add(a0, f2_pack(ex2_approx(v[e]), ex2_approx(v[e + 1])));
            a1 = f2_add(a1, f2_pack(ex2_approx(v[e + 2]), ex2_approx(v[e + 3])));
          }
          float s0, s1;
          f2_unpack(f2_add(a0, a1), &s0, &s1);
          acc += s0 + s1;
        }
      };
      for (int q = x.q0; q < x.q1; ++q, ++qc) {
        const int s = qc % NS, b = qc & 1;
        const int hc = q / x.nvis, pb = x.pb_lo + q % x.nvis;
        if (MAXMODE && hc != cur_hc) {
          if (cur_hc >= 0) flush(cur_hc);
          cur_hc = hc;
        }
        if ((qc & 1) != hh) continue;  // the other group's tile
        if (!mbar_wait(&S.s_full[b], (qc >> 1) & 1, abort_flag) ||
            !mbar_wait(&S.q_full[s], (qc / NS) & 1, abort_flag)) {  // the staged offsets arrived with the tile
          ok = false;
          break;
        }
        tc_fence_after();
        if (j == 0 || (x.two && pb >= x.pb_lo1)) {
          const int pmin = geo.q_pos0 + pb * P;
          const bool diag = pmin < t0 + 127;
          const uint32_t base = lane_base + b * 256;
          tmem_issue32(base, va);
          tmem_wait32(va);
          tmem_issue32(base + 32, vb);
          chunk(va, S.bv[s], 0, pmin, diag);
          tmem_wait32(vb);
          tmem_issue32(base + 64, va);
          chunk(vb, S.bv[s] + 32, 32, pmin, diag);
          tmem_wait32(va);
          tmem_issue32(base + 96, vb);
          chunk(va, S.bv[s] + 64, 64, pmin, diag);
          tmem_wait32(vb);
          tc_fence_before();  // this warp is done with the TMEM buffer
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.s_empty[b]);
          chunk(vb, S.bv[s] + 96, 96, pmin, diag);
        } else {  // key tile kt0+1 precedes every query of this tile: only release the buffer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.s_empty[b]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.q_empty[s]);  // done reading bv[s]
      }
      if (!ok) break;
      if (MAXMODE && cur_hc >= 0) flush(cur_hc);
      // the two groups' values of this key, combined in a fixed order
      const float mine = MAXMODE ? best : acc;
      if (hh == 1) {
        if (!mbar_wait(&S.c_empty, (n_it & 1) ^ 1u, abort_flag)) break;
        S.comb[j][krow] = mine;
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.c_full);
      } else {
        if (!mbar_wait(&S.c_full, n_it & 1, abort_flag)) break;
        const float other = S.comb[j][krow];
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.c_empty);
        const float res = MAXMODE ? fmaxf(mine, other) : mine + other;
        if (t < geo.N) {
          const size_t o = static_cast<size_t>(x.g) * geo.N + t;
          if (n_split == 1)
            out_direct[o] = res;
          else
            out_partial[static_cast<size_t>(x.split) * geo.Hkv * geo.N + o] = res;
        }
      }
      ++n_it;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Sums (or maxes) pass-2 partials over the key tile's splits, in split order.
template <bool MAXMODE>
__global__ void colreduce_finalize_kernel(const ScoreGeom geo, const int qt_chunk, const int n_split,
                                          const float* __restrict__ part, float* __restrict__ out) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  if (timeout_recorded()) return;  // the partials were never written: leave the outputs untouched
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  const int total = geo.Hkv * geo.N;
  if (idx >= total) return;
  const int t = idx % geo.N;
  // a key's splits are those of its key-tile pair, whose query list is the first tile's
  const int ns = ceil_div_i(kt_nvis(geo, (t / 128) & ~1) * geo.n_hc, qt_chunk);
  float r = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float v = part[static_cast<size_t>(s) * total + idx];
    r = MAXMODE ? fmaxf(r, v) : r + v;
  }
  out[idx] = r;
}

// ---------------------------------------------------------------------------
// KVzip+ norms   [KVzap §2.1: |h_j| and |W_O v_i|]
// ---------------------------------------------------------------------------
// out[r] = |X[r, :]|_2, one warp per row, 16-byte loads, fixed-order reduction
__global__ void row_norm_kernel(const uint16_t* __restrict__ X, const int rows, const int cols,
                                float* __restrict__ out) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  const int warps = blockDim.x >> 5;
  const int r = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const uint4* p = reinterpret_cast<const uint4*>(X + static_cast<size_t>(r) * cols);
  const int n16 = cols / 8;
  float acc = 0.f;
  for (int i = lane; i < n16; i += 32) {
    const uint4 u = __ldg(p + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xFFFF0000u);
      acc = fmaf(lo, lo, acc);
      acc = fmaf(hi, hi, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (lane == 0) out[r] = sqrtf(acc);
}

// Partial Gram matrices of the per-head output projections:
//   gram[s][h][c1][c2] = sum_{i in slice s} W_O[i, h*DH + c1] W_O[i, h*DH + c2]
// grid (n_slices, Hq, DH/64); 256 threads; each thread 4 x (DH/16) outputs.
template <int DH>
__global__ void __launch_bounds__(256) gram_kernel(const uint16_t* __restrict__ WO, const int D, const int Hq,
                                                   const int slice_len, float* __restrict__ gram) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  constexpr int CPT = DH / 16;
  __shared__ float T[32][DH + 4];
  const int s = blockIdx.x, h = blockIdx.y, c1b = blockIdx.z * 64;
  const int tid = threadIdx.x;
  const int r4 = (tid / 16) * 4, cg = (tid % 16) * CPT;
  float acc[4][CPT];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < CPT; ++b) acc[a][b] = 0.f;
  const int i_begin = s * slice_len, i_end = min(D, i_begin + slice_len);
  const size_t ld = static_cast<size_t>(Hq) * DH;
  for (int i0 = i_begin; i0 < i_end; i0 += 32) {
    for (int e = tid; e < 32 * DH; e += 256) {
      const int rr = e / DH, cc = e % DH;
      const int i = i0 + rr;
      float v = 0.f;
      if (i < i_end) v = __uint_as_float(static_cast<uint32_t>(WO[i * ld + h * DH + cc]) << 16);
      T[rr][cc] = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < 32; ++k) {
      float a[4], b[CPT];
#pragma unroll
      for (int x = 0; x < 4; ++x) a[x] = T[k][c1b + r4 + x];
#pragma unroll
      for (int y = 0; y < CPT; ++y) b[y] = T[k][cg + y];
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < CPT; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
    }
    __syncthreads();
  }
  float* out = gram + ((static_cast<size_t>(s) * Hq + h) * DH) * DH;
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < CPT; ++y) out[(c1b + r4 + x) * DH + cg + y] = acc[x][y];
}

// vn[h][t] = sqrt(v_t^T G_h v_t) = |W_O^h v_t|, G_h = sum of the Gram slices
// (fixed order).  grid (ceil(N/64), Hq); 256 threads: 16 token quads x 16 column groups.
template <int DH>
__global__ void __launch_bounds__(256) vnorm_kernel(const uint16_t* __restrict__ V,
                                                    const float* __restrict__ gram, const int n_slices,
                                                    const int Hq, const int G, const int N,
                                                    float* __restrict__ vn) {
  pdl_wait();  // inputs may come from the previous kernel on the stream
  pdl_trigger();
  constexpr int CPT = DH / 16;
  extern __shared__ uint8_t smem_raw[];
  float* Gs = reinterpret_cast<float*>(smem_raw);  // [DH][DH]
  float* Vs = Gs + DH * DH;                        // [DH][64] (transposed tile)
  const int h = blockIdx.y, t0 = blockIdx.x * 64, tid = threadIdx.x;
  const int g = h / G;
  for (int e = tid; e < DH * DH; e += 256) {
    float a = 0.f;
    for (int s = 0; s < n_slices; ++s) a += gram[(static_cast<size_t>(s) * Hq + h) * DH * DH + e];
    Gs[e] = a;
  }
  for (int e = tid; e < 64 * DH; e += 256) {
    const int tt = e / DH, cc = e % DH;
    const int t = t0 + tt;
    float v = 0.f;
    if (t < N) v = __uint_as_float(static_cast<uint32_t>(V[(static_cast<size_t>(g) * N + t) * DH + cc]) << 16);
    Vs[cc * 64 + tt] = v;
  }
  __syncthreads();
  const int tq = (tid / 16) * 4, cg = (tid % 16) * CPT;
  float acc[4][CPT];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < CPT; ++b) acc[a][b] = 0.f;
#pragma unroll 4
  for (int k = 0; k < DH; ++k) {
    const float4 a4 = *reinterpret_cast<const float4*>(&Vs[k * 64 + tq]);
    const float a[4] = {a4.x, a4.y, a4.z, a4.w};
    float b[CPT];
#pragma unroll
    for (int y = 0; y < CPT; ++y) b[y] = Gs[k * DH + cg + y];
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < CPT; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
  }
  float part[4];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    float p = 0.f;
#pragma unroll
    for (int y = 0; y < CPT; ++y) p = fmaf(acc[x][y], Vs[(cg + y) * 64 + tq + x], p);
    part[x] = p;
  }
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) part[x] += __shfl_xor_sync(0xFFFFFFFFu, part[x], o);
  if ((tid % 16) == 0) {
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int t = t0 + tq + x;
      if (t < N) vn[static_cast<size_t>(h) * N + t] = sqrtf(fmaxf(part[x], 0.f));
    }
  }
}

// ---------------------------------------------------------------------------
// |W_O^h v_t| on the tensor cores (d = 128): vn^2 = v_t^T G_h v_t with
// G_h = W_O^h^T W_O^h.  G_h (fp32, the sum of the Gram slices in slice order)
// is split into two bf16 matrices, G = G_hi + G_lo (16 significant bits), and
// P = V_tile G_h is two tcgen05 MMAs into TMEM (bf16 products exact, fp32
// sums); the epilogue thread of token t then forms sum_c P[t, c] V[t, c],
// reading its value row from global memory (L2-resident: TMA just brought the
// tile in for the MMA).  Reading the row from the staged shared-memory tile
// instead gave wrong sums, varying run to run, whenever both tile stages and
// both accumulator buffers were in flight (with one of either, it was exact);
// the global read is exact with the full pipeline.
// grid (n_split, Hq), 192 threads: warps 0-3 the epilogue (one token row per
// thread), warp 4 TMA (the value tiles of KV head h / G), warp 5 the MMAs.
// ---------------------------------------------------------------------------
constexpr int kVnThreads = 192;
constexpr int kVnStages = 2;

struct VnSmem {
  uint8_t g_hi[2 * 16384];            // G_h high part, K-major 128-byte-swizzle panels (B operand)
  uint8_t g_lo[2 * 16384];            // G_h low part
  uint8_t v[kVnStages][2 * 16384];    // value tiles: 128 tokens x 128 channels (A operand)
  uint64_t v_full[kVnStages], v_empty[kVnStages], acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  int abort_flag;
};

// byte offset of element (row r, column c) of a K-major 128-byte-swizzle tile of 128-column rows
__device__ __forceinline__ uint32_t sw128_elem(int r, int c) {
  return static_cast<uint32_t>((c >> 6) * 16384 + (r >> 3) * 1024 + (r & 7) * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) +
                               (c & 7) * 2);
}

__global__ void __launch_bounds__(kVnThreads, 1)
    vnorm_tc_kernel(const __grid_constant__ CUtensorMap mapV, const float* __restrict__ gram, const int n_slices,
                    const int Hq, const int G, const int N, const int tiles_per_cta, float* __restrict__ vn,
                    const uint16_t* __restrict__ V) {
  extern __shared__ uint8_t smem_raw[];
  VnSmem& S = *reinterpret_cast<VnSmem*>(align1024(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, g = h / G;
  const int n_tiles = (N + 127) / 128;
  const int tile0 = blockIdx.x * tiles_per_cta;
  const int tile1 = min(n_tiles, tile0 + tiles_per_cta);
  if (tile0 >= tile1 || timeout_recorded()) return;  // uniform over the CTA, before any barrier
  if (threadIdx.x == 0) {
    for (int s = 0; s < kVnStages; ++s) {
      mbar_init(&S.v_full[s], 1);
      mbar_init(&S.v_empty[s], 1 + 4);  // the MMAs and the 4 epilogue warps (they read the tile too)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.acc_full[b], 1);
      mbar_init(&S.acc_empty[b], 4);
    }
    mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, 256);
    tmem_relinquish();
  }
  pdl_wait();  // the Gram slices come from the previous kernel on the stream
  // G_h = sum of the slices (fixed order), split into bf16 high and low parts
  const float* gh = gram + static_cast<size_t>(h) * 128 * 128;
  const size_t slice = static_cast<size_t>(Hq) * 128 * 128;
  for (int e = threadIdx.x; e < 128 * 128; e += kVnThreads) {
    float a = 0.f;
    for (int s = 0; s < n_slices; ++s) a += gh[s * slice + e];
    const int r = e >> 7, c = e & 127;  // B operand row n = r (G is symmetric), K index c
    const __nv_bfloat16 hi = __float2bfloat16_rn(a);
    const __nv_bfloat16 lo = __float2bfloat16_rn(a - __bfloat162float(hi));
    *reinterpret_cast<__nv_bfloat16*>(S.g_hi + sw128_elem(r, c)) = hi;
    *reinterpret_cast<__nv_bfloat16*>(S.g_lo + sw128_elem(r, c)) = lo;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the stores above are visible to the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;
  const int nt = tile1 - tile0;

  if (warp == 4) {
    if (lane == 0) {  // TMA producer
      prefetch_tensormap(&mapV);
      int issued = 0;
      for (int i = 0; i < nt; ++i) {
        const int s = i % kVnStages;
        if (!mbar_wait(&S.v_empty[s], ((i / kVnStages) & 1) ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(&S.v_full[s], 2 * 16384);
#pragma unroll
        for (int p = 0; p < 2; ++p) tma_load_3d(S.v[s] + p * 16384, &mapV, &S.v_full[s], p * 64, (tile0 + i) * 128, g);
        issued = i + 1;
      }
      if (*abort_flag) {
        volatile int never = 0;
        for (int i = max(0, issued - kVnStages); i < issued; ++i)
          mbar_wait(&S.v_full[i % kVnStages], (i / kVnStages) & 1, &never);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {  // MMA issuer: P = V_tile (M = 128 tokens) x G_h (N = 128 channels), hi then lo
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      for (int i = 0; i < nt; ++i) {
        const int s = i % kVnStages, b = i & 1;
        if (!mbar_wait(&S.v_full[s], (i / kVnStages) & 1, abort_flag) ||
            !mbar_wait(&S.acc_empty[b], ((i >> 1) & 1) ^ 1u, abort_flag))
          break;
        tc_fence_after();
        const uint32_t a = smem_u32(S.v[s]);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t bm = smem_u32(part ? S.g_lo : S.g_hi);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * 16384u + (kk & 3) * 32u;
            umma_bf16(tmem + b * 128, sdesc_kmajor_sw128(a + off), sdesc_kmajor_sw128(bm + off), idesc,
                      (part > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(&S.v_empty[s]);
        umma_commit(&S.acc_full[b]);
      }
      if (*abort_flag) {
        volatile int never = 0;
        umma_commit(&S.drain);
        mbar_wait(&S.drain, 0, &never);
      }
    }
  } else {  // warps 0-3: token row 32 warp + lane of each tile
    const int row = warp * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint16_t* Vg = V + static_cast<long long>(g) * N * 128;
    uint32_t pv[32];
    for (int i = 0; i < nt; ++i) {
      const int s = i % kVnStages, b = i & 1;
      if (!mbar_wait(&S.acc_full[b], (i >> 1) & 1, abort_flag)) break;
      tc_fence_after();
      const int t = (tile0 + i) * 128 + row;
      const uint16_t* vrow = Vg + static_cast<long long>(min(t, N - 1)) * 128;
      float acc = 0.f;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        tmem_issue32(lane_base + b * 128 + ch * 32, pv);
        tmem_wait32(pv);
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {  // 8 channels of the value row per 16-byte load
          const int c = ch * 32 + j8 * 8;
          const uint4 q = __ldg(reinterpret_cast<const uint4*>(vrow + c));
          const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc = fmaf(__uint_as_float(pv[j8 * 8 + 2 * k]), __uint_as_float(wv[k] << 16), acc);
            acc = fmaf(__uint_as_float(pv[j8 * 8 + 2 * k + 1]), __uint_as_float(wv[k] & 0xFFFF0000u), acc);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.acc_empty[b]);
        mbar_arrive(&S.v_empty[s]);
      }
      if (t < N) vn[static_cast<size_t>(h) * N + t] = sqrtf(fmaxf(acc, 0.f));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace kvs
