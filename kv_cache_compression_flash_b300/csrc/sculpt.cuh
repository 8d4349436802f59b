// KVSculpt: the attention targets of the compression zone and the closed-form
// values for fixed compressed keys   [KVSculpt §2: the compressed pairs are
// fitted to the block's attention output and LSE; with the keys fixed, the
// values are a ridge least-squares solution].
//
//   block_attention_tc_kernel<DH>  flash-style on tcgen05 (S, P and O in
//       TMEM, P read there as the A operand of the second MMA; see below).  Row r sees
//       keys t < n_block, t <= q_pos0 + r.
//   ridge_softmax_kernel<DH>    A = softmax over all k compressed keys (no
//       mask: every training query sees the whole compressed block), the
//       logits by mma.sync m16n8k16 (bf16 products, fp32 sums), in two sweeps
//       over the keys (row max and sum, then the weights).
//   ridge_atb_kernel            A^T A + lam I (its lower 64 x 64 tiles) and
//       A^T Y in one launch, 4 x 4 outputs a thread over 32-row slices of R,
//       R split in two halves whose partial sums the solve adds.
//   ridge_solve_cluster_kernel<DH>  a cluster of 8 CTAs per head: blocked
//       Cholesky of A^T A + lam I and the forward and backward solves for
//       the d right-hand sides, the matrix in the cluster's shared memory.
// A^T A, A^T Y and the solve are fp32 on the FMA pipes.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace kvs {

constexpr int kRidgeMaxK = 512;
constexpr int kRidgeMaxD = 128;

// ---- mma.sync helpers (the ridge's softmax): m16n8k16, bf16 -> fp32 ----
constexpr int kBaThreads = 128;  // 4 warps x 16 rows
constexpr int kBaKeys = 64;      // keys per chunk

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


// ---- block attention on tcgen05 ---------------------------------------------
// One CTA per 128-row query tile (Gt heads of one KV group x P = 128 / Gt
// window positions, as in the scoring passes), looping over the block's keys
// 128 at a time.  The key tiles alternate between two softmax groups of four
// warps (group g takes tiles j = g, g + 2, ...; warp w of a group reads TMEM
// lanes 32 (w % 4) .., one query row a thread, all 128 keys of its tile); each
// group keeps its own running max m, sum l and output accumulator O_g, so the
// groups never wait on each other and one group's softmax overlaps the other
// group's products on the tensor pipe:
//   S = Q K^T                 tcgen05.mma into TMEM buffer j & 1
//   P = 2^(S c - m_g)         the row max m_g in the log2 domain is raised
//                             only when a row's tile max exceeds it by
//                             kBtRescale, and then the row's O_g and l_g are
//                             scaled by 2^(m_old - m_new); P is split into a
//                             high part (its upper 16 bits: bf16 by
//                             truncation) and the bf16 of the remainder (16
//                             significant bits together), written as bf16
//                             pairs into TMEM over the tile's own S columns
//   O_g += P_hi V + P_lo V    two tcgen05.mma into TMEM, A = P read from TMEM,
//                             V straight from its TMA tile as an MN-major B
//                             operand (channels contiguous; the instruction's
//                             transpose bit)
// and at the end the two groups' parts are merged, m = max(m_0, m_1),
// O = sum_g 2^(m_g - m) O_g, l likewise, Y = O / l, lse = (m + log2 l) ln 2
// (group g writes channels g DH / 2 .. of Y).  Warp 8 issues TMA (K and V
// each in a 3-stage ring), warp 9 the MMAs: S of tile j + 2 goes into buffer
// j & 1 once the O product of tile j has read its P.  Warps 10 and 11 only
// complete the third warpgroup, which hands its registers to the softmax
// warpgroups (setmaxnreg), so the softmax runs without register spills.  Every
// wait is bounded.
// TMEM: S/P buffers at columns 0 and 128, O_0 at 256, O_1 at 256 + DH.
constexpr int kBtThreads = 384;  // three warpgroups: softmax groups 0 and 1, then TMA, MMA and two idle warps
// registers a thread after the split: the softmax warpgroups take what the
// third gives up (the sum stays within the launch's threads x registers)
constexpr int kBtRegsSoft = 216, kBtRegsCtl = 56;
constexpr int kBtRegPool = 2 * 128 * kBtRegsSoft + 128 * kBtRegsCtl;
constexpr int kBtSoftWarps = 8;  // two groups of four
constexpr int kBtTmaWarp = 8, kBtMmaWarp = 9;
constexpr int kBtKStages = 3;
constexpr int kBtVStages = 3;
constexpr float kBtRescale = 8.f;

template <int DH>
struct BtSmem {
  uint8_t q[TileCfg<DH>::kTileBytes];              // 128 rows x DH, K-major, DH / 64 panels
  uint8_t k[kBtKStages][TileCfg<DH>::kTileBytes];  // 128 keys x DH
  uint8_t v[kBtVStages][TileCfg<DH>::kTileBytes];  // 128 keys x DH as TMA brings it: the MN-major B operand
  uint64_t q_full, k_full[kBtKStages], k_empty[kBtKStages], v_full[kBtVStages], v_empty[kBtVStages], s_full[2],
      p_full[2], pv_done[2], o_full, drain;
  uint32_t tmem_base;
  int abort_flag;
};

// byte offset of element (row r, column c) of a K-major 128-byte-swizzle
// operand whose 64-column panels hold `rows` rows each
__device__ __forceinline__ uint32_t bt_sw(int r, int c, int rows) {
  return static_cast<uint32_t>((c >> 6) * rows * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}

// 32 consecutive fp32 columns of this thread's TMEM lane, written back
__device__ __forceinline__ void tmem_store32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]),
      "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]),
      "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]),
      "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}
// barrier `id` (not 0: __syncthreads) over the first `n` threads of the CTA
__device__ __forceinline__ void named_barrier_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// 16 consecutive 32-bit columns of this thread's TMEM lane, written back
__device__ __forceinline__ void tmem_store16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// one fp32 column of this thread's TMEM lane: store (waited), load (waited)
__device__ __forceinline__ void tmem_store1(uint32_t taddr, float v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};\n\ttcgen05.wait::st.sync.aligned;" ::"r"(taddr),
               "f"(v)
               : "memory");
}
__device__ __forceinline__ float tmem_load1(uint32_t taddr) {
  float v;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\ttcgen05.wait::ld.sync.aligned;"
               : "=f"(v)
               : "r"(taddr)
               : "memory");
  return v;
}

// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle
// (rows along K, each row 64 MN elements = 128 bytes): 8-row atoms every 1024
// bytes along K (stride byte offset), 64-element blocks along MN every `lbo`
// bytes (leading byte offset).
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// D[tmem] (+)= A[tmem] * B[smem]: the A operand read from tensor memory (one
// row per lane, two 16-bit elements per 32-bit column)
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// O (+)= P V over the 128 keys of a tile: A = P in TMEM (64 columns of bf16
// pairs, keys 2c and 2c + 1 in column c), B = V as loaded (128 keys x DH,
// MN-major: the transpose bit of the instruction)
template <int DH>
__device__ __forceinline__ void bt_issue_pv(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, DH) | (1u << 16);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)  // 16 keys a step: 8 columns of A, two 8-row atoms of B
    umma_bf16_ts(d_tmem, a_tmem + kk * 8, sdesc_mnmajor_sw128(b_base + kk * 2048u, 16384u), idesc,
                 (accumulate || kk > 0) ? 1u : 0u);
}

// grid: Hkv * n_hc * n_pb query tiles (tile rt: group rt / (n_hc n_pb), head chunk (rt / n_pb) % n_hc,
// position block rt % n_pb); kBtThreads threads.
template <int DH>
__global__ void __launch_bounds__(kBtThreads, 1)
    block_attention_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                              const __grid_constant__ CUtensorMap mapV, const int G, const int Gt, const int W,
                              const int q_pos0, const int n_block, const int n_hc, const int n_pb,
                              const float c_log2, float* __restrict__ Y, float* __restrict__ lse) {
  extern __shared__ uint8_t smem_raw[];
  BtSmem<DH>& S = *reinterpret_cast<BtSmem<DH>*>(align1024(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (timeout_recorded()) return;  // uniform over the CTA, before any barrier
  const int P = 128 / Gt;
  const int rt = blockIdx.x;
  const int g = rt / (n_hc * n_pb), hc = (rt / n_pb) % n_hc, pb = rt % n_pb;
  const int h0 = g * G + hc * Gt;  // the tile's first query head
  const int p_last = min((pb + 1) * P, W) - 1;
  const int n_keys = min(n_block, q_pos0 + p_last + 1);
  const int n_kt = (n_keys + 127) / 128;

  if (threadIdx.x == 0) {
    mbar_init(&S.q_full, 1);
    for (int i = 0; i < kBtKStages; ++i) {
      mbar_init(&S.k_full[i], 1);
      mbar_init(&S.k_empty[i], 1);
    }
    for (int i = 0; i < kBtVStages; ++i) {
      mbar_init(&S.v_full[i], 1);
      mbar_init(&S.v_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.s_full[b], 1);
      mbar_init(&S.p_full[b], kBtSoftWarps / 2);  // the four warps of group b
      mbar_init(&S.pv_done[b], 1);                // the O product that read P from buffer b is done
    }
    mbar_init(&S.o_full, 1);
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
  pdl_wait();
  pdl_trigger();
  const uint32_t tmem = S.tmem_base;  // S/P buffers at columns 0 and 128, O_0 at 256, O_1 at 256 + DH
  volatile int* abort_flag = &S.abort_flag;
  constexpr uint32_t kTile = TileCfg<DH>::kTileBytes;

  if (warp >= kBtSoftWarps) {  // the third warpgroup gives registers up, then its TMA and MMA warps run
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kBtRegsCtl));
  if (warp == kBtTmaWarp) {
    if (lane == 0) {  // TMA producer
      prefetch_tensormap(&mapQ);
      prefetch_tensormap(&mapK);
      prefetch_tensormap(&mapV);
      mbar_arrive_expect_tx(&S.q_full, kTile);
#pragma unroll
      for (int p = 0; p < TileCfg<DH>::kPanels; ++p)
        tma_load_3d(S.q + p * 16384, &mapQ, &S.q_full, p * 64, pb * P, h0);
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int s = j % kBtKStages;
        if (j >= kBtKStages && !mbar_wait(&S.k_empty[s], ((j / kBtKStages) - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(&S.k_full[s], kTile);
#pragma unroll
        for (int p = 0; p < TileCfg<DH>::kPanels; ++p)
          tma_load_3d(S.k[s] + p * 16384, &mapK, &S.k_full[s], p * 64, j * 128, g);
        issued_k = j + 1;
        const int sv = j % kBtVStages;
        if (j >= kBtVStages && !mbar_wait(&S.v_empty[sv], ((j / kBtVStages) - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(&S.v_full[sv], kTile);
#pragma unroll
        for (int p = 0; p < TileCfg<DH>::kPanels; ++p)
          tma_load_3d(S.v[sv] + p * 16384, &mapV, &S.v_full[sv], p * 64, j * 128, g);
        issued_v = j + 1;
      }
      if (*abort_flag) {  // let our copies land before the CTA goes away
        volatile int never = 0;
        mbar_wait(&S.q_full, 0, &never);
        for (int i = max(0, issued_k - kBtKStages); i < issued_k; ++i)
          mbar_wait(&S.k_full[i % kBtKStages], (i / kBtKStages) & 1, &never);
        for (int i = max(0, issued_v - kBtVStages); i < issued_v; ++i)
          mbar_wait(&S.v_full[i % kBtVStages], (i / kBtVStages) & 1, &never);
      }
    }
  } else if (warp == kBtMmaWarp) {
    if (lane == 0) {  // MMA issuer
      bool ok = mbar_wait(&S.q_full, 0, abort_flag);
      auto mma_s = [&](int j) {  // S of tile j into buffer j & 1
        const int s = j % kBtKStages;
        if (!mbar_wait(&S.k_full[s], (j / kBtKStages) & 1, abort_flag)) return false;
        tc_fence_after();
        issue_tile_mma<DH>(tmem + (j & 1) * 128, smem_u32(S.q), smem_u32(S.k[s]));
        umma_commit(&S.k_empty[s]);
        umma_commit(&S.s_full[j & 1]);
        return true;
      };
      if (ok) ok = mma_s(0);
      if (ok && n_kt > 1) ok = mma_s(1);
      for (int j = 0; j < n_kt && ok; ++j) {
        const int b = j & 1, sv = j % kBtVStages;
        if (!mbar_wait(&S.p_full[b], (j >> 1) & 1, abort_flag) ||
            !mbar_wait(&S.v_full[sv], (j / kBtVStages) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pt = tmem + b * 128, ot = tmem + 256 + b * DH;  // P of tile j sits over its S
        bt_issue_pv<DH>(ot, pt, smem_u32(S.v[sv]), j >= 2);
        bt_issue_pv<DH>(ot, pt + 64, smem_u32(S.v[sv]), true);
        umma_commit(&S.v_empty[sv]);
        if (j + 2 < n_kt) {  // the buffer takes S of tile j + 2 once this product has read P
          umma_commit(&S.pv_done[b]);
          if (!mbar_wait(&S.pv_done[b], (j >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          ok = mma_s(j + 2);
        }
      }
      if (ok) umma_commit(&S.o_full);
      if (*abort_flag) {
        volatile int never = 0;
        umma_commit(&S.drain);
        mbar_wait(&S.drain, 0, &never);
      }
    }
  }
  } else {  // warps 0-7: softmax; group grp = warp / 4 takes tiles grp, grp + 2, ...; TMEM lanes 32 (warp % 4) ..
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kBtRegsSoft));
    const int grp = warp >> 2, q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const int hl = row / P, pos = pb * P + row % P;
    const int posc = min(pos, W - 1);
    const int vis = min(n_block, q_pos0 + posc + 1);  // keys this row sees
    // the lowest visible count over the warp's rows: tiles below it need no mask
    int vis_w = vis;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) vis_w = min(vis_w, __shfl_xor_sync(0xFFFFFFFFu, vis_w, o));
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const uint32_t sb = lane_base + grp * 128;       // this group's S/P buffer
    const uint32_t ob = lane_base + 256 + grp * DH;  // and its O
    const float c = c_log2;
    const unsigned long long c2 = f2_pack(c, c);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = grp; j < n_kt; j += 2) {
      const int t0 = j * 128;
      const bool full = t0 + 128 <= vis_w;  // every key of the tile is visible to all the warp's rows
      const int lim = vis - t0;             // keys of the tile this row sees (may be <= 0 or >= 128)
      if (!mbar_wait(&S.s_full[grp], (j >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the tile's row max, masked keys left out: keys 0-63 first, then 64-127
      // (kept in registers; 0-63 are read again for P)
      auto mask = [&](uint32_t (&r)[32], int k0) {  // keys the row does not see: -inf (2^-inf = 0 in P)
        if (!full) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (k0 + e >= lim) r[e] = 0xFF800000u;
        }
      };
      auto chunk_max = [&](const uint32_t (&r)[32], int k0) {
        const float* x = reinterpret_cast<const float*>(r);
        float u[11];
#pragma unroll
        for (int k = 0; k < 10; ++k) u[k] = fmax3(x[3 * k], x[3 * k + 1], x[3 * k + 2]);
        u[10] = fmaxf(x[30], x[31]);
        return fmax3(fmax3(u[0], u[1], u[2]), fmax3(u[3], u[4], u[5]), fmax3(u[6], u[7], fmax3(u[8], u[9], u[10])));
      };
      float z;
      {
        uint32_t ra[32], rb[32];
        tmem_issue32(sb, ra);
        tmem_issue32(sb + 32, rb);
        tmem_wait32(ra);
        tmem_wait32(rb);
        mask(ra, 0);
        mask(rb, 32);
        z = fmaxf(chunk_max(ra, 0), chunk_max(rb, 32));
      }
      uint32_t rc[32], rd[32];
      tmem_issue32(sb + 64, rc);
      tmem_issue32(sb + 96, rd);
      tmem_wait32(rc);
      tmem_wait32(rd);
      mask(rc, 64);
      mask(rd, 96);
      z = fmax3(z, chunk_max(rc, 64), chunk_max(rd, 96));
      z *= c;
      // raised only past the margin (never by a tile with no visible key: z = -inf)
      const bool raise = z > m + kBtRescale;
      float alpha = 1.f;
      if (raise) {
        alpha = ex2_approx(m - z);  // 0 on the row's first visible tile
        m = z;
      }
      l *= alpha;
      // P = 2^(s c - m), its row sum, and its two bf16 parts into TMEM over
      // this tile's S: keys 2i, 2i + 1 of the tile as a bf16 pair in column i
      // (high part) and 64 + i (low part).  Keys 0-63 are read again first
      // (their parts land on columns 0-31 and 64-95: S of keys 0-31, read,
      // and of keys 64-95, in registers); keys 64-127 come from registers.
      const float m_sub = m == -INFINITY ? 0.f : m;  // a row with no visible key yet: P = 0, not NaN
      const unsigned long long nm2 = f2_pack(-m_sub, -m_sub);
      unsigned long long acc2 = 0ull;
      auto chunk_p = [&](const uint32_t (&r)[32], int q) {
        const float* x = reinterpret_cast<const float*>(r);
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float e0, e1;
          f2_unpack(f2_fma(f2_pack(x[e], x[e + 1]), c2, nm2), &e0, &e1);
          const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
          acc2 = f2_add(acc2, f2_pack(p0, p1));
          const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
          hi[e / 2] = __byte_perm(b0, b1, 0x7632);  // the upper halves: bf16 by truncation
          float r0, r1;
          f2_unpack(f2_add(f2_pack(p0, p1),
                           f2_pack(-__uint_as_float(b0 & 0xFFFF0000u), -__uint_as_float(b1 & 0xFFFF0000u))),
                    &r0, &r1);
          lo[e / 2] = ba_bf2(r0, r1);
        }
        tmem_store16(sb + q * 16, hi);
        tmem_store16(sb + 64 + q * 16, lo);
      };
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t ra[32];
        tmem_load32(sb + q * 32, reinterpret_cast<float(&)[32]>(ra));
        mask(ra, q * 32);
        chunk_p(ra, q);
      }
      chunk_p(rc, 2);
      chunk_p(rd, 3);
      // scale this warp's rows of O_g (after P, with S out of the registers):
      // its last product (tile j - 2) is done, for S of tile j was issued
      // after it had read its P
      if (j >= 2 && __any_sync(0xFFFFFFFFu, raise)) {
#pragma unroll
        for (int ch = 0; ch < DH / 32; ++ch) {
          float o[32];
          tmem_load32(ob + ch * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_store32(ob + ch * 32, o);
        }
      }
      tmem_wait_st();
      float s0, s1;
      f2_unpack(acc2, &s0, &s1);
      l += s0 + s1;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.p_full[grp]);
    }
    // merge the two groups' parts: each thread leaves its row's m_g and l_g
    // in columns 2 grp, 2 grp + 1 of buffer 0 (free: every product is done)
    const bool good = ok && mbar_wait(&S.o_full, 0, abort_flag);
    if (good) {
      tc_fence_after();
      tmem_store1(lane_base + 2 * grp, m);
      tmem_store1(lane_base + 2 * grp + 1, l);
    }
    tc_fence_before();
    named_barrier_sync(1, kBtSoftWarps * 32);  // every softmax warp reaches it once
    tc_fence_after();
    if (good && !*abort_flag) {
      const float m_o = tmem_load1(lane_base + 2 * (grp ^ 1));
      const float l_o = tmem_load1(lane_base + 2 * (grp ^ 1) + 1);
      const float m0 = grp == 0 ? m : m_o, l0 = grp == 0 ? l : l_o;
      const float m1 = grp == 0 ? m_o : m, l1 = grp == 0 ? l_o : l;
      const bool two = n_kt > 1;  // O_1 holds a product
      const float mt = two ? fmaxf(m0, m1) : m0;
      const float a0 = ex2_approx(m0 - mt), a1 = two ? ex2_approx(m1 - mt) : 0.f;
      const float lt = l0 * a0 + l1 * a1;
      const bool store = pos < W && hl < Gt;
      const long long hd = h0 + hl;
      const int o_lo = grp * (DH / 2);  // this group's channels of Y
      float* yr = Y + (hd * W + posc) * DH + o_lo;
      const float inv = 1.f / lt;
      const float w0 = a0 * inv, w1 = a1 * inv;
#pragma unroll
      for (int ch = 0; ch < DH / 64; ++ch) {
        float o[32], o1[32];
        tmem_load32(lane_base + 256 + o_lo + ch * 32, o);
        if (two) {
          tmem_load32(lane_base + 256 + DH + o_lo + ch * 32, o1);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = o[e] * w0 + o1[e] * w1;
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= w0;
        }
        if (store) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(yr + ch * 32 + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
        }
      }
      if (store && lse && grp == 0) lse[hd * W + posc] = (mt + lg2_approx(lt)) * kLn2;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


// A[g][r][i] = softmax_i(Qt[g][r] . Kc[g][i] / sqrt(d)) over the k compressed keys.
// grid (ceil(R / 64), Hkv), 128 threads, 16 rows a warp; the logits from
// mma.sync m16n8k16 over chunks of 64 keys (cp.async, double-buffered, rows
// past k clamped and masked), in two sweeps: the row max and sum, then the
// normalised weights written to A.
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
constexpr int kAtbTile = 64, kAtbSlice = 32;
constexpr int kAtbSplit = 2;  // partial sums over the halves of R, added by the solve as it loads them

// One launch for both products of a head: tile t < kt (kt + 1) / 2 is a lower
// tile of A^T A (+ lam I on the diagonal of split 0), the rest the tiles of
// A^T Y; blockIdx.y = the split s (rows s Rs .. (s + 1) Rs - 1 of R), blockIdx.z
// = the head.  Split s writes M + s mstride and B + s bstride.
__global__ void __launch_bounds__(256) ridge_atb_kernel(const float* __restrict__ A, const float* __restrict__ Y,
                                                        int R, int k, int d, float lam, float* __restrict__ M,
                                                        long long mstride, float* __restrict__ B,
                                                        long long bstride) {
  pdl_wait();
  pdl_trigger();
  const int kt = (k + kAtbTile - 1) / kAtbTile, nlow = kt * (kt + 1) / 2;
  int t = blockIdx.x;
  const bool gram = t < nlow;
  int ti = 0, tj;
  if (gram) {
    while ((ti + 1) * (ti + 2) / 2 <= t) ++ti;
    tj = t - ti * (ti + 1) / 2;
  } else {
    t -= nlow;
    const int dt = (d + kAtbTile - 1) / kAtbTile;
    ti = t / dt;
    tj = t % dt;
  }
  const int n = gram ? k : d;
  const int i0 = ti * kAtbTile, j0 = tj * kAtbTile;
  const int split = blockIdx.y, g = blockIdx.z;
  const int Rs = (R + kAtbSplit * kAtbSlice - 1) / (kAtbSplit * kAtbSlice) * kAtbSlice;  // rows of a split
  const int rb = split * Rs, re = min(R, rb + Rs);
  __shared__ __align__(16) float ps[kAtbSlice][kAtbTile];
  __shared__ __align__(16) float qs[kAtbSlice][kAtbTile];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const float* Pg = A + static_cast<long long>(g) * R * k;
  const float* Qg = gram ? Pg : Y + static_cast<long long>(g) * R * d;
  // this thread's loads per slice: element e = tid + 256 u -> row e / 64, column e % 64
  constexpr int kLoads = kAtbSlice * kAtbTile / 256;
  float pv[kLoads], qv[kLoads];
  auto fetch = [&](int r0) {
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int e = tid + 256 * u, rr = e >> 6, cc = e & 63, r = r0 + rr;
      pv[u] = (r < re && i0 + cc < k) ? Pg[static_cast<long long>(r) * k + i0 + cc] : 0.f;
      qv[u] = (r < re && j0 + cc < n) ? Qg[static_cast<long long>(r) * n + j0 + cc] : 0.f;
    }
  };
  float acc[4][4];
#pragma unroll
  for (int u = 0; u < 4; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
  fetch(rb);
  for (int r0 = rb; r0 < re; r0 += kAtbSlice) {
    __syncthreads();  // the previous slice is consumed
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int e = tid + 256 * u;
      ps[e >> 6][e & 63] = pv[u];
      qs[e >> 6][e & 63] = qv[u];
    }
    __syncthreads();
    if (r0 + kAtbSlice < re) fetch(r0 + kAtbSlice);
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
  float* C = gram ? M + split * mstride : B + split * bstride;
  const bool diag = gram && split == 0;
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int i = i0 + 4 * ty + u, j = j0 + 4 * tx + v;
      if (i < k && j < n)
        C[(static_cast<long long>(g) * k + i) * n + j] = acc[u][v] + ((diag && i == j) ? lam : 0.f);
    }
}

// ---- ridge solve across a cluster ---------------------------------------------
// (A^T A + lam I) Vc = A^T Y for each head: a blocked Cholesky factorisation
// L L^T and two blocked triangular solves, on a cluster of kRsCluster CTAs
// per head that hold the matrix in their shared memory.  The k x k matrix is
// padded with the identity to nblk <= 16 row blocks of 32 (a padded row
// solves to 0); block i lives in CTA i (i < 8) or 15 - i (i >= 8): its rows,
// columns 0 .. 32 i + 31 (the lower triangle up to its diagonal block), so
// every CTA holds 17 blocks' worth of columns and the updates of one column
// step are spread evenly.  Column step b:
//   the owner of block b factors the diagonal block in one warp (L_bb) and
//   inverts it, one lane per column; cluster barrier;
//   every CTA turns its blocks i > b into L_ib = M_ib L_bb^-T (L_bb^-1 read
//   from the owner); cluster barrier;
//   every CTA copies the rows of the column panel L_jb (j > b) it needs from
//   their owners and updates its blocks, M_ij -= L_ib L_jb^T for b < j <= i,
//   8 x 4 outputs a thread.
// The diagonal block is factored and inverted in registers (warp shuffles).
// The two solves split the d channels over the cluster (CTA r takes
// d / 8 of them for every row) and need no further barrier; both are
// right-looking: the forward solve L y = A^T Y takes y_b = L_bb^-1 r_b and
// subtracts L_ib y_b from the rows below (column block b of L read from the
// owners of those rows), the backward solve L^T x = y takes x_b = L_bb^-T y_b
// from the last block up and subtracts L_bi^T x_b from the rows above (row
// block b read from its owner).  fp32 FMA throughout.  A pivot that is not positive
// records KVS_ERR_RANGE and the head's values are 0.
constexpr int kRsCluster = 8;
constexpr int kRsThreads = 512;
constexpr int kRsMaxBlocks = kRidgeMaxK / 32;  // 16 = 2 kRsCluster
constexpr int kRsLd = 33;                      // a 32 x 32 block in shared memory
constexpr int kRsBlk = 32 * kRsLd;
constexpr int kRsLdAt = 36;                        // a transposed panel block L_ib^T
constexpr int kRsLdp = 32 * (kRsMaxBlocks - 1) + 4;  // the column panel, transposed: 32 x (rows below the diagonal)
// shared memory layout (floats), the same in every CTA of the cluster
constexpr int kRsOffB = 32 * (32 * (kRsMaxBlocks + 1) + 8);  // after the rows of the CTA's two blocks
constexpr int kRsOffAt = kRsOffB + 2 * 32 * kRidgeMaxD;       // the solves' right-hand sides (the CTA's channels)
constexpr int kRsOffPt = kRsOffAt + 2 * 32 * kRsLdAt;         // panel; in the solves a row or column block of L
constexpr int kRsOffDinv = kRsOffPt + 32 * kRsLdp;            // L_bb^-1 of the two blocks
constexpr int kRsOffTinv = kRsOffDinv + 2 * kRsBlk;           // a copy of the current L_bb^-1
constexpr int kRsOffFlag = kRsOffTinv + kRsBlk;               // a pivot was not positive
constexpr size_t kRsSmemBytes = static_cast<size_t>(kRsOffFlag + 4) * sizeof(float);
static_assert(kRidgeMaxK * (kRidgeMaxD / kRsCluster) <= 2 * 32 * kRidgeMaxD, "the channel slice fits");
static_assert(32 * (kRidgeMaxK - 32) <= 32 * kRsLdp, "a row or column block of L fits in the panel's space");
static_assert(kRsMaxBlocks == 2 * kRsCluster, "two blocks per CTA");

__device__ __forceinline__ int rs_owner(int i) { return i < kRsCluster ? i : 2 * kRsCluster - 1 - i; }
__device__ __forceinline__ int rs_slot(int i) { return i < kRsCluster ? 0 : 1; }
// row stride of block i's rows at its owner, and where they start there
__device__ __forceinline__ int rs_ld(int i) { return 32 * (i + 1) + 4; }
__device__ __forceinline__ int rs_off(int i) { return i < kRsCluster ? 0 : 32 * rs_ld(2 * kRsCluster - 1 - i); }

// grid (kRsCluster, Hkv), clusters of kRsCluster along x; kRsThreads threads.
template <int DH>
__global__ void __launch_bounds__(kRsThreads, 1)
    ridge_solve_cluster_kernel(const float* __restrict__ M, long long mstride, const float* __restrict__ B,
                               long long bstride, const int k, float* __restrict__ Vc) {
  namespace cgr = cooperative_groups;
  cgr::cluster_group cluster = cgr::this_cluster();
  extern __shared__ float4 rs_smem4[];
  float* sm = reinterpret_cast<float*>(rs_smem4);
  const int rank = static_cast<int>(cluster.block_rank());
  const int g = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nblk = (k + 31) >> 5;
  const float* Mg = M + static_cast<long long>(g) * k * k;
  const float* Bg = B + static_cast<long long>(g) * k * DH;
  float* Vg = Vc + static_cast<long long>(g) * k * DH;
  float* PT = sm + kRsOffPt;
  float* dinv = sm + kRsOffDinv;
  float* tinv = sm + kRsOffTinv;
  int* flag = reinterpret_cast<int*>(sm + kRsOffFlag);
  const int own[2] = {rank, 2 * kRsCluster - 1 - rank};  // slot 0 holds the lower block
  const bool has[2] = {own[0] < nblk, own[1] < nblk};
  float* Ms[2] = {sm + rs_off(own[0]), sm + rs_off(own[1])};
  const int lds[2] = {rs_ld(own[0]), rs_ld(own[1])};
  float* At[2] = {sm + kRsOffAt, sm + kRsOffAt + 32 * kRsLdAt};
  const int imax = has[1] ? own[1] : own[0];  // the CTA's last block (when it has one)
  pdl_wait();

  // the CTA's rows of M (padded with the identity)
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    if (!has[s]) continue;
    const int i = own[s], wdt = 32 * (i + 1);
    for (int e = tid; e < 32 * wdt; e += kRsThreads) {
      const int rr = e / wdt, c = e - rr * wdt, gr = 32 * i + rr;
      float v = gr == c ? 1.f : 0.f;
      if (gr < k && c < k) {
        const long long o = static_cast<long long>(gr) * k + c;
        v = __ldg(Mg + o);
#pragma unroll
        for (int sp = 1; sp < kAtbSplit; ++sp) v += __ldg(Mg + sp * mstride + o);
      }
      Ms[s][rr * lds[s] + c] = v;
    }
  }
  if (tid == 0) *flag = 0;
  cluster.sync();

  // ---- factorisation ----
  bool bad = false;
  for (int b = 0; b < nblk; ++b) {
    const int ob = rs_owner(b), sb = rs_slot(b);
    if (rank == ob && warp == 0) {  // L_bb in registers (lane = row), then L_bb^-1 (lane = column)
      const float* Db = (sb ? Ms[1] : Ms[0]) + 32 * b;
      const int ldb = sb ? lds[1] : lds[0];
      float a[32];  // row `lane` of the block, straight from the CTA's rows; the lower triangle becomes L_bb
#pragma unroll
      for (int c = 0; c < 32; ++c) a[c] = Db[lane * ldb + c];
      bool ok = true;  // the same value in every lane (no early exit: a[] stays in registers)
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p = __shfl_sync(0xFFFFFFFFu, a[c], c);
        ok = ok && p > 0.f;
        const float rp = __frsqrt_rn(p);  // 1 / L_cc
        if (lane == c) a[c] = p * rp;
        if (lane > c) a[c] *= rp;
#pragma unroll
        for (int c2 = 1; c2 < 32; ++c2) {  // row c2 > c of the trailing block, for the rows that reach it
          if (c2 > c) {
            const float l = __shfl_sync(0xFFFFFFFFu, a[c], c2);
            if (lane >= c2) a[c2] = fmaf(-a[c], l, a[c2]);
          }
        }
      }
      if (!ok) {
        if (lane == 0) *flag = 1;
      } else {
        float dl = a[0];
#pragma unroll
        for (int c = 1; c < 32; ++c) dl = lane == c ? a[c] : dl;
        const float rd = __frcp_rn(dl);  // 1 / L_{lane, lane}
        float x[32];  // column `lane` of L_bb^-1: L x = e_lane by forward substitution
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) {
          float v = rr == lane ? 1.f : 0.f;
#pragma unroll
          for (int q = 0; q < 31; ++q)
            if (q < rr) v = fmaf(-__shfl_sync(0xFFFFFFFFu, a[q], rr), x[q], v);
          x[rr] = v * __shfl_sync(0xFFFFFFFFu, rd, rr);
        }
        float* dv = dinv + sb * kRsBlk;
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) dv[rr * kRsLd + lane] = x[rr];
      }
    }
    cluster.sync();  // L_bb^-1, or the flag, at the owner
    if (*cluster.map_shared_rank(flag, ob)) {  // the same value in every CTA
      bad = true;
      break;
    }
    const bool t0 = has[0] && own[0] > b, t1 = has[1] && own[1] > b;  // blocks below the diagonal block
    if (t0 || t1) {  // L_ib = M_ib L_bb^-T
      const float4* src = reinterpret_cast<const float4*>(cluster.map_shared_rank(dinv + sb * kRsBlk, ob));
      if (tid < kRsBlk / 4) reinterpret_cast<float4*>(tinv)[tid] = src[tid];
      __syncthreads();
      const int rr = tid >> 4, c2 = tid & 15;
      float a[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (!(s == 0 ? t0 : t1)) continue;
        const float* mr = Ms[s] + rr * lds[s] + 32 * b;
#pragma unroll 8
        for (int q = 0; q < 32; ++q) {
          const float m = mr[q];
          a[s][0] = fmaf(m, tinv[c2 * kRsLd + q], a[s][0]);
          a[s][1] = fmaf(m, tinv[(c2 + 16) * kRsLd + q], a[s][1]);
        }
      }
      __syncthreads();
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (!(s == 0 ? t0 : t1)) continue;
        float* mr = Ms[s] + rr * lds[s] + 32 * b;
        mr[c2] = a[s][0];
        mr[c2 + 16] = a[s][1];
        At[s][c2 * kRsLdAt + rr] = a[s][0];
        At[s][(c2 + 16) * kRsLdAt + rr] = a[s][1];
      }
    }
    cluster.sync();  // the column panel L_jb, j > b, at the blocks' owners
    if (t0 || t1) {
      const int np = (imax - b) * 32;  // the panel's rows this CTA needs (at most 480: one a thread)
      if (tid < np) {
        const int jb = b + 1 + (tid >> 5), rr = tid & 31;
        const float4* src = reinterpret_cast<const float4*>(cluster.map_shared_rank(sm, rs_owner(jb)) + rs_off(jb) +
                                                            rr * rs_ld(jb) + 32 * b);
        float4 v[8];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) v[q4] = src[q4];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          PT[(4 * q4) * kRsLdp + tid] = v[q4].x;
          PT[(4 * q4 + 1) * kRsLdp + tid] = v[q4].y;
          PT[(4 * q4 + 2) * kRsLdp + tid] = v[q4].z;
          PT[(4 * q4 + 3) * kRsLdp + tid] = v[q4].w;
        }
      }
      __syncthreads();
      const int cgi = tid & 127, rg = tid >> 7;  // columns 4 cgi .., rows 8 rg ..
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (!(s == 0 ? t0 : t1) || 4 * cgi >= 32 * (own[s] - b)) continue;
        float acc[8][4];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
#pragma unroll 4
        for (int q = 0; q < 32; ++q) {
          const float4 pv = *reinterpret_cast<const float4*>(PT + q * kRsLdp + 4 * cgi);
          const float4 x0 = *reinterpret_cast<const float4*>(At[s] + q * kRsLdAt + 8 * rg);
          const float4 x1 = *reinterpret_cast<const float4*>(At[s] + q * kRsLdAt + 8 * rg + 4);
          const float xa[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            acc[u][0] = fmaf(xa[u], pv.x, acc[u][0]);
            acc[u][1] = fmaf(xa[u], pv.y, acc[u][1]);
            acc[u][2] = fmaf(xa[u], pv.z, acc[u][2]);
            acc[u][3] = fmaf(xa[u], pv.w, acc[u][3]);
          }
        }
        float* out = Ms[s] + 8 * rg * lds[s] + 32 * (b + 1) + 4 * cgi;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          float4* o = reinterpret_cast<float4*>(out + u * lds[s]);
          float4 v = *o;
          v.x -= acc[u][0];
          v.y -= acc[u][1];
          v.z -= acc[u][2];
          v.w -= acc[u][3];
          *o = v;
        }
      }
      __syncthreads();
    }
  }

  if (!bad) {
    // ---- the two solves, CTA `rank` taking channels rank NCH .. + NCH - 1 of
    // every row: L and the L_bb^-1 are final (read from their owners); no
    // cluster barrier until the end ----
    constexpr int NCH = DH / kRsCluster;  // 16 or 8
    float* Yc = sm + kRsOffB;             // [32 nblk][NCH]: A^T Y, then y, then x
    const int kp = 32 * nblk;
    for (int e = tid; e < kp * NCH; e += kRsThreads) {
      const int row = e / NCH, c = e % NCH;
      float v = 0.f;
      if (row < k) {
        const long long o = static_cast<long long>(row) * DH + rank * NCH + c;
        v = __ldg(Bg + o);
#pragma unroll
        for (int sp = 1; sp < kAtbSplit; ++sp) v += __ldg(Bg + sp * bstride + o);
      }
      Yc[e] = v;
    }
    const int orow = tid / NCH, oc = tid % NCH;  // this thread's output of a 32-row block (if orow < 32)
    const bool active = tid < 32 * NCH;
    float* lbuf = PT;  // pulled rows or columns of L
    // pulls of step b from the owners, every remote load of a thread in flight
    // at once: L_bb^-1 into tinv, and either column block b of the rows below
    // it (lbuf[p][0..31], p < 32 (nblk - 1 - b)) or row block b left of its
    // diagonal block (lbuf[q][0..32 b - 1], row stride 32 b + 4)
    auto pull = [&](int b, bool column) {
      const int ob = rs_owner(b), sb = rs_slot(b);
      const float* ob_sm = cluster.map_shared_rank(sm, ob);
      const int nq = 32 * b, np = 32 * (nblk - 1 - b);
      const int n4 = column ? np * 8 : 32 * (nq / 4);  // at most 3840 = 7.5 a thread
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = tid + u * kRsThreads;
        if (e < n4) {
          if (column) {
            const int p = e >> 3, ib = b + 1 + (p >> 5);
            v[u] = reinterpret_cast<const float4*>(cluster.map_shared_rank(sm, rs_owner(ib)) + rs_off(ib) +
                                                   (p & 31) * rs_ld(ib) + 32 * b)[e & 7];
          } else {
            v[u] = reinterpret_cast<const float4*>(ob_sm + rs_off(b) + (e / (nq / 4)) * rs_ld(b))[e % (nq / 4)];
          }
        }
      }
      const float4 t = tid < kRsBlk / 4 ? reinterpret_cast<const float4*>(ob_sm + kRsOffDinv + sb * kRsBlk)[tid]
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = tid + u * kRsThreads;
        if (e < n4) {
          if (column)
            reinterpret_cast<float4*>(lbuf + (e >> 3) * 32)[e & 7] = v[u];
          else
            reinterpret_cast<float4*>(lbuf + (e / (nq / 4)) * (nq + 4))[e % (nq / 4)] = v[u];
        }
      }
      if (tid < kRsBlk / 4) reinterpret_cast<float4*>(tinv)[tid] = t;
    };
    // block b's 32 x NCH solution in place: z = L_bb^-1 r (forward) or L_bb^-T r (backward)
    auto solve_block = [&](int b, bool transposed) {
      float z = 0.f;
      if (active) {
#pragma unroll 8
        for (int q = 0; q < 32; ++q)
          z = fmaf(transposed ? tinv[q * kRsLd + orow] : tinv[orow * kRsLd + q], Yc[(32 * b + q) * NCH + oc], z);
      }
      __syncthreads();
      if (active) Yc[(32 * b + orow) * NCH + oc] = z;
      __syncthreads();
    };
    // rows p of the update (p < nrows, global row row0 + p) minus their products
    // with block b's solution: coef(p, q) is the factor entry for row p, column q
    // of the block; each thread keeps channel tid % NCH of the solution in registers
    auto update = [&](int b, int row0, int nrows, auto coef) {
      const int c = tid % NCH;
      float z[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) z[q] = Yc[(32 * b + q) * NCH + c];
      for (int p = tid / NCH; p < nrows; p += kRsThreads / NCH) {
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          a0 = fmaf(coef(p, q), z[q], a0);
          a1 = fmaf(coef(p, q + 1), z[q + 1], a1);
          a2 = fmaf(coef(p, q + 2), z[q + 2], a2);
          a3 = fmaf(coef(p, q + 3), z[q + 3], a3);
        }
        Yc[(row0 + p) * NCH + c] -= (a0 + a1) + (a2 + a3);
      }
      __syncthreads();
    };
    // L y = A^T Y, right-looking: y_b = L_bb^-1 r_b, then r_i -= L_ib y_b for the rows below
    for (int b = 0; b < nblk; ++b) {
      pull(b, true);
      __syncthreads();
      solve_block(b, false);
      update(b, 32 * (b + 1), 32 * (nblk - 1 - b), [&](int p, int q) { return lbuf[p * 32 + q]; });
    }
    // L^T x = y, from the last block up: x_b = L_bb^-T y_b, then y_i -= L_bi^T x_b for the rows above
    for (int b = nblk - 1; b >= 0; --b) {
      pull(b, false);
      __syncthreads();
      solve_block(b, true);
      const int ld = 32 * b + 4;
      update(b, 0, 32 * b, [&](int p, int q) { return lbuf[q * ld + p]; });
    }
    for (int e = tid; e < k * NCH; e += kRsThreads)
      Vg[static_cast<long long>(e / NCH) * DH + rank * NCH + e % NCH] = Yc[e];
  } else {
    if (rank == 0 && tid == 0) record_error(KVS_ERR_RANGE);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      if (!has[s]) continue;
      for (int e = tid; e < 32 * DH; e += kRsThreads) {
        const int gr = 32 * own[s] + e / DH;
        if (gr < k) Vg[static_cast<long long>(gr) * DH + e % DH] = 0.f;
      }
    }
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

}  // namespace kvs
