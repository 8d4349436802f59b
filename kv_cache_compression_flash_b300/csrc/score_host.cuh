// Host side of the scoring passes: TMA tensor maps, the work plan (split of
// the query tiles and key tiles over the SMs), workspace carving and the
// launches of score.cuh.  Included once, by kvs.cu, inside its anonymous
// namespace (it uses sm_count, as_stream, aligned16 and cdiv from there).
#pragma once

// ---- TMA tensor maps ---------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D bf16 map over [dim2][dim1][dim0] (dim0 contiguous), 128-byte swizzle,
// out-of-range elements read as zero.
// `rows2` is the row count between consecutive dim2 slices (dim1 when dense).
int make_map_3d(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2, uint32_t box0,
                uint32_t box1, uint32_t box2, uint64_t rows2 = 0) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return KVS_ERR_CUDA;
  const cuuint64_t gdim[3] = {dim0, dim1, dim2};
  const cuuint64_t gstride[2] = {dim0 * 2, dim0 * (rows2 ? rows2 : dim1) * 2};
  const cuuint32_t box[3] = {box0, box1, box2};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstride, box,
                        estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KVS_OK : KVS_ERR_CUDA;
}

// ---- scoring plan -------------------------------------------------------------
constexpr int kGramSlices = 8;

struct ScorePlan {
  ScoreGeom geo;
  int d, D;
  int kt_chunk, n_split1;
  int qt_chunk, n_split2;
  int gram_slice_len;
  bool want_wt, want_max, want_plus, lse_given;
  long long k_rows;  // rows of K per KV head in memory (N unless the keys are a leading block)
};

int validate_shape(int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d, int64_t q_pos0) {
  if (Hq <= 0 || Hkv <= 0 || W <= 0 || N <= 0 || d <= 0 || q_pos0 < 0) return KVS_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || q_pos0 + W > N) return KVS_ERR_INVALID_ARG;
  const int64_t G = Hq / Hkv;
  if (d != 64 && d != 128) return KVS_ERR_UNSUPPORTED;
  // a 128-row query tile packs Gt = min(G, 4) heads of P = 128 / Gt rows:
  // exact only for G in {1, 2, 4} or a multiple of 4
  if (!(G == 1 || G == 2 || G % 4 == 0)) return KVS_ERR_UNSUPPORTED;
  if (N >= (1ll << 31) || Hkv * N >= (1ll << 31) || Hq * W >= (1ll << 31) || Hq >= (1 << 16))
    return KVS_ERR_UNSUPPORTED;
  return KVS_OK;
}

// n_keys > 0: the keys are rows [0, n_keys) of each head of an N-row cache and
// only the row LSE is computed (queries at or after n_keys see every key).
int plan_score(int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d, int64_t D, int64_t q_pos0,
               uint32_t mode, ScorePlan* pl, int64_t n_keys = 0) {
  int st = validate_shape(Hq, Hkv, W, N, d, q_pos0);
  if (st) return st;
  if (n_keys < 0 || n_keys > N || (n_keys > 0 && mode != KVS_MODE_LSE)) return KVS_ERR_INVALID_ARG;
  pl->k_rows = N;
  if (n_keys > 0) N = n_keys;
  if ((mode & ~(KVS_MODE_LSE | KVS_MODE_RDKV_WT | KVS_MODE_KVZIP | KVS_MODE_KVZIP_PLUS | KVS_MODE_LSE_GIVEN)) != 0)
    return KVS_ERR_INVALID_ARG;
  if ((mode & KVS_MODE_KVZIP) && (mode & KVS_MODE_KVZIP_PLUS)) return KVS_ERR_INVALID_ARG;
  if ((mode & KVS_MODE_KVZIP_PLUS) && (D <= 0 || D % 8 != 0)) return KVS_ERR_INVALID_ARG;
  ScoreGeom& g = pl->geo;
  g.Hq = static_cast<int>(Hq);
  g.Hkv = static_cast<int>(Hkv);
  g.G = static_cast<int>(Hq / Hkv);
  g.Gt = g.G <= 4 ? g.G : 4;
  g.P = 128 / g.Gt;
  g.W = static_cast<int>(W);
  g.N = static_cast<int>(N);
  g.q_pos0 = static_cast<int>(q_pos0);
  g.pos_cap = static_cast<int>(N - 1);
  g.n_hc = g.G / g.Gt;
  g.n_pb = static_cast<int>(cdiv(W, g.P));
  g.n_rt = g.Hkv * g.n_hc * g.n_pb;
  g.n_kt = static_cast<int>(cdiv(N, 128));
  g.c_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  pl->d = static_cast<int>(d);
  pl->D = static_cast<int>(D);
  pl->want_wt = (mode & KVS_MODE_RDKV_WT) != 0;
  pl->want_plus = (mode & KVS_MODE_KVZIP_PLUS) != 0;
  pl->want_max = (mode & (KVS_MODE_KVZIP | KVS_MODE_KVZIP_PLUS)) != 0;
  pl->lse_given = (mode & KVS_MODE_LSE_GIVEN) != 0;
  // Split long loops so that the persistent pass-1 CTAs see about eight work
  // items each and the pass-2 CTAs (key-tile pairs) about four; measured on
  // the 8 192-key layer, more splits cost more in pipeline fill and merging
  // than they gain in balance.
  const long long target = static_cast<long long>(sm_count()) * 8, target2 = static_cast<long long>(sm_count()) * 4;
  long long w1 = 0;
  for (int pb = 1; pb < g.n_pb + 1; pb += 2) w1 += pb_nkt(g, std::min(pb, g.n_pb - 1));  // per pair of row tiles
  w1 *= static_cast<long long>(g.Hkv) * g.n_hc;
  pl->kt_chunk = static_cast<int>(std::max<long long>(4, cdiv(w1, target)));
  pl->n_split1 = static_cast<int>(cdiv(pb_nkt(g, g.n_pb - 1), pl->kt_chunk));
  long long w2 = 0;  // query tiles over the key-tile pairs (a pair's list is its first tile's)
  for (int kt = 0; kt < g.n_kt; kt += 2) w2 += kt_nvis(g, kt);
  w2 *= static_cast<long long>(g.Hkv) * g.n_hc;
  pl->qt_chunk = static_cast<int>(std::max<long long>(4, cdiv(w2, target2)));
  pl->n_split2 = static_cast<int>(cdiv(static_cast<long long>(kt_nvis(g, 0)) * g.n_hc, pl->qt_chunk));
  if (pl->n_split2 < 1) pl->n_split2 = 1;
  pl->gram_slice_len = static_cast<int>(cdiv(cdiv(std::max<int64_t>(D, 1), kGramSlices), 32) * 32);
  return KVS_OK;
}

struct ScoreWs {
  float2* part1;
  float* b_plain;
  float* b_scaled;
  float* part_sum;
  float* part_max;
  float* hn;
  float* gram;
  float* vn;
};

size_t carve_score(const ScorePlan& pl, void* base, size_t cap, ScoreWs* w) {
  WsCarver c{static_cast<char*>(base), 0, cap};
  const ScoreGeom& g = pl.geo;
  w->part1 = pl.lse_given ? nullptr : c.take<float2>(static_cast<size_t>(g.n_rt) * pl.n_split1 * 256);
  w->b_plain = (pl.want_wt || (pl.want_max && !pl.want_plus)) ? c.take<float>(static_cast<size_t>(g.n_rt) * 128)
                                                              : nullptr;
  w->b_scaled = pl.want_plus ? c.take<float>(static_cast<size_t>(g.n_rt) * 128) : nullptr;
  const size_t kn = static_cast<size_t>(g.Hkv) * g.N;
  w->part_sum = (pl.want_wt && pl.n_split2 > 1) ? c.take<float>(kn * pl.n_split2) : nullptr;
  w->part_max = (pl.want_max && pl.n_split2 > 1) ? c.take<float>(kn * pl.n_split2) : nullptr;
  w->hn = pl.want_plus ? c.take<float>(g.W) : nullptr;
  w->gram = pl.want_plus ? c.take<float>(static_cast<size_t>(kGramSlices) * g.Hq * pl.d * pl.d) : nullptr;
  w->vn = pl.want_plus ? c.take<float>(static_cast<size_t>(g.Hq) * g.N) : nullptr;
  return c.used;
}

template <class K>
cudaError_t allow_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

constexpr int kStages2 = 4;  // pass-2 query-tile ring
constexpr int kStages1 = 3;  // pass-1 K ring

template <int DH>
int launch_lse(const ScorePlan& pl, const CUtensorMap& mq, const CUtensorMap& mk, float2* part,
               cudaStream_t st) {
  auto kern = lse_pass_kernel<DH, kStages1>;
  // at least half the shared memory: one CTA per SM (it holds all 512 TMEM columns)
  const size_t smem = std::max(sizeof(LseSmem<DH, kStages1>) + 1024, static_cast<size_t>(116 * 1024));
  KVS_CUDA_TRY(allow_smem(kern, smem));
  const int n_pairs = pl.geo.Hkv * pl.geo.n_hc * ((pl.geo.n_pb + 1) / 2);
  const int n_items = n_pairs * pl.n_split1;
  const int grid = std::min(n_items, sm_count());  // persistent: one CTA per SM
  KVS_CUDA_TRY(launch_k(kern, dim3(grid), dim3(kScoreThreads1), smem, st, 0, mq, mk, pl.geo, pl.kt_chunk, pl.n_split1, n_items, part));
  return KVS_OK;
}

template <int DH, int GT, bool MAXM>
int launch_col_gt(const ScorePlan& pl, const CUtensorMap& mq, const CUtensorMap& mk, const float* bvals,
                  const float* vn, float* out, float* part, cudaStream_t st) {
  auto kern = colreduce_pass_kernel<DH, kStages2, GT, MAXM>;
  // at least half the shared memory: one CTA per SM (it holds all 512 TMEM columns)
  const size_t smem = std::max(sizeof(ColSmem<DH, kStages2>) + 1024, static_cast<size_t>(116 * 1024));
  KVS_CUDA_TRY(allow_smem(kern, smem));
  const int n_items = col_pairs(pl.geo) * pl.geo.Hkv * pl.n_split2;
  const int grid = std::min(n_items, sm_count());  // persistent: one CTA per SM
  KVS_CUDA_TRY(launch_k(kern, dim3(grid), dim3(kScoreThreads2), smem, st, 0, mq, mk, pl.geo, pl.qt_chunk, pl.n_split2,
                        n_items, bvals, vn, out, part));
  if (pl.n_split2 > 1) {
    const int total = pl.geo.Hkv * pl.geo.N;
    KVS_CUDA_TRY(launch_k(colreduce_finalize_kernel<MAXM>, dim3(static_cast<unsigned>(cdiv(total, 256))), dim3(256),
                          0, st, 0, pl.geo, pl.qt_chunk, pl.n_split2, part, out));
  }
  return KVS_OK;
}

template <int DH, bool MAXM>
int launch_col(const ScorePlan& pl, const CUtensorMap& mq, const CUtensorMap& mk, const float* bvals,
               const float* vn, float* out, float* part, cudaStream_t st) {
  switch (pl.geo.Gt) {
    case 1: return launch_col_gt<DH, 1, MAXM>(pl, mq, mk, bvals, vn, out, part, st);
    case 2: return launch_col_gt<DH, 2, MAXM>(pl, mq, mk, bvals, vn, out, part, st);
    case 4: return launch_col_gt<DH, 4, MAXM>(pl, mq, mk, bvals, vn, out, part, st);
    default: return KVS_ERR_UNSUPPORTED;
  }
}

template <int DH>
int score_dh(const ScorePlan& pl, const uint16_t* Q, const uint16_t* K, const uint16_t* V, const uint16_t* h,
             const uint16_t* WO, float* lse, float* w_t, float* s_plus, const ScoreWs& w, cudaStream_t st) {
  const ScoreGeom& g = pl.geo;
  CUtensorMap mq, mk;
  int rc = make_map_3d(&mq, Q, DH, g.W, g.Hq, 64, g.P, g.Gt);
  if (rc) return rc;
  rc = make_map_3d(&mk, K, DH, g.N, g.Hkv, 64, 128, 1, static_cast<uint64_t>(pl.k_rows));
  if (rc) return rc;
  if (pl.want_plus) {
    KVS_CUDA_TRY(launch_k(row_norm_kernel, dim3(static_cast<unsigned>(cdiv(g.W, 8))), dim3(256), 0, st, 0, h, g.W,
                          pl.D, w.hn));
    if (DH == kGramD) {
      // W_O^h^T W_O^h on the tensor cores: head h's 128 columns of W_O as a
      // [D, 128] matrix with row stride Hq * 128; the slices' partial Grams
      // are summed by the vnorm kernel in slice order
      KVS_CUDA_TRY(allow_smem(gram_partial_kernel, kGramSmem));
      const int per = static_cast<int>(cdiv(cdiv(pl.D, kGramTile), kGramSlices) * kGramTile);
      KVS_CUDA_TRY(launch_k(gram_partial_kernel, dim3(kGramSlices, g.Hq), dim3(kGramThreads), kGramSmem, st, 0, WO, pl.D,
                            static_cast<long long>(g.Hq) * DH, static_cast<long long>(DH),
                            static_cast<const uint8_t*>(nullptr), per, w.gram));
    } else {
      KVS_CUDA_TRY(launch_k(gram_kernel<DH>, dim3(kGramSlices, g.Hq, DH / 64), dim3(256), 0, st, 0, WO, pl.D, g.Hq,
                            pl.gram_slice_len, w.gram));
    }
    if (DH == kGramD) {  // the quadratic forms on the tensor cores
      CUtensorMap mv;
      rc = make_map_3d(&mv, V, DH, g.N, g.Hkv, 64, 128, 1);
      if (rc) return rc;
      const size_t vs = sizeof(VnSmem) + 1024;
      KVS_CUDA_TRY(allow_smem(vnorm_tc_kernel, vs));
      const int n_tiles = static_cast<int>(cdiv(g.N, 128));
      const int per_head = static_cast<int>(std::max<long long>(1, sm_count() / g.Hq));  // CTAs per head: one wave
      const int tiles_per_cta = static_cast<int>(cdiv(n_tiles, per_head));
      const int n_split = static_cast<int>(cdiv(n_tiles, tiles_per_cta));
      KVS_CUDA_TRY(launch_k(vnorm_tc_kernel, dim3(static_cast<unsigned>(n_split), g.Hq), dim3(kVnThreads), vs, st, 0, mv,
                            static_cast<const float*>(w.gram), kGramSlices, g.Hq, g.G, g.N, tiles_per_cta, w.vn, V));
    } else {
    const size_t vsmem = (static_cast<size_t>(DH) * DH + static_cast<size_t>(DH) * 64) * sizeof(float);
    KVS_CUDA_TRY(allow_smem(vnorm_kernel<DH>, vsmem));
    KVS_CUDA_TRY(launch_k(vnorm_kernel<DH>, dim3(static_cast<unsigned>(cdiv(g.N, 64)), g.Hq), dim3(256), vsmem, st, 0,
                          V, w.gram, kGramSlices, g.Hq, g.G, g.N, w.vn));
    }
  }
  if (pl.lse_given) {
    if (w.b_plain || w.b_scaled) KVS_CUDA_TRY(launch_k(lse_offsets_kernel, dim3(g.n_rt), dim3(128), 0, st, 0, g, lse, w.hn, w.b_plain, w.b_scaled));
  } else {
    rc = launch_lse<DH>(pl, mq, mk, w.part1, st);
    if (rc) return rc;
    KVS_CUDA_TRY(launch_k(lse_finalize_kernel, dim3(g.n_rt), dim3(128), 0, st, 0, g, pl.kt_chunk, pl.n_split1, w.part1, w.hn, lse, w.b_plain,
                                                 w.b_scaled));
  }
  if (pl.want_wt) {
    rc = launch_col<DH, false>(pl, mq, mk, w.b_plain, nullptr, w_t, w.part_sum, st);
    if (rc) return rc;
  }
  if (pl.want_max) {
    rc = launch_col<DH, true>(pl, mq, mk, pl.want_plus ? w.b_scaled : w.b_plain, pl.want_plus ? w.vn : nullptr,
                              s_plus, w.part_max, st);
    if (rc) return rc;
  }
  return KVS_OK;
}

