// libkvs.so: host side of the C ABI declared in include/kvs.h.  Validates
// arguments, carves the caller's workspace, encodes TMA tensor maps and
// enqueues the kernels of score.cuh, norms.cuh, alloc.cuh and pack.cuh on the
// caller's stream.  One translation unit, so every kernel shares the device
// error word.
#include <cmath>
#include <cstring>
#include <mutex>

#include "alloc.cuh"
#include "api.cuh"
#include "alloc_cluster.cuh"
#include "common.cuh"
#include "norms.cuh"
#include "pack.cuh"
#include "score.cuh"
#include "decode.cuh"
#include "core.cuh"
#include "sculpt.cuh"

using namespace kvs;

namespace {

constexpr int kVersion = 101;

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

#include "score_host.cuh"

// ---- allocation ---------------------------------------------------------------
int alloc_blocks_max() { return sm_count() * 8; }
constexpr long long kAllocUnitsPerBlock = 2048;

// workspace of the grid allocator for `pools` pools of nb blocks each
size_t alloc_ws_bytes(long long nb, long long pools = 1) {
  WsCarver c{nullptr, 0, 0};
  c.take<AllocHeader>(static_cast<size_t>(pools));
  c.take<unsigned long long>(static_cast<size_t>(pools) * kRadixPasses * kRadixBins);
  c.take<unsigned long long>(static_cast<size_t>(pools * nb));
  c.take<FixCand>(static_cast<size_t>(pools) * kMaxFixRounds * nb);
  return c.used;
}

// The one-cluster allocator, one instantiation per cluster size.
using ClusterAllocFn = void (*)(AllocParams, int);
ClusterAllocFn cluster_alloc_fn(int cl) {
  switch (cl) {
    case 1: return allocate_cluster_kernel<1>;
    case 2: return allocate_cluster_kernel<2>;
    case 4: return allocate_cluster_kernel<4>;
    case 8: return allocate_cluster_kernel<8>;
    case 16: return allocate_cluster_kernel<16>;
    default: return nullptr;
  }
}

cudaLaunchConfig_t cluster_cfg(int cl, size_t smem, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cl));
  cfg.blockDim = dim3(kCAThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Cluster size, units per CTA, candidate capacity and shared memory of the
// one-cluster allocator, or *CL = 0 when the pool does not fit one cluster
// (or no cluster of the needed size can be scheduled).
int plan_cluster_alloc(long long U, int K, int* CL, long long* per, int* cand_cap, size_t* smem) {
  *CL = 0;
  // once per process: the shared-memory cap and which cluster sizes can be
  // scheduled with that much shared memory per CTA
  static size_t cap = 0;
  static bool sched[kCAMaxCluster + 1] = {};
  static std::once_flag once;
  static cudaError_t init_err = cudaSuccess;
  std::call_once(once, [] {
    int dev = 0, max_smem = 0;
    init_err = cudaGetDevice(&dev);
    if (init_err == cudaSuccess)
      init_err = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cap = max_smem > 4096 ? static_cast<size_t>(max_smem - 4096) : 0;  // room for the static part
    for (int cl = 1; init_err == cudaSuccess && cl <= kCAMaxCluster; cl *= 2) {
      ClusterAllocFn fn = cluster_alloc_fn(cl);
      init_err = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (init_err == cudaSuccess)
        init_err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(cap));
      if (init_err != cudaSuccess) break;
      cudaLaunchAttribute attr[1];
      const cudaLaunchConfig_t cfg = cluster_cfg(cl, cap, nullptr, attr);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
      sched[cl] = n > 0;
    }
  });
  if (init_err != cudaSuccess) return KVS_ERR_CUDA;
  const long long items = U * K;
  int cl = 1;
  while (cl < kCAMaxCluster && static_cast<long long>(cl) * 8192 < items) cl *= 2;
  for (; cl <= kCAMaxCluster; cl *= 2) {
    const long long pr = cdiv(U, cl);
    const size_t base = ca_smem_bytes(pr, K, cl, 0);
    if (base + 256 * sizeof(CACand) > cap || !sched[cl]) continue;
    const int cc = static_cast<int>(std::min<size_t>(4096, (cap - base) / sizeof(CACand)));
    *CL = cl;
    *per = pr;
    *cand_cap = cc;
    *smem = ca_smem_bytes(pr, K, cl, cc);
    return KVS_OK;
  }
  return KVS_OK;
}

// ---- packing --------------------------------------------------------------------
StreamPtrs to_ptrs(const kvs_stream_set* s, bool with_counts) {
  StreamPtrs p;
  for (int i = 0; i < 4; ++i) {
    p.codes[i] = s->codes[i];
    p.scales[i] = s->scales[i];
    p.ids[i] = s->unit_ids[i];
    p.goff[i] = s->group_offsets[i];
    p.cap_units[i] = s->cap_units[i];
    p.cap_groups[i] = s->cap_groups[i];
  }
  p.counts = with_counts ? s->counts : nullptr;
  return p;
}

bool streams_ok(const kvs_stream_set* s) {
  if (!s) return false;
  for (int i = 0; i < 4; ++i) {
    if (s->cap_units[i] < 0 || s->cap_groups[i] < 0) return false;
    if (s->cap_units[i] > 0 && (!s->unit_ids[i] || !s->group_offsets[i])) return false;
    if (s->cap_groups[i] > 0 && !s->codes[i]) return false;
    if (s->cap_groups[i] > 0 && i < 3 && !s->scales[i]) return false;
    if ((reinterpret_cast<uintptr_t>(s->codes[i]) & 7u) != 0) return false;
  }
  return true;
}

struct PackWs {
  int* kept;
  int* n_kept;
  long long* chan_base;
  uint32_t* row_counts;  // axis 0: per pool and chunk of kRowChunk units, the units of each stored width
};

size_t carve_pack(int64_t n_pools, int64_t Hkv, int64_t N, int64_t d, int axis, void* base, size_t cap, PackWs* w) {
  WsCarver c{static_cast<char*>(base), 0, cap};
  const int64_t HKV = n_pools * Hkv;  // heads of every pool together
  w->kept = w->n_kept = nullptr;
  w->chan_base = nullptr;
  w->row_counts = nullptr;
  if (axis == 1) {
    w->kept = c.take<int>(static_cast<size_t>(HKV * N));
    w->n_kept = c.take<int>(static_cast<size_t>(HKV));
    w->chan_base = c.take<long long>(static_cast<size_t>(HKV * d));
  } else {
    w->row_counts = c.take<uint32_t>(static_cast<size_t>(n_pools * cdiv(Hkv * N, kRowChunk) * 4));
  }
  return c.used;
}

int pack_shape_ok(int64_t n_pools, int64_t Hkv, int64_t N, int64_t d, int axis) {
  if (n_pools <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || (axis != 0 && axis != 1)) return KVS_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return KVS_ERR_UNSUPPORTED;
  if (Hkv * N >= (1ll << 31) || n_pools * Hkv * N >= (1ll << 40) || n_pools > 65535) return KVS_ERR_UNSUPPORTED;
  // channel plan: per-width unit counts in 16 bits, group counts in 32 bits;
  // the channel kernels' grid rows run over every pool's heads
  if (axis == 1 && (Hkv * d >= (1ll << 16) || Hkv * d * cdiv(N, 64) >= (1ll << 32) || n_pools * Hkv > 65535))
    return KVS_ERR_UNSUPPORTED;
  return KVS_OK;
}

template <class F>
cudaError_t set_cluster_attrs(F fn) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <class F, class... A>
cudaError_t launch_cluster(F fn, dim3 grid, int cl, int threads, size_t smem, cudaStream_t st, A... args) {
  return launch_k(fn, grid, dim3(static_cast<unsigned>(threads)), smem, st, cl, args...);
}

template <int DH>
int pack_dh(const uint16_t* X, int64_t n_pools, int64_t Hkv, int64_t N, int axis, const uint8_t* bits,
            const uint8_t* keep, const kvs_stream_set* s, const PackWs& w, cudaStream_t st, bool dequant, float* out) {
  const int hkv = static_cast<int>(Hkv);
  const unsigned gy = static_cast<unsigned>(n_pools * Hkv);  // channel kernels: every pool's heads
  if (axis == 0) {
    // per chunk of kRowChunk units, the count of each width; then one CTA per chunk, in unit order
    const long long U = Hkv * N;
    const StreamPtrs sp = to_ptrs(s, !dequant);
    const int n_chunks = static_cast<int>(cdiv(U, kRowChunk));
    const dim3 grid(static_cast<unsigned>(n_chunks), static_cast<unsigned>(n_pools));
    KVS_CUDA_TRY(launch_k(rows_count_kernel, grid, dim3(kRowThreads), 0, st, 0, bits, U, n_chunks, w.row_counts));
    if (dequant)
      KVS_CUDA_TRY(launch_k(dequant_rows_kernel<DH>, grid, dim3(kRowThreads), 0, st, 0, sp, bits, U, n_chunks,
                            static_cast<const uint32_t*>(w.row_counts), out));
    else
      KVS_CUDA_TRY(launch_k(pack_rows_kernel<DH>, grid, dim3(kRowThreads), 0, st, 0, X, bits, U, n_chunks,
                            static_cast<const uint32_t*>(w.row_counts), sp));
  } else {
    const StreamPtrs sp = to_ptrs(s, !dequant);
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
      err = set_cluster_attrs(channels_plan_kernel<64>);
      if (err == cudaSuccess) err = set_cluster_attrs(channels_plan_kernel<128>);
      if (err == cudaSuccess) err = allow_smem(pack_channels_kernel<64>, chan_pack_smem<64>());
      if (err == cudaSuccess) err = allow_smem(pack_channels_kernel<128>, chan_pack_smem<128>());
    });
    if (err != cudaSuccess) return KVS_ERR_CUDA;
    const int cl = static_cast<int>(std::min<int64_t>(Hkv, 16));
    KVS_CUDA_TRY(launch_cluster(channels_plan_kernel<DH>, dim3(static_cast<unsigned>(cl * n_pools)), cl, kPlanThreads,
                                0, st, keep, static_cast<int>(N), hkv, bits, w.kept, w.n_kept, w.chan_base, sp,
                                dequant ? 0 : 1));
    constexpr int TG = chan_groups_per_cta<DH>();
    if (dequant) {
      const dim3 grid(static_cast<unsigned>(cdiv(N, 64 * TG) + 1), gy);
      KVS_CUDA_TRY(launch_k(dequant_channels_kernel<DH>, grid, dim3(kChanThreads), 0, st, 0, sp, static_cast<int>(N),
                            bits, w.chan_base, w.kept, w.n_kept, out, hkv));
    } else {
      const dim3 grid(static_cast<unsigned>(cdiv(cdiv(N, 64), TG)), gy);
      KVS_CUDA_TRY(launch_k(pack_channels_kernel<DH>, grid, dim3(kChanThreads), chan_pack_smem<DH>(), st, 0, X,
                            static_cast<int>(N), bits, w.chan_base, w.kept, w.n_kept, sp, hkv));
    }
  }
  return KVS_OK;
}

int pack_common(const uint16_t* X, int64_t n_pools, int64_t Hkv, int64_t N, int64_t d, int axis, const uint8_t* bits,
                const uint8_t* keep, const kvs_stream_set* s, void* ws, size_t ws_bytes, void* stream,
                bool dequant, float* out) {
  int rc = pack_shape_ok(n_pools, Hkv, N, d, axis);
  if (rc) return rc;
  if (!bits || !streams_ok(s) || (axis == 1 && !keep) || (dequant ? !out : !X)) return KVS_ERR_INVALID_ARG;
  if (!dequant && !s->counts) return KVS_ERR_INVALID_ARG;
  if (X && !aligned16(X)) return KVS_ERR_INVALID_ARG;
  if (out && !aligned16(out)) return KVS_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i) {  // the code blocks are written and read 16 bytes at a time
    if (!aligned16(s->codes[i])) return KVS_ERR_INVALID_ARG;
    // a stored token has d / 64 groups: entry k's groups must fit the group arrays
    if (axis == 0 && s->cap_groups[i] < s->cap_units[i] * (d / 64)) return KVS_ERR_INVALID_ARG;
  }
  PackWs w;
  if (carve_pack(n_pools, Hkv, N, d, axis, ws, ws_bytes, &w) > ws_bytes || !ws) return KVS_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return KVS_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  rc = d == 64 ? pack_dh<64>(X, n_pools, Hkv, N, axis, bits, keep, s, w, st, dequant, out)
               : pack_dh<128>(X, n_pools, Hkv, N, axis, bits, keep, s, w, st, dequant, out);
  if (rc) return rc;
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

// cluster size for column reductions over `rows` rows per group: about
// kColRowsPerCta rows a CTA, at most 16 CTAs
constexpr long long kColRowsPerCta = 2048;
int colsq_cluster(long long rows) {
  int cl = 1;
  while (cl < 16 && static_cast<long long>(cl) * kColRowsPerCta < rows) cl *= 2;
  return cl;
}

int launch_colsq(const uint16_t* A, long long rows_a, const uint8_t* keep, const uint16_t* B, long long rows_b,
                 int64_t groups, int64_t d, int mode, float scale, float* out, cudaStream_t st, float* out2 = nullptr) {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = set_cluster_attrs(colsq_cluster_kernel<64, false>);
    if (err == cudaSuccess) err = set_cluster_attrs(colsq_cluster_kernel<128, false>);
    if (err == cudaSuccess) err = set_cluster_attrs(colsq_cluster_kernel<64, true>);
    if (err == cudaSuccess) err = set_cluster_attrs(colsq_cluster_kernel<128, true>);
    if (err == cudaSuccess) err = allow_smem(colsq_cluster_kernel<64, false>, col_ring_bytes<64>());
    if (err == cudaSuccess) err = allow_smem(colsq_cluster_kernel<128, false>, col_ring_bytes<128>());
    if (err == cudaSuccess) err = allow_smem(colsq_cluster_kernel<64, true>, col_ring_bytes<64>());
    if (err == cudaSuccess) err = allow_smem(colsq_cluster_kernel<128, true>, col_ring_bytes<128>());
  });
  if (err != cudaSuccess) return KVS_ERR_CUDA;
  const int cl = colsq_cluster(std::max(rows_a, rows_b));
  const dim3 grid(static_cast<unsigned>(cl), static_cast<unsigned>(groups));
  const int ra = static_cast<int>(rows_a), rb = static_cast<int>(rows_b);
  const bool stats = mode == kColChannelStats;
  cudaError_t e;
  const size_t sm64 = col_ring_bytes<64>(), sm128 = col_ring_bytes<128>();
  if (d == 64)
    e = stats ? launch_cluster(colsq_cluster_kernel<64, true>, grid, cl, kColThreads, sm64, st, A, ra, keep, B, rb,
                               mode, scale, out, out2)
              : launch_cluster(colsq_cluster_kernel<64, false>, grid, cl, kColThreads, sm64, st, A, ra, keep, B, rb,
                               mode, scale, out, out2);
  else
    e = stats ? launch_cluster(colsq_cluster_kernel<128, true>, grid, cl, kColThreads, sm128, st, A, ra, keep, B, rb,
                               mode, scale, out, out2)
              : launch_cluster(colsq_cluster_kernel<128, false>, grid, cl, kColThreads, sm128, st, A, ra, keep, B, rb,
                               mode, scale, out, out2);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return KVS_ERR_CUDA;
  }
  return KVS_OK;
}
}  // namespace

// =============================================================================
// C ABI
// =============================================================================
extern "C" {

const char* kvs_status_string(int status) {
  switch (status) {
    case KVS_OK: return "KVS_OK";
    case KVS_ERR_INVALID_ARG: return "KVS_ERR_INVALID_ARG";
    case KVS_ERR_UNSUPPORTED: return "KVS_ERR_UNSUPPORTED";
    case KVS_ERR_RANGE: return "KVS_ERR_RANGE";
    case KVS_ERR_CUDA: return "KVS_ERR_CUDA";
    case KVS_ERR_TIMEOUT: return "KVS_ERR_TIMEOUT";
    case KVS_ERR_WORKSPACE: return "KVS_ERR_WORKSPACE";
    case KVS_ERR_BOUNDS: return "KVS_ERR_BOUNDS";
    default: return "KVS_ERR_UNKNOWN";
  }
}

int kvs_version(void) { return kVersion; }

int kvs_get_device_error(void* stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) {
    (void)cudaGetLastError();
    return KVS_ERR_CUDA;
  }
  int v = 0;
  const int zero = 0;
  KVS_CUDA_TRY(cudaMemcpyFromSymbol(&v, kvs::g_device_error, sizeof(int)));
  KVS_CUDA_TRY(cudaMemcpyToSymbol(kvs::g_device_error, &zero, sizeof(int)));
  return v;
}

namespace {
__global__ void debug_exp2_kernel(const float* __restrict__ x, float* __restrict__ y, const long long n) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    y[i] = ex2_fma(x[i]);
}
}  // namespace

int kvs_debug_exp2(const float* x, float* y, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return KVS_ERR_INVALID_ARG;
  if (n == 0) return KVS_OK;
  const int blocks = static_cast<int>(std::min<long long>(cdiv(n, 256), 1024));
  KVS_CUDA_TRY(launch_k(debug_exp2_kernel, dim3(blocks), dim3(256), 0, as_stream(stream), 0, x, y,
                        static_cast<long long>(n)));
  return KVS_OK;
}

int kvs_debug_inject(uint32_t fault, uint64_t wait_limit_ns) {
  if (fault != KVS_DEBUG_NONE && fault != KVS_DEBUG_WITHHOLD_LSE_ARRIVE) return KVS_ERR_INVALID_ARG;
  unsigned long long lim = wait_limit_ns == 0 ? kWaitLimitNs : wait_limit_ns;
  lim = std::min<unsigned long long>(std::max<unsigned long long>(lim, 1000000ull), kWaitLimitNs);
  const int f = static_cast<int>(fault);
  KVS_CUDA_TRY(cudaDeviceSynchronize());
  KVS_CUDA_TRY(cudaMemcpyToSymbol(kvs::g_debug_fault, &f, sizeof(int)));
  KVS_CUDA_TRY(cudaMemcpyToSymbol(kvs::g_wait_limit_ns, &lim, sizeof(lim)));
  KVS_CUDA_TRY(cudaDeviceSynchronize());
  return KVS_OK;
}

size_t kvs_score_workspace_size(int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d, int64_t D,
                                int64_t q_pos0, uint32_t mode) {
  ScorePlan pl;
  if (plan_score(Hq, Hkv, W, N, d, D, q_pos0, mode, &pl) != KVS_OK) return 0;
  ScoreWs w;
  return carve_score(pl, nullptr, 0, &w);
}

int kvs_score_plan_info(int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d, int64_t D, int64_t q_pos0,
                        uint32_t mode, int64_t* info) {
  if (!info) return KVS_ERR_INVALID_ARG;
  ScorePlan pl;
  const int rc = plan_score(Hq, Hkv, W, N, d, D, q_pos0, mode, &pl);
  if (rc) return rc;
  info[0] = pl.kt_chunk;
  info[1] = pl.n_split1;
  info[2] = pl.qt_chunk;
  info[3] = pl.n_split2;
  const int per_col = 1 + (pl.n_split2 > 1 ? 1 : 0);
  const int head = pl.lse_given ? ((pl.want_wt || pl.want_max) ? 1 : 0) : 2;
  info[4] = (pl.want_plus ? 3 : 0) + head + (pl.want_wt ? per_col : 0) + (pl.want_max ? per_col : 0);
  return KVS_OK;
}

int kvs_score_attention(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const uint16_t* h,
                        const uint16_t* W_O, int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d, int64_t D,
                        int64_t q_pos0, uint32_t mode, float* lse, float* w_t, float* s_plus, void* workspace,
                        size_t workspace_bytes, void* stream) {
  KVS_API_ENTRY();
  ScorePlan pl;
  int rc = plan_score(Hq, Hkv, W, N, d, D, q_pos0, mode, &pl);
  if (rc) return rc;
  if (!Q || !K || !lse) return KVS_ERR_INVALID_ARG;
  if (pl.want_wt && !w_t) return KVS_ERR_INVALID_ARG;
  if (pl.want_max && !s_plus) return KVS_ERR_INVALID_ARG;
  if (pl.want_plus && (!V || !h || !W_O)) return KVS_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || (pl.want_plus && (!aligned16(V) || !aligned16(h) || !aligned16(W_O))))
    return KVS_ERR_INVALID_ARG;
  ScoreWs w;
  if (carve_score(pl, workspace, workspace_bytes, &w) > workspace_bytes || !workspace) return KVS_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KVS_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  rc = d == 64 ? score_dh<64>(pl, Q, K, V, h, W_O, lse, w_t, s_plus, w, st)
               : score_dh<128>(pl, Q, K, V, h, W_O, lse, w_t, s_plus, w, st);
  if (rc) return rc;
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

size_t kvs_block_lse_workspace_size(int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d, int64_t q_pos0,
                                    int64_t n_block) {
  ScorePlan pl;
  if (n_block < 1 || plan_score(Hq, Hkv, W, N, d, 0, q_pos0, KVS_MODE_LSE, &pl, n_block) != KVS_OK) return 0;
  ScoreWs w;
  return carve_score(pl, nullptr, 0, &w);
}

int kvs_block_lse(const uint16_t* Q, const uint16_t* K, int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d,
                  int64_t q_pos0, int64_t n_block, float* lse, void* workspace, size_t workspace_bytes,
                  void* stream) {
  KVS_API_ENTRY();
  if (n_block < 1) return KVS_ERR_INVALID_ARG;
  ScorePlan pl;
  int rc = plan_score(Hq, Hkv, W, N, d, 0, q_pos0, KVS_MODE_LSE, &pl, n_block);
  if (rc) return rc;
  if (!Q || !K || !lse) return KVS_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K)) return KVS_ERR_INVALID_ARG;
  ScoreWs w;
  if (carve_score(pl, workspace, workspace_bytes, &w) > workspace_bytes || !workspace) return KVS_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KVS_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  rc = d == 64 ? score_dh<64>(pl, Q, K, nullptr, nullptr, nullptr, lse, nullptr, nullptr, w, st)
               : score_dh<128>(pl, Q, K, nullptr, nullptr, nullptr, lse, nullptr, nullptr, w, st);
  if (rc) return rc;
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

size_t kvs_channel_weights_workspace_size(int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d) {
  (void)Hq, (void)Hkv, (void)W, (void)N, (void)d;
  return 0;  // one cluster per group reduces in shared memory
}


int kvs_channel_weights(const uint16_t* Q, const uint16_t* K, int64_t Hq, int64_t Hkv, int64_t W, int64_t N,
                        int64_t d, float* w_c, void* workspace, size_t workspace_bytes, void* stream) {
  KVS_API_ENTRY();
  (void)workspace, (void)workspace_bytes;
  if (Hq <= 0 || Hkv <= 0 || W <= 0 || N <= 0 || d <= 0 || Hq % Hkv) return KVS_ERR_INVALID_ARG;
  if (!Q || !K || !w_c || !aligned16(Q) || !aligned16(K)) return KVS_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return KVS_ERR_UNSUPPORTED;
  if (Hkv * N >= (1ll << 31) || Hq * W >= (1ll << 31)) return KVS_ERR_UNSUPPORTED;
  const long long rq = (Hq / Hkv) * W;  // the group's query rows are contiguous in Q
  const int rc = launch_colsq(Q, rq, nullptr, K, N, Hkv, d, kColChannelWeight,
                              static_cast<float>(1.0 / std::sqrt(static_cast<double>(d))), w_c, as_stream(stream));
  if (rc) return rc;
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

int kvs_channel_stats(const uint16_t* Q, const uint16_t* K, const uint8_t* keep_bits, int64_t Hq, int64_t Hkv,
                      int64_t W, int64_t N, int64_t d, float* w_c, float* sigma_c, void* stream) {
  KVS_API_ENTRY();
  if (Hq <= 0 || Hkv <= 0 || W <= 0 || N <= 0 || d <= 0 || Hq % Hkv) return KVS_ERR_INVALID_ARG;
  if (!Q || !K || !w_c || !sigma_c || !aligned16(Q) || !aligned16(K)) return KVS_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return KVS_ERR_UNSUPPORTED;
  if (Hkv * N >= (1ll << 31) || Hq * W >= (1ll << 31)) return KVS_ERR_UNSUPPORTED;
  const long long rq = (Hq / Hkv) * W;  // the group's query rows are contiguous in Q
  const int rc = launch_colsq(K, N, keep_bits, Q, rq, Hkv, d, kColChannelStats,
                              static_cast<float>(1.0 / std::sqrt(static_cast<double>(d))), sigma_c, as_stream(stream),
                              w_c);
  if (rc) return rc;
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

size_t kvs_unit_rms_workspace_size(int64_t Hkv, int64_t N, int64_t d, int axis) {
  (void)Hkv, (void)N, (void)d, (void)axis;
  return 0;
}

int kvs_unit_rms(const uint16_t* X, int64_t Hkv, int64_t N, int64_t d, int axis, const uint8_t* keep_bits,
                 float* sigma, void* workspace, size_t workspace_bytes, void* stream) {
  KVS_API_ENTRY();
  (void)workspace, (void)workspace_bytes;
  if (Hkv <= 0 || N <= 0 || d <= 0 || (axis != 0 && axis != 1)) return KVS_ERR_INVALID_ARG;
  if (!X || !sigma || !aligned16(X)) return KVS_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return KVS_ERR_UNSUPPORTED;
  if (Hkv * N >= (1ll << 31)) return KVS_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  const int sms = sm_count();
  if (axis == 0) {
    const long long rows = Hkv * N;
    const int rpb = kNormThreads / (static_cast<int>(d) / 8) * 4;
    const int blocks = static_cast<int>(std::min<long long>(cdiv(rows, rpb), static_cast<long long>(sms) * 8));
    if (d == 64)
      KVS_CUDA_TRY(launch_k(row_rms_kernel<64>, dim3(blocks), dim3(kNormThreads), 0, st, 0, X, static_cast<int>(rows), sigma));
    else
      KVS_CUDA_TRY(launch_k(row_rms_kernel<128>, dim3(blocks), dim3(kNormThreads), 0, st, 0, X, static_cast<int>(rows), sigma));
  } else {
    const int rc = launch_colsq(X, N, keep_bits, nullptr, 0, Hkv, d, kColMaskedRms, 1.f, sigma, st);
    if (rc) return rc;
  }
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

size_t kvs_allocate_workspace_size(int64_t U) {
  (void)U;
  return alloc_ws_bytes(alloc_blocks_max());
}

size_t kvs_allocate_pools_workspace_size(int64_t n_pools, int64_t U) {
  const size_t one = alloc_ws_bytes(alloc_blocks_max());
  if (n_pools <= 1 || U <= 0) return one;
  // the side-by-side grid: at most every block the GPU holds at once, over the pools
  const long long nb = std::max<long long>(1, static_cast<long long>(alloc_blocks_max()) / n_pools);
  return std::max(one, alloc_ws_bytes(nb, n_pools));
}

}  // extern "C"

namespace {
// Width set, step costs and chord slopes of the allocation, from the mask.
// Returns false when the mask allows no width but 0.
bool alloc_widths(uint32_t width_mask, AllocParams* p) {
  std::memset(p, 0, sizeof(*p));
  int nw = 1;
  p->width[0] = 0;
  for (int b : {2, 4, 8, 16})
    if (width_mask & (1u << b)) p->width[nw++] = b;
  p->K = nw - 1;
  if (p->K == 0) return false;
  p->min_cost = 1 << 30;
  for (int k = 0; k < p->K; ++k) {
    const int b0 = p->width[k], b1 = p->width[k + 1];
    p->cost[k] = b1 - b0;
    p->min_cost = std::min(p->min_cost, p->cost[k]);
    p->c[k] = (std::ldexp(1.0, -b0) - std::ldexp(1.0, -b1)) / static_cast<double>(b1 - b0);
  }
  // c_k = (2^(b1-b0) - 1) / ((b1-b0) 2^b1): dyadic unless b1-b0 keeps an odd factor
  p->dyadic = 1;
  for (int k = 0; k < p->K; ++k) {
    const int b0 = p->width[k], b1 = p->width[k + 1], d = b1 - b0;
    unsigned long long num = (1ull << d) - 1ull, den = static_cast<unsigned long long>(d);
    int e = b1;
    for (unsigned long long q = 3; q <= den; q += 2)
      while (den % q == 0 && num % q == 0) {
        den /= q;
        num /= q;
      }
    while ((den & 1ull) == 0ull) {
      den >>= 1;
      ++e;
    }
    if (den != 1ull || num >= (1ull << 16)) {
      p->dyadic = 0;
      break;
    }
    p->n[k] = static_cast<unsigned>(num);
    p->e[k] = e;
  }
  return true;
}

// How a pool of U units is solved: on one cluster (*CL > 0, no workspace) or
// on a cooperative grid of *nb blocks (cached: thetas kept in shared memory).
struct AllocPlan {
  int CL, cand_cap;
  long long per;
  size_t ca_smem;
  long long nb;
  bool cached;
};

int plan_alloc(long long U, int K, AllocPlan* ap) {
  std::memset(ap, 0, sizeof(*ap));
  int rc = plan_cluster_alloc(U, K, &ap->CL, &ap->per, &ap->cand_cap, &ap->ca_smem);
  if (rc) return rc;
  if (ap->CL > 0) return KVS_OK;
  const int sms = sm_count();
  const size_t cache_smem = static_cast<size_t>(kAllocUnitsPerBlock) * K * sizeof(unsigned long long);
  KVS_CUDA_TRY(allow_smem(allocate_kernel<true>, cache_smem));
  int occ_c = 0, occ_u = 0;
  KVS_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_c, allocate_kernel<true>, kAllocThreads, cache_smem));
  KVS_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_u, allocate_kernel<false>, kAllocThreads, 0));
  long long nb = std::max<long long>(1, cdiv(U, kAllocUnitsPerBlock));
  ap->cached = nb <= static_cast<long long>(occ_c) * sms && nb <= alloc_blocks_max();
  if (!ap->cached)
    nb = std::max<long long>(1, std::min<long long>(cdiv(U, kAllocUnitsPerBlock),
                                                    std::min<long long>(static_cast<long long>(std::max(occ_u, 1)) * sms,
                                                                        alloc_blocks_max())));
  ap->nb = nb;
  ap->per = cdiv(U, nb);
  if (ap->per * 16 >= (1ll << 32)) return KVS_ERR_UNSUPPORTED;  // per-block histogram counts are 32-bit
  return KVS_OK;
}

// Several pools too large for one cluster, solved at once: one cooperative
// grid with a block row per pool.  Thetas stay cached in shared memory when
// every pool's blocks fit on the GPU together with their caches, and are
// recomputed from w and sigma in every pass otherwise.  nb = 0: the pools do
// not fit side by side (they then run one after the other).
struct MultiAllocPlan {
  long long nb, per;
  bool cached;
};

int plan_alloc_multi(long long U, int K, long long n_pools, MultiAllocPlan* mp) {
  std::memset(mp, 0, sizeof(*mp));
  const int sms = sm_count();
  const size_t cache_smem = static_cast<size_t>(kAllocUnitsPerBlock) * K * sizeof(unsigned long long);
  KVS_CUDA_TRY(allow_smem(allocate_kernel<true>, cache_smem));
  int occ_c = 0, occ_u = 0;
  KVS_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_c, allocate_kernel<true>, kAllocThreads, cache_smem));
  KVS_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_u, allocate_kernel<false>, kAllocThreads, 0));
  const long long nb_c = std::max<long long>(1, cdiv(U, kAllocUnitsPerBlock));
  if (nb_c * n_pools <= static_cast<long long>(occ_c) * sms) {
    mp->nb = nb_c;
    mp->cached = true;
  } else {
    mp->nb = std::min<long long>(cdiv(U, kAllocThreads), static_cast<long long>(occ_u) * sms / n_pools);
    mp->cached = false;
  }
  if (mp->nb < 1 || mp->nb > 65535) {
    mp->nb = 0;
    return KVS_OK;
  }
  mp->per = cdiv(U, mp->nb);
  if (mp->per * 16 >= (1ll << 32)) mp->nb = 0;  // per-block histogram counts are 32-bit
  return KVS_OK;
}

int allocate_pools(const float* w, const float* sigma, int64_t n_pools, int64_t U, int64_t budget_bits,
                   uint32_t width_mask, uint8_t* bits, void* workspace, size_t workspace_bytes, void* stream) {
  if (U < 0 || budget_bits < 0 || n_pools < 0) return KVS_ERR_INVALID_ARG;
  if ((width_mask & ~KVS_WIDTHS_ALL & ~1u) != 0) return KVS_ERR_INVALID_ARG;
  if (U == 0 || n_pools == 0) return KVS_OK;
  if (!w || !sigma || !bits) return KVS_ERR_INVALID_ARG;
  if (n_pools > 65535 || n_pools * U >= (1ll << 40)) return KVS_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  AllocParams p;
  if (!alloc_widths(width_mask, &p)) {
    KVS_CUDA_TRY(cudaMemsetAsync(bits, 0, static_cast<size_t>(n_pools * U), st));
    return KVS_OK;
  }
  p.w = w;
  p.sigma = sigma;
  p.bits = bits;
  p.U = U;
  p.B = static_cast<unsigned long long>(budget_bits);
  AllocPlan ap;
  int rc = plan_alloc(U, p.K, &ap);
  if (rc) return rc;
  if (ap.CL > 0) {
    // one thread-block cluster per pool holds every item's threshold in
    // shared memory and needs no workspace
    p.per = ap.per;
    KVS_CUDA_TRY(launch_k(cluster_alloc_fn(ap.CL), dim3(static_cast<unsigned>(ap.CL * n_pools)), dim3(kCAThreads),
                          ap.ca_smem, st, ap.CL, p, ap.cand_cap));
    return KVS_OK;
  }
  if (n_pools > 1 && workspace) {
    MultiAllocPlan mp;
    rc = plan_alloc_multi(U, p.K, n_pools, &mp);
    if (rc) return rc;
    if (mp.nb > 0 && alloc_ws_bytes(mp.nb, n_pools) <= workspace_bytes) {
      p.per = mp.per;
      WsCarver c{static_cast<char*>(workspace), 0, workspace_bytes};
      p.hdr = c.take<AllocHeader>(static_cast<size_t>(n_pools));
      p.hist = c.take<unsigned long long>(static_cast<size_t>(n_pools) * kRadixPasses * kRadixBins);
      p.tie_block = c.take<unsigned long long>(static_cast<size_t>(n_pools * mp.nb));
      p.cand = c.take<FixCand>(static_cast<size_t>(n_pools) * kMaxFixRounds * mp.nb);
      KVS_CUDA_TRY(cudaMemsetAsync(p.hdr, 0, static_cast<size_t>(n_pools) * sizeof(AllocHeader), st));
      void* args[] = {&p};
      const dim3 grid(static_cast<unsigned>(mp.nb), static_cast<unsigned>(n_pools));
      if (mp.cached) {
        const size_t smem = static_cast<size_t>(p.per) * p.K * sizeof(unsigned long long);
        KVS_CUDA_TRY(cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(allocate_kernel<true>), grid,
                                                 dim3(kAllocThreads), args, smem, st));
      } else {
        KVS_CUDA_TRY(cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(allocate_kernel<false>), grid,
                                                 dim3(kAllocThreads), args, 0, st));
      }
      return KVS_OK;
    }
  }
  // a cooperative grid per pool, one pool after the other on the stream (they
  // share the workspace): a few thousand units per block with their thetas
  // cached in shared memory (every block co-resident), or, failing that,
  // thetas recomputed from w and sigma in every pass
  const long long nb = ap.nb;
  p.per = ap.per;
  WsCarver c{static_cast<char*>(workspace), 0, workspace_bytes};
  p.hdr = c.take<AllocHeader>(1);
  p.hist = c.take<unsigned long long>(static_cast<size_t>(kRadixPasses) * kRadixBins);
  p.tie_block = c.take<unsigned long long>(static_cast<size_t>(nb));
  p.cand = c.take<FixCand>(static_cast<size_t>(kMaxFixRounds) * nb);
  if (!c.ok() || !workspace) return KVS_ERR_WORKSPACE;
  for (int64_t q = 0; q < n_pools; ++q) {
    p.w = w + q * U;
    p.sigma = sigma + q * U;
    p.bits = bits + q * U;
    KVS_CUDA_TRY(cudaMemsetAsync(p.hdr, 0, sizeof(AllocHeader), st));
    void* args[] = {&p};
    if (ap.cached) {
      const size_t smem = static_cast<size_t>(p.per) * p.K * sizeof(unsigned long long);
      KVS_CUDA_TRY(cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(allocate_kernel<true>),
                                               dim3(static_cast<unsigned>(nb)), dim3(kAllocThreads), args, smem, st));
    } else {
      KVS_CUDA_TRY(cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(allocate_kernel<false>),
                                               dim3(static_cast<unsigned>(nb)), dim3(kAllocThreads), args, 0, st));
    }
  }
  return KVS_OK;
}
}  // namespace

extern "C" {

int kvs_allocate_bits(const float* w, const float* sigma, int64_t U, int64_t budget_bits, uint32_t width_mask,
                      uint8_t* bits, void* workspace, size_t workspace_bytes, void* stream) {
  KVS_API_ENTRY();
  return allocate_pools(w, sigma, 1, U, budget_bits, width_mask, bits, workspace, workspace_bytes, stream);
}

int kvs_allocate_bits_pools(const float* w, const float* sigma, int64_t n_pools, int64_t U, int64_t budget_bits,
                            uint32_t width_mask, uint8_t* bits, void* workspace, size_t workspace_bytes,
                            void* stream) {
  KVS_API_ENTRY();
  return allocate_pools(w, sigma, n_pools, U, budget_bits, width_mask, bits, workspace, workspace_bytes, stream);
}

int kvs_allocate_plan_info(int64_t U, uint32_t width_mask, int64_t* info) {
  if (U < 0 || !info || (width_mask & ~KVS_WIDTHS_ALL & ~1u) != 0) return KVS_ERR_INVALID_ARG;
  info[0] = info[1] = info[2] = 0;
  AllocParams p;
  if (U == 0 || !alloc_widths(width_mask, &p)) return KVS_OK;
  AllocPlan ap;
  const int rc = plan_alloc(U, p.K, &ap);
  if (rc) return rc;
  info[0] = ap.CL;
  info[1] = ap.CL > 0 ? 0 : ap.nb;
  info[2] = ap.CL > 0 ? 0 : static_cast<int64_t>(alloc_ws_bytes(static_cast<int>(ap.nb)));
  return KVS_OK;
}

int kvs_pack_capacity(int64_t Hkv, int64_t N, int64_t d, int axis, int64_t budget_bits, int64_t* cap_units,
                      int64_t* cap_groups) {
  const int rc = pack_shape_ok(1, Hkv, N, d, axis);
  if (rc) return rc;
  if (budget_bits < 0 || !cap_units || !cap_groups) return KVS_ERR_INVALID_ARG;
  const long long U = axis == 0 ? Hkv * N : Hkv * d;
  const long long gpu = axis == 0 ? d / 64 : cdiv(N, 64);
  const int widths[4] = {2, 4, 8, 16};
  for (int i = 0; i < 4; ++i) {
    cap_units[i] = std::min<long long>(U, budget_bits / widths[i]);
    cap_groups[i] = cap_units[i] * gpu;
  }
  return KVS_OK;
}

size_t kvs_pack_workspace_size(int64_t Hkv, int64_t N, int64_t d, int axis) {
  return kvs_pack_pools_workspace_size(1, Hkv, N, d, axis);
}

size_t kvs_pack_pools_workspace_size(int64_t n_pools, int64_t Hkv, int64_t N, int64_t d, int axis) {
  if (pack_shape_ok(n_pools, Hkv, N, d, axis)) return 0;
  PackWs w;
  return carve_pack(n_pools, Hkv, N, d, axis, nullptr, 0, &w);
}

int kvs_quantize_pack(const uint16_t* X, int64_t Hkv, int64_t N, int64_t d, int axis, const uint8_t* bits,
                      const uint8_t* keep_bits, const kvs_stream_set* streams, void* workspace,
                      size_t workspace_bytes, void* stream) {
  KVS_API_ENTRY();
  return pack_common(X, 1, Hkv, N, d, axis, bits, keep_bits, streams, workspace, workspace_bytes, stream, false,
                     nullptr);
}

int kvs_dequantize(const kvs_stream_set* streams, int64_t Hkv, int64_t N, int64_t d, int axis, const uint8_t* bits,
                   const uint8_t* keep_bits, float* out, void* workspace, size_t workspace_bytes, void* stream) {
  KVS_API_ENTRY();
  return pack_common(nullptr, 1, Hkv, N, d, axis, bits, keep_bits, streams, workspace, workspace_bytes, stream, true,
                     out);
}

int kvs_quantize_pack_pools(const uint16_t* X, int64_t n_pools, int64_t Hkv, int64_t N, int64_t d, int axis,
                            const uint8_t* bits, const uint8_t* keep_bits, const kvs_stream_set* streams,
                            void* workspace, size_t workspace_bytes, void* stream) {
  KVS_API_ENTRY();
  return pack_common(X, n_pools, Hkv, N, d, axis, bits, keep_bits, streams, workspace, workspace_bytes, stream, false,
                     nullptr);
}

int kvs_dequantize_pools(const kvs_stream_set* streams, int64_t n_pools, int64_t Hkv, int64_t N, int64_t d, int axis,
                         const uint8_t* bits, const uint8_t* keep_bits, float* out, void* workspace,
                         size_t workspace_bytes, void* stream) {
  KVS_API_ENTRY();
  return pack_common(nullptr, n_pools, Hkv, N, d, axis, bits, keep_bits, streams, workspace, workspace_bytes, stream,
                     true, out);
}

int kvs_threshold_keep(const float* score, int64_t Hkv, int64_t N, float tau, int64_t window,
                       uint32_t keep_width, uint8_t* bits, void* stream) {
  KVS_API_ENTRY();
  if (Hkv <= 0 || N <= 0 || window < 0 || !score || !bits) return KVS_ERR_INVALID_ARG;
  if (keep_width != 2 && keep_width != 4 && keep_width != 8 && keep_width != 16) return KVS_ERR_INVALID_ARG;
  if (Hkv * N >= (1ll << 31)) return KVS_ERR_UNSUPPORTED;
  if (N % 4 == 0 && (!aligned16(score) || (reinterpret_cast<uintptr_t>(bits) & 3u))) return KVS_ERR_INVALID_ARG;
  const long long total = Hkv * N;
  const int blocks = static_cast<int>(std::min<long long>(cdiv(total, 1024), static_cast<long long>(sm_count()) * 8));
  KVS_CUDA_TRY(launch_k(threshold_keep_kernel, dim3(blocks), dim3(256), 0, as_stream(stream), 0, score, total, static_cast<int>(N), tau,
                                                               static_cast<int>(std::min<int64_t>(window, N)),
                                                               static_cast<uint8_t>(keep_width), bits));
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

// ---- TriZone decode attention ------------------------------------------------
size_t kvs_trizone_index_size(int64_t Hkv, int64_t N) {
  if (Hkv <= 0 || N <= 0) return 0;
  return static_cast<size_t>(tz_layout(Hkv, N).total);
}

int kvs_trizone_index(const kvs_stream_set* k_streams, const kvs_stream_set* v_streams, const uint8_t* bits_v,
                      int64_t Hkv, int64_t N, int64_t d, void* index, size_t index_bytes, void* stream) {
  KVS_API_ENTRY();
  if (Hkv <= 0 || N <= 0 || d <= 0 || !bits_v || !index) return KVS_ERR_INVALID_ARG;
  if (!streams_ok(k_streams) || !streams_ok(v_streams) || !k_streams->counts || !v_streams->counts)
    return KVS_ERR_INVALID_ARG;
  if (d != kTzD || Hkv * N >= (1ll << 31) || Hkv * d >= (1ll << 31)) return KVS_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(index) & 255u) || index_bytes < kvs_trizone_index_size(Hkv, N))
    return KVS_ERR_WORKSPACE;
  const TzLayout lay = tz_layout(Hkv, N);
  char* base = static_cast<char*>(index);
  KVS_CUDA_TRY(launch_k(trizone_index_kernel, dim3(static_cast<unsigned>(Hkv)), dim3(1024), 0, as_stream(stream), 0,
                        to_ptrs(k_streams, true), to_ptrs(v_streams, true), bits_v, static_cast<int>(N),
                        static_cast<int>(d), reinterpret_cast<long long*>(base),
                        reinterpret_cast<int*>(base + lay.vstart), reinterpret_cast<uint8_t*>(base + lay.vslot)));
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

// partial records the decode may write: one per (query head, CTA column)
static long long tz_slot_cap(int64_t N, int64_t nc_cap) { return cdiv(N, 64) + cdiv(nc_cap, kTzChunkC); }

size_t kvs_trizone_workspace_size(int64_t Hq, int64_t Hkv, int64_t N, int64_t d, int64_t nc_cap) {
  if (Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || nc_cap < 0) return 0;
  const long long rec = Hq * tz_slot_cap(N, nc_cap);
  return static_cast<size_t>(2 * cdiv(rec * 4, 256) * 256 + cdiv(rec * d * 4, 256) * 256);
}

int kvs_trizone_decode(const uint16_t* q, int64_t Hq, int64_t Hkv, int64_t N, int64_t d,
                       const kvs_stream_set* k_streams, const kvs_stream_set* v_streams, const void* index,
                       const uint16_t* k_new, const uint16_t* v_new, const int32_t* n_new, int64_t nc_cap,
                       float* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  KVS_API_ENTRY();
  if (Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || nc_cap < 0 || !q || !index || !out || !lse)
    return KVS_ERR_INVALID_ARG;
  if (Hq % Hkv) return KVS_ERR_INVALID_ARG;
  if (nc_cap > 0 && (!k_new || !v_new || !n_new)) return KVS_ERR_INVALID_ARG;
  if (!streams_ok(k_streams) || !streams_ok(v_streams)) return KVS_ERR_INVALID_ARG;
  const long long G = Hq / Hkv;
  if (d != kTzD || !(G == 1 || G == 2 || G % 4 == 0) || Hkv * N >= (1ll << 31) || nc_cap >= (1ll << 30))
    return KVS_ERR_UNSUPPORTED;
  for (int i = 0; i < 4; ++i)
    if (!aligned16(k_streams->codes[i]) || !aligned16(v_streams->codes[i]) ||
        (reinterpret_cast<uintptr_t>(v_streams->scales[i]) & 3u))
      return KVS_ERR_INVALID_ARG;
  if (!aligned16(q) || (nc_cap > 0 && (!aligned16(k_new) || !aligned16(v_new)))) return KVS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(index) & 255u)) return KVS_ERR_WORKSPACE;
  const size_t need = kvs_trizone_workspace_size(Hq, Hkv, N, d, nc_cap);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return KVS_ERR_WORKSPACE;
  const int HG = G >= 4 ? 4 : static_cast<int>(G);
  const long long Z = G / HG;
  // flash-decoding split: about two CTAs per SM over the (KV head, head slice) pairs
  const long long per_pair = std::min<long long>(512, std::max<long long>(1, 2LL * sm_count() / (Hkv * Z)));
  const int n_split = static_cast<int>(std::min<long long>(cdiv(N, 64), per_pair));
  const int n_csplit = static_cast<int>(std::min<long long>(cdiv(nc_cap, kTzChunkC), per_pair));
  const int slots = n_split + n_csplit;
  const long long rec_cap = Hq * tz_slot_cap(N, nc_cap);   // the layout of the workspace size
  float* pm = static_cast<float*>(workspace);
  float* pl = reinterpret_cast<float*>(static_cast<char*>(workspace) + cdiv(rec_cap * 4, 256) * 256);
  float* po = reinterpret_cast<float*>(static_cast<char*>(workspace) + 2 * cdiv(rec_cap * 4, 256) * 256);
  const TzLayout lay = tz_layout(Hkv, N);
  const char* ib = static_cast<const char*>(index);
  const long long* hdr = reinterpret_cast<const long long*>(ib);
  const int* vstart = reinterpret_cast<const int*>(ib + lay.vstart);
  const uint8_t* vslot = reinterpret_cast<const uint8_t*>(ib + lay.vslot);
  const dim3 grid(static_cast<unsigned>(slots), static_cast<unsigned>(Hkv), static_cast<unsigned>(Z));
  const float qscale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  const StreamPtrs ks = to_ptrs(k_streams, false), vs = to_ptrs(v_streams, false);
  cudaStream_t st = as_stream(stream);
  const int g_ = static_cast<int>(G), n_ = static_cast<int>(N), ncap = static_cast<int>(nc_cap);
  if (HG == 4)
    KVS_CUDA_TRY(launch_k(trizone_decode_kernel<4>, grid, dim3(kTzThreads), 0, st, 0, q, g_, n_, ks, vs, hdr, vstart,
                          vslot, k_new, v_new, n_new, ncap, n_split, qscale, pm, pl, po));
  else if (HG == 2)
    KVS_CUDA_TRY(launch_k(trizone_decode_kernel<2>, grid, dim3(kTzThreads), 0, st, 0, q, g_, n_, ks, vs, hdr, vstart,
                          vslot, k_new, v_new, n_new, ncap, n_split, qscale, pm, pl, po));
  else
    KVS_CUDA_TRY(launch_k(trizone_decode_kernel<1>, grid, dim3(kTzThreads), 0, st, 0, q, g_, n_, ks, vs, hdr, vstart,
                          vslot, k_new, v_new, n_new, ncap, n_split, qscale, pm, pl, po));
  KVS_CUDA_TRY(launch_k(trizone_combine_kernel, dim3(static_cast<unsigned>(Hq)), dim3(kTzCombineThreads), 0, st, 0,
                        slots, pm, pl, po, out, lse));
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

// ---- KV-CoRE: Gram accumulation and spectrum --------------------------------
static int gram_split(int64_t Hkv, int64_t N) {
  return static_cast<int>(std::max<long long>(1, std::min<long long>(cdiv(N, kGramTile), 2LL * sm_count() / Hkv)));
}

size_t kvs_gram_workspace_size(int64_t Hkv, int64_t N, int64_t d) {
  if (Hkv <= 0 || N <= 0 || d != kGramD) return 0;
  return static_cast<size_t>(gram_split(Hkv, N)) * Hkv * kGramD * kGramD * 4;
}

int kvs_gram(const uint16_t* X, int64_t Hkv, int64_t N, int64_t d, const uint8_t* keep_bits, int accumulate,
             float* G, void* workspace, size_t workspace_bytes, void* stream) {
  KVS_API_ENTRY();
  if (Hkv <= 0 || N <= 0 || d <= 0 || !X || !G) return KVS_ERR_INVALID_ARG;
  if (d != kGramD || Hkv * N >= (1ll << 31)) return KVS_ERR_UNSUPPORTED;
  if (!aligned16(X) || !aligned16(G)) return KVS_ERR_INVALID_ARG;
  const size_t need = kvs_gram_workspace_size(Hkv, N, d);
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return KVS_ERR_WORKSPACE;
  const int ns = gram_split(Hkv, N);
  const int per = static_cast<int>(cdiv(cdiv(N, kGramTile), ns) * kGramTile);
  cudaStream_t st = as_stream(stream);
  KVS_CUDA_TRY(allow_smem(gram_partial_kernel, kGramSmem));
  float* part = static_cast<float*>(workspace);
  KVS_CUDA_TRY(launch_k(gram_partial_kernel, dim3(static_cast<unsigned>(ns), static_cast<unsigned>(Hkv)),
                        dim3(kGramThreads), kGramSmem, st, 0, X, static_cast<int>(N), static_cast<long long>(kGramD),
                        static_cast<long long>(N) * kGramD, keep_bits, per, part));
  const long long per_split = Hkv * kGramD * kGramD;
  KVS_CUDA_TRY(launch_k(gram_reduce_kernel, dim3(static_cast<unsigned>(cdiv(per_split, 256))), dim3(256), 0, st, 0,
                        static_cast<const float*>(part), ns, per_split, accumulate ? 1 : 0, G));
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

int kvs_spectrum(const float* G, int64_t Hkv, int64_t d, float rtol, float* sigma, float* ner, int32_t* rank,
                 void* stream) {
  KVS_API_ENTRY();
  if (Hkv <= 0 || d <= 0 || !G || !sigma || !ner || !rank || !(rtol >= 0.f) || !(rtol < 1.f))
    return KVS_ERR_INVALID_ARG;
  if (d != kGramD) return KVS_ERR_UNSUPPORTED;
  KVS_CUDA_TRY(allow_smem(spectrum_kernel, kSpecSmem));
  KVS_CUDA_TRY(launch_k(spectrum_kernel, dim3(static_cast<unsigned>(Hkv)), dim3(kSpecThreads), kSpecSmem,
                        as_stream(stream), 0, G, rtol, sigma, ner, rank));
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

// ---- KVSculpt: block attention targets, ridge values -----------------------
int kvs_block_attention(const uint16_t* Q, const uint16_t* K, const uint16_t* V, int64_t Hq, int64_t Hkv, int64_t W,
                        int64_t N, int64_t d, int64_t q_pos0, int64_t n_block, float* Y, float* lse, void* stream) {
  KVS_API_ENTRY();
  int rc = validate_shape(Hq, Hkv, W, N, d, q_pos0);
  if (rc) return rc;
  if (n_block < 1 || n_block > N) return KVS_ERR_INVALID_ARG;
  if (!Q || !K || !V || !Y) return KVS_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(Y)) return KVS_ERR_INVALID_ARG;
  // tcgen05: one CTA per 128-row query tile of Gt heads x 128 / Gt positions
  const int G = static_cast<int>(Hq / Hkv);
  const int Gt = G >= 4 ? 4 : G;  // G is 1, 2 or a multiple of 4 (validate_shape)
  const int Pp = 128 / Gt;
  const int n_hc = G / Gt, n_pb = static_cast<int>(cdiv(W, Pp));
  const float c_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  cudaStream_t st = as_stream(stream);
  CUtensorMap mq, mk, mv;
  rc = make_map_3d(&mq, Q, d, W, Hq, 64, Pp, Gt);
  if (!rc) rc = make_map_3d(&mk, K, d, N, Hkv, 64, 128, 1);
  if (!rc) rc = make_map_3d(&mv, V, d, N, Hkv, 64, 128, 1);
  if (rc) return rc;
  const dim3 grid(static_cast<unsigned>(Hkv * n_hc * n_pb));
  const int Wi = static_cast<int>(W), p0 = static_cast<int>(q_pos0), nb = static_cast<int>(n_block);
  // the kernel's register split must fit the registers it is launched with
  // (otherwise the softmax warpgroups would wait for registers forever);
  // checked once per kernel: its attributes do not change
  auto split_fits = [](const void* kern) {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, kern) == cudaSuccess && fa.numRegs * kBtThreads >= kBtRegPool;
  };
  static const bool fits64 = split_fits(reinterpret_cast<const void*>(block_attention_tc_kernel<64>));
  static const bool fits128 = split_fits(reinterpret_cast<const void*>(block_attention_tc_kernel<128>));
  if (!(d == 64 ? fits64 : fits128)) return KVS_ERR_UNSUPPORTED;
  if (d == 64) {
    const size_t smem = sizeof(BtSmem<64>) + 1024;
    KVS_CUDA_TRY(allow_smem(block_attention_tc_kernel<64>, smem));
    KVS_CUDA_TRY(launch_k(block_attention_tc_kernel<64>, grid, dim3(kBtThreads), smem, st, 0, mq, mk, mv, G, Gt, Wi,
                          p0, nb, n_hc, n_pb, c_log2, Y, lse));
  } else {
    const size_t smem = sizeof(BtSmem<128>) + 1024;
    KVS_CUDA_TRY(allow_smem(block_attention_tc_kernel<128>, smem));
    KVS_CUDA_TRY(launch_k(block_attention_tc_kernel<128>, grid, dim3(kBtThreads), smem, st, 0, mq, mk, mv, G, Gt,
                          Wi, p0, nb, n_hc, n_pb, c_log2, Y, lse));
  }
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

namespace {
int ridge_check(int64_t Hkv, int64_t R, int64_t k, int64_t d) {
  if (Hkv <= 0 || R <= 0 || k <= 0 || d <= 0) return KVS_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return KVS_ERR_UNSUPPORTED;
  if (k > kRidgeMaxK || Hkv >= 65536 || Hkv * R * k >= (1ll << 40) || R >= (1ll << 31)) return KVS_ERR_UNSUPPORTED;
  return KVS_OK;
}

// A [Hkv, R, k], then M [kAtbSplit, Hkv, k, k] and B [kAtbSplit, Hkv, k, d], each 256-byte aligned
size_t carve_ridge(int64_t Hkv, int64_t R, int64_t k, int64_t d, void* base, float** A, float** M, float** B) {
  WsCarver c{static_cast<char*>(base), 0, 0};
  *A = c.take<float>(static_cast<size_t>(Hkv * R * k));
  *M = c.take<float>(static_cast<size_t>(kAtbSplit * Hkv * k * k));  // one partial sum per split of R
  *B = c.take<float>(static_cast<size_t>(kAtbSplit * Hkv * k * d));
  return c.used;
}
}  // namespace

size_t kvs_ridge_values_workspace_size(int64_t Hkv, int64_t R, int64_t k, int64_t d) {
  if (ridge_check(Hkv, R, k, d) != KVS_OK) return 0;
  float *A, *M, *B;
  return carve_ridge(Hkv, R, k, d, nullptr, &A, &M, &B);
}

int kvs_ridge_values(const uint16_t* Qt, const uint16_t* Kc, const float* Y, int64_t Hkv, int64_t R, int64_t k,
                     int64_t d, float lam, float* Vc, void* workspace, size_t workspace_bytes, void* stream) {
  KVS_API_ENTRY();
  int rc = ridge_check(Hkv, R, k, d);
  if (rc) return rc;
  if (!(lam > 0.f) || !std::isfinite(lam)) return KVS_ERR_INVALID_ARG;
  if (!Qt || !Kc || !Y || !Vc) return KVS_ERR_INVALID_ARG;
  if (!aligned16(Qt) || !aligned16(Kc) || !aligned16(Y) || !aligned16(Vc)) return KVS_ERR_INVALID_ARG;
  float *A, *M, *B;
  const size_t need = carve_ridge(Hkv, R, k, d, workspace, &A, &M, &B);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return KVS_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  const float c_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  const dim3 gs(static_cast<unsigned>(cdiv(R, 64)), static_cast<unsigned>(Hkv));
  const int Ri = static_cast<int>(R), ki = static_cast<int>(k), di = static_cast<int>(d);
  if (d == 64) {
    KVS_CUDA_TRY(allow_smem(ridge_softmax_kernel<64>, RsCfg<64>::kSmem));
    KVS_CUDA_TRY(launch_k(ridge_softmax_kernel<64>, gs, dim3(kBaThreads), RsCfg<64>::kSmem, st, 0, Qt, Kc, Ri, ki,
                          c_log2, A));
  } else {
    KVS_CUDA_TRY(allow_smem(ridge_softmax_kernel<128>, RsCfg<128>::kSmem));
    KVS_CUDA_TRY(launch_k(ridge_softmax_kernel<128>, gs, dim3(kBaThreads), RsCfg<128>::kSmem, st, 0, Qt, Kc, Ri, ki,
                          c_log2, A));
  }
  const unsigned kt = static_cast<unsigned>(cdiv(k, kAtbTile)), dt = static_cast<unsigned>(cdiv(d, kAtbTile));
  const long long mstride = Hkv * k * k, bstride = Hkv * k * d;  // between the partial sums
  KVS_CUDA_TRY(launch_k(ridge_atb_kernel, dim3(kt * (kt + 1) / 2 + kt * dt, kAtbSplit, static_cast<unsigned>(Hkv)),
                        dim3(256), 0, st, 0, static_cast<const float*>(A), Y, Ri, ki, di, lam, M, mstride, B,
                        bstride));
  const dim3 gsolve(kRsCluster, static_cast<unsigned>(Hkv));  // a cluster of kRsCluster CTAs per head
  if (d == 64) {
    KVS_CUDA_TRY(allow_smem(ridge_solve_cluster_kernel<64>, kRsSmemBytes));
    KVS_CUDA_TRY(launch_k(ridge_solve_cluster_kernel<64>, gsolve, dim3(kRsThreads), kRsSmemBytes, st, kRsCluster,
                          static_cast<const float*>(M), mstride, static_cast<const float*>(B), bstride, ki, Vc));
  } else {
    KVS_CUDA_TRY(allow_smem(ridge_solve_cluster_kernel<128>, kRsSmemBytes));
    KVS_CUDA_TRY(launch_k(ridge_solve_cluster_kernel<128>, gsolve, dim3(kRsThreads), kRsSmemBytes, st, kRsCluster,
                          static_cast<const float*>(M), mstride, static_cast<const float*>(B), bstride, ki, Vc));
  }
  KVS_CUDA_TRY(cudaGetLastError());
  return KVS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// kvs_allocate_bits_static: the allocator with library-owned scratch, for
// callers that cannot allocate device memory themselves.
// ---------------------------------------------------------------------------
// Host code must not pass this name to a kernel: on the host it only stands
// in for the symbol; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_alloc_scratch[KVS_STATIC_ALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxStaticDevices = 64;
std::mutex g_static_scratch_mu;
// per device: the context the address was looked up in, and the address
void* g_static_scratch_ctx[kMaxStaticDevices] = {};
void* g_static_scratch_addr[kMaxStaticDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the scratch array in the current device's context.  It
// is looked up once per (device, context): a context made after
// cudaDeviceReset holds the array at a new address, so a change of context
// triggers a new lookup instead of reusing a dangling pointer.
int static_scratch_address(void** out) {
  int dev = 0;
  KVS_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxStaticDevices) return KVS_ERR_UNSUPPORTED;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (!get_ctx) return KVS_ERR_CUDA;
  CUcontext ctx = nullptr;  // null until the runtime has made a context current on this thread
  if (get_ctx(&ctx) != CUDA_SUCCESS) return KVS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  if (g_static_scratch_addr[dev] == nullptr || ctx == nullptr || g_static_scratch_ctx[dev] != static_cast<void*>(ctx)) {
    void* p = nullptr;
    KVS_CUDA_TRY(cudaGetSymbolAddress(&p, g_static_alloc_scratch));  // makes the primary context current if needed
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return KVS_ERR_CUDA;
    g_static_scratch_addr[dev] = p;
    g_static_scratch_ctx[dev] = static_cast<void*>(ctx);
  }
  *out = g_static_scratch_addr[dev];
  return KVS_OK;
}
}  // namespace

extern "C" int kvs_allocate_bits_static(const float* w, const float* sigma, int64_t U, int64_t budget_bits,
                                        uint32_t width_mask, uint8_t* bits, void* stream) {
  KVS_API_ENTRY();
  if (U < 0 || budget_bits < 0) return KVS_ERR_INVALID_ARG;
  if (kvs_allocate_workspace_size(U) > KVS_STATIC_ALLOC_SCRATCH_BYTES) return KVS_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = static_scratch_address(&scratch);
  if (rc) return rc;
  // the allocator zeroes its own header on the stream before its kernel runs
  return kvs_allocate_bits(w, sigma, U, budget_bits, width_mask, bits, scratch, KVS_STATIC_ALLOC_SCRATCH_BYTES,
                           stream);
}
