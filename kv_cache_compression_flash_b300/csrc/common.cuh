// Shared device helpers for libkvs: error word, bounded waits, mbarrier, TMA
// and tcgen05 (5th-generation tensor core + tensor memory) wrappers for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvs.h"

namespace kvs {

// ---------------------------------------------------------------------------
// device error word: the first error code any kernel records (0 = none)
// ---------------------------------------------------------------------------
__device__ int g_device_error;

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_device_error, 0, code); }

// Bounds check of a data-dependent index (a gathered token, a stream entry, a
// computed head).  In the checked build (KVS_DEBUG defined) a false condition
// records KVS_ERR_BOUNDS and the caller skips the access; otherwise the
// condition is not evaluated.  Use: if (kvs_in_bounds(i < n)) a[i] = x;
#ifdef KVS_DEBUG
__device__ __forceinline__ bool kvs_in_bounds(const bool ok) {
  if (!ok) record_error(KVS_ERR_BOUNDS);
  return ok;
}
#define KVS_IN_BOUNDS(cond) ::kvs::kvs_in_bounds(cond)
#else
#define KVS_IN_BOUNDS(cond) true
#endif

// true once any kernel gave up on a wait: later CTAs skip their work so a
// broken launch ends quickly instead of timing out wave after wave
__device__ __forceinline__ bool timeout_recorded() {
  return *reinterpret_cast<volatile int*>(&g_device_error) == KVS_ERR_TIMEOUT;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// every wait on another agent gives up after this long and records KVS_ERR_TIMEOUT
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Test hooks (kvs_debug_inject): the wait limit in force, and a fault the
// kernels plant on purpose so that a test can watch a bounded wait run out.
// Read only where a wait has already spun, or once per launch.
__device__ unsigned long long g_wait_limit_ns = kWaitLimitNs;
__device__ int g_debug_fault;

__device__ __forceinline__ uint64_t wait_limit_ns() {
  return *reinterpret_cast<volatile unsigned long long*>(&g_wait_limit_ns);
}

// ---------------------------------------------------------------------------
// 2^x on the FMA pipe, to take part of the softmax exponentials off the
// special-function unit.  Cody and Waite's range reduction (1980): x = n + f
// with n = round(x) and |f| <= 1/2; 2^f by the degree-3 polynomial of relative
// minimax error on [-1/2, 1/2] (coefficients from a Remez exchange,
// kv_cache_compression_flash_b300/exp2_fit.py: max relative error 7.5e-5); 2^n
// by adding n to the exponent field.  x below -125 (and -inf) gives 0: such
// terms are under 2^-125, nothing next to the sums they join.
// ---------------------------------------------------------------------------
constexpr float kExp2C0 = 0x1.fff692p-1f;
constexpr float kExp2C1 = 0x1.62f31ap-1f;
constexpr float kExp2C2 = 0x1.f0de1ap-3f;
constexpr float kExp2C3 = 0x1.c3f76p-5f;

__device__ __forceinline__ float ex2_fma(float x) {
  const float xc = fmaxf(x, -127.f);
  const float t = xc + 12582912.f;       // 1.5 * 2^23: the nearest integer lands in the low mantissa bits
  const float f = xc - (t - 12582912.f);  // exact, |f| <= 1/2
  float p = fmaf(kExp2C3, f, kExp2C2);
  p = fmaf(p, f, kExp2C1);
  p = fmaf(p, f, kExp2C0);
  // (bits(t) << 23) mod 2^32 = n << 23: the exponent bits of t shift out
  const float r = __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
  return x >= -125.f ? r : 0.f;  // keeps the result a normal float
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// when *abort_flag becomes nonzero or after the wait limit (then sets the flag
// and records KVS_ERR_TIMEOUT).  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (timeout_recorded()) {
        *abort_flag = 1;
        return false;
      }
      if (global_timer_ns() - t0 > wait_limit_ns()) {
        *abort_flag = 1;
        record_error(KVS_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// plain bulk copy: both addresses 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory allocation, MMA, loads, fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {  // whole warp
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major operand with the 128-byte swizzle:
// 8-row x 128-byte swizzle atoms stacked every 1024 bytes (SBO), version 1.
// The operand tile must start on a 1024-byte boundary; stepping along K inside
// the 128-byte row is a plain byte offset on the start address.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);       // start address
  d |= static_cast<uint64_t>(16u >> 4) << 16;                // leading byte offset (unused with swizzle)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;              // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;                      // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 x bf16 -> fp32, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                                  // D format f32
         | (1u << 7)                                // A format bf16
         | (1u << 10)                               // B format bf16
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// arrive on `bar` once every tcgen05 op this thread issued so far has completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane; the wait for the
// load sits in the same asm statement so no use can be scheduled before it.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, float (&v)[32]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Split form: the load is issued now and its 32 registers may only be read
// after tmem_wait32() on the same array (the wait takes them as in/out
// operands, so no use can be scheduled before it).  Lets the next chunk's
// load overlap the current chunk's arithmetic.
__device__ __forceinline__ void tmem_issue32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                 "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                 "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// ---------------------------------------------------------------------------
// packed fp32 pairs (one instruction for two lanes of arithmetic) and the
// three-input max
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float* a, float* b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(*a), "=f"(*b) : "l"(v));
}
// a * b + c on both halves, round to nearest
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ---------------------------------------------------------------------------
// fast math on the special-function unit (PTX approximate instructions)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// grid-wide barrier for cooperative launches (all blocks co-resident)
// ---------------------------------------------------------------------------
struct GridSync {
  unsigned int count;
  unsigned int generation;
};

// Returns false (in every thread of the block) when the wait timed out.
__device__ __forceinline__ bool grid_barrier(GridSync* gs, unsigned int nblocks) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    volatile unsigned int* gen = &gs->generation;
    const unsigned int g0 = *gen;
    __threadfence();
    const unsigned int arrived = atomicAdd(&gs->count, 1u) + 1u;
    if (arrived == nblocks) {
      gs->count = 0u;
      __threadfence();
      atomicAdd(&gs->generation, 1u);
    } else {
      const uint64_t t0 = global_timer_ns();
      while (*gen == g0) {
        __nanosleep(64);
        if (global_timer_ns() - t0 > wait_limit_ns()) {
          record_error(KVS_ERR_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: every kernel of the library is launched so
// that it may start while the kernel before it on the stream drains.  A
// kernel calls pdl_wait() before it touches memory the previous kernel may
// still be writing (or reading), and pdl_trigger() to let the next kernel
// launch; both are no-ops when the launch did not ask for this.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// small host helpers
// ---------------------------------------------------------------------------
// Launches `kern` with programmatic stream serialization (and, with cluster
// > 0, as clusters of that many CTAs along x).
template <typename... Params, typename... Args>
inline cudaError_t launch_k(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
}
struct WsCarver {
  char* base;
  size_t used;
  size_t cap;
  template <class T>
  T* take(size_t count) {
    size_t off = (used + 255) & ~static_cast<size_t>(255);
    used = off + count * sizeof(T);
    return reinterpret_cast<T*>(base ? base + off : nullptr);
  }
  bool ok() const { return used <= cap; }
};

}  // namespace kvs

#define KVS_CUDA_TRY(expr)                 \
  do {                                     \
    cudaError_t e_ = (expr);               \
    if (e_ != cudaSuccess) {               \
      (void)cudaGetLastError();            \
      return KVS_ERR_CUDA;                 \
    }                                      \
  } while (0)
