/*
 * kvs.h - C ABI of libkvs.so: attention-derived importance scoring and
 * rate-distortion compression of a prefilled KV cache, for NVIDIA B300 (sm_103a).
 *
 * Sources (web summaries of the papers; section as printed there):
 *   [RDKV]     "RDKV - Asignacion de Bits de Tasa-Distorsion para Eviccion y
 *              Cuantizacion Conjunta de la Cache KV" (gist.science 2605.08317)
 *   [KVzap]    "KVzap - Poda del KV Cache Rapida, Adaptativa y Fiel"
 *              (gist.science 2601.07891)
 *   [KVSculpt] "KVSculpt: KV Cache Compression as Distillation"
 *              (gist.science 2603.27819)
 *
 * Conventions shared by every call
 *  - Tensors are row-major and contiguous.  bf16 data is passed as its 16-bit
 *    patterns (uint16_t).  Shapes:
 *        Q    [Hq,  W, d]  queries of the observation window; row r is at
 *                          absolute position q_pos0 + r
 *        K, V [Hkv, N, d]  the cache; row t is at position t
 *        h    [W, D]       hidden states of the window positions
 *        W_O  [D, Hq*d]    output projection; head hd uses columns hd*d .. hd*d+d-1
 *    Query head hd reads KV head hd / G with G = Hq / Hkv.  A query at
 *    position p sees keys t <= p.  Logits are q.k / sqrt(d).
 *  - Every pointer that is not marked "host" is a DEVICE pointer owned by the
 *    caller.  The library allocates no device memory: scratch space is the
 *    caller's workspace, sized by the matching *_workspace_size() call and
 *    aligned to 256 bytes.  Workspace contents need not be initialised.
 *  - Every call enqueues its kernels on `stream` (a cudaStream_t passed as
 *    void*; NULL = the legacy default stream) and returns without
 *    synchronising.  Outputs are valid once the stream reaches that point.
 *  - Return value: KVS_OK or an error code.  Argument errors are detected on
 *    the host before anything is enqueued.  Data-dependent errors found on
 *    the device (non-finite weights, an fp16 scale overflow, a stream
 *    capacity exceeded, a device wait that timed out) are recorded in a device
 *    error word that kvs_get_device_error() reads; the kernels that detect
 *    them skip the offending writes and return normally.
 *  - Device waits are bounded: a wait that exceeds about two seconds sets
 *    KVS_ERR_TIMEOUT in the error word and the kernel returns.
 *  - Supported: d in {64, 128}; G in {1, 2} or a positive multiple of 4;
 *    0 <= q_pos0 and q_pos0 + W <= N; N, W >= 1; N < 2^31; Hkv*N < 2^31.
 */
#ifndef KVS_H_
#define KVS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define KVS_OK               0
#define KVS_ERR_INVALID_ARG  1  /* null pointer, negative or inconsistent size */
#define KVS_ERR_UNSUPPORTED  2  /* shape outside the supported set */
#define KVS_ERR_RANGE        3  /* non-finite / negative weight, fp16 scale overflow, capacity */
#define KVS_ERR_CUDA         4  /* a CUDA runtime call failed */
#define KVS_ERR_TIMEOUT      5  /* a bounded device wait ran out */
#define KVS_ERR_WORKSPACE    6  /* workspace too small or misaligned */
#define KVS_ERR_BOUNDS       7  /* bounds-checked build only (libkvs_debug.so, compiled with
                                   KVS_DEBUG): a data-dependent index fell outside its array;
                                   the access was skipped */

/* Human-readable name of a status code (static string). */
const char* kvs_status_string(int status);

/* Library ABI version (major*100 + minor). */
int kvs_version(void);

/* Reads and clears the device error word after synchronising `stream`.
 * Returns KVS_OK when no kernel recorded an error since the last call,
 * else the first recorded code; KVS_ERR_CUDA if the read itself failed. */
int kvs_get_device_error(void* stream);

/* Test hook for failure handling; the papers have no counterpart.  Plants a
 * fault in later launches so that a test can watch a bounded device wait run
 * out, and shortens the wait limit so that it runs out quickly:
 *   fault = KVS_DEBUG_WITHHOLD_LSE_ARRIVE: in each pass-1 CTA the MMA issuer
 *           withholds the arrive that hands its first logit tile to the
 *           reducers, whose wait then times out (KVS_ERR_TIMEOUT in the error
 *           word; the CTA drains its copies and MMAs, frees its tensor memory
 *           and returns; later kernels of the call skip their work);
 *   fault = KVS_DEBUG_NONE: no fault;
 *   wait_limit_ns = 0 restores the default limit (2 s); otherwise it is
 *           clamped to [1 ms, 2 s].
 * Synchronous (waits for the device); returns KVS_ERR_CUDA if the update fails.
 * Reset with kvs_debug_inject(KVS_DEBUG_NONE, 0) before normal use. */
#define KVS_DEBUG_NONE 0u
#define KVS_DEBUG_WITHHOLD_LSE_ARRIVE 1u
int kvs_debug_inject(uint32_t fault, uint64_t wait_limit_ns);

/* Test hook; the papers have no counterpart.  y[i] = the library's FMA-pipe
 * 2^x[i] (Cody-Waite reduction and a degree-3 minimax polynomial, relative
 * error below 1e-4; 0 for x < -125), the routine that takes part of the
 * softmax exponentials off the special-function unit.  x, y: device float [n]. */
int kvs_debug_exp2(const float* x, float* y, int64_t n, void* stream);

/* ---- importance scoring ------------------------------------------------ */
#define KVS_MODE_LSE         1u  /* lse[Hq, W]  = ln sum_{t<=p_r} exp(s_{r,t})         [KVSculpt §2, LSE term] */
#define KVS_MODE_RDKV_WT     2u  /* w_t[Hkv, N] = sum over the group's heads and window rows of a_{r,t}
                                                                                     [RDKV §2.1, w_t] */
#define KVS_MODE_KVZIP       4u  /* s_plus[Hkv, N] = max over heads and rows of a_{r,t}  [KVzap §2.1, KVzip] */
#define KVS_MODE_KVZIP_PLUS  8u  /* s_plus[Hkv, N] = max_heads max_r a^h_{r,t} |h_r| / |W_O^h v_t|
                                                                                     [KVzap §2.1, KVzip+] */
#define KVS_MODE_LSE_GIVEN  16u  /* lse is an INPUT (from an earlier call): pass 1 is skipped and pass 2
                                    reuses it.  Lets a caller time or schedule the two passes apart. */

/* Bytes of workspace kvs_score_attention needs for these sizes and mode. */
size_t kvs_score_workspace_size(int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d,
                                int64_t D, int64_t q_pos0, uint32_t mode);

/* Attention-derived scores of a prefilled cache, without materialising the
 * attention matrix.  Pass 1 computes every window row's log-sum-exp; pass 2
 * recomputes the probabilities a = exp(s - lse) and reduces them per key.
 *   mode    : KVS_MODE_LSE is implied; add KVS_MODE_RDKV_WT and at most one of
 *             KVS_MODE_KVZIP / KVS_MODE_KVZIP_PLUS; with KVS_MODE_LSE_GIVEN the
 *             lse buffer is read instead of written.
 *   Q, K    : bf16, required.  V, h, W_O: bf16, required for KVZIP_PLUS only
 *             (D = hidden size, ignored otherwise).  Every one of them
 *             16-byte aligned.
 *   lse     : float [Hq, W], natural log, required.
 *   w_t     : float [Hkv, N], required with RDKV_WT, else may be NULL.
 *   s_plus  : float [Hkv, N], required with KVZIP or KVZIP_PLUS.  Keys no
 *             query sees get w_t = 0 and s_plus = 0.
 * Deterministic: the same inputs give the same bits. */
int kvs_score_attention(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                        const uint16_t* h, const uint16_t* W_O,
                        int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d, int64_t D,
                        int64_t q_pos0, uint32_t mode,
                        float* lse, float* w_t, float* s_plus,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Host-only: how kvs_score_attention splits its work for these sizes and
 * mode (same rules as the call itself).  info: host int64[5] =
 *   {key tiles per pass-1 CTA, pass-1 splits, query tiles per pass-2 CTA,
 *    pass-2 splits, kernels the call launches}. */
int kvs_score_plan_info(int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d, int64_t D,
                        int64_t q_pos0, uint32_t mode, int64_t* info);

/* ---- block LSE ------------------------------------------------------------ */
/* The row log-sum-exp over a leading block of keys   [KVSculpt §2: the LSE
 * term of the loss matches the attention mass of the compressed block, the
 * zone [0, N - m) of a cache whose last m tokens are retained]:
 *     lse[hd, r] = ln sum_{t < n_block, t <= q_pos0 + r} exp(s_{r,t})
 * with the keys K[g, 0 .. n_block) of the [Hkv, N, d] cache (each head's rows
 * stay at their place: no copy of the block is needed).  Queries at or after
 * n_block see the whole block.  1 <= n_block <= N; other arguments, layouts
 * and errors as kvs_score_attention with KVS_MODE_LSE (whose result this is
 * for n_block = N). */
size_t kvs_block_lse_workspace_size(int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d, int64_t q_pos0,
                                    int64_t n_block);
int kvs_block_lse(const uint16_t* Q, const uint16_t* K, int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d,
                  int64_t q_pos0, int64_t n_block, float* lse, void* workspace, size_t workspace_bytes,
                  void* stream);

/* Channel distortion weights  w_c[g, c] = |Q_{:,c}| |K_{:,c}| / sqrt(d)   [RDKV §2.1, w_c]
 * The query column stacks the G heads' W window rows of group g; the key
 * column spans all N tokens of KV head g.  w_c: float [Hkv, d]. */
size_t kvs_channel_weights_workspace_size(int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d);
int kvs_channel_weights(const uint16_t* Q, const uint16_t* K,
                        int64_t Hq, int64_t Hkv, int64_t W, int64_t N, int64_t d,
                        float* w_c, void* workspace, size_t workspace_bytes, void* stream);

/* Per-unit RMS sigma_u, the scale of a unit in the RD objective   [RDKV §2.1]
 *   axis 0: unit = token row,  sigma[g*N + t] = sqrt(mean_c X[g,t,c]^2)      (V cache)
 *   axis 1: unit = channel,    sigma[g*d + c] = sqrt(mean_{t kept} X[g,t,c]^2) (K cache)
 *           token t of head g is kept iff keep_bits[g*N + t] != 0 (stage 2's
 *           V widths; stage 3 allocates K over kept tokens only [RDKV §2.2]);
 *           keep_bits NULL keeps every token; a head keeping none gives 0. */
size_t kvs_unit_rms_workspace_size(int64_t Hkv, int64_t N, int64_t d, int axis);
int kvs_unit_rms(const uint16_t* X, int64_t Hkv, int64_t N, int64_t d, int axis,
                 const uint8_t* keep_bits, float* sigma,
                 void* workspace, size_t workspace_bytes, void* stream);

/* Stage 3's two channel quantities from ONE read of the keys: w_c as
 * kvs_channel_weights computes it (every token of K) and sigma_c as
 * kvs_unit_rms(K, axis 1, keep_bits) computes it (the kept tokens)
 * [RDKV §2.1 w_c; §2.2 stage 3 over the retained tokens].  keep_bits NULL
 * keeps every token.  w_c, sigma_c: float [Hkv, d].  No workspace. */
int kvs_channel_stats(const uint16_t* Q, const uint16_t* K, const uint8_t* keep_bits, int64_t Hq, int64_t Hkv,
                      int64_t W, int64_t N, int64_t d, float* w_c, float* sigma_c, void* stream);

/* ---- bit allocation ---------------------------------------------------- */
/* Width set as a bit mask: bit b set <=> width b allowed.  Width 0 (evict) is
 * always allowed.  Allowed widths: 2, 4, 8, 16. */
#define KVS_WIDTHS_ALL  ((1u << 2) | (1u << 4) | (1u << 8) | (1u << 16))
#define KVS_WIDTHS_KEEP_OR_EVICT  (1u << 16)

size_t kvs_allocate_workspace_size(int64_t U);
/* Workspace bytes that let kvs_allocate_bits_pools solve n_pools pools of U
 * units side by side (never less than kvs_allocate_workspace_size(U)). */
size_t kvs_allocate_pools_workspace_size(int64_t n_pools, int64_t U);

/* min sum_u w_u sigma_u 2^-b_u  s.t.  sum_u b_u <= budget_bits, b_u in the
 * width set   [RDKV §2.1 objective; §2.2 reverse water-filling / Lagrangian
 * relaxation of the multiple-choice knapsack over {0,2,4,8,16}].
 * key_u = (double)w_u * (double)sigma_u; the Lagrangian moves unit u from
 * width b_k to b_{k+1} at multiplier theta = c_k * key_u (fp64), with c_k the
 * chord slope of 2^-b.  Upgrades are taken in theta-descending order (ties:
 * lower unit, then lower step) while they fit; a budget-fix scan then takes
 * any later upgrade that still fits and whose previous step was taken.
 *   w, sigma : float [U], finite and >= 0 (else KVS_ERR_RANGE in the error word)
 *   bits     : uint8 [U] output widths.
 * Bit-exact and deterministic. */
int kvs_allocate_bits(const float* w, const float* sigma, int64_t U, int64_t budget_bits,
                      uint32_t width_mask, uint8_t* bits,
                      void* workspace, size_t workspace_bytes, void* stream);

/* kvs_allocate_bits over n_pools independent pools of U units each, in one
 * call: pool q is units q*U .. q*U + U-1 of w, sigma and bits, solved on its
 * own with the same budget_bits and width set (one pool = one (layer,
 * sequence) of a batch   [RDKV §2.2: one allocation per cache]).  Results are
 * bit for bit those of n_pools kvs_allocate_bits calls.  Pools that fit one
 * thread-block cluster run side by side on the GPU, one cluster each.  Larger
 * ones run side by side too, as one cooperative grid with a row of blocks per
 * pool, when the workspace holds kvs_allocate_pools_workspace_size(n_pools,
 * U) bytes and the pools' blocks fit on the GPU at once; otherwise they run
 * one after the other on the stream, sharing a workspace of
 * kvs_allocate_workspace_size(U) bytes.  n_pools < 65536. */
int kvs_allocate_bits_pools(const float* w, const float* sigma, int64_t n_pools, int64_t U, int64_t budget_bits,
                            uint32_t width_mask, uint8_t* bits, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Host-only: how a pool of U units is allocated with this width mask.
 * info: host int64[3] = {CTAs of the thread-block cluster that solves the
 * pool without workspace (0: it does not fit one cluster), blocks of the
 * cooperative grid that solves it otherwise (0 with a cluster), workspace
 * bytes that grid uses}.  Queries the current device. */
int kvs_allocate_plan_info(int64_t U, uint32_t width_mask, int64_t* info);

/* kvs_allocate_bits for callers that must not allocate device memory.  The
 * papers have no counterpart: this entry point exists for host code that
 * cannot call cudaMalloc (or any allocating library), e.g. an inference
 * engine that reserves all device memory for its own pool at start-up, or a
 * plug-in that runs where only the engine may allocate.  Instead of a caller
 * workspace it uses one fixed scratch array of KVS_STATIC_ALLOC_SCRATCH_BYTES
 * that lives inside the library; every GPU that loads libkvs.so holds those
 * bytes until the process exits.  Inputs and outputs are as for
 * kvs_allocate_bits, and so are the results (bit for bit).
 *  - The first call on a device looks up the array's device address (once
 *    per device and context, with that device current); make that first call
 *    before any stream capture.  After cudaDeviceReset the next call looks
 *    the address up again in the new context.
 *  - All calls share the one array and it keeps the previous call's
 *    contents; each call clears the part that must start at zero.  Calls
 *    whose kernels overlap on the GPU (different streams, or several host
 *    threads) race on the array: serialise them.
 *  - Returns KVS_ERR_WORKSPACE when this GPU would need more scratch than the
 *    array holds (more than about 300 SMs); other errors as kvs_allocate_bits. */
#define KVS_STATIC_ALLOC_SCRATCH_BYTES (1u << 20)
int kvs_allocate_bits_static(const float* w, const float* sigma, int64_t U, int64_t budget_bits,
                             uint32_t width_mask, uint8_t* bits, void* stream);

/* ---- quantise / pack / dequantise --------------------------------------- */
/* Width-grouped streams, one per width 2, 4, 8, 16 (index 0..3)   [RDKV §2.3, TriZone].
 * A unit is a token row (axis 0, V cache) or a channel over the kept tokens
 * in ascending order (axis 1, K cache).  Its elements form groups of 64; a
 * short last group is padded with code 0.  Units of one width are stored in
 * ascending unit id (g*N + t, or g*d + c).
 *   codes[i]         : uint8, 8*w bytes per group.  Widths 2/4/8: element e of
 *                      a group is the w-bit two's-complement code q_e in bits
 *                      [w*e, w*e + w) of the group's block, least significant
 *                      first.  Width 16: the raw bf16 values, little-endian.
 *   scales[i]        : fp16 bit patterns, one per group (widths 2/4/8 only):
 *                      s = smallest fp16 >= absmax/qmax, qmax = 2^(w-1)-1,
 *                      q = round-half-even(x / s); x_hat = q * s.
 *   unit_ids[i]      : int32, the unit id of each stored unit.
 *   group_offsets[i] : int64, the first group of each stored unit.
 *   cap_units[i], cap_groups[i] : capacities (host values) of those arrays.
 *   counts           : device int64[8]: units stored per width, then groups
 *                      per width; written by kvs_quantize_pack.
 * Overflowing a capacity records KVS_ERR_RANGE and drops the excess. */
typedef struct kvs_stream_set {
    uint8_t*  codes[4];
    uint16_t* scales[4];
    int32_t*  unit_ids[4];
    int64_t*  group_offsets[4];
    int64_t   cap_units[4];
    int64_t   cap_groups[4];
    int64_t*  counts;
} kvs_stream_set;

/* Every codes[i] pointer must be 16-byte aligned, and for token units (axis
 * 0) every cap_groups[i] must be at least cap_units[i] * d / 64 (a stored
 * token has d / 64 groups); KVS_ERR_INVALID_ARG otherwise. */

/* Host-only: capacities that always suffice for an allocation of at most
 * budget_bits (a unit of width w costs w bits, so at most budget/w units of
 * that width exist).  cap_units, cap_groups: host int64[4]. */
int kvs_pack_capacity(int64_t Hkv, int64_t N, int64_t d, int axis, int64_t budget_bits,
                      int64_t* cap_units, int64_t* cap_groups);

size_t kvs_pack_workspace_size(int64_t Hkv, int64_t N, int64_t d, int axis);

/* Quantise and pack X [Hkv, N, d] (bf16) at the widths `bits` (uint8, one per
 * unit: Hkv*N for axis 0, Hkv*d for axis 1)   [RDKV §2.2 stages 2-3, §2.3].
 * axis 1 needs keep_bits (uint8 [Hkv*N], nonzero = kept); axis 0 ignores it.
 * `streams` is a HOST pointer to a struct of device pointers.  An fp16
 * scale overflow records KVS_ERR_RANGE. */
int kvs_quantize_pack(const uint16_t* X, int64_t Hkv, int64_t N, int64_t d, int axis,
                      const uint8_t* bits, const uint8_t* keep_bits,
                      const kvs_stream_set* streams,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Inverse of kvs_quantize_pack: out float [Hkv, N, d], x_hat = q * s (exact in
 * fp32), width 16 -> the bf16 value, width 0 and tokens not kept -> 0. */
int kvs_dequantize(const kvs_stream_set* streams, int64_t Hkv, int64_t N, int64_t d, int axis,
                   const uint8_t* bits, const uint8_t* keep_bits, float* out,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Pooled variants: n_pools independent caches of one shape, one (layer,
 * sequence) each, packed (or unpacked) by one call   [RDKV §2.2-2.3, applied
 * to every cache of a batch].  X [n_pools, Hkv, N, d]; bits [n_pools, U] (U =
 * Hkv*N for axis 0, Hkv*d for axis 1); keep_bits [n_pools, Hkv*N]; out
 * [n_pools, Hkv, N, d].  cap_units / cap_groups in `streams` are the capacities
 * of ONE pool (kvs_pack_capacity), and every array holds n_pools of them back
 * to back: pool q's codes start at byte q*cap_groups[i]*8*w, its scales at
 * q*cap_groups[i], its unit ids and group offsets at q*cap_units[i] and its
 * counts at counts[8*q].  Within a pool, unit ids and group offsets are local
 * (as in a one-pool set), so pointers offset that way give a stream set that
 * the one-pool calls accept.  Results are bit for bit those of n_pools
 * one-pool calls.  n_pools < 65536 (axis 1: n_pools*Hkv < 65536).
 * Workspace: kvs_pack_pools_workspace_size bytes. */
size_t kvs_pack_pools_workspace_size(int64_t n_pools, int64_t Hkv, int64_t N, int64_t d, int axis);
int kvs_quantize_pack_pools(const uint16_t* X, int64_t n_pools, int64_t Hkv, int64_t N, int64_t d, int axis,
                            const uint8_t* bits, const uint8_t* keep_bits, const kvs_stream_set* streams,
                            void* workspace, size_t workspace_bytes, void* stream);
int kvs_dequantize_pools(const kvs_stream_set* streams, int64_t n_pools, int64_t Hkv, int64_t N, int64_t d, int axis,
                         const uint8_t* bits, const uint8_t* keep_bits, float* out, void* workspace,
                         size_t workspace_bytes, void* stream);

/* ---- threshold pruning with a sliding window ------------------------------ */
/* KVzap's adaptive eviction   [KVzap §2.3: tokens whose score falls below a
 * fixed threshold tau are dropped; the last w tokens are always kept]:
 *   bits[g*N + t] = keep_width  if score[g*N + t] >= tau or t >= N - window
 *                   0           otherwise (evicted)
 *   score      : float [Hkv, N], e.g. s_plus from kvs_score_attention; compare
 *                in the score's own domain (pass exp(tau) to threshold log-scores)
 *   window     : 0 <= window; window >= N keeps everything
 *   keep_width : the width kept tokens get, one of 2, 4, 8, 16
 *   bits       : uint8 [Hkv, N], usable as the widths (and keep mask) of
 *                kvs_quantize_pack.
 * A non-finite score records KVS_ERR_RANGE in the error word; that token is
 * evicted unless the window keeps it. */
int kvs_threshold_keep(const float* score, int64_t Hkv, int64_t N, float tau, int64_t window,
                       uint32_t keep_width, uint8_t* bits, void* stream);

/* ---- TriZone decode attention ------------------------------------------- */
/* One decode step of attention over a compressed pool, with dequantisation
 * inside both products   [RDKV §2.3, TriZone: zone A = the packed K channels
 * and V rows at widths 2/4/8, zone B = the width-16 streams read as raw bf16,
 * zone C = bf16 K/V rows of tokens generated after compression].  For query
 * head hd (KV head g = hd / G):
 *     s_t = q_hd . k_t / sqrt(d) over the kept old tokens t (bits_V > 0; an
 *           evicted token takes no part) and the n_new new tokens,
 *     lse[hd] = ln sum_t exp(s_t),   out[hd] = sum_t exp(s_t - lse[hd]) v_t,
 * where k_t, v_t of an old token are the dequantised values kvs_dequantize
 * returns (a K channel of width 0 contributes zero).  No visible token:
 * out = 0, lse = -inf.
 * Supported: d = 128; G in {1, 2} or a multiple of 4.
 *
 * kvs_trizone_index builds, once per compressed pool (after kvs_quantize_pack
 * of both caches), the per-KV-head lookup the decode kernel reads:
 *     k_streams : K streams (axis 1) and v_streams : V streams (axis 0), as
 *                 written by kvs_quantize_pack, counts included (HOST pointers
 *                 to structs of device pointers)
 *     bits_v    : uint8 [Hkv, N], the V widths the V streams were packed with
 *     index     : device, kvs_trizone_index_size(Hkv, N) bytes, 256-aligned;
 *                 opaque to the caller, valid while the streams are unchanged.
 * Streams that do not match bits_v record KVS_ERR_RANGE; the decode then skips
 * what it cannot locate and stays inside the stream capacities.
 *
 * kvs_trizone_decode:
 *     q        : bf16 [Hq, d], the decode step's queries, 16-byte aligned
 *     k_new, v_new : bf16 [Hkv, nc_cap, d], zone C rows (row j of KV head g at
 *                (g*nc_cap + j)*d); may be NULL when nc_cap = 0
 *     n_new    : DEVICE int32 scalar, the valid zone C rows (0 <= n_new <=
 *                nc_cap; outside that range records KVS_ERR_RANGE and is
 *                clamped).  Read on the device, so a captured CUDA graph
 *                replays across decode steps while zone C grows.
 *     out      : float [Hq, d];  lse : float [Hq] (natural log)
 *     workspace: kvs_trizone_workspace_size(Hq, Hkv, N, d, nc_cap) bytes,
 *                256-aligned.
 * Stream codes must be 16-byte aligned. */
size_t kvs_trizone_index_size(int64_t Hkv, int64_t N);
int kvs_trizone_index(const kvs_stream_set* k_streams, const kvs_stream_set* v_streams, const uint8_t* bits_v,
                      int64_t Hkv, int64_t N, int64_t d, void* index, size_t index_bytes, void* stream);
size_t kvs_trizone_workspace_size(int64_t Hq, int64_t Hkv, int64_t N, int64_t d, int64_t nc_cap);
int kvs_trizone_decode(const uint16_t* q, int64_t Hq, int64_t Hkv, int64_t N, int64_t d,
                       const kvs_stream_set* k_streams, const kvs_stream_set* v_streams, const void* index,
                       const uint16_t* k_new, const uint16_t* v_new, const int32_t* n_new, int64_t nc_cap,
                       float* out, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* ---- KV-CoRE: Gram accumulation, spectrum and NER ------------------------ */
/* The covariance of a cache, updated over its tokens, and the singular values
 * it yields   [KV-CoRE §2: incremental covariance -> singular values and right
 * singular vectors; Eckart-Young-Mirsky; NER].
 *
 * kvs_gram:  G[g] (+)= sum_t x_t x_t^T over the tokens t of KV head g
 *     X        : bf16 [Hkv, N, d], d = 128, 16-byte aligned (a whole cache, or
 *                one block of new tokens when accumulating)
 *     keep_bits: uint8 [Hkv, N] or NULL; a token with keep_bits[t] == 0 is left
 *                out (pass bits_V to take the RDKV kept set)
 *     accumulate: 0 writes G, nonzero adds to it (token-block by token-block
 *                accumulation; the sum over blocks equals the sum over all)
 *     G        : float [Hkv, d, d], 16-byte aligned.  bf16 products are exact
 *                in fp32; the sums are fp32 (tensor cores), adding the token
 *                ranges' partial sums in a fixed order (deterministic).
 *     workspace: kvs_gram_workspace_size(Hkv, N, d) bytes, 16-byte aligned.
 *
 * kvs_spectrum: per KV head, from G[g] (symmetrised):
 *     sigma[g, i] = sqrt(max(lambda_i, 0)) in descending order (fp32 cyclic
 *                   Jacobi, run until the off-diagonal norm is below
 *                   1e-5 |G|_F or stops shrinking, at most 24 sweeps),
 *     rank[g]     = #{i : sigma_i > rtol * sigma_max}, 0 <= rtol < 1,
 *     ner[g]      = exp(-sum_{i<rank} p_i ln p_i) / rank with
 *                   p_i = sigma_i / sum_{j<rank} sigma_j   (the normalised
 *                   effective rank, 1/rank <= ner <= 1; 0 for G = 0).
 * The page gives no NER formula: this is the entropy effective rank over the
 * numerical rank. */
size_t kvs_gram_workspace_size(int64_t Hkv, int64_t N, int64_t d);
int kvs_gram(const uint16_t* X, int64_t Hkv, int64_t N, int64_t d, const uint8_t* keep_bits, int accumulate,
             float* G, void* workspace, size_t workspace_bytes, void* stream);
int kvs_spectrum(const float* G, int64_t Hkv, int64_t d, float rtol, float* sigma, float* ner, int32_t* rank,
                 void* stream);

/* ---- KVSculpt: attention targets and closed-form values ------------------ */
/* kvs_block_attention: the attention output and LSE of the window queries over
 * the leading keys [0, n_block) of each KV head, the targets the compressed
 * pairs of the compression zone are fitted to   [KVSculpt §2, the loss: the
 * output term and the LSE term]:
 *     Y[hd, r, :] = sum_t softmax_t(q_r . k_t / sqrt(d)) v_t,
 *     lse[hd, r]  = ln sum_t exp(q_r . k_t / sqrt(d)),
 * both over t < n_block with t <= q_pos0 + r (queries at or after n_block see
 * the whole block).
 *   Q      : bf16 [Hq, W, d];  K, V : bf16 [Hkv, N, d] (the cache itself; only
 *            rows [0, n_block) of each head are read);
 *   Y      : float [Hq, W, d], written;  lse : float [Hq, W] or NULL.
 * Shapes and errors as kvs_block_lse (1 <= n_block <= N, d in {64, 128});
 * every pointer 16-byte aligned.  No workspace.  Tensor cores: the logits are
 * bf16 products summed in fp32; the weights enter the output product split
 * into two bf16 parts (16 significant bits), so Y keeps fp32-level error; an
 * online softmax over tiles of 128 keys, the tiles taken alternately by two
 * groups of warps whose partial results merge at the end.  Returns
 * KVS_ERR_UNSUPPORTED (nothing launched) if the kernel's register split does
 * not fit the registers it was built to launch with.
 *
 * kvs_ridge_values: per KV head g, the values of k compressed pairs whose keys
 * Kc[g] are fixed   [KVSculpt §2: with the keys fixed the values solve a
 * ridge least-squares problem in closed form]:
 *     A     = softmax_rows(Qt[g] Kc[g]^T / sqrt(d))            [R, k]
 *     Vc[g] = (A^T A + lam I)^-1 A^T Y[g]                      [k, d]
 *   Qt : bf16 [Hkv, R, d], the training queries of each head (Q [Hq, W, d]
 *        is this layout with R = (Hq / Hkv) W);
 *   Kc : bf16 [Hkv, k, d], 1 <= k <= 512;
 *   Y  : float [Hkv, R, d], the targets (Y of kvs_block_attention is this
 *        layout);
 *   lam: > 0 and finite;
 *   Vc : float [Hkv, k, d], written;
 *   workspace: kvs_ridge_values_workspace_size(Hkv, R, k, d) bytes, 256-byte
 *        aligned.
 * The logits as in kvs_block_attention (bf16 products, fp32 sums), then fp32:
 * A, the lower triangle of A^T A + lam I and A^T Y (as two partial sums over
 * the halves of R), and a blocked Cholesky solve on a cluster of 8 CTAs per
 * head (one cluster per head at a time: about 183 KB of shared memory each).  A pivot that is not positive (lam too small for fp32
 * against |A^T A|) records KVS_ERR_RANGE in the error word and sets that
 * head's values to 0.  d in {64, 128}, else KVS_ERR_UNSUPPORTED; k > 512
 * gives KVS_ERR_UNSUPPORTED. */
int kvs_block_attention(const uint16_t* Q, const uint16_t* K, const uint16_t* V, int64_t Hq, int64_t Hkv, int64_t W,
                        int64_t N, int64_t d, int64_t q_pos0, int64_t n_block, float* Y, float* lse, void* stream);
size_t kvs_ridge_values_workspace_size(int64_t Hkv, int64_t R, int64_t k, int64_t d);
int kvs_ridge_values(const uint16_t* Qt, const uint16_t* Kc, const float* Y, int64_t Hkv, int64_t R, int64_t k,
                     int64_t d, float lam, float* Vc, void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KVS_H_ */
