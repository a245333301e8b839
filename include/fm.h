/*
 * fm.h - masked scaled-dot-product attention for GB300 (sm_103a), C ABI.
 *
 * The mask is given in the column-wise sparse form of FlashMask (page
 * "FlashMask-3: ядро внимания с масками для GPU Hopper и распределённого
 * обучения", introduction and «Ключевые факты»): for every key column j four
 * int32 bounds along the query axis, LTS[j], LTE[j], UTS[j], UTE[j].  Key j is
 * hidden from query row i iff  LTS[j] <= i < LTE[j]  or  UTS[j] <= i < UTE[j].
 * An interval with start >= end hides nothing.  Bound values must lie in
 * [0, Sq]; other values are reported as FM_ERR_BOUNDS (see fm_device_status).
 *
 * The attention is exact (page "FlashAttention-2 ... work partitioning",
 * «Блочная обработка сохраняет общую нормализацию»): a streaming softmax with
 * rescaling, results equal to softmax(scale * Q K^T + mask) V up to
 * floating-point order.  128 x 128 tiles are classified from per-block
 * min/max of the bounds as empty (skipped), full (no mask arithmetic) or
 * partial (element-wise mask), the "fewer non-matmul operations" step of the
 * same page («Три способа повысить загрузку GPU»).
 *
 * Conventions for every entry point:
 *  - Tensors are caller-owned DEVICE pointers.  The library allocates and
 *    frees nothing.  Its scratch is the caller's workspace `ws`, except for
 *    fm_fwd_static, whose scratch is a fixed array of device memory inside
 *    the library (see its declaration below).
 *  - Q, K, V, O, dO, dQ, dK, dV are bf16 in BSHD layout: element (b, s, h, c)
 *    at  b*stride[0] + s*stride[1] + h*stride[2] + c  (elements; the head
 *    dimension is contiguous).  Base pointers must be 16-byte aligned and the
 *    three strides multiples of 8 elements (16 bytes).  Outputs (O, dQ, dK,
 *    dV) whose base is 32-byte aligned and whose strides are multiples of 16
 *    elements are written with 32-byte stores, which is faster; the results
 *    are the same either way.
 *  - Bounds are int32 arrays of shape [B][Hm][Skv], contiguous.  Query head h
 *    reads mask head 0 if Hm == 1, else mask head h.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *    enqueued on it and the call returns without synchronising.  Errors found
 *    on the host (bad shapes, pointers, workspace size) are returned at once
 *    and nothing is enqueued.  Errors found on the device (bound values out of
 *    range, an internal wait that expired) are or-ed into a status word in
 *    `ws`; read it with fm_device_status().  No device code traps or asserts.
 *  - No exception or C++ type crosses this interface.
 */
#ifndef FM_H_
#define FM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FM_OK = 0,
  FM_ERR_INVALID = 1,      /* bad argument: null pointer, shape, stride, alignment, chunk map */
  FM_ERR_BOUNDS = 2,       /* a bound value outside [0, Sq] (device-detected) */
  FM_ERR_UNSUPPORTED = 3,  /* valid but not built: head_dim other than 64 or 128 */
  FM_ERR_WORKSPACE = 4,    /* workspace pointer null/misaligned or smaller than fm_workspace_size */
  FM_ERR_CUDA = 5,         /* a CUDA runtime call failed */
  FM_ERR_TIMEOUT = 6       /* a device-side wait expired; outputs are undefined */
} fm_status;

/* Problem description.  H query heads; Hkv K/V heads (grouped-query
 * attention, listed as a key feature on the ROCm page): Hkv divides H, query
 * head h reads K/V head h / (H / Hkv), and the backward's dK and dV of a K/V
 * head sum over its query heads; Hkv = 0 means Hkv = H (multi-head).  q, o,
 * dO, dQ have H heads, k, v, dK, dV have Hkv.  Hm (mask heads, per query
 * head) is 1 or H; d (head_dim) is 64 or 128; Sq, Skv >= 1.  Strides are in
 * elements, for the (b, s, h) axes.  For the backward pass dO uses o_stride,
 * dQ uses q_stride, dK uses k_stride and dV uses v_stride. */
typedef struct {
  int B, H, Hm, Sq, Skv, d;
  int Hkv;
  int64_t q_stride[3];
  int64_t k_stride[3];
  int64_t v_stride[3];
  int64_t o_stride[3];
} fm_desc;

/* Byte offsets of the regions inside a workspace (all 256-byte aligned).
 * nQ = ceil(Sq/128), nK = ceil(Skv/128).  List entries are
 * (tile_index << 2) | class with class 1 = PARTIAL, 2 = FULL. */
typedef struct {
  size_t status;     /* int32[8]: [0] device status bits, [1] units claimed by the
                        CTAs of the forward or of the dK/dV kernel, [2..3] uint64
                        count of mask slots asked for, [4] units claimed by the
                        CTAs of the dQ kernel; zeroed by every call              */
  size_t summary;    /* int32 [B][Hm][nK][8]: min/max of LTS, LTE, UTS, UTE per k-block */
  size_t table;      /* uint8 [B][Hm][nQ][nK]: 0 EMPTY, 1 PARTIAL, 2 FULL           */
  size_t row_count;  /* int32 [B][Hm][nQ]: non-empty tiles per q-tile row             */
  size_t row_list;   /* int32 [B][Hm][nQ][nK]: ascending k-tiles of each row          */
  size_t col_count;  /* int32 [B][Hm][nK]: non-empty tiles per k-tile column          */
  size_t col_list;   /* int32 [B][Hm][nK][nQ]: ascending q-tiles of each column       */
  size_t fwd_order;  /* int32 [B*H*nP], nP = ceil(nQ/2): forward units u=(b*H+h)*nP+p
                        (q-tiles 2p and 2p+1), longest first                       */
  size_t bwd_order;  /* int32 [B*Hkv*nK]: dK/dV units u=(b*Hkv+hk)*nK+kj, longest
                        first; a unit walks the k-tile column of each of the H/Hkv
                        query heads that read K/V head hk, and costs their sum */
  size_t row_mask;   /* int32 [B][Hm][nQ]: first visibility-mask slot of the row's partial
                        tiles (consecutive in list order), -1 if none              */
  size_t masks;      /* uint8 [cap][128][16], cap = min(B*Hm*nQ*nK, 65536): per partial
                        tile (and the ragged last k-tile) 128 rows of 128 column bits,
                        bit c of 32-bit word w = column 32w+c, set = hidden (the last
                        region).  Rows whose tiles do not fit get row_mask -1 and the
                        forward and dQ kernels build their bits themselves         */
  size_t pair_info;  /* int32 [B][Hm][nP][4]: entries of the pair list, non-empty tiles
                        of q-tile 2p, of q-tile 2p+1, and their sum (forward only) */
  size_t pair_list;  /* int32 [B][Hm][nP][nK]: union of the two q-tiles' non-empty
                        k-tiles, ascending, (kj << 4) | (class_2p << 2) | class_2p+1,
                        a non-empty ragged last k-tile as PARTIAL (forward only)   */
  size_t delta;      /* float [B][H][nQ*128]: D_i = dO_i . O_i, 0 past Sq (backward)  */
  size_t lse_log2;   /* float [B][H][nQ*128]: -LSE_i * log2(e), -inf for rows that see
                        no key and past Sq (backward only)                          */
  size_t row_order;  /* int32 [B*H*nQ]: dQ units u=(b*H+h)*nQ+qi (q-tile rows), longest
                        first (backward only)                                      */
  size_t total;      /* bytes needed */
} fm_ws_layout;

/* Workspace kinds (the `mode` argument below; 0 and 1 may also be read as
 * "for_bwd"): the forward's, the backward's, or a step workspace that holds
 * the regions of both and the analysis of both passes. */
#define FM_WS_FWD 0
#define FM_WS_BWD 1
#define FM_WS_STEP 2

/* Workspace bytes needed by fm_fwd (mode FM_WS_FWD), fm_bwd (FM_WS_BWD), or
 * fm_fwd_planned and fm_bwd_planned (FM_WS_STEP).  Returns 0 for an invalid
 * description or mode. */
size_t fm_workspace_size(const fm_desc* desc, int mode);

/* Fill `out` with the region offsets fm_workspace_size() accounts for;
 * regions a mode does not have are 0. */
fm_status fm_workspace_layout(const fm_desc* desc, int mode, fm_ws_layout* out);

/* Mask analysis into `ws`: validate the bounds (status word), the per-k-block
 * summary, the tile table, the q-tile row lists with the partial tiles' bit
 * masks, and then for FM_WS_FWD the q-tile pair lists and the forward's
 * longest-first unit order, for FM_WS_BWD the k-tile column lists and the
 * longest-first orders of the dK/dV units (columns) and the dQ units (rows),
 * and for FM_WS_STEP all of these.  fm_fwd and fm_bwd run it themselves; a
 * training step runs it once with FM_WS_STEP and then calls fm_fwd_planned
 * and fm_bwd_planned (FlashMask-3 page, introduction: the bounds do not
 * change between the forward and the backward pass).  Zeroes the whole
 * status word first. */
fm_status fm_plan(const fm_desc* desc, const int32_t* lts, const int32_t* lte,
                  const int32_t* uts, const int32_t* ute, void* ws, size_t ws_bytes,
                  int mode, void* stream);

/* Forward pass.  q [B][Sq][H][d], k and v [B][Skv][H][d] bf16 (inputs);
 * o [B][Sq][H][d] bf16 and lse [B][H][Sq] fp32 (outputs, natural log of the
 * row's softmax normaliser including `scale`).  A query row that sees no key
 * gets O = 0 and LSE = -inf.  `ws` must hold fm_workspace_size(desc, 0) bytes,
 * 256-byte aligned.  `scale` multiplies Q K^T (1/sqrt(d) is usual). */
fm_status fm_fwd(const fm_desc* desc, const void* q, const void* k, const void* v,
                 const int32_t* lts, const int32_t* lte, const int32_t* uts,
                 const int32_t* ute, float scale, void* o, float* lse, void* ws,
                 size_t ws_bytes, void* stream);

/* Backward pass.  Inputs q, k, v, o (bf16), lse (fp32, from fm_fwd with the
 * same bounds and scale), dout = dO (bf16, o_stride); outputs dq, dk, dv
 * (bf16).  Gradients of rows that see no key, and of columns no row sees,
 * are 0.  `ws` must hold fm_workspace_size(desc, 1) bytes.  dK and dV are
 * accumulated per k-tile column and dQ per q-tile row, each on chip, so the
 * outputs are written once and need no clearing beforehand. */
fm_status fm_bwd(const fm_desc* desc, const void* q, const void* k, const void* v,
                 const void* o, const float* lse, const void* dout, const int32_t* lts,
                 const int32_t* lte, const int32_t* uts, const int32_t* ute, float scale,
                 void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream);

/* fm_fwd and fm_bwd without the mask analysis: `ws` is a step workspace
 * (fm_workspace_size(desc, FM_WS_STEP) bytes) on which fm_plan(FM_WS_STEP)
 * has run, on `stream` or before it, with this `desc` and these bounds, and
 * which nothing has written since but fm_fwd_planned and fm_bwd_planned.
 * The bounds are still read (per-key masks of partial tiles).  Each call
 * zeroes only its kernels' unit counters in the status word, so the
 * analysis' device status bits stay for fm_device_status.  Results are
 * identical to fm_fwd / fm_bwd's.  Same arguments and errors otherwise. */
fm_status fm_fwd_planned(const fm_desc* desc, const void* q, const void* k, const void* v,
                         const int32_t* lts, const int32_t* lte, const int32_t* uts,
                         const int32_t* ute, float scale, void* o, float* lse, void* ws,
                         size_t ws_bytes, void* stream);
fm_status fm_bwd_planned(const fm_desc* desc, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout,
                         const int32_t* lts, const int32_t* lte, const int32_t* uts,
                         const int32_t* ute, float scale, void* dq, void* dk, void* dv,
                         void* ws, size_t ws_bytes, void* stream);

/* Size of the fixed device scratch used by fm_fwd_static (8 MiB per GPU). */
#define FM_STATIC_SCRATCH_BYTES (8u << 20)

/* Forward pass for callers that cannot allocate device memory when they call
 * it (for instance a plugin inside a framework that owns all device memory
 * through its own allocator, or a latency-critical path that must not call
 * cudaMalloc/cudaFree).  The pages describe no such interface; it has no
 * counterpart there.  Same arguments and results as fm_fwd, without `ws`:
 * the scratch lives in a fixed array of FM_STATIC_SCRATCH_BYTES in device
 * memory that belongs to the library image, so every GPU that loads the
 * library keeps those bytes until the process exits.  The visibility-mask
 * region gets what the other regions leave of the array (possibly nothing;
 * the forward kernel then builds the partial tiles' bits itself: slower,
 * same results); problems whose other regions alone exceed
 * FM_STATIC_SCRATCH_BYTES are rejected with FM_ERR_WORKSPACE before anything
 * is enqueued.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current); make that first call before any stream capture.
 * The function allocates nothing (no cudaMalloc, cudaFree or allocating
 * library call).  All calls on a device share the array: calls whose work
 * may overlap on the GPU (other streams, other host threads) race and give
 * undefined results, so serialise them.  Device-side findings (bound values
 * out of range) are recorded in the shared array and cannot be read back
 * through this entry point; check bounds with fm_plan on a caller workspace
 * if that is needed. */
fm_status fm_fwd_static(const fm_desc* desc, const void* q, const void* k, const void* v,
                        const int32_t* lts, const int32_t* lte, const int32_t* uts,
                        const int32_t* ute, float scale, void* o, float* lse, void* stream);

/* Mask localisation ("clip, shift, max" over the bound vectors; FlashMask-3
 * page, introduction and «Ключевые факты»).  A rank holds the query rows of
 * n_chunks chunks of the global sequence, chunk c covering global rows
 * [chunk_start[c], chunk_start[c] + chunk_len[c]), laid out one after the
 * other in its local query tensor.  Every bound value x becomes
 *     x' = max over chunks c with chunk_start[c] <= x of
 *              (offset[c] + min(x - chunk_start[c], chunk_len[c])),   0 if none,
 * offset[c] = sum of the lengths of the chunks before c: the number of local
 * rows whose global row is below x.  The key axis is unchanged, so the
 * rank runs fm_fwd / fm_bwd with Sq = sum(chunk_len), its local Q/dO and the
 * full K/V.  No data moves between ranks.
 *   bounds, local_bounds: DEVICE int32 [4][B][Hm][Skv] (LTS, LTE, UTS, UTE
 *     arrays one after the other); may not overlap.
 *   chunk_start, chunk_len: HOST int32[n_chunks], in local order, which must
 *     be ascending in global position and non-overlapping, with positive
 *     lengths (else FM_ERR_INVALID: the preimage of an interval would not be
 *     an interval); 1 <= n_chunks <= 128. */
fm_status fm_localize(const int32_t* bounds, int B, int Hm, int Skv,
                      const int32_t* chunk_start, const int32_t* chunk_len, int n_chunks,
                      int32_t* local_bounds, void* stream);

/* FP8 (e4m3) forward, head_dim 128 only (FM_ERR_UNSUPPORTED otherwise).  The
 * ROCm page («Современное состояние Flash Attention на ROCm») names an FP8
 * FlashAttention as the fastest in its comparison and gives no formula; the
 * reading here is per-tile scaling:
 *
 * fm_quantize_fp8: for each (batch, head) and 128-row tile of Q, K and V, the
 * scale s = amax / 448 and its reciprocal r = 448 / amax in fp32 (both 1
 * for an all-zero tile; one IEEE division each per tile) and the codes
 * e4m3(x * r) (fp32 product, round to nearest even, saturating at +-448).
 * Inputs q, k, v: bf16 with desc's strides.  Outputs (caller-owned device
 * memory): q8 uint8 [B][Sq][H][128] and k8 uint8 [B][Skv][Hkv][128] (BSHD,
 * contiguous); v8t uint8 [B][Hkv][128][nK*128], V transposed per head with the
 * key axis padded to whole tiles (padding 0); q_scale fp32 [B][H][nQ],
 * k_scale and v_scale fp32 [B][Hkv][nK], v_head_scale fp32 [B][Hkv] (the
 * largest V tile scale of the head).
 *
 * fm_fwd_fp8: the forward pass on those codes and scales, with the same
 * masks, scale, outputs (o bf16 with o_stride, lse fp32) and workspace
 * (FM_WS_FWD) as fm_fwd; desc's q/k/v strides are not used.  Per query row
 * i and visible key j: s_ij = scale * sq * sk * (q8_i . k8_j), c = s log2 e;
 * P is taken against an integral reference exponent M (ceil of the running
 * row maximum of c, moved only when it grows by more than 8), multiplied by
 * the V tile's ratio sv / sv_head and rounded to e4m3 for the P V product;
 * O = sv_head * sum_j P8_ij v8_j / sum_j 2^(c_ij - M), LSE = (M + log2 l) ln 2.
 * Both products run as e4m3 tensor-core MMAs with fp32 accumulation. */
fm_status fm_quantize_fp8(const fm_desc* desc, const void* q, const void* k, const void* v,
                          void* q8, void* k8, void* v8t, float* q_scale, float* k_scale,
                          float* v_scale, float* v_head_scale, void* stream);
fm_status fm_fwd_fp8(const fm_desc* desc, const void* q8, const void* k8, const void* v8t,
                     const float* q_scale, const float* k_scale, const float* v_scale,
                     const float* v_head_scale, const int32_t* lts, const int32_t* lte,
                     const int32_t* uts, const int32_t* ute, float scale, void* o, float* lse,
                     void* ws, size_t ws_bytes, void* stream);

/* Bounds of a packed variable-length batch: the FlashAttention-2 page's
 * fixed-token batch («Как понимать заявленное ускорение»: 16K tokens per
 * batch) in the column-bound form of the FlashMask-3 page.  Sequence s holds
 * rows and keys [cu_seqlens[s], cu_seqlens[s+1]) of one axis of `total`
 * tokens; a row sees only keys of its own sequence, and with `causal` only
 * keys at or before it.  cu_seqlens: device int32 [n_seqs + 1], 0 first,
 * non-decreasing, `total` last (zero-length sequences allowed).  bounds:
 * device int32 [4][total] (LTS, LTE, UTS, UTE; the [4][B=1][Hm=1][Skv] layout
 * of fm_fwd with Sq = Skv = total), written by a kernel on `stream`.  `bad`
 * (device int, may be null) has 1 or-ed into it if cu_seqlens is not such a
 * partition; keys then outside every sequence are hidden from all rows.
 * Returns FM_ERR_INVALID for null pointers or sizes out of range. */
fm_status fm_varlen_bounds(const int32_t* cu_seqlens, int n_seqs, int total, int causal,
                           int32_t* bounds, int* bad, void* stream);

/* Kernel timing, for benchmarks.  While enabled, every kernel the library
 * launches is bracketed by a pair of CUDA events recorded on its own stream
 * (event objects are created on first use and reused; no device memory is
 * allocated).  fm_profile_read() waits for the recorded events, writes per
 * kernel id the summed device time in milliseconds and the launch count into
 * total_ms[0..n) and launches[0..n) (either may be NULL), and clears the
 * record.  Kernel ids: 0 block summary, 1 classify, 2 unit order,
 * 3 localize, 4 forward, 5 backward preprocess, 6 backward dK/dV, 7 backward
 * dQ, 8 partial-tile visibility masks, 9 FP8 quantisation, 10 FP8 forward;
 * fm_kernel_name(id) names them.  At most 65536 launches are recorded per
 * read; later launches are counted but not timed. */
fm_status fm_profile_enable(int on);
fm_status fm_profile_read(double* total_ms, int* launches, int n);
const char* fm_kernel_name(int id);

/* Measured exp2 throughput of this GPU: a kernel of one 1024-thread block
 * per SM, each thread eight independent chains of ex2.approx.f32 (the
 * instruction that computes P in the attention kernels), timed with CUDA
 * events on `stream` (synchronises it).  Writes exp2 evaluations per second
 * for the whole GPU; the host turns it into a ceiling on effective TFLOP/s
 * (one exp2 per visible entry in the forward, two in the backward).  No
 * counterpart on the pages: it measures the secondary (non-matmul) limit
 * the FlashAttention-2 page's «Три способа повысить загрузку GPU» is about. */
fm_status fm_measure_exp2_rate(double* per_second, void* stream);

/* Test hooks for the device-side wait limit (process-wide; they apply to
 * every launch made after the call).  Every mbarrier wait in the attention
 * kernels gives up after wait_limit_ns nanoseconds (0 restores the default of
 * 2 s); the launch then records FM_ERR_TIMEOUT in its status word, finishes
 * the copies and MMAs it has issued, frees its tensor memory and returns,
 * leaving its outputs undefined.  withhold_release makes one consumer
 * release never happen, so that a wait runs out on purpose: 0 none,
 * 1 fm_fwd (the softmax warps of the first q-tile of each unit pair skip
 * their first "P ready" arrival in each CTA), 2 fm_bwd's dK/dV pass (the
 * compute warps skip their first "P ready" arrival in each CTA), 3 fm_bwd's
 * dQ pass (the compute warps skip their first "dS ready" arrival in each
 * CTA).  For tests of the unwind
 * path only; calls that overlap a change of these settings see either value.
 * FM_ERR_INVALID for other withhold values. */
fm_status fm_test_hooks(uint64_t wait_limit_ns, int withhold_release);

/* Synchronise `stream` and read the device status word of `ws`: FM_OK,
 * FM_ERR_BOUNDS, FM_ERR_TIMEOUT, or FM_ERR_CUDA if a kernel found its shared
 * memory misaligned and did nothing (precedence: CUDA, timeout, bounds). */
fm_status fm_device_status(const void* ws, void* stream);

/* Static description of a status code. */
const char* fm_status_string(fm_status s);

/* Library version, major*10000 + minor*100 + patch. */
int fm_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FM_H_ */
