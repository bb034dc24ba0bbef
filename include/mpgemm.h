/*
 * mpgemm — mixed-precision tensor-core matrix product for sm_103a (GB300).
 *
 * C ABI.  Plain pointers and integer sizes only; no C++ or framework types.
 *
 * Computes, for every batch index b,
 *     C_b = alpha * A_b * B_b + beta * C_b
 * with A_b (m x k), B_b (k x n), C_b (m x n, row-major fp32), under an explicit
 * precision policy.  The operation and its parameters follow:
 *   - "tile_matmul(): use the cuBLASDx register-accumulator API with suggested
 *     shared layouts for Tensor Core precisions", section "Description": every
 *     call computes C = alpha*A*B + beta*C in place;
 *   - "Tensor Core operands: a matrix instruction still needs a layout
 *     contract", first paragraph: row-major / column-major operands and the
 *     leading dimension (element distance between successive rows, resp.
 *     columns; padding may make it larger than the visible extent);
 *   - same page, third paragraph: FP16 or BF16 multiplicands with FP32
 *     accumulation, TF32, and the rounding each conversion adds;
 *   - "qsa_prompt_attn: Volta (sm_70) m8n8k4 kernel - keep the hi and lo halves
 *     in separate accumulator chains", sections "What's going on" and "The fix":
 *     FP32 operands split into FP16 hi and lo halves, with the hi and lo
 *     products accumulated in separate chains and summed in plain FP32.
 *
 * Conventions common to every entry point:
 *   - Device pointers are raw CUDA device addresses owned by the caller; the
 *     library never frees or retains them after the call returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Compute calls are asynchronous on that stream.
 *   - Compute calls launch only stream-ordered work (kernels, and one
 *     cudaMemsetAsync for the split tail), so they can be captured in CUDA
 *     graphs; make the first call on a device outside a capture (it sets
 *     kernel attributes and queries cluster occupancy once).
 *   - Every call returns an mpg_status; on failure the reason is available
 *     from mpg_last_error_string() (thread-local, valid until the next call
 *     on the same thread).  Argument errors are detected on the host before
 *     anything is launched.
 *   - No entry point allocates device memory on the compute path.  Scratch
 *     (split-K partial sums) lives in a caller-provided workspace sized by
 *     mpg_gemm_workspace_size().
 */
#ifndef MPGEMM_H_
#define MPGEMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage order of an operand (layout contract, "Tensor Core operands: a
 * matrix instruction still needs a layout contract", first paragraph).
 *   ROW_MAJOR: element (r, c) at r*ld + c, ld >= number of columns.
 *   COL_MAJOR: element (r, c) at c*ld + r, ld >= number of rows. */
typedef enum { MPG_ROW_MAJOR = 0, MPG_COL_MAJOR = 1 } mpg_layout;

/* Storage type of A and B.  C is always fp32, row-major. */
typedef enum { MPG_F32 = 0, MPG_F16 = 1, MPG_BF16 = 2 } mpg_dtype;

/* Precision policy ("Tensor Core operands ...", third paragraph; "qsa_prompt_attn
 * ...", "The fix").
 *   FP16_F32ACC  multiplicands rounded to fp16 (RNE) — fp32 inputs are
 *                converted on load, fp16 inputs are used as stored; products
 *                accumulated in fp32 on the tensor cores.
 *   BF16_F32ACC  same with bf16 (fp32 or bf16 inputs).
 *   TF32         fp32 inputs fed to the tf32 tensor-core path, fp32 accumulate.
 *   SPLIT_FP16_3CHAIN  fp32 inputs split on load into fp16 hi/lo halves
 *                (see mpg_options for the exact split); hi*hi, hi*lo and lo*hi
 *                accumulate in three separate fp32 accumulators that are summed
 *                in plain fp32 in the epilogue: acc = hh + 2^-L * (hl + lh)
 *                (L = 11 by default, 0 with split_plain_lo), per K chunk, the
 *                chunk totals added in fp32 (split_chunk_k).
 *   SPLIT_FP16_1CHAIN  the same three products accumulated in ONE accumulator
 *                over the whole K range (the shared-chain variant, kept for
 *                comparison; its lo is the plain fp16(x*2^s - hi), without the
 *                2^11 scale).
 *   FP32_FFMA    plain fp32 CUDA-core product: each output is one sequential
 *                fmaf chain over k in ascending order (the comparator).
 *   SPLIT_A_FP16_2CHAIN  the split of "qsa_prompt_attn ...", "What's going
 *                on": only A is split into fp16 hi and lo (lo scaled by 2^L,
 *                L = 11 by default), B is rounded to fp16 (RNE); A_hi*B and
 *                A_lo*B accumulate in two separate chains summed in fp32:
 *                acc = hb + 2^-L * lb (per K chunk, as for the three-chain
 *                split).  fp32 inputs.
 *   SPLIT_FP16_4CHAIN  the three-chain split plus the lo*lo product in a
 *                fourth chain: acc = hh + (2^-L * (hl + lh) + 2^-2L * ll).
 *                fp32 inputs; 128 x 64 tiles. */
typedef enum {
  MPG_FP16_F32ACC = 0,
  MPG_BF16_F32ACC = 1,
  MPG_TF32 = 2,
  MPG_SPLIT_FP16_3CHAIN = 3,
  MPG_SPLIT_FP16_1CHAIN = 4,
  MPG_FP32_FFMA = 5,
  MPG_SPLIT_A_FP16_2CHAIN = 6,
  MPG_SPLIT_FP16_4CHAIN = 7
} mpg_precision;

typedef enum {
  MPG_OK = 0,
  MPG_ERR_INVALID_ARG = 1,  /* bad size, leading dimension, stride or pointer */
  MPG_ERR_UNSUPPORTED = 2,  /* dtype / mode combination the library does not offer */
  MPG_ERR_NO_DEVICE = 3,    /* no CUDA device, or not an sm_103 device */
  MPG_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required */
  MPG_ERR_CUDA = 5,         /* a CUDA runtime / driver call failed */
  MPG_ERR_TIMEOUT = 6       /* a kernel's bounded wait expired (see mpg_device_status) */
} mpg_status;

/* Optional knobs.  Initialise with mpg_options_init(); a NULL options pointer
 * means the defaults. */
typedef struct {
  /* Split modes: A is split as x*2^split_exp_a and B as x*2^split_exp_b before
   * hi = fp16(x*2^s), lo = fp16((x*2^s - hi) * 2^L) (L: see split_plain_lo);
   * the scale is undone exactly in the epilogue.  Use it to lift
   * operands whose magnitudes sit below fp16's normal range (2^-14), e.g.
   * softmax probabilities.  Default 0.  Range [-100, 100]. */
  int32_t split_exp_a;
  int32_t split_exp_b;
  /* Number of K partitions (split-K).  0 = chosen by the library. */
  int32_t splitk;
  /* 1 = load operands with plain global loads even where TMA applies
   * (exercises the path used for unaligned leading dimensions).  Default 0. */
  int32_t force_generic_load;
  /* Tile width along N: 0 = chosen by the library, else 64, 128 or 256
   * (256 only for the direct fp16/bf16/tf32 paths). */
  int32_t tile_n;
  /* Upper bound for any single wait inside a kernel, in nanoseconds.
   * 0 = default (2 s).  On expiry the kernel stops, records MPG_ERR_TIMEOUT in
   * the device status word and returns without hanging the GPU. */
  int64_t wait_timeout_ns;
  /* The split modes except the one-chain form: the K loop accumulates in chunks of this many k
   * elements.  Each chunk starts fresh hh / hl / lh accumulators on the tensor
   * cores; the epilogue adds the chunk's hh + 2^-L*(hl + lh) to an fp32
   * running sum with round-to-nearest.  This bounds how long the tensor
   * cores' own fp32 accumulation runs (its rounding is not round-to-nearest).
   * 0 = default: 512 for the three- and four-chain splits, one chunk for the
   * A-only two-chain split (whose error is set by B's fp16 rounding);
   * negative = one chunk covering the whole K range.  Rounded up to a
   * multiple of the k-block (32 or 64). */
  int32_t split_chunk_k;
  /* The separate conversion pass for fp32 operands (FP16_F32ACC, BF16_F32ACC
   * and the split modes): one extra kernel reads A and B once and writes
   * packed 16-bit copies (hi and lo halves for the split) into the caller's
   * workspace, then the product runs on those copies on its direct TMA path.
   * Same conversions and same results as converting on the fly in the load
   * stage; it needs a workspace of mpg_gemm_workspace_size() bytes queried
   * with the same options (4 bytes per operand element for the split, 2
   * otherwise, plus split-K partials).
   *   1  = always (MPG_ERR_WORKSPACE if the workspace is too small);
   *   0  (default) = the library's choice: the pass when m >= 256,
   *        n >= 256 and m*n*k >= 2^32 (both operands re-read by many tiles)
   *        and the workspace holds the copies; mpg_gemm_workspace_size
   *        includes them for the split modes, mpg_gemm_workspace_size_ex
   *        (which sees the operand types) also for fp16 / bf16 modes on
   *        fp32 operands; otherwise conversion happens on the fly;
   *   -1 = never. */
  int32_t prepass;
  /* Storage type of C (an mpg_dtype): MPG_F32 (default), MPG_F16 or MPG_BF16.
   * With a 16-bit C the `C` argument points to 16-bit storage (ldc and
   * strideC in its elements); beta*C is read in that type and the fp32
   * result alpha*acc + beta*C is rounded once, to nearest even, when stored:
   * the extra rounding stage of a reduced-precision output ("Tensor Core
   * operands: a matrix instruction still needs a layout contract", third
   * paragraph). */
  int32_t c_dtype;
  /* CTA pairs for 16-bit and TF32 products on the direct TMA path (FP16 /
   * BF16 operands, TF32 with a row-major A and a column-major B, or the
   * copies made by the conversion pass or the aligned-copy path): a cluster
   * of two CTAs on two SMs computes a 256 x 256 tile with cta_group::2
   * tensor-core instructions, each CTA holding half of A's rows and half of
   * B's columns; the same products, accumulated in fp32 on the tensor cores
   * along K in the same order.  0 (default) = used when m > 128, n > 128
   * and the 256 x 256 tiles give every pair of SMs at least one tile (many
   * small batched products keep the finer one-CTA tiles), 1 = always where
   * it applies,
   * -1 = never (one CTA per 128-row tile).  The three-chain split on the
   * conversion pass's copies takes pairs (256 x 128 tiles, the same bits as
   * single CTAs) only with 1: on a GB300 it measured slower than single
   * CTAs.  Other configurations ignore it. */
  int32_t cta_pair;
  /* Split tail for the CTA-pair kernel.  A persistent grid of P clusters
   * takes tiles in rounds of P; when the last round holds R < P tiles, the
   * other clusters would idle for a whole tile.  With the split tail each of
   * those R tiles is cut in two along K at the middle k-block: 2R workers
   * each multiply one half, write their fp32 partial sums to the workspace,
   * and the second half to arrive adds the two (fp32, round to nearest: the
   * same sum in either order) and applies alpha, beta and C's type, so the
   * result does not depend on timing.  Needs the workspace that
   * mpg_gemm_workspace_size reports (at most 128 x 256 x 4 bytes per SM plus
   * counters) and clears its counters with one cudaMemsetAsync per call.
   *   0 (default) = where it pays on a GB300: 1 to 6 full rounds, then
   *       1 <= R <= P/2 tiles, and at least 128 k-blocks (k >= 8192, tf32
   *       k >= 4096: half a tile's time outweighs
   *       waiting for the later of two clusters and exchanging the partial
   *       sums, about 16 us), when the workspace holds it;
   *   1 = whenever the tile count is not a multiple of P (all tiles when
   *       there are fewer than P) and K has two k-blocks
   *       (MPG_ERR_WORKSPACE if the workspace is too small);
   *   -1 = never.  Other kernels ignore it. */
  int32_t tail_split;
  /* The lo half's scale 2^L in the split modes.
   *   0 (default) = L = 11 in the forms with separate lo chains (3CHAIN,
   *       A-only 2CHAIN, 4CHAIN): lo = fp16((x*2^s - hi) * 2^11), the lo
   *       chains scaled back by 2^-11 in fp32 in the epilogue, which keeps
   *       lo out of fp16's subnormals for |x*2^s| >= 2^-3; L = 0 in the
   *       one-chain form (its single accumulator holds hi and lo products
   *       at one scale);
   *   1 = L = 0 in every split form: the plain lo = fp16(x*2^s - hi).  With
   *       3CHAIN this is the three-chain split with the unscaled lo, whose
   *       operands are bit for bit those of 1CHAIN: the two then differ in
   *       the number of accumulator chains alone.
   * Other values: MPG_ERR_INVALID_ARG. */
  int32_t split_plain_lo;
  /* SPLIT_FP16_3CHAIN only: 1 = the hi*lo and lo*hi products share one
   * accumulator, so the product keeps two (hh, and hl + lh), summed in fp32
   * in the epilogue as acc = hh + 2^-L * (hl + lh).  The two lo products
   * have the same magnitude (about 2^-11 of hh), so sharing their
   * accumulator keeps them apart from hh as the separate chains do.  Two
   * such accumulators fit in TMEM at once, so the epilogue of one tile
   * overlaps the products of the next: the form for short K, e.g. attention
   * scores (k = 128).  Taken when the whole K range is one accumulation
   * chunk (k <= split_chunk_k, 512 by default, or split_chunk_k < 0); longer
   * products keep the three chains.  0 (default) = three chains.  Other
   * values: MPG_ERR_INVALID_ARG. */
  int32_t split_lo_shared;
  int32_t reserved[1];
} mpg_options;

void mpg_options_init(mpg_options* opt);

/* The product.
 *   m, n, k      >= 0; batch >= 0.  m == 0, n == 0 or batch == 0: no-op.
 *                k == 0: C = beta*C.  beta == 0: C is not read.
 *                alpha == 0: A and B are not read.
 *   A            device pointer; a_layout ROW_MAJOR requires lda >= k,
 *                COL_MAJOR requires lda >= m (lda >= 1 always).
 *   strideA      elements between consecutive batch matrices of A; 0 means
 *                packed (m*lda for row-major, k*lda for column-major).
 *   B            likewise with (k x n): ROW_MAJOR ldb >= n, COL_MAJOR ldb >= k.
 *   C            device pointer, row-major fp32 (or 16-bit, see
 *                mpg_options.c_dtype), ldc >= n; strideC 0 = m*ldc; with
 *                batch > 1 a nonzero strideC must keep the batch matrices
 *                of C apart (strideC >= (m-1)*ldc + n), else
 *                MPG_ERR_INVALID_ARG.
 *   mode         precision policy; allowed input dtypes per mode:
 *                  FP16_F32ACC: A, B both F32 or both F16
 *                  BF16_F32ACC: A, B both F32 or both BF16
 *                  TF32, SPLIT_* (all split forms), FP32_FFMA: A, B both F32
 *                anything else returns MPG_ERR_UNSUPPORTED.
 *   workspace    device scratch of at least mpg_gemm_workspace_size(...)
 *                bytes (may be NULL when that size is 0).  Its contents on
 *                entry are ignored.  Calls that share a workspace must be
 *                ordered on one stream.
 * Pointers need only element alignment; 16-byte aligned pointers and leading
 * dimensions whose byte size is a multiple of 16 take the TMA load path; for
 * any other alignment the call copies the operands to aligned lines in the
 * workspace when it has room (mpg_gemm_workspace_size reserves it for large
 * products), else takes the generic-load path (same results, lower speed).
 * The memory C_b occupies must not overlap A or B. */
mpg_status mpg_gemm(int64_t m, int64_t n, int64_t k, int64_t batch,
                    const void* A, int64_t lda, int64_t strideA, mpg_dtype a_dtype, mpg_layout a_layout,
                    const void* B, int64_t ldb, int64_t strideB, mpg_dtype b_dtype, mpg_layout b_layout,
                    float* C, int64_t ldc, int64_t strideC,
                    float alpha, float beta, mpg_precision mode,
                    void* workspace, size_t workspace_bytes, void* stream);

/* mpg_gemm with options (NULL = defaults). */
mpg_status mpg_gemm_ex(int64_t m, int64_t n, int64_t k, int64_t batch,
                       const void* A, int64_t lda, int64_t strideA, mpg_dtype a_dtype, mpg_layout a_layout,
                       const void* B, int64_t ldb, int64_t strideB, mpg_dtype b_dtype, mpg_layout b_layout,
                       float* C, int64_t ldc, int64_t strideC,
                       float alpha, float beta, mpg_precision mode,
                       void* workspace, size_t workspace_bytes, void* stream,
                       const mpg_options* opt);

/* The product for callers that cannot allocate device memory.
 *
 * No counterpart on the pages: this is a convenience of this library.  Some
 * callers cannot call cudaMalloc and so cannot hand mpg_gemm a workspace:
 * plugins inside a host framework that owns all device memory and forbids
 * raw allocations, and real-time or long-running services that allow no
 * allocation (and no allocation failure) after start-up.  This entry point
 * takes the same arguments as
 * mpg_gemm_ex minus the workspace and behaves as mpg_gemm_ex given a
 * workspace of MPG_NOALLOC_SCRATCH_BYTES bytes: that workspace is a scratch
 * array compiled into the library (16 MiB of device memory, present on every
 * GPU that loads the library until the process exits).  It holds split-K
 * partial sums, and the copies that the conversion pass or the aligned-copy
 * path make when they fit.  It allocates nothing.
 *   - With a split count forced by mpg_options.splitk whose partial sums
 *     (splits x batch x m x n x 4 bytes) exceed the scratch, the call returns
 *     MPG_ERR_WORKSPACE before anything is launched; an automatic split
 *     count falls back to one split instead.  A conversion pass forced with
 *     mpg_options.prepass = 1 whose copies exceed the scratch also returns
 *     MPG_ERR_WORKSPACE.  Use mpg_gemm with a workspace for those.
 *   - The first call on a device looks up the scratch array's device address
 *     (once per device, with that device current) and keeps it for the life
 *     of the process; make that first call before any stream capture.  After
 *     cudaDeviceReset the kept address (like the library's other per-device
 *     state) is no longer valid: do not call the library again in that
 *     process.
 *   - Every call on a device shares the one scratch array, and each call
 *     overwrites the part it uses (nothing in it needs to start at zero):
 *     calls that can overlap on the GPU (different streams without ordering)
 *     race.  Order them on one stream.
 *   - The split tail (mpg_options.tail_split) is never taken here: its
 *     partial sums can outgrow the scratch.
 * Results are bit for bit those of mpg_gemm_ex for the same arguments and
 * options with tail_split = -1 and a workspace of MPG_NOALLOC_SCRATCH_BYTES
 * bytes. */
#define MPG_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
mpg_status mpg_gemm_noalloc(int64_t m, int64_t n, int64_t k, int64_t batch,
                            const void* A, int64_t lda, int64_t strideA, mpg_dtype a_dtype, mpg_layout a_layout,
                            const void* B, int64_t ldb, int64_t strideB, mpg_dtype b_dtype, mpg_layout b_layout,
                            float* C, int64_t ldc, int64_t strideC,
                            float alpha, float beta, mpg_precision mode, void* stream,
                            const mpg_options* opt);

/* Bytes of workspace mpg_gemm / mpg_gemm_ex need for this problem (0 if none).
 * Depends only on the sizes, the mode, the options and the current device,
 * so it covers every layout and alignment of the operands: for fp16 / bf16 /
 * tf32 products with m >= 256, n >= 256 and m*n*k >= 2^32 it includes room
 * for copies of both operands with 16-byte aligned lines (2 bytes per
 * element, 4 for tf32, at the larger of the two line paddings), which the
 * call uses for operands TMA cannot take as given (unaligned base, leading
 * dimension or batch stride; tf32 in the wrong majorness), multiplying the
 * copies on its TMA path, and, for fp32 operands in the fp16 / bf16 modes,
 * for the conversion pass.  mpg_gemm_workspace_size_ex gives the exact need
 * of one call (0 for aligned operands of those modes, the split tail aside).
 * For the fp16 / bf16 / tf32 modes it includes the split tail's partial sums
 * (mpg_options.tail_split) when the library may take it (1 to 6 full rounds
 * of 256 x 256 tiles on SMs / 2 clusters, k >= 8192, tf32 k >= 4096): up to
 * SMs / 4 tiles x 512 KiB, about 20 MB on 152 SMs. */
size_t mpg_gemm_workspace_size(int64_t m, int64_t n, int64_t k, int64_t batch,
                               mpg_precision mode, const mpg_options* opt);

/* The product with A, B and C in HOST memory: the call copies the operands
 * in, multiplies on the device and copies C back, all enqueued on `stream`.
 *
 * The same arguments as mpg_gemm_ex, except that A, B and C are host
 * pointers (page-locked memory, e.g. from cudaHostAlloc, lets the copies run
 * asynchronously and overlap; pageable memory works but its copies block the
 * calling thread).  C's padding columns (n .. ldc-1) are never written.
 *   workspace   device memory of at least mpg_gemm_host_workspace_size()
 *               bytes for the same arguments, 16-byte aligned: packed device
 *               copies of A, B and C with lines padded to 16 bytes (so the
 *               product takes the TMA path whatever the host leading
 *               dimensions), plus the product's own workspace.
 * Inside one call the copies overlap the product: B is copied first, then A
 * and C are processed in chunks of rows (of whole matrices when batch > 1),
 * the copy of chunk i+1 and the copy back of chunk i-1 running beside the
 * product of chunk i on two internal copy streams of the library, ordered
 * against `stream` by events.  When the call returns, the work is enqueued;
 * C holds the result once `stream` has completed it (e.g. after
 * cudaStreamSynchronize(stream)).  Calls on different streams with separate
 * workspaces and host buffers overlap each other's copies and products.
 * Errors: those of mpg_gemm_ex; MPG_ERR_WORKSPACE if the workspace is too
 * small.  No counterpart on the pages: this is the library's entry point for
 * data that lives on the host. */
size_t mpg_gemm_host_workspace_size(int64_t m, int64_t n, int64_t k, int64_t batch,
                                    int64_t lda, int64_t strideA, mpg_dtype a_dtype, mpg_layout a_layout,
                                    int64_t ldb, int64_t strideB, mpg_dtype b_dtype, mpg_layout b_layout,
                                    int64_t ldc, int64_t strideC, float alpha, float beta,
                                    mpg_precision mode, const mpg_options* opt);
mpg_status mpg_gemm_host(int64_t m, int64_t n, int64_t k, int64_t batch,
                         const void* A, int64_t lda, int64_t strideA, mpg_dtype a_dtype, mpg_layout a_layout,
                         const void* B, int64_t ldb, int64_t strideB, mpg_dtype b_dtype, mpg_layout b_layout,
                         void* C, int64_t ldc, int64_t strideC,
                         float alpha, float beta, mpg_precision mode,
                         void* workspace, size_t workspace_bytes, void* stream,
                         const mpg_options* opt);

/* Fused prompt attention: O = softmax(scale * Q K^T) V, row by row, with the
 * scores and probabilities never written to memory ("qsa_prompt_attn: Volta
 * m8n8k4 kernel - keep the hi and lo halves in separate accumulator chains",
 * sections "What's going on" and "The fix").
 *   Q     device, fp32, lq x d row-major (ldq >= d).  Multiplied by
 *         scale * log2(e) in fp32 on load (the scores come out in base-2
 *         units for the base-2 exponential) and split into an FP16 hi half
 *         and a lo half for q.k.
 *   K, V  device, fp16 (the key/value cache), lk x d row-major; ldk and ldv
 *         >= d, multiples of 8, pointers 16-byte aligned (TMA).
 *   O     device, fp32, lq x d row-major (ldo >= d).
 *   d     the head dimension; 128 is supported (else MPG_ERR_UNSUPPORTED).
 *   scale the softmax scale (e.g. 1/sqrt(d)); scores are scale * q.k.
 *   mode  MPG_ATTN_SPLIT_2CHAIN: q and the probabilities p are split into
 *         hi = fp16(x) and lo = fp16((x - hi) * 2^11); the hi and lo products
 *         accumulate in separate tensor-core chains added in fp32 (the fix).
 *         MPG_ATTN_SPLIT_1CHAIN: lo = fp16(x - hi) accumulated into the same
 *         chain as hi (the form the fix replaced), for comparison.
 *   key_splits  0 = chosen by the library: the keys are divided among CTAs
 *         so that about one CTA per SM works; > 1 forces that many ranges
 *         (at most one per block of 128 keys).
 *         Several ranges need a workspace of mpg_attention_workspace_size()
 *         bytes for their partial results (a merge kernel combines them);
 *         with a smaller workspace an automatic choice falls back to one range.
 * lq == 0 is a no-op; lk must be >= 1. */
typedef enum { MPG_ATTN_SPLIT_2CHAIN = 0, MPG_ATTN_SPLIT_1CHAIN = 1 } mpg_attn_mode;
size_t mpg_attention_workspace_size(int64_t lq, int64_t lk, int64_t d, int32_t key_splits);
mpg_status mpg_attention(int64_t lq, int64_t lk, int64_t d, const float* Q, int64_t ldq, const void* K, int64_t ldk,
                         const void* V, int64_t ldv, float* O, int64_t ldo, float scale, mpg_attn_mode mode,
                         int32_t key_splits, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace for this exact call: mpg_gemm_workspace_size() plus
 * room for copies of the operands the TMA path cannot take as given:
 * 16-bit operands (FP16 / BF16 modes) and fp32 operands (TF32) whose base is
 * not 16-byte aligned or whose leading dimension or batch stride is not a
 * multiple of 16 bytes, and in TF32 a column-major A or a row-major B (the
 * tensor cores take tf32 tiles K-major only; those copies are transposed).
 * Given that workspace, mpg_gemm_ex copies such operands (one extra read
 * and write of each) and multiplies the copies on its TMA path instead of
 * loading the originals element by element. */
size_t mpg_gemm_workspace_size_ex(int64_t m, int64_t n, int64_t k, int64_t batch,
                                  const void* A, int64_t lda, int64_t strideA, mpg_dtype a_dtype,
                                  mpg_layout a_layout, const void* B, int64_t ldb, int64_t strideB,
                                  mpg_dtype b_dtype, mpg_layout b_layout, mpg_precision mode,
                                  const mpg_options* opt);

/* Synchronises `stream`, then reads and clears the library's device status
 * word on the current device.  Returns MPG_ERR_TIMEOUT if any kernel since the
 * last call gave up a bounded wait, MPG_ERR_CUDA if the stream reports an
 * error, else MPG_OK. */
mpg_status mpg_device_status(void* stream);

/* Thread-local description of the last failure on this thread. */
const char* mpg_last_error_string(void);

/* Library version, major*10000 + minor*100 + patch. */
int mpg_version(void);

/* ---- accumulator fragment map of mma.sync m16n8k16 (f32 accumulator) ------
 * "feat(cuda-device): derive the m16n8k16 accumulator fragment layout",
 * sections "The layout is a mixed-radix numeral" and "API".  Pure host
 * functions, no CUDA.  lane in [0, 32), j in [0, 4). */

/* Position (row in [0,16), col in [0,8)) of value j of lane `lane`.
 * Returns 0, or -1 for an out-of-range argument (outputs untouched). */
int mpg_acc_coords(int lane, int j, int* row, int* col);

/* Row-major offset in the 16x8 tile, in numeral form
 * (j&1)*1 + (lane%4)*2 + (lane/4)*8 + (j>>1)*64; -1 if out of range. */
int mpg_acc_offset(int lane, int j);

/* Offset of value j of lane `lane` in a strided destination whose tile starts
 * at (tile_row, tile_col) with row stride row_stride:
 *     (tile_row + row) * row_stride + tile_col + col.
 * Returns -1 (the "None" of the page) when an argument is out of range, a
 * coordinate is negative, col would not fit in the row (tile_col + col >=
 * row_stride), or the offset would reach `limit` or overflow int64. */
int64_t mpg_acc_matrix_offset(int lane, int j, int64_t tile_row, int64_t tile_col,
                              int64_t row_stride, int64_t limit);

/* Inverse of mpg_acc_offset: offset in [0,128) -> (lane, j).  Returns 0 or -1. */
int mpg_acc_decode(int offset, int* lane, int* j);

/* Accumulator map of the tcgen05 paths of this library: cta_group::1 with
 * M = 128 (m_shape 128) and cta_group::2 with M = 256 (m_shape 256, the CTA
 * pair, where each CTA's TMEM holds 128 of the rows and every column).  The
 * tcgen05 counterpart of the fragment map of "feat(cuda-device): derive the
 * m16n8k16 accumulator fragment layout", section "API".
 * Value `reg` returned by tcgen05.ld.32x32b to lane `lane` of warp `warp` of
 * the CTA of rank `cta_rank` in the pair (0 for M = 128), reading columns
 * from `col_base` on, holds D(row, col) with
 *     row = 128*cta_rank + 32*(warp % 4) + lane,   col = col_base + reg.
 * col_base + reg < 512 (the TMEM columns of an SM).  Returns 0, or -1 for an
 * out-of-range argument (outputs untouched). */
int mpg_tmem_acc_coords(int m_shape, int cta_rank, int warp, int lane, int reg, int col_base, int* row, int* col);

/* Inverse of mpg_tmem_acc_coords for loads of `load_cols` columns per
 * tcgen05.ld (a power of two, 1 .. 128; col_base a multiple of it): D(row,
 * col), row < m_shape, col < 512, comes from register `reg` of lane `lane`
 * of warp `warp` (the lowest index, 0 .. 3, of the warps that reach its lane
 * quarter; warp + 4j reads the same lanes) of CTA `cta_rank`, in the load
 * that starts at column `col_base`.  Returns 0 or -1. */
int mpg_tmem_acc_decode(int m_shape, int row, int col, int load_cols, int* cta_rank, int* warp, int* lane, int* reg,
                        int* col_base);

/* ---- operand fragment maps of mma.sync m16n8k16 (f16 / bf16 operands) -----
 * The cuda-oxide page derives the accumulator numeral and notes that the A
 * and B operands are different numerals ("Scope").  From the PTX ISA operand
 * layouts, with group = lane/4 and tig = lane%4:
 *   A (16x16, row-major): value i in [0,8) of a lane (register i/2, half i%2)
 *     sits at row = group + 8*((i>>1)&1), col = 2*tig + (i&1) + 8*(i>>2);
 *     row-major offset = (i&1)*1 + tig*2 + (i>>2)*8 + group*16 + ((i>>1)&1)*128.
 *   B (16x8, column-major): value i in [0,4) (register i/2, half i%2) sits at
 *     k = 2*tig + (i&1) + 8*(i>>1), n = group;
 *     column-major offset = (i&1)*1 + tig*2 + (i>>1)*8 + group*16.
 * Each is a bijection (256 resp. 128 points).  Return 0, or -1 for an
 * out-of-range argument. */
int mpg_frag_a_coords(int lane, int i, int* row, int* col);
int mpg_frag_a_decode(int row, int col, int* lane, int* i);
int mpg_frag_b_coords(int lane, int i, int* k, int* n);
int mpg_frag_b_decode(int k, int n, int* lane, int* i);

/* ---- hardware checks ------------------------------------------------------ */

/* One mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 by one warp.
 *   A: device, 16x16 fp16 (raw 16-bit codes), row-major, ld 16.
 *   B: device, 16x8 fp16, column-major (element (k, n) at n*16 + k).
 *   D: device, 128 floats; D[lane*4 + j] receives the raw accumulator value j
 *      of lane `lane` (C = 0), unscattered, so the caller can place it with
 *      mpg_acc_coords and compare with a host product.
 * Fragments are gathered with the A/B operand layouts of the PTX ISA. */
mpg_status mpg_probe_mma_m16n8k16(const void* A, const void* B, float* D, void* stream);

/* The same mma.sync with the operand fragments supplied per lane by the
 * caller: Afrag[lane*4 + r] is A register r of `lane` (two fp16 values, low
 * half first), Bfrag[lane*2 + r] is B register r.  The kernel loads them
 * verbatim, so a product equal to the host product checks the caller's
 * fragment maps on the hardware.  D as above (device pointers, C = 0). */
mpg_status mpg_probe_mma_m16n8k16_fragments(const uint32_t* Afrag, const uint32_t* Bfrag, float* D, void* stream);

/* Probe of the epilogue's shared-memory staging, for measuring its bank
 * conflicts apart from the tensor core's and TMA's shared-memory traffic
 * (the swizzled shared layouts of "tile_matmul(): use the cuBLASDx
 * register-accumulator API ...", "Proposed change").  `blocks` blocks of
 * 32 x 32 fp32 (row-major, packed, 4 KB each) are copied from `in` to `out`
 * through the staging buffer of one warp, with the product epilogues' own
 * code: each lane writes one row, then the warp reads the block back by
 * 16-byte chunks of rows (scalar = 0, the vector-store path) or by columns
 * (scalar = 1, the scalar path of unaligned destinations).  out equals in on
 * return.  in, out: device pointers, 16-byte aligned, blocks * 1024 floats
 * each, not overlapping; blocks in [0, 2^40].  MPG_ERR_INVALID_ARG for bad
 * arguments, before any launch. */
mpg_status mpg_probe_epilogue_staging(const float* in, float* out, int64_t blocks, int scalar, void* stream);

/* One tcgen05.mma pass of the library's one-CTA path (cta_group::1, M = 128,
 * N = n, K = 64 as four K = 16 instructions of kind::f16, fp32 accumulator in
 * TMEM, both operands K-major in 128-byte swizzled shared memory, the
 * operand layout and descriptors of the product kernels), followed by
 * tcgen05.ld.32x32b.x32 of every column by the four warps of the CTA.
 *   A: device, 128 x 64 fp16 (raw codes), row-major, ld 64.
 *   B: device, n x 64 fp16: row j holds column j of the K x N operand (B
 *      column-major with ld 64).
 *   n: 64, 128 or 256.
 *   D: device, 128 * n floats, the loads unscattered:
 *      D[((warp*32 + lane) * (n/32) + c) * 32 + reg] is register `reg` of lane
 *      `lane` of warp `warp` in the load of columns 32c .. 32c+31.  Placing
 *      each value with mpg_tmem_acc_coords(128, 0, warp, lane, reg, 32c, ...)
 *      and comparing with the host product checks the map on the hardware.
 * Waits are bounded (1 s); MPG_ERR_INVALID_ARG for bad arguments, before any
 * launch; a wait that expires shows in mpg_device_status. */
mpg_status mpg_probe_tmem_acc(const void* A, const void* B, int n, float* D, void* stream);

/* The same check for the CTA-pair path (cta_group::2, M = 256): a cluster of
 * two CTAs runs one k-block (K = 64) with the pair kernels' operand layout;
 * the CTA of rank r holds rows 128r .. 128r+127 of A and columns
 * (n/2) r .. (n/2) r + n/2 - 1 of B, and each CTA's TMEM receives its 128
 * rows of D and every column.
 *   A: device, 256 x 64 fp16, row-major, ld 64.
 *   B: device, n x 64 fp16 (row j = column j of B), n = 64, 128 or 256.
 *   D: device, 256 * n floats:
 *      D[(((4 r + warp)*32 + lane) * (n/32) + c) * 32 + reg] is register `reg`
 *      of lane `lane` of warp `warp` of the CTA of rank r in the load of
 *      columns 32c .. 32c+31; placed with mpg_tmem_acc_coords(256, r, warp,
 *      lane, reg, 32c, ...).
 * Waits are bounded (1 s); MPG_ERR_INVALID_ARG for bad arguments, before any
 * launch. */
mpg_status mpg_probe_tmem_acc_pair(const void* A, const void* B, int n, float* D, void* stream);

/* Throughput probe of the fp32 multiply-add pipe that bounds MPG_FP32_FFMA
 * (the plain fp32 comparator of "tile_matmul(): use the cuBLASDx
 * register-accumulator API ...", spike results, second bullet: fp32 stays
 * FFMA-bound).  Launches `blocks` blocks of 256 threads; every thread runs
 * `iters` rounds of 32 independent fp32 multiply-adds held in registers, as
 * scalar fmaf (packed = 0) or as 16 packed pairs (packed = 1), with no memory
 * traffic inside the loop: 2 * 32 * iters * 256 * blocks flops.  Time it with
 * events on `stream` to measure the pipe's sustained rate on this GPU.
 *   out: device, `blocks` floats; out[b] = 496 + 32 * iters on return (the
 *        chains' exact end values, so the work cannot be skipped).
 *   blocks in [1, 65535], iters in [1, 2^19], packed 0 or 1.
 * MPG_ERR_INVALID_ARG for bad arguments, before any launch. */
mpg_status mpg_probe_fma_rate(float* out, int64_t blocks, int iters, int packed, void* stream);

/* Failure-detection self test: launches one kernel whose single wait is on an
 * mbarrier nothing ever arrives at, bounded by timeout_ns (1 ms .. 10 s), then
 * synchronises.  Returns MPG_ERR_TIMEOUT when the kernel gave up the wait and
 * returned cleanly (the expected outcome); the device status word is cleared
 * afterwards.  Touches no caller memory. */
mpg_status mpg_selftest_wait_timeout(int64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MPGEMM_H_ */
