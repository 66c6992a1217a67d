/*
 * gemvfuse -- decode-path GEMV with a fused element-wise epilogue and a signed
 * Walsh-Hadamard prologue, for GB300 (sm_103a).  C ABI.
 *
 * Operations defined by the pages this library restates (cited by title, section):
 *  [EPI]  "feat(cuda): fuse activations and residual add into mmv f/q epilogues",
 *         Summary / What changed: y = W x for one output column (ncols_dst == 1), with
 *         the tail sigmoid | silu | silu(y)*m | y + r folded into the GEMV; a reshape
 *         between the product and the tail is an index identity; the destination may
 *         alias the mul/add operand (same element index) but never the product inputs.
 *  [FWHT] "vulkan: fuse the sign multiply into the Hadamard FWHT", Overview: the sign
 *         vector is multiplied in while the row is loaded, before the transform, and is
 *         broadcast over its own length.
 *  [CPU]  "ggml-cpu: fuse element-wise epilogues (ADD, MUL, SILU) into
 *         ggml_compute_forward_mul_mat", Guards / Correctness: epilogue operands are F32,
 *         same shape, contiguous; F32/F16/Q8_0/Q4_0 weights; fused == unfused values.
 *         What: the SwiGLU gate (MUL_MAT + SILU) and the gate x up product (MUL_MAT +
 *         MUL) of one FFN -- taken together as the gated dual GEMV gemv_glu() -- and
 *         the RMS_NORM + MUL pair ahead of a matmul (the RMS-normalisation prologue).
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers owned by the caller (gf_copy's may also be
 *    pinned host memory).  The library never allocates, frees or keeps a pointer after
 *    the call returns, except for handles: a prepared call keeps its pointers (host
 *    memory only), and a step graph owns its CUDA graph.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is enqueued
 *    asynchronously; the call returns once it is launched.
 *  - Arguments are validated on the host before anything is launched.  A non-zero
 *    return means nothing was launched, except GF_ERR_CUDA (launch failure; see
 *    gf_last_cuda_error()).
 *  - Vectors are contiguous float32.  A batch of ncols columns is column-major:
 *    x is [ncols][K], aux and dst are [ncols][M].
 *  - The library holds no state between calls other than per-device launch limits,
 *    a device error word (see gf_device_status()), a repair counter
 *    (gf_repair_count()) and a host-side cache of encoded tensor maps (address, shape
 *    and box of recent tensor-core operands; an entry never goes stale, as it holds
 *    no data).
 */
#ifndef GEMVFUSE_H
#define GEMVFUSE_H

#include <stdint.h>

#if defined(__GNUC__)
#define GF_API __attribute__((visibility("default")))
#else
#define GF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Weight storage formats; each row of W holds K elements, rows are contiguous.
 *  GF_F32  : float32 [M][K].
 *  GF_F16  : IEEE binary16 [M][K].
 *  GF_Q8_0 : per 32 elements a 34-byte block {binary16 d; int8 q[32]}; w = d*q.
 *  GF_Q4_0 : per 32 elements an 18-byte block {binary16 d; uint8 qs[16]}; byte j holds
 *            element j (low nibble) and element j+16 (high nibble); w = d*(nibble-8).
 *  GF_Q4_K : per 256 elements a 144-byte super-block {binary16 d; binary16 dmin;
 *            uint8 scales[12]; uint8 qs[128]}: eight 32-element sub-blocks j with 6-bit
 *            scale sc[j] and min m[j] (scales[j] low 6 bits = sc[j], scales[j+4] low 6
 *            bits = m[j] for j < 4; for j >= 4 the low 4 bits are the low/high nibble of
 *            scales[j+4] and the top 2 bits those of scales[j-4] / scales[j]); qs holds
 *            four 32-byte groups, group g sub-block 2g in the low nibbles and 2g+1 in the
 *            high nibbles; w = d*sc[j]*q - dmin*m[j].  K % 256 == 0.
 * (Format names from [CPU] Correctness; the layouts are the ggml block convention.) */
typedef enum { GF_F32 = 0, GF_F16 = 1, GF_Q8_0 = 2, GF_Q4_0 = 3, GF_Q4_K = 4 } gf_wtype;

/* Fused tails ([EPI] What changed; [CPU] What):
 *  NONE      dst = y
 *  SIGMOID   dst = 1/(1+exp(-y))
 *  SILU      dst = y*sigmoid(y)
 *  SILU_MUL  dst = silu(y)*aux          (aux = the per-row activation_mul operand)
 *  ADD       dst = y + aux              (residual add; dst == aux allowed, in place) */
typedef enum {
  GF_EPI_NONE = 0, GF_EPI_SIGMOID = 1, GF_EPI_SILU = 2, GF_EPI_SILU_MUL = 3, GF_EPI_ADD = 4
} gf_epilogue;

/* Stand-alone element-wise ops (the unfused control path): dst[i] = op(a[i], b[i % nb]). */
typedef enum { GF_EW_SIGMOID = 1, GF_EW_SILU = 2, GF_EW_MUL = 3, GF_EW_ADD = 4 } gf_ewop;

typedef enum {
  GF_OK = 0,
  GF_ERR_INVALID = -1,      /* bad enum, size, null pointer or view shape            */
  GF_ERR_ALIAS = -2,        /* dst overlaps an input it may not alias                */
  GF_ERR_UNSUPPORTED = -3,  /* valid but outside what is implemented (e.g. K%32 != 0 */
                            /* for a block format, ncols > 256, FWHT block > 8192)   */
  GF_ERR_ALIGN = -4,        /* pointer not aligned to its element type               */
  GF_ERR_CUDA = -5,         /* a CUDA runtime call or launch failed                  */
  GF_ERR_TIMEOUT = -6       /* a kernel gave up on a bounded wait (device status)    */
} gf_status;

/* gf_opts.flags */
#define GF_FLAG_PDL 1u   /* launch with programmatic dependent launch: the kernel may
                            start while the previous kernel in `stream` still runs and
                            streams W before waiting for it.  Only valid when no kernel
                            still running in `stream` writes W. */
#define GF_FLAG_NO_TENSOR_CORES 4u  /* use the CUDA-core kernels only.  By default F16 weights
                            with 3 or more columns (16 per launch), K % 64 == 0 and
                            16-byte aligned W and x run on the tensor cores: tcgen05 MMAs
                            of the f16 weights with x split into scaled f16 hi + lo parts,
                            fp32 accumulation. */
#define GF_FLAG_NO_SPLIT_K 2u  /* never split K over a cluster of CTAs (by default a GEMV
                            with M <= SMs/2 rows gives each row range to a cluster of
                            2..8 CTAs that each stream a slice of K and add their
                            partial sums in a fixed order through distributed shared
                            memory; the result is deterministic either way, but the
                            summation order, hence the rounding, differs). */

typedef struct {
  int64_t ncols;             /* columns in the batch, 1..256 (0 is read as 1); up to 8 */
                             /* share one pass over W, wider batches run as blocks of 8 */
  const float* fwht_signs;   /* non-NULL: signed-FWHT prologue on every column of x     */
  int64_t fwht_block;        /* FWHT block B: power of two, 1..8192, K % B == 0         */
  int64_t nsigns;            /* length of fwht_signs; K % nsigns == 0; element k of a   */
                             /* column uses fwht_signs[k % nsigns]                      */
  int64_t view_ne[4];        /* optional view of each dst column (all 0 = none); the    */
                             /* product of the non-zero entries must equal M. A view of */
                             /* contiguous memory is an index identity ([EPI] What      */
                             /* changed: result written with the matmul geometry).      */
  uint32_t flags;            /* GF_FLAG_*                                              */
  float* fwht_workspace;     /* optional device buffer of ncols*K floats (16-byte       */
                             /* aligned, overlapping no other argument).  Given, the    */
                             /* prologue runs once as a stand-alone transform into it   */
                             /* and the GEMV reads it, chained with programmatic        */
                             /* dependent launch; NULL: every CTA transforms x on chip. */
  const float* rms_norm_weight;  /* non-NULL: RMS-normalisation prologue on every column */
                             /* of x: x'_c = x_c / sqrt(mean_k(x_c[k]^2) + eps) * gamma, */
                             /* gamma = rms_norm_weight [K] (device float32, overlapping */
                             /* no output).  Not combinable with the FWHT prologue       */
                             /* (GF_ERR_UNSUPPORTED).                                    */
  float rms_norm_eps;        /* eps of the normalisation: finite, >= 0                 */
} gf_opts;

/* y = W x with the fused tail, one column.  [EPI] Summary, What changed.
 *  W    : device, M rows in format `wtype` (see gf_wtype).  Alignment: 4 B for F32,
 *         2 B otherwise; 16 B (and K % 256 == 0 for block formats) selects the
 *         TMA-streamed fast kernel, anything else the generic kernel.
 *  x    : device float32 [K].           aux : device float32 [M], required iff the
 *  dst  : device float32 [M].                 epilogue is SILU_MUL or ADD.
 *  Aliasing: dst may equal aux exactly; any other overlap of dst with W, x or aux
 *  returns GF_ERR_ALIAS.  M == 0 launches nothing.  K == 0 gives y = 0. */
GF_API int gemv_fused(const void* W, int wtype, const float* x, int64_t M, int64_t K,
               int epilogue, const float* aux, float* dst, void* stream);

/* gemv_fused plus the options in `opts` (may be NULL): a batch of ncols independent
 * columns sharing one pass over W; the signed-FWHT prologue
 *     x'_c[b*B + j] = (1/sqrt(B)) sum_t H_B[j][t] s[(b*B + t) % nsigns] x_c[b*B + t]
 * (Sylvester H, [FWHT] Overview) applied to each column before the product -- on chip
 * in every CTA, or once into opts->fwht_workspace; the dst view check; and
 * GF_FLAG_PDL.  fwht_signs must not overlap dst.  With a workspace two kernels are
 * launched (the transform, then the GEMV). */
GF_API int gemv_fused_ex(const void* W, int wtype, const float* x, int64_t M, int64_t K,
                  int epilogue, const float* aux, float* dst, const gf_opts* opts,
                  void* stream);

/* Gated dual GEMV, the gate and up projections of one FFN in a single pass:
 *     dst_c[i] = silu(G_i . x'_c) * (U_i . x'_c),   silu(g) = g / (1 + exp(-g))
 * ([CPU] What: MUL_MAT + SILU on the gate, then MUL by the up projection; [EPI] Summary
 * names this gated branch, which it leaves to its own GLU path).  W_gate and W_up are
 * two M x K matrices of the same format `wtype` (same rules as W of gemv_fused); x'
 * is x after the prologue chosen in `opts` (none, signed FWHT, RMS normalisation).
 * Every tile the kernel streams holds rows of both matrices, so each weight byte is
 * read once and the gate result never leaves the chip.  opts may be NULL; its ncols,
 * prologues, view and flags apply as in gemv_fused_ex.  dst may not overlap W_gate,
 * W_up, x or the prologue operands. */
GF_API int gemv_glu(const void* W_gate, const void* W_up, int wtype, const float* x, int64_t M,
                    int64_t K, float* dst, const gf_opts* opts, void* stream);

/* Several matrices that share x, in one pass (no counterpart on the pages; it carries
 * their fusion one step further): for each item i,
 *     dst_i = epilogue_i(W_i x')          (x' = x after the prologue in `opts`)
 * e.g. a layer's q, k and v projections (and a small gate such as a sigmoid head) on the
 * same activations, without concatenating their weights.  One launch streams every
 * matrix once, as one matrix of sum_i M_i rows: the fixed cost of a launch is paid once.
 *  items : n items (1 <= n <= GF_MULTI_MAX, else GF_ERR_INVALID / GF_ERR_UNSUPPORTED),
 *          each a matrix W (M rows of format `wtype`, K columns; the rules of W in
 *          gemv_fused) with its own epilogue, aux ([ncols][M], required iff SILU_MUL or
 *          ADD) and dst ([ncols][M]).
 *  x, K, wtype, opts : shared; opts as in gemv_fused_ex (ncols, either prologue,
 *          flags) except `view_ne`, which must be all zero.
 *  Aliasing: each dst as in gemv_fused against its own operands, and it may not overlap
 *  any other item's W, aux or dst (GF_ERR_ALIAS).  The results equal those of the n
 *  separate calls bit for bit (the same per-row arithmetic).  Shapes the streamed kernel
 *  cannot take in one pass run as one launch per matrix. */
#define GF_MULTI_MAX 4
typedef struct {
  const void* W;
  int64_t M;
  int epilogue;
  const float* aux;
  float* dst;
} gf_multi_item;
GF_API int gemv_multi(const gf_multi_item* items, int n, int wtype, const float* x, int64_t K,
                      const gf_opts* opts, void* stream);

/* Prepared calls: plan once, launch many times.  A decode loop issues the same GEMVs
 * with the same buffers every step; gf_prepare / gf_prepare_glu validate and plan a
 * call exactly as gemv_fused_ex / gemv_glu would (same arguments, same rules, same
 * status codes) and keep every launch argument, so gf_launch_prepared only issues the
 * kernels: no validation, planning or allocation per step.  The results are the ones
 * the direct call gives (the same kernels with the same arguments).
 *  out      : receives a handle owned by the caller, released with gf_free_prepared;
 *             NULL on failure.  A call with M == 0 gives a handle that launches nothing.
 *  (gf_prepare_multi plans gemv_multi the same way.)
 *  Buffers  : the handle holds the device pointers given here (W, x, aux, dst, opts'
 *             signs, workspace and RMS weight); their contents may change between
 *             launches, the allocations must stay valid while the handle is used.
 *  Device   : the handle belongs to the device current at gf_prepare; launching it
 *             with another device current returns GF_ERR_INVALID. */
typedef struct gf_prepared gf_prepared;
GF_API int gf_prepare(const void* W, int wtype, const float* x, int64_t M, int64_t K, int epilogue,
                      const float* aux, float* dst, const gf_opts* opts, gf_prepared** out);
GF_API int gf_prepare_glu(const void* W_gate, const void* W_up, int wtype, const float* x, int64_t M,
                          int64_t K, float* dst, const gf_opts* opts, gf_prepared** out);
GF_API int gf_prepare_multi(const gf_multi_item* items, int n, int wtype, const float* x, int64_t K,
                            const gf_opts* opts, gf_prepared** out);
/* Issues the launches of calls[0], ..., calls[n-1] in order on `stream` (n >= 0; the
 * calls' GF_FLAG_PDL settings apply as given to gf_prepare).  Stops at the first
 * failing launch and returns its status; GF_ERR_INVALID (nothing launched) for a NULL
 * handle or one prepared on another device. */
GF_API int gf_launch_prepared(const gf_prepared* const* calls, int n, void* stream);
/* Releases a handle (NULL is ignored).  Launches already issued are not affected. */
GF_API void gf_free_prepared(gf_prepared* p);

/* Host staging of a decode step by a kernel instead of the copy engine, so that a step's
 * input upload, its GEMVs and its result download can be one stream sequence or one CUDA
 * graph (gf_graph_create takes the handle of gf_prepare_copy like any prepared call).
 * Copies `bytes` bytes from src to dst; each range may be device memory of the current
 * device, managed memory, or pinned host memory (cudaHostAlloc / cudaMallocHost, or
 * registered with cudaHostRegister).
 *  - src and dst 16-byte aligned (GF_ERR_ALIGN), bytes >= 0 and a multiple of 16
 *    (GF_ERR_INVALID), the ranges disjoint (GF_ERR_ALIAS); pageable host memory, or
 *    device memory of another device: GF_ERR_INVALID (nothing launched).  bytes == 0
 *    launches nothing.
 *  - flags: GF_FLAG_PDL launches it with programmatic dependent launch; the kernel
 *    waits for the preceding grid before reading src, so it may read what that grid
 *    wrote, and the next launch may start early (every kernel of this library waits
 *    before reading what a preceding grid writes).
 *  - Host memory written here is complete when the stream (or graph launch) is; the
 *    copy uses no copy engine and is not ordered with copies in other streams. */
GF_API int gf_copy(void* dst, const void* src, int64_t bytes, uint32_t flags, void* stream);
GF_API int gf_prepare_copy(void* dst, const void* src, int64_t bytes, uint32_t flags, gf_prepared** out);

/* A decode step as one launch: gf_graph_create records the launches of calls[0..n)
 * (n >= 1, in order, as gf_launch_prepared would issue them, programmatic dependent
 * launches included) into a CUDA graph and instantiates it; gf_graph_launch replays it
 * on `stream` -- one host call for the whole sequence, and the launch overhead of a
 * graph instead of one per kernel.  The graph keeps the prepared calls' arguments
 * (the handles may be freed afterwards; their buffers must stay allocated).  It belongs
 * to the device current at creation (another one: GF_ERR_INVALID).  Errors: NULL or
 * foreign handles GF_ERR_INVALID; a failing capture or instantiation GF_ERR_CUDA. */
typedef struct gf_graph gf_graph;
GF_API int gf_graph_create(const gf_prepared* const* calls, int n, gf_graph** out);
GF_API int gf_graph_launch(const gf_graph* g, void* stream);
GF_API void gf_graph_free(gf_graph* g);

/* Allocation-free variant of gemv_fused_ex with the signed-FWHT prologue.  The pages
 * have no counterpart: this entry point exists for callers that cannot allocate a
 * device workspace -- a C host that links only this library and has no device
 * allocator of its own, or a serving process whose device memory is fixed at start-up
 * and may not grow while requests run.  It computes exactly what gemv_fused_ex computes
 * with opts = {ncols, fwht_signs, fwht_block, nsigns, flags} and a workspace, but the
 * workspace (the transformed x', ncols*K floats) is a static device array inside the
 * library; nothing is allocated or freed.
 *  - Limit: ncols*K <= GF_NOALLOC_MAX_WORKSPACE_FLOATS, else GF_ERR_UNSUPPORTED with
 *    nothing launched.  fwht_signs must be non-NULL (GF_ERR_INVALID otherwise).
 *  - The array (1 MiB) is held on every GPU that loads the library until the process
 *    exits.  The first call on a device looks up its address (cudaGetSymbolAddress,
 *    with that device current); make that first call before any stream capture.
 *  - Every call on a device shares the one array and overwrites it before reading it;
 *    calls whose work overlaps on the GPU (e.g. on different streams without ordering)
 *    race on it and give undefined results: order them, e.g. on one stream.
 *  - The address is kept for the life of the process.  Destroying the device's primary
 *    context (cudaDeviceReset) invalidates it, as it does the library's device error
 *    word: after a reset, reload the library before calling it again. */
#define GF_NOALLOC_MAX_WORKSPACE_FLOATS 262144
GF_API int gemv_fused_fwht_noalloc(const void* W, int wtype, const float* x, int64_t M, int64_t K,
                                   int epilogue, const float* aux, float* dst, int64_t ncols,
                                   const float* fwht_signs, int64_t fwht_block, int64_t nsigns,
                                   uint32_t flags, void* stream);

/* Signed FWHT, stand-alone ([FWHT] Overview): for every block of `block` consecutive
 * elements of x[0..n), dst_b = H_block (x_b * s) / sqrt(block), with element i using
 * signs[i % nsigns]; signs == NULL means all +1 (the plain normalised transform).
 *  block : power of two, 1..16384, n % block == 0;  n % nsigns == 0 when signs != NULL.
 *  dst == x is allowed (in place); other overlaps with x or signs: GF_ERR_ALIAS. */
GF_API int fwht_signed(const float* x, const float* signs, float* dst, int64_t n,
                int64_t block, int64_t nsigns, void* stream);

/* Unfused control ([CPU] Correctness compares fused against unfused outputs):
 * dst[i] = op(a[i], b[i % nb]) for i < n; SIGMOID and SILU ignore b.  Uses the same
 * device functions as the fused tails.  dst may equal a or b exactly. */
GF_API int gf_elementwise(int op, const float* a, const float* b, int64_t nb, float* dst,
                   int64_t n, void* stream);

/* Test hook: out[i*K + k] = decoded W[i][k] as float32, through the same unit decoders
 * the fast GEMV kernel uses.  Every decoded value is exact in float32. */
GF_API int gf_dequantize(const void* W, int wtype, int64_t M, int64_t K, float* out, void* stream);

/* Which kernel gemv_fused_ex would launch for these arguments (host only, launches
 * nothing): 0 = none (M == 0), 1 = TMA-streamed kernel, 2 = generic kernel, 3 = tensor-core
 * kernel (F16 batches), <0 = the gf_status the call would return.  `info` (may be NULL) receives
 *   {grid, block_threads, stage_rows, stages, k_chunk, smem_bytes, row_chunk,
 *    ctas_per_cluster (split K; 1 = no split)}. */
GF_API int gf_plan(const void* W, int wtype, const float* x, int64_t M, int64_t K, int epilogue,
            const float* aux, const float* dst, const gf_opts* opts, int64_t info[8]);

/* gf_plan for gemv_glu. */
GF_API int gf_plan_glu(const void* W_gate, const void* W_up, int wtype, const float* x, int64_t M,
                       int64_t K, const float* dst, const gf_opts* opts, int64_t info[8]);

/* Failure-path self-test (no GEMV): one GPU thread waits, through the same bounded wait
 * every kernel uses, on a barrier that nothing completes.  After limit_us microseconds
 * (1..1000000) the wait gives up, sets the device error word (gf_device_status then
 * reports GF_ERR_TIMEOUT) and the kernel returns; the context stays usable.  out: device
 * int[4] = {first wait succeeded (0), second wait succeeded (0: it returns at once on the
 * abort flag), microseconds spent in the first wait, microseconds in the second}. */
GF_API int gf_selftest_wait_timeout(int64_t limit_us, int* out, void* stream);

/* Device error word of the current device: GF_OK, or GF_ERR_TIMEOUT if a kernel gave up
 * on a bounded wait since the last reset.  Synchronises with the device.  reset != 0
 * clears it. */
GF_API int gf_device_status(int reset);

/* Row chunks (a CTA's rows of one launch, or of one row chunk of it) whose sums the
 * single-column Q4_0 / Q8_0 / Q4_K kernels recomputed in fp32 because some 16-element
 * unit of x could not be carried by their integer dot products (an outlier far above
 * the values around it, or a NaN / Inf): a count since the last reset, on the current
 * device.  Such a launch reads its weights twice; the count says how often that
 * happens for a workload.  Synchronises with the device; reset != 0 clears it.
 * Negative: a gf_status (GF_ERR_CUDA). */
GF_API int64_t gf_repair_count(int reset);

/* Human-readable name of a gf_status value. */
GF_API const char* gf_status_string(int status);

/* cudaError_t of the last failing CUDA call made by this library in this thread. */
GF_API int gf_last_cuda_error(void);

/* Library ABI version. */
GF_API int gf_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GEMVFUSE_H */
