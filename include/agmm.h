/*
 * agmm -- fused all-gather matmul for one GB300 (sm_103a).  C ABI.
 *
 * The operation ("Add all gather matmul benchmark", pytorch/helion PR #400,
 * statement of the op):
 *
 *     (a, out) = ag_matmul(a_shared, b),  a = all_gather(a_shared),  out = a @ b
 *
 * Here the D row shards of A are D separate device allocations on the same
 * GPU (they stand in for D ranks).  The library writes the gathered matrix
 * a_gathered = concat_rows(a_shards[0..D-1]) ([M, K], M = D * m_per_shard) and
 * out = a_gathered @ b (+ bias) ([M, N]).  Inputs and outputs are 16-bit
 * (bf16 by default, or fp16); products are summed in fp32 and rounded once,
 * to nearest even, after the optional fp32 bias is added ("Fused
 * all-gather+GEMM HBM-buffer kernel for iris.ops", ROCm/iris #346, section
 * "New kernel": optional bias in the epilogue).
 *
 * ag_matmul runs the fused design of that Iris kernel (section "New kernel"
 * and its description): one persistent kernel in which A tiles are copied
 * from the shards into an HBM staging buffer and per-tile ready flags are
 * published, while tensor-core warps wait on those flags and compute each
 * output tile as soon as its A rows are staged -- no whole-gather barrier.
 * Here every chunk of A (a 128-row block x k_per_flag k-blocks) has an owner
 * tile, which loads it from its shard with TMA for its own MMA and hands it
 * to its CTA's copier warps; they copy it into the staging buffer and publish
 * its flag, and the other tiles wait on that flag and read the staged copy.
 * When a call takes at most three waves and the last one is partial, the CTAs
 * with one tile fewer copy all of A first instead, and every tile waits on the
 * flags.  Tiles that lie inside the local shard (option `rank`) are read
 * straight from that shard without waiting (the local-tile shortcut
 * described in the Helion PR).  ag_then_matmul is the barrier baseline of the
 * Iris result tables ("Baseline" column): gather everything, then run the
 * GEMM.
 *
 * Common argument contract (every entry point below that takes these):
 *   a_shards      HOST array of D DEVICE pointers; shard r is row-major
 *                 [m_per_shard, K], contiguous, 16-byte aligned.  Read only.
 *   D             number of shards, 1 <= D <= AG_MAX_SHARDS.
 *   m_per_shard   rows per shard, >= 1.  M = D * m_per_shard <= 2^31 - 1.
 *   K             columns of A / rows of b; >= 8 and a multiple of 8 (row
 *                 pitches must be multiples of 16 bytes for TMA).
 *   b             DEVICE pointer, row-major [K, N], 16-byte aligned.  Read only.
 *   N             columns of b and out; >= 8 and a multiple of 8.
 *   bias_or_null  DEVICE pointer to N fp32 values (4-byte aligned) or NULL.
 *   a_gathered    DEVICE pointer, row-major [M, K], 16-byte aligned.  Written.
 *   out           DEVICE pointer, row-major [M, N], 16-byte aligned.  Written.
 *   stream        CUDA stream the work is enqueued on (0 = legacy default).
 * The caller allocates and owns every pointer argument.  Outputs must not
 * overlap each other or any input.  The dtype of a_shards, b, a_gathered and
 * out is the same (ag_options.dtype; bf16 for the entry points without
 * options), except with AG_DTYPE_FP8_E4M3 (8-bit inputs, b transposed, bf16
 * out; see ag_dtype).
 *
 * Semantics: asynchronous.  A call validates its arguments, enqueues one
 * (fused) or two (barrier) kernels on `stream` and returns; it never
 * synchronises the host.  On any error return nothing has been enqueued.
 * Inputs must stay unchanged until the stream has executed the call.
 *
 * Errors: the return value is an ag_status.  Device-side failures (a ready
 * flag or pipeline wait that exceeded its time limit) cannot be returned by
 * an asynchronous call; the kernel records them and ag_get_device_error()
 * reports them.  No kernel of this library traps or faults on purpose: every
 * device-side wait is bounded by a time limit.
 *
 * Workspace: the fused path needs ready flags (8 bytes per (128-row block,
 * k-group)) and one word per output tile (8 bytes per 128 x 256 tile); both
 * paths need a [K, M] staging buffer for the m-contiguous layout.  By default
 * the library owns them (one set per device, grown on demand; growing
 * synchronises the device).  Calls on one workspace must not overlap on the
 * GPU.  For the library workspace this is checked: the library remembers the
 * stream of the last call that used it and an event recorded after that
 * call; a call on another stream while that event has not completed returns
 * AG_ERR_BUSY and enqueues nothing (the library cannot see an ordering that
 * the caller set up between streams with events, so such a call is refused
 * rather than allowed to race).  Calls on the same stream are ordered by the
 * stream and never busy.  Work that must overlap on several streams passes a
 * caller workspace per stream (ag_options.workspace); the library does not
 * track those.
 */
#ifndef AGMM_H_
#define AGMM_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AG_MAX_SHARDS 16

/* Return codes. */
typedef enum ag_status {
  AG_OK = 0,
  AG_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment, overlap or option value */
  AG_ERR_UNSUPPORTED = 2, /* valid request the library cannot run (device, dtype/layout combo, D > AG_MAX_SHARDS) */
  AG_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed; see ag_status_string */
  AG_ERR_TIMEOUT = 4,     /* device-side: a bounded wait ran out (reported by ag_get_device_error) */
  AG_ERR_WORKSPACE = 5,   /* caller workspace smaller than ag_workspace_size() */
  AG_ERR_TOO_LARGE = 6,   /* problem needs more than ag_matmul_noalloc's fixed scratch */
  AG_ERR_BUSY = 7,        /* the library workspace is in use by an unfinished call on another
                             stream; nothing was enqueued (see "Workspace" above) */
  AG_ERR_BOUNDS = 8       /* device-side, bounds-checked build only (libagmm_debug.so): an
                             index fell outside its buffer; the access was skipped
                             (reported by ag_get_device_error; info = site << 24 | index) */
} ag_status;

/* Storage types.  AG_DTYPE_FP8_E4M3 is an extension the pages do not cover:
 * 8-bit A and b in the OCP FP8 E4M3 encoding (1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN), with per-tensor
 * scales ag_options.scale_a and scale_b.  With it:
 *   a_shards[r]  [m_per_shard, K] e4m3, row-major;
 *   b            given TRANSPOSED: [N, K] e4m3, row-major (K fastest), the
 *                layout FP8 GEMMs take their second operand in;
 *   a_gathered   [M, K] e4m3;
 *   out          [M, N] bf16:  out = bf16(scale_a * scale_b * (a @ b) + bias),
 *                products and sums in fp32, the scale applied to the fp32 sum;
 *   K % 16 == 0 (16-byte rows), N % 8 == 0, layout k-contiguous only (the
 *   m-contiguous staging returns AG_ERR_UNSUPPORTED for it); every entry
 *   point (fused, barrier, chunked, no-alloc) accepts it. */
typedef enum ag_dtype { AG_DTYPE_BF16 = 0, AG_DTYPE_FP16 = 1, AG_DTYPE_FP8_E4M3 = 2 } ag_dtype;

/* Layout of the staged A in HBM ("Fused all-gather+GEMM HBM-buffer kernel for
 * iris.ops", section "New kernel": k_contiguous and m_contiguous staged-A
 * layouts; the page names them without defining them).  Reading used here:
 *   AG_LAYOUT_K_CONTIGUOUS  staged A is [M, K] row-major (K fastest); this is
 *                           a_gathered itself.
 *   AG_LAYOUT_M_CONTIGUOUS  staged A is additionally written as [K, M]
 *                           row-major (M fastest) and the GEMM reads it from
 *                           there; requires M % 8 == 0.
 * a_gathered is [M, K] row-major in both cases. */
typedef enum ag_layout { AG_LAYOUT_K_CONTIGUOUS = 0, AG_LAYOUT_M_CONTIGUOUS = 1 } ag_layout;

/* Options of the *_ex entry points.  Start from ag_options_default(). */
typedef struct ag_options {
  int32_t dtype;            /* ag_dtype of a_shards, b, a_gathered, out (default bf16) */
  int32_t layout;           /* ag_layout of the staged A (default k-contiguous) */
  int32_t rank;             /* the local shard, 0 <= rank < D (default 0) */
  int32_t k_per_flag;       /* 64-column K blocks covered by one ready flag; 0 = automatic
                               (default): when every output tile fits in one wave of the
                               grid, K blocks per 256-column block clamped to [4, 8], else
                               8 (k-contiguous) or 16 (m-contiguous); at most the number
                               of K blocks */
  int32_t num_sms;          /* cap on the persistent grid (CTAs); 0 = every SM */
  int32_t inject_skip_flag; /* fault injection: the producer never publishes this flag index
                               (-1 = off); the consumer wait then times out */
  int64_t timeout_ns;       /* limit of one device-side ready-flag wait; 0 = 2 s.  Pipeline
                               waits inside a CTA use 4x this plus 2 s. */
  uint64_t* trace;          /* DEVICE buffer for timeline records or NULL; see ag_trace_* */
  int64_t trace_words;      /* capacity of `trace` in 64-bit words */
  void* workspace;          /* caller-owned DEVICE workspace or NULL (library-owned) */
  int64_t workspace_bytes;  /* its size; must be >= ag_workspace_size() */
  float scale_a;            /* AG_DTYPE_FP8_E4M3: per-tensor scale of A (default 1); ignored otherwise */
  float scale_b;            /* AG_DTYPE_FP8_E4M3: per-tensor scale of b (default 1); must be finite */
  int64_t inject_delay_ns;  /* stress testing (fused calls): every publisher of a ready flag
                               waits a pseudo-random 0 .. inject_delay_ns after its copies and
                               before the release store that publishes them, so readers meet
                               late publishers.  0 = off (default); at most timeout_ns / 16
                               (the default 2 s timeout allows 125 ms), else
                               AG_ERR_INVALID_ARG.  Results are unchanged. */
  /* Tile and pipeline shape.  The pages' tunables ("Fused all-gather+GEMM
   * HBM-buffer kernel for iris.ops", the defaults table: block sizes,
   * num_stages, fetch SMs).  0 = automatic (default).  Only the shapes the
   * library is compiled for are accepted; any other positive value is
   * AG_ERR_UNSUPPORTED, a negative one AG_ERR_INVALID_ARG. */
  int32_t block_m;          /* output rows per tile: 256 (a CTA pair per tile) or 128 (one CTA
                               per tile).  Automatic: 256 when at least two SMs are allowed,
                               except calls with K of at most 32 k-blocks (2048 16-bit
                               elements) whose 128-row tiles all fit one wave: 128 */
  int32_t block_n;          /* output columns per tile: 256 */
  int32_t block_k;          /* K per pipeline stage, in elements: 64 (16-bit) or 128 (FP8) */
  int32_t stages;           /* pipeline depth: 6 with block_m 256, 4 with block_m 128 (a value
                               alone also selects block_m) */
  int32_t producer_warps;   /* copier warps per CTA that stage A chunks: 4 */
} ag_options;

/* Fill `opt` with the defaults listed above.  Never fails (NULL is ignored). */
void ag_options_default(ag_options* opt);

/* Fused all-gather matmul, bf16, k-contiguous staging, rank 0.
 * Equivalent to ag_matmul_ex with ag_options_default(). */
int ag_matmul(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
              const void* bias_or_null, void* a_gathered, void* out, cudaStream_t stream);

/* Barrier baseline: a gather kernel writes a_gathered, then a GEMM kernel
 * (the same tensor-core mainloop and epilogue, without flags) reads it.
 * Results are bit-identical to ag_matmul's.  bf16. */
int ag_then_matmul(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
                   const void* bias_or_null, void* a_gathered, void* out, cudaStream_t stream);

/* As above with options (opt may be NULL for the defaults).  ag_then_matmul_ex
 * honours dtype, layout, num_sms, timeout_ns, trace and the tile options
 * (block_m ... producer_warps): with the m-contiguous layout its gather kernel
 * also writes the [K, M] staging (library-owned) and the GEMM reads A from
 * there.  It ignores rank, k_per_flag, inject_skip_flag, inject_delay_ns and
 * the caller workspace. */
int ag_matmul_ex(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
                 const void* bias_or_null, void* a_gathered, void* out, cudaStream_t stream,
                 const ag_options* opt);
int ag_then_matmul_ex(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
                      const void* bias_or_null, void* a_gathered, void* out, cudaStream_t stream,
                      const ag_options* opt);

/* The chunked pipeline: the same operation as ag_then_matmul_ex, run as the
 * stream-pipelined AG+GEMM of "Lower distributed matmul to pipelined
 * algorithm for fine-grained overlap: AG+GEMM layout" (NVIDIA/Fuser #3695,
 * section "What"): A is taken as [S, D, m_per_shard / S, K] with S = `chunks`
 * (at most m_per_shard / 128, at least 1: a shorter sub-block would be padded
 * to a 128-row tile), so chunk s is the s-th sub-block of every shard
 * (local rows [s*m/S, (s+1)*m/S)).  Chunk by chunk, round-robin over four
 * library-owned streams that fork from and join back to `stream`: gather the
 * chunk into a_gathered (every shard contributes), then multiply its D row
 * segments into the same rows of out (one launch of the barrier GEMM core over
 * the D segments).  A chunk's GEMMs wait for the chunk's whole gather; different
 * chunks overlap.  Results equal ag_then_matmul_ex's bitwise (same GEMM core
 * and k order).  Arguments and errors as for ag_then_matmul_ex; chunks < 1 or
 * > 4096 is AG_ERR_INVALID_ARG, the m-contiguous layout AG_ERR_UNSUPPORTED.
 * The first call on a device creates the four streams and five events (no
 * device memory); they live until the process ends. */
int ag_chunked_matmul_ex(const void** a_shards, int D, int m_per_shard, int K, const void* b,
                         int N, const void* bias_or_null, void* a_gathered, void* out,
                         cudaStream_t stream, const ag_options* opt, int chunks);

/* Bytes a caller workspace must hold for a fused call of this shape and
 * these options (flags, plus the [K, M] staging for the m-contiguous layout).
 * With the automatic k_per_flag the flags are sized for the finest automatic
 * granularity (4), which covers whatever a launch picks.
 * The workspace must be 256-byte aligned and zero-filled before its first use
 * with this library; after that the library owns its contents.  Returns 0 on
 * invalid sizes. */
size_t ag_workspace_size(int D, int m_per_shard, int K, int N, const ag_options* opt);

/* Synchronises `stream`, then reports the newest device-side error recorded
 * on the current device by a call made since the previous report.  Errors are
 * kept in two places -- the library's error word and ag_matmul_noalloc's
 * scratch -- and when both hold an unreported error, the one of the later
 * call is reported and the other stays for the next report.  *code is AG_OK
 * when there is none; *info is the flag index or pipeline site that timed
 * out.  Either pointer may be NULL.  Returns AG_OK or AG_ERR_CUDA. */
int ag_get_device_error(cudaStream_t stream, int* code, int* info);

/* Frees the library-owned workspace of the current device (synchronises the
 * device first).  The next call allocates it again. */
int ag_release_workspace(void);

/* Static description of a status code; for AG_ERR_CUDA the text of the most
 * recent CUDA failure seen by this thread.  Never NULL. */
const char* ag_status_string(int status);

/* Number of SMs the persistent kernels size their grid by on the current
 * device (0 if no device). */
int ag_num_sms(void);

/* The launch plan of a fused call (ag_matmul, ag_matmul_ex,
 * ag_matmul_noalloc) with these sizes and options, on a device with `sms`
 * SMs where `pair_clusters` clusters of two CTAs fit at once (0: single
 * CTAs).  Host arithmetic only: no CUDA call and nothing launched, so it runs
 * without a GPU too.  K counts elements (FP8: bytes), as in the calls.
 * Returns AG_OK and fills *plan (caller-owned), or the status the calls
 * would return for these sizes and options (pointers are not checked). */
typedef struct ag_plan {
  int32_t grid;           /* CTAs launched (even with CTA pairs) */
  int32_t cta_pairs;      /* 1: 256 x 256 tiles on CTA pairs; 0: 128 x 256 on single CTAs */
  int32_t tiles;          /* output tiles (pair tiles with CTA pairs) */
  int32_t k_per_flag;     /* k-blocks (64 elements; FP8: 128 bytes) per ready flag */
  int32_t prologue_cta0;  /* fetch prologue: CTAs from this index first stage all of A; -1: none */
  int32_t l2_prefetch;    /* 1: the kernel first prefetches all of A into L2 */
  int32_t block_m;        /* output rows per tile (256: CTA pairs, 128: single CTAs) */
  int32_t stages;         /* pipeline depth */
  int32_t k_ascending;    /* 1: every tile runs k ascending (calls of four or more waves; the
                             results then equal ag_then_matmul_ex's with the same tile
                             options bit for bit); 0: each tile starts at the k-range it
                             owns.  With the m-contiguous layout on CTA pairs, such calls
                             also read pairs wholly in the local shard straight from it */
} ag_plan;
int ag_plan_fused(int D, int m_per_shard, int K, int N, const ag_options* opt, int sms,
                  int pair_clusters, ag_plan* plan);

/* Size of the fixed device scratch that ag_matmul_noalloc uses (see below). */
#define AG_NOALLOC_SCRATCH_BYTES (256 * 1024)

/* ag_matmul_noalloc -- the fused all-gather matmul for callers that cannot
 * allocate device memory.  (No counterpart on the pages: this is a library
 * convenience, not part of the method.)
 *
 * Who needs it: code that must not call cudaMalloc/cudaFree (or any routine
 * that may allocate, torch's caching allocator included) when it runs --
 * e.g. a host framework that plans and owns every device allocation up
 * front, or a latency-critical loop where an allocation's implicit device
 * synchronisation is not acceptable.  ag_matmul may allocate: its first call
 * on a device creates the error word and the flag workspace, and a larger
 * problem later grows the workspace.
 *
 * What it does: exactly what ag_matmul_ex does for the k-contiguous layout
 * (same kernel, same results bit for bit), but the kernel's scratch -- its
 * error word, the ready flags and the per-tile words -- lives in one
 * file-scope device array of AG_NOALLOC_SCRATCH_BYTES bytes inside this
 * library.  Every GPU that loads the library holds that array until the
 * process exits.  The caller still passes (and owns) every input and output.
 *
 * Limits and errors: ag_options.layout must be AG_LAYOUT_K_CONTIGUOUS
 * (m-contiguous staging needs K * M * 2 bytes; AG_ERR_UNSUPPORTED otherwise)
 * and ag_options.workspace must be NULL (AG_ERR_INVALID_ARG).  A problem whose
 * scratch -- 256 bytes plus ag_workspace_size() for the k-contiguous layout --
 * exceeds AG_NOALLOC_SCRATCH_BYTES is rejected with AG_ERR_TOO_LARGE before
 * anything is enqueued.  With the automatic k_per_flag that admits, for
 * example, M = 16384, N = 3584, K = 8192 (about 48 KB of scratch).  All other
 * arguments and errors are as for ag_matmul_ex; device-side timeouts are
 * reported by ag_get_device_error.
 *
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents.  Nothing in it needs clearing between calls: flags and
 * per-tile words carry the call's epoch, so values left by earlier calls
 * read as untouched.  Calls whose kernels may overlap on the GPU (different
 * streams without ordering) race on the array and give wrong results; order
 * them on one stream or with events.
 *
 * Set-up: the first call on each device, made with that device current, does
 * one-time set-up: it looks up the array's device address (the array's name
 * in host code is only a stand-in for it) and sets the kernel's shared-memory
 * limit.  Those are CUDA runtime calls that should not run while a stream is
 * being captured, so make that first call before any stream capture begins.
 * No call performs a device allocation or free. */
int ag_matmul_noalloc(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
                      const void* bias_or_null, void* a_gathered, void* out,
                      cudaStream_t stream, const ag_options* opt);

/* Timeline records.  When ag_options.trace is set, word 0 of the buffer is an
 * atomic record counter (the caller zeroes it) and record i occupies words
 * 1 + 4*i .. 4 + 4*i: {t_start_ns, t_end_ns, meta, 0}, times from the GPU's
 * global nanosecond timer.  meta = role << 56 | cta << 40 | a << 20 | b with
 * the roles below.  Records beyond the capacity are dropped (the counter
 * still counts them). */
#define AG_TRACE_CLAIM 1u    /* a CTA claimed a chunk and loads it from its shard
                                (a = 128-row block, b = k-group; t_start = t_end) */
#define AG_TRACE_WAIT 2u     /* a CTA waited for a chunk's ready flag (a = block, b = k-group) */
#define AG_TRACE_TILE 3u     /* epilogue stored an output tile (a = row block, b = column block) */
#define AG_TRACE_GATHER 4u   /* barrier path: a gather-kernel CTA ran (a = CTA, b = 0) */
#define AG_TRACE_REGFETCH 5u /* a chunk TMA cannot address was copied by registers (a, b) */
#define AG_TRACE_ISSUE 6u    /* one chunk's A loads were decided (barrier GEMM: issued; fused:
                                the protocol warp handed the chunk to the A loader, flag checks
                                included) (a = block, b = k-group | 1 << 16 if read straight
                                from a shard | 2 << 16 if this CTA staged it) */

#ifdef __cplusplus
}
#endif

#endif /* AGMM_H_ */
