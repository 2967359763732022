/*
 * moe_router.h -- C ABI of the GB300 (sm_103a) routed mixture-of-experts
 * forward for small decode, speculative-verify and prefill sub-chunks
 * (1..8 token rows).
 *
 * The operation is the routed MoE layer of page "Function forward_moe"
 * (forward_moe(gpu, k, cfg, w, x, out, rows, ws, stream), which applies the
 * routed experts to each of `rows` token rows and runs the shared expert once
 * for all of them) and of page
 * "metrale_model_layers/layers/moe/forward_token_major.rs"
 * (MoeLayer::forward_token_major_decode: gate projection, batched top-k,
 * gate+up, silu+down, weighted sum + shared-expert blend).  The union of the
 * experts selected by all rows is built on the device by pairwise scan, as
 * the forward_moe page's RETRACTED note describes, and every union expert's
 * NVFP4 weights are streamed once for all the rows that selected it; the
 * selected ids never travel to the host.
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" point to GPU global memory of the current
 *     device; "host" pointers to CPU memory.  The caller owns every buffer;
 *     the library never allocates, frees or synchronises inside moe_route,
 *     moe_union or moe_forward.  Work is enqueued on `stream` (a
 *     cudaStream_t passed as void*, NULL = the legacy default stream) and
 *     returns immediately.
 *   - bf16 values travel as uint16_t bit patterns.
 *   - Every argument check runs on the host before the first launch; a
 *     refused call enqueues nothing and returns a non-zero moe_status whose
 *     text moe_last_error() gives (per calling thread).
 *   - A launch failure reported by the CUDA runtime returns MOE_ERR_CUDA.
 *   - Faults the device detects (an expert id out of range, a weight pointer
 *     that is not 16-byte aligned, a wait that ran out of time) never trap:
 *     the kernel records a code in the workspace's status word, skips the
 *     offending work and finishes; moe_read_device_status() returns it.
 *
 * NVFP4 matrix [N][K] (N outputs, K inputs, "untransposed"):
 *   packed  uint8 [N][K/2], row-major; the low nibble holds the even input
 *           index, each nibble an FP4 E2M1 code (sign, 2 exponent bits with
 *           bias 1, 1 mantissa bit);
 *   scales  uint8 [N][K/16], row-major; one FP8 E4M3 (bias 7, no infinity)
 *           scale per 16 contiguous inputs;
 *   scale2  fp32, one per matrix.
 *   weight[n][k] = e2m1(code) * e4m3(scale) * scale2.
 *   Both arrays must start on a 16-byte boundary.
 *
 * The same matrix in the t layout (the transposed decode layout that the
 * forward_token_major.rs page names -- use_t_layout_for_decode -- without
 * defining it; this library stores the down projections that way when
 * moe_config.t_layout = 1): the same codes and the same 16-input scale
 * blocks, stored input-major:
 *   packed  uint8 [K][N/2]; element (n, k) in byte k * N/2 + n/2, the low
 *           nibble holding the even output index;
 *   scales  uint8 [K/16][N]; the scale of (n, inputs 16b .. 16b+15) in
 *           byte b * N + n;
 *   scale2  unchanged.
 * moe_nvfp4_to_t_layout converts a matrix (or a stack of them).
 */
#ifndef MOE_ROUTER_H
#define MOE_ROUTER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#define MOE_ABI_VERSION 3
#define MOE_MAX_ROWS 32       /* rows per call */
#define MOE_MAX_IDS 256       /* rows * top_k per call (the union's capacity) */
#define MOE_CHUNK_ROWS 8      /* rows per sub-chunk of the expert sweep ... */
#define MOE_CHUNK_IDS 64      /* ... whose union of at most 64 ids fits one
                                 block's pairwise scan (forward_moe page,
                                 WIDENED note: 8 * 8 == 64) */
#define MOE_MAX_HIDDEN 4096
#define MOE_MAX_EXPERTS 1024

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* null / misaligned pointer, size out of range */
    MOE_ERR_UNSUPPORTED = 2,    /* a configuration this path refuses */
    MOE_ERR_WORKSPACE = 3,      /* workspace missing, too small or misaligned */
    MOE_ERR_CUDA = 4,           /* the CUDA runtime reported an error */
    MOE_ERR_DEVICE_STATUS = 5   /* the device recorded a fault (see below) */
} moe_status;

/* Device-side fault codes (moe_read_device_status). */
#define MOE_DEV_OK 0
#define MOE_DEV_BAD_EXPERT_ID 1     /* an id outside [0, num_experts) */
#define MOE_DEV_MISALIGNED_PTR 2    /* an expert matrix not 16-byte aligned */
#define MOE_DEV_WAIT_TIMEOUT 3      /* an on-chip wait exceeded its bound
                                       (about two seconds); the launch skipped
                                       the rest of its work.  The workspace
                                       stays usable as it is: the next launch
                                       runs its grid barriers on a counter the
                                       failed launch zeroed, so no
                                       moe_workspace_init is needed */

enum { MOE_SCORING_SOFTMAX = 0, MOE_SCORING_SIGMOID = 1 };
enum { MOE_ROUTER_BF16 = 0, MOE_ROUTER_NVFP4 = 1 };
/* Expert matrix formats (moe_config.expert_fmt; routed and shared experts):
 *   NVFP4: as described at the top of this file;
 *   FP8:   packed uint8 [N][K], one E4M3 (bias 7, no infinity) code per
 *          weight, row-major; scales not used (may be NULL); weight =
 *          e4m3(code) * scale2;
 *   BF16:  packed [N][K] bfloat16 (2 bytes per weight, little-endian),
 *          row-major; scales not used (may be NULL); weight = bf16 * scale2.
 * The forward_token_major.rs page names BF16 and FP8 experts as formats its
 * token-major path hands to another path, without giving their layout; the
 * layouts above are this library's reading.  A 16-row tile of an FP8 or
 * BF16 matrix is 16*K or 32*K bytes.  BF16 gate/up tiles too large for two
 * shared-memory ring slots are streamed in two K-halves (hidden up to 4096,
 * when hidden/128 is even), and FP8 or BF16 down tiles too large for two
 * slots in K-parts of whole 128-input chunks (intermediates up to 4096);
 * configurations whose tiles still do not fit (BF16 gate/up tiles of an odd
 * number of chunks beyond the ring, for example) are refused at the first
 * forward (MOE_ERR_UNSUPPORTED). */
enum { MOE_EXPERT_NVFP4 = 0, MOE_EXPERT_FP8 = 1, MOE_EXPERT_BF16 = 2 };

/* One NVFP4 matrix whose pointers the host knows (router, shared expert). */
typedef struct moe_nvfp4 {
    const uint8_t *packed;   /* device, [N][K/2] */
    const uint8_t *scales;   /* device, [N][K/16] */
    float scale2;            /* per-tensor scale */
} moe_nvfp4;

/* Layer configuration (page "Function forward_moe": Glm5NextMlpConfig;
 * forward_token_major.rs: hidden_size, moe_intermediate_size, num_experts,
 * num_experts_per_tok, norm_topk_prob, routed_scaling_factor). */
typedef struct moe_config {
    int hidden;                  /* H: multiple of 128, 128..4096 */
    int num_experts;             /* E: 1..1024 routed experts */
    int router_width;            /* router output count; must equal E (wider
                                    "zero-computation" routers are refused, as
                                    both source pages refuse them) */
    int top_k;                   /* k: 1..min(E, 64) */
    int moe_inter;               /* I: multiple of 128 */
    int shared_inter;            /* Is: multiple of 128 (ignored if no shared) */
    int scoring;                 /* MOE_SCORING_SOFTMAX or _SIGMOID */
    int norm_topk_prob;          /* renormalise the k weights to sum 1 */
    float routed_scaling_factor; /* sigmoid scoring only; softmax requires 1 */
    int router_fmt;              /* MOE_ROUTER_BF16 or MOE_ROUTER_NVFP4 */
    int has_shared;              /* 1 = a shared expert is present */
    int shared_gate;             /* 1 = blend sigmoid(x . shared_expert_gate),
                                    0 = plain add of the shared expert */
    int per_row_mode;            /* 1 = no de-duplication: every (row, slot)
                                    pair streams its expert separately (the
                                    token-major reference order); the output
                                    is byte-identical to the union mode */
    int gemv_lever;              /* one-row sub-chunks only (a one-row call,
                                    or the one-row last sub-chunk of a
                                    longer call; see moe_forward): 0 = the
                                    expert projections on the tensor cores
                                    (NVFP4 unpacked to f16, mma.sync, fp32
                                    accumulation); 1 = on the CUDA cores as
                                    a GEMV (f16x2 products and 16-input block
                                    sums, block scales and the rest of each
                                    dot product in fp32).  The two give
                                    results within the parity tolerance of
                                    each other, not the same bytes; union and
                                    per-row mode are byte-identical within
                                    either.  The forward_ep.rs page switches
                                    its one-row GEMV kernels the same way
                                    (ctx.levers.gemv_sw).  Sub-chunks of
                                    more rows ignore it. */
    int t_layout;                /* 0: every down projection (routed and
                                    shared) in the NVFP4 layout above,
                                    [H][I/2] + [H][I/16]; 1: in the t layout
                                    ([I][H/2] + [I/16][H]).  The t layout is
                                    a decode layout: moe_forward then takes
                                    every row as a sub-chunk of its own and
                                    runs the fused one-row form (see
                                    moe_forward).  Gate and up projections
                                    keep the layout above either way; NVFP4
                                    experts only. */
    int expert_fmt;              /* MOE_EXPERT_NVFP4, _FP8 or _BF16 (every
                                    routed and shared expert matrix; the
                                    router has its own router_fmt).
                                    gemv_lever applies to NVFP4 experts
                                    only; the other formats ignore it. */
} moe_config;

/* Per-expert matrices (in the config's expert_fmt): device arrays indexed by
 * expert id (forward_token_major.rs: packed_ptrs / scale_ptrs / scale2_vals).
 * FP8 and BF16 experts leave `scales` unused (it may be NULL).  moe_nvfp4
 * likewise describes a shared-expert matrix of any expert format. */
typedef struct moe_expert_table {
    const uint8_t *const *packed;  /* device array [E] of device pointers */
    const uint8_t *const *scales;  /* device array [E] of device pointers */
    const float *scale2;           /* device array [E] */
} moe_expert_table;

typedef struct moe_weights {
    const uint16_t *router_bf16;     /* device [E][H] bf16 (router_fmt BF16) */
    moe_nvfp4 router_nvfp4;          /* [E][H] (router_fmt NVFP4) */
    const float *correction_bias;    /* device [E] fp32 (sigmoid scoring) */
    moe_expert_table gate;           /* each [I][H] */
    moe_expert_table up;             /* each [I][H] */
    moe_expert_table down;           /* each [H][I] */
    moe_nvfp4 shared_gate_proj;      /* [Is][H] */
    moe_nvfp4 shared_up_proj;        /* [Is][H] */
    moe_nvfp4 shared_down_proj;      /* [H][Is] */
    const uint16_t *shared_expert_gate; /* device [H] bf16 (shared_gate = 1) */
} moe_weights;

/* Union of the experts selected by all rows of a call (device-resident;
 * moe_union and moe_read_routing copy it out): the first occurrences of the
 * ids in row-major (row, slot) order.  Positions p = row * top_k + slot. */
typedef struct moe_union_table {
    int32_t num_union;                  /* U <= min(rows * top_k, E) */
    int32_t rows;
    int32_t top_k;
    int32_t per_row_mode;
    int32_t expert[MOE_MAX_IDS];        /* union[u]: expert id, u < U */
    uint32_t rowmask[MOE_MAX_IDS];      /* bit r: row r selected union[u] */
    uint8_t slot2u[MOE_MAX_IDS];        /* [p]: union index of position p */
    uint8_t uslot[MOE_MAX_IDS][MOE_MAX_ROWS]; /* [u][r]: slot of union[u] in
                                           row r, 0xFF if r did not pick it */
} moe_union_table;

/* Convert `count` NVFP4 matrices of N outputs x K inputs, stored back to
 * back in the layout above (packed: count x [N][K/2], scales: count x
 * [N][K/16]), into the t layout (packed_t: count x [K][N/2], scales_t: count
 * x [K/16][N]), asynchronously on `stream`.  N and K: multiples of 16, 16 ..
 * 65536; all four arrays device memory, 16-byte aligned, the outputs not
 * overlapping the inputs.  A one-off load-time step (one launch), not part
 * of the forward; scale2 is unchanged. */
MOE_API moe_status moe_nvfp4_to_t_layout(const uint8_t *packed, const uint8_t *scales,
                                         int count, int n_out, int k_in,
                                         uint8_t *packed_t, uint8_t *scales_t,
                                         void *stream);

/* ABI version of the loaded library (MOE_ABI_VERSION when built). */
MOE_API int moe_abi_version(void);

/* Text of the last refusal or error on the calling thread ("" if none). */
MOE_API const char *moe_last_error(void);

/* Host-only validation of a configuration (no CUDA call).  Returns MOE_OK or
 * the refusal; moe_route / moe_union / moe_forward run the same checks. */
MOE_API moe_status moe_check_config(const moe_config *cfg);

/* Bytes of caller-owned device workspace the calls below need for `cfg`
 * (routing scratch, union and pointer tables, intermediate activations,
 * tile counters and the status word; the scratch layout starts with the
 * top-k ids followed by the routing weights, as forward_token_major.rs lays
 * out its scratch).  Returns 0 when the configuration is refused.  The
 * workspace must be 256-byte aligned. */
MOE_API size_t moe_workspace_size(const moe_config *cfg);

/* Zero the whole workspace, its counters and status word included (async
 * on `stream`).  Call once after allocating a workspace.  The kernels keep
 * the counters consistent from then on -- a launch ticket that only grows,
 * and two grid-barrier counters that alternate between launches, each
 * zeroed by the launch before the one that uses it -- so no later call,
 * change of row count or timed-out launch needs a second initialisation. */
MOE_API moe_status moe_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Router + top-k for `rows` rows, 1..MOE_MAX_ROWS with rows * top_k <=
 * MOE_MAX_IDS (forward_token_major.rs: gate projection then
 * moe_topk_softmax_batched / moe_topk_sigmoid_batched).
 *   x       device [rows][H] bf16, 16-byte aligned
 *   ids     device [rows][top_k] int32, descending score, ties -> lower id
 *   wts     device [rows][top_k] fp32 routing weights
 *   logits  device [rows][E] fp32 router logits, or NULL */
MOE_API moe_status moe_route(const moe_config *cfg, const moe_weights *w,
                     const uint16_t *x, int rows, int32_t *ids, float *wts,
                     float *logits, void *ws, size_t ws_bytes, void *stream);

/* Union of caller-given ids [rows][top_k] (device int32, rows * top_k <=
 * MOE_MAX_IDS) by pairwise scan (forward_moe page, RETRACTED note: no
 * sort), with the device pointer table of the union experts built in the
 * workspace.  The ids are scanned in blocks of MOE_CHUNK_IDS: a position
 * opens a union entry when no earlier position, in its own block or an
 * earlier one, holds the same id, so the entries keep first-occurrence
 * order across blocks.  `out` is a device moe_union_table.  `w` supplies
 * the expert tables for the pointer table and may be NULL (no pointer
 * table).  Ids outside [0, E) are recorded as MOE_DEV_BAD_EXPERT_ID and
 * skipped. */
MOE_API moe_status moe_union(const moe_config *cfg, const moe_weights *w,
                     const int32_t *ids, int rows, moe_union_table *out,
                     void *ws, size_t ws_bytes, void *stream);

/* The whole routed MoE layer (page "Function forward_moe": forward_moe(x,
 * out, rows)) for rows = 1..MOE_MAX_ROWS with rows * top_k <= MOE_MAX_IDS:
 *   out[r] = sum_{slot < k} wts[r][slot] * Expert_{ids[r][slot]}(x[r])
 *            + g_r * Shared(x[r]),
 *   Expert(x) = Wd (silu(Wg x) * (Wu x)), g_r = sigmoid(x[r] . gs) with
 *   shared_gate = 1, 1 with shared_gate = 0, 0 without a shared expert.
 *   x    device [rows][H] bf16, 16-byte aligned
 *   out  device [rows][H] bf16, 16-byte aligned, must not overlap x
 * `out` is the MoE output only (the residual add is the caller's).  Nothing
 * is read back to the host, so the call can be captured in a CUDA graph.
 * Rows are taken in consecutive sub-chunks of min(MOE_CHUNK_ROWS,
 * MOE_CHUNK_IDS / top_k) rows, one kernel launch each, as the page batches
 * prefill in 8-row sub-chunks: a sub-chunk's union (at most MOE_CHUNK_IDS
 * ids, one block) is swept once for all its rows, and every row's output
 * bytes are those a call with that sub-chunk alone would give.  A call of
 * more than one sub-chunk then resolves the union of all its rows (as
 * moe_union does) for moe_read_routing.
 *
 * With t_layout = 1 every row is a sub-chunk of its own and runs in a fused
 * form: each 16-row gate/up tile's h goes straight into the 16 rows of the
 * transposed down projection that it multiplies, every SM keeps a partial
 * sum of every output, and after one grid barrier the partials are added in
 * a fixed order (the down sweep, the blend and their two grid barriers do
 * not exist in this form).  Its results agree with t_layout = 0 within the
 * parity tolerance, not byte for byte; union and per-row mode give the same
 * bytes. */
MOE_API moe_status moe_forward(const moe_config *cfg, const moe_weights *w,
                       const uint16_t *x, uint16_t *out, int rows, void *ws,
                       size_t ws_bytes, void *stream);

/* moe_forward with CUDA events recorded just before and just after the
 * layer's kernel launch (ev[0], ev[1]: cudaEvent_t passed as void*), for
 * timing the kernel alone.  The event records sit between launches, so the
 * kernel does not overlap its prologue with the previous launch as it does
 * in moe_forward; the result bytes are the same.  Diagnostics. */
MOE_API moe_status moe_forward_timed(const moe_config *cfg, const moe_weights *w,
                                     const uint16_t *x, uint16_t *out, int rows,
                                     void *ws, size_t ws_bytes, void *stream,
                                     void *const ev[2]);

/* Bytes of the library-owned device workspace behind moe_forward_static;
 * it covers every configuration moe_check_config accepts (at most about
 * 9.3 MB, with the t layout at hidden 4096, 1024 experts, intermediate
 * 4096). */
#define MOE_STATIC_WORKSPACE_BYTES (10u << 20)

/* moe_forward for callers that cannot allocate device memory themselves --
 * for example a plug-in running inside a host framework that owns every
 * device allocation through its own pool and forbids side allocations, or a
 * latency-critical path that must never enter the CUDA allocator.  The
 * source pages have no counterpart to this entry point.
 *
 * Same arguments and result as moe_forward, minus the workspace: the scratch
 * lives in one file-scope device array of MOE_STATIC_WORKSPACE_BYTES, which
 * every GPU that loads the library holds until the process exits.  The call
 * allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine).  The first call on each device looks up the array's device
 * address; make that first call before any stream capture.  Every call
 * clears the array's counters and status word on `stream`, then runs the
 * layer.  All calls share the one array, so calls that overlap on the GPU
 * (different streams, or host threads without ordering) race and must be
 * serialised by the caller.  Device fault codes recorded by this path are
 * cleared by the next call and are not reported.  A configuration whose
 * workspace would exceed the array is refused with MOE_ERR_WORKSPACE. */
MOE_API moe_status moe_forward_static(const moe_config *cfg, const moe_weights *w,
                                      const uint16_t *x, uint16_t *out, int rows,
                                      void *stream);

/* Copy the routing of the last moe_forward / moe_route on this workspace
 * into caller buffers (async device-to-device copies on `stream`; any
 * pointer may be NULL): ids / wts device [rows][top_k], uni a device
 * moe_union_table of all the call's rows (valid after moe_forward or
 * moe_union). */
MOE_API moe_status moe_read_routing(const moe_config *cfg, const void *ws,
                            size_t ws_bytes, int rows, int32_t *ids,
                            float *wts, moe_union_table *uni, void *stream);

/* Synchronise `stream`, read the workspace's device status word into *code
 * (MOE_DEV_*), and clear it (only the status word and its detail: the
 * counters need no reset, even after MOE_DEV_WAIT_TIMEOUT).  Returns
 * MOE_ERR_DEVICE_STATUS when the code is non-zero.  Test and diagnostics
 * use only: it blocks the host. */
MOE_API moe_status moe_read_device_status(void *ws, size_t ws_bytes, int *code,
                                  void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTER_H */
