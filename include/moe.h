/*
 * moe.h - C ABI of the GB300 (sm_103a) routed Mixture-of-Experts FFN forward.
 *
 * The library computes, on one GPU, the routed MoE FFN forward pass whose
 * expert-grouped pipeline the Motivation of "perf: add small-batch route MMA
 * for MoE" describes: top-k routing; grouping the routes by expert (counts and
 * a stable order); gathering the rows; prefix sums and a GEMM task map; the
 * Gate/Up grouped GEMM; SwiGLU with optional FP8 re-quantisation; the Down
 * grouped GEMM; and the weighted reduction of each token's k expert outputs
 * (the index_shuffling and scatter_add_dense_tokens steps of "Port necessary
 * FBGEMM MoE kernels").  It also has the route-direct small-batch path of the
 * route-MMA page's Summary: each route reads its expert directly, with no
 * sort, gather, prefix sum or task map; the long Gate/Up K dimension is split
 * for parallelism; and the split reduction, SwiGLU and the quantisation of the
 * Down input are done in one pass.
 *
 * Definitions used throughout:
 *   T tokens, E experts, k = top_k, H hidden size, I expert intermediate size,
 *   R = T*k routes; route r = t*k + j is slot j of token t.
 *   Routing: ids[t, 0..k-1] = the k experts with the largest router score,
 *   ordered by score descending, ties to the lower expert id (-0.0 == +0.0);
 *   w[t, j] = softmax over the k selected scores.
 *   Gate/Up weights W1 [E, 2I, H]: rows 0..I-1 of W1[e] are the gate
 *   projection, rows I..2I-1 the up projection.  Down weights W2 [E, H, I].
 *   y[t] = sum_j w[t, j] * W2[ids[t, j]] (silu(gate) * up), rounded to bf16.
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers to row-major, contiguous
 *     arrays, unless stated otherwise.  Bases of bf16 / e4m3 arrays and of
 *     the workspace must be 16-byte aligned (a TMA requirement); int32 and
 *     fp32 arrays 4-byte aligned.
 *   - The caller owns and allocates every buffer, including outputs and the
 *     workspace.  The library never allocates, frees or synchronises inside
 *     moe_route / moe_shuffle / moe_tile_map / moe_forward / moe_forward_ex /
 *     moe_round_bf16: work is enqueued
 *     on `stream` in order, with no device-to-host copy, so these calls can be
 *     captured in a CUDA graph.  Inputs are never written.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Arguments are validated on the host BEFORE anything is enqueued; on a
 *     validation error nothing is launched and outputs are untouched.
 *   - A launch failure returns MOE_ERR_CUDA.  Conditions detected on the device
 *     (a bounded wait that timed out, an index out of range) are recorded in
 *     a status word at the head of the workspace and reported by
 *     moe_read_device_status(); the library never traps.
 *   - Results are deterministic: the same inputs give bitwise identical
 *     outputs, eager or replayed from a CUDA graph.
 */
#ifndef MOE_GB300_MOE_H_
#define MOE_GB300_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so that the header needs no CUDA headers. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* bad shape, null or misaligned pointer, inconsistent scales */
  MOE_ERR_UNSUPPORTED = 2,    /* valid, but outside what this library implements (limits below) */
  MOE_ERR_WORKSPACE = 3,      /* workspace missing or smaller than the *_workspace_size() value */
  MOE_ERR_CUDA = 4,           /* a CUDA runtime/driver call or a launch failed, or no usable GPU */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait expired (reported by moe_read_device_status) */
  MOE_ERR_DEVICE_BOUNDS = 6   /* a kernel saw an out-of-range index (reported by moe_read_device_status) */
} moe_status;

typedef enum {
  MOE_BF16 = 0,           /* bf16 x, W1, W2; bf16 h; fp32 accumulation */
  MOE_FP8_PER_TENSOR = 1, /* e4m3 W1/W2 with one fp32 scale per expert matrix; x and h quantised to
                             e4m3 with one dynamic scale each (amax/448 over the whole tensor) */
  MOE_FP8_BLOCK128 = 2,   /* e4m3 W1/W2 with fp32 scales per 128x128 block; x quantised per
                             (token, 128 columns); h per (route, 128 columns) */
  MOE_MXFP8 = 3           /* MXFP8: e4m3 W1/W2 with one E8M0 (power-of-two) scale per 32
                             consecutive values of a row along K; x and h quantised the same
                             way (grouped path only; see moe_forward) */
} moe_quant;

typedef enum {
  MOE_PATH_AUTO = 0,        /* library chooses (see moe_select_path) */
  MOE_PATH_GROUPED = 1,     /* group routes by expert, tile map, grouped GEMMs, combine */
  MOE_PATH_ROUTE_DIRECT = 2 /* route-order decode path, no sort / gather / tile map */
} moe_path;

typedef struct {
  int T, E, k, H, I;
  moe_quant quant;
  moe_path path;
} moe_problem;

/* Limits of this library (MOE_ERR_UNSUPPORTED beyond them):
 *   1 <= E <= 512;  1 <= k <= min(E, 32);  0 <= T;  T*k < 2^31;
 *   H % 64 == 0, I % 64 == 0 (bf16, FP8 per-tensor);  H % 128 == 0, I % 64 == 0 (FP8
 *   blockwise, whose last 128-column scale group of I may hold 64 columns, and MXFP8);
 *   MOE_PATH_GROUPED: all four modes;  MOE_PATH_ROUTE_DIRECT: per-tensor and blockwise
 *   FP8, T*k <= 1024. */

/* ---------------------------------------------------------------- routing
 * moe_route - top-k routing (the routing step of "perf: add small-batch route
 * MMA for MoE", Motivation).
 *   scores [T, E] fp32 (finite; NaN/inf are outside the contract)
 *   ids    [T, k] int32 out: selected experts in slot order (score desc, id asc)
 *   w      [T, k] fp32  out: softmax over the k selected scores
 * ids are exact; w is computed in fp32 (expf, IEEE division).
 * T == 0 is a no-op.  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
moe_status moe_route(const float* scores, int T, int E, int k, int32_t* ids, float* w,
                     moe_stream_t stream);

/* ---------------------------------------------------------------- shuffle
 * moe_shuffle - index shuffling (index_shuffling of "Port necessary FBGEMM
 * MoE kernels"; the counting and sorting step of the route-MMA page's
 * Motivation).
 *   ids     [T, k] int32 in: expert of each route, each in [0, E)
 *   counts  [E]    int32 out: routes per expert
 *   offsets [E+1]  int32 out: exclusive prefix sum of counts (offsets[E] = R)
 *   perm    [R]    int32 out: sorted position -> route r; stable (routes of one
 *                             expert keep increasing r, i.e. token order)
 *   inv     [R]    int32 out: route -> sorted position (inv[perm[p]] == p)
 *   ws      device scratch of at least moe_shuffle_workspace_size(T, E, k) bytes
 * All outputs are unique and therefore bit-exact.  An id outside [0, E) is
 * recorded as MOE_ERR_DEVICE_BOUNDS in the status word at the head of ws and
 * that route is left out of the outputs.  Errors: INVALID_ARG, UNSUPPORTED,
 * WORKSPACE, CUDA. */
size_t moe_shuffle_workspace_size(int T, int E, int k);
moe_status moe_shuffle(const int32_t* ids, int T, int E, int k, int32_t* counts, int32_t* offsets,
                       int32_t* perm, int32_t* inv, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- shuffle, no allocation
 * moe_shuffle_noalloc - moe_shuffle without a caller-provided workspace.  The
 * pages have no counterpart to this entry point: it exists for callers that
 * cannot allocate device memory when they need the shuffle - code running while
 * a stream is captured into a CUDA graph (cudaMalloc is not allowed there),
 * plugins of a host framework that owns all device memory and provides no
 * scratch, and serving loops that forbid allocation after start-up.
 *   Arguments and outputs: as moe_shuffle (caller-owned device arrays).
 *   Scratch: a fixed array of MOE_NOALLOC_SCRATCH_BYTES inside the library;
 *   every GPU that loads the library holds it until the process exits.  Neither
 *   this call nor the library allocates or frees anything.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  The looked-up address is cached for the life
 *   of the process: destroying the device's context after the first call
 *   (cudaDeviceReset) and calling again is not supported.
 *   Every call uses the same array: calls whose work overlaps on the GPU (e.g.
 *   on two streams) race and must be serialised by the caller.
 *   Errors: as moe_shuffle; MOE_ERR_WORKSPACE when the problem needs more than
 *   the fixed array (moe_shuffle_workspace_size(T, E, k) >
 *   MOE_NOALLOC_SCRATCH_BYTES; e.g. up to 131072 routes with E = 128 fit).
 *   An out-of-range id is skipped as in moe_shuffle; its status word is the
 *   array's and is not exposed. */
#define MOE_NOALLOC_SCRATCH_BYTES (1u << 20)
moe_status moe_shuffle_noalloc(const int32_t* ids, int T, int E, int k, int32_t* counts, int32_t* offsets,
                               int32_t* perm, int32_t* inv, moe_stream_t stream);

/* ---------------------------------------------------------------- tile map
 * moe_tile_map - the grouped GEMMs' task map (the task-map step of the
 * route-MMA page's Motivation, sized by the experts that actually have routes,
 * as its Code changes do), built on the device with no device-to-host copy.
 *   counts    [E] int32 in (e.g. from moe_shuffle)
 *   BM        row-tile height (1..1024; moe_forward uses 128)
 *   tiles     [max_tiles, 4] int32 out: {expert, first sorted row, rows, 0} for
 *             each tile, experts in id order, ceil(counts[e]/BM) tiles each
 *   num_tiles [1] int32 out: number of tiles written
 *   max_tiles capacity of `tiles`; floor(sum(counts)/BM) + E always suffices.
 * If the tiles do not fit, num_tiles holds the required count, only
 * max_tiles tiles are written and MOE_ERR_DEVICE_BOUNDS is recorded in the
 * status word at the head of ws.  ws needs moe_shuffle_workspace_size(0, E, 1)
 * bytes.  Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
moe_status moe_tile_map(const int32_t* counts, int E, int BM, int32_t* tiles, int32_t* num_tiles,
                        int max_tiles, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- forward
 * moe_select_path - the path moe_forward takes for *p (AUTO resolved):
 * bf16 and MXFP8 -> GROUPED; per-tensor FP8 -> ROUTE_DIRECT for T <= 96,
 * blockwise FP8 -> ROUTE_DIRECT for T <= 64 (both also need T*k <= 1024), else
 * GROUPED: the crossovers measured on GB300.  Returns p->path when it is not
 * AUTO. */
moe_path moe_select_path(const moe_problem* p);

/* moe_workspace_size - bytes of device workspace moe_forward needs for *p
 * (0 if *p is invalid or unsupported). */
size_t moe_workspace_size(const moe_problem* p);

/* moe_forward - the whole routed MoE FFN forward.
 *   x        [T, H]  bf16 activations
 *   scores   [T, E]  fp32 router scores
 *   w1       [E, 2I, H] bf16 (MOE_BF16) or e4m3 codes (FP8 modes); rows 0..I-1 gate, I..2I-1 up
 *   w2       [E, H, I]  bf16 or e4m3
 *   w1_scale NULL (bf16) | fp32 [E] (per-tensor) | fp32 [E, 2I/128, H/128] (blockwise; a block
 *            row of W1 may hold the last gate rows and the first up rows when I % 128 == 64)
 *            | uint8 E8M0 codes [E, 2I, H/32] (MXFP8, passed through this pointer)
 *   w2_scale NULL (bf16) | fp32 [E] (per-tensor) | fp32 [E, H/128, ceil(I/128)] (blockwise)
 *            | uint8 E8M0 codes [E, H, I/32] (MXFP8)
 *   y        [T, H]  bf16 out, preallocated by the caller (written, never read)
 *   ws       device workspace of at least moe_workspace_size(p) bytes; its
 *            contents on entry do not matter and are overwritten
 * Quantisation (FP8 modes): scale = amax/448 in fp32 (1 when amax == 0),
 * code = e4m3(v / scale) rounded to nearest even with saturation.  MXFP8 (the
 * OCP Microscaling format named by "[mxfp8 moe training] add per group blocked
 * scale kernels"): each run of 32 values along the contraction dimension
 * shares the scale 2^X, X = floor(log2(amax)) - 8 clamped to [-127, 127] (-127
 * for a zero run), stored as the E8M0 code X + 127; code = e4m3(v / 2^X), RNE,
 * saturating.  The MXFP8 forward converts x's, h's and the weights' scales
 * into the blocked layout of moe_mx_blocked_scales (groups = the experts'
 * row segments) on every call and multiplies with the tensor cores'
 * block-scaled MMA; h is quantised in the Gate/Up epilogue.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
moe_status moe_forward(const moe_problem* p, const void* x, const float* scores, const void* w1,
                       const void* w2, const float* w1_scale, const float* w2_scale, void* y,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- forward, extended
 * moe_forward_ex - moe_forward with the optional parts below (opt NULL or all
 * zero = moe_forward).
 *
 * Shared experts (the "shared output" that the Summary of "perf: add small-batch
 * route MMA for MoE" lists; the page does not define it, and this library takes
 * the common reading): n_shared = S experts, each with the routed experts'
 * shapes and formats, that every token passes through with weight 1:
 *   y[t] = sum_j w[t, j] * o_(t, j)  +  sum_s FFN_shared[s](x_t),
 * summed j ascending then s ascending, rounded once.  Their rows are more rows
 * of the same intermediate tensor: x is quantised once for both, and in
 * per-tensor FP8 the dynamic scale of h spans the routed and the shared rows.
 *   w1_shared        [S, 2I, H] bf16 | e4m3 (rows 0..I-1 gate, I..2I-1 up)
 *   w2_shared        [S, H, I]
 *   w1_shared_scale  NULL (bf16) | fp32 [S] | fp32 [S, 2I/128, H/128]
 *   w2_shared_scale  NULL (bf16) | fp32 [S] | fp32 [S, H/128, ceil(I/128)]
 * Shared experts run on the grouped path (AUTO takes it; an explicit
 * MOE_PATH_ROUTE_DIRECT with S > 0 is UNSUPPORTED).  0 <= S <= 16.
 *
 * Unrounded output (y_fp32 = 1): y is fp32 [T, H], the sum above before its
 * rounding.  This is the partial output of one slice of a tensor-parallel
 * split of I (the TP8 deployment in the route-MMA page's Performance section):
 * each slice holds gate rows and up rows [p*I/P, (p+1)*I/P) of every W1[e] (and
 * the same columns of W2[e], and for blockwise FP8 the matching scale blocks, so
 * I/P must be a multiple of 128) and runs moe_forward_ex with I/P as its I; the
 * caller sums the slices' partial outputs (e.g. an all-reduce) and rounds the sum
 * with moe_round_bf16.  In bf16 and blockwise FP8 that equals the unsplit
 * forward up to fp32 summation order; per-tensor FP8 then scales h per slice.
 *
 * moe_workspace_size_ex gives the workspace for (*p, *opt); moe_forward_views_ex
 * the views of that workspace.  Errors: as moe_forward. */
typedef struct {
  int n_shared;
  const void* w1_shared;
  const void* w2_shared;
  const float* w1_shared_scale;
  const float* w2_shared_scale;
  int y_fp32;
  int mx_weight_scales_blocked; /* MXFP8: 1 = the weight scale pointers (routed and shared) hold
                                   the blocked layouts of moe_mx_weight_scales instead of the
                                   row-major E8M0 codes (no per-call conversion) */
} moe_forward_options;
size_t moe_workspace_size_ex(const moe_problem* p, const moe_forward_options* opt);
moe_status moe_forward_ex(const moe_problem* p, const moe_forward_options* opt, const void* x, const float* scores,
                          const void* w1, const void* w2, const float* w1_scale, const float* w2_scale, void* y,
                          void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_mx_weight_scales - the MXFP8 weights' scales in the blocked layout the
 * forward's block-scaled MMAs read, converted once (e.g. when the weights are
 * loaded) instead of on every call (moe_forward_options.mx_weight_scales_blocked).
 *   w1_scale [E, 2I, H/32], w2_scale [E, H, I/32] uint8 E8M0 codes (4-byte aligned)
 *   w1_blocked, w2_blocked  outputs of moe_mx_weight_scales_bytes(E, H, I, 1 / 2)
 *                           bytes (16-byte aligned): W1 as the B operands of the
 *                           Gate/Up units (96 gate rows and the matching 96 up rows
 *                           of one expert, two 128-row blocks per unit, adjacent
 *                           per column block), W2 likewise as the B operands of the
 *                           Down units (192 rows, two blocks each); blocks are the
 *                           512-byte blocks of moe_mx_blocked_scales.
 * Errors: INVALID_ARG, UNSUPPORTED (the MXFP8 shape limits), CUDA. */
size_t moe_mx_weight_scales_bytes(int E, int H, int I, int which);
moe_status moe_mx_weight_scales(const uint8_t* w1_scale, const uint8_t* w2_scale, int E, int H, int I,
                                uint8_t* w1_blocked, uint8_t* w2_blocked, moe_stream_t stream);

/* moe_round_bf16 - y[i] = bf16(y32[i]) for i < n (round to nearest even): the
 * single rounding of a sum of partial outputs (moe_forward_ex, y_fp32 = 1).
 * y32 fp32 [n], y bf16 [n], both 16-byte aligned, n a multiple of 8.
 * Errors: INVALID_ARG, CUDA. */
moe_status moe_round_bf16(const float* y32, void* y, size_t n, moe_stream_t stream);

/* ---------------------------------------------------------------- MX scale layout
 * moe_mx_blocked_scales - the per-group blocked scale conversion of "[mxfp8 moe
 * training] add per group blocked scale kernels" (Summary): MX scales of row
 * groups (e.g. the expert groups of a grouped GEMM's activations) converted
 * into the blocked, swizzled layout that block-scaled tensor-core MMAs read,
 * each group on its own and padded to whole 128-row blocks, with every group's
 * start row in the padded output computed on the device (no device-to-host
 * copy).
 *   scales        [rows, cols] uint8 (one byte per scale, row-major; base 4-byte aligned)
 *   group_offsets [groups + 1] int32: group g = rows [off[g], off[g+1]),
 *                 nondecreasing, off[groups] <= rows
 *   out           blocked output, at least moe_mx_blocked_bytes(rows, cols,
 *                 groups) bytes; group g's padded rows start at row
 *                 group_starts[g] of an [*, ceil(cols/4)*4] byte matrix
 *   group_starts  [groups + 1] int32 out: padded start rows; entry groups = total
 *   ws            scratch of moe_mx_blocked_workspace_size(rows, groups) bytes
 * Layout: each group's scales are zero-padded to a multiple of 128 rows and of
 * 4 columns and cut into 128 x 4 blocks, stored block row by block row; inside
 * a 512-byte block the scale of (row r, column c) is at byte (r % 32) * 16 +
 * (r / 32) * 4 + c.  Output bytes past group_starts[groups] rows are not
 * written.  A negative group size is recorded as MOE_ERR_DEVICE_BOUNDS (status
 * word at the head of ws) and treated as empty.  1 <= groups <= 4096.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
size_t moe_mx_blocked_bytes(int rows, int cols, int groups);
size_t moe_mx_blocked_workspace_size(int rows, int groups);
moe_status moe_mx_blocked_scales(const uint8_t* scales, int rows, int cols, const int32_t* group_offsets,
                                 int groups, uint8_t* out, size_t out_bytes, int32_t* group_starts, void* ws,
                                 size_t ws_bytes, moe_stream_t stream);

/* moe_forward_views - device pointers to the intermediate results moe_forward
 * leaves in the workspace (read-only diagnostics; valid after the call's
 * work on the stream completed).  Pointers not produced by the path chosen
 * for *p are set to NULL.  ids/w: [T, k]; counts [E]; offsets [E+1];
 * perm/inv [R]; tiles [*, 4] and num_tiles [1] as for moe_tile_map (BM 128).
 * The activations as the Gate/Up GEMM reads them (the quantisation of x is
 * unique, so these can be checked bit for bit):
 *   xs       grouped path: [R, H] rows in expert-sorted order, row p = x row
 *            of token perm[p] / k (bf16 copies, or e4m3 codes in the FP8
 *            modes); route-direct path: [T, H] e4m3 codes in token order.
 *            NULL for the bf16 variant that gathers x inside the GEMM.
 *   x_scale  blockwise FP8: fp32 scales of xs, one per row and 128 columns
 *            ([R, H/128] sorted, or [T, H/128] route-direct); MXFP8: uint8
 *            E8M0 codes, one per row and 32 columns ([R, H/32] sorted); else
 *            NULL.
 *   amax_x   per-tensor FP8: the fp32 amax of x over the whole [T, H]
 *            (scale = amax / 448, 1 when it is 0); else NULL. */
typedef struct {
  const int32_t* ids;
  const float* w;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* inv;
  const int32_t* tiles;
  const int32_t* num_tiles;
  const void* xs;
  const float* x_scale;
  const float* amax_x;
} moe_views;
moe_status moe_forward_views(const moe_problem* p, const void* ws, size_t ws_bytes, moe_views* out);
/* The same for a workspace of moe_forward_ex(p, opt, ...); with shared experts
 * xs (and x_scale) hold T*k + S*T rows, shared expert s's row of token t at
 * T*k + s*T + t. */
moe_status moe_forward_views_ex(const moe_problem* p, const moe_forward_options* opt, const void* ws,
                                size_t ws_bytes, moe_views* out);

/* ---------------------------------------------------------------- diagnostics
 * moe_read_device_status - synchronises `stream`, then returns the status
 * recorded on the device in the status word at the head of `ws` (MOE_OK,
 * MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_DEVICE_BOUNDS), or MOE_ERR_CUDA if the
 * synchronisation failed.  Diagnostic only: it blocks, so it is never part of
 * the hot path.  Each moe_forward / moe_shuffle / moe_tile_map call resets the
 * word at its start. */
moe_status moe_read_device_status(const void* ws, moe_stream_t stream);

/* ---------------------------------------------------------------- stage timing
 * While profiling is on, each kernel launch of the entry points above is
 * bracketed by a pair of CUDA events recorded on the caller's stream (host-side
 * records only: nothing is synchronised or allocated on the device, and
 * launches on a stream that is being captured into a graph are not timed).
 *
 * moe_profile_start - clears earlier records and turns profiling on.
 * moe_profile_stop  - waits for the recorded events, writes one entry per
 *   kernel stage (in order of first launch) to out[0 .. max_stages-1], turns
 *   profiling off and returns the number of stages, or -1 if waiting on an
 *   event failed.  total_ms sums the stage's launches; launches counts them.
 * moe_profile_start_stage - the same, but only launches of the stage named
 *   `stage` are timed (NULL or "" times every stage).  Each event pair recorded
 *   between two kernels costs GPU time (about 2 us per stage on GB300), so a
 *   measurement of the whole call brackets only the kernel it needs.
 * Stage names: route_rank (with the per-tensor FP8 amax of x), scan_tiles,
 * scatter_gather, gateup_gemm, quant_h, down_gemm, combine (grouped path);
 * rd_prep, rd_gateup, rd_reduce, rd_down, combine (route-direct path); scatter,
 * tile_map, header_reset. */
typedef struct {
  char name[32];
  double total_ms;
  int launches;
} moe_stage_time;
int moe_profile_start(void);
int moe_profile_start_stage(const char* stage);
int moe_profile_stop(moe_stage_time* out, int max_stages);

/* moe_status_string - static, NUL-terminated description of a status code. */
const char* moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_MOE_H_ */
