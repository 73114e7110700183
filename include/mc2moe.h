/*
 * mc2moe.h -- C ABI of the GB300 (sm_103a) MoE expert block.
 *
 * The block is the expert-parallel forward of "NPU Training Operators - MC2"
 * (shaojiemike.top), section "Execution path": histc per-expert token counts,
 * the all_gather of those counts, send_counts / recv_counts, permute, the
 * fc1 grouped matmul, SwiGLU, the fc2 grouped matmul and the routing-weighted
 * unpermute.  Here the W expert-parallel ranks are logical: rank r owns tokens
 * [r*T/W, (r+1)*T/W) and experts [r*E/W, (r+1)*E/W) of one GPU, so the two
 * AllToAllv exchanges become a row gather folded into the fc1 operand load
 * and an ordered per-token sum of the fc2 rows (a separate pass by default,
 * inside the fc2 kernel when selected).  The int8 variant uses the
 * dequantisation of "torch_npu.npu_mm_reduce_scatter_base" (Ascend op-plugin
 * docs), section "Function description": (x1_scale * x2_scale) * (x1 @ x2),
 * with no bias.
 *
 * Conventions for every entry point
 *  - Pointers marked [dev] are CUDA device pointers; the caller owns every
 *    buffer, including the workspace `ws` and the device status word.  The
 *    library never allocates, frees or synchronises; all work is enqueued on
 *    `stream`, in order.  Inputs are read-only; outputs are fully written.
 *  - Tensors are dense row-major with the shapes given; element types follow
 *    mc2_shape_t.act (activations and weights) and mc2_shape_t.out.
 *  - Every array pointer is 16-byte aligned and the workspace 256-byte
 *    aligned (the kernels use 16-byte vector and TMA accesses); a misaligned
 *    pointer returns MC2_ERR_INVALID_ARG.
 *  - A synchronous return other than MC2_OK means nothing was enqueued.
 *  - Conditions found on the device (an expert id outside [0, E); a bounded
 *    device-side wait that expired) are OR-ed into *dev_status as
 *    MC2_DEV_* bits; read it after synchronising `stream`.  dev_status may be
 *    NULL, in which case those conditions are not reported.
 *  - Ids outside [0, E) are never used as addresses: they are left out of
 *    every count, sorted after every valid pair in the permutation, skipped
 *    by both matmuls and contribute zero to the combine.
 */
#ifndef MC2MOE_H
#define MC2MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MC2_OK = 0,
  MC2_ERR_INVALID_ARG = 1,    /* shape rule or pointer rule broken; nothing launched */
  MC2_ERR_UNSUPPORTED = 2,    /* valid request the library does not implement */
  MC2_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed */
  MC2_ERR_DEVICE_TIMEOUT = 4, /* never returned synchronously: the device reports MC2_DEV_TIMEOUT;
                                 the code exists so callers can map that bit to a status */
  MC2_ERR_BAD_EXPERT_ID = 5   /* likewise, for the MC2_DEV_BAD_EXPERT_ID bit */
} mc2_status_t;

/* bits of the device status word */
#define MC2_DEV_BAD_EXPERT_ID 0x1
#define MC2_DEV_TIMEOUT 0x2
#define MC2_DEV_INTERNAL 0x4  /* the two CTAs of a pair were given different TMEM; work skipped */

typedef enum {
  MC2_F32 = 0,   /* fp32 values; matmuls on tensor cores in tf32 (inputs rounded to nearest) */
  MC2_BF16 = 1,  /* bf16 values, fp32 accumulation */
  MC2_I8 = 2,    /* int8 values with fp32 per-token / per-channel scales, exact int32 accumulation */
  MC2_I32 = 3    /* out only, with act = MC2_I8: raw int32 accumulators (test mode) */
} mc2_dtype_t;

typedef struct {
  int32_t T;    /* tokens (rows of hidden_states after view(-1, H)) */
  int32_t H;    /* hidden size; multiple of 64 */
  int32_t I;    /* per-expert intermediate size; fc1 emits 2I (gate | up); multiple of 64 */
  int32_t E;    /* experts, 1..1024; E % W == 0 */
  int32_t k;    /* top-k, 1..E */
  int32_t W;    /* logical expert-parallel ranks; T % W == 0 and E % W == 0 */
  int32_t act;  /* mc2_dtype_t of x, w1, w2 (and of h for F32/BF16) */
  int32_t out;  /* mc2_dtype_t of the block output: F32 (act F32), BF16 (act BF16 or I8),
                   or I32 (act I8, accumulator test mode) */
} mc2_shape_t;

/* Check a shape against the rules above.  Host only, pure. */
mc2_status_t mc2_check_shape(const mc2_shape_t* s);

/* Bytes of device workspace the block needs for this shape (0 for an invalid
 * shape).  Host only, pure and deterministic; the same workspace serves all
 * entry points below.  Alignment: 256 bytes. */
size_t mc2_workspace_bytes(const mc2_shape_t* s);

/*
 * mc2_moe_counts -- steps 2-6 of the execution path: per-rank histc, the
 * logical all_gather, send/recv counts and the permutation indices.
 *   sel            [dev] int32 [T, k]  selected_experts (flat index i = t*k + j)
 *   cnt            [dev] int32 [W, E]  out: num_global_tokens_per_expert; row r is
 *                                      rank r's histc(bins=E, min=0, max=E) of its
 *                                      own tokens, i.e. its send_counts
 *   recv           [dev] int32 [W, W*E/W] out: recv_counts of rank r =
 *                                      cnt[:, r*E_l:(r+1)*E_l].reshape(-1)
 *                                      (source-rank-major), E_l = E/W
 *   offsets        [dev] int32 [E + 1] out: first permuted row of each expert;
 *                                      offsets[E] = number of valid pairs
 *   permute_src    [dev] int32 [T*k]   out: flat index of the pair in permuted row p;
 *                                      rows ordered by (expert, t, j) -- a stable
 *                                      sort by expert; invalid ids last
 *   unpermute_dst  [dev] int32 [T*k]   out: inverse of permute_src
 *   ws             [dev] workspace of mc2_workspace_bytes(s)
 */
mc2_status_t mc2_moe_counts(const mc2_shape_t* s, const int32_t* sel, int32_t* cnt,
                            int32_t* recv, int32_t* offsets, int32_t* permute_src,
                            int32_t* unpermute_dst, void* ws, int32_t* dev_status,
                            void* stream);

/*
 * mc2_alltoallv_gmm -- dispatch segment, steps 6-8: the permute (a gather of
 * token rows by permute_src), the fc1 grouped matmul and SwiGLU, named after
 * npu_alltoallv_gmm of the same page, section "Low-level API comparison".
 *   x         [dev] [T, H] act                 hidden_states
 *   x_scale   [dev] fp32 [T]                   per-token scale (act I8 only, else NULL)
 *   w1        [dev] [E, H, 2I] act             fc1_weight = gate_up_proj; columns
 *                                              [0, I) gate, [I, 2I) up; y = x @ w1[e]
 *   w1_scale  [dev] fp32 [E, 2I]               per-channel scale (act I8 only, else NULL)
 *   offsets, permute_src                       from mc2_moe_counts
 *   h         [dev] out, permuted (expert-major) rows:
 *                act BF16/F32: [T*k, I] act, h = silu(gate) * up
 *                act I8, out BF16: [T*k, I] int8, h re-quantised per row
 *                act I8, out I32: [T*k, 2I] int32, the raw fc1 accumulators
 *             rows p >= offsets[E] are not written.
 *   h_scale   [dev] fp32 [T*k] out (act I8 and out BF16 only, else NULL):
 *             per-row scale of the int8 h (max|h| / 127, 1 for an all-zero row)
 * With T = 0 nothing is launched and x, w1, the scales, permute_src and h may
 * be NULL (as in mc2_gmm_alltoallv).
 */
mc2_status_t mc2_alltoallv_gmm(const mc2_shape_t* s, const void* x, const float* x_scale,
                               const void* w1, const float* w1_scale, const int32_t* offsets,
                               const int32_t* permute_src, void* ws, void* h, float* h_scale,
                               int32_t* dev_status, void* stream);

/*
 * mc2_gmm_alltoallv -- combine segment, steps 9-10: the fc2 grouped matmul
 * and the unpermute with probs, named after npu_gmm_alltoallv.
 *   h, h_scale         [dev] as produced by mc2_alltoallv_gmm (h_scale: act I8 only)
 *   w2        [dev] [E, I, H] act              fc2_weight = down_proj
 *   w2_scale  [dev] fp32 [E, H]                per-channel scale (act I8 only, else NULL)
 *   offsets, permute_src, unpermute_dst        from mc2_moe_counts
 *   probs     [dev] fp32 [T, k]                routing_weights
 *   out       [dev] out dtype:
 *                F32/BF16: [T, H], out[t] = sum_j probs[t, j] * y(t, j), summed in
 *                          fp32 in ascending j, one rounding at the end; the sum is
 *                          bit-identical from run to run
 *                I32 (act I8): [T*k, H] int32 raw fc2 accumulators, permuted rows;
 *                          h is then the int8 h of an out=BF16 fc1 call
 */
mc2_status_t mc2_gmm_alltoallv(const mc2_shape_t* s, const void* h, const float* h_scale,
                               const void* w2, const float* w2_scale, const int32_t* offsets,
                               const int32_t* permute_src, const int32_t* unpermute_dst,
                               const float* probs, void* ws, void* out, int32_t* dev_status,
                               void* stream);

/*
 * mc2_moe_counts_static -- mc2_moe_counts for callers that cannot allocate
 * device memory: same arguments and results, minus the workspace.  The paper
 * has no counterpart; it exists because some callers cannot call cudaMalloc
 * (a plugin inside a host application that owns all device memory through its
 * own pool, a service whose device-memory budget is fixed at start-up).
 *   - Scratch is a fixed array inside this library's device image (1 MiB on
 *     every GPU that loads the library, held until the process exits).  The
 *     shape must satisfy (E + 1) * W * ceil(T*k / W / 256) <= 131072, else the
 *     call returns MC2_ERR_UNSUPPORTED and launches nothing.
 *   - The first call on a device looks up that array's device address (with
 *     that device current) and caches it, keyed on the device's current
 *     context (after cudaDeviceReset the next call looks it up again); make
 *     that first call before any stream capture.
 *   - Pointer rules as for mc2_moe_counts (16-byte aligned arrays, else
 *     MC2_ERR_INVALID_ARG with nothing launched).
 *   - Allocates nothing and calls no allocating routine.
 *   - Every call shares the one array: calls whose kernels may overlap on the
 *     GPU (other streams, other host threads) race and corrupt each other's
 *     results.  Serialise them, e.g. on one stream.
 */
mc2_status_t mc2_moe_counts_static(const mc2_shape_t* s, const int32_t* sel, int32_t* cnt,
                                   int32_t* recv, int32_t* offsets, int32_t* permute_src,
                                   int32_t* unpermute_dst, int32_t* dev_status, void* stream);

/*
 * The non-fused baseline of the same block: the data flow of the "alltoall"
 * dispatcher that MC2 replaces ("NPU Training Operators - MC2", sections
 * "Execution path" and "Migration checks": permute, then the plain grouped
 * matmul).  mc2_moe_counts, then mc2_permute_rows, then mc2_gmm_swiglu, then
 * mc2_gmm_alltoallv computes exactly what mc2_moe_forward computes (h and out
 * are bitwise equal), with the permuted token rows materialised in between
 * instead of gathered inside fc1.  It exists to measure what that fusion
 * buys.  bf16 only (act = out = MC2_BF16; other types: MC2_ERR_UNSUPPORTED).
 *
 * mc2_permute_rows -- xp[p, :] = x[permute_src[p] / k, :] for every p < T*k.
 *   x [T, H] and xp [T*k, H] bf16 [dev]; permute_src [T*k] int32 [dev] from
 *   mc2_moe_counts (every entry a valid flat index).
 * mc2_gmm_swiglu -- for each expert e and each row p in [offsets[e],
 *   offsets[e+1]): h[p, :] = SwiGLU(xp[p, :] @ w1[e]); rows from offsets[E]
 *   on (invalid ids) are not written.  xp [T*k, H], w1 [E, H, 2I], h [T*k, I]
 *   bf16 [dev]; offsets [E+1] int32 [dev].  dev_status as above (may be NULL).
 * Pointer and shape rules as for the other entry points.
 */
mc2_status_t mc2_permute_rows(const mc2_shape_t* s, const void* x, const int32_t* permute_src,
                              void* xp, void* stream);
mc2_status_t mc2_gmm_swiglu(const mc2_shape_t* s, const void* xp, const void* w1,
                            const int32_t* offsets, void* h, int32_t* dev_status, void* stream);

/*
 * Backward of the block (bf16): the gradients of L = sum(out * dout) with
 * respect to x, w1, w2 and probs, by the chain rule back through the steps of
 * "NPU Training Operators - MC2", section "Execution path" (10 back to 6; the
 * fused AllToAllGroupedMatmul / GroupedMatmulAllToAll operators of the pages
 * wrap forward and backward).  Ids outside [0, E) get no gradient (their
 * dprobs is 0).  The forward's h passes through its bf16 rounding with
 * derivative 1; G = x[t] @ w1[e] is recomputed in bf16.
 *
 * mc2_transpose_weights -- w1t [E, 2I, H] = w1 transposed per expert, w2t
 *   [E, H, I] = w2 transposed, bf16 [dev]; once whenever the weights change.
 * mc2_alltoallv_gmm_keep -- the training form of mc2_alltoallv_gmm (bf16):
 *   also keeps the pre-activation rows g [T*k, 2I] bf16 [dev] (gate | up of
 *   every valid permuted row) for the backward; h [T*k, I] is then
 *   bf16(silu(gate) * up) of those bf16 rows.  Same rules as
 *   mc2_alltoallv_gmm otherwise.
 * mc2_moe_backward -- inputs: x [T, H] bf16, probs [T, k] fp32, w1 [E, H, 2I],
 *   g (the rows kept by mc2_alltoallv_gmm_keep, or NULL: then they are
 *   recomputed from x and w1, bitwise the same),
 *   w1t, w2t (from mc2_transpose_weights), dout [T, H] bf16, and offsets,
 *   permute_src, unpermute_dst of mc2_moe_counts for the same ids.  Outputs:
 *   dx [T, H] bf16, dw1 [E, H, 2I] fp32, dw2 [E, I, H] fp32 (zero for experts
 *   without rows), dprobs [T, k] fp32.  ws: mc2_backward_workspace_bytes(s)
 *   bytes [dev], 256-byte aligned.  act = out = MC2_BF16 only (else
 *   MC2_ERR_UNSUPPORTED).  Pointer rules, errors and dev_status as above.
 */
size_t mc2_backward_workspace_bytes(const mc2_shape_t* s);
mc2_status_t mc2_alltoallv_gmm_keep(const mc2_shape_t* s, const void* x, const void* w1,
                                    const int32_t* offsets, const int32_t* permute_src, void* h,
                                    void* g, int32_t* dev_status, void* stream);
mc2_status_t mc2_transpose_weights(const mc2_shape_t* s, const void* w1, const void* w2,
                                   void* w1t, void* w2t, void* stream);
mc2_status_t mc2_moe_backward(const mc2_shape_t* s, const void* x, const float* probs,
                              const void* w1, const void* g, const void* w1t, const void* w2t,
                              const void* dout,
                              const int32_t* offsets, const int32_t* permute_src,
                              const int32_t* unpermute_dst, void* dx, float* dw1, float* dw2,
                              float* dprobs, void* ws, int32_t* dev_status, void* stream);

/*
 * Quantised matmul + reduce-scatter over W logical tensor-parallel ranks, the
 * operation of "torch_npu.npu_mm_reduce_scatter_base" (Ascend op-plugin docs,
 * sections "Function description" and "Parameters") in its quantised form:
 * rank r holds x1_r [m, k] int8 with per-token scales x1_scale_r [m] (fp32)
 * and x2_r [k, n] int8 with per-channel scales x2_scale_r [n] (fp32); the
 * reduce op is a sum, no bias, bf16 output:
 *   total = sum over r of (x1_scale_r * x2_scale_r) * (x1_r @ x2_r)
 * and rank r's result is rows [r*m/W, (r+1)*m/W) of total.
 *
 * Inputs [dev], stacked over ranks: x1 [W, m, k], x1_scale [W, m], x2 [W, k,
 * n], x2_scale [W, n].  Output out [m, n] bf16 [dev]: all ranks' results,
 * rank r's block at rows r*m/W.  Each rank's x1_r @ x2_r is summed exactly
 * (int32); the products (x1_scale * x2_scale) * float(acc) are summed in fp32
 * in rank order, then rounded once to bf16.
 * Rules: W >= 1, m >= 0, m % W == 0 (the pages: m divisible by world_size),
 * k and n multiples of 64, 64 <= k <= 4096 (the pages allow k up to 65535;
 * here K is summed in exact chunks of 1024 in at most four accumulators),
 * n >= 64; W*m < 2^31.  ws: mc2_mm_reduce_scatter_workspace_bytes(s) bytes
 * [dev], 256-byte aligned (bf16 copies of x1 and x2, then room for the int32
 * partial products of every rank, which only the two-pass form of
 * mc2_set_mmrs_path writes).  Errors and dev_status as for the block.
 */
typedef struct {
  int32_t m;  /* rows of each rank's x1 */
  int32_t k;  /* each rank's reduction length */
  int32_t n;  /* columns */
  int32_t W;  /* logical ranks (world_size) */
} mc2_mmrs_shape_t;

size_t mc2_mm_reduce_scatter_workspace_bytes(const mc2_mmrs_shape_t* s);
mc2_status_t mc2_mm_reduce_scatter_i8(const mc2_mmrs_shape_t* s, const int8_t* x1,
                                      const float* x1_scale, const int8_t* x2,
                                      const float* x2_scale, void* out, void* ws,
                                      int32_t* dev_status, void* stream);

/*
 * mc2_prepack_weights -- int8 path only (a no-op returning MC2_OK for other
 * activation types): expands the int8 weights w1 [E, H, 2I] and w2 [E, I, H]
 * into bf16 copies held in `ws`.  Every int8 value is exact in bf16; the
 * int8 GEMMs run on the bf16 tensor cores (sm_103a has no integer tcgen05
 * MMA) and read these copies, so call this once whenever the weights change
 * and before any act=I8 mc2_alltoallv_gmm / mc2_gmm_alltoallv / mc2_moe_forward
 * that uses this workspace.  w1/w2 passed to those calls must be the same
 * tensors.  The int8 path requires H <= 4096 and I <= 4096 (K is summed in
 * at most four exact chunks of 1024).
 */
mc2_status_t mc2_prepack_weights(const mc2_shape_t* s, const void* w1, const void* w2, void* ws,
                                 void* stream);

/*
 * mc2_moe_forward -- the whole block (the three calls above, in order) on
 * device buffers.  cnt/recv/offsets/permute_src/unpermute_dst/h/h_scale are
 * outputs as above (h_scale may be NULL unless act is I8); out is [T, H].
 */
mc2_status_t mc2_moe_forward(const mc2_shape_t* s, const void* x, const float* x_scale,
                             const int32_t* sel, const float* probs, const void* w1,
                             const float* w1_scale, const void* w2, const float* w2_scale,
                             int32_t* cnt, int32_t* recv, int32_t* offsets,
                             int32_t* permute_src, int32_t* unpermute_dst, void* h,
                             float* h_scale, void* out, void* ws, int32_t* dev_status,
                             void* stream);

/*
 * mc2_selftest_wait -- exercises the bounded device-side wait used by every
 * kernel: one CTA waits on an mbarrier phase that nothing completes, gives up
 * after `limit_ns` nanoseconds, ORs MC2_DEV_TIMEOUT into *dev_status and
 * returns.  Test hook only; never hangs the GPU.
 */
mc2_status_t mc2_selftest_wait(uint64_t limit_ns, int32_t* dev_status, void* stream);

/*
 * Test and diagnostic hooks.  A production caller needs none of them.  Each
 * setting holds for later calls made on the host thread that set it (and on
 * no other thread) until that thread sets it again; apart from the wait
 * limit, none of them changes any result bit (the tests check this).
 */

/* Set the device-side wait limit (nanoseconds) used by later launches of
 * this thread's calls; 0 restores the default (2 s). Host only. */
void mc2_set_wait_limit_ns(uint64_t limit_ns);

/* Grouped-GEMM tiling for later calls of this thread: 0 = automatic
 * (bf16/tf32 fc2 on CTA pairs with 256x256 tiles when experts average >= 256
 * rows; everything else on one CTA per 128x256 tile, the int8 GEMMs with
 * their K chunks folded in TMEM), 1 = always single CTAs (int8 GEMMs:
 * 128x128 tiles), 2 = always CTA pairs (int8 GEMMs: 256x128 tiles); other
 * values mean 0.  The choice does not change any result bit: every tiling
 * accumulates each output in the same K order.  Host only. */
void mc2_set_tile_pairing(int32_t mode);

/* Which counts pass later calls of this thread use: 0 (default) one launch
 * of a thread-block cluster (up to 16 CTAs, per-CTA tables in shared memory)
 * whenever its tables fit, else three launches over the workspace tables;
 * 1 always three launches; 2 the same as 0 (the cluster pass when it fits).
 * Outputs are identical either way.  Host only. */
void mc2_set_counts_path(int32_t mode);

/* Which form later mc2_mm_reduce_scatter_i8 calls of this thread take:
 * 0 (default) fused, one CTA-pair kernel after the int8 -> bf16 copies that
 * folds every rank's dequantised product into an on-chip fp32 sum; 1 two
 * passes, the int32 partial product of every rank written to the workspace
 * (as [W, m, n] int32, after the two bf16 copies, each region 256-byte
 * aligned), then a reduce kernel.  Both fold rank r in as
 * fma(x1_scale * x2_scale, float(acc), sum), r ascending: the outputs are
 * identical bit for bit.  Host only. */
void mc2_set_mmrs_path(int32_t mode);

/* Where later bf16/fp32 mc2_gmm_alltoallv calls of this thread do the
 * weighted combine: 0 (default) in a separate kernel after fc2; 1 inside
 * the fc2 kernel (top-k up to 8; larger k take the separate kernel): the
 * fc2 kernel counts the rows of every (token, 256-column tile) as their
 * stores complete, sums a few completed tokens per stored row block itself
 * and leaves the rest to a follow-up kernel.  Both sum the same products in
 * the same order: the outputs are identical bit for bit.  Host only. */
void mc2_set_combine_path(int32_t mode);

/* Timing of a grouped-matmul kernel alone (a diagnostic hook).  While set,
 * every later call of this thread that launches an fc1 or fc2 kernel
 * (mc2_alltoallv_gmm, mc2_gmm_alltoallv, mc2_gmm_swiglu, mc2_moe_forward)
 * records `before` on its stream right before that kernel's launch and
 * `after` right after it, so the time between the two events is that
 * kernel's.  A call with two such kernels (mc2_moe_forward) records both
 * events twice; the second pair, around fc2, is what remains.  A call that
 * launches nothing (T = 0) records nothing.  The bf16 fc1
 * call launches only its kernel; the int8 calls also convert their
 * activations to bf16 before it and re-quantise h or combine after it.
 * The handles are cudaEvent_t created by the caller on the stream's device
 * (the library does not own them); either may be NULL (that event is not
 * recorded), and both NULL, the default, records nothing.  A failed record
 * returns MC2_ERR_CUDA.  Results are identical either way.  Host only. */
void mc2_set_gemm_events(void* before, void* after);

/* Programmatic dependent launch between the kernels of later calls of this
 * thread: 1 (default) lets each kernel's set-up overlap the end of the
 * previous kernel on the stream (each kernel still waits for its
 * predecessors' results before reading or writing global memory); 0 launches
 * them in plain stream order.  Results are identical either way.  Host only. */
void mc2_set_launch_overlap(int32_t enabled);

/* Number of kernel launches the last successful call on this host thread
 * enqueued. Host only. */
int32_t mc2_last_launch_count(void);

const char* mc2_status_str(mc2_status_t st);

#ifdef __cplusplus
}
#endif

#endif /* MC2MOE_H */
