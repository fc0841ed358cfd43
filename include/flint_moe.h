/*
 * flint_moe: routed-expert MoE block with NVFP4 (W4) experts and BF16 (A16)
 * activations, for one NVIDIA GB300 (sm_103a).
 *
 * The block is the one the vLLM API page "vllm.models.flint.ops.moe"
 * describes in its module docstring ("Numerics") and in flint_moe / route:
 * BF16 router logits, fp32 sigmoid top-k renormalised and rounded to BF16,
 * per selected expert an NVFP4 gate/up projection (E2M1 codes times E4M3
 * block scales, fp32 accumulation, per-expert fp32 global scale on the
 * accumulator), act = bf16(silu(g) * u), an NVFP4 down projection
 * y_e = bf16(acc * gs_e), the routed sum bf16(sum_j tw_j * y_j) accumulated
 * in fp32 in rank order, plus an ungated BF16 shared expert:
 * out = bf16(routed + shared).  Variants take an NVFP4 shared expert, BF16
 * routed experts or an add-RMSNorm prologue; flint_qkv_fused is the decode
 * step before attention (page "vllm.models.flint.ops.qkv_fused").
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers, row-major, contiguous and
 *    16-byte aligned (fp32 scalars and int32/int64 index arrays: aligned to
 *    their size; the paged KV caches of flint_qkv_fused take strides).  The
 *    caller owns every buffer; the library keeps no per-call global state
 *    and allocates nothing.
 *  - Work is enqueued on `stream` and returns before it completes.  Argument
 *    errors are reported synchronously (negative return, nothing enqueued);
 *    launch failures return FLINT_ERR_CUDA.
 *  - `workspace` is caller-owned device memory of at least
 *    flint_moe_workspace_bytes(shape) bytes (256-byte aligned), zero-filled
 *    ONCE after allocation (e.g. cudaMemsetAsync).  Every launch leaves its
 *    counters at zero again, so the same workspace serves any number of calls
 *    in stream order (and CUDA-graph replays) with the same H, E, I and SI
 *    and any M up to the one it was sized for.  Calls that may overlap on the
 *    GPU (two streams) need separate workspaces.
 */
#ifndef FLINT_MOE_H_
#define FLINT_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* flint_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum {
  FLINT_OK = 0,
  FLINT_ERR_INVALID_ARG = -1, /* null/misaligned pointer, bad shape */
  FLINT_ERR_UNSUPPORTED = -2, /* shape outside what the kernels support */
  FLINT_ERR_WORKSPACE = -3,   /* workspace missing or too small */
  FLINT_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed */
  FLINT_ERR_TIMEOUT = -5,     /* a bounded device-side wait gave up */
  FLINT_ERR_SCRATCH = -6,     /* shape needs more than the fixed static scratch */
};

/* Problem shape.
 *   M      tokens (rows of x), M >= 0.  M = 0 (an empty batch) is checked
 *          as a shape and returns FLINT_OK without any launch or memory
 *          access; the M-sized buffers and the workspace may then be NULL.
 *   H      hidden size; multiple of 64
 *   E      routed experts, 1..256
 *   top_k  experts per token, 1..min(E, 32)
 *   I      routed-expert intermediate size; multiple of 64
 *   SI     shared-expert intermediate size; 0 (no shared expert) or a
 *          multiple of 64
 * A shape outside these limits is invalid (FLINT_ERR_INVALID_ARG).  The
 * kernels run K in 128-wide slices: a valid shape whose H, I or SI is an odd
 * multiple of 64 is not supported yet, and every entry point returns
 * FLINT_ERR_UNSUPPORTED for it without enqueuing anything (the size queries
 * return 0). */
typedef struct {
  int M, H, E, top_k, I, SI;
} flint_moe_shape;

/* Bytes of device workspace flint_moe_route / flint_moe_forward need for
 * `shape`; 0 if the shape is invalid or not supported. */
size_t flint_moe_workspace_bytes(const flint_moe_shape* shape);

/* Routing only: "route" on the page above (BF16 router logits -> top-k ids
 * int32 and renormalised fp32 weights), with the _topk_row rules: experts
 * ranked by BF16 logit (bit order: -0 below +0), ties to the lower expert
 * index; s = 1 / (1 + exp(-logit)) in fp32; tw = bf16(s / (sum_k s + 1e-20))
 * stored as fp32; both outputs in rank order (column 0 = largest logit).
 * The fp32 logit sum is taken in one fixed order (32 strided partial sums
 * combined by a xor butterfly), so ids are reproducible bit for bit.
 *
 *   x          bf16 [M, H]
 *   router_w   bf16 [E, H]
 *   ids        int32 [M, top_k]   (output)
 *   tw         fp32  [M, top_k]   (output)
 */
int flint_moe_route(const void* x, const void* router_w, const flint_moe_shape* shape,
                    int32_t* ids, float* tw, void* workspace, size_t workspace_bytes,
                    flint_stream_t stream);

/* The whole MoE block: "flint_moe" on the page above (routing, NVFP4 experts,
 * weighted combine) plus the ungated shared expert's output added in.
 *
 *   x            bf16 [M, H]
 *   router_w     bf16 [E, H]
 *   w13          uint8 [E, 2I, H/2]  e2m1 codes, gate rows [0, I) then up rows
 *                                     [I, 2I); even K index in the low nibble
 *   w13_sf       uint8 [E, 2I, H/16] e4m3 (float8_e4m3fn) block scales, one per
 *                                     16 consecutive K of a row
 *   w13_gs       fp32  [E]           global scale of gate and up (ModelOpt
 *                                     weight_scale_2; gate and up must share it)
 *   w2           uint8 [E, H, I/2], w2_sf uint8 [E, H, I/16], w2_gs fp32 [E]
 *   shared_gu    bf16 [2*SI, H]      shared expert gate rows then up rows
 *                                     (NULL when SI == 0)
 *   shared_down  bf16 [H, SI]        (NULL when SI == 0)
 *   out          bf16 [M, H]         (output)
 *   ids_out, tw_out  optional int32 / fp32 [M, top_k] copies of the routing
 *                    (NULL to skip)
 *
 * Numerics: BF16 activations, E2M1 x E4M3 weights dequantised exactly,
 * fp32 accumulation with the global scale applied to the accumulator;
 * act = bf16(silu(g) * u); y_e = bf16(acc * gs2_e); shared expert
 * gS, uS = bf16(dot), sact = bf16(silu(gS) * uS), ys = bf16(dot);
 * out = bf16(bf16(sum_j tw_j y_j) + ys), the routed sum in rank order.
 * How close the sums come to the exact ones depends on the path (see
 * flint_moe_plan):
 *  - FLINT_PATH_SINGLE_LAUNCH forms every gate/up sum (routed and shared) as
 *    the exact sum of the exact products rounded once to fp32, the down sums
 *    from exact 128-K partial sums added with TwoSum, and every sigmoid with
 *    the correctly rounded exp wherever the BF16 rounding depends on it;
 *  - FLINT_PATH_DECODE forms the shared expert's gate/up sums exactly (its
 *    activation reaches every output of a token) and evaluates act and sact
 *    with the correctly rounded exp; the routed sums follow the tensor
 *    cores' fp32 order in 128-K chains;
 *  - the fallback and grouped paths accumulate in the tensor cores' fp32
 *    order with sigmoid = rcp.approx(1 + ex2.approx(-g log2 e)).
 * Where a sum is not exact, its BF16 rounding now and then moves by one ulp.
 * The kernels of the decode paths multiply activations by weights scaled by
 * 2^-7 (exactly) and scale the fp32 accumulator back by 2^7, so single
 * products below 2^-119 in magnitude are formed as fp32 subnormals; no sum
 * of realistic size resolves them. */
int flint_moe_forward(const void* x, const void* router_w, const uint8_t* w13,
                      const uint8_t* w13_sf, const float* w13_gs, const uint8_t* w2,
                      const uint8_t* w2_sf, const float* w2_gs, const void* shared_gu,
                      const void* shared_down, const flint_moe_shape* shape, void* out,
                      int32_t* ids_out, float* tw_out, void* workspace, size_t workspace_bytes,
                      flint_stream_t stream);

/* The decode MoE block with its add-RMSNorm prologue: "flint_moe_ll" on the
 * page above.  residual' = attn_out + residual and x = rms_norm(residual')
 * are formed as norm.fused_add_rms_norm (_add_rms_norm on that page): from
 * the unrounded fp32 sum s = a + r, residual' = bf16(s),
 * v = sum_h(s^2) / H + eps (the sum of squares as the exact sum rounded once
 * to fp32), inv = 1 / sqrt(v) rounded once to fp32, xn = bf16((s * inv) * w);
 * then the MoE block of flint_moe_forward runs on xn.
 *
 *   attn_out, residual  bf16 [M, H]   (inputs, not modified)
 *   ln_weight           bf16 [H]      norm weight
 *   eps                 0 <= eps <= 1
 *   residual_out        bf16 [M, H]   (output) residual'
 *   xn_out              bf16 [M, H]   (optional output) the normalised rows;
 *                                      NULL keeps them in the workspace
 *   the other arguments as for flint_moe_forward; out is the MoE output.
 * One more kernel (one warp per token) runs ahead of the block's kernels,
 * chained to them with programmatic dependent launch.  The workspace is the
 * one flint_moe_workspace_bytes(shape) sizes. */
int flint_moe_forward_add_norm(const void* attn_out, const void* residual, const void* ln_weight,
                               float eps, const void* router_w, const uint8_t* w13,
                               const uint8_t* w13_sf, const float* w13_gs, const uint8_t* w2,
                               const uint8_t* w2_sf, const float* w2_gs, const void* shared_gu,
                               const void* shared_down, const flint_moe_shape* shape, void* out,
                               void* residual_out, void* xn_out, int32_t* ids_out, float* tw_out,
                               void* workspace, size_t workspace_bytes, flint_stream_t stream);

/* The MoE block with an NVFP4 shared expert (the shared expert of
 * "LLMoEWeights" on the page above: ModelOpt-packed gate/up and down with
 * block scales and an fp32 global scale each).  The shared expert follows
 * the routed experts' rule: g, u = fp32(sum) * sgu_gs,
 * sact = bf16(silu(g) * u), ys = bf16(fp32(sum) * sdown_gs), and
 * out = bf16(bf16(routed) + ys); its sums are exact (as in the single-launch
 * path).  The routed part takes the path flint_moe_plan names for the shape
 * with SI = 0.
 *
 *   sgu       uint8 [2*SI, H/2]   e2m1 codes, gate rows then up rows
 *   sgu_sf    uint8 [2*SI, H/16]  e4m3 block scales;  sgu_gs fp32 [1]
 *   sdown     uint8 [H, SI/2],  sdown_sf uint8 [H, SI/16],  sdown_gs fp32 [1]
 *   the other arguments as for flint_moe_forward (shape->SI >= 128; the
 *   workspace is the one flint_moe_workspace_bytes(shape) sizes). */
int flint_moe_forward_nvfp4_shared(const void* x, const void* router_w, const uint8_t* w13,
                                   const uint8_t* w13_sf, const float* w13_gs, const uint8_t* w2,
                                   const uint8_t* w2_sf, const float* w2_gs, const uint8_t* sgu,
                                   const uint8_t* sgu_sf, const float* sgu_gs,
                                   const uint8_t* sdown, const uint8_t* sdown_sf,
                                   const float* sdown_gs, const flint_moe_shape* shape, void* out,
                                   int32_t* ids_out, float* tw_out, void* workspace,
                                   size_t workspace_bytes, flint_stream_t stream);

/* Fused decode qkv: "flint_qkv_fused" on the page
 * "vllm.models.flint.ops.qkv_fused".  Per token t < M:
 *   s = x + residual (fp32; s = x without a residual), residual_out =
 *   bf16(s), xn = bf16((s * inv) * norm_weight) with inv = 1 / sqrt(mean(s^2)
 *   + eps) (the add-RMSNorm of flint_moe_forward_add_norm);
 *   qkv = bf16(fp32(xn . W row) * global_scale) for NVFP4 weights (every sum
 *   the exact sum of the products rounded once to fp32), bf16(fp32 sum) for
 *   BF16 weights; rows [0, 128 nq) are the q heads, then nkv k heads, then
 *   nkv v heads;
 *   per q and k head (128 values v): n = (v * inv) * w (w = q_norm_weight or
 *   k_norm_weight, inv = 1 / sqrt(sum(v^2) / 128 + qk_eps), the sum of the
 *   squares exact and rounded once), then NeoX RoPE with the fp32 table row
 *   c | s = cos_sin_cache[positions[t]]: o[d] = n[d] c[d] - n[d+64] s[d],
 *   o[d+64] = n[d+64] c[d] + n[d] s[d] (d < 64), fp32 math, o = n without a
 *   table; q_out[t, 128 h + d] = bf16(o) for q head h;
 *   with slot = slot_mapping[t] (t < num_slots) and slot >= 0: the k head h's
 *   bf16(o) and the v head h's values go to k_cache / v_cache at element
 *   offset (slot / block_size) * stride_block + (slot % block_size) *
 *   stride_slot + h * stride_head + d.
 *
 *   x, residual  bf16 [M, H] (residual NULL: plain RMSNorm, residual_out
 *                unused)
 *   norm_weight  bf16 [H]
 *   weight       NVFP4 codes uint8 [N, H/2] (even K in the low nibble) with
 *                weight_scale uint8 [N, H/16] e4m3 row-major and one fp32
 *                global_scale; or BF16 [N, H] with weight_scale and
 *                global_scale NULL.  N = (num_q_heads + 2 num_kv_heads) * 128.
 *                (The page's 128x4-swizzled scale order is a permutation of
 *                the same bytes; this entry point takes them row-major.)
 *   q_norm_weight, k_norm_weight  bf16 [128]
 *   cos_sin_cache  fp32 [max_pos, 128] (cos | sin) or NULL (no RoPE);
 *                positions int64 [M]
 *   k_cache, v_cache  bf16 paged caches (same strides, in elements), with
 *                num_blocks blocks of block_size slots; slot_mapping int64
 *                [num_slots]
 *   q_out        bf16 [M, num_q_heads * 128] (output)
 *   residual_out bf16 [M, H] (output, with a residual)
 *   workspace    flint_qkv_workspace_bytes(M, H, nq, nkv) bytes, 256-byte
 *                aligned; its first word is a status word that
 *                flint_moe_status reads.
 * H must be a multiple of 64 (FLINT_ERR_INVALID_ARG otherwise); an odd
 * multiple returns FLINT_ERR_UNSUPPORTED.  M = 0 is a no-op.  A position
 * outside [0, max_pos) leaves that token's heads without RoPE, and a slot at
 * or past num_blocks * block_size is not written; either records
 * FLINT_ERR_INVALID_ARG in the status word.  Three launches (input norm,
 * GEMV, heads) chained with programmatic dependent launch on `stream`. */
size_t flint_qkv_workspace_bytes(int M, int H, int num_q_heads, int num_kv_heads);
int flint_qkv_fused(const void* x, const void* residual, const void* norm_weight, float eps,
                    const void* weight, const uint8_t* weight_scale, const float* global_scale,
                    const void* q_norm_weight, const void* k_norm_weight, float qk_eps,
                    const float* cos_sin_cache, long long max_pos, const long long* positions,
                    void* k_cache, void* v_cache, long long stride_block, long long stride_slot,
                    long long stride_head, int block_size, long long num_blocks,
                    const long long* slot_mapping, int num_slots, int M, int H, int num_q_heads,
                    int num_kv_heads, void* q_out, void* residual_out, void* workspace,
                    size_t workspace_bytes, flint_stream_t stream);

/* The decode MoE block on BF16 routed experts: "flint_moe_bf16_decode" on
 * the page above.  The same routing as flint_moe_route, then per selected
 * expert act = bf16(silu(g) * u) from the fp32 gate/up sums (no global
 * scale), y_e = bf16(acc), routed = bf16(sum_j tw_j y_j) in fp32 in rank
 * order, out = bf16(routed + shared_out).  Every gate/up and down sum is the
 * exact sum of the products rounded once to fp32.
 *
 *   x            bf16 [M, H]
 *   router_w     bf16 [E, H]
 *   w13          bf16 [E, 2I, H]   gate rows [0, I) then up rows [I, 2I)
 *                                   (row-major; the page's blocked storage
 *                                   order is not used)
 *   w2           bf16 [E, H, I]
 *   shared_out   bf16 [M, H]       the shared expert's output, added to the
 *                                   routed part (NULL: no shared expert)
 *   out          bf16 [M, H]       (output)
 *   ids_out, tw_out, workspace, stream: as for flint_moe_forward.
 * The shape's SI must be 0 (FLINT_ERR_INVALID_ARG otherwise); M above 64
 * returns FLINT_ERR_UNSUPPORTED.  Four launches (router, gate/up, down,
 * combine) chained with programmatic dependent launch. */
int flint_moe_forward_bf16(const void* x, const void* router_w, const void* w13, const void* w2,
                           const void* shared_out, const flint_moe_shape* shape, void* out,
                           int32_t* ids_out, float* tw_out, void* workspace, size_t workspace_bytes,
                           flint_stream_t stream);

/* Routing without caller memory: the same kernel, numerics and outputs as
 * flint_moe_route, but its intermediates live in a fixed scratch array that
 * the library itself holds in device memory (2 MiB per device, a file-scope
 * __device__ array).  The pages describe no such entry point; it exists for
 * callers that cannot hand over or allocate device memory at the point of the
 * call (inside an allocator hook, a memory-pool callback, or code that must
 * not touch the caching allocator), and it makes no cudaMalloc/cudaFree or
 * other allocating call.
 *
 *   x, router_w, ids, tw, shape, stream: as for flint_moe_route (I and SI of
 *   the shape are ignored).
 *
 * Size limit: the call needs flint_moe_route_noalloc_bytes(shape) bytes of
 * scratch, 256-aligned regions for ceil(M/8) int32 counters, bf16 [M, E]
 * logits and int32 + fp32 [M, top_k]; when that exceeds
 * flint_moe_route_noalloc_capacity() the call returns FLINT_ERR_SCRATCH and
 * enqueues nothing (at E = 128, top_k = 8 about 6500 tokens fit).
 * The first call in each CUDA context looks up the scratch's device address
 * in that context (cudaGetSymbolAddress, which may load the module) and
 * caches it under the context's process-unique id, so a context created
 * later (another device, a driver-API context, or the primary context
 * re-created after cudaDeviceReset) gets its own lookup; make the first call
 * in a context outside any stream capture.  Every call clears the counters
 * (cudaMemsetAsync on `stream`) before the kernel; nothing else needs an
 * initial value.  All calls on one device share the one scratch: two calls
 * that may run at the same time on the GPU (different streams or host threads
 * without ordering between them) race and give wrong results; order them on
 * one stream or with events. */
int flint_moe_route_noalloc(const void* x, const void* router_w, const flint_moe_shape* shape,
                            int32_t* ids, float* tw, flint_stream_t stream);

/* Scratch bytes flint_moe_route_noalloc needs for `shape` (0 if invalid or
 * not supported). */
size_t flint_moe_route_noalloc_bytes(const flint_moe_shape* shape);

/* Size of the fixed scratch (bytes per device). */
size_t flint_moe_route_noalloc_capacity(void);

/* Synchronises `stream`, then reads and clears the device status word of
 * `workspace`: FLINT_OK, or the error a kernel recorded (FLINT_ERR_TIMEOUT
 * when a bounded device-side wait gave up).  FLINT_ERR_CUDA if the stream
 * reports an error.  This call blocks the calling host thread: it waits for
 * `stream` and then reads (and, when non-zero, clears) the word with
 * synchronous copies on the legacy default stream, so it does not belong
 * inside stream capture or a latency-critical loop. */
int flint_moe_status(void* workspace, flint_stream_t stream);

/* Which kernels flint_moe_forward runs for `shape` on the calling thread's
 * current device (a host-side query; nothing is enqueued):
 *   FLINT_PATH_NONE            M = 0: nothing
 *   FLINT_PATH_SINGLE_LAUNCH   one cooperative kernel: router, top-k, expert
 *                              grouping, gate/up, down and combine (few tokens;
 *                              every gate/up sum exact before its rounding)
 *   FLINT_PATH_DECODE          router, gate/up and down kernels chained with
 *                              programmatic dependent launch (M <= 64)
 *   FLINT_PATH_DECODE_FALLBACK the same three steps for shapes outside the
 *                              limits of the two paths above
 *   FLINT_PATH_GROUPED         many tokens: router with expert histogram,
 *                              per-expert tcgen05 GEMMs, combine
 * or a negative FLINT_ERR_* code (invalid / unsupported shape, CUDA error). */
enum {
  FLINT_PATH_NONE = 0,
  FLINT_PATH_SINGLE_LAUNCH = 1,
  FLINT_PATH_DECODE = 2,
  FLINT_PATH_DECODE_FALLBACK = 3,
  FLINT_PATH_GROUPED = 4,
};
int flint_moe_plan(const flint_moe_shape* shape);

/* Path preference (process-wide, default FLINT_PATH_NONE).  By default a
 * batch of at most 64 tokens runs FLINT_PATH_DECODE, which measures faster.
 * With FLINT_PATH_SINGLE_LAUNCH, flint_moe_forward runs the single-launch
 * kernel wherever it supports the shape (M <= 8, M * top_k <= 64,
 * H <= 2048, I <= 2048, SI <= 1024 and E <= twice the SM count): its gate/up
 * sums are the exact sums rounded once to fp32.  Returns FLINT_OK, or
 * FLINT_ERR_INVALID_ARG for another value.  Set it between calls, not while
 * another host thread enqueues work. */
int flint_moe_prefer_path(int path);

/* Kernel spans for profiling (process-wide, default off).  With a device
 * buffer of FLINT_SPAN_KERNELS * FLINT_SPAN_CTAS * 2 uint64 words that the
 * caller zero-fills, every later launch records, for each of its kernels
 * (index FLINT_SPAN_*) and CTA c (slot c mod FLINT_SPAN_CTAS), the
 * %globaltimer value (ns) at the CTA's start, stored as its bitwise
 * complement (word 2 * slot), and at its last warp's exit (word 2 * slot + 1).
 * A kernel's span is then [min start, max exit] over its slots.  The cost
 * is one atomic per CTA and one per warp; NULL turns it off.  Set it between
 * calls; the buffer must outlive the launches that write it. */
enum {
  FLINT_SPAN_ROUTE = 0, FLINT_SPAN_GATE_UP = 1, FLINT_SPAN_DOWN = 2, FLINT_SPAN_SINGLE_LAUNCH = 3,
  FLINT_SPAN_GROUP_COUNT = 4, FLINT_SPAN_GROUP_SCAN = 5, FLINT_SPAN_GROUP_SCATTER = 6,
  FLINT_SPAN_PLAN = 7, FLINT_SPAN_GATHER = 8, FLINT_SPAN_GEMM1 = 9, FLINT_SPAN_GEMM2 = 10,
  FLINT_SPAN_COMBINE = 11, FLINT_SPAN_ADD_NORM = 12, FLINT_SPAN_SHARED_GATE_UP = 13,
  FLINT_SPAN_SHARED_DOWN = 14, FLINT_SPAN_SHARED_ADD = 15, FLINT_SPAN_QKV_GEMV = 16,
  FLINT_SPAN_QKV_HEADS = 17,
  FLINT_SPAN_KERNELS = 18, FLINT_SPAN_CTAS = 1024
};
int flint_moe_record_spans(unsigned long long* spans);

/* Static description of an error code. */
const char* flint_moe_strerror(int code);

/* Test hook for the failure path (process-wide, default off).  With
 * site = FLINT_FAULT_DOWN_HANDOVER the next forward launches leave out one
 * hand-over signal into the down projection: in the three-kernel decode
 * path the warp holding the second half of an item's K never raises its
 * flag; in the single-launch path the CTA that sees the grid barrier before
 * the down phase complete never passes that on to its down records.  The
 * waiting warps give up after their bounded wait (200 ms), record
 * FLINT_ERR_TIMEOUT with the wait site (17), CTA and stage in status words
 * 1..3 of the workspace, and every warp of the launch exits; the outputs of
 * such a call are undefined, the context stays usable and the next call
 * without the hook is exact again.  Nothing faults, traps or hangs.
 * site = 0 turns the hook off.  Returns FLINT_OK, or FLINT_ERR_INVALID_ARG
 * for an unknown site. */
enum { FLINT_FAULT_NONE = 0, FLINT_FAULT_DOWN_HANDOVER = 17 };
int flint_moe_debug_fault(int site);

#ifdef __cplusplus
}
#endif

#endif /* FLINT_MOE_H_ */
