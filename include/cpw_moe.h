/*
 * cpw_moe.h -- C ABI of the fused FP8 Mixture-of-Experts layer ("Mega-MoE") on one GPU.
 *
 * One call of moe_forward computes, for every token t,
 *     out[t] = bf16( sum_k  w[t,k] * Expert_{idx[t,k]}(x[t]) ),   idx == -1 skipped,
 * where Expert_e(x) = W_down[e] . requant_1x128( silu(W_gate[e] . x) * (W_up[e] . x) )
 * with FP8 e4m3 operands and fp32 block scales.  The steps follow the fused layer of the
 * source pages, on one GPU whose tokens are split into R logical source partitions:
 *   routing count + packed 64-bit slot claim      ("Mega-MoE 内核代码导读：从 Dispatch 到
 *                                                   WGMMA 的融合流水线" §4.1-4.2)
 *   [expert][source][slot] index table            (same page §4.3; Mega-MoE walkthrough,
 *                                                   part 2, kwkr.cn/news/1317662, §1.1)
 *   expert segments + round-robin min-peeling      (walkthrough part 2 §2.4-2.5)
 *   gather into the expert-major FP8 pool          (walkthrough part 2 §2.6)
 *   grouped FP8 GEMMs gate_up -> SwiGLU -> down    (first page §六, §八)
 *   weighted scatter through {source,token,topk}   ("DeepGEMM Mega MoE 对称内存（Symmetric
 *   metadata + top-k combine reduce                 Memory）深度分析" §8-§9)
 *   Output(T) = sum_k w_k Expert_k(T)              ("Dispatch/Combine: 博客理论 ↔ DeepEP 源码
 *                                                   ↔ DeepGEMM Mega MoE 三方对比分析" §1)
 *
 * Conventions for every call below:
 *   - All tensor pointers are DEVICE pointers unless the name says host; they are
 *     row-major, contiguous, and owned by the caller.  FP8 tensors are e4m3 bytes
 *     (OCP FP8 E4M3, largest finite 448).  FP8 row pointers must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Every function returns a moe_status code.  Host-detectable problems are returned
 *     synchronously; problems found by the GPU (bad expert id, slot overflow, a wait
 *     that ran past its time limit) are recorded in a sticky per-handle word that
 *     moe_get_error returns; while it is set, forwards skip their work and `out` is
 *     undefined.
 *   - A handle serves one forward at a time: its workspace is shared by its calls.
 */
#ifndef CPW_MOE_H
#define CPW_MOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_ctx *moe_handle_t;

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,        /* bad size, null or misaligned pointer            */
    MOE_ERR_CUDA = 2,               /* a CUDA runtime/driver call failed               */
    MOE_ERR_CAPACITY = 3,           /* T above the reserved maximum                    */
    MOE_ERR_NO_WEIGHTS = 4,         /* forward before the weights (routed and shared) are loaded */
    MOE_ERR_UNSUPPORTED_DEVICE = 5, /* not an sm_103 GPU, or a shape this build lacks  */
    MOE_ERR_BAD_INDEX = 6,          /* device: an expert id outside [0,E) other than -1 */
    MOE_ERR_TIMEOUT = 7,            /* device: a bounded wait gave up                  */
    MOE_ERR_SLOT_OVERFLOW = 8,      /* device: > T/R rows of one source for one expert */
    MOE_ERR_NOT_RESERVED = 9,       /* forward before moe_reserve                      */
    MOE_ERR_BAD_SCALE = 10          /* block-scaled mode: a weight scale (at the forward) or
                                       an activation scale (device) is not a power of two;
                                       MXFP4 weights: a NaN scale byte (at load), or a forward
                                       forced to the fp32-scale kernel */
};

/* Create a layer for E experts, hidden size H, expert intermediate size I, top-k, and R
 * logical source partitions (the layer object the pages' Python API builds before its
 * forward: "DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析" §10.1).  Requires
 * H % 128 == 0, I % 128 == 0, H <= 16384, I <= 16384, 1 <= topk <= 32, topk <= E <= 1024,
 * 1 <= R <= 64, E*R <= 16384, on the current device, which must be sm_103.  Allocates no
 * device memory.  *out receives the handle. */
int moe_create(int E, int H, int I, int topk, int R, moe_handle_t *out);

/* As moe_create, with n_shared shared experts besides the E routed ones ("DeepGEMM Mega MoE
 * 对称内存（Symmetric Memory）深度分析" §8.2: the combine buffer gets a plane after the top-k
 * ones when shared experts exist, and §10.1 passes their weights separately).  Every token
 * also goes through each shared expert (same H and I as the routed ones), whose output is
 * added to the token's top-k sum with weight 1.  The caller's topk_idx / topk_w stay
 * [T][topk] (routed only); the shared experts' weights come from moe_load_shared_weights.
 * Requires E + n_shared <= 1024, topk + n_shared <= 32, (E + n_shared)*R <= 16384;
 * n_shared = 0 is moe_create. */
int moe_create_shared(int E, int H, int I, int topk, int R, int n_shared, moe_handle_t *out);

/* Allocate the device workspace for up to max_tokens tokens per forward (the pages'
 * host pre-sizing: a larger batch is an error, not a reallocation).  May be called
 * again to grow; not while a forward is in flight. */
int moe_reserve(moe_handle_t h, int max_tokens);

/* Copy the expert weights into the handle (re-laid-out for the GEMMs; the caller keeps
 * ownership of its buffers, which may be freed after the stream has run the copies).
 *   w_gate_up  [E][2I][H] e4m3, rows 0..I-1 = gate, rows I..2I-1 = up
 *   sf_gate_up [E][2I/128][H/128] fp32, one scale per 128x128 block
 *   w_down     [E][H][I] e4m3
 *   sf_down    [E][H/128][I/128] fp32
 * The gate/up rows are interleaved in groups of 8 inside the handle
 * ("DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析" §10.2). */
int moe_load_weights(moe_handle_t h, const uint8_t *w_gate_up, const float *sf_gate_up,
                     const uint8_t *w_down, const float *sf_down, void *stream);

/* Weights of the n_shared shared experts, layouts as moe_load_weights with n_shared in
 * place of E.  Required before a forward of a handle made with n_shared > 0;
 * MOE_ERR_INVALID_ARG on a handle without shared experts. */
int moe_load_shared_weights(moe_handle_t h, const uint8_t *w_gate_up, const float *sf_gate_up,
                            const uint8_t *w_down, const float *sf_down, void *stream);

/* Weight formats (moe_info.weight_format). */
enum moe_weight_format {
    MOE_WEIGHTS_FP8 = 0,    /* e4m3 with fp32 128x128 block scales (moe_load_weights)     */
    MOE_WEIGHTS_MXFP4 = 1   /* E2M1 with UE8M0 1x32 scales (moe_load_weights_mxfp4)       */
};

/* MXFP4 expert weights (FP8 activations x FP4 weights: the pages name an FP8 x FP4 variant
 * of the SM100 kernel, "DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析" §11, without
 * its format; this is the OCP Microscaling MXFP4 block: 32 consecutive elements of a row
 * share one power-of-two scale).
 *   w_gate_up  [E][2I][H/2] bytes of packed E2M1 codes (element 2j in the low nibble of byte
 *              j, element 2j+1 in the high nibble), rows 0..I-1 = gate, I..2I-1 = up
 *   sf_gate_up [E][2I][H/32] UE8M0 bytes (scale 2^(b-127) of elements 32j..32j+31 of a row)
 *   w_down     [E][H][I/2] packed E2M1
 *   sf_down    [E][H][I/32] UE8M0
 * Weight pointers 16-byte aligned, scale pointers 4-byte aligned.  The forward then runs the
 * block-scaled UMMA with E2M1 weight operands; the activation scales (x_sf) must be powers of
 * two, and MOE_OPT_SCALE_MODE 0 makes moe_forward return MOE_ERR_BAD_SCALE.  A scale byte
 * 0xFF (NaN) makes this call return MOE_ERR_BAD_SCALE and leaves the weights unloaded.
 * Routed and shared weights must be loaded in one format: until they are, moe_forward
 * returns MOE_ERR_NO_WEIGHTS. */
int moe_load_weights_mxfp4(moe_handle_t h, const uint8_t *w_gate_up, const uint8_t *sf_gate_up,
                           const uint8_t *w_down, const uint8_t *sf_down, void *stream);

/* The n_shared shared experts' weights as MXFP4, layouts as moe_load_weights_mxfp4. */
int moe_load_shared_weights_mxfp4(moe_handle_t h, const uint8_t *w_gate_up, const uint8_t *sf_gate_up,
                                  const uint8_t *w_down, const uint8_t *sf_down, void *stream);

/* The layer on T tokens (0 <= T <= max_tokens, T % R == 0; source r owns tokens
 * [r*T/R, (r+1)*T/R)): Output(T) = sum_k w_k Expert_k(T) ("Dispatch/Combine: 博客理论 ↔
 * DeepEP 源码 ↔ DeepGEMM Mega MoE 三方对比分析" §1), by the fused call sequence of "DeepGEMM
 * Mega MoE 对称内存（Symmetric Memory）深度分析" §10.1.  Asynchronous on `stream`.
 *   x        [T][H] e4m3            x_sf [T][H/128] fp32 (1x128 activation scales)
 *   topk_idx [T][topk] int64, -1 = skip this slot
 *   topk_w   [T][topk] fp32 gate weights
 *   out      [T][H] bf16 bits, fully written (a token with no valid slot gets 0). */
int moe_forward(moe_handle_t h, int T, const uint8_t *x, const float *x_sf,
                const int64_t *topk_idx, const float *topk_w, uint16_t *out, void *stream);

/* moe_forward from HOST buffers (same shapes as above), all on `stream`, returning after
 * the stream has finished.  Inputs in pinned (page-locked, device-mapped) memory with
 * 16-byte aligned addresses are read in place by one staging kernel into the handle's
 * device staging buffers; others are copied there by cudaMemcpyAsync.  A pinned, 16-byte
 * aligned `host_out` is written in place by the kernel that completes the combine (with
 * power-of-two scales or MXFP4 weights the FFN kernel itself in the default combine mode, see
 * MOE_OPT_COMBINE_MODE); otherwise the result is
 * copied back from a staging buffer.  Pageable buffers work but are slower. */
int moe_forward_host(moe_handle_t h, int T, const uint8_t *host_x, const float *host_x_sf,
                     const int64_t *host_topk_idx, const float *host_topk_w,
                     uint16_t *host_out, void *stream);

/* As moe_forward_host, but returns once the work is enqueued: the host buffers must stay
 * valid and unchanged, and `host_out` is complete, once `stream` has been synchronized
 * (moe_get_error synchronizes it too).  Forwards enqueued on one stream run in order, so a
 * caller may enqueue the next batch before the previous one has finished. */
int moe_forward_host_async(moe_handle_t h, int T, const uint8_t *host_x, const float *host_x_sf,
                           const int64_t *host_topk_idx, const float *host_topk_w,
                           uint16_t *host_out, void *stream);

/* Wait for the handle's last stream, then return (and clear) the sticky device status in
 * *device_status (a moe_status value; MOE_OK if none).  The pages' kernel stops with an
 * assertion when a bounded wait runs out ("DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度
 * 分析" §6.2); here the kernels record the failure and this call reports it.  Clearing also resets the
 * workspace counters so the next forward starts clean. */
int moe_get_error(moe_handle_t h, int *device_status);

/* Routing results of the last forward (host copies, after syncing its stream), i.e. the
 * per-expert counts, expert segments and pool metadata of "Mega-MoE walkthrough part 2"
 * (kwkr.cn/news/1317662) §2.4-2.6:
 *   counts [E] rows per expert, recv [E][R] rows per (expert, source),
 *   block_offset [E+1] first M-block of each expert in the pool (last = total blocks),
 *   meta [P][3] {source, token, topk slot} of every pool row (rows past an expert's
 *   count hold padding), *P = pool rows used = block_offset[E] * block_m,
 *   *block_m = rows per M-block.  Any output pointer may be NULL.  meta needs room for
 *   the pool rows of the last forward: (ceil(T*topk/block_m) + E) * block_m rows. */
int moe_debug_routing(moe_handle_t h, uint32_t *counts, uint32_t *recv, int32_t *block_offset,
                      uint32_t *meta, int *P, int *block_m);

/* Per-expert routed rows accumulated over every forward since the handle was created
 * (host copy, [E]). */
int moe_cumulative_expert_rows(moe_handle_t h, uint64_t *rows);

/* Host copy of an intermediate buffer of the last forward (for stage-by-stage tests):
 *   MOE_BUF_POOL_X   [P][H] e4m3 gathered rows      MOE_BUF_POOL_SF [H/128][P] fp32
 *   MOE_BUF_ACT      [P][I] e4m3 SwiGLU output      MOE_BUF_ACT_SF  [I/128][P] fp32
 *   MOE_BUF_COMBINE  [topk][T][H] bf16 weighted expert outputs
 *   MOE_BUF_TABLE    [E][R][max_tokens/R] int32 index table (token_in_source*topk + k)
 * where P is the reserved pool row capacity (moe_info).  `bytes` must equal the
 * buffer's size; returns MOE_ERR_INVALID_ARG otherwise. */
enum moe_buffer {
    MOE_BUF_POOL_X = 0, MOE_BUF_POOL_SF = 1, MOE_BUF_ACT = 2, MOE_BUF_ACT_SF = 3,
    MOE_BUF_COMBINE = 4, MOE_BUF_TABLE = 5
};
int moe_debug_buffer(moe_handle_t h, int which, void *host_dst, uint64_t bytes);

/* Sizes and launch shape of the handle. */
typedef struct moe_info {
    int E, H, I, topk, R;
    int max_tokens;       /* reserved tokens per forward                     */
    int pool_rows;        /* reserved pool row capacity P                    */
    int block_m;          /* rows per M-block (GEMM tile rows)               */
    int block_n;          /* GEMM tile columns                               */
    int num_sms;          /* persistent grid size                            */
    uint64_t workspace_bytes;
    uint64_t weight_bytes;
    int n_shared;         /* shared experts; E and topk above include them: shared expert s
                             is expert slot E - n_shared + s and combine plane
                             topk - n_shared + s (the debug buffers use these sizes) */
    int weight_format;    /* moe_weight_format of the routed weights last loaded          */
} moe_info;
int moe_get_info(moe_handle_t h, moe_info *info);

/* Options.  MOE_OPT_TIMEOUT_NS: time limit of every device-side wait (default 2e9 ns);
 * MOE_OPT_DEBUG_SKIP_BARRIER: when 1, one CTA of the routing kernel skips its arrival
 * at the grid barrier, so the others give up after the time limit and the forward
 * ends with MOE_ERR_TIMEOUT (failure-path test; never on in normal use);
 * MOE_OPT_FFN_MODE: how the expert FFN kernel covers its tiles: 0 = automatic (default) and
 * 1 = one CTA per 128-row tile, which are the same kernel; other values are refused;
 * MOE_OPT_SCALE_MODE: 0 = arbitrary fp32 block scales (the UMMA accumulates each 128-deep
 * K block in TMEM and the scales are applied on the CUDA cores); 1 = every scale (x_sf, both
 * weight scale tensors) is a power of two: the UMMA applies them itself as UE8M0 scale
 * factors and accumulates the whole K range in TMEM ("DeepGEMM Mega MoE 对称内存
 * （Symmetric Memory）深度分析" §8.1), and the SwiGLU requant uses the smallest power-of-two
 * scale >= max(amax, 1e-4)/448; 2 = automatic (default): mode 1 when every scale of the
 * loaded weights is a power of two (checked by moe_load_weights), else mode 0.  In mode 1
 * weights that are not all powers of two make moe_forward return MOE_ERR_BAD_SCALE; in
 * modes 1 and 2 an activation scale that is not, on the block-scaled path, is reported by
 * the device the same way (sticky);
 * MOE_OPT_COMBINE_MODE: where the top-k combine runs ("DeepGEMM Mega MoE 对称内存（Symmetric
 * Memory）深度分析" §9: the per-token fp32 reduce of the top-k expert outputs).  0 = a
 * separate kernel after the expert FFN kernel; 1 = inside the expert FFN kernel: a down tile's
 * scattered rows are counted per (token, 256-column n-tile), and the epilogue warps reduce every
 * (token, n-tile) whose routed rows are all scattered while other tiles are still being
 * computed (the forward is then two kernels, three with shared experts); 2 = automatic
 * (default): 1 when a host-buffer entry point writes the output into pinned host memory in
 * place and the block-scaled FFN kernel runs (power-of-two scales or MXFP4 weights: its rows
 * then cross to the host while the GEMMs still run), else 0 (with arbitrary fp32 scales the
 * reduce would lengthen the FFN kernel's critical epilogue more than it saves).  All modes
 * give the same output bits.  Other values are refused. */
enum moe_option {
    MOE_OPT_TIMEOUT_NS = 0,
    MOE_OPT_DEBUG_SKIP_BARRIER = 1,
    MOE_OPT_FFN_MODE = 2,
    MOE_OPT_SCALE_MODE = 3,
    MOE_OPT_COMBINE_MODE = 4
};
int moe_set_option(moe_handle_t h, int option, int64_t value);

/* Stage timing with CUDA events recorded on the forward's own stream.  enable = N > 0:
 * the 1st, (N+1)-th, (2N+1)-th ... moe_forward from now records an event before and after
 * each of its three kernels (dispatch; expert FFN = gate_up GEMM + SwiGLU + down GEMM +
 * weighted scatter; combine) — N > 1 samples the forwards, so the events (which serialise
 * the kernels they sit between) disturb only one step in N; enable = 0 stops.  With the
 * combine inside the FFN kernel the combine stage brackets no kernel (its time is ~0 and the
 * FFN stage includes the reduce).
 * moe_profile_read waits for the last stream, returns the summed milliseconds of each
 * stage over the recorded forwards in stage_ms[3] and their number in *calls, and starts
 * a new window.  At most 8192 forwards are recorded per window (later ones are counted in
 * *dropped, not timed). */
int moe_profile_enable(moe_handle_t h, int enable);
int moe_profile_read(moe_handle_t h, double *stage_ms, int *calls, int *dropped);

/* Routing without any device allocation, for callers that may not allocate GPU memory
 * themselves or through this library (code running under another framework's memory
 * pool or a fixed memory budget, real-time loops that must stay out of the allocator,
 * plug-ins whose host owns every allocation).  The pages have no counterpart: it is a
 * deployment convenience, not a step of the method.  It needs no handle and no weights.
 * It computes what moe_debug_routing reports after a forward: counts [E], recv [E][R],
 * block_offset [E+1] (M-blocks of 128 rows) and, for every received row, its pool row's
 * {source, token, topk slot} in meta [(ceil(T*topk/128) + E) * 128][3] (padding rows are
 * left untouched), plus *status (device int32: MOE_OK, MOE_ERR_BAD_INDEX or
 * MOE_ERR_SLOT_OVERFLOW; on an error the other outputs are left untouched).  All pointers
 * are device pointers owned by the caller; topk_idx is [T][topk] int64 with -1 = skip.
 * Scratch (slot counters and the index table) lives in one fixed array of about 4 MB per
 * GPU, kept until the process exits; sizes beyond it return MOE_ERR_CAPACITY: at most
 * E*R <= 4096, T*topk <= 131072 and E*T <= 1048576 (plus the moe_create limits on E, topk
 * and R, and T % R == 0).  The first call on a device looks up that array's device
 * address and should come before any stream capture; the address is kept until the process
 * exits, so the entry point must not be used on a device after that device was reset
 * (cudaDeviceReset).  Asynchronous on `stream`, which must belong to the current device
 * (MOE_ERR_INVALID_ARG otherwise); calls that overlap on the GPU share the scratch and race. */
int moe_route_noalloc(int T, int E, int topk, int R, const int64_t *topk_idx, uint32_t *counts,
                      uint32_t *recv, int32_t *block_offset, uint32_t *meta, int32_t *status,
                      void *stream);

/* Release every device buffer of the handle (after syncing its last stream): the teardown
 * of the buffers the layer object of "DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析"
 * §10.1 allocates. */
int moe_destroy(moe_handle_t h);

/* Static description of a status code. */
const char *moe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* CPW_MOE_H */
