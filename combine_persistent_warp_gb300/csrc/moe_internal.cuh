// moe_internal.cuh -- workspace layout, kernel argument blocks and launchers shared by
// the translation units of the CUDA library (not part of the public C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace cpw {

#ifndef CPW_BKS
#define CPW_BKS 128
#endif

constexpr int BM = 128;            // pool rows per M-block = UMMA M = TMEM lanes
constexpr int BN = 256;            // GEMM tile columns (UMMA N)
constexpr int BK = 128;            // K of one fp32 scale block = one TMEM partial
constexpr int BKS = CPW_BKS;       // K (bytes of an FP8 operand row) per pipeline stage
constexpr int SUBS = BK / BKS;     // pipeline stages per scale block
constexpr int STAGES = 4 * BK / BKS;   // TMA -> UMMA ring depth (192 KB of operand tiles)
constexpr int MAX_KB = 128;        // 128-deep K blocks of H and of I at most (H, I <= 16384)
constexpr int GEMM_THREADS = 384;  // 4 producer/issuer warps + 2 epilogue warpgroups
constexpr int DISPATCH_THREADS = 1024;
constexpr int COMBINE_THREADS = 256;
static_assert(BKS == 32 || BKS == 64 || BKS == 128, "stage depth must match a swizzle width");

constexpr int STAGE_A_BYTES = BM * BKS;                // 16 KB at BKS = 128
constexpr int STAGE_B_BYTES = BN * BKS;                // 32 KB at BKS = 128
constexpr int STAGE_BYTES = STAGE_A_BYTES + STAGE_B_BYTES;

// 32-bit words of the workspace header; hot words sit on separate 128-byte lines.
enum HdrWord : int {
    HDR_GRID_SYNC = 0,     // XOR-tag grid barrier counter of the routing kernel
    HDR_ERR_CALL = 32,     // first device error of the forward in flight
    HDR_ERR_STICKY = 64,   // errors of finished forwards, until moe_get_error
    HDR_TILE_NEXT = 96,    // next tile of the FFN kernel's dynamic tile list
    HDR_FFN_EXIT = 128,    // FFN CTAs finished (in-kernel combine: the last one resets)
    HDR_WORDS = 160
};

// Device workspace of one handle.  Sizes: P = pool row capacity, MB = P / BM.
struct Workspace {
    uint32_t *hdr;                 // [HDR_WORDS]
    unsigned long long *send;      // [R][E] packed (arrivals << 32 | rows)
    uint32_t *counts;              // [E] rows per expert (last forward)
    uint32_t *recv;                // [E][R] rows per (expert, source)
    int32_t *blk_off;              // [E+1] first M-block of each expert
    int32_t *block_expert;         // [MB] expert of each M-block
    int32_t *block_rows;           // [MB] valid rows of each M-block
    unsigned long long *cum_rows;  // [E] rows per expert over all forwards
    int32_t *table;                // [E][R][tsrc_cap] token_in_source * topk + k
    uint8_t *pool_x;               // [P][H]   e4m3 gathered activations
    float *pool_sf;                // [H/128][P]
    uint8_t *pool_sfe;             // [P/128][H/128][512] UE8M0 scale blocks (block-scaled mode)
    uint32_t *meta;                // [P][3]   {source, token, topk slot}
    uint8_t *act;                  // [P][I]   e4m3 SwiGLU output
    float *act_sf;                 // [I/128][P]
    uint8_t *act_sfe;              // [P/128][I/128][512] UE8M0 scale blocks (block-scaled mode)
    uint16_t *combine;             // [topk][max_tokens][H] bf16 weighted expert outputs
    uint32_t *arrive;              // [MB] rows gathered per M-block
    uint32_t *l1_done;             // [MB] finished gate_up (tile, epilogue warp) pairs
    uint32_t *tok_mask;            // [max_tokens] routed top-k slots of each token (bit k)
    uint32_t *tok_cnt;             // [max_tokens][ceil(H/256)] scattered rows per (token, n-tile)
    int tsrc_cap;                  // max_tokens / R
    int P;                         // pool rows
    int max_blocks;                // P / BM
    int max_tokens;
};

struct Dims {
    int E, H, I, K, R;   // K = topk
};

struct CallArgs {
    int T;
    const uint8_t *x;
    const float *x_sf;
    const int64_t *idx;
    const float *w;
    uint16_t *out;
    long long timeout_ns;
    int debug_skip_barrier;
    int block_scaled;   // 1: power-of-two scales, hardware block-scaled UMMA (ffn_bs.cu)
    int fused_combine;  // 1: the top-k combine runs inside the FFN kernel (topk_combine.cuh)
};

// Device error codes (same values as the public moe_status).
enum DevErr : uint32_t { DEV_BAD_INDEX = 6, DEV_TIMEOUT = 7, DEV_SLOT_OVERFLOW = 8, DEV_BAD_SCALE = 10 };

__device__ __forceinline__ void record_error(uint32_t *hdr, uint32_t code)
{
    atomicCAS(hdr + HDR_ERR_CALL, 0u, code);
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) holds per device: raises a kernel's limit
// to `bytes` on the current device unless a call for that (kernel, device) already has
// (thread-safe; defined in api.cu).
cudaError_t ensure_max_dynamic_smem(const void *kernel, int bytes);

// Launch with programmatic stream serialization: the kernel may start while the previous
// kernel of the stream still runs, and must call ptx::grid_dependency_wait() before it reads
// anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*kern)(KArgs...), int grid, int block, int smem, cudaStream_t s, Args... args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Launchers (one per translation unit).
cudaError_t launch_dispatch(const Dims &d, const Workspace &ws, const CallArgs &c, int num_sms,
                            cudaStream_t s);
constexpr int A_ROWS_PART = 32;   // row granularity of partial A-tile loads
struct FfnMaps {
    CUtensorMap a1, b1, a2, b2;   // pool x / W1 tiles (gate_up), act / W2 tiles (down)
    CUtensorMap a1p, a2p;         // pool x / act with 32-row boxes (partly filled M-blocks)
    CUtensorMap a1h, a2h;         // pool x / act with 64-row boxes (block-scaled kernel)
};
// the fp32-scale FFN kernel (ffn.cu): one CTA per SM, tiles claimed in list order
cudaError_t launch_ffn(const FfnMaps &maps, const Dims &d, const Workspace &ws, const CallArgs &c,
                       const float *sf1, const float *sf2, int wave_blocks, int num_sms, cudaStream_t s);
#ifdef CPW_TRACE
cudaError_t trace_read(void *dst, size_t bytes);
cudaError_t trace_clear();
#endif
// power-of-two scales: the block-scaled FFN kernel (ffn_bs.cu) and the load-time UE8M0
// scale blocks of the weight tiles; fp4: MXFP4 weight tiles (packed E2M1, maps of the
// 16U4_ALIGN16B type) with per-K-block scale blocks
cudaError_t launch_ffn_bs(const FfnMaps &maps, const Dims &d, const Workspace &ws, const CallArgs &c,
                          const uint8_t *sfb1, const uint8_t *sfb2, int wave_blocks, int num_sms, bool fp4,
                          cudaStream_t s);
cudaError_t launch_build_sfb(const float *s, uint8_t *dst, int E, int N, int K, int gate_up_I, uint32_t *bad,
                             cudaStream_t st);
cudaError_t launch_build_sfb4(const uint8_t *s, uint8_t *dst, int E, int N, int K, int gate_up_I, uint32_t *bad,
                              cudaStream_t st);
cudaError_t launch_combine(const Dims &d, const Workspace &ws, const CallArgs &c, int num_sms,
                           cudaStream_t s);
// shared experts: idx_ext / w_ext [T][K + S] = the caller's [T][K] route plus slots K + s naming
// expert E_routed + s with weight 1
cudaError_t launch_extend_route(const int64_t *idx, const float *w, int64_t *idx_ext, float *w_ext, int T, int K,
                                int S, int E_routed, int num_sms, cudaStream_t s);
cudaError_t launch_stage_inputs(const void *const src[4], void *const dst[4], const long long bytes[4], int num_sms,
                                cudaStream_t s);
// kb_bytes: bytes of a 128-element K block of a weight row (128 e4m3, 64 packed E2M1)
cudaError_t launch_relayout_weights(const uint8_t *src, uint8_t *dst, int E, int N, int K, int gate_up_I,
                                    int kb_bytes, cudaStream_t s);

}  // namespace cpw
