// routing.cu -- the data-movement kernels of the fused MoE layer:
//   dispatch_kernel : route + count, packed 64-bit slot claim, [expert][source][slot] index
//                     table, grid barrier, expert segments, round-robin gather of token rows
//                     into the expert-major FP8 pool (one cooperative persistent launch);
//   combine_kernel  : top-k reduce of the weighted expert outputs into token order, then
//                     the workspace reset for the next forward;
//   relayout_weights_kernel: load-time weight re-layout into contiguous GEMM tiles, with the
//                     gate/up row interleave of the gate_up weights.
//
// The routing steps themselves (count, claim, table, grid barrier, segments, round-robin
// gather) are device functions in route_device.cuh, with their source pages.  The combine
// follows "DeepGEMM Mega
// MoE 对称内存（Symmetric Memory）深度分析" §9.2 (per-token top-k reduce in fp32 over the valid
// slots).
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "route_device.cuh"
#include "topk_combine.cuh"

namespace cpw {

// Dynamic shared memory of the routing kernel: cnt [R*E] u32 | recv [E*R] u32 | cum [E+1] |
// blk [E+1] | flag, then (16-byte aligned) the gather warps' barriers [gwarps][2] and
// (128-byte aligned) their row buffers [gwarps][2][H]: up to 192 KB of rows in flight per SM.
struct DispatchSmem {
    size_t bars, bufs, total;
    int gwarps;   // warps of a CTA that gather
};
__host__ __device__ inline DispatchSmem dispatch_smem(const Dims &d, int threads)
{
    constexpr size_t SMEM_MAX = 227 * 1024, STAGING = 192 * 1024;
    DispatchSmem L;
    const size_t base = sizeof(uint32_t) * (2 * static_cast<size_t>(d.R) * d.E) +
                        sizeof(int32_t) * 2 * (static_cast<size_t>(d.E) + 1) + 16;
    L.bars = (base + 15) & ~static_cast<size_t>(15);
    const int maxw = threads / 32;
    const size_t used = L.bars + 16 * static_cast<size_t>(maxw) + 128;
    const size_t room = used < SMEM_MAX ? SMEM_MAX - used : 0;
    const size_t stg = room < STAGING ? room : STAGING;
    const size_t per_warp = 2 * static_cast<size_t>(d.H);
    L.gwarps = static_cast<int>(stg / per_warp) < maxw ? static_cast<int>(stg / per_warp) : maxw;
    L.bufs = (L.bars + 16 * static_cast<size_t>(L.gwarps) + 127) & ~static_cast<size_t>(127);
    L.total = L.bufs + per_warp * static_cast<size_t>(L.gwarps);
    return L;
}


__global__ void __launch_bounds__(DISPATCH_THREADS, 1)
    dispatch_kernel(const Dims d, const Workspace ws, const CallArgs c)
{
    extern __shared__ uint32_t smem_u[];
    const int E = d.E, R = d.R;
    uint32_t *cnt = smem_u;                                  // [R][E]
    uint32_t *recv_s = cnt + R * E;                          // [E][R]
    int32_t *cum = reinterpret_cast<int32_t *>(recv_s + E * R);
    int32_t *blk = cum + (E + 1);
    volatile int *s_ok = reinterpret_cast<volatile int *>(blk + (E + 1));
    const DispatchSmem L = dispatch_smem(d, blockDim.x);
    uint64_t *gbar = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(smem_u) + L.bars);
    uint8_t *gbuf = reinterpret_cast<uint8_t *>(smem_u) + L.bufs;
    if (threadIdx.x == 0) {   // the gather warps' row barriers (first used after the grid barrier)
        for (int i = 0; i < 2 * L.gwarps; ++i)
            ptx::mbar_init(&gbar[i], 1);
        ptx::fence_mbar_init();
    }

    // the expert FFN kernel may be scheduled at once: its CTAs run their prologue as this
    // kernel's CTAs leave and then wait for the whole grid
    ptx::launch_dependents();
    // A forward after an unreported device error does nothing (every CTA sees the same
    // sticky word: nothing writes it while this kernel runs).
    if (*reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_STICKY) != 0)
        return;
    const uint64_t deadline = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);

    // ---- count, packed claim, index table ------------------------------------------------
    route::count_claim_table(d, ws, c, cnt);
    // each token's routed slots (read by either combine), and with the in-kernel combine the
    // zero rows of unrouted tokens
    route::token_masks(d, ws, c);

    // ---- grid barrier: every claim and table entry is visible past this point -----------
    const bool skip = c.debug_skip_barrier != 0 && blockIdx.x == 0;
    if (!route::grid_barrier(ws.hdr + HDR_GRID_SYNC, ws.hdr, skip, deadline, s_ok))
        return;
    if (*reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_CALL) != 0)
        return;

    // ---- received counts, expert segments, M-block map -----------------------------------
    route::segments(d, ws, recv_s, cum, blk);

    // ---- gather, one warp per received row at a time (global order across experts) ------
    // (warps numbered CTA-minor, so a small batch's rows spread over every SM)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < L.gwarps)
        route::gather_rows(d, ws, c, cum, blk, recv_s, warp * gridDim.x + blockIdx.x, L.gwarps * gridDim.x,
                           gbar + 2 * warp, gbuf + static_cast<size_t>(warp) * 2 * d.H, deadline, lane);
}

cudaError_t launch_dispatch(const Dims &d, const Workspace &ws, const CallArgs &c, int num_sms,
                            cudaStream_t s)
{
    // the routing steps of a large batch want every warp an SM can hold; a small batch is bound
    // by the routing steps and the launch, which half the block does faster
    const long long rows = static_cast<long long>(c.T) * d.K;
    const int threads = rows >= 8LL * 1024 ? DISPATCH_THREADS : DISPATCH_THREADS / 2;
    const DispatchSmem L = dispatch_smem(d, threads);
    if (L.gwarps < 1)   // cannot happen for the shapes moe_create accepts (H <= 16384, R*E <= 16384)
        return cudaErrorInvalidConfiguration;
    const size_t smem = L.total;
    cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void *>(dispatch_kernel), static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    Dims dd = d;
    Workspace ww = ws;
    CallArgs cc = c;
    void *args[] = {&dd, &ww, &cc};
    return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(dispatch_kernel), dim3(num_sms), dim3(threads), args,
                                       smem, s);
}

// ------------------------------------------------------------------ combine -------------
// out[t] = bf16( sum over valid k, ascending, of combine[k][t] ) in fp32; no valid k -> 0.
// Then the workspace reset of the pages' cleanup step (reset_after_forward).  With the
// in-kernel combine (topk_combine.cuh) this kernel is not launched.
__global__ void __launch_bounds__(COMBINE_THREADS, 2)
    combine_kernel(const Dims d, const Workspace ws, const CallArgs c)
{
    // launched programmatically for small batches: the FFN kernel's results are complete and
    // visible past this point (a no-op for an ordinary launch)
    ptx::grid_dependency_wait();
    const int K = d.K, H = d.H;
    const uint32_t err = *reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_CALL) |
                         *reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_STICKY);
    if (err == 0) {
        // two 16-byte output vectors (8 bf16 each) per thread per round; every valid plane
        // load of both is issued before any of them is summed
        const int H8 = H / 8;
        const long long plane = static_cast<long long>(ws.max_tokens) * H8;   // uint4 per plane
        const uint4 *cb = reinterpret_cast<const uint4 *>(ws.combine);
        uint4 *out = reinterpret_cast<uint4 *>(c.out);
        const long long n = static_cast<long long>(c.T) * H8;
        const long long G = static_cast<long long>(gridDim.x) * blockDim.x;
        for (long long g0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g0 < n; g0 += 2 * G) {
            const long long g[2] = {g0, g0 + G};
            const bool live1 = g[1] < n;
            uint32_t mask[2] = {0u, 0u};
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                if (v == 1 && !live1)
                    break;
                mask[v] = __ldcg(ws.tok_mask + g[v] / H8);   // the routing kernel's slot mask
            }
            float acc[2][8];
#pragma unroll
            for (int v = 0; v < 2; ++v)
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    acc[v][q] = 0.0f;
            for (int k0 = 0; k0 < K; k0 += 8) {
                uint4 u[2][8];
#pragma unroll
                for (int v = 0; v < 2; ++v)
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if ((mask[v] >> (k0 + j)) & 1u)   // bits >= K are clear
                            u[v][j] = __ldcs(cb + (k0 + j) * plane + g[v]);
#pragma unroll
                for (int v = 0; v < 2; ++v)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (!((mask[v] >> (k0 + j)) & 1u))
                            continue;
                        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u[v][j]);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = __bfloat1622float2(b[q]);
                            acc[v][2 * q] += f.x;
                            acc[v][2 * q + 1] += f.y;
                        }
                    }
            }
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                if (v == 1 && !live1)
                    break;
                uint4 o;
                __nv_bfloat162 *ob = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    ob[q] = __floats2bfloat162_rn(acc[v][2 * q], acc[v][2 * q + 1]);
                out[g[v]] = o;
            }
        }
    }
    // reset for the next forward
    reset_after_forward(d, ws, blockIdx.x * blockDim.x + threadIdx.x, gridDim.x * blockDim.x);
}

cudaError_t launch_combine(const Dims &d, const Workspace &ws, const CallArgs &c, int num_sms,
                           cudaStream_t s)
{
    // two CTAs per SM (128 registers a thread keep 16 plane loads in flight), all resident.
    // A small batch (at most 4096 routed rows, the threshold at which "MOE融合算子",
    // vllm-ascend dispatch_ffn_combine §4, switches to its small-batch combine) is launched
    // programmatically, so the launch overlaps the FFN kernel's last
    // CTAs; a large one ordinarily (programmatic there measured 1.3% slower: its CTAs wait on the
    // SMs the FFN CTAs leave)
    if (static_cast<long long>(c.T) * d.K <= 4096)
        return launch_programmatic(combine_kernel, num_sms * 2, COMBINE_THREADS, 0, s, d, ws, c);
    combine_kernel<<<num_sms * 2, COMBINE_THREADS, 0, s>>>(d, ws, c);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ shared experts -----
// Every token also goes through each shared expert, whose output enters the top-k sum
// unweighted, in a combine plane of its own after the routed slots ("DeepGEMM Mega MoE 对称内存
// （Symmetric Memory）深度分析" §8.2: num_topk + 1 planes when shared experts exist).  Here a
// shared expert is an expert slot after the routed ones that every token's route names in
// slot K + s with weight 1, so routing, the grouped GEMMs and the combine need nothing else.
__global__ void extend_route_kernel(const int64_t *__restrict__ idx, const float *__restrict__ w,
                                    int64_t *__restrict__ idx_ext, float *__restrict__ w_ext, int T, int K, int S,
                                    int E_routed)
{
    const int KS = K + S;
    const long long n = static_cast<long long>(T) * KS;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long t = i / KS;
        const int k = static_cast<int>(i - t * KS);
        if (k < K) {
            idx_ext[i] = idx[t * K + k];
            w_ext[i] = w[t * K + k];
        } else {
            idx_ext[i] = E_routed + (k - K);
            w_ext[i] = 1.0f;
        }
    }
}

cudaError_t launch_extend_route(const int64_t *idx, const float *w, int64_t *idx_ext, float *w_ext, int T, int K,
                                int S, int E_routed, int num_sms, cudaStream_t s)
{
    extend_route_kernel<<<num_sms, 256, 0, s>>>(idx, w, idx_ext, w_ext, T, K, S, E_routed);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ host inputs --------
// Copies of the host-buffer entry point's inputs, read straight from pinned (device-mapped)
// host memory in one launch instead of one copy-engine transfer per buffer.  Every pointer
// is 16-byte aligned; a tail of fewer than 16 bytes is copied byte by byte.
struct StageCopy {
    const uint8_t *src;
    uint8_t *dst;
    long long bytes;
};
struct StageArgs {
    StageCopy cp[4];
};

__global__ void __launch_bounds__(256) stage_inputs_kernel(const StageArgs a)
{
    const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long gthreads = static_cast<long long>(gridDim.x) * blockDim.x;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const StageCopy c = a.cp[i];
        const long long n16 = c.bytes / 16;
        const uint4 *s = reinterpret_cast<const uint4 *>(c.src);
        uint4 *d = reinterpret_cast<uint4 *>(c.dst);
        for (long long q = gtid; q < n16; q += gthreads)
            d[q] = s[q];
        for (long long b = n16 * 16 + gtid; b < c.bytes; b += gthreads)
            c.dst[b] = c.src[b];
    }
}

cudaError_t launch_stage_inputs(const void *const src[4], void *const dst[4], const long long bytes[4], int num_sms,
                                cudaStream_t s)
{
    StageArgs a;
    for (int i = 0; i < 4; ++i)
        a.cp[i] = StageCopy{static_cast<const uint8_t *>(src[i]), static_cast<uint8_t *>(dst[i]), bytes[i]};
    stage_inputs_kernel<<<num_sms * 2, 256, 0, s>>>(a);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ weights -------------
// Load-time weight re-layout into GEMM tiles.  A weight row of K elements is K/128 blocks of
// kb_bytes bytes (128 for e4m3; 64 for packed 4-bit E2M1, two elements per byte).  dst =
// [E][N/256][K/128][256][kb_bytes] bytes: every 256-row tile the FFN kernel loads per 128-deep
// K block is one contiguous block (32 KB / 16 KB), so each weight load streams whole DRAM
// pages instead of 256 rows several KB apart.
// N need not be a multiple of 256: the last tile's rows past N are written as zeros (the
// down weight with H an odd multiple of 128).
// With gate_up_I > 0 (the gate_up weight, N = 2I) the rows are also gate/up interleaved:
// within each group of 16 rows, rows 0..7 are gate rows 8j..8j+7 and rows 8..15 are up rows
// I+8j..I+8j+7 (granularity 8, the layout of "DeepGEMM Mega MoE 对称内存（Symmetric Memory）
// 深度分析" §10.2), so one 256-row tile holds 128 gate rows and the 128 matching up rows.
__global__ void relayout_weights_kernel(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int E,
                                        int N, int K, int gate_up_I, int kb_bytes)
{
    const int KB = K / 128, NT = (N + BN - 1) / BN, C16 = kb_bytes / 16;
    const long long row_bytes = static_cast<long long>(KB) * kb_bytes;
    const long long chunks = static_cast<long long>(E) * NT * BN * KB * C16;
    for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < chunks;
         q += static_cast<long long>(gridDim.x) * blockDim.x) {
        long long t = q;
        const int c16 = static_cast<int>(t % C16);
        t /= C16;
        const int r = static_cast<int>(t % BN);
        t /= BN;
        const int kb = static_cast<int>(t % KB);
        t /= KB;
        const int nt = static_cast<int>(t % NT);
        const long long e = t / NT;
        const int n = nt * BN + r;
        if (n >= N) {
            reinterpret_cast<uint4 *>(dst)[q] = make_uint4(0u, 0u, 0u, 0u);
            continue;
        }
        int srow = n;
        if (gate_up_I > 0) {
            const int j = n / 16, i = n % 16;
            srow = i < 8 ? 8 * j + i : gate_up_I + 8 * j + (i - 8);
        }
        const uint4 *sp = reinterpret_cast<const uint4 *>(src + (e * N + srow) * row_bytes + kb * kb_bytes + c16 * 16);
        reinterpret_cast<uint4 *>(dst)[q] = *sp;
    }
}

cudaError_t launch_relayout_weights(const uint8_t *src, uint8_t *dst, int E, int N, int K, int gate_up_I,
                                    int kb_bytes, cudaStream_t s)
{
    if (kb_bytes != 128 && kb_bytes != 64)
        return cudaErrorInvalidValue;
    relayout_weights_kernel<<<2048, 256, 0, s>>>(src, dst, E, N, K, gate_up_I, kb_bytes);
    return cudaGetLastError();
}

}  // namespace cpw
