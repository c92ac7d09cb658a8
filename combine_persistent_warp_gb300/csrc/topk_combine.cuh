// topk_combine.cuh -- the top-k combine run inside the expert FFN kernels, and the workspace
// reset that ends a forward (shared by the combine kernel and the FFN kernels).
//
// The combine reduces each token's top-k weighted expert outputs, one bf16 plane per top-k
// slot ("DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析" §8.2), in fp32 over the valid
// slots (same page §9.2).  The pages run that reduce in the epilogue warps of the persistent
// kernel itself, after every rank's scatter is complete (same page §9.1; "MOE融合算子",
// DeepGEMM MegaMoE §4: scatter, then the reduce behind one cross-GPU barrier).  On one GPU
// nothing has to wait for the whole scatter: a token's reduce needs only its own top-k rows.
// So, with the in-kernel combine on,
//   * one warp of every FFN CTA (the counting warp) counts every down tile the CTA's epilogue
//     warps have stored, per (token, n-tile): it adds 1 for each valid row of the tile to the
//     counter of (the row's token, the tile's n-tile); the add that brings a counter to the
//     token's number of routed slots finds that token's columns of the n-tile complete and
//     lists the pair in the tile's ring slot;
//   * the CTA's epilogue warps reduce the listed pairs at the end of their next tile, each
//     pair's 256 columns by one warp (8 columns a lane, fp32 over the valid slots in
//     ascending order, then bf16 into the output row): the same arithmetic, in the same
//     order, as the separate combine kernel, so the two give identical bits.
// Tokens without any routed slot (all top-k ids -1) get their zero output row from the
// routing kernel.  The last FFN CTA to finish resets the workspace for the next forward.
#pragma once

#include <cuda_bf16.h>

#include "moe_internal.cuh"

namespace cpw {
namespace topk {

// Per tile-ring slot: the (token, slot mask) pairs a down tile completed, its n-tile and their
// number, and the barrier (one arrival per tile) that hands them to the epilogue warps.
template <int RING>
struct Lists {
    uint64_t ready[RING];
    int n[RING];
    int nt[RING];
    uint32_t tok[RING][BM];
    uint32_t mask[RING][BM];
};

// Warp-collective, by the counting warp once it has seen (through a CTA barrier) that every
// epilogue warp of its CTA has stored down tile (row0 = first pool row of the M-block, `rows`
// valid rows, n-tile nt): counts the tile's rows and writes the pairs it completed into tok[] /
// mask[]; returns their number (the same in every lane).
__device__ __forceinline__ int count_rows(const Dims &d, const Workspace &ws, long long row0, int rows, int nt,
                                          uint32_t *tok, uint32_t *mask, int lane)
{
    constexpr int RPL = BM / 32;
    const int NB = (d.H + BN - 1) / BN;
    uint32_t t[RPL], m[RPL];
#pragma unroll
    for (int j = 0; j < RPL; ++j)
        t[j] = lane + 32 * j < rows ? __ldg(ws.meta + (row0 + lane + 32 * j) * 3 + 1) : 0u;
#pragma unroll
    for (int j = 0; j < RPL; ++j)
        m[j] = lane + 32 * j < rows ? __ldg(ws.tok_mask + t[j]) : 0u;
    // release: the tile's stores, ordered before this point by the CTA barrier, are ordered
    // before the counts (the fence is cumulative)
    __threadfence();
    bool done[RPL];
#pragma unroll
    for (int j = 0; j < RPL; ++j) {
        done[j] = false;
        if (lane + 32 * j < rows) {
            uint32_t *cnt = ws.tok_cnt + static_cast<long long>(t[j]) * NB + nt;
            done[j] = atomicAdd(cnt, 1u) + 1u == static_cast<uint32_t>(__popc(m[j]));
            if (done[j])
                *cnt = 0u;   // every row of this (token, n-tile) has been counted
        }
    }
    // acquire: the other CTAs' stores these counts have seen are ordered before the reduce's
    // loads, which come after this warp's barrier arrival
    __threadfence();
    int n = 0;
#pragma unroll
    for (int j = 0; j < RPL; ++j) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, done[j]);
        if (done[j]) {
            const int at = n + __popc(b & ((1u << lane) - 1u));
            tok[at] = t[j];
            mask[at] = m[j];
        }
        n += __popc(b);
    }
    return n;
}

// Warp-collective: reduce pairs first, first + step, ... of a list (n-tile nt).  Lane l covers
// columns nt*256 + 8l .. +7 of the output row (nothing past H), with the loads of a pair's
// valid slots in flight eight at a time.
__device__ __forceinline__ void reduce(const Dims &d, const Workspace &ws, const CallArgs &c, const uint32_t *tok,
                                       const uint32_t *mask, int n, int nt, int first, int step, int lane)
{
    const int K = d.K, H = d.H;
    const int col = nt * BN + lane * 8;
    if (col >= H)
        return;
    const long long plane = static_cast<long long>(ws.max_tokens) * H;
    for (int i = first; i < n; i += step) {
        const uint32_t t = tok[i];
        const uint64_t m = mask[i];   // bits >= K are clear
        const uint16_t *p = ws.combine + static_cast<long long>(t) * H + col;
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            acc[q] = 0.0f;
        for (int k0 = 0; k0 < K; k0 += 8) {
            uint4 u[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if ((m >> (k0 + j)) & 1u)
                    u[j] = __ldcg(reinterpret_cast<const uint4 *>(p + (k0 + j) * plane));
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (!((m >> (k0 + j)) & 1u))
                    continue;
                const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u[j]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = __bfloat1622float2(b[q]);
                    acc[2 * q] += f.x;
                    acc[2 * q + 1] += f.y;
                }
            }
        }
        uint4 o;
        __nv_bfloat162 *ob = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            ob[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
        *reinterpret_cast<uint4 *>(c.out + static_cast<long long>(t) * H + col) = o;
    }
}

}  // namespace topk

// The reset of the pages' cleanup step, by threads tid, tid + nthreads, ... of whatever runs
// last in a forward: send counts, arrival and gate_up completion counters back to zero, the
// tile counter rewound; a device error of this forward moves into the sticky word and the
// grid barrier counter is cleared (an aborted barrier leaves it mid-phase).
__device__ __forceinline__ void reset_after_forward(const Dims &d, const Workspace &ws, int tid, int nthreads)
{
    for (int i = tid; i < d.R * d.E; i += nthreads)
        ws.send[i] = 0ull;
    for (int i = tid; i < ws.max_blocks; i += nthreads) {
        ws.arrive[i] = 0u;
        ws.l1_done[i] = 0u;
    }
    if (tid == 0) {
        ws.hdr[HDR_TILE_NEXT] = 0u;
        const uint32_t call = *reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_CALL);
        if (call != 0) {
            if (ws.hdr[HDR_ERR_STICKY] == 0)
                ws.hdr[HDR_ERR_STICKY] = call;
            ws.hdr[HDR_GRID_SYNC] = 0u;
            ws.hdr[HDR_ERR_CALL] = 0u;
        }
    }
}

// The last step of every thread of an FFN CTA when the combine runs inside the FFN kernel:
// the CTA that finishes last (every other CTA has made its last access to the workspace)
// resets it.  `flag` is a shared-memory word of the CTA.
__device__ __forceinline__ void ffn_cta_exit(const Dims &d, const Workspace &ws, int *flag)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t done = atomicAdd(ws.hdr + HDR_FFN_EXIT, 1u) + 1u;
        const bool last = done == gridDim.x;
        if (last)
            __threadfence();
        *flag = last ? 1 : 0;
    }
    __syncthreads();
    if (*flag) {
        reset_after_forward(d, ws, threadIdx.x, blockDim.x);
        if (threadIdx.x == 0)
            ws.hdr[HDR_FFN_EXIT] = 0u;
    }
}

}  // namespace cpw
