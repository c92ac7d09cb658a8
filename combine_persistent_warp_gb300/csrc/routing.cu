// routing.cu -- the data-movement kernels of the fused MoE layer:
//   dispatch_kernel : route + count, packed 64-bit slot claim, [expert][source][slot] index
//                     table, grid barrier, expert segments, round-robin gather of token rows
//                     into the expert-major FP8 pool (one cooperative persistent launch);
//   combine_kernel  : top-k reduce of the weighted expert outputs into token order, then
//                     the workspace reset for the next forward;
//   relayout_weights_kernel: load-time weight re-layout into contiguous GEMM tiles, with the
//                     gate/up row interleave of the gate_up weights.
//
// Source pages, by title and section:
//   "Mega-MoE 内核代码导读：从 Dispatch 到 WGMMA 的融合流水线" §4.1 (token x top-k scan),
//     §4.2 (per-expert count with block atomics, packed (1<<32)|count global claim),
//     §4.3 (index table [local_expert][source][slot] = token*topk + k), §4.4 (grid sync)
//   Mega-MoE walkthrough part 2 (kwkr.cn/news/1317662) §2.4 (expert segments, pool block
//     offsets by ceil_div), §2.5 (round-robin source choice by min-peeling), §2.6 (row copy,
//     scale copy, {source, token, topk} metadata, per-M-block arrival count)
//   "DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析" §6.2 (XOR-tag grid barrier with a
//     time limit), §9.2 (per-token top-k reduce in fp32 over the valid slots)
//
// On one GPU the pages' ranks become R logical source partitions of the token batch:
// source r owns tokens [r*T/R, (r+1)*T/R).  A "remote" store is a plain global store.
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace cpw {

namespace {

// XOR-tag grid barrier: CTA 0 adds 0x80000000 - (n-1), every other CTA adds 1, so bit 31
// of the counter flips exactly when all n CTAs have arrived.  Bounded: on the deadline the
// CTA records DEV_TIMEOUT and returns false.  `skip_arrive` is the failure-path test hook.
__device__ bool grid_barrier(uint32_t *counter, uint32_t *hdr, bool skip_arrive,
                             uint64_t deadline, volatile int *s_ok)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const uint32_t add = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1) : 1u;
        __threadfence();
        uint32_t old = skip_arrive ? ptx::ld_acquire_gpu(counter) : atomicAdd(counter, add);
        for (uint32_t i = 0;; ++i) {
            const uint32_t v = ptx::ld_acquire_gpu(counter);
            if ((v ^ old) & 0x80000000u)
                break;
            if ((i & 255u) == 255u && ptx::globaltimer() > deadline) {
                record_error(hdr, DEV_TIMEOUT);
                ok = 0;
                break;
            }
        }
        __threadfence();
        *s_ok = ok;
    }
    __syncthreads();
    return *s_ok != 0;
}

// Largest i in [0, n) with a[i] <= v (a non-decreasing, a[0] <= v).
__device__ __forceinline__ int last_le(const int32_t *a, int n, int32_t v)
{
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a[mid] <= v)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Round-robin by min-peeling: position p among one expert's received rows -> (source,
// slot).  Each round: A sources with rows left, L = their smallest remainder, A*L rows;
// position q of the round goes to the (q mod A)-th active source at slot offset + q / A.
__device__ __forceinline__ void round_robin(const uint32_t *recv, int R, uint32_t p,
                                            uint32_t &src, uint32_t &slot)
{
    uint32_t offset = 0, peeled = 0;   // rows every active source has used so far
    src = 0;
    slot = 0;
    for (int round = 0; round <= R; ++round) {
        uint32_t A = 0, L = 0xFFFFFFFFu;
        for (int r = 0; r < R; ++r) {
            const uint32_t rem = recv[r] > peeled ? recv[r] - peeled : 0u;
            if (rem > 0) {
                ++A;
                L = rem < L ? rem : L;
            }
        }
        if (A == 0)
            return;
        if (p < A * L) {
            const uint32_t which = p % A;
            uint32_t nth = 0;
            for (int r = 0; r < R; ++r) {
                if (recv[r] > peeled) {
                    if (nth == which) {
                        src = static_cast<uint32_t>(r);
                        break;
                    }
                    ++nth;
                }
            }
            slot = offset + p / A;
            return;
        }
        p -= A * L;
        offset += L;
        peeled += L;
    }
}

}  // namespace

// Dynamic shared memory: cnt [R*E] u32 | recv [E*R] u32 | cum [E+1] | blk [E+1] | flag
size_t dispatch_smem_bytes(const Dims &d)
{
    return sizeof(uint32_t) * (2 * static_cast<size_t>(d.R) * d.E) +
           sizeof(int32_t) * 2 * (static_cast<size_t>(d.E) + 1) + 16;
}

__global__ void __launch_bounds__(DISPATCH_THREADS, 1)
    dispatch_kernel(const Dims d, const Workspace ws, const CallArgs c)
{
    extern __shared__ uint32_t smem_u[];
    const int E = d.E, R = d.R, K = d.K, H = d.H;
    const int T = c.T, Tsrc = T / R;
    uint32_t *cnt = smem_u;                                  // [R][E]
    uint32_t *recv_s = cnt + R * E;                          // [E][R]
    int32_t *cum = reinterpret_cast<int32_t *>(recv_s + E * R);
    int32_t *blk = cum + (E + 1);
    volatile int *s_ok = reinterpret_cast<volatile int *>(blk + (E + 1));

    // A forward after an unreported device error does nothing (every CTA sees the same
    // sticky word: nothing writes it while this kernel runs).
    if (*reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_STICKY) != 0)
        return;
    const uint64_t deadline = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);

    // ---- phase 1: count (token x top-k entries of this CTA's contiguous token chunk) ----
    const int chunk = (T + gridDim.x - 1) / gridDim.x;
    const int t0 = min(T, static_cast<int>(blockIdx.x) * chunk);
    const int t1 = min(T, t0 + chunk);
    for (int i = threadIdx.x; i < R * E; i += blockDim.x)
        cnt[i] = 0;
    __syncthreads();
    for (long long f = static_cast<long long>(t0) * K + threadIdx.x; f < static_cast<long long>(t1) * K;
         f += blockDim.x) {
        const long long e = c.idx[f];
        if (e == -1)
            continue;
        if (e < -1 || e >= E) {
            record_error(ws.hdr, DEV_BAD_INDEX);
            continue;
        }
        const int r = static_cast<int>(f / K) / Tsrc;
        atomicAdd(&cnt[r * E + static_cast<int>(e)], 1u);
    }
    __syncthreads();

    // ---- phase 2: packed claim per (source, expert) this CTA holds tokens of -------------
    // old = atomicAdd(send, (1<<32) | count): high word counts arriving CTAs, the old low
    // word is this CTA's first slot.  Zero counts are claimed too, as the pages do.
    if (t1 > t0) {
        const int r0 = t0 / Tsrc, r1 = (t1 - 1) / Tsrc;
        const int n = (r1 - r0 + 1) * E;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const int r = r0 + i / E, e = i % E;
            const unsigned long long add = (1ull << 32) | cnt[r * E + e];
            const unsigned long long old = atomicAdd(&ws.send[r * E + e], add);
            cnt[r * E + e] = static_cast<uint32_t>(old);
        }
    }
    __syncthreads();

    // ---- phase 3: index table [e][r][slot] = token_in_source * topk + k -----------------
    for (long long f = static_cast<long long>(t0) * K + threadIdx.x; f < static_cast<long long>(t1) * K;
         f += blockDim.x) {
        const long long e = c.idx[f];
        if (e < 0 || e >= E)
            continue;
        const int t = static_cast<int>(f / K), kk = static_cast<int>(f % K);
        const int r = t / Tsrc;
        const uint32_t slot = atomicAdd(&cnt[r * E + static_cast<int>(e)], 1u);
        if (slot >= static_cast<uint32_t>(Tsrc)) {
            record_error(ws.hdr, DEV_SLOT_OVERFLOW);
            continue;
        }
        ws.table[(static_cast<long long>(e) * R + r) * ws.tsrc_cap + slot] = (t - r * Tsrc) * K + kk;
    }

    // ---- grid barrier: every claim and table entry is visible past this point -----------
    const bool skip = c.debug_skip_barrier != 0 && blockIdx.x == 0;
    if (!grid_barrier(ws.hdr + HDR_GRID_SYNC, ws.hdr, skip, deadline, s_ok))
        return;
    if (*reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_CALL) != 0)
        return;

    // ---- phase 4: received counts, expert segments, M-block map --------------------------
    for (int i = threadIdx.x; i < E * R; i += blockDim.x) {
        const int e = i / R, r = i % R;
        recv_s[i] = static_cast<uint32_t>(__ldcg(&ws.send[r * E + e]));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int rows = 0, blocks = 0;
        for (int e = e0; e < e1; ++e) {
            int n = 0;
            for (int r = 0; r < R; ++r)
                n += static_cast<int>(recv_s[e * R + r]);
            rows += n;
            blocks += (n + BM - 1) / BM;
        }
        int inc_rows = rows, inc_blocks = blocks;
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xFFFFFFFFu, inc_rows, o);
            const int b = __shfl_up_sync(0xFFFFFFFFu, inc_blocks, o);
            if (lane >= o) {
                inc_rows += a;
                inc_blocks += b;
            }
        }
        int base_rows = inc_rows - rows, base_blocks = inc_blocks - blocks;
        for (int e = e0; e < e1; ++e) {
            int n = 0;
            for (int r = 0; r < R; ++r)
                n += static_cast<int>(recv_s[e * R + r]);
            cum[e] = base_rows;
            blk[e] = base_blocks;
            base_rows += n;
            base_blocks += (n + BM - 1) / BM;
        }
        if (lane == 31) {
            cum[E] = inc_rows;
            blk[E] = inc_blocks;
        }
    }
    __syncthreads();
    const int total_rows = cum[E];
    const int total_blocks = blk[E];
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const uint32_t n = static_cast<uint32_t>(cum[e + 1] - cum[e]);
            ws.counts[e] = n;
            ws.cum_rows[e] += n;
            for (int r = 0; r < R; ++r)
                ws.recv[e * R + r] = recv_s[e * R + r];
        }
        for (int e = threadIdx.x; e <= E; e += blockDim.x)
            ws.blk_off[e] = blk[e];
    }
    const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
    const int gthreads = gridDim.x * blockDim.x;
    for (int g = gtid; g < total_blocks; g += gthreads) {
        const int e = last_le(blk, E + 1, g);
        const int n = cum[e + 1] - cum[e];
        ws.block_expert[g] = e;
        ws.block_rows[g] = min(BM, n - (g - blk[e]) * BM);
    }

    // ---- phase 5: gather, one warp per received row (global order across experts) -------
    const int lane = threadIdx.x & 31;
    const int gw = gtid >> 5, nw = gthreads >> 5;
    const int H16 = H / 16, KBH = H / 128;
    for (int j = gw; j < total_rows; j += nw) {
        const int e = last_le(cum, E + 1, j);
        const uint32_t i = static_cast<uint32_t>(j - cum[e]);
        uint32_t r, slot;
        round_robin(recv_s + e * R, R, i, r, slot);
        const int v = __ldcg(&ws.table[(static_cast<long long>(e) * R + r) * ws.tsrc_cap + slot]);
        const int t = static_cast<int>(r) * Tsrc + v / K;
        const int kk = v % K;
        const long long row = static_cast<long long>(blk[e]) * BM + i;
        const uint4 *__restrict__ src = reinterpret_cast<const uint4 *>(c.x + static_cast<long long>(t) * H);
        uint4 *__restrict__ dst = reinterpret_cast<uint4 *>(ws.pool_x + row * H);
        constexpr int U = 8;
        for (int q0 = lane; q0 < H16; q0 += 32 * U) {
            uint4 buf[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (q0 + u * 32 < H16)
                    buf[u] = __ldg(src + q0 + u * 32);
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (q0 + u * 32 < H16)
                    dst[q0 + u * 32] = buf[u];
        }
        for (int kb = lane; kb < KBH; kb += 32)
            ws.pool_sf[static_cast<long long>(kb) * ws.P + row] = __ldg(c.x_sf + static_cast<long long>(t) * KBH + kb);
        if (lane == 0) {
            ws.meta[row * 3 + 0] = r;
            ws.meta[row * 3 + 1] = static_cast<uint32_t>(t);
            ws.meta[row * 3 + 2] = static_cast<uint32_t>(kk);
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence();
            atomicAdd(&ws.arrive[row / BM], 1u);
        }
    }
}

cudaError_t launch_dispatch(const Dims &d, const Workspace &ws, const CallArgs &c, int num_sms,
                            cudaStream_t s)
{
    const size_t smem = dispatch_smem_bytes(d);
    static size_t configured = 0;
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
        configured = smem;
    }
    Dims dd = d;
    Workspace ww = ws;
    CallArgs cc = c;
    void *args[] = {&dd, &ww, &cc};
    return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(dispatch_kernel), dim3(num_sms),
                                       dim3(DISPATCH_THREADS), args, smem, s);
}

// ------------------------------------------------------------------ combine -------------
// out[t] = bf16( sum over valid k, ascending, of combine[k][t] ) in fp32; no valid k -> 0.
// Then the workspace reset of the pages' cleanup step: send counts and arrival counters go
// back to zero; a device error of this forward moves into the sticky word and the grid
// barrier counter is cleared (an aborted barrier leaves it mid-phase).
__global__ void __launch_bounds__(COMBINE_THREADS)
    combine_kernel(const Dims d, const Workspace ws, const CallArgs c)
{
    const int K = d.K, H = d.H;
    const uint32_t err = *reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_CALL) |
                         *reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_STICKY);
    if (err == 0) {
        // one thread per 16-byte output vector (8 bf16); its top-k plane loads are
        // independent, so they are all in flight together
        const int H8 = H / 8;
        const long long plane = static_cast<long long>(ws.max_tokens) * H8;   // uint4 per plane
        const uint4 *cb = reinterpret_cast<const uint4 *>(ws.combine);
        uint4 *out = reinterpret_cast<uint4 *>(c.out);
        const long long n = static_cast<long long>(c.T) * H8;
        const long long gthreads_l = static_cast<long long>(gridDim.x) * blockDim.x;
        for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < n;
             g += gthreads_l) {
            const long long t = g / H8;
            uint32_t mask = 0;
            for (int kk = 0; kk < K; ++kk)
                mask |= (__ldg(c.idx + t * K + kk) >= 0 ? 1u : 0u) << kk;
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                acc[q] = 0.0f;
#pragma unroll 8
            for (int kk = 0; kk < K; ++kk) {
                if (mask & (1u << kk)) {
                    const uint4 u = __ldcs(cb + kk * plane + g);
                    const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
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
            out[g] = o;
        }
    }
    // reset for the next forward
    const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
    const int gthreads = gridDim.x * blockDim.x;
    for (int i = gtid; i < d.R * d.E; i += gthreads)
        ws.send[i] = 0ull;
    for (int i = gtid; i < ws.max_blocks; i += gthreads) {
        ws.arrive[i] = 0u;
        ws.l1_done[i] = 0u;
    }
    if (gtid == 0) {
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

cudaError_t launch_combine(const Dims &d, const Workspace &ws, const CallArgs &c, int num_sms,
                           cudaStream_t s)
{
    combine_kernel<<<num_sms * 4, COMBINE_THREADS, 0, s>>>(d, ws, c);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ weights -------------
// Load-time weight re-layout into GEMM tiles.  dst = [E][N/256][K/128][256][128] bytes: every
// 256-row x 128-byte tile the FFN kernel loads per 128-deep K block is one contiguous 32 KB
// block, so each weight load streams whole DRAM pages instead of 256 rows 7 KB apart.
// With gate_up_I > 0 (the gate_up weight, N = 2I) the rows are also gate/up interleaved:
// within each group of 16 rows, rows 0..7 are gate rows 8j..8j+7 and rows 8..15 are up rows
// I+8j..I+8j+7 (granularity 8, the layout of "DeepGEMM Mega MoE 对称内存（Symmetric Memory）
// 深度分析" §10.2), so one 256-row tile holds 128 gate rows and the 128 matching up rows.
__global__ void relayout_weights_kernel(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int E,
                                        int N, int K, int gate_up_I)
{
    const int KB = K / 128, NT = N / BN;
    const long long chunks = static_cast<long long>(E) * N * (K / 16);
    for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < chunks;
         q += static_cast<long long>(gridDim.x) * blockDim.x) {
        long long t = q;
        const int c16 = static_cast<int>(t % 8);
        t /= 8;
        const int r = static_cast<int>(t % BN);
        t /= BN;
        const int kb = static_cast<int>(t % KB);
        t /= KB;
        const int nt = static_cast<int>(t % NT);
        const long long e = t / NT;
        const int n = nt * BN + r;
        int srow = n;
        if (gate_up_I > 0) {
            const int j = n / 16, i = n % 16;
            srow = i < 8 ? 8 * j + i : gate_up_I + 8 * j + (i - 8);
        }
        const uint4 *sp = reinterpret_cast<const uint4 *>(src + (e * N + srow) * static_cast<long long>(K) +
                                                          kb * 128 + c16 * 16);
        reinterpret_cast<uint4 *>(dst)[q] = *sp;
    }
}

cudaError_t launch_relayout_weights(const uint8_t *src, uint8_t *dst, int E, int N, int K, int gate_up_I,
                                    cudaStream_t s)
{
    relayout_weights_kernel<<<2048, 256, 0, s>>>(src, dst, E, N, K, gate_up_I);
    return cudaGetLastError();
}

}  // namespace cpw
