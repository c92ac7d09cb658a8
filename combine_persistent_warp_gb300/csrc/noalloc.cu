// noalloc.cu -- routing of one batch for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: code that runs inside another
// framework's memory pool or a fixed memory budget, a real-time loop that must not
// enter the driver's allocator, or a plug-in whose host owns every device allocation.
// moe_route_noalloc gives them the routing part of the layer (per-expert counts,
// per-(expert, source) counts, expert block offsets and the round-robin pool row
// metadata) with no allocation: the scratch it needs (the packed per-(source, expert)
// slot counters and the [expert][source][slot] index table) lives in one file-scope
// device array of fixed size, held by every GPU that loads the library until exit.
//
// The array's name is only a host-side stand-in in host code, so the real device address
// is looked up once per device with cudaGetSymbolAddress (with that device current) and
// passed to the kernels.  The address is kept for the life of the process: a device reset
// (cudaDeviceReset, which unloads the module) makes it stale, so the entry point must not be
// called on a device after a reset of that device.  Every call shares the array and leaves its contents behind: the
// counters are cleared on the caller's stream at the start of each call, the table needs
// no clearing (every entry read is written first by the same call).  Calls that overlap on
// the GPU (different streams, or different host threads on one device) race on the array.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "../../include/cpw_moe.h"
#include "moe_internal.cuh"

namespace cpw {

namespace {

constexpr long long NA_MAX_TABLE = 1ll << 20;   // E * T index table entries (4 MB)
constexpr long long NA_MAX_ROUTED = 1ll << 17;  // T * topk routed entries
constexpr int NA_MAX_ER = 4096;                 // E * R slot counters
constexpr size_t NA_SEND_BYTES = static_cast<size_t>(NA_MAX_ER) * sizeof(unsigned long long);
constexpr size_t NA_SCRATCH_BYTES = NA_SEND_BYTES + static_cast<size_t>(NA_MAX_TABLE) * sizeof(int32_t);
constexpr int NA_THREADS = 512;
constexpr int NA_MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NA_SCRATCH_BYTES];

struct DeviceScratch {
    bool ready = false;
    unsigned char *ptr = nullptr;
    int num_sms = 0;
};
std::mutex g_mu;
DeviceScratch g_dev[NA_MAX_DEVICES];

// Device address of the scratch array (and the SM count) of the current device; the first
// call on a device looks them up.
int scratch_of_current_device(unsigned char **ptr, int *num_sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (dev < 0 || dev >= NA_MAX_DEVICES)
        return MOE_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceScratch &d = g_dev[dev];
    if (!d.ready) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return MOE_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
            return MOE_ERR_CUDA;
        d.ptr = static_cast<unsigned char *>(p);
        d.num_sms = sms;
        d.ready = true;
    }
    *ptr = d.ptr;
    *num_sms = d.num_sms;
    return MOE_OK;
}

__device__ __forceinline__ void na_error(int32_t *status, int32_t code)
{
    atomicCAS(status, 0, code);
}

// Largest i in [0, n) with a[i] <= v (a non-decreasing, a[0] <= v).
__device__ __forceinline__ int na_last_le(const int32_t *a, int n, int32_t v)
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

// Round-robin source choice by min-peeling for position p of one expert's rows.
__device__ __forceinline__ void na_round_robin(const uint32_t *recv, int R, uint32_t p, uint32_t &src,
                                               uint32_t &slot)
{
    uint32_t peeled = 0;
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
            slot = peeled + p / A;
            return;
        }
        p -= A * L;
        peeled += L;
    }
}

// Kernel 1: per-(source, expert) counts of this CTA's token chunk, packed claim
// old = atomicAdd(send, (1<<32) | count), then table[e][r][slot] = token_in_source*topk + k.
__global__ void __launch_bounds__(NA_THREADS)
    na_count_claim_table(const int64_t *__restrict__ idx, int T, int E, int K, int R,
                         unsigned long long *send, int32_t *table, int32_t *status)
{
    extern __shared__ uint32_t cnt[];   // [R][E]
    const int Tsrc = T / R;
    const int chunk = (T + gridDim.x - 1) / gridDim.x;
    const int t0 = min(T, static_cast<int>(blockIdx.x) * chunk);
    const int t1 = min(T, t0 + chunk);
    for (int i = threadIdx.x; i < R * E; i += blockDim.x)
        cnt[i] = 0;
    __syncthreads();
    for (long long f = static_cast<long long>(t0) * K + threadIdx.x; f < static_cast<long long>(t1) * K;
         f += blockDim.x) {
        const long long e = idx[f];
        if (e == -1)
            continue;
        if (e < -1 || e >= E) {
            na_error(status, MOE_ERR_BAD_INDEX);
            continue;
        }
        atomicAdd(&cnt[(static_cast<int>(f / K) / Tsrc) * E + static_cast<int>(e)], 1u);
    }
    __syncthreads();
    if (t1 > t0) {
        const int r0 = t0 / Tsrc, r1 = (t1 - 1) / Tsrc;
        for (int i = threadIdx.x; i < (r1 - r0 + 1) * E; i += blockDim.x) {
            const int r = r0 + i / E, e = i % E;
            const unsigned long long old = atomicAdd(&send[r * E + e], (1ull << 32) | cnt[r * E + e]);
            cnt[r * E + e] = static_cast<uint32_t>(old);
        }
    }
    __syncthreads();
    for (long long f = static_cast<long long>(t0) * K + threadIdx.x; f < static_cast<long long>(t1) * K;
         f += blockDim.x) {
        const long long e = idx[f];
        if (e < 0 || e >= E)
            continue;
        const int t = static_cast<int>(f / K), kk = static_cast<int>(f % K);
        const int r = t / Tsrc;
        const uint32_t slot = atomicAdd(&cnt[r * E + static_cast<int>(e)], 1u);
        if (slot >= static_cast<uint32_t>(Tsrc)) {
            na_error(status, MOE_ERR_SLOT_OVERFLOW);
            continue;
        }
        table[(e * R + r) * static_cast<long long>(Tsrc) + slot] = (t - r * Tsrc) * K + kk;
    }
}

// Kernel 2: received counts, expert segments (block offsets), and for every received row
// its pool row and {source, token, topk slot} metadata in round-robin order.
__global__ void __launch_bounds__(NA_THREADS)
    na_offsets_meta(int T, int E, int K, int R, const unsigned long long *send, const int32_t *table,
                    const int32_t *status, uint32_t *counts, uint32_t *recv, int32_t *block_offset,
                    uint32_t *meta)
{
    extern __shared__ uint32_t sm[];
    uint32_t *recv_s = sm;                                     // [E][R]
    int32_t *cum = reinterpret_cast<int32_t *>(recv_s + E * R);
    int32_t *blk = cum + (E + 1);
    if (*reinterpret_cast<const volatile int32_t *>(status) != 0)
        return;   // written only by the previous kernel: every CTA sees the same value
    const int Tsrc = R > 0 ? T / R : 0;
    for (int i = threadIdx.x; i < E * R; i += blockDim.x) {
        const int e = i / R, r = i % R;
        recv_s[i] = static_cast<uint32_t>(send[r * E + e]);
    }
    __syncthreads();
    {
        // expert row and M-block prefixes: each thread sums a run of at most two experts,
        // then a block-wide scan (warp shuffles, then the warp totals)
        __shared__ int wtot[2][NA_THREADS / 32];
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const int per = (E + NA_THREADS - 1) / NA_THREADS;
        const int e0 = min(E, static_cast<int>(threadIdx.x) * per), e1 = min(E, e0 + per);
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
        if (lane == 31) {
            wtot[0][warp] = inc_rows;
            wtot[1][warp] = inc_blocks;
        }
        __syncthreads();
        if (warp == 0) {
            int wr = lane < NA_THREADS / 32 ? wtot[0][lane] : 0;
            int wb = lane < NA_THREADS / 32 ? wtot[1][lane] : 0;
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xFFFFFFFFu, wr, o);
                const int b = __shfl_up_sync(0xFFFFFFFFu, wb, o);
                if (lane >= o) {
                    wr += a;
                    wb += b;
                }
            }
            if (lane < NA_THREADS / 32) {
                wtot[0][lane] = wr;   // inclusive prefix over warps
                wtot[1][lane] = wb;
            }
        }
        __syncthreads();
        int base_rows = inc_rows - rows + (warp > 0 ? wtot[0][warp - 1] : 0);
        int base_blocks = inc_blocks - blocks + (warp > 0 ? wtot[1][warp - 1] : 0);
        for (int e = e0; e < e1; ++e) {
            int n = 0;
            for (int r = 0; r < R; ++r)
                n += static_cast<int>(recv_s[e * R + r]);
            cum[e] = base_rows;
            blk[e] = base_blocks;
            base_rows += n;
            base_blocks += (n + BM - 1) / BM;
        }
        if (threadIdx.x == NA_THREADS - 1) {
            cum[E] = wtot[0][NA_THREADS / 32 - 1];
            blk[E] = wtot[1][NA_THREADS / 32 - 1];
        }
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            counts[e] = static_cast<uint32_t>(cum[e + 1] - cum[e]);
            for (int r = 0; r < R; ++r)
                recv[e * R + r] = recv_s[e * R + r];
        }
        for (int e = threadIdx.x; e <= E; e += blockDim.x)
            block_offset[e] = blk[e];
    }
    const int total = cum[E];
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < total; j += gridDim.x * blockDim.x) {
        const int e = na_last_le(cum, E + 1, j);
        const uint32_t i = static_cast<uint32_t>(j - cum[e]);
        uint32_t r, slot;
        na_round_robin(recv_s + e * R, R, i, r, slot);
        const int v = table[(static_cast<long long>(e) * R + r) * Tsrc + slot];
        const long long row = static_cast<long long>(blk[e]) * BM + i;
        meta[row * 3 + 0] = r;
        meta[row * 3 + 1] = static_cast<uint32_t>(static_cast<int>(r) * Tsrc + v / K);
        meta[row * 3 + 2] = static_cast<uint32_t>(v % K);
    }
}

}  // namespace

}  // namespace cpw

extern "C" int moe_route_noalloc(int T, int E, int topk, int R, const int64_t *topk_idx,
                                 uint32_t *counts, uint32_t *recv, int32_t *block_offset,
                                 uint32_t *meta, int32_t *status, void *stream)
{
    using namespace cpw;
    if (T < 0 || E < 1 || E > 1024 || topk < 1 || topk > 32 || topk > E || R < 1 || R > 64 ||
        T % R != 0)
        return MOE_ERR_INVALID_ARG;
    if (static_cast<long long>(E) * R > NA_MAX_ER || static_cast<long long>(T) * topk > NA_MAX_ROUTED ||
        static_cast<long long>(E) * T > NA_MAX_TABLE)
        return MOE_ERR_CAPACITY;
    if (!counts || !recv || !block_offset || !status || (T > 0 && (!topk_idx || !meta)))
        return MOE_ERR_INVALID_ARG;
    unsigned char *scratch = nullptr;
    int num_sms = 0;
    const int rc = scratch_of_current_device(&scratch, &num_sms);
    if (rc != MOE_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the scratch address is the current device's: the stream must belong to that device
    int cur = 0, sdev = 0;
    if (cudaGetDevice(&cur) != cudaSuccess || cudaStreamGetDevice(s, &sdev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (sdev != cur)
        return MOE_ERR_INVALID_ARG;
    auto *send = reinterpret_cast<unsigned long long *>(scratch);
    auto *table = reinterpret_cast<int32_t *>(scratch + NA_SEND_BYTES);
    if (cudaMemsetAsync(send, 0, sizeof(unsigned long long) * E * R, s) != cudaSuccess ||
        cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    const int grid1 = std::max(1, std::min(num_sms, (T + 31) / 32));
    na_count_claim_table<<<grid1, NA_THREADS, sizeof(uint32_t) * E * R, s>>>(topk_idx, T, E, topk, R, send,
                                                                             table, status);
    if (cudaGetLastError() != cudaSuccess)
        return MOE_ERR_CUDA;
    const size_t smem2 = sizeof(uint32_t) * E * R + sizeof(int32_t) * 2 * (E + 1);
    na_offsets_meta<<<num_sms, NA_THREADS, smem2, s>>>(T, E, topk, R, send, table, status, counts, recv,
                                                       block_offset, meta);
    if (cudaGetLastError() != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
