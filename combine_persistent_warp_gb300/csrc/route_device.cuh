// route_device.cuh -- the routing steps of the fused MoE layer as device functions (count,
// packed claim, index table, grid barrier, segments, round-robin gather of one row), used by
// the routing kernel in routing.cu.
//
// Source pages, by title and section:
//   "Mega-MoE 内核代码导读：从 Dispatch 到 WGMMA 的融合流水线" §4.1 (token x top-k scan),
//     §4.2 (per-expert count with block atomics, packed (1<<32)|count global claim),
//     §4.3 (index table [local_expert][source][slot] = token*topk + k), §4.4 (grid sync)
//   Mega-MoE walkthrough part 2 (kwkr.cn/news/1317662) §2.4 (expert segments, pool block
//     offsets by ceil_div), §2.5 (round-robin source choice by min-peeling), §2.6 (row copy,
//     scale copy, {source, token, topk} metadata, per-M-block arrival count)
//   "DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析" §6.2 (XOR-tag grid barrier with a
//     time limit)
//
// On one GPU the pages' ranks become R logical source partitions of the token batch:
// source r owns tokens [r*T/R, (r+1)*T/R).  A "remote" store is a plain global store.
#pragma once

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace cpw {
namespace route {

// XOR-tag grid barrier: CTA 0 adds 0x80000000 - (n-1), every other CTA adds 1, so bit 31
// of the counter flips exactly when all n CTAs have arrived.  Bounded: on the deadline the
// CTA records DEV_TIMEOUT and returns false.  `skip_arrive` is the failure-path test hook.
// Every thread of the CTA calls it; `s_ok` is a shared-memory word.
__device__ inline bool grid_barrier(uint32_t *counter, uint32_t *hdr, bool skip_arrive, uint64_t deadline,
                                    volatile int *s_ok)
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
__device__ __forceinline__ void round_robin(const uint32_t *recv, int R, uint32_t p, uint32_t &src,
                                            uint32_t &slot)
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

// Steps of one CTA before the grid barrier, over its contiguous chunk of tokens:
//   count: shared histogram cnt[R][E] of its (token, k) entries (block atomics);
//   claim: old = atomicAdd(send[r][e], (1<<32) | count) for every (source, expert) it holds
//          tokens of (zero counts too, as the pages do); the old low word is its first slot;
//   table: table[e][r][slot] = token_in_source * topk + k.
// Bad expert ids and slot overflow are recorded as device errors.  All threads call it.
__device__ inline void count_claim_table(const Dims &d, const Workspace &ws, const CallArgs &c, uint32_t *cnt)
{
    const int E = d.E, R = d.R, K = d.K;
    const int T = c.T, Tsrc = T / R;
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
}

// tok_mask[t] = the routed top-k slots of token t (bit k set when topk_idx[t][k] >= 0; topk +
// shared slots <= 32), read by the combine kernel and by the combine inside the FFN kernel
// (topk_combine.cuh); for the latter the output row of a token with no routed slot is zero (the
// combine's empty sum), written here because no down tile will ever count it.  One thread per
// token of the grid.
__device__ inline void token_masks(const Dims &d, const Workspace &ws, const CallArgs &c)
{
    const int K = d.K;
    const int G = gridDim.x * blockDim.x;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < c.T; t += G) {
        const int64_t *id = c.idx + static_cast<long long>(t) * K;
        uint32_t m = 0;
#pragma unroll 8
        for (int k = 0; k < K; ++k)
            m |= (id[k] >= 0 ? 1u : 0u) << k;
        ws.tok_mask[t] = m;
        if (m == 0 && c.fused_combine) {
            uint4 *o = reinterpret_cast<uint4 *>(c.out + static_cast<long long>(t) * d.H);
            for (int v = 0; v < d.H / 8; ++v)
                o[v] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// Step after the grid barrier: rows per (expert, source) from the claim words into recv_s
// [E][R] (shared), expert row prefix cum[E+1] and M-block prefix blk[E+1] (shared, by one
// warp's scan), then CTA 0 publishes counts, recv, block offsets and the cumulative rows, and
// the grid writes the M-block map (expert, valid rows of every block).  All threads call it.
__device__ inline void segments(const Dims &d, const Workspace &ws, uint32_t *recv_s, int32_t *cum, int32_t *blk)
{
    const int E = d.E, R = d.R;
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
    for (int g = gtid; g < blk[E]; g += gthreads) {
        const int e = last_le(blk, E + 1, g);
        const int n = cum[e + 1] - cum[e];
        ws.block_expert[g] = e;
        ws.block_rows[g] = min(BM, n - (g - blk[e]) * BM);
    }
}

// Step a5: the gather of the expert-major pool, one warp per pool row at a time (rows in
// expert order).  For pool row j of expert e (recv_e = rows of expert e per source) the round
// robin picks (source, slot) and the index table gives (token, k); the token's H bytes move
// global -> shared -> global by two bulk (TMA) copies through a double buffer of the warp, the
// next row's load issued before the current row's store, while the lanes write the row's H/128
// scales (and, on the block-scaled path, their UE8M0 bytes), its {source, token, k} and add one
// to the M-block's arrival count.  The FFN kernel that reads the pool is a later launch on the
// same stream, which orders all of these stores before its loads, so the count is a plain
// (relaxed) increment.
struct PoolRow {
    long long row;   // pool row
    int t, kk;       // token, top-k slot
    uint32_t r;      // source
};

__device__ __forceinline__ PoolRow resolve_row(const Dims &d, const Workspace &ws, const CallArgs &c, int j,
                                               const int32_t *cum, const int32_t *blk, const uint32_t *recv_s)
{
    const int e = last_le(cum, d.E + 1, j);
    const uint32_t i = static_cast<uint32_t>(j - cum[e]);
    PoolRow x;
    uint32_t slot;
    round_robin(recv_s + e * d.R, d.R, i, x.r, slot);
    const int v = __ldcg(&ws.table[(static_cast<long long>(e) * d.R + x.r) * ws.tsrc_cap + slot]);
    x.t = static_cast<int>(x.r) * (c.T / d.R) + v / d.K;
    x.kk = v % d.K;
    x.row = static_cast<long long>(blk[e]) * BM + i;
    return x;
}

// the row's scales, UE8M0 bytes, metadata and arrival (all lanes of the warp)
__device__ __forceinline__ void row_side_data(const Dims &d, const Workspace &ws, const CallArgs &c, const PoolRow &x,
                                              int lane)
{
    const int KBH = d.H / 128;
    for (int kb = lane; kb < KBH; kb += 32) {
        const float sf = __ldg(c.x_sf + static_cast<long long>(x.t) * KBH + kb);
        ws.pool_sf[static_cast<long long>(kb) * ws.P + x.row] = sf;
        if (c.block_scaled) {
            // UE8M0 byte of this row and K block kb in its M-block's 512-byte scale block of
            // the group of four K blocks kb / 4 (row r's word at byte 16*(r%32) + 4*(r/32),
            // byte kb % 4); the scale must be a power of two
            const uint32_t b = __float_as_uint(sf), ex = (b >> 23) & 0xFFu;
            if ((b & 0x807FFFFFu) != 0u || ex == 0u || ex == 0xFFu)
                record_error(ws.hdr, DEV_BAD_SCALE);
            const int rr = static_cast<int>(x.row % BM);
            ws.pool_sfe[((x.row / BM) * ((KBH + 3) / 4) + kb / 4) * 512 + 16 * (rr % 32) + 4 * (rr / 32) + kb % 4] =
                static_cast<uint8_t>(ex);
        }
    }
    if (lane == 0) {
        ws.meta[x.row * 3 + 0] = x.r;
        ws.meta[x.row * 3 + 1] = static_cast<uint32_t>(x.t);
        ws.meta[x.row * 3 + 2] = static_cast<uint32_t>(x.kk);
        atomicAdd(ws.arrive + x.row / BM, 1u);
    }
}

// One gather warp: rows gw, gw + nw, ...; bar[2] (initialised, count 1) and buf (2 * H bytes,
// 16-byte aligned) are the warp's own.  Every wait is bounded; on a time-out the warp records
// DEV_TIMEOUT, waits (bounded again) for its loads in flight and stops.  Before returning, lane
// 0 waits for its bulk stores to complete.
__device__ inline void gather_rows(const Dims &d, const Workspace &ws, const CallArgs &c, const int32_t *cum,
                                   const int32_t *blk, const uint32_t *recv_s, int gw, int nw, uint64_t *bar,
                                   uint8_t *buf, uint64_t deadline, int lane)
{
    const int total = cum[d.E];
    if (gw >= total)
        return;
    const uint32_t H = static_cast<uint32_t>(d.H);
    PoolRow cur = resolve_row(d, ws, c, gw, cum, blk, recv_s);
    if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&bar[0], H);
        ptx::bulk_load(buf, c.x + static_cast<long long>(cur.t) * H, H, &bar[0]);
    }
    uint32_t it = 0;
    bool ok = true;
    for (int j = gw; j < total; j += nw, ++it) {
        const bool more = j + nw < total;
        PoolRow nxt{};
        if (more) {
            nxt = resolve_row(d, ws, c, j + nw, cum, blk, recv_s);
            if (lane == 0) {
                // the other buffer's last store (row j - nw) has read it
                ptx::bulk_wait_read<0>();
                const uint32_t nb = (it + 1) & 1u;
                ptx::mbar_arrive_expect_tx(&bar[nb], H);
                ptx::bulk_load(buf + nb * H, c.x + static_cast<long long>(nxt.t) * H, H, &bar[nb]);
            }
        }
        row_side_data(d, ws, c, cur, lane);
        if (lane == 0) {
            const uint32_t b = it & 1u;
            if (ptx::mbar_wait(&bar[b], (it >> 1) & 1u, deadline)) {
                ptx::bulk_store(ws.pool_x + cur.row * H, buf + b * H, H);
                ptx::bulk_commit();
            } else {
                ok = false;
            }
        }
        if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) {
            if (lane == 0) {
                record_error(ws.hdr, DEV_TIMEOUT);
                const uint64_t dl = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);
                ptx::mbar_wait(&bar[it & 1u], (it >> 1) & 1u, dl);
                if (more)
                    ptx::mbar_wait(&bar[(it + 1) & 1u], ((it + 1) >> 1) & 1u, dl);
            }
            break;
        }
        cur = nxt;
    }
    if (lane == 0)
        ptx::bulk_wait<0>();
}

}  // namespace route
}  // namespace cpw
