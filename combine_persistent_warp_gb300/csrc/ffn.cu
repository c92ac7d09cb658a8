// ffn.cu -- the expert FFN of the fused MoE layer as ONE persistent, warp-specialised
// FP8 grouped-GEMM kernel on tcgen05 (sm_103a).
//
// Both expert GEMMs run in the same launch ("Mega-MoE 内核代码导读：从 Dispatch 到 WGMMA 的融合
// 流水线" §六: Linear1 gate_up then Linear2 down; "MOE融合算子", DeepGEMM MegaMoE §2 and §5:
// within an expert wave, all Linear1 tiles, then all Linear2 tiles; a Linear2 block waits
// only for the Linear1 tiles of its own M-block):
//   phase 1 tile (blk, nt):  A = gathered pool rows [P][H] e4m3 with 1x128 scales,
//                            B = gate/up-interleaved W1 tiles (contiguous 256 x 128-byte
//                            blocks per 128-deep K block) e4m3 with 128x128 scales;
//                            epilogue: SwiGLU, per-row 1x128 requant -> act [P][I], then
//                            one release-increment of l1_done[blk] per epilogue warp.
//   phase 2 tile (blk, nt):  producer first waits for l1_done[blk] == 8 * (2I/256), then
//                            A = act [P][I] with scales, B = W2 tiles with 128x128 scales;
//                            epilogue: times the top-k gate weight, bf16, scatter through the
//                            {source, token, topk} metadata into combine[topk][T][H]
//                            ("DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析" §8.1).
// Tiles are listed wave by wave ([phase-1 tiles of the wave's blocks][phase-2 tiles of the
// same blocks]) and handed out in list order from one global counter (the producer warp of
// a CTA takes its next tile when it starts one and passes the index to the UMMA and
// epilogue warps through a small ring), so a phase-2 wait only ever waits on phase-1 tiles
// that were handed out earlier: the smallest unfinished phase-1 tile is always being worked
// on.  The launch is cooperative (all CTAs resident), so those tiles always finish.
//
// Roles of the 12 warps of a CTA (one CTA per SM):
//   warp 0     TMA producer: A and B tiles of one BKS-deep K slice per stage into a
//              STAGES-deep ring (192 KB), plus L2 prefetch of B PREFETCH_KB blocks ahead
//   warp 1     UMMA issuer: (128x256x32) tcgen05.mma, 128/32 of them per scale block, into
//              a fresh TMEM partial per 128-deep scale block
//   warps 2-3  idle (the epilogue warpgroups must start at a warpgroup boundary)
//   warps 4-11 two epilogue warpgroups, columns [0,128) and [128,256) of the tile
// The fp32 scales are arbitrary per 128-deep K block (1x128 for A rows, 128x128 for B), so
// each K block's product lands in its own TMEM partial (double-buffered, 2 x 256 columns)
// and the epilogue warps promote it into fp32 registers with the product of the two scales
// (the promotion of the first page, §8.1), overlapped with the next block's UMMA through
// the TMEM full/empty barriers.
// 2-CTA mode (clusters of two CTAs on neighbouring SMs): one cta_group::2 UMMA of
// 256 x 256 x 32 covers two M-blocks of one expert; each CTA stages its own 128 A rows and
// one 128-row half of the weight tile (32 KB per stage, six stages), the even CTA issues
// the UMMAs and each CTA's epilogue promotes the 128 rows in its own TMEM.  Per FLOP this
// moves a third fewer operand bytes from L2 than the one-CTA tile; tiles are dealt to the
// clusters round-robin in list order.
// All waits carry a deadline; on expiry the CTA records MOE_ERR_TIMEOUT and leaves after
// draining the copies and MMAs it has in flight.
#include <cuda_bf16.h>

#include <algorithm>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace cpw {

namespace {

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = ptx::idesc_e4m3_f32(BM, BN);
#ifndef CPW_PREFETCH_KB
#define CPW_PREFETCH_KB 0
#endif
constexpr int PREFETCH_KB = CPW_PREFETCH_KB;   // L2 prefetch distance of B, in scale blocks
constexpr int EPI_WARPS = 8;
constexpr int TILE_RING = 4;   // tiles the producer may run ahead of the UMMA/epilogue warps
// Two-CTA mode (cta_group::2): one UMMA of M = 256 rows covers two M-blocks, one in each
// CTA of a cluster pair; each CTA stages its own 128 A rows and one half (128 rows) of the
// 256-row weight tile, so a stage is 32 KB instead of 48 KB and the same 192 KB holds six.
constexpr uint32_t PAIR_B_BYTES = STAGE_B_BYTES / 2;
constexpr uint32_t PAIR_STAGE_BYTES = STAGE_A_BYTES + PAIR_B_BYTES;
constexpr int PAIR_STAGES = static_cast<int>((STAGES * STAGE_BYTES) / PAIR_STAGE_BYTES);
constexpr int MAX_STAGES = PAIR_STAGES > STAGES ? PAIR_STAGES : STAGES;
constexpr uint32_t IDESC_PAIR = ptx::idesc_e4m3_f32(2 * BM, BN);
// One CTA, one stage per scale block: the UMMA issuer commits once per K block (to the
// TMEM-full barrier) and the epilogue, having seen that the MMAs are done, releases the
// operand stage to the producer.  A second commit per K block for the stage cost ~95 cycles
// of UMMA issue each time.
template <bool PAIRED>
constexpr bool EPI_RELEASES_STAGE = !PAIRED && SUBS == 1;
static_assert(PAIR_STAGES * PAIR_STAGE_BYTES <= STAGES * STAGE_BYTES, "pair stages exceed the ring");

#ifdef CPW_TRACE
// Development trace (compiled only with -DCPW_TRACE): SM clock stamps of two CTAs, per
// pipeline stage for the producer (0: load issue) and the UMMA issuer (1: stage full,
// 2: MMAs issued), per scale block for one epilogue warp (3: TMEM full, 4: promoted,
// 5: tile epilogue start).
// 6: producer tile start, 7: producer done waiting for a down tile's gate_up blocks,
// 8: UMMA issuer done waiting for an empty TMEM partial (per scale block), 9: the epilogue
// warp's TMEM-empty arrival (per scale block).
// g_cta_span: global-timer ns at every CTA's start and end (cross-SM comparable).
constexpr int TRACE_CTAS = 2, TRACE_EVENTS = 10, TRACE_ITERS = 4096, TRACE_MAX_GRID = 1024;
__device__ unsigned long long g_trace[TRACE_CTAS][TRACE_EVENTS][TRACE_ITERS];
__device__ unsigned long long g_cta_span[2][TRACE_MAX_GRID];
__device__ __forceinline__ int trace_slot()
{
    return blockIdx.x == 0 ? 0 : (blockIdx.x == gridDim.x / 2 ? 1 : -1);
}
#define CPW_STAMP(ev, it)                                                                   \
    do {                                                                                     \
        const int ts_ = trace_slot();                                                        \
        if (ts_ >= 0 && (it) < static_cast<uint32_t>(TRACE_ITERS))                           \
            g_trace[ts_][ev][it] = static_cast<unsigned long long>(clock64());               \
    } while (0)
#else
#define CPW_STAMP(ev, it) \
    do {                  \
    } while (0)
#endif

struct __align__(8) FfnBars {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t xbar;          // row-amax exchange between the two epilogue warpgroups
    uint64_t tile_full[TILE_RING];    // producer -> UMMA issuer + epilogue: next tile index
    uint64_t tile_empty[TILE_RING];   // UMMA issuer + 8 epilogue warps have read the slot
    int tile_ring[TILE_RING];
    uint32_t tmem_base;
    int abort;
    float amax[2][2][BM];   // [tile parity][column half][row]
    int32_t pair_off[1025]; // 2-CTA mode: first block pair of each expert (E <= 1024)
};

// Tile list: waves of `wave_blocks` M-blocks; inside a wave all phase-1 tiles (block-major,
// n-tile minor), then all phase-2 tiles of the same blocks.
struct TileList {
    int NT1, NT2, nblocks, wave_blocks;

    __device__ __forceinline__ int total() const { return nblocks * (NT1 + NT2); }

    __device__ __forceinline__ void at(int tile, int &phase, int &blk, int &nt) const
    {
        const int full = wave_blocks * (NT1 + NT2);
        const int w = tile / full;
        const int r = tile - w * full;
        const int b0 = w * wave_blocks;
        const int nb = min(wave_blocks, nblocks - b0);
        if (r < nb * NT1) {
            phase = 1;
            blk = b0 + r / NT1;
            nt = r % NT1;
        } else {
            const int r2 = r - nb * NT1;
            phase = 2;
            blk = b0 + r2 / NT2;
            nt = r2 % NT2;
        }
    }
};

}  // namespace

// Tile of the list as one CTA sees it.  In 2-CTA mode a list entry is a pair of
// consecutive M-blocks of one expert (one M = 256 UMMA tile); CTA rank r takes the r-th
// block, and an expert with an odd block count leaves rank 1 a null half (it loads no A
// rows, only its half of the weight tile, and stores nothing).
struct TileView {
    int phase, nt, blk, e;
    bool null_half;
};

template <bool PAIRED>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    ffn_kernel(const __grid_constant__ FfnMaps maps, const Dims d, const Workspace ws, const CallArgs c,
               const float *__restrict__ sf1, const float *__restrict__ sf2, const int wave_blocks)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    FfnBars *bars = reinterpret_cast<FfnBars *>(smem + STAGES * STAGE_BYTES);
    constexpr int NST = PAIRED ? PAIR_STAGES : STAGES;                  // stages in the ring
    constexpr uint32_t SBYTES = PAIRED ? PAIR_STAGE_BYTES : STAGE_BYTES;   // bytes per stage
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        const uint32_t err = *reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_CALL) |
                             *reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_STICKY);
        bars->abort = err != 0;
        if (!err) {
            // 2-CTA mode: only the even CTA's full and TMEM-empty barriers are used; both
            // CTAs' loads count on its full barrier, both CTAs' epilogue warps arrive on its
            // TMEM-empty barrier, and its UMMA commits arrive on both CTAs' empty / TMEM-full
            for (int s = 0; s < NST; ++s) {
                ptx::mbar_init(&bars->full[s], 1);
                ptx::mbar_init(&bars->empty[s], 1);
            }
            for (int b = 0; b < 2; ++b) {
                ptx::mbar_init(&bars->tfull[b], 1);
                ptx::mbar_init(&bars->tempty[b], (PAIRED ? 2 : 1) * EPI_WARPS);   // one per epilogue warp
            }
            ptx::mbar_init(&bars->xbar, 32 * EPI_WARPS);       // every epilogue thread
            for (int i = 0; i < TILE_RING; ++i) {
                ptx::mbar_init(&bars->tile_full[i], 1);
                ptx::mbar_init(&bars->tile_empty[i], 1 + EPI_WARPS);
            }
            ptx::fence_mbar_init();
        }
    }
    __syncthreads();
    uint32_t rank = 0;
    if constexpr (PAIRED) {
        // both CTAs' barriers are initialised before any remote load, commit or arrive, and
        // both take the same abort decision (a CTA must not leave while its peer may still
        // write into its shared memory)
        ptx::cluster_sync();
        rank = ptx::cluster_ctarank();
        const int peer_abort = ptx::ld_cluster_s32(ptx::map_cluster(&bars->abort, rank ^ 1u));
        const bool stop = bars->abort || peer_abort;
        ptx::cluster_sync();
        if (stop)
            return;
        if (threadIdx.x == 0) {
            int acc = 0;
            for (int e = 0; e < d.E; ++e) {
                bars->pair_off[e] = acc;
                acc += (ws.blk_off[e + 1] - ws.blk_off[e] + 1) / 2;
            }
            bars->pair_off[d.E] = acc;
        }
    } else {
        if (bars->abort)
            return;
    }
    if (warp == 1) {
        if constexpr (PAIRED) {
            ptx::tmem_alloc_pair(&bars->tmem_base, TMEM_COLS);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(&bars->tmem_base, TMEM_COLS);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (PAIRED)
        ptx::cluster_sync();   // both CTAs hold their TMEM before the even CTA's first UMMA
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    const TileList tl{(2 * d.I) / BN, (d.H + BN - 1) / BN, PAIRED ? bars->pair_off[d.E] : ws.blk_off[d.E],
                      PAIRED ? max(1, wave_blocks / 2) : wave_blocks};
    const int ntiles = tl.total();
    const int nclusters = static_cast<int>(gridDim.x) / 2, cluster_id = static_cast<int>(blockIdx.x) / 2;
    auto view_of = [&](int tile, uint32_t r) {
        TileView v;
        int unit;
        tl.at(tile, v.phase, unit, v.nt);
        if (PAIRED) {
            int lo = 0, hi = d.E - 1;          // expert of pair `unit`: last e with pair_off[e] <= unit
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (bars->pair_off[mid] <= unit)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            v.e = lo;
            const int b = ws.blk_off[lo] + 2 * (unit - bars->pair_off[lo]) + static_cast<int>(r);
            v.null_half = b >= ws.blk_off[lo + 1];
            v.blk = v.null_half ? b - 1 : b;
        } else {
            v.blk = unit;
            v.e = ws.block_expert[unit];
            v.null_half = false;
        }
        return v;
    };
    auto view = [&](int tile) { return view_of(tile, rank); };
    // A bytes a CTA stages per K slice for a tile: a partly filled M-block loads only its
    // 32-row groups that hold valid rows (the UMMA still reads 128 rows; the rest only feed
    // padding rows of the tile, which are never stored); a null half loads no A
    auto a_parts = [&](const TileView &v) {
        return v.null_half ? 0 : (ws.block_rows[v.blk] + A_ROWS_PART - 1) / A_ROWS_PART;
    };
    auto a_stage_bytes = [&](int n_part) {
        return n_part < BM / A_ROWS_PART ? static_cast<uint32_t>(n_part * A_ROWS_PART * BKS) : STAGE_A_BYTES;
    };
    const int NKB1 = d.H / BK, NKB2 = d.I / BK;
    const uint32_t l1_target = static_cast<uint32_t>(EPI_WARPS * tl.NT1);
    const uint64_t deadline = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);
#ifdef CPW_TRACE
    if (threadIdx.x == 0 && blockIdx.x < TRACE_MAX_GRID)
        g_cta_span[0][blockIdx.x] = ptx::globaltimer();
#endif

    // Registers: launched at 168 per thread (384 x 168 = 64512); the producer warpgroup
    // gives (168-40) x 128 back and the two epilogue warpgroups take (232-168) x 256.
    if (warp < 4) {
        ptx::setmaxnreg_dec<40>();   // one instruction for all four warps of the group
        if (warp == 0) {
            // -------------------------------------------------------- TMA producer ----
            if (lane == 0) {
                ptx::prefetch_tmap(&maps.a1);
                ptx::prefetch_tmap(&maps.b1);
                ptx::prefetch_tmap(&maps.a2);
                ptx::prefetch_tmap(&maps.b2);
                const uint64_t pol_a = ptx::policy_evict_last();
                const uint64_t pol_b_once = ptx::policy_evict_first();    // read by one block
                const uint64_t pol_b_shared = ptx::policy_evict_normal(); // read by several
                uint32_t it = 0;
                bool ok = true;
                uint32_t tcount = 0;
                while (ok) {
                    // tiles are taken in list order: from the global counter (one CTA per tile),
                    // or round-robin over clusters (2-CTA mode, both CTAs see the same list)
                    const int tile = PAIRED ? cluster_id + static_cast<int>(tcount) * nclusters
                                            : static_cast<int>(atomicAdd(ws.hdr + HDR_TILE_NEXT, 1u));
                    const uint32_t slot = tcount % TILE_RING, sph = (tcount / TILE_RING) & 1u;
                    if (!ptx::mbar_wait(&bars->tile_empty[slot], sph ^ 1u, deadline)) {
                        ok = false;
                        break;
                    }
                    bars->tile_ring[slot] = tile < ntiles ? tile : -1;
                    ptx::mbar_arrive(&bars->tile_full[slot]);
                    if (tile >= ntiles)
                        break;
                    const TileView tv = view(tile);
                    const int phase = tv.phase, blk = tv.blk, nt = tv.nt, e = tv.e;
                    CPW_STAMP(6, tcount);
                    ++tcount;
                    // an expert's weight tile is re-read by each of its M-blocks: keep it in L2
                    // unless this block is the expert's only one
                    const uint64_t pol_b = ws.blk_off[e + 1] - ws.blk_off[e] > 1 ? pol_b_shared : pol_b_once;
                    const int n_part = a_parts(tv);
                    const bool part = n_part < BM / A_ROWS_PART;
                    const uint32_t a_bytes = a_stage_bytes(n_part);
                    // bytes the stage's full barrier waits for: this CTA's, plus (2-CTA mode,
                    // even CTA) the odd CTA's, whose loads count on the even CTA's barrier
                    uint32_t tx_bytes = a_bytes + (PAIRED ? PAIR_B_BYTES : STAGE_B_BYTES);
                    if (PAIRED && rank == 0)
                        tx_bytes += a_stage_bytes(a_parts(view_of(tile, 1))) + PAIR_B_BYTES;
                    const CUtensorMap *ta = phase == 1 ? (part ? &maps.a1p : &maps.a1)
                                                       : (part ? &maps.a2p : &maps.a2);
                    const CUtensorMap *tb = PAIRED ? (phase == 1 ? &maps.b1h : &maps.b2h)
                                                   : (phase == 1 ? &maps.b1 : &maps.b2);
                    const int nkb = phase == 1 ? NKB1 : NKB2;
                    // weight tiles are contiguous [E][NT][KB][256][128]: this tile's K block
                    // kb starts at row (tile0 + kb) * 256 of the 128-byte-wide tensor map
                    const int tile0 = (e * (phase == 1 ? tl.NT1 : tl.NT2) + nt) * nkb;
                    for (int kb = 0; kb < PREFETCH_KB && kb < nkb; ++kb)
                        for (int j = 0; j < SUBS; ++j)
                            ptx::tma_prefetch_l2_2d(tb, j * BKS, (tile0 + kb) * BN);
                    if (phase == 2 && !tv.null_half) {
                        // the act rows of this block are complete once every epilogue warp
                        // of every gate_up tile of the block has released its stores
                        for (uint32_t i = 0;; ++i) {
                            if (ptx::ld_acquire_gpu(ws.l1_done + blk) >= l1_target)
                                break;
                            if ((i & 63u) == 63u && ptx::globaltimer() > deadline) {
                                ok = false;
                                break;
                            }
                        }
                        if (!ok)
                            break;
                        CPW_STAMP(7, tcount);
                        ptx::fence_proxy_async_global();
                    }
                    for (int kb = 0; kb < nkb && ok; ++kb) {
                        if (kb + PREFETCH_KB < nkb)
                            for (int j = 0; j < SUBS; ++j)
                                ptx::tma_prefetch_l2_2d(tb, j * BKS, (tile0 + kb + PREFETCH_KB) * BN);
                        for (int j = 0; j < SUBS; ++j, ++it) {
                            const uint32_t s = it % NST, ph = (it / NST) & 1u;
                            if (!ptx::mbar_wait(&bars->empty[s], ph ^ 1u, deadline)) {
                                ok = false;
                                break;
                            }
                            uint8_t *sa = smem + s * SBYTES;
                            CPW_STAMP(0, it);
                            const int kx = kb * BK + j * BKS;
                            if (!PAIRED || rank == 0)
                                ptx::mbar_arrive_expect_tx(&bars->full[s], tx_bytes);
                            if constexpr (PAIRED) {
                                // own A rows and own half of the weight tile, counted on the
                                // even CTA's full barrier
                                const uint32_t fb = ptx::map_cluster(&bars->full[s], 0);
                                if (part) {
                                    for (int g = 0; g < n_part; ++g)
                                        ptx::tma_load_2d_pair(sa + g * A_ROWS_PART * BKS, ta, fb, kx,
                                                              blk * BM + g * A_ROWS_PART, pol_a);
                                } else {
                                    ptx::tma_load_2d_pair(sa, ta, fb, kx, blk * BM, pol_a);
                                }
                                ptx::tma_load_2d_pair(sa + STAGE_A_BYTES, tb, fb, j * BKS,
                                                      (tile0 + kb) * BN + static_cast<int>(rank) * (BN / 2), pol_b);
                            } else {
                                if (part) {
                                    for (int g = 0; g < n_part; ++g)
                                        ptx::tma_load_2d(sa + g * A_ROWS_PART * BKS, ta, &bars->full[s], kx,
                                                         blk * BM + g * A_ROWS_PART, pol_a);
                                } else {
                                    ptx::tma_load_2d(sa, ta, &bars->full[s], kx, blk * BM, pol_a);
                                }
                                ptx::tma_load_2d(sa + STAGE_A_BYTES, tb, &bars->full[s], j * BKS,
                                                 (tile0 + kb) * BN, pol_b);
                            }
                        }
                    }
                }
                if (!ok)
                    record_error(ws.hdr, DEV_TIMEOUT);
                // drain: every issued load has landed before the CTA may exit (2-CTA mode:
                // has been consumed by the UMMA, whose commit reaches both CTAs)
                const uint64_t dl = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);
                for (uint32_t i = it > NST ? it - NST : 0; i < it; ++i)
                    ptx::mbar_wait(PAIRED ? &bars->empty[i % NST] : &bars->full[i % NST], (i / NST) & 1u, dl);
            }
        } else if (warp == 1) {
            // -------------------------------------------------------- UMMA issuer -----
            // (2-CTA mode: the even CTA issues every UMMA of the pair; the odd CTA's issuer
            // only takes its tile slots)
            if (lane == 0) {
                uint32_t it = 0, pit = 0, tcount = 0;
                bool ok = true;
                const bool issuer = !PAIRED || rank == 0;
                while (ok) {
                    const uint32_t slot = tcount % TILE_RING, sph = (tcount / TILE_RING) & 1u;
                    if (!ptx::mbar_wait(&bars->tile_full[slot], sph, deadline)) {
                        ok = false;
                        break;
                    }
                    const int tile = bars->tile_ring[slot];
                    ptx::mbar_arrive(&bars->tile_empty[slot]);
                    ++tcount;
                    if (tile < 0)
                        break;
                    if (!issuer)
                        continue;
                    const TileView tv = view(tile);
                    const int nkb = tv.phase == 1 ? NKB1 : NKB2;
                    for (int kb = 0; kb < nkb && ok; ++kb, ++pit) {
                        const uint32_t buf = pit & 1u, bph = (pit >> 1) & 1u;
                        if (!ptx::mbar_wait(&bars->tempty[buf], bph ^ 1u, deadline)) {
                            ok = false;
                            break;
                        }
                        CPW_STAMP(8, pit);
                        const uint32_t dt = tmem + buf * BN;
                        // the SUBS stages of one scale block accumulate into one TMEM partial
                        for (int j = 0; j < SUBS; ++j, ++it) {
                            const uint32_t s = it % NST, ph = (it / NST) & 1u;
                            if (!ptx::mbar_wait(&bars->full[s], ph, deadline)) {
                                ok = false;
                                break;
                            }
                            CPW_STAMP(1, it);
                            ptx::tc_fence_after();
                            const uint32_t a_addr = ptx::smem_u32(smem + s * SBYTES);
                            const uint64_t adesc = ptx::kmajor_swizzled_desc<BKS>(a_addr);
                            const uint64_t bdesc = ptx::kmajor_swizzled_desc<BKS>(a_addr + STAGE_A_BYTES);
#pragma unroll
                            for (int k = 0; k < BKS / 32; ++k) {   // +32 bytes along K = +2 in the >>4 field
                                if constexpr (PAIRED)
                                    ptx::umma_f8_pair(dt, adesc + 2 * k, bdesc + 2 * k, IDESC_PAIR,
                                                      (j > 0 || k > 0) ? 1u : 0u);
                                else
                                    ptx::umma_f8(dt, adesc + 2 * k, bdesc + 2 * k, IDESC,
                                                 (j > 0 || k > 0) ? 1u : 0u);
                            }
                            if constexpr (PAIRED)
                                ptx::umma_commit_pair(&bars->empty[s], static_cast<uint16_t>(0x3));
                            else if constexpr (!EPI_RELEASES_STAGE<PAIRED>)
                                ptx::umma_commit(&bars->empty[s]);
                            CPW_STAMP(2, it);
                        }
                        if (!ok)
                            break;
                        if constexpr (PAIRED)
                            ptx::umma_commit_pair(&bars->tfull[buf], static_cast<uint16_t>(0x3));
                        else
                            ptx::umma_commit(&bars->tfull[buf]);
                    }
                }
                if (!ok)
                    record_error(ws.hdr, DEV_TIMEOUT);
                // drain: the last commit arrives once every issued MMA has completed
                if (it > 0) {
                    const uint64_t dl = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);
                    const uint32_t i = it - 1;
                    ptx::mbar_wait(&bars->empty[i % NST], (i / NST) & 1u, dl);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue --------
        ptx::setmaxnreg_inc<232>();
        const int wg = (warp - 4) >> 2;          // column half of the tile
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;           // tile row = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        uint32_t pit = 0, xcount = 0, tcount = 0;
        bool ok = true;
        while (ok) {
            const uint32_t slot = tcount % TILE_RING, sph = (tcount / TILE_RING) & 1u;
            if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&bars->tile_full[slot], sph, deadline))) {
                ok = false;
                break;
            }
            const int tile = bars->tile_ring[slot];
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(&bars->tile_empty[slot]);
            ++tcount;
            if (tile < 0)
                break;
            const TileView tv = view(tile);
            const int phase = tv.phase, blk = tv.blk, nt = tv.nt, e = tv.e;
            const int nkb = phase == 1 ? NKB1 : NKB2;
            // TMEM-empty arrivals go to the even CTA's barrier in 2-CTA mode
            const uint32_t tempty0 = PAIRED ? ptx::map_cluster(&bars->tempty[0], 0) : 0u;
            if (tv.null_half) {
                // no rows of this CTA in this tile (odd CTA, odd block count): the UMMA still
                // writes its TMEM partials, so take each one and hand it back unread
                for (int kb = 0; kb < nkb; ++kb, ++pit) {
                    const uint32_t buf = pit & 1u, bph = (pit >> 1) & 1u;
                    if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&bars->tfull[buf], bph, deadline))) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        ptx::mbar_arrive_cluster(tempty0 + buf * static_cast<uint32_t>(sizeof(uint64_t)));
                }
                continue;
            }
            const long long prow = static_cast<long long>(blk) * BM + row;
            // a warp whose 32 rows are all padding of a partly filled M-block (most warps at
            // decode) only hands each TMEM partial back: its results are never stored; so does
            // the second column half of the last down tile when H is an odd multiple of 128
            // (its weight rows are zero and lie past H)
            const bool dead = q * 32 >= ws.block_rows[blk] || (phase == 2 && nt * BN + wg * 128 >= d.H);
            const float *sfa = (phase == 1 ? ws.pool_sf : ws.act_sf) + prow;
            const float *sb0;
            const float *sb1;
            if (phase == 1) {
                sb0 = sf1 + (static_cast<long long>(e) * (2 * d.I / 128) + nt) * NKB1;              // gate
                sb1 = sf1 + (static_cast<long long>(e) * (2 * d.I / 128) + d.I / 128 + nt) * NKB1;  // up
            } else {
                sb0 = sf2 + (static_cast<long long>(e) * (d.H / 128) + 2 * nt + wg) * NKB2;
                sb1 = sb0;
            }
            if (phase == 2 && !dead) {
                // act_sf of this block is written by other CTAs in this launch: acquire the
                // block's completion counter (as the producer does before its TMA loads)
                // before the first scale read, and read the scales coherently (L2), not
                // through the read-only path.
                bool ready = true;
                for (uint32_t i = 0;; ++i) {
                    if (ptx::ld_acquire_gpu(ws.l1_done + blk) >= l1_target)
                        break;
                    if ((i & 63u) == 63u && ptx::globaltimer() > deadline) {
                        ready = false;
                        break;
                    }
                }
                if (!__all_sync(0xFFFFFFFFu, ready)) {
                    ok = false;
                    break;
                }
            }
            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j)
                acc[j] = 0.0f;
            float a_nx = 0.0f, b0_nx = 0.0f, b1_nx = 0.0f;
            if (!dead) {
                a_nx = phase == 1 ? __ldg(sfa) : __ldcg(sfa);
                b0_nx = __ldg(sb0);
                b1_nx = __ldg(sb1);
            }
            for (int kb = 0; kb < nkb; ++kb, ++pit) {
                const float s0 = a_nx * b0_nx, s1 = a_nx * b1_nx;
                if (kb + 1 < nkb && !dead) {
                    const float *na = sfa + static_cast<long long>(kb + 1) * ws.P;
                    a_nx = phase == 1 ? __ldg(na) : __ldcg(na);
                    b0_nx = __ldg(sb0 + kb + 1);
                    b1_nx = __ldg(sb1 + kb + 1);
                }
                const uint32_t buf = pit & 1u, bph = (pit >> 1) & 1u;
                // all lanes wait; the warp acts on a uniform verdict (tcgen05.ld is .aligned)
                if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&bars->tfull[buf], bph, deadline))) {
                    ok = false;
                    break;
                }
                if constexpr (EPI_RELEASES_STAGE<PAIRED>) {
                    if (warp == 4 && lane == 0)
                        ptx::mbar_arrive(&bars->empty[pit % NST]);   // this K block's operand stage
                }
                if (warp == 4 && lane == 0)
                    CPW_STAMP(3, pit);
                ptx::tc_fence_after();
                if (dead) {
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIRED)
                            ptx::mbar_arrive_cluster(tempty0 + buf * static_cast<uint32_t>(sizeof(uint64_t)));
                        else
                            ptx::mbar_arrive(&bars->tempty[buf]);
                    }
                    continue;
                }
                const uint32_t taddr = tmem + lane_base + buf * BN + wg * 128;
                // two 32-column loads in flight per round; the partial is handed back to the
                // UMMA issuer as soon as its last columns are in registers, before the last
                // 64 FMAs.  Gate/up interleave by 8: in phase 1 columns 8..15 of every 16 are
                // "up" (scale s1); in phase 2 s1 == s0.
                uint32_t r0[32], r1[32];
                ptx::tmem_ld32(taddr, r0);
                ptx::tmem_ld32(taddr + 32, r1);
                ptx::tmem_ld_wait(r0);
                ptx::reg_tie(r1);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float sj = ((j >> 3) & 1) ? s1 : s0;
                    acc[j] = fmaf(__uint_as_float(r0[j]), sj, acc[j]);
                    acc[32 + j] = fmaf(__uint_as_float(r1[j]), sj, acc[32 + j]);
                }
                ptx::tmem_ld32(taddr + 64, r0);
                ptx::tmem_ld32(taddr + 96, r1);
                ptx::tmem_ld_wait(r0);
                ptx::reg_tie(r1);
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIRED)
                        ptx::mbar_arrive_cluster(tempty0 + buf * static_cast<uint32_t>(sizeof(uint64_t)));
                    else
                        ptx::mbar_arrive(&bars->tempty[buf]);
                }
                if (warp == 4 && lane == 0)
                    CPW_STAMP(9, pit);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float sj = ((j >> 3) & 1) ? s1 : s0;
                    acc[64 + j] = fmaf(__uint_as_float(r0[j]), sj, acc[64 + j]);
                    acc[96 + j] = fmaf(__uint_as_float(r1[j]), sj, acc[96 + j]);
                }
                if (warp == 4 && lane == 0)
                    CPW_STAMP(4, pit);
            }
            if (!ok)
                break;
            if (warp == 4 && lane == 0)
                CPW_STAMP(5, pit);

            if (phase == 1) {
                // SwiGLU on the 64 (gate, up) pairs of this thread's row and column half,
                // then 1x128 requant of the row's 128 outputs of this n-tile (the two
                // column halves exchange their absolute maxima through shared memory).
                // This tail runs once per tile while the UMMA pipe waits for the next
                // tile's first promotions, so it is kept short: fast exp and reciprocal,
                // one multiply per code, and warps whose 32 rows are all padding of a
                // partly filled block skip it (they only take part in the exchange).
                const bool live = q * 32 < ws.block_rows[blk];
                float amax = 0.0f;
                if (live) {
#pragma unroll
                    for (int m = 0; m < 64; ++m) {
                        const float g = acc[(m >> 3) * 16 + (m & 7)];
                        const float u = acc[(m >> 3) * 16 + 8 + (m & 7)];
                        const float hval = __fdividef(g, 1.0f + __expf(-g)) * u;
                        acc[m] = hval;   // acc[m] is no longer needed as a gate/up input
                        amax = fmaxf(amax, fabsf(hval));
                    }
                }
                // slots of this tile's parity, behind a bounded mbarrier (a slot is rewritten
                // two phase-1 tiles later, after every thread has read it)
                const uint32_t tp = xcount & 1u;
                ++xcount;
                bars->amax[tp][wg][row] = amax;
                ptx::mbar_arrive(&bars->xbar);
                if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&bars->xbar, tp, deadline))) {
                    ok = false;
                    break;
                }
                if (live) {
                    amax = fmaxf(fmaxf(bars->amax[tp][0][row], bars->amax[tp][1][row]), 1e-4f);
                    const float sf = amax / 448.0f;
                    const float inv = 448.0f / amax;
                    uint4 *dst = reinterpret_cast<uint4 *>(ws.act + prow * d.I + nt * 128 + wg * 64);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint32_t w4[4];
#pragma unroll
                        for (int p = 0; p < 4; ++p) {
                            const int m = v * 16 + p * 4;
                            const uint32_t lo = ptx::cvt_e4m3x2(acc[m] * inv, acc[m + 1] * inv);
                            const uint32_t hi = ptx::cvt_e4m3x2(acc[m + 2] * inv, acc[m + 3] * inv);
                            w4[p] = lo | (hi << 16);
                        }
                        dst[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    if (wg == 0)
                        ws.act_sf[static_cast<long long>(nt) * ws.P + prow] = sf;
                }
                // publish: this warp's part of the block's act rows is written (the warp
                // barrier orders every lane's stores before lane 0's release)
                __syncwarp();
                ptx::fence_proxy_async_global();
                if (lane == 0)
                    ptx::red_release_add(ws.l1_done + blk, 1u);
            } else {
                // Weighted scatter of this warp's 32 rows x 128 columns (256 bytes of bf16 per
                // row, each row to its own (slot, token) row of the combine buffer).  Stored
                // straight from the TMEM layout (a lane per row), every store instruction would
                // touch 32 rows with 16 bytes each, and that stream of partial-line writes holds
                // up this SM's TMA loads of the next tile.  So each group of 8 lanes first
                // transposes its 8 rows x 8 16-byte chunks (per 128-byte half) with three
                // xor-shuffle stages; then store (h, i) has the group write row i's half h as
                // one full 128-byte line, four lines per instruction.
                const int rows = ws.block_rows[blk];
                if (!dead) {
                    float gw = 0.0f;
                    uint32_t roff = 0;   // combine row: slot * max_tokens + token
                    if (row < rows) {
                        const uint32_t t = ws.meta[prow * 3 + 1];
                        const uint32_t kk = ws.meta[prow * 3 + 2];
                        gw = __ldg(c.w + static_cast<long long>(t) * d.K + kk);
                        roff = kk * static_cast<uint32_t>(ws.max_tokens) + t;
                    }
                    uint32_t w[64];   // chunk k (columns 8k..8k+7) = w[4k..4k+3]
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(gw * acc[2 * j], gw * acc[2 * j + 1]);
                        w[j] = *reinterpret_cast<const uint32_t *>(&b2);
                    }
                    // stage b swaps bit b of (lane, chunk) wherever they differ: afterwards lane
                    // p of a group holds, in chunk slot 8h + i, chunk 8h + p of the group's row i
                    const int p8 = lane & 7, g8 = lane & ~7;
#pragma unroll
                    for (int b = 4; b >= 1; b >>= 1) {
                        const bool hi = (p8 & b) != 0;
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int c0 = 0; c0 < 8; ++c0) {
                                if (c0 & b)
                                    continue;
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    uint32_t &e0 = w[(8 * h + c0) * 4 + u];
                                    uint32_t &e1 = w[(8 * h + (c0 | b)) * 4 + u];
                                    const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, hi ? e0 : e1, b);
                                    e0 = hi ? y : e0;
                                    e1 = hi ? e1 : y;
                                }
                            }
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t ro = __shfl_sync(0xFFFFFFFFu, roff, g8 + i);
                        if (q * 32 + g8 + i < rows) {
                            uint16_t *dst = ws.combine + static_cast<long long>(ro) * d.H + nt * BN + wg * 128 + p8 * 8;
#pragma unroll
                            for (int h = 0; h < 2; ++h)
                                *reinterpret_cast<uint4 *>(dst + h * 64) =
                                    make_uint4(w[(8 * h + i) * 4], w[(8 * h + i) * 4 + 1], w[(8 * h + i) * 4 + 2],
                                               w[(8 * h + i) * 4 + 3]);
                        }
                    }
                }
            }
        }
        if (!ok)
            record_error(ws.hdr, DEV_TIMEOUT);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (PAIRED)
        ptx::cluster_sync();   // the peer neither reads this CTA's stages nor writes its TMEM any more
#ifdef CPW_TRACE
    if (threadIdx.x == 0 && blockIdx.x < TRACE_MAX_GRID)
        g_cta_span[1][blockIdx.x] = ptx::globaltimer();
#endif
    if (warp == 1) {
        ptx::tc_fence_after();
        if constexpr (PAIRED)
            ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
        else
            ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

#ifdef CPW_TRACE
cudaError_t trace_read(void *dst, size_t bytes)
{
    if (bytes != sizeof(g_trace) + sizeof(g_cta_span))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaMemcpyFromSymbol(dst, g_trace, sizeof(g_trace));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyFromSymbol(static_cast<char *>(dst) + sizeof(g_trace), g_cta_span, sizeof(g_cta_span));
}
cudaError_t trace_clear()
{
    static unsigned long long zeros[TRACE_CTAS][TRACE_EVENTS][TRACE_ITERS];
    return cudaMemcpyToSymbol(g_trace, zeros, sizeof(zeros));
}
#endif

cudaError_t launch_ffn(const FfnMaps &maps, const Dims &d, const Workspace &ws, const CallArgs &c,
                       const float *sf1, const float *sf2, int wave_blocks, int num_sms, bool paired,
                       cudaStream_t s)
{
    static int paired_grid = 0;
    static int paired_coop = 1;   // cooperative attribute accepted together with clusters
    void *kern = paired ? reinterpret_cast<void *>(ffn_kernel<true>) : reinterpret_cast<void *>(ffn_kernel<false>);
    cudaError_t e0 = ensure_max_dynamic_smem(kern, GEMM_SMEM_BYTES);
    if (e0 != cudaSuccess)
        return e0;
    FfnMaps m = maps;
    Dims dd = d;
    Workspace ww = ws;
    CallArgs cc = c;
    const float *p1 = sf1;
    const float *p2 = sf2;
    int wb = wave_blocks;
    void *args[] = {&m, &dd, &ww, &cc, &p1, &p2, &wb};
    // phase-2 tiles wait on phase-1 tiles of other CTAs, so all CTAs must be resident at once
    if (!paired)
        return cudaLaunchCooperativeKernel(kern, dim3(num_sms), dim3(GEMM_THREADS), args, GEMM_SMEM_BYTES, s);

    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = 2;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    attrs[1].id = cudaLaunchAttributeCooperative;
    attrs[1].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = GEMM_SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attrs;
    if (paired_grid == 0) {
        // every cluster resident at once: as many clusters as can be active together
        cfg.gridDim = dim3(num_sms);
        cfg.numAttrs = 1;
        int clusters = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
        if (e != cudaSuccess)
            return e;
        if (clusters < 1)
            return cudaErrorInvalidConfiguration;
        paired_grid = 2 * std::min(clusters, num_sms / 2);
    }
    cfg.gridDim = dim3(paired_grid);
    if (paired_coop) {
        cfg.numAttrs = 2;
        if (cudaLaunchKernelExC(&cfg, kern, args) == cudaSuccess)
            return cudaSuccess;
        cudaGetLastError();   // this runtime rejects cooperative + cluster: clusters alone
        paired_coop = 0;
    }
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace cpw
