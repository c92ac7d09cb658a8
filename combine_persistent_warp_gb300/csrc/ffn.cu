// ffn.cu -- the expert FFN of the fused MoE layer as ONE persistent, warp-specialised
// FP8 grouped-GEMM kernel on tcgen05 (sm_103a), for arbitrary fp32 block scales.
//
// Both expert GEMMs run in the same launch ("Mega-MoE 内核代码导读：从 Dispatch 到 WGMMA 的融合
// 流水线" §六: Linear1 gate_up then Linear2 down; "MOE融合算子", DeepGEMM MegaMoE §2 and §5:
// within an expert wave, all Linear1 tiles, then all Linear2 tiles; a Linear2 block waits
// only for the Linear1 tiles of its own M-block):
//   phase 1 tile (blk, nt):  A = gathered pool rows [P][H] e4m3 with 1x128 scales,
//                            B = gate/up-interleaved W1 tiles (contiguous 256 x 128-byte
//                            blocks per 128-deep K block) e4m3 with 128x128 scales;
//                            epilogue: SwiGLU, per-row 1x128 requant -> act [P][I]; the
//                            release warp then adds the tile to l1_done[blk].
//   phase 2 tile (blk, nt):  producer first waits for l1_done[blk] == 8 * (2I/256), then
//                            A = act [P][I] with scales, B = W2 tiles with 128x128 scales;
//                            epilogue: times the top-k gate weight, bf16, scatter through the
//                            {source, token, topk} metadata into combine[topk][T][H]
//                            ("DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析" §8.1).
// Tiles are listed wave by wave ([phase-1 tiles of the wave's blocks][phase-2 tiles of the
// same blocks]) and handed out in list order from one global counter (the producer warp of
// a CTA takes its next tile when it starts one and passes it, with the tile's expert and
// valid rows, to the other warps through a small ring), so a phase-2 wait only ever waits
// on phase-1 tiles that were handed out earlier to running CTAs: the smallest unfinished
// tile is always being worked on, and the launch needs no co-residency guarantee.
//
// The fp32 scales are arbitrary per 128-deep K block (1x128 for A rows, 128x128 for B), so
// each K block's product lands in its own TMEM partial (double-buffered, 2 x 256 columns)
// and the epilogue warps promote it into fp32 registers with the product of the two scales
// (the promotion of the first page, §8.1).  On this GPU that FP32 work slows the tensor pipe
// running beside it, and the UMMA can run only two K blocks ahead of the promotion, so every
// other piece of work is kept off the epilogue warps' path:
//
// Roles of the 12 warps of a CTA (one CTA per SM):
//   warp 0     TMA producer: A and B tiles of one 128-deep K block per stage into a 3-deep
//              ring (144 KB)
//   warp 1     UMMA issuer: four 128x256x32 tcgen05.mma per K block into a fresh TMEM partial
//   warp 2     stager: per tile, the weight scales of all its K blocks, the A-row scales of
//              its first K block and (down tiles) each row's gate weight and combine row,
//              into the tile's ring slot, so a tile starts without a dependent global load
//   warp 3     release warp: stores each tile's output rows, which the epilogue warps stage
//              in shared memory (64 KB), as full-line warp stores, so the epilogue goes on to
//              the next tile at once; then publishes a gate_up tile's SwiGLU rows to the down
//              tiles of every CTA (proxy fence + GPU-scope release add on l1_done); with the
//              top-k combine inside this kernel it counts a down tile's rows per (token,
//              n-tile) and lists the (token, n-tile) pairs the tile completed (topk_combine.cuh)
//   warps 4-11 two epilogue warpgroups, columns [0,128) and [128,256) of the tile; with the
//              in-kernel combine they reduce the previous tile's completed pairs after each
//              tile
// All waits carry a deadline; on expiry the CTA records MOE_ERR_TIMEOUT and leaves after
// draining the copies and MMAs it has in flight.
#include <cuda_bf16.h>

#include <algorithm>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "topk_combine.cuh"

namespace cpw {

namespace {

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = ptx::idesc_e4m3_f32(BM, BN);
constexpr int EPI_WARPS = 8;
constexpr int TILE_RING = 4;   // tiles the producer may run ahead of the slowest consumer
static_assert(BKS == BK, "one pipeline stage per 128-deep scale block");

#ifdef CPW_TRACE
// Development trace (compiled only with -DCPW_TRACE): SM clock stamps of two CTAs, per
// pipeline stage for the producer (0: load issue) and the UMMA issuer (1: stage full,
// 2: MMAs issued), per scale block for one epilogue warp (3: TMEM full, 4: promoted,
// 5: tile epilogue start).
// 6: producer tile start, 7: producer done waiting for a down tile's gate_up blocks,
// 8: UMMA issuer done waiting for an empty TMEM partial (per scale block), 9: the epilogue
// warp's TMEM-empty arrival (per scale block), 10: epilogue warp 4 has the tile's staged
// data (per tile), 11: stager done with a tile, 12: release warp saw a tile's act_done,
// 13: release warp done (per tile).
// g_cta_span: global-timer ns at every CTA's start and end (cross-SM comparable).
constexpr int TRACE_CTAS = 2, TRACE_EVENTS = 14, TRACE_ITERS = 4096, TRACE_MAX_GRID = 1024;
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

// Shared memory: a 3-stage operand ring of [A 16 KB | B 32 KB], then a tile's output, staged by
// the epilogue warps for the release warp's stores: a down tile's bf16 rows (128 x 512 bytes,
// 16-byte chunk c of row r at r*512 + 16*(c ^ (r % 32))) or a gate_up tile's FP8 act rows (128
// x 128 bytes, chunk c at r*128 + 16*(c ^ (r % 8))); both conflict-free for a lane per row or a
// lane per chunk.  Three stages keep a tensor-bound batch's pipe fed (four measured the same at the
// large and prefill batches and 2.5% faster at decode, which the staged stores do not pay for).
constexpr int FSTAGES = 3;
constexpr int OUT_STAGE_BYTES = BM * 2 * BN;
struct __align__(16) FfnBars {
    uint64_t full[FSTAGES];
    uint64_t empty[FSTAGES];           // epilogue warp 4, once the stage's MMAs are complete
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t xbar;                    // row-amax exchange between the two epilogue warpgroups
    uint64_t tile_full[TILE_RING];    // producer -> all: next tile, its expert and valid rows
    uint64_t tile_empty[TILE_RING];   // issuer, stager, release warp and epilogue warps are done with the slot
    uint64_t meta_ready[TILE_RING];   // stager -> epilogue: the slot's scales / row data are in place
    uint64_t act_done[TILE_RING];     // epilogue -> release warp: the slot's tile is stored (a down tile: staged)
    uint64_t out_free;                // release warp -> epilogue: the staged down tile is stored
    int tile_ring[TILE_RING];
    int tile_e[TILE_RING];
    int tile_rows[TILE_RING];
    uint32_t tmem_base;
    int abort;
    float amax[2][2][BM];              // [tile parity][column half][row]
    float sa0[TILE_RING][BM];          // A-row scales of a tile's first K block
    float sb[TILE_RING][2][MAX_KB];    // weight scales of a tile: gate | up, or down row group 2nt | 2nt+1
    float gw[TILE_RING][BM];           // down tile: gate weight of each row
    uint32_t roff[TILE_RING][BM];      // down tile: combine row (slot * max_tokens + token)
    topk::Lists<TILE_RING> tk;         // in-kernel combine: pairs completed by a down tile
    int exit_flag;
    int max_rows;                      // valid rows of the fullest M-block of the forward
};
constexpr int FFN_SMEM_BYTES = 1024 /*align slack*/ + FSTAGES * STAGE_BYTES + OUT_STAGE_BYTES + static_cast<int>(sizeof(FfnBars));
static_assert(FFN_SMEM_BYTES <= 227 * 1024, "shared memory per CTA");

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

// all 32 lanes wait; the warp acts on a uniform verdict
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t deadline)
{
    return __all_sync(0xFFFFFFFFu, ptx::mbar_wait(bar, parity, deadline));
}

}  // namespace

// FUSED: the top-k combine runs inside this kernel (topk_combine.cuh); a separate
// instantiation, so the other one carries none of its code.
template <bool FUSED>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    ffn_kernel(const __grid_constant__ FfnMaps maps, const Dims d, const Workspace ws, const CallArgs c,
               const float *__restrict__ sf1, const float *__restrict__ sf2, const int wave_blocks)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *out_stage = smem + FSTAGES * STAGE_BYTES;
    FfnBars *bars = reinterpret_cast<FfnBars *>(out_stage + OUT_STAGE_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // prologue (barriers, TMEM, tensor maps) while the routing kernel may still run
    if (threadIdx.x == 0) {
        for (int s = 0; s < FSTAGES; ++s) {
            ptx::mbar_init(&bars->full[s], 1);
            ptx::mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bars->tfull[b], 1);
            ptx::mbar_init(&bars->tempty[b], EPI_WARPS);
        }
        ptx::mbar_init(&bars->xbar, 32 * EPI_WARPS);       // every epilogue thread
        ptx::mbar_init(&bars->out_free, 1);
        for (int i = 0; i < TILE_RING; ++i) {
            ptx::mbar_init(&bars->tile_full[i], 1);
            ptx::mbar_init(&bars->tile_empty[i], 3 + EPI_WARPS);
            ptx::mbar_init(&bars->meta_ready[i], 1);
            ptx::mbar_init(&bars->act_done[i], EPI_WARPS);
            ptx::mbar_init(&bars->tk.ready[i], 1);
        }
        bars->max_rows = 0;
        ptx::fence_mbar_init();
    } else if (threadIdx.x == 32) {
        ptx::prefetch_tmap(&maps.a1);
        ptx::prefetch_tmap(&maps.b1);
        ptx::prefetch_tmap(&maps.a2);
        ptx::prefetch_tmap(&maps.b2);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&bars->tmem_base, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // the routing kernel's results are complete and visible past this point
    ptx::grid_dependency_wait();
    if (threadIdx.x == 0) {
        const uint32_t err = *reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_CALL) |
                             *reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_STICKY);
        bars->abort = err != 0;
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    if (bars->abort) {   // a device error earlier in this forward: nothing to do
        if (warp == 1)
            ptx::tmem_dealloc(tmem, TMEM_COLS);
        if (FUSED)
            ffn_cta_exit(d, ws, &bars->exit_flag);
        return;
    }
    // Who hands an operand stage back to the producer.  With M-blocks of at most 64 rows
    // (decode-sized batches) the weight stream sets the rate and most epilogue warps hold only
    // padding rows: the UMMA issuer commits the stage's release itself, so a refill never waits
    // for an epilogue warp busy promoting.  Otherwise epilogue warp 4 releases it when it sees
    // the partial, which keeps a second commit off the issuer of a tensor-bound batch.
    {
        const int nblocks = min(ws.blk_off[d.E], ws.max_blocks);
        int mr = 0;
        for (int b = threadIdx.x; b < nblocks; b += blockDim.x)
            mr = max(mr, ws.block_rows[b]);
        mr = __reduce_max_sync(0xFFFFFFFFu, mr);
        if (lane == 0 && mr > 0)
            atomicMax(&bars->max_rows, mr);
        __syncthreads();
    }
    const bool issuer_releases = bars->max_rows <= 2 * A_ROWS_PART;

    const TileList tl{(2 * d.I) / BN, (d.H + BN - 1) / BN, ws.blk_off[d.E], wave_blocks};
    const int ntiles = tl.total();
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
                const uint64_t pol_a = ptx::policy_evict_last();
                const uint64_t pol_b_once = ptx::policy_evict_first();    // read by one block
                const uint64_t pol_b_shared = ptx::policy_evict_normal(); // read by several
                uint32_t it = 0, tcount = 0;
                bool ok = true;
                // Tiles are claimed and published one ahead: while the loads of one tile are
                // issued, the next one is already in the ring, so the stager has a whole tile's
                // time to stage it.  A CTA holds at most one claimed tile it has not started,
                // and it claimed that one after the tile it works on.
                struct Claimed {
                    int tile, phase, blk, nt, e, rows, eblocks;
                };
                auto claim_and_push = [&](Claimed &t) {
                    t.tile = static_cast<int>(atomicAdd(ws.hdr + HDR_TILE_NEXT, 1u));
                    t.phase = t.blk = t.nt = t.e = t.rows = t.eblocks = 0;
                    if (t.tile < ntiles) {
                        tl.at(t.tile, t.phase, t.blk, t.nt);
                        t.e = ws.block_expert[t.blk];
                        t.rows = ws.block_rows[t.blk];
                        t.eblocks = ws.blk_off[t.e + 1] - ws.blk_off[t.e];
                    }
                    const uint32_t slot = tcount % TILE_RING, sph = (tcount / TILE_RING) & 1u;
                    ++tcount;
                    if (!ptx::mbar_wait(&bars->tile_empty[slot], sph ^ 1u, deadline))
                        return false;
                    bars->tile_ring[slot] = t.tile < ntiles ? t.tile : -1;
                    bars->tile_e[slot] = t.e;
                    bars->tile_rows[slot] = t.rows;
                    ptx::mbar_arrive(&bars->tile_full[slot]);
                    return true;
                };
                Claimed cur, nxt;
                ok = claim_and_push(cur);
                while (ok && cur.tile < ntiles) {
                    const int phase = cur.phase, blk = cur.blk, nt = cur.nt, e = cur.e, rows = cur.rows;
                    bool pushed = false;   // the next tile is published after this tile's first stage
                    CPW_STAMP(6, tcount - 1);
                    // an expert's weight tile is re-read by each of its M-blocks: keep it in L2
                    // unless this block is the expert's only one
                    const uint64_t pol_b = cur.eblocks > 1 ? pol_b_shared : pol_b_once;
                    // A rows in one load per K block: the first 32 or 64 rows of a partly filled
                    // M-block that holds no more valid rows, else all 128 (the UMMA reads 128
                    // rows; the rest only feed padding rows, never stored)
                    const int n_part = max(1, (rows + A_ROWS_PART - 1) / A_ROWS_PART);
                    const uint32_t a_bytes = n_part <= 2 ? static_cast<uint32_t>(n_part * A_ROWS_PART * BKS) : STAGE_A_BYTES;
                    const uint32_t tx_bytes = a_bytes + STAGE_B_BYTES;
                    const CUtensorMap *ta = phase == 1 ? (n_part == 1 ? &maps.a1p : n_part == 2 ? &maps.a1h : &maps.a1)
                                                       : (n_part == 1 ? &maps.a2p : n_part == 2 ? &maps.a2h : &maps.a2);
                    const CUtensorMap *tb = phase == 1 ? &maps.b1 : &maps.b2;
                    const int nkb = phase == 1 ? NKB1 : NKB2;
                    // weight tiles are contiguous [E][NT][KB][256][128]: this tile's K block
                    // kb starts at row (tile0 + kb) * 256 of the 128-byte-wide tensor map
                    const int tile0 = (e * (phase == 1 ? tl.NT1 : tl.NT2) + nt) * nkb;
                    if (phase == 2) {
                        // the act rows and scales of this block are complete once every
                        // gate_up tile of the block has been published by its release warp
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
                        CPW_STAMP(7, tcount - 1);
                        ptx::fence_proxy_async_global();
                    }
                    for (int kb = 0; kb < nkb && ok; ++kb, ++it) {
                        const uint32_t s = it % FSTAGES, ph = (it / FSTAGES) & 1u;
                        if (!ptx::mbar_wait(&bars->empty[s], ph ^ 1u, deadline)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sa = smem + s * STAGE_BYTES;
                        CPW_STAMP(0, it);
                        ptx::mbar_arrive_expect_tx(&bars->full[s], tx_bytes);
                        ptx::tma_load_2d(sa, ta, &bars->full[s], kb * BK, blk * BM, pol_a);
                        ptx::tma_load_2d(sa + STAGE_A_BYTES, tb, &bars->full[s], 0, (tile0 + kb) * BN, pol_b);
                        if (!pushed) {
                            pushed = true;
                            ok = claim_and_push(nxt);
                        }
                    }
                    if (ok && !pushed)
                        ok = claim_and_push(nxt);
                    cur = nxt;
                }
                if (!ok)
                    record_error(ws.hdr, DEV_TIMEOUT);
                // drain: every issued load has landed before the CTA may exit
                const uint64_t dl = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);
                for (uint32_t i = it > FSTAGES ? it - FSTAGES : 0; i < it; ++i)
                    ptx::mbar_wait(&bars->full[i % FSTAGES], (i / FSTAGES) & 1u, dl);
            }
        } else if (warp == 1) {
            // -------------------------------------------------------- UMMA issuer -----
            if (lane == 0) {
                uint32_t it = 0, tcount = 0;
                bool ok = true;
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
                    int phase, blk, nt;
                    tl.at(tile, phase, blk, nt);
                    const int nkb = phase == 1 ? NKB1 : NKB2;
                    // one stage and one TMEM partial per K block (partial = it & 1)
                    for (int kb = 0; kb < nkb && ok; ++kb, ++it) {
                        const uint32_t buf = it & 1u, bph = (it >> 1) & 1u;
                        if (!ptx::mbar_wait(&bars->tempty[buf], bph ^ 1u, deadline)) {
                            ok = false;
                            break;
                        }
                        CPW_STAMP(8, it);
                        const uint32_t s = it % FSTAGES, ph = (it / FSTAGES) & 1u;
                        if (!ptx::mbar_wait(&bars->full[s], ph, deadline)) {
                            ok = false;
                            break;
                        }
                        CPW_STAMP(1, it);
                        ptx::tc_fence_after();
                        const uint32_t dt = tmem + buf * BN;
                        const uint32_t a_addr = ptx::smem_u32(smem + s * STAGE_BYTES);
                        const uint64_t adesc = ptx::kmajor_swizzled_desc<BKS>(a_addr);
                        const uint64_t bdesc = ptx::kmajor_swizzled_desc<BKS>(a_addr + STAGE_A_BYTES);
#pragma unroll
                        for (int k = 0; k < BKS / 32; ++k)   // +32 bytes along K = +2 in the >>4 field
                            ptx::umma_f8(dt, adesc + 2 * k, bdesc + 2 * k, IDESC, k > 0 ? 1u : 0u);
                        CPW_STAMP(2, it);
                        // the epilogue warps, once they see the partial, also release the stage
                        // (or, for small M-blocks, this commit does)
                        ptx::umma_commit(&bars->tfull[buf]);
                        if (issuer_releases)
                            ptx::umma_commit(&bars->empty[s]);
                    }
                }
                if (!ok)
                    record_error(ws.hdr, DEV_TIMEOUT);
                // drain: the last commit arrives once every issued MMA has completed
                if (it > 0) {
                    const uint64_t dl = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);
                    const uint32_t i = it - 1;
                    ptx::mbar_wait(&bars->tfull[i & 1u], (i >> 1) & 1u, dl);
                }
            }
        } else if (warp == 2) {
            // -------------------------------------------------------- stager ----------
            // For each published tile: the weight scales of all its K blocks (phase 1: the
            // gate row group nt and the up row group I/128 + nt; phase 2: the down weight's
            // row groups 2nt and 2nt+1, the second one only below H), the A-row scales of its
            // first K block, and for a down tile each valid row's gate weight and combine row,
            // into the tile's ring slot.  A down tile's A-row scales are SwiGLU scales that
            // gate_up tiles of other CTAs write: this warp first acquires the block's l1_done
            // count, and the epilogue, which waits for this warp's barrier, then reads the later
            // K blocks' scales coherently.
            uint32_t tcount = 0;
            bool ok = true;
            while (ok) {
                const uint32_t slot = tcount % TILE_RING, sph = (tcount / TILE_RING) & 1u;
                ++tcount;
                if (!warp_wait(&bars->tile_full[slot], sph, deadline)) {
                    ok = false;
                    break;
                }
                const int tile = bars->tile_ring[slot];
                const int e = bars->tile_e[slot];
                const int rows = bars->tile_rows[slot];
                if (tile >= 0) {
                    int phase, blk, nt;
                    tl.at(tile, phase, blk, nt);
                    const long long row0 = static_cast<long long>(blk) * BM;
                    constexpr int RPL = BM / 32;   // rows per lane
                    if (phase == 1) {
                        const float *g = sf1 + (static_cast<long long>(e) * (2 * d.I / 128) + nt) * NKB1;
                        const float *u = g + static_cast<long long>(d.I / 128) * NKB1;
                        float a0[RPL];
#pragma unroll
                        for (int j = 0; j < RPL; ++j)
                            a0[j] = __ldg(ws.pool_sf + row0 + lane + 32 * j);
                        for (int k = lane; k < NKB1; k += 32) {
                            bars->sb[slot][0][k] = __ldg(g + k);
                            bars->sb[slot][1][k] = __ldg(u + k);
                        }
#pragma unroll
                        for (int j = 0; j < RPL; ++j)
                            bars->sa0[slot][lane + 32 * j] = a0[j];
                    } else {
                        // row data and weight scales first (they do not depend on other CTAs),
                        // every load of a round issued before its results are used
                        const float *g0 = sf2 + (static_cast<long long>(e) * (d.H / 128) + 2 * nt) * NKB2;
                        const bool second = (2 * nt + 1) * 128 < d.H;
                        uint32_t t[RPL], kk[RPL];
#pragma unroll
                        for (int j = 0; j < RPL; ++j) {
                            const int r = lane + 32 * j;
                            t[j] = r < rows ? __ldg(ws.meta + (row0 + r) * 3 + 1) : 0u;
                            kk[j] = r < rows ? __ldg(ws.meta + (row0 + r) * 3 + 2) : 0u;
                        }
                        for (int k = lane; k < NKB2; k += 32) {
                            bars->sb[slot][0][k] = __ldg(g0 + k);
                            bars->sb[slot][1][k] = second ? __ldg(g0 + NKB2 + k) : 0.0f;
                        }
                        float gw[RPL];
#pragma unroll
                        for (int j = 0; j < RPL; ++j)
                            gw[j] = lane + 32 * j < rows ? __ldg(c.w + static_cast<long long>(t[j]) * d.K + kk[j]) : 0.0f;
#pragma unroll
                        for (int j = 0; j < RPL; ++j) {
                            bars->gw[slot][lane + 32 * j] = gw[j];
                            bars->roff[slot][lane + 32 * j] = kk[j] * static_cast<uint32_t>(ws.max_tokens) + t[j];
                        }
                        // then the first K block's A-row scales: SwiGLU scales written by the
                        // gate_up tiles of this block, published through l1_done
                        bool ready = true;
                        if (lane == 0) {
                            for (uint32_t i = 0;; ++i) {
                                if (ptx::ld_acquire_gpu(ws.l1_done + blk) >= l1_target)
                                    break;
                                if ((i & 63u) == 63u && ptx::globaltimer() > deadline) {
                                    ready = false;
                                    break;
                                }
                            }
                        }
                        // the other lanes' reads below are ordered after lane 0's acquire by the
                        // warp barrier
                        __syncwarp();
                        if (!__shfl_sync(0xFFFFFFFFu, ready, 0)) {
                            ok = false;
                            break;
                        }
                        float a0[RPL];
#pragma unroll
                        for (int j = 0; j < RPL; ++j)
                            a0[j] = __ldcg(ws.act_sf + row0 + lane + 32 * j);
#pragma unroll
                        for (int j = 0; j < RPL; ++j)
                            bars->sa0[slot][lane + 32 * j] = a0[j];
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    CPW_STAMP(11, tcount - 1);
                    ptx::mbar_arrive(&bars->meta_ready[slot]);
                    ptx::mbar_arrive(&bars->tile_empty[slot]);
                }
                if (tile < 0)
                    break;
            }
            if (!ok && lane == 0)
                record_error(ws.hdr, DEV_TIMEOUT);
        } else {
            // -------------------------------------------------------- release warp ----
            // The epilogue warps arrive on the slot's act_done barrier when they are done with
            // a tile: its output rows are staged in shared memory (and a gate_up tile's row
            // scales stored).  This warp stores the rows and hands the buffer back; for a
            // gate_up tile lane 0 then publishes them for the down tiles of every CTA: the
            // CTA-scope barriers order the stores before this thread's GPU-scope release
            // (release is cumulative), and the proxy fence covers the TMA loads that read them.  With the combine inside this kernel the warp
            // then counts the down tile's rows per (token, n-tile) (its own stores, fenced
            // first) and lists the pairs the tile completed for the epilogue warps, which
            // reduce them at the end of their next tile (topk_combine.cuh).
            uint32_t tcount = 0;
            bool ok = true;
            while (ok) {
                const uint32_t slot = tcount % TILE_RING, sph = (tcount / TILE_RING) & 1u;
                ++tcount;
                if (!warp_wait(&bars->tile_full[slot], sph, deadline)) {
                    ok = false;
                    break;
                }
                const int tile = bars->tile_ring[slot];
                if (tile < 0) {
                    __syncwarp();
                    if (lane == 0)
                        ptx::mbar_arrive(&bars->tile_empty[slot]);
                    break;
                }
                if (!warp_wait(&bars->act_done[slot], sph, deadline)) {
                    ok = false;
                    break;
                }
                if (lane == 0)
                    CPW_STAMP(12, tcount - 1);
                int phase, blk, nt;
                tl.at(tile, phase, blk, nt);
                if (phase == 1) {
                    // the staged act rows: lanes 8i..8i+7 store row 4k+i's 128 bytes (a full line)
                    const int rows = bars->tile_rows[slot];
                    const int c = lane & 7;
                    for (int r = lane >> 3; r < rows; r += 4) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(out_stage + r * 128 + ((c ^ (r & 7)) << 4));
                        *reinterpret_cast<uint4 *>(ws.act + (static_cast<long long>(blk) * BM + r) * d.I + nt * 128 + c * 16) = v;
                    }
                    __syncwarp();
                    if (lane == 0) {
                        ptx::mbar_arrive(&bars->out_free);
                        ptx::fence_proxy_async_global();
                        ptx::red_release_add(ws.l1_done + blk, static_cast<uint32_t>(EPI_WARPS));
                    }
                }
                if (phase == 2) {
                    // the staged down tile: lane l stores 16-byte chunk l of each valid row, the
                    // warp one full 512-byte row per instruction (only its first half when the
                    // tile's second column half lies past H); then the buffer is free again
                    const int rows = bars->tile_rows[slot];
                    const bool half2 = nt * BN + 128 < d.H;
                    const bool mine = lane < 16 || half2;
                    uint16_t *dst0 = ws.combine + nt * BN + lane * 8;
#pragma unroll 4
                    for (int r = 0; r < rows; ++r) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(out_stage + r * (2 * BN) + ((lane ^ (r & 31)) << 4));
                        if (mine)
                            *reinterpret_cast<uint4 *>(dst0 + static_cast<long long>(bars->roff[slot][r]) * d.H) = v;
                    }
                    __syncwarp();
                    if (lane == 0)
                        ptx::mbar_arrive(&bars->out_free);
                }
                if (FUSED) {
                    const int n = phase == 2 ? topk::count_rows(d, ws, static_cast<long long>(blk) * BM,
                                                                bars->tile_rows[slot], nt, bars->tk.tok[slot],
                                                                bars->tk.mask[slot], lane)
                                             : 0;
                    __syncwarp();
                    if (lane == 0) {
                        bars->tk.n[slot] = n;
                        bars->tk.nt[slot] = nt;
                        ptx::mbar_arrive(&bars->tk.ready[slot]);
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    CPW_STAMP(13, tcount - 1);
                    ptx::mbar_arrive(&bars->tile_empty[slot]);
                }
            }
            if (!ok && lane == 0)
                record_error(ws.hdr, DEV_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ epilogue --------
        ptx::setmaxnreg_inc<232>();
        const int wg = (warp - 4) >> 2;          // column half of the tile
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;           // tile row = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        uint32_t it = 0, xcount = 0, tcount = 0, dcount = 0;   // dcount: tiles staged
        bool ok = true;
        // in-kernel combine: the (token, n-tile) pairs the release warp listed for the previous
        // tile are reduced by the eight epilogue warps at the end of the next one
        int prev = -1;   // ring slot of the previous tile, -1 before the first
        uint32_t prev_ph = 0;
        auto reduce_listed = [&](int sl, uint32_t ph) {
            if (!warp_wait(&bars->tk.ready[sl], ph, deadline))
                return false;
            const int n = bars->tk.n[sl];
            if (n > 0)
                topk::reduce(d, ws, c, bars->tk.tok[sl], bars->tk.mask[sl], n, bars->tk.nt[sl], warp - 4, EPI_WARPS,
                             lane);
            return true;
        };
        while (ok) {
            const uint32_t slot = tcount % TILE_RING, sph = (tcount / TILE_RING) & 1u;
            ++tcount;
            if (!warp_wait(&bars->tile_full[slot], sph, deadline)) {
                ok = false;
                break;
            }
            const int tile = bars->tile_ring[slot];
            const int rows = bars->tile_rows[slot];
            if (tile < 0) {
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(&bars->tile_empty[slot]);
                if (FUSED && prev >= 0 && !reduce_listed(prev, prev_ph))
                    ok = false;
                break;
            }
            int phase, blk, nt;
            tl.at(tile, phase, blk, nt);
            const int nkb = phase == 1 ? NKB1 : NKB2;
            const long long prow = static_cast<long long>(blk) * BM + row;
            // a warp whose 32 rows are all padding of a partly filled M-block (most warps at
            // decode) only hands each TMEM partial back: its results are never stored; so does
            // the second column half of the last down tile when H is an odd multiple of 128
            // (its weight rows are zero and lie past H)
            const bool dead = q * 32 >= rows || (phase == 2 && nt * BN + wg * 128 >= d.H);
            // the tile's weight scales (and down-tile row data), staged by warp 2
            if (!warp_wait(&bars->meta_ready[slot], sph, deadline)) {
                ok = false;
                break;
            }
            if (warp == 4 && lane == 0)
                CPW_STAMP(10, tcount - 1);
            const float *sb0 = bars->sb[slot][phase == 1 ? 0 : wg];
            const float *sb1 = bars->sb[slot][phase == 1 ? 1 : wg];
            // A-row scales: the first K block's from the slot, the next one's loaded a K block
            // ahead ([K block][P] floats; a down tile's were acquired by the stager)
            const float *sfa = (phase == 1 ? ws.pool_sf : ws.act_sf) + prow;
            float a_nx = bars->sa0[slot][row];
            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j)
                acc[j] = 0.0f;
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const uint32_t s = it % FSTAGES;
                const uint32_t buf = it & 1u, bph = (it >> 1) & 1u;
                const float s0 = a_nx * sb0[kb], s1 = a_nx * sb1[kb];
                if (kb + 1 < nkb && !dead) {
                    const float *na = sfa + static_cast<long long>(kb + 1) * ws.P;
                    a_nx = phase == 1 ? __ldg(na) : __ldcg(na);
                }
                if (!warp_wait(&bars->tfull[buf], bph, deadline)) {
                    ok = false;
                    break;
                }
                // the MMAs that read this K block's operand stage are complete
                if (!issuer_releases && warp == 4 && lane == 0)
                    ptx::mbar_arrive(&bars->empty[s]);
                if (warp == 4 && lane == 0)
                    CPW_STAMP(3, it);
                ptx::tc_fence_after();
                if (dead) {
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        ptx::mbar_arrive(&bars->tempty[buf]);
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
                if (lane == 0)
                    ptx::mbar_arrive(&bars->tempty[buf]);
                if (warp == 4 && lane == 0)
                    CPW_STAMP(9, it);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float sj = ((j >> 3) & 1) ? s1 : s0;
                    acc[64 + j] = fmaf(__uint_as_float(r0[j]), sj, acc[64 + j]);
                    acc[96 + j] = fmaf(__uint_as_float(r1[j]), sj, acc[96 + j]);
                }
                if (warp == 4 && lane == 0)
                    CPW_STAMP(4, it);
            }
            if (!ok)
                break;
            if (warp == 4 && lane == 0)
                CPW_STAMP(5, it);

            if (phase == 1) {
                // SwiGLU on the 64 (gate, up) pairs of this thread's row and column half,
                // then 1x128 requant of the row's 128 outputs of this n-tile (the two
                // column halves exchange their absolute maxima through shared memory).
                // This tail runs once per tile while the UMMA pipe waits for the next
                // tile's first promotions, so it is kept short: fast exp and reciprocal,
                // one multiply per code, and warps whose 32 rows are all padding of a
                // partly filled block skip it (they only take part in the exchange).
                const bool live = q * 32 < rows;
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
                if (!warp_wait(&bars->xbar, tp, deadline)) {
                    ok = false;
                    break;
                }
                // the act rows go through the staging buffer too (row r's 128 bytes at r*128,
                // 16-byte chunk c at 16*(c ^ (r % 8))): the release warp stores them as full
                // lines before it publishes the tile
                if (!warp_wait(&bars->out_free, (dcount & 1u) ^ 1u, deadline)) {
                    ok = false;
                    break;
                }
                ++dcount;
                if (live) {
                    amax = fmaxf(fmaxf(bars->amax[tp][0][row], bars->amax[tp][1][row]), 1e-4f);
                    const float sf = amax / 448.0f;
                    const float inv = 448.0f / amax;
                    uint8_t *orow = out_stage + row * 128;
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
                        *reinterpret_cast<uint4 *>(orow + (((wg * 4 + v) ^ (row & 7)) << 4)) =
                            make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    if (wg == 0)
                        ws.act_sf[static_cast<long long>(nt) * ws.P + prow] = sf;
                }
            } else {
                // Weighted scatter of this warp's 32 rows x 128 columns: bf16(gate weight x row)
                // into the output staging buffer (row r's 512 bytes, this column half's 16-byte
                // chunks at 16*(c ^ (r % 32)) for c = 16*wg .. 16*wg+15); the release warp stores
                // each staged row with one full-line warp store into its (slot, token) combine
                // row while these warps go on with the next tile.  The buffer is rewritten once
                // the release warp has stored the previous tile.
                if (!warp_wait(&bars->out_free, (dcount & 1u) ^ 1u, deadline)) {
                    ok = false;
                    break;
                }
                ++dcount;
                if (!dead) {
                    const float gw = bars->gw[slot][row];
                    uint8_t *orow = out_stage + row * (2 * BN);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        uint32_t w4[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const __nv_bfloat162 b2 =
                                __floats2bfloat162_rn(gw * acc[8 * k + 2 * u], gw * acc[8 * k + 2 * u + 1]);
                            w4[u] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        const int ch = (wg * 16 + k) ^ (row & 31);
                        *reinterpret_cast<uint4 *>(orow + ch * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            }
            // done with the slot: the release warp publishes a gate_up tile's rows, and the
            // slot's staged data may be overwritten
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(&bars->act_done[slot]);
                ptx::mbar_arrive(&bars->tile_empty[slot]);
            }
            if (FUSED) {
                if (prev >= 0 && !reduce_listed(prev, prev_ph)) {
                    ok = false;
                    break;
                }
                prev = static_cast<int>(slot);
                prev_ph = sph;
            }
        }
        if (!ok)
            record_error(ws.hdr, DEV_TIMEOUT);
    }

    ptx::tc_fence_before();
    __syncthreads();
#ifdef CPW_TRACE
    if (threadIdx.x == 0 && blockIdx.x < TRACE_MAX_GRID)
        g_cta_span[1][blockIdx.x] = ptx::globaltimer();
#endif
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
    if (FUSED)
        ffn_cta_exit(d, ws, &bars->exit_flag);
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
                       const float *sf1, const float *sf2, int wave_blocks, int num_sms, cudaStream_t s)
{
    const void *kern = c.fused_combine ? reinterpret_cast<const void *>(ffn_kernel<true>)
                                       : reinterpret_cast<const void *>(ffn_kernel<false>);
    cudaError_t e0 = ensure_max_dynamic_smem(kern, FFN_SMEM_BYTES);
    if (e0 != cudaSuccess)
        return e0;
    return c.fused_combine ? launch_programmatic(ffn_kernel<true>, num_sms, GEMM_THREADS, FFN_SMEM_BYTES, s, maps, d,
                                                 ws, c, sf1, sf2, wave_blocks)
                           : launch_programmatic(ffn_kernel<false>, num_sms, GEMM_THREADS, FFN_SMEM_BYTES, s, maps, d,
                                                 ws, c, sf1, sf2, wave_blocks);
}

}  // namespace cpw
