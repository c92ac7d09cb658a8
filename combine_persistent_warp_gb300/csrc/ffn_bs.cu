// ffn_bs.cu -- the expert FFN of the fused MoE layer for power-of-two (UE8M0) block scales:
// one persistent, warp-specialised kernel on the block-scaled tcgen05 UMMA
// (kind::mxf8f6f4.block_scale.scale_vec::1X, sm_103a).
//
// Same tile list, phases and memory layouts as the fp32-scale kernel in ffn.cu (gate_up
// tiles then down tiles per wave, SwiGLU + 1x128 requant in the gate_up epilogue, weighted
// bf16 scatter in the down epilogue).  The difference is where the scales are applied: every
// scale is a power of two, so the tensor core applies them itself (one UE8M0 scale per row
// of A and per N-row of B for each 32-deep K slice) and accumulates the whole K range of a
// tile in TMEM.  There is no per-128-K promotion on the CUDA cores: the UMMA issuer runs the
// K loop back to back and the epilogue reads each tile's accumulator once.  This is the
// hardware block-scaled path of the pages' SM100 design ("DeepGEMM Mega MoE 对称内存
// （Symmetric Memory）深度分析" §8.1 and the UE8M0 scale format it names); with arbitrary fp32
// scales the layer uses ffn.cu instead.
//
// Scale factors reach TMEM through shared memory, once per group of four 128-deep K blocks:
// with a group's first stage the producer bulk-copies a 512-byte A block (the 128 rows'
// scale words, row r at byte 16*(r%32) + 4*(r/32)) and a 1 KB B block (two 512-byte halves;
// tile column n at 512*(n/128) + 16*(n%32) + 4*((n%128)/32)), each word holding the UE8M0
// bytes of the group's four K blocks (byte j = K block 4g + j), into a ring of three scale
// slots.  The UMMA issuer copies them into the group's TMEM slot with tcgen05.cp
// 32x128b.warpx4 (every lane quarter gets the same 32 lanes); the UMMA reads row m's scale at lane m, column base + m/32, and tile
// column n's at lane 32*q + n%32, column base + n/32, byte = the instruction's scale id, here
// K block % 4 for all four 32-deep UMMAs of a K block.  Copying once per group instead of
// once per K block took the issue sequence from ~830 to ~700 cycles per K block.
//
// MXFP4 weights (FP4 = true): the weight tiles are packed E2M1 (64 bytes per row and 128-deep
// K block) with one UE8M0 scale per row and 32-deep K slice (the OCP Microscaling block).  TMA
// loads them with the 16U4_ALIGN16B element type, which widens every 8 bytes (16 values) to a
// 16-byte slot in shared memory: the 128-byte-row image the UMMA reads for a 4-bit operand of
// kind::mxf8f6f4 (B format E2M1), at the same swizzle and descriptor as an e4m3 tile, while
// only the packed 16 KB per stage comes from memory.  The B scale words then change every K
// block (byte j = the scale of the block's j-th 32-deep slice, instruction B scale id = j):
// the group's B scales are its K blocks' 1 KB blocks, consecutive in memory, so they still
// come in one bulk copy per group (up to 4 KB); the issuer copies each K block's to its own
// columns of the group's TMEM slot just before that K block's UMMAs.
//
// Copies per K block: each load, bulk or tiled, that the producer issues costs the SM's TMA
// unit more than its bytes at decode sizes, where a weight tile moves only 16 KB (MXFP4).  So
// a K block stages A in one load (32, 64 or 128 rows, whichever first covers the M-block's
// valid rows) and the scales come once per group.
//
// Roles (one CTA per SM, 12 warps): warp 0 TMA producer (A and B of a 128-deep K block per
// stage, 4 or 5 stages, and a scale group's blocks with its first stage); warp 1 UMMA issuer
// (a group's scale copies, then 4 block-scaled UMMAs per stage into one 256-column TMEM
// accumulator); warp 2 dependency warp (a down
// tile's gate_up completion count); warp 3, with the top-k combine inside this kernel, counts
// each stored down tile's rows per (token, n-tile) and lists the pairs it completed
// (topk_combine.cuh); warps 4-11 epilogue (two warpgroups, columns [0,128) / [128,256)): one
// TMEM read per tile, then SwiGLU + UE8M0 requant (phase 1) or the weighted scatter (phase 2),
// and with the in-kernel combine the reduce of the previous tile's completed pairs.  TMEM:
// accumulator columns 0-255, scale group slots 256 + 40*j.  All waits carry a deadline
// (MOE_ERR_TIMEOUT).
#include <cuda_bf16.h>

#include <algorithm>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "topk_combine.cuh"

namespace cpw {

namespace {

constexpr uint32_t TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;
constexpr int TILE_RING = 4;
constexpr int SF_GROUP = 4;               // K blocks per scale group (bytes of an FP8 scale word)
constexpr uint32_t SFA_BYTES = 512, SFB_BYTES = 1024;
// Scale groups in shared memory: a ring of SF_SLOTS slots of [A 512 | B up to 4 x 1 KB], each
// filled by one bulk copy per kind with a group's first stage.  The producer refills a slot
// once the UMMAs of the last K block that read it have completed (that K block's release in
// the stage ring, waited for only when it is less than a ring's length back).
constexpr int SF_SLOTS = 3;
constexpr uint32_t SF_SLOT_BYTES = SFA_BYTES + SF_GROUP * SFB_BYTES;
// Scale groups in TMEM: group slot j at columns SF_COL + SF_TCOLS*j (A: +0..3; B: +4..11, or
// with MXFP4 weights K block i of the group at +4+8i..+11+8i)
constexpr uint32_t SF_COL = 256, SF_TCOLS = 40;
static_assert(BKS == BK, "the block-scaled kernel stages whole 128-deep K blocks");
// Stage ring layouts.  Standard: STAGES stages of [A 16 KB | B 32 KB].  Compact, when no M-block
// of the forward holds more than 64 rows (decode-sized batches): NST_MAX stages of [A 8 KB |
// B 32 KB] in about the same space, i.e. one more weight tile in flight per SM.  The UMMA
// still reads 128 A rows from the stage base; rows 64-127 then lie in the stage's own B tile
// and only feed padding rows of the accumulator, which are never stored.
constexpr int NST_MAX = 5;
constexpr uint32_t COMPACT_A_BYTES = 2 * A_ROWS_PART * BKS;
constexpr uint32_t COMPACT_STAGE_BYTES = COMPACT_A_BYTES + STAGE_B_BYTES;
constexpr int RING_BYTES = STAGES * STAGE_BYTES > NST_MAX * static_cast<int>(COMPACT_STAGE_BYTES)
                               ? STAGES * STAGE_BYTES
                               : NST_MAX * static_cast<int>(COMPACT_STAGE_BYTES);
static_assert(NST_MAX >= STAGES, "the compact ring has at least as many stages");
static_assert(COMPACT_STAGE_BYTES % 1024 == 0 && COMPACT_A_BYTES % 1024 == 0, "128-byte swizzle atoms");
static_assert(SF_COL + SF_TCOLS * NST_MAX <= TMEM_COLS, "scale slots exceed TMEM");
static_assert(4 + 8 * SF_GROUP <= SF_TCOLS, "a group's scale columns");

// block-scaled instruction descriptor: B scale id (byte of the scale word) at bits 4-5, A
// format e4m3 (0) at bits 7-9, B format at bits 10-12 (e4m3 = 0, E2M1 = 5), K-major A and B,
// N>>3 at 17-22, UE8M0 scales (bit 23), M>>4 at 24-28, A scale id at 29-30
template <int M, bool FP4>
__device__ __forceinline__ uint32_t idesc_bs(int a_sf_id, int b_sf_id)
{
    return (static_cast<uint32_t>(b_sf_id) << 4) | ((FP4 ? 5u : 0u) << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
           (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) | (static_cast<uint32_t>(a_sf_id) << 29);
}

// D (128 rows) (+)= A x B^T with the A and B scale factors read from this CTA's TMEM
__device__ __forceinline__ void umma_bs(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
                 "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
                 : "memory");
}

// shared -> TMEM copy of 32 rows x 16 bytes (no swizzle, 8-row groups 128 B apart) into
// four columns of every lane quarter
__device__ __forceinline__ void sf_copy(uint32_t taddr, uint32_t smem_addr)
{
    const uint64_t desc = static_cast<uint64_t>((smem_addr >> 4) & 0x3FFF) | (static_cast<uint64_t>(8) << 16) |
                          (static_cast<uint64_t>(128 >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

// the smallest power of two >= v for a positive normal fp32 v (exact)
__device__ __forceinline__ float pow2_ceil(float v)
{
    const uint32_t b = __float_as_uint(v);
    return (b & 0x007FFFFFu) == 0u ? v : __uint_as_float((b & 0x7F800000u) + 0x00800000u);
}

struct __align__(8) BsBars {
    uint64_t full[NST_MAX];
    uint64_t empty[NST_MAX];
    uint64_t tfull;
    uint64_t tempty;
    uint64_t xbar;
    uint64_t tile_full[TILE_RING];
    uint64_t tile_empty[TILE_RING];
    uint64_t dep[TILE_RING];   // dependency warp -> producer: this slot's tile may be loaded
    uint64_t act_done[TILE_RING];   // in-kernel combine: epilogue -> counting warp, tile stored
    int tile_ring[TILE_RING];
    uint32_t tmem_base;
    int abort;
    int exit_flag;
    int max_rows;   // valid rows of the fullest M-block of the forward
    float amax[2][2][BM];
    topk::Lists<TILE_RING> tk;   // in-kernel combine: pairs completed by a down tile
};

struct BsTiles {
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

// Tile of the list: phase, n-tile, M-block and its expert.
struct BsView {
    int phase, nt, blk, e;
};

}  // namespace

// FUSED: the top-k combine runs inside this kernel (topk_combine.cuh); a separate
// instantiation, so the other one carries none of its code.
template <bool FP4, bool FUSED>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    ffn_bs_kernel(const __grid_constant__ FfnMaps maps, const Dims d,
                  const Workspace ws, const CallArgs c, const uint8_t *__restrict__ sfb1,
                  const uint8_t *__restrict__ sfb2, const int wave_blocks)
{
    // weight bytes a stage's TMA brings from memory (packed E2M1: half the shared-memory image)
    constexpr uint32_t B_TX = STAGE_B_BYTES / (FP4 ? 2u : 1u);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    BsBars *bars = reinterpret_cast<BsBars *>(smem + RING_BYTES);
    uint8_t *sf_smem = smem + RING_BYTES + 8192;   // [SF_SLOTS][A 512 | B 4 x 1 KB]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // prologue (barriers, TMEM, tensor maps) while the routing kernel may still run
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST_MAX; ++s) {
            ptx::mbar_init(&bars->full[s], 1);
            ptx::mbar_init(&bars->empty[s], 1);
        }
        bars->max_rows = 0;
        ptx::mbar_init(&bars->tfull, 1);
        ptx::mbar_init(&bars->tempty, EPI_WARPS);
        ptx::mbar_init(&bars->xbar, 32 * EPI_WARPS);
        for (int i = 0; i < TILE_RING; ++i) {
            ptx::mbar_init(&bars->tile_full[i], 1);
            // issuer, dependency warp, epilogue (and the counting warp with the in-kernel combine)
            ptx::mbar_init(&bars->tile_empty[i], 2 + EPI_WARPS + (FUSED ? 1 : 0));
            ptx::mbar_init(&bars->dep[i], 1);
            ptx::mbar_init(&bars->act_done[i], EPI_WARPS);
            ptx::mbar_init(&bars->tk.ready[i], 1);
        }
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
    // the fullest M-block of the forward decides the stage layout (the same in every CTA)
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
    const bool compact = bars->max_rows <= 2 * A_ROWS_PART;
    const uint32_t nst = compact ? NST_MAX : STAGES;                    // stages in the ring
    const uint32_t sbytes = compact ? COMPACT_STAGE_BYTES : STAGE_BYTES;   // bytes per stage
    const uint32_t a_reg = compact ? COMPACT_A_BYTES : STAGE_A_BYTES;      // B tile offset in a stage

    const BsTiles tl{(2 * d.I) / BN, (d.H + BN - 1) / BN, ws.blk_off[d.E], wave_blocks};
    const int ntiles = tl.total();
    auto view = [&](int tile) {
        BsView v;
        tl.at(tile, v.phase, v.blk, v.nt);
        v.e = ws.block_expert[v.blk];
        return v;
    };
    // A bytes a CTA stages per K block for a tile, in one load: the first 32 or 64 rows of an
    // M-block that holds no more valid rows, else all 128 (padding rows feed only accumulator
    // rows that are never stored)
    auto a_stage_bytes = [&](int n_part) {
        return n_part <= 2 ? static_cast<uint32_t>(n_part * A_ROWS_PART * BKS) : STAGE_A_BYTES;
    };
    const int NKB1 = d.H / BK, NKB2 = d.I / BK;
    const uint32_t l1_target = static_cast<uint32_t>(EPI_WARPS * tl.NT1);
    const uint64_t deadline = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);

    // Registers: launched at 168 per thread (384 x 168 = 64512); the producer / issuer
    // warpgroup gives (168-72) x 128 back and the two epilogue warpgroups take (216-168) x 256
    // (the producer keeps the next tile's metadata live without spilling).
    if (warp < 4) {
        ptx::setmaxnreg_dec<72>();
        if (warp == 0) {
            // -------------------------------------------------------- TMA producer ----
            if (lane == 0) {
                const uint64_t pol_a = ptx::policy_evict_last();
                const uint64_t pol_b_once = ptx::policy_evict_first();
                const uint64_t pol_b_shared = ptx::policy_evict_normal();
                uint32_t it = 0, tcount = 0, gcount = 0;   // K blocks, tiles, scale groups loaded
                // the last K block whose TMEM copies read the scale slots of the last three groups
                // (g-1, g-2, g-3; none yet: ~0): group g refills g-3's slot
                static_assert(SF_SLOTS == 3, "one reader per slot of the ring");
                uint32_t last1 = ~0u, last2 = ~0u, last3 = ~0u;
                uint32_t s = 0, ph = 0;   // stage of K block `it` and its ring pass parity
                bool ok = true;
                // Tiles are claimed from the global counter one ahead (a CTA holds at most one
                // claimed, unstarted tile; the smallest unfinished tile is always being worked on).
                auto claim_after = [&](int) { return static_cast<int>(atomicAdd(ws.hdr + HDR_TILE_NEXT, 1u)); };
                // The next tile is claimed, published to the ring (so the issuer, the epilogue
                // and the dependency warp see it a tile ahead), and its metadata (its M-block's
                // expert and valid rows, the expert's M-block count) read, in three steps taken
                // while the producer waits for free stages of the current tile, two K blocks
                // apart so each step's reads land before the next uses them.  Otherwise a chain of dependent
                // global reads sits between a tile's last load and the next tile's first, and
                // short (down) tiles start with the UMMA pipe dry.
                uint32_t pcount = 0;   // ring slots filled
                auto push = [&](int t) {
                    const uint32_t slot = pcount % TILE_RING, sph = (pcount / TILE_RING) & 1u;
                    if (!ptx::mbar_wait(&bars->tile_empty[slot], sph ^ 1u, deadline))
                        return false;
                    bars->tile_ring[slot] = t < ntiles ? t : -1;
                    ptx::mbar_arrive(&bars->tile_full[slot]);
                    ++pcount;
                    return true;
                };
                int m_tile = static_cast<int>(atomicAdd(ws.hdr + HDR_TILE_NEXT, 1u));
                BsView m_v{};
                int m_rows = 0, m_eblocks = 0;
                auto fetch = [&](int step, int cur) {
                    if (step == 0) {
                        m_tile = claim_after(cur);
                        return true;
                    }
                    if (step == 1) {
                        if (!push(m_tile))
                            return false;
                        if (m_tile < ntiles) {
                            m_v = view(m_tile);
                            m_rows = ws.block_rows[m_v.blk];
                        }
                    } else if (m_tile < ntiles) {
                        m_eblocks = ws.blk_off[m_v.e + 1] - ws.blk_off[m_v.e];
                    }
                    return true;
                };
                ok = fetch(1, 0) && fetch(2, 0);
                while (ok) {
                    const int tile = m_tile;
                    const BsView tv = m_v;
                    const int tv_rows = m_rows, tv_eblocks = m_eblocks;
                    const uint32_t slot = tcount % TILE_RING, sph = (tcount / TILE_RING) & 1u;
                    ++tcount;
                    if (tile >= ntiles)
                        break;
                    int fstep = 0, fkb = -2;   // next tile's steps done; K block of the last one
                    const int phase = tv.phase, blk = tv.blk, nt = tv.nt, e = tv.e;
                    const uint64_t pol_b = tv_eblocks > 1 ? pol_b_shared : pol_b_once;
                    const int n_part = max(1, (tv_rows + A_ROWS_PART - 1) / A_ROWS_PART);
                    const uint32_t a_bytes = a_stage_bytes(n_part);
                    // bytes the stage's full barrier waits for (the scale blocks only with the
                    // first stage of a group of K blocks)
                    const uint32_t tx_bytes = a_bytes + B_TX;
                    const CUtensorMap *ta = phase == 1 ? (n_part == 1 ? &maps.a1p : n_part == 2 ? &maps.a1h : &maps.a1)
                                                       : (n_part == 1 ? &maps.a2p : n_part == 2 ? &maps.a2h : &maps.a2);
                    const CUtensorMap *tb = phase == 1 ? &maps.b1 : &maps.b2;
                    const int nkb = phase == 1 ? NKB1 : NKB2;
                    const int wtile = e * (phase == 1 ? tl.NT1 : tl.NT2) + nt;
                    const int tile0 = wtile * nkb;
                    // scale blocks: A per (M-block, K-block group), B per (weight tile, group), or
                    // with MXFP4 weights per (weight tile, K block)
                    const int ng = (nkb + SF_GROUP - 1) / SF_GROUP;
                    const int nbb = FP4 ? nkb : ng;   // B scale blocks per weight tile
                    const uint8_t *sfa_src = (phase == 1 ? ws.pool_sfe : ws.act_sfe) +
                                             static_cast<long long>(blk) * ng * SFA_BYTES;
                    const uint8_t *sfb_src = (phase == 1 ? sfb1 : sfb2) + static_cast<long long>(wtile) * nbb * SFB_BYTES;
                    if (phase == 2) {
                        // the act rows and their scales of this block are complete: the
                        // dependency warp has acquired the block's gate_up completion count
                        // (a GPU-scope acquire here would also wait for this thread's loads in
                        // flight)
                        if (!ptx::mbar_wait(&bars->dep[slot], sph, deadline)) {
                            ok = false;
                            break;
                        }
                        ptx::fence_proxy_async_global();
                    }
                    for (int kb = 0; kb < nkb; ++kb, ++it, s = s + 1 == nst ? 0u : s + 1, ph ^= s == 0 ? 1u : 0u) {
                        // a step of the next tile's claim / publication / metadata, only when the
                        // stage is not free yet (the loads of a starving pipe are never held back)
                        // and two K blocks after the step before (whose reads it uses)
                        if (fstep < 3 && kb >= fkb + 2 && !ptx::mbar_try_wait(&bars->empty[s], ph ^ 1u)) {
                            fkb = kb;
                            if (!fetch(fstep++, tile)) {
                                ok = false;
                                break;
                            }
                        }
                        if (!ptx::mbar_wait(&bars->empty[s], ph ^ 1u, deadline)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sa = smem + s * sbytes;
                        // the first K block of a scale group brings the group's scale blocks into
                        // the next scale slot: A 512 bytes, B 1 KB (MXFP4: 1 KB per K block of the
                        // group, copied to TMEM with that K block)
                        const bool sf_k = kb % SF_GROUP == 0;
                        uint8_t *ss = nullptr;
                        uint32_t sfb_bytes = 0;
                        if (sf_k) {
                            const uint32_t j = gcount % SF_SLOTS;
                            ++gcount;
                            const int glen = min(SF_GROUP, nkb - kb);
                            // the slot's last reader: released above unless less than nst K blocks
                            // back (short groups); its stage is not refilled before that release
                            const uint32_t x = last3;
                            if (x != ~0u && x + nst > it &&
                                !ptx::mbar_wait(&bars->empty[x % nst], (x / nst) & 1u, deadline)) {
                                ok = false;
                                break;
                            }
                            last3 = last2;
                            last2 = last1;
                            last1 = it + (FP4 ? static_cast<uint32_t>(glen - 1) : 0u);
                            ss = sf_smem + j * SF_SLOT_BYTES;
                            sfb_bytes = (FP4 ? static_cast<uint32_t>(glen) : 1u) * SFB_BYTES;
                        }
                        ptx::mbar_arrive_expect_tx(&bars->full[s], tx_bytes + (sf_k ? SFA_BYTES + sfb_bytes : 0u));
                        ptx::tma_load_2d(sa, ta, &bars->full[s], kb * BK, blk * BM, pol_a);
                        ptx::tma_load_2d(sa + a_reg, tb, &bars->full[s], 0, (tile0 + kb) * BN, pol_b);
                        if (sf_k) {
                            const int grp = kb / SF_GROUP;
                            ptx::bulk_load(ss, sfa_src + grp * SFA_BYTES, SFA_BYTES, &bars->full[s]);
                            ptx::bulk_load(ss + SFA_BYTES, sfb_src + static_cast<long long>(FP4 ? kb : grp) * SFB_BYTES,
                                           sfb_bytes, &bars->full[s]);
                        }
                    }
                    while (ok && fstep < 3)
                        ok = fetch(fstep++, tile);
                }
                if (!ok)
                    record_error(ws.hdr, DEV_TIMEOUT);
                // drain: every issued load has landed before the CTA may exit
                const uint64_t dl = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);
                for (uint32_t i = it > nst ? it - nst : 0; i < it; ++i)
                    ptx::mbar_wait(&bars->full[i % nst], (i / nst) & 1u, dl);
            }
        } else if (warp == 2) {
            // -------------------------------------------------------- dependency warp --
            // A down tile reads act rows and scales that gate_up tiles of other CTAs wrote:
            // for each published tile this lane acquires (GPU scope) the M-block's gate_up
            // completion count, then releases the tile to the producer through the slot's
            // CTA-scope barrier (gate_up tiles and null halves at once).
            if (lane == 0) {
                uint32_t tcount = 0;
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
                    const BsView v = view(tile);
                    if (v.phase == 2) {
                        for (uint32_t i = 0;; ++i) {
                            if (ptx::ld_acquire_gpu(ws.l1_done + v.blk) >= l1_target)
                                break;
                            if ((i & 63u) == 63u && ptx::globaltimer() > deadline) {
                                ok = false;
                                break;
                            }
                        }
                        if (!ok)
                            break;
                    }
                    ptx::mbar_arrive(&bars->dep[slot]);
                }
                if (!ok)
                    record_error(ws.hdr, DEV_TIMEOUT);
            }
        } else if (warp == 1) {
            // -------------------------------------------------------- UMMA issuer -----
            if (lane == 0) {
                uint32_t it = 0, tcount = 0, acc_n = 0, gcount = 0;
                uint32_t s = 0, ph = 0, gslot = 0;   // stage of K block `it`, its pass parity; next TMEM scale slot
                // Scale group g is copied from shared-memory slot g % SF_SLOTS (MXFP4: each K
                // block's B scales with that K block) to TMEM group slot g % NST_MAX.  That TMEM
                // slot is reused only after NST_MAX more groups, i.e. at least NST_MAX K blocks
                // after group g's last, whose first stage's arrival implies (through the stage
                // ring of at most NST_MAX stages) that every UMMA reading group g has completed.
                uint32_t sfa = 0, ssg = 0;   // TMEM slot and shared-memory slot of the current group
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
                    int phase, unit, nt;
                    tl.at(tile, phase, unit, nt);
                    const int nkb = phase == 1 ? NKB1 : NKB2;
                    // the previous tile's accumulator has been read by every epilogue warp
                    if (!ptx::mbar_wait(&bars->tempty, (acc_n & 1u) ^ 1u, deadline)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    for (int kb = 0; kb < nkb; ++kb, ++it, s = s + 1 == nst ? 0u : s + 1, ph ^= s == 0 ? 1u : 0u) {
                        if (!ptx::mbar_wait(&bars->full[s], ph, deadline)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        if (kb % SF_GROUP == 0) {
                            ssg = ptx::smem_u32(sf_smem + (gcount % SF_SLOTS) * SF_SLOT_BYTES);
                            ++gcount;
                            sfa = tmem + SF_COL + SF_TCOLS * gslot;
                            gslot = gslot + 1 == NST_MAX ? 0u : gslot + 1;
                            sf_copy(sfa, ssg);
                            if constexpr (!FP4) {
                                sf_copy(sfa + 4, ssg + SFA_BYTES);
                                sf_copy(sfa + 8, ssg + SFA_BYTES + 512);
                            }
                        }
                        uint32_t sfb = sfa + 4;
                        if constexpr (FP4) {
                            // copied per K block: the group's copies spread over its K blocks
                            // measured faster than all at its start
                            const uint32_t i = static_cast<uint32_t>(kb % SF_GROUP);
                            sfb += 8 * i;
                            sf_copy(sfb, ssg + SFA_BYTES + i * SFB_BYTES);
                            sf_copy(sfb + 4, ssg + SFA_BYTES + i * SFB_BYTES + 512);
                        }
                        const uint32_t a_addr = ptx::smem_u32(smem + s * sbytes);
                        const uint64_t adesc = ptx::kmajor_swizzled_desc<BKS>(a_addr);
                        const uint64_t bdesc = ptx::kmajor_swizzled_desc<BKS>(a_addr + a_reg);
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k)   // +32 bytes along K = +2 in the >>4 field
                            umma_bs(tmem, adesc + 2 * k, bdesc + 2 * k,
                                    idesc_bs<BM, FP4>(kb % SF_GROUP, FP4 ? k : kb % SF_GROUP), sfa, sfb,
                                    (kb > 0 || k > 0) ? 1u : 0u);
                        ptx::umma_commit(&bars->empty[s]);
                    }
                    if (!ok)
                        break;
                    ptx::umma_commit(&bars->tfull);
                    ++acc_n;
                }
                if (!ok)
                    record_error(ws.hdr, DEV_TIMEOUT);
                // drain: the last commit arrives once every issued copy and MMA has completed
                if (it > 0) {
                    const uint64_t dl = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);
                    const uint32_t i = it - 1;
                    ptx::mbar_wait(&bars->empty[i % nst], (i / nst) & 1u, dl);
                }
            }
        } else if (FUSED) {
            // -------------------------------------------------------- counting warp ---
            // In-kernel combine: once the epilogue warps have stored a down tile (act_done),
            // count its rows per (token, n-tile) and list the pairs it completed for the
            // epilogue warps, which reduce them at the end of their next tile
            // (topk_combine.cuh); every tile gets its list barrier arrival.
            uint32_t tcount = 0;
            bool ok = true;
            while (ok) {
                const uint32_t slot = tcount % TILE_RING, sph = (tcount / TILE_RING) & 1u;
                ++tcount;
                if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&bars->tile_full[slot], sph, deadline))) {
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
                if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&bars->act_done[slot], sph, deadline))) {
                    ok = false;
                    break;
                }
                int phase, blk, nt;
                tl.at(tile, phase, blk, nt);
                const int n = phase == 2 ? topk::count_rows(d, ws, static_cast<long long>(blk) * BM, ws.block_rows[blk],
                                                            nt, bars->tk.tok[slot], bars->tk.mask[slot], lane)
                                         : 0;
                __syncwarp();
                if (lane == 0) {
                    bars->tk.n[slot] = n;
                    bars->tk.nt[slot] = nt;
                    ptx::mbar_arrive(&bars->tk.ready[slot]);
                    ptx::mbar_arrive(&bars->tile_empty[slot]);
                }
            }
            if (!ok && lane == 0)
                record_error(ws.hdr, DEV_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ epilogue --------
        ptx::setmaxnreg_inc<216>();
        const int wg = (warp - 4) >> 2;          // column half of the tile
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;           // tile row = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        uint32_t tcount = 0, xcount = 0, acc_n = 0;
        bool ok = true;
        // in-kernel combine: the (token, n-tile) pairs the counting warp listed for the previous
        // tile are reduced by the eight epilogue warps at the end of the next one
        int prev = -1;   // ring slot of the previous tile, -1 before the first
        uint32_t prev_ph = 0;
        auto reduce_listed = [&](int sl, uint32_t ph) {
            if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&bars->tk.ready[sl], ph, deadline)))
                return false;
            const int n = bars->tk.n[sl];
            if (n > 0)
                topk::reduce(d, ws, c, bars->tk.tok[sl], bars->tk.mask[sl], n, bars->tk.nt[sl], warp - 4, EPI_WARPS,
                             lane);
            return true;
        };
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
            if (tile < 0) {
                if (FUSED && prev >= 0 && !reduce_listed(prev, prev_ph))
                    ok = false;
                break;
            }
            int phase, blk, nt;
            tl.at(tile, phase, blk, nt);
            const long long prow = static_cast<long long>(blk) * BM + row;
            // the whole tile, already scaled, in one read of this warp's 32 rows x 128 columns
            if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&bars->tfull, acc_n & 1u, deadline))) {
                ok = false;
                break;
            }
            ++acc_n;
            ptx::tc_fence_after();
            float acc[128];
            const uint32_t taddr = tmem + lane_base + wg * 128;
#pragma unroll
            for (int ch = 0; ch < 4; ch += 2) {
                uint32_t r0[32], r1[32];
                ptx::tmem_ld32(taddr + ch * 32, r0);
                ptx::tmem_ld32(taddr + ch * 32 + 32, r1);
                ptx::tmem_ld_wait(r0);
                ptx::reg_tie(r1);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    acc[ch * 32 + j] = __uint_as_float(r0[j]);
                    acc[ch * 32 + 32 + j] = __uint_as_float(r1[j]);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(&bars->tempty);
            const int rows = ws.block_rows[blk];
            if (phase == 1) {
                // SwiGLU on the 64 (gate, up) pairs of this row and column half, then 1x128
                // requant with the smallest power-of-two scale >= max(amax, 1e-4)/448
                const bool live = q * 32 < rows;
                float amax = 0.0f;
                if (live) {
#pragma unroll
                    for (int m = 0; m < 64; ++m) {
                        const float g = acc[(m >> 3) * 16 + (m & 7)];
                        const float u = acc[(m >> 3) * 16 + 8 + (m & 7)];
                        const float hval = __fdividef(g, 1.0f + __expf(-g)) * u;
                        acc[m] = hval;
                        amax = fmaxf(amax, fabsf(hval));
                    }
                }
                const uint32_t tp = xcount & 1u;
                ++xcount;
                bars->amax[tp][wg][row] = amax;
                ptx::mbar_arrive(&bars->xbar);
                if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&bars->xbar, tp, deadline))) {
                    ok = false;
                    break;
                }
                if (live) {
                    amax = fmaxf(bars->amax[tp][0][row], bars->amax[tp][1][row]);
                    const float sf = pow2_ceil(fmaxf(amax, 1e-4f) / 448.0f);
                    // 1/sf is exact for a power of two
                    const float inv = __uint_as_float((254u << 23) - (__float_as_uint(sf) & 0x7F800000u));
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
                    if (wg == 0) {
                        ws.act_sf[static_cast<long long>(nt) * ws.P + prow] = sf;
                        // UE8M0 byte of this row and K block nt of the down GEMM, in the block's
                        // 512-byte scale block of group nt / 4
                        ws.act_sfe[(static_cast<long long>(blk) * ((NKB2 + SF_GROUP - 1) / SF_GROUP) + nt / SF_GROUP) *
                                       SFA_BYTES +
                                   16 * (row % 32) + 4 * (row / 32) + nt % SF_GROUP] =
                            static_cast<uint8_t>(__float_as_uint(sf) >> 23);
                    }
                }
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
                // (with H an odd multiple of 128 the last down tile's second column half lies
                // past H: its weight rows are zero and nothing is stored)
                if (q * 32 < rows && nt * BN + wg * 128 < d.H) {
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
            if (FUSED) {
                // the tile is stored: the counting warp may count it; then the previous tile's
                // completed pairs
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(&bars->act_done[slot]);
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
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
    if (FUSED)
        ffn_cta_exit(d, ws, &bars->exit_flag);
}

cudaError_t launch_ffn_bs(const FfnMaps &maps, const Dims &d, const Workspace &ws, const CallArgs &c,
                          const uint8_t *sfb1, const uint8_t *sfb2, int wave_blocks, int num_sms, bool fp4,
                          cudaStream_t s)
{
    constexpr int SMEM = 1024 + RING_BYTES + 8192 + SF_SLOTS * static_cast<int>(SF_SLOT_BYTES);
    static_assert(sizeof(BsBars) <= 8192, "barrier block");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
    const bool fu = c.fused_combine != 0;
    void *kern = fp4 ? (fu ? reinterpret_cast<void *>(ffn_bs_kernel<true, true>)
                           : reinterpret_cast<void *>(ffn_bs_kernel<true, false>))
                     : (fu ? reinterpret_cast<void *>(ffn_bs_kernel<false, true>)
                           : reinterpret_cast<void *>(ffn_bs_kernel<false, false>));
    cudaError_t e0 = ensure_max_dynamic_smem(kern, SMEM);
    if (e0 != cudaSuccess)
        return e0;
    // Tiles are claimed in list order by running CTAs only, so the launch needs no
    // co-residency guarantee: a down tile waits only on gate_up tiles claimed before it.
    if (fp4)
        return fu ? launch_programmatic(ffn_bs_kernel<true, true>, num_sms, GEMM_THREADS, SMEM, s, maps, d, ws, c, sfb1,
                                        sfb2, wave_blocks)
                  : launch_programmatic(ffn_bs_kernel<true, false>, num_sms, GEMM_THREADS, SMEM, s, maps, d, ws, c, sfb1,
                                        sfb2, wave_blocks);
    return fu ? launch_programmatic(ffn_bs_kernel<false, true>, num_sms, GEMM_THREADS, SMEM, s, maps, d, ws, c, sfb1,
                                    sfb2, wave_blocks)
              : launch_programmatic(ffn_bs_kernel<false, false>, num_sms, GEMM_THREADS, SMEM, s, maps, d, ws, c, sfb1,
                                    sfb2, wave_blocks);
}

// ------------------------------------------------------------------ weight scales -----
// Load-time UE8M0 scale blocks of the weight tiles: for weight tile (e, nt) and group g of
// four K blocks, 1 KB at ((e*NT + nt)*G + g)*1024 (G = ceil(KB/4)) with tile column n's word
// at 512*(n/128) + 16*(n%32) + 4*((n%128)/32), byte kb % 4 = K block kb's scale.  Column n of a gate_up tile (gate_up_I > 0) is the gate row group nt if
// (n/8) is even, else the up group I/128 + nt (the interleave by 8); of a down tile, the row
// group 2*nt + n/128.  Any scale that is not a positive normal power of two sets *bad.  A
// last tile that covers fewer than 256 rows (N an odd multiple of 128) gets the byte 127
// (scale 1) for its missing rows, whose re-laid weights are zero.
__global__ void build_sfb_kernel(const float *__restrict__ s, uint8_t *__restrict__ dst, int E, int N, int K,
                                 int gate_up_I, uint32_t *bad)
{
    const int KB = K / 128, NT = (N + BN - 1) / BN;
    const long long words = static_cast<long long>(E) * NT * KB * BN;
    for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < words;
         q += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(q % BN);
        const long long tk = q / BN;   // (e*NT + nt)*KB + kb
        const int kb = static_cast<int>(tk % KB);
        const long long et = tk / KB;
        const int nt = static_cast<int>(et % NT);
        const int e = static_cast<int>(et / NT);
        int group;
        if (gate_up_I > 0)
            group = ((n >> 3) & 1) ? gate_up_I / 128 + nt : nt;
        else
            group = 2 * nt + n / 128;
        uint32_t ex = 127u;
        if (nt * BN + n < N) {
            const float v = s[(static_cast<long long>(e) * (N / 128) + group) * KB + kb];
            const uint32_t b = __float_as_uint(v);
            ex = (b >> 23) & 0xFFu;
            if ((b & 0x807FFFFFu) != 0u || ex == 0u || ex == 0xFFu)
                atomicOr(bad, 1u);
        }
        const long long g = et * ((KB + SF_GROUP - 1) / SF_GROUP) + kb / SF_GROUP;
        dst[g * SFB_BYTES + 512 * (n / 128) + 16 * (n % 32) + 4 * ((n % 128) / 32) + kb % SF_GROUP] =
            static_cast<uint8_t>(ex);
    }
}

cudaError_t launch_build_sfb(const float *s, uint8_t *dst, int E, int N, int K, int gate_up_I, uint32_t *bad,
                             cudaStream_t st)
{
    build_sfb_kernel<<<1024, 256, 0, st>>>(s, dst, E, N, K, gate_up_I, bad);
    return cudaGetLastError();
}

// MXFP4 weights: scale blocks per weight tile and K block.  s = [E][N][K/32] UE8M0 bytes in
// the caller's row order; for weight tile (e, nt) and K block kb, 1 KB at
// ((e*NT + nt)*KB + kb)*1024 with tile column n's word at 512*(n/128) + 16*(n%32) +
// 4*((n%128)/32), byte j = the scale of the row's 32-deep slice 4*kb + j.  Tile column n is
// weight row nt*256 + n, through the gate/up interleave by 8 for the gate_up weight (the
// row order of the re-laid weight tiles).  A byte 0xFF (NaN in the UE8M0 format) sets *bad.
// Rows past N of a last tile that covers fewer than 256 rows get the bytes 127 (zero weights).
__global__ void build_sfb4_kernel(const uint8_t *__restrict__ s, uint8_t *__restrict__ dst, int E, int N, int K,
                                  int gate_up_I, uint32_t *bad)
{
    const int KB = K / 128, NT = (N + BN - 1) / BN;
    const long long words = static_cast<long long>(E) * NT * KB * BN;
    for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < words;
         q += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(q % BN);
        const long long tk = q / BN;   // (e*NT + nt)*KB + kb
        const int kb = static_cast<int>(tk % KB);
        const long long et = tk / KB;
        const int nt = static_cast<int>(et % NT);
        const long long e = et / NT;
        const int row = nt * BN + n;
        int srow = row;
        if (gate_up_I > 0) {
            const int j = row / 16, i = row % 16;
            srow = i < 8 ? 8 * j + i : gate_up_I + 8 * j + (i - 8);
        }
        // K/32 is a multiple of 4: the four bytes of K block kb are one aligned word
        const uint32_t w = row < N ? *reinterpret_cast<const uint32_t *>(s + (e * N + srow) * (K / 32) + 4 * kb)
                                   : 0x7F7F7F7Fu;
        if (((w & 0xFFu) == 0xFFu) || ((w >> 8 & 0xFFu) == 0xFFu) || ((w >> 16 & 0xFFu) == 0xFFu) || ((w >> 24) == 0xFFu))
            atomicOr(bad, 1u);
        *reinterpret_cast<uint32_t *>(dst + tk * SFB_BYTES + 512 * (n / 128) + 16 * (n % 32) + 4 * ((n % 128) / 32)) = w;
    }
}

cudaError_t launch_build_sfb4(const uint8_t *s, uint8_t *dst, int E, int N, int K, int gate_up_I, uint32_t *bad,
                              cudaStream_t st)
{
    build_sfb4_kernel<<<1024, 256, 0, st>>>(s, dst, E, N, K, gate_up_I, bad);
    return cudaGetLastError();
}

}  // namespace cpw
