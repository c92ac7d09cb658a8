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
// Scale factors reach TMEM through shared memory: per stage the producer bulk-copies a
// 512-byte A block (the 128 rows' scale words, row r at byte 16*(r%32) + 4*(r/32)) and a
// 1 KB B block (two 512-byte halves; tile column n at 512*(n/128) + 16*(n%32) + 4*((n%128)/32)),
// each word holding the UE8M0 byte four times (one per 32-deep K slice).  The UMMA issuer
// copies them into TMEM with tcgen05.cp 32x128b.warpx4 (every lane quarter gets the same
// 32 lanes), where the UMMA reads row m's scale at lane m, column base + m/32, and tile
// column n's at lane 32*q + n%32, column base + n/32, byte = the K slice.
//
// Roles (one CTA per SM, 12 warps): warp 0 TMA producer (A, B and the two scale blocks of
// a 128-deep K block per stage, 4 stages); warp 1 UMMA issuer (scale copies + 4 block-scaled
// UMMAs per stage into one 256-column TMEM accumulator); warps 4-11 epilogue (two
// warpgroups, columns [0,128) / [128,256)): one TMEM read per tile, then SwiGLU + UE8M0
// requant (phase 1) or the weighted scatter (phase 2).  TMEM: accumulator columns 0-255,
// scale slots 256 + 16*s.  All waits carry a deadline (MOE_ERR_TIMEOUT).
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace cpw {

namespace {

constexpr uint32_t TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;
constexpr int TILE_RING = 4;
constexpr uint32_t SF_COL = 256;          // scale slot s: columns SF_COL + 16*s (A: +0..3, B: +4..11)
constexpr uint32_t SFA_BYTES = 512, SFB_BYTES = 1024, SF_STAGE_BYTES = SFA_BYTES + SFB_BYTES;
static_assert(BKS == BK, "the block-scaled kernel stages whole 128-deep K blocks");

// block-scaled instruction descriptor: B scale slice at bits 4-5, e4m3 A/B (formats 0),
// K-major A and B, N>>3 at 17-22, UE8M0 scales (bit 23), M>>4 at 24-28, A scale slice at
// 29-30
__device__ __forceinline__ uint32_t idesc_bs(int k)
{
    return (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
           (static_cast<uint32_t>(BM >> 4) << 24) | (static_cast<uint32_t>(k) << 29);
}

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
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull;
    uint64_t tempty;
    uint64_t xbar;
    uint64_t tile_full[TILE_RING];
    uint64_t tile_empty[TILE_RING];
    int tile_ring[TILE_RING];
    uint32_t tmem_base;
    int abort;
    float amax[2][2][BM];
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

}  // namespace

__global__ void __launch_bounds__(GEMM_THREADS, 1)
    ffn_bs_kernel(const __grid_constant__ FfnMaps maps, const Dims d, const Workspace ws, const CallArgs c,
                  const uint8_t *__restrict__ sfb1, const uint8_t *__restrict__ sfb2, const int wave_blocks)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    BsBars *bars = reinterpret_cast<BsBars *>(smem + STAGES * STAGE_BYTES);
    uint8_t *sf_smem = smem + STAGES * STAGE_BYTES + 8192;   // [STAGES][A 512 | B 1024]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        const uint32_t err = *reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_CALL) |
                             *reinterpret_cast<volatile uint32_t *>(ws.hdr + HDR_ERR_STICKY);
        bars->abort = err != 0;
        if (!err) {
            for (int s = 0; s < STAGES; ++s) {
                ptx::mbar_init(&bars->full[s], 1);
                ptx::mbar_init(&bars->empty[s], 1);
            }
            ptx::mbar_init(&bars->tfull, 1);
            ptx::mbar_init(&bars->tempty, EPI_WARPS);
            ptx::mbar_init(&bars->xbar, 32 * EPI_WARPS);
            for (int i = 0; i < TILE_RING; ++i) {
                ptx::mbar_init(&bars->tile_full[i], 1);
                ptx::mbar_init(&bars->tile_empty[i], 1 + EPI_WARPS);
            }
            ptx::fence_mbar_init();
        }
    }
    __syncthreads();
    if (bars->abort)
        return;
    if (warp == 1) {
        ptx::tmem_alloc(&bars->tmem_base, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    const BsTiles tl{(2 * d.I) / BN, d.H / BN, ws.blk_off[d.E], wave_blocks};
    const int ntiles = tl.total();
    const int NKB1 = d.H / BK, NKB2 = d.I / BK;
    const uint32_t l1_target = static_cast<uint32_t>(EPI_WARPS * tl.NT1);
    const uint64_t deadline = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);

    if (warp < 4) {
        ptx::setmaxnreg_dec<40>();
        if (warp == 0) {
            // -------------------------------------------------------- TMA producer ----
            if (lane == 0) {
                ptx::prefetch_tmap(&maps.a1);
                ptx::prefetch_tmap(&maps.b1);
                ptx::prefetch_tmap(&maps.a2);
                ptx::prefetch_tmap(&maps.b2);
                const uint64_t pol_a = ptx::policy_evict_last();
                const uint64_t pol_b_once = ptx::policy_evict_first();
                const uint64_t pol_b_shared = ptx::policy_evict_normal();
                uint32_t it = 0, tcount = 0;
                bool ok = true;
                // tiles are claimed one ahead, so the claim's round trip to L2 overlaps the
                // loads of the tile before (a CTA holds at most one claimed, unstarted tile;
                // the smallest unfinished tile is always being worked on)
                int next = static_cast<int>(atomicAdd(ws.hdr + HDR_TILE_NEXT, 1u));
                while (ok) {
                    const int tile = next;
                    if (tile < ntiles)
                        next = static_cast<int>(atomicAdd(ws.hdr + HDR_TILE_NEXT, 1u));
                    const uint32_t slot = tcount % TILE_RING, sph = (tcount / TILE_RING) & 1u;
                    if (!ptx::mbar_wait(&bars->tile_empty[slot], sph ^ 1u, deadline)) {
                        ok = false;
                        break;
                    }
                    bars->tile_ring[slot] = tile < ntiles ? tile : -1;
                    ptx::mbar_arrive(&bars->tile_full[slot]);
                    ++tcount;
                    if (tile >= ntiles)
                        break;
                    int phase, blk, nt;
                    tl.at(tile, phase, blk, nt);
                    const int e = ws.block_expert[blk];
                    const uint64_t pol_b = ws.blk_off[e + 1] - ws.blk_off[e] > 1 ? pol_b_shared : pol_b_once;
                    const int n_part = (ws.block_rows[blk] + A_ROWS_PART - 1) / A_ROWS_PART;
                    const bool part = n_part < BM / A_ROWS_PART;
                    const uint32_t a_bytes = part ? static_cast<uint32_t>(n_part * A_ROWS_PART * BKS) : STAGE_A_BYTES;
                    const CUtensorMap *ta = phase == 1 ? (part ? &maps.a1p : &maps.a1) : (part ? &maps.a2p : &maps.a2);
                    const CUtensorMap *tb = phase == 1 ? &maps.b1 : &maps.b2;
                    const int nkb = phase == 1 ? NKB1 : NKB2;
                    const int tile0 = (e * (phase == 1 ? tl.NT1 : tl.NT2) + nt) * nkb;
                    // scale blocks: A per (M-block, K block), B per (weight tile, K block)
                    const uint8_t *sfa_src = (phase == 1 ? ws.pool_sfe : ws.act_sfe) +
                                             static_cast<long long>(blk) * nkb * SFA_BYTES;
                    const uint8_t *sfb_src = (phase == 1 ? sfb1 : sfb2) + static_cast<long long>(tile0) * SFB_BYTES;
                    if (phase == 2) {
                        // the act rows and their scales of this block are complete once every
                        // epilogue warp of every gate_up tile of the block has released them
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
                        ptx::fence_proxy_async_global();
                    }
                    for (int kb = 0; kb < nkb; ++kb, ++it) {
                        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                        if (!ptx::mbar_wait(&bars->empty[s], ph ^ 1u, deadline)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sa = smem + s * STAGE_BYTES;
                        uint8_t *ss = sf_smem + s * SF_STAGE_BYTES;
                        ptx::mbar_arrive_expect_tx(&bars->full[s], a_bytes + STAGE_B_BYTES + SF_STAGE_BYTES);
                        if (part) {
                            for (int g = 0; g < n_part; ++g)
                                ptx::tma_load_2d(sa + g * A_ROWS_PART * BKS, ta, &bars->full[s], kb * BK,
                                                 blk * BM + g * A_ROWS_PART, pol_a);
                        } else {
                            ptx::tma_load_2d(sa, ta, &bars->full[s], kb * BK, blk * BM, pol_a);
                        }
                        ptx::tma_load_2d(sa + STAGE_A_BYTES, tb, &bars->full[s], 0, (tile0 + kb) * BN, pol_b);
                        ptx::bulk_load(ss, sfa_src + kb * SFA_BYTES, SFA_BYTES, &bars->full[s]);
                        ptx::bulk_load(ss + SFA_BYTES, sfb_src + static_cast<long long>(kb) * SFB_BYTES, SFB_BYTES,
                                       &bars->full[s]);
                    }
                }
                if (!ok)
                    record_error(ws.hdr, DEV_TIMEOUT);
                const uint64_t dl = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);
                for (uint32_t i = it > STAGES ? it - STAGES : 0; i < it; ++i)
                    ptx::mbar_wait(&bars->full[i % STAGES], (i / STAGES) & 1u, dl);
            }
        } else if (warp == 1) {
            // -------------------------------------------------------- UMMA issuer -----
            if (lane == 0) {
                uint32_t it = 0, tcount = 0, acc_n = 0;
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
                    // the previous tile's accumulator has been read by every epilogue warp
                    if (!ptx::mbar_wait(&bars->tempty, (acc_n & 1u) ^ 1u, deadline)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    for (int kb = 0; kb < nkb; ++kb, ++it) {
                        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                        if (!ptx::mbar_wait(&bars->full[s], ph, deadline)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t ss = ptx::smem_u32(sf_smem + s * SF_STAGE_BYTES);
                        const uint32_t sfa = tmem + SF_COL + 16 * s, sfb = sfa + 4;
                        sf_copy(sfa, ss);
                        sf_copy(sfb, ss + SFA_BYTES);
                        sf_copy(sfb + 4, ss + SFA_BYTES + 512);
                        const uint32_t a_addr = ptx::smem_u32(smem + s * STAGE_BYTES);
                        const uint64_t adesc = ptx::kmajor_swizzled_desc<BKS>(a_addr);
                        const uint64_t bdesc = ptx::kmajor_swizzled_desc<BKS>(a_addr + STAGE_A_BYTES);
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k)   // +32 bytes along K = +2 in the >>4 field
                            umma_bs(tmem, adesc + 2 * k, bdesc + 2 * k, idesc_bs(k), sfa, sfb,
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
                if (it > 0) {
                    const uint64_t dl = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);
                    const uint32_t i = it - 1;
                    ptx::mbar_wait(&bars->empty[i % STAGES], (i / STAGES) & 1u, dl);
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
        uint32_t tcount = 0, xcount = 0, acc_n = 0;
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
                        // UE8M0 scale word of this row in the block's 512-byte scale block
                        const uint32_t byte = (__float_as_uint(sf) >> 23) & 0xFFu;
                        *reinterpret_cast<uint32_t *>(ws.act_sfe + (static_cast<long long>(blk) * NKB2 + nt) * SFA_BYTES +
                                                      16 * (row % 32) + 4 * (row / 32)) = byte * 0x01010101u;
                    }
                }
                __syncwarp();
                ptx::fence_proxy_async_global();
                if (lane == 0)
                    ptx::red_release_add(ws.l1_done + blk, 1u);
            } else {
                if (row < rows) {
                    const uint32_t t = ws.meta[prow * 3 + 1];
                    const uint32_t kk = ws.meta[prow * 3 + 2];
                    const float gw = __ldg(c.w + static_cast<long long>(t) * d.K + kk);
                    uint4 *dst = reinterpret_cast<uint4 *>(
                        ws.combine + (static_cast<long long>(kk) * ws.max_tokens + t) * d.H + nt * BN + wg * 128);
#pragma unroll
                    for (int v = 0; v < 16; ++v) {
                        uint32_t w4[4];
#pragma unroll
                        for (int p = 0; p < 4; ++p) {
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(gw * acc[v * 8 + 2 * p],
                                                                            gw * acc[v * 8 + 2 * p + 1]);
                            w4[p] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        dst[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
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
}

cudaError_t launch_ffn_bs(const FfnMaps &maps, const Dims &d, const Workspace &ws, const CallArgs &c,
                          const uint8_t *sfb1, const uint8_t *sfb2, int wave_blocks, int num_sms, cudaStream_t s)
{
    static bool configured = false;
    constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + 8192 + STAGES * SF_STAGE_BYTES;
    static_assert(sizeof(BsBars) <= 8192, "barrier block");
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(ffn_bs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    FfnMaps m = maps;
    Dims dd = d;
    Workspace ww = ws;
    CallArgs cc = c;
    const uint8_t *p1 = sfb1;
    const uint8_t *p2 = sfb2;
    int wb = wave_blocks;
    void *args[] = {&m, &dd, &ww, &cc, &p1, &p2, &wb};
    // down tiles wait on gate_up tiles of other CTAs: all CTAs must be resident at once
    return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(ffn_bs_kernel), dim3(num_sms), dim3(GEMM_THREADS), args,
                                       SMEM, s);
}

// ------------------------------------------------------------------ weight scales -----
// Load-time UE8M0 scale blocks of the weight tiles: for weight tile (e, nt) and K block kb,
// 1 KB at ((e*NT + nt)*KB + kb)*1024 with tile column n's word at 512*(n/128) + 16*(n%32) +
// 4*((n%128)/32).  Column n of a gate_up tile (gate_up_I > 0) is the gate row group nt if
// (n/8) is even, else the up group I/128 + nt (the interleave by 8); of a down tile, the row
// group 2*nt + n/128.  Any scale that is not a positive normal power of two sets *bad.
__global__ void build_sfb_kernel(const float *__restrict__ s, uint8_t *__restrict__ dst, int E, int N, int K,
                                 int gate_up_I, uint32_t *bad)
{
    const int KB = K / 128, NT = N / BN;
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
        const float v = s[(static_cast<long long>(e) * (N / 128) + group) * KB + kb];
        const uint32_t b = __float_as_uint(v);
        const uint32_t ex = (b >> 23) & 0xFFu;
        if ((b & 0x807FFFFFu) != 0u || ex == 0u || ex == 0xFFu)
            atomicOr(bad, 1u);
        *reinterpret_cast<uint32_t *>(dst + tk * SFB_BYTES + 512 * (n / 128) + 16 * (n % 32) + 4 * ((n % 128) / 32)) =
            ex * 0x01010101u;
    }
}

cudaError_t launch_build_sfb(const float *s, uint8_t *dst, int E, int N, int K, int gate_up_I, uint32_t *bad,
                             cudaStream_t st)
{
    build_sfb_kernel<<<1024, 256, 0, st>>>(s, dst, E, N, K, gate_up_I, bad);
    return cudaGetLastError();
}

}  // namespace cpw
