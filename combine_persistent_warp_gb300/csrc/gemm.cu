// gemm.cu -- persistent, warp-specialised FP8 grouped GEMM on tcgen05 (sm_103a).
//
// One kernel template serves both expert GEMMs of the layer ("Mega-MoE 内核代码导读：从
// Dispatch 到 WGMMA 的融合流水线" §六: Linear1 gate_up, Linear2 down; §八: per-tile life of
// a GEMM block):
//   PHASE 1 (gate_up):  A = expert-major pool [P][H] e4m3 + 1x128 scales,
//                       B = gate/up-interleaved W1 [E*2I][H] e4m3 + 128x128 scales;
//                       epilogue: SwiGLU, per-row 1x128 requant to e4m3 -> act [P][I].
//   PHASE 2 (down):     A = act [P][I] + scales, B = W2 [E*H][I] + 128x128 scales;
//                       epilogue: multiply by the top-k gate weight, bf16, scatter through
//                       the {source, token, topk} metadata into combine[topk][T][H]
//                       ("DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析" §8.1).
//
// Roles of the 12 warps of a CTA (one CTA per SM, persistent over a static tile list):
//   warp 0     TMA producer: A and B tiles of one 128-deep K block into a 4-stage ring
//   warp 1     UMMA issuer: 4 x (128x256x32) tcgen05.mma into a fresh TMEM partial
//   warps 2-3  idle (keep the epilogue warpgroups aligned for TMEM lane access)
//   warps 4-11 two epilogue warpgroups, columns [0,128) and [128,256) of the tile
// The fp32 scales are arbitrary per 128-deep K block (1x128 for A rows, 128x128 for B), so
// each K block's product is accumulated separately in TMEM (double-buffered, 2 x 256
// columns) and the epilogue warps promote it into fp32 registers with the product of the
// two scales -- the scale promotion of the pages' SM90 kernel (§8.1 of the first page),
// here overlapped with the next K block's UMMA through the TMEM full/empty barriers.
// All waits carry a deadline; on expiry the CTA records MOE_ERR_TIMEOUT and leaves after
// draining the copies and MMAs it has in flight.
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace cpw {

namespace {

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = ptx::idesc_e4m3_f32(BM, BN);

struct __align__(8) GemmBars {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t xbar;          // row-amax exchange between the two epilogue warpgroups
    uint32_t tmem_base;
    int abort;
    float amax[2][2][BM];   // [tile parity][column half][row]
};

}  // namespace

template <int PHASE>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const Dims d, const Workspace ws, const CallArgs c, const float *__restrict__ sf_w)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    GemmBars *bars = reinterpret_cast<GemmBars *>(smem + STAGES * STAGE_BYTES);
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
            for (int b = 0; b < 2; ++b) {
                ptx::mbar_init(&bars->tfull[b], 1);
                ptx::mbar_init(&bars->tempty[b], 8);   // one arrival per epilogue warp
            }
            ptx::mbar_init(&bars->xbar, 256);          // every epilogue thread, once per tile
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

    const int Kdim = PHASE == 1 ? d.H : d.I;
    const int NKB = Kdim / BK;
    const int NT = PHASE == 1 ? (2 * d.I) / BN : d.H / BN;
    const int ntiles = ws.blk_off[d.E] * NT;
    const uint64_t deadline = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);

    // Registers: launched at 168 per thread (384 x 168 = 64512); the producer warpgroup
    // gives (168-40) x 128 back and the two epilogue warpgroups take (232-168) x 256.
    if (warp < 4) {
        ptx::setmaxnreg_dec<40>();   // one instruction for all four warps of the group
        if (warp == 0) {
            // ------------------------------------------------------------ TMA producer ----
            if (lane == 0) {
                ptx::prefetch_tmap(&tm_a);
                ptx::prefetch_tmap(&tm_b);
                const uint64_t pol_a = ptx::policy_evict_last();
                const uint64_t pol_b = ptx::policy_evict_first();
                uint32_t it = 0;
                bool ok = true;
                for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                    const int blk = tile / NT, nt = tile % NT;
                    const int e = ws.block_expert[blk];
                    const int brow = (PHASE == 1 ? e * 2 * d.I : e * d.H) + nt * BN;
                    for (int kb = 0; kb < NKB; ++kb, ++it) {
                        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                        if (!ptx::mbar_wait(&bars->empty[s], ph ^ 1u, deadline)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sa = smem + s * STAGE_BYTES;
                        ptx::mbar_arrive_expect_tx(&bars->full[s], STAGE_BYTES);
                        ptx::tma_load_2d(sa, &tm_a, &bars->full[s], kb * BK, blk * BM, pol_a);
                        ptx::tma_load_2d(sa + STAGE_A_BYTES, &tm_b, &bars->full[s], kb * BK, brow, pol_b);
                    }
                }
                if (!ok)
                    record_error(ws.hdr, DEV_TIMEOUT);
                // drain: every issued load has landed before the CTA may exit
                const uint64_t dl = ptx::globaltimer() + static_cast<uint64_t>(c.timeout_ns);
                for (uint32_t i = it > STAGES ? it - STAGES : 0; i < it; ++i)
                    ptx::mbar_wait(&bars->full[i % STAGES], (i / STAGES) & 1u, dl);
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------ UMMA issuer -----
            if (lane == 0) {
                uint32_t it = 0, pit = 0;
                bool ok = true;
                for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                    for (int kb = 0; kb < NKB; ++kb, ++it, ++pit) {
                        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                        const uint32_t buf = pit & 1u, bph = (pit >> 1) & 1u;
                        if (!ptx::mbar_wait(&bars->full[s], ph, deadline) ||
                            !ptx::mbar_wait(&bars->tempty[buf], bph ^ 1u, deadline)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t a_addr = ptx::smem_u32(smem + s * STAGE_BYTES);
                        const uint64_t adesc = ptx::sw128_kmajor_desc(a_addr);
                        const uint64_t bdesc = ptx::sw128_kmajor_desc(a_addr + STAGE_A_BYTES);
                        const uint32_t dt = tmem + buf * BN;
    #pragma unroll
                        for (int k = 0; k < BK / 32; ++k)   // +32 bytes along K = +2 in the >>4 field
                            ptx::umma_f8(dt, adesc + 2 * k, bdesc + 2 * k, IDESC, k > 0 ? 1u : 0u);
                        ptx::umma_commit(&bars->empty[s]);
                        ptx::umma_commit(&bars->tfull[buf]);
                    }
                }
                if (!ok)
                    record_error(ws.hdr, DEV_TIMEOUT);
                // drain: the last commit arrives once every issued MMA has completed
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
        const float *sfa_base = PHASE == 1 ? ws.pool_sf : ws.act_sf;
        uint32_t pit = 0, tcount = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++tcount) {
            const int blk = tile / NT, nt = tile % NT;
            const int e = ws.block_expert[blk];
            const long long prow = static_cast<long long>(blk) * BM + row;
            const float *sfa = sfa_base + prow;
            const float *sb0;
            const float *sb1;
            if (PHASE == 1) {
                sb0 = sf_w + (static_cast<long long>(e) * (2 * d.I / 128) + nt) * NKB;              // gate
                sb1 = sf_w + (static_cast<long long>(e) * (2 * d.I / 128) + d.I / 128 + nt) * NKB;  // up
            } else {
                sb0 = sf_w + (static_cast<long long>(e) * (d.H / 128) + 2 * nt + wg) * NKB;
                sb1 = sb0;
            }
            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j)
                acc[j] = 0.0f;
            float a_nx = __ldg(sfa), b0_nx = __ldg(sb0), b1_nx = __ldg(sb1);
            for (int kb = 0; kb < NKB; ++kb, ++pit) {
                const float s0 = a_nx * b0_nx, s1 = a_nx * b1_nx;
                if (kb + 1 < NKB) {
                    a_nx = __ldg(sfa + static_cast<long long>(kb + 1) * ws.P);
                    b0_nx = __ldg(sb0 + kb + 1);
                    b1_nx = __ldg(sb1 + kb + 1);
                }
                const uint32_t buf = pit & 1u, bph = (pit >> 1) & 1u;
                // all lanes wait; the warp acts on a uniform verdict (tcgen05.ld is .aligned)
                if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&bars->tfull[buf], bph, deadline))) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t taddr = tmem + lane_base + buf * BN + wg * 128;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t r[32];
                    ptx::tmem_ld32(taddr + ch * 32, r);
                    ptx::tmem_ld_wait(r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        // gate/up interleave by 8: columns 8..15 of every 16 are "up"
                        const float sc = (PHASE == 1 && ((j >> 3) & 1)) ? s1 : s0;
                        acc[ch * 32 + j] = fmaf(__uint_as_float(r[j]), sc, acc[ch * 32 + j]);
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(&bars->tempty[buf]);
            }
            if (!ok)
                break;

            if (PHASE == 1) {
                // SwiGLU on the 64 (gate, up) pairs of this thread's row and column half,
                // then 1x128 requant of the row's 128 outputs of this n-tile (the two
                // column halves exchange their absolute maxima through shared memory).
                float amax = 0.0f;
#pragma unroll
                for (int m = 0; m < 64; ++m) {
                    const float g = acc[(m >> 3) * 16 + (m & 7)];
                    const float u = acc[(m >> 3) * 16 + 8 + (m & 7)];
                    const float hval = g / (1.0f + expf(-g)) * u;
                    acc[m] = hval;   // acc[m] is no longer needed as a gate/up input
                    amax = fmaxf(amax, fabsf(hval));
                }
                // exchange through slots of this tile's parity, behind a bounded mbarrier
                // (a slot is rewritten two tiles later, after every thread has passed the
                // next tile's exchange and so has read it)
                const uint32_t tp = tcount & 1u;
                bars->amax[tp][wg][row] = amax;
                ptx::mbar_arrive(&bars->xbar);
                if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&bars->xbar, tp, deadline))) {
                    ok = false;
                    break;
                }
                amax = fmaxf(bars->amax[tp][0][row], bars->amax[tp][1][row]);
                const float sf = fmaxf(amax, 1e-4f) / 448.0f;
                uint4 *dst = reinterpret_cast<uint4 *>(ws.act + prow * d.I + nt * 128 + wg * 64);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint32_t w4[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const int m = v * 16 + p * 4;
                        const uint32_t lo = ptx::cvt_e4m3x2(__fdiv_rn(acc[m], sf), __fdiv_rn(acc[m + 1], sf));
                        const uint32_t hi = ptx::cvt_e4m3x2(__fdiv_rn(acc[m + 2], sf), __fdiv_rn(acc[m + 3], sf));
                        w4[p] = lo | (hi << 16);
                    }
                    dst[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
                if (wg == 0)
                    ws.act_sf[static_cast<long long>(nt) * ws.P + prow] = sf;
            } else {
                if (row < ws.block_rows[blk]) {
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

template <int PHASE>
static cudaError_t launch_gemm(const CUtensorMap &tm_a, const CUtensorMap &tm_b, const Dims &d,
                               const Workspace &ws, const CallArgs &c, const float *sf_w, int num_sms,
                               cudaStream_t s)
{
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel<PHASE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             GEMM_SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    gemm_kernel<PHASE><<<num_sms, GEMM_THREADS, GEMM_SMEM_BYTES, s>>>(tm_a, tm_b, d, ws, c, sf_w);
    return cudaGetLastError();
}

cudaError_t launch_gemm_gate_up(const CUtensorMap &tm_a, const CUtensorMap &tm_b, const Dims &d,
                                const Workspace &ws, const CallArgs &c, const float *sf_w, int num_sms,
                                cudaStream_t s)
{
    return launch_gemm<1>(tm_a, tm_b, d, ws, c, sf_w, num_sms, s);
}

cudaError_t launch_gemm_down(const CUtensorMap &tm_a, const CUtensorMap &tm_b, const Dims &d,
                             const Workspace &ws, const CallArgs &c, const float *sf_w, int num_sms,
                             cudaStream_t s)
{
    return launch_gemm<2>(tm_a, tm_b, d, ws, c, sf_w, num_sms, s);
}

}  // namespace cpw
