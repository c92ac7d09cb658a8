// api.cu -- the C ABI declared in include/cpw_moe.h: handle, argument checks, workspace
// planning and allocation, weight re-layout, TMA descriptors, and the launch sequence of
// one forward:
//   dispatch (cooperative, one CTA per SM)  ->  expert FFN (cooperative, one CTA per SM:
//   gate_up GEMM + SwiGLU/requant, then down GEMM + weighted scatter)  ->
//   combine reduce + workspace reset
// all on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "../../include/cpw_moe.h"
#include "moe_internal.cuh"

using namespace cpw;

cudaError_t cpw::ensure_max_dynamic_smem(const void *kernel, int bytes)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, int> set_to;
    std::lock_guard<std::mutex> lock(mu);
    int &cur = set_to[{kernel, dev}];
    if (bytes <= cur)
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        cur = bytes;
    return e;
}

struct moe_ctx {
    int dev = -1;
    int num_sms = 0;
    Dims d{};                    // E, K include the shared experts (experts E_routed.., slots K_routed..)
    int E_routed = 0, K_routed = 0, S = 0;   // routed experts, routed top-k, shared experts
    bool reserved = false;
    bool have_weights = false;
    bool routed_loaded = false, shared_loaded = false;
    bool routed_pow2 = false, shared_pow2 = false;
    int fmt_routed = MOE_WEIGHTS_FP8, fmt_shared = MOE_WEIGHTS_FP8;   // format of each loaded set
    bool mxfp4 = false;          // the loaded weights are MXFP4 (block-scaled kernel, FP4 B tiles)
    Workspace ws{};
    void *small_mem = nullptr;   // header + routing arrays (size depends on E, R only)
    void *big_mem = nullptr;     // table, pools, combine, staging (depends on max_tokens)
    size_t small_bytes = 0, big_bytes = 0;
    uint8_t *w1 = nullptr;       // [E][2I/256][H/128][256][128] tiles, gate/up interleaved
    float *s1 = nullptr;         // [E][2I/128][H/128]
    uint8_t *w2 = nullptr;       // [E][H/256][I/128][256][128] tiles
    float *s2 = nullptr;         // [E][H/128][I/128]
    uint8_t *sfb1 = nullptr;     // UE8M0 scale blocks of the W1 / W2 tiles (1 KB per tile and
    uint8_t *sfb2 = nullptr;     // 128-deep K block), valid when every weight scale is 2^k
    uint32_t *sfb_bad = nullptr; // device flag: a weight scale is not a power of two
    bool weights_pow2 = false;
    void *w_mem = nullptr;
    size_t w_bytes = 0;
    FfnMaps maps{};              // a1 pool x, b1 W1, a2 act, b2 W2
    // MXFP4 weights (allocated by the first MXFP4 load): packed E2M1 tiles
    // [E][N/256][K/128][256][64] and UE8M0 scale blocks of 1 KB per weight tile and K block
    uint8_t *w41 = nullptr, *w42 = nullptr, *sfb41 = nullptr, *sfb42 = nullptr;
    uint32_t *sfb4_bad = nullptr;
    void *w4_mem = nullptr;
    size_t w4_bytes = 0;
    CUtensorMap b41{}, b42{};    // 16U4_ALIGN16B maps of the E2M1 tiles
    // staging buffers of moe_forward_host
    // (two input sets: an asynchronous call fills one with the copy engines on copy_stream
    // while the previous call's kernels still read the other)
    uint8_t *st_x[2] = {nullptr, nullptr};
    float *st_sf[2] = {nullptr, nullptr};
    int64_t *st_idx[2] = {nullptr, nullptr};
    float *st_w[2] = {nullptr, nullptr};
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t ev_staged[2] = {nullptr, nullptr};   // copy_stream: set filled
    cudaEvent_t ev_free[2] = {nullptr, nullptr};     // forward's stream: set no longer read
    bool free_recorded[2] = {false, false};
    unsigned host_calls = 0;
    uint16_t *st_out = nullptr;
    // shared experts: every token's route extended by slots K_routed.. (expert E_routed + s, weight 1)
    int64_t *ext_idx = nullptr;
    float *ext_w = nullptr;
    cudaStream_t last_stream = nullptr;
    bool have_last = false;
    int last_T = 0;
    long long timeout_ns = 2000000000LL;
    int debug_skip_barrier = 0;
    int ffn_mode = 0;            // 0 automatic, 1 one CTA per tile (the same kernel)
    int combine_mode = 2;        // 0 separate combine kernel, 1 inside the FFN kernel, 2 automatic
    int scale_mode = 2;          // 0 fp32 scales, 1 power-of-two scales (block-scaled UMMA),
                                 // 2 block-scaled exactly when the weights' scales are 2^k
    // stage profiling (events on the forward's stream)
    bool profile = false;
    int prof_every = 1;                // record every prof_every-th forward
    long long prof_seen = 0;           // forwards since profiling was enabled
    std::vector<cudaEvent_t> events;   // 4 per recorded forward
    int prof_calls = 0, prof_dropped = 0;
};

static constexpr int PROF_MAX_CALLS = 8192;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder()
{
    if (g_encode)
        return MOE_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return MOE_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return MOE_OK;
}

// 2-D byte matrix [rows][cols] (row-major), tiles of BKS bytes x box_rows, swizzled at
// BKS bytes (the layout the UMMA shared-memory descriptors of the FFN kernel expect).
int encode_tile_map(CUtensorMap *m, void *base, uint64_t rows, uint64_t cols, uint32_t box_rows)
{
    if (get_encoder() != MOE_OK)
        return MOE_ERR_CUDA;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BKS), box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = BKS == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : BKS == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// Packed E2M1 weight tiles as rows of 64 bytes (128 four-bit values), element type
// 16U4_ALIGN16B: a box of 128 values x box_rows lands in shared memory as 128-byte rows (each
// 8 packed bytes followed by an 8-byte gap), swizzled at 128 bytes like an e4m3 tile; the
// transaction count is the packed bytes.  Needs a 32-byte aligned base.
int encode_fp4_tile_map(CUtensorMap *m, void *base, uint64_t rows, uint32_t box_rows)
{
    if (get_encoder() != MOE_OK || reinterpret_cast<uintptr_t>(base) % 32 != 0)
        return MOE_ERR_CUDA;
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {64};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// 256-row tiles of the down weight (H rows; the last tile is half zero rows when H is an odd
// multiple of 128)
inline int h_tiles(const Dims &d) { return (d.H + BN - 1) / BN; }

// Bump allocator over one cudaMalloc'd block.
struct Carver {
    char *base;
    size_t off = 0;
    template <typename T>
    T *take(size_t count)
    {
        off = align_up(off, 256);
        T *p = reinterpret_cast<T *>(base ? base + off : nullptr);
        off += count * sizeof(T);
        return p;
    }
};

#define CK(x)                                  \
    do {                                       \
        if ((x) != cudaSuccess)                \
            return MOE_ERR_CUDA;               \
    } while (0)

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

void free_big(moe_ctx *h)
{
    if (h->copy_stream)
        cudaStreamSynchronize(h->copy_stream);
    h->free_recorded[0] = h->free_recorded[1] = false;
    if (h->big_mem)
        cudaFree(h->big_mem);
    h->big_mem = nullptr;
    h->big_bytes = 0;
    h->reserved = false;
}

// Carve the max_tokens-dependent part of the workspace; with base == nullptr only sizes it.
size_t carve_big(moe_ctx *h, char *base, int max_tokens, Workspace &ws)
{
    const Dims &d = h->d;
    Carver c{base};
    const int tsrc_cap = std::max(1, max_tokens / d.R);
    const long long routed = static_cast<long long>(max_tokens) * d.K;
    const int max_blocks = static_cast<int>((routed + BM - 1) / BM) + d.E;
    const long long P = static_cast<long long>(max_blocks) * BM;
    ws.tsrc_cap = tsrc_cap;
    ws.max_blocks = max_blocks;
    ws.P = static_cast<int>(P);
    ws.max_tokens = max_tokens;
    ws.block_expert = c.take<int32_t>(max_blocks);
    ws.block_rows = c.take<int32_t>(max_blocks);
    ws.arrive = c.take<uint32_t>(max_blocks);
    ws.l1_done = c.take<uint32_t>(max_blocks);
    ws.tok_mask = c.take<uint32_t>(max_tokens);
    ws.tok_cnt = c.take<uint32_t>(static_cast<size_t>(max_tokens) * ((d.H + BN - 1) / BN));
    ws.table = c.take<int32_t>(static_cast<size_t>(d.E) * d.R * tsrc_cap);
    ws.meta = c.take<uint32_t>(static_cast<size_t>(P) * 3);
    ws.pool_x = c.take<uint8_t>(static_cast<size_t>(P) * d.H);
    ws.pool_sf = c.take<float>(static_cast<size_t>(P) * (d.H / 128));
    ws.pool_sfe = c.take<uint8_t>(static_cast<size_t>(P) * (d.H / 32));
    ws.act = c.take<uint8_t>(static_cast<size_t>(P) * d.I);
    ws.act_sf = c.take<float>(static_cast<size_t>(P) * (d.I / 128));
    ws.act_sfe = c.take<uint8_t>(static_cast<size_t>(P) * (d.I / 32));
    ws.combine = c.take<uint16_t>(static_cast<size_t>(d.K) * max_tokens * d.H);
    for (int i = 0; i < 2; ++i) {
        h->st_x[i] = c.take<uint8_t>(static_cast<size_t>(max_tokens) * d.H);
        h->st_sf[i] = c.take<float>(static_cast<size_t>(max_tokens) * (d.H / 128));
        h->st_idx[i] = c.take<int64_t>(static_cast<size_t>(max_tokens) * d.K);
        h->st_w[i] = c.take<float>(static_cast<size_t>(max_tokens) * d.K);
    }
    h->st_out = c.take<uint16_t>(static_cast<size_t>(max_tokens) * d.H);
    if (h->S > 0) {
        h->ext_idx = c.take<int64_t>(static_cast<size_t>(max_tokens) * d.K);
        h->ext_w = c.take<float>(static_cast<size_t>(max_tokens) * d.K);
    }
    return align_up(c.off, 256);
}

// M-blocks per expert wave of the FFN kernel: the SwiGLU output of one wave
// (blocks x 128 rows x I bytes) should stay within half of the 129 MB L2 until the
// down-projection tiles of the same wave read it back.
int wave_blocks(const moe_ctx *h)
{
    const long long per_block = static_cast<long long>(BM) * h->d.I;
    const long long half_l2 = 64ll << 20;
    return static_cast<int>(std::max(1ll, half_l2 / per_block));
}

int sync_last(moe_ctx *h)
{
    if (h->have_last)
        CK(cudaStreamSynchronize(h->last_stream));
    return MOE_OK;
}

}  // namespace

extern "C" {

const char *moe_status_string(int s)
{
    switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_CAPACITY: return "token count above the reserved maximum";
    case MOE_ERR_NO_WEIGHTS: return "weights not loaded";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "unsupported device or shape";
    case MOE_ERR_BAD_INDEX: return "expert id outside [0,E) (device)";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_SLOT_OVERFLOW: return "more than T/R rows of one source for one expert (device)";
    case MOE_ERR_NOT_RESERVED: return "workspace not reserved";
    case MOE_ERR_BAD_SCALE: return "a scale is not a power of two in the block-scaled mode";
    default: return "unknown status";
    }
}

int moe_create(int E, int H, int I, int topk, int R, moe_handle_t *out)
{
    return moe_create_shared(E, H, I, topk, R, 0, out);
}

int moe_create_shared(int E, int H, int I, int topk, int R, int n_shared, moe_handle_t *out)
{
    if (!out)
        return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    if (E < 1 || H < 128 || H % 128 != 0 || H / 128 > MAX_KB || I / 128 > MAX_KB || I < 128 || I % 128 != 0 || topk < 1 || topk > E || R < 1 ||
        R > 64 || n_shared < 0 || E + n_shared > 1024 || topk + n_shared > 32 || (E + n_shared) * R > 16384)
        return MOE_ERR_INVALID_ARG;
    int dev = 0;
    CK(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    CK(cudaGetDeviceProperties(&prop, dev));
    if (!(prop.major == 10 && prop.minor == 3))
        return MOE_ERR_UNSUPPORTED_DEVICE;
    moe_ctx *h = new (std::nothrow) moe_ctx();
    if (!h)
        return MOE_ERR_INVALID_ARG;
    h->dev = dev;
    h->num_sms = prop.multiProcessorCount;
    h->d = Dims{E + n_shared, H, I, topk + n_shared, R};
    h->E_routed = E;
    h->K_routed = topk;
    h->S = n_shared;
    *out = h;
    return MOE_OK;
}

int moe_reserve(moe_handle_t h, int max_tokens)
{
    if (!h || max_tokens < 1)
        return MOE_ERR_INVALID_ARG;
    if (h->reserved && h->ws.max_tokens >= max_tokens)
        return MOE_OK;
    CK(cudaSetDevice(h->dev));
    if (sync_last(h) != MOE_OK)
        return MOE_ERR_CUDA;
    const Dims &d = h->d;
    if (!h->small_mem) {
        Carver c{nullptr};
        Workspace &ws = h->ws;
        auto carve_small = [&](char *base) {
            c = Carver{base};
            ws.hdr = c.take<uint32_t>(HDR_WORDS);
            ws.send = c.take<unsigned long long>(static_cast<size_t>(d.R) * d.E);
            ws.counts = c.take<uint32_t>(d.E);
            ws.recv = c.take<uint32_t>(static_cast<size_t>(d.E) * d.R);
            ws.blk_off = c.take<int32_t>(d.E + 1);
            ws.cum_rows = c.take<unsigned long long>(d.E);
            return align_up(c.off, 256);
        };
        const size_t bytes = carve_small(nullptr);
        CK(cudaMalloc(&h->small_mem, bytes));
        carve_small(static_cast<char *>(h->small_mem));
        h->small_bytes = bytes;
        CK(cudaMemset(h->small_mem, 0, bytes));
    }
    free_big(h);
    Workspace ws = h->ws;
    const size_t bytes = carve_big(h, nullptr, max_tokens, ws);
    if (cudaMalloc(&h->big_mem, bytes) != cudaSuccess) {
        h->big_mem = nullptr;
        return MOE_ERR_CUDA;
    }
    carve_big(h, static_cast<char *>(h->big_mem), max_tokens, ws);
    h->ws = ws;
    h->big_bytes = bytes;
    CK(cudaMemset(ws.arrive, 0, sizeof(uint32_t) * ws.max_blocks));
    CK(cudaMemset(ws.l1_done, 0, sizeof(uint32_t) * ws.max_blocks));
    CK(cudaMemset(ws.tok_cnt, 0, sizeof(uint32_t) * static_cast<size_t>(max_tokens) * ((d.H + BN - 1) / BN)));
    CK(cudaMemset(ws.pool_sf, 0, sizeof(float) * static_cast<size_t>(ws.P) * (d.H / 128)));
    CK(cudaMemset(ws.act_sf, 0, sizeof(float) * static_cast<size_t>(ws.P) * (d.I / 128)));
    CK(cudaMemset(ws.pool_x, 0, static_cast<size_t>(ws.P) * d.H));
    CK(cudaMemset(ws.act, 0, static_cast<size_t>(ws.P) * d.I));
    if (encode_tile_map(&h->maps.a1, ws.pool_x, ws.P, d.H, BM) != MOE_OK ||
        encode_tile_map(&h->maps.a2, ws.act, ws.P, d.I, BM) != MOE_OK ||
        encode_tile_map(&h->maps.a1p, ws.pool_x, ws.P, d.H, A_ROWS_PART) != MOE_OK ||
        encode_tile_map(&h->maps.a2p, ws.act, ws.P, d.I, A_ROWS_PART) != MOE_OK ||
        encode_tile_map(&h->maps.a1h, ws.pool_x, ws.P, d.H, 2 * A_ROWS_PART) != MOE_OK ||
        encode_tile_map(&h->maps.a2h, ws.act, ws.P, d.I, 2 * A_ROWS_PART) != MOE_OK)
        return MOE_ERR_CUDA;
    CK(cudaDeviceSynchronize());
    h->reserved = true;
    return MOE_OK;
}

namespace {

// Weights of experts [e0, e0 + n) of the handle's expert slots (routed experts first, then
// the shared ones): re-laid into GEMM tiles, scales copied, UE8M0 scale blocks built;
// *pow2 = every scale of these experts is a power of two.
int load_expert_weights(moe_ctx *h, int e0, int n, const uint8_t *w_gate_up, const float *sf_gate_up,
                        const uint8_t *w_down, const float *sf_down, cudaStream_t s, bool *pow2)
{
    if (!w_gate_up || !sf_gate_up || !w_down || !sf_down)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(w_gate_up, 16) || !aligned(w_down, 16) || !aligned(sf_gate_up, 4) || !aligned(sf_down, 4))
        return MOE_ERR_INVALID_ARG;
    CK(cudaSetDevice(h->dev));
    const Dims &d = h->d;
    // down-weight tiles cover H rounded up to the 256-row tile (zero rows past H)
    const size_t w1e = static_cast<size_t>(2) * d.I * d.H, w2e = static_cast<size_t>(h_tiles(d)) * BN * d.I;
    const size_t s1e = static_cast<size_t>(2 * d.I / 128) * (d.H / 128), s2e = static_cast<size_t>(d.H / 128) * (d.I / 128);
    // UE8M0 scale blocks: 1 KB per weight tile and group of four 128-deep K blocks
    const size_t b1e = static_cast<size_t>(2 * d.I / BN) * ((d.H / 128 + 3) / 4) * 1024,
                 b2e = static_cast<size_t>(h_tiles(d)) * ((d.I / 128 + 3) / 4) * 1024;
    const size_t n1 = d.E * w1e, n2 = d.E * w2e;
    if (!h->w_mem) {
        Carver c{nullptr};
        auto carve = [&](char *base) {
            c = Carver{base};
            h->w1 = c.take<uint8_t>(n1);
            h->s1 = c.take<float>(d.E * s1e);
            h->w2 = c.take<uint8_t>(n2);
            h->s2 = c.take<float>(d.E * s2e);
            h->sfb1 = c.take<uint8_t>(d.E * b1e);
            h->sfb2 = c.take<uint8_t>(d.E * b2e);
            h->sfb_bad = c.take<uint32_t>(1);
            return align_up(c.off, 256);
        };
        const size_t bytes = carve(nullptr);
        CK(cudaMalloc(&h->w_mem, bytes));
        carve(static_cast<char *>(h->w_mem));
        h->w_bytes = bytes;
    }
    if (launch_relayout_weights(w_gate_up, h->w1 + e0 * w1e, n, 2 * d.I, d.H, d.I, 128, s) != cudaSuccess ||
        launch_relayout_weights(w_down, h->w2 + e0 * w2e, n, d.H, d.I, 0, 128, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    CK(cudaMemcpyAsync(h->s1 + e0 * s1e, sf_gate_up, n * s1e * sizeof(float), cudaMemcpyDeviceToDevice, s));
    CK(cudaMemcpyAsync(h->s2 + e0 * s2e, sf_down, n * s2e * sizeof(float), cudaMemcpyDeviceToDevice, s));
    // UE8M0 scale blocks for the block-scaled path; usable only if every scale is 2^k
    CK(cudaMemsetAsync(h->sfb_bad, 0, sizeof(uint32_t), s));
    if (launch_build_sfb(sf_gate_up, h->sfb1 + e0 * b1e, n, 2 * d.I, d.H, d.I, h->sfb_bad, s) != cudaSuccess ||
        launch_build_sfb(sf_down, h->sfb2 + e0 * b2e, n, d.H, d.I, 0, h->sfb_bad, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    uint32_t bad = 1;
    CK(cudaMemcpyAsync(&bad, h->sfb_bad, sizeof(uint32_t), cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    *pow2 = bad == 0;
    // weight tiles as rows of 128 bytes: tile (e, nt, kb) starts at row ((e*NT + nt)*KB + kb)*256
    if (encode_tile_map(&h->maps.b1, h->w1, n1 / 128, 128, BN) != MOE_OK ||
        encode_tile_map(&h->maps.b2, h->w2, n2 / 128, 128, BN) != MOE_OK)
        return MOE_ERR_CUDA;
    h->last_stream = s;
    h->have_last = true;
    return MOE_OK;
}

// MXFP4 weights of experts [e0, e0 + n): packed E2M1 rows re-laid into 16 KB GEMM tiles,
// UE8M0 scales into per-(tile, K block) scale blocks.  MOE_ERR_BAD_SCALE if a scale byte is
// 0xFF (NaN).
int load_expert_weights_mxfp4(moe_ctx *h, int e0, int n, const uint8_t *w_gate_up, const uint8_t *sf_gate_up,
                              const uint8_t *w_down, const uint8_t *sf_down, cudaStream_t s)
{
    if (!w_gate_up || !sf_gate_up || !w_down || !sf_down)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(w_gate_up, 16) || !aligned(w_down, 16) || !aligned(sf_gate_up, 4) || !aligned(sf_down, 4))
        return MOE_ERR_INVALID_ARG;
    CK(cudaSetDevice(h->dev));
    const Dims &d = h->d;
    const size_t w1e = static_cast<size_t>(2) * d.I * (d.H / 2), w2e = static_cast<size_t>(h_tiles(d)) * BN * (d.I / 2);
    const size_t b1e = static_cast<size_t>(2 * d.I / BN) * (d.H / 128) * 1024,
                 b2e = static_cast<size_t>(h_tiles(d)) * (d.I / 128) * 1024;
    const size_t n1 = d.E * w1e, n2 = d.E * w2e;
    if (!h->w4_mem) {
        Carver c{nullptr};
        auto carve = [&](char *base) {
            c = Carver{base};
            h->w41 = c.take<uint8_t>(n1);
            h->w42 = c.take<uint8_t>(n2);
            h->sfb41 = c.take<uint8_t>(d.E * b1e);
            h->sfb42 = c.take<uint8_t>(d.E * b2e);
            h->sfb4_bad = c.take<uint32_t>(1);
            return align_up(c.off, 256);
        };
        const size_t bytes = carve(nullptr);
        CK(cudaMalloc(&h->w4_mem, bytes));
        carve(static_cast<char *>(h->w4_mem));
        h->w4_bytes = bytes;
    }
    if (launch_relayout_weights(w_gate_up, h->w41 + e0 * w1e, n, 2 * d.I, d.H, d.I, 64, s) != cudaSuccess ||
        launch_relayout_weights(w_down, h->w42 + e0 * w2e, n, d.H, d.I, 0, 64, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    CK(cudaMemsetAsync(h->sfb4_bad, 0, sizeof(uint32_t), s));
    if (launch_build_sfb4(sf_gate_up, h->sfb41 + e0 * b1e, n, 2 * d.I, d.H, d.I, h->sfb4_bad, s) != cudaSuccess ||
        launch_build_sfb4(sf_down, h->sfb42 + e0 * b2e, n, d.H, d.I, 0, h->sfb4_bad, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    uint32_t bad = 1;
    CK(cudaMemcpyAsync(&bad, h->sfb4_bad, sizeof(uint32_t), cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    // tile (e, nt, kb) starts at 64-byte row ((e*NT + nt)*KB + kb)*256
    if (encode_fp4_tile_map(&h->b41, h->w41, n1 / 64, BN) != MOE_OK ||
        encode_fp4_tile_map(&h->b42, h->w42, n2 / 64, BN) != MOE_OK)
        return MOE_ERR_CUDA;
    h->last_stream = s;
    h->have_last = true;
    return bad ? MOE_ERR_BAD_SCALE : MOE_OK;
}

void update_weight_state(moe_ctx *h)
{
    // routed and shared experts run in one kernel: both sets in one format
    h->have_weights = h->routed_loaded && (h->S == 0 || (h->shared_loaded && h->fmt_shared == h->fmt_routed));
    h->weights_pow2 = h->routed_pow2 && (h->S == 0 || h->shared_pow2);
    h->mxfp4 = h->fmt_routed == MOE_WEIGHTS_MXFP4;
}

}  // namespace

int moe_load_weights(moe_handle_t h, const uint8_t *w_gate_up, const float *sf_gate_up,
                     const uint8_t *w_down, const float *sf_down, void *stream)
{
    if (!h)
        return MOE_ERR_INVALID_ARG;
    h->routed_loaded = false;
    const int rc = load_expert_weights(h, 0, h->E_routed, w_gate_up, sf_gate_up, w_down, sf_down,
                                       static_cast<cudaStream_t>(stream), &h->routed_pow2);
    if (rc == MOE_OK) {
        h->routed_loaded = true;
        h->fmt_routed = MOE_WEIGHTS_FP8;
    }
    update_weight_state(h);
    return rc;
}

int moe_load_shared_weights(moe_handle_t h, const uint8_t *w_gate_up, const float *sf_gate_up,
                            const uint8_t *w_down, const float *sf_down, void *stream)
{
    if (!h || h->S == 0)
        return MOE_ERR_INVALID_ARG;
    h->shared_loaded = false;
    const int rc = load_expert_weights(h, h->E_routed, h->S, w_gate_up, sf_gate_up, w_down, sf_down,
                                       static_cast<cudaStream_t>(stream), &h->shared_pow2);
    if (rc == MOE_OK) {
        h->shared_loaded = true;
        h->fmt_shared = MOE_WEIGHTS_FP8;
    }
    update_weight_state(h);
    return rc;
}

int moe_load_weights_mxfp4(moe_handle_t h, const uint8_t *w_gate_up, const uint8_t *sf_gate_up,
                           const uint8_t *w_down, const uint8_t *sf_down, void *stream)
{
    if (!h)
        return MOE_ERR_INVALID_ARG;
    h->routed_loaded = false;
    const int rc = load_expert_weights_mxfp4(h, 0, h->E_routed, w_gate_up, sf_gate_up, w_down, sf_down,
                                             static_cast<cudaStream_t>(stream));
    if (rc == MOE_OK) {
        h->routed_loaded = true;
        h->fmt_routed = MOE_WEIGHTS_MXFP4;
        h->routed_pow2 = true;
    }
    update_weight_state(h);
    return rc;
}

int moe_load_shared_weights_mxfp4(moe_handle_t h, const uint8_t *w_gate_up, const uint8_t *sf_gate_up,
                                  const uint8_t *w_down, const uint8_t *sf_down, void *stream)
{
    if (!h || h->S == 0)
        return MOE_ERR_INVALID_ARG;
    h->shared_loaded = false;
    const int rc = load_expert_weights_mxfp4(h, h->E_routed, h->S, w_gate_up, sf_gate_up, w_down, sf_down,
                                             static_cast<cudaStream_t>(stream));
    if (rc == MOE_OK) {
        h->shared_loaded = true;
        h->fmt_shared = MOE_WEIGHTS_MXFP4;
        h->shared_pow2 = true;
    }
    update_weight_state(h);
    return rc;
}

// out_is_host: the output is pinned host memory the kernels write in place (host-buffer entry
// points); the automatic combine mode then runs the combine inside the FFN kernel, so the
// output rows cross to the host while the GEMMs still run instead of in one burst at the end.
static int forward_impl(moe_handle_t h, int T, const uint8_t *x, const float *x_sf, const int64_t *topk_idx,
                        const float *topk_w, uint16_t *out, void *stream, bool out_is_host)
{
    if (!h || T < 0)
        return MOE_ERR_INVALID_ARG;
    if (!h->reserved)
        return MOE_ERR_NOT_RESERVED;
    if (!h->have_weights)
        return MOE_ERR_NO_WEIGHTS;
    if (T > h->ws.max_tokens)
        return MOE_ERR_CAPACITY;
    if (T % h->d.R != 0)
        return MOE_ERR_INVALID_ARG;
    if (T == 0)
        return MOE_OK;
    if (!x || !x_sf || !topk_idx || !topk_w || !out)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(out, 16) || !aligned(x_sf, 4) || !aligned(topk_idx, 8) ||
        !aligned(topk_w, 4))
        return MOE_ERR_INVALID_ARG;
    CK(cudaSetDevice(h->dev));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // power-of-two scales: the block-scaled kernel (the weights were checked at load time,
    // the activation scales are checked by the routing kernel's gather); MXFP4 weights run
    // only there
    if ((h->scale_mode == 1 && !h->weights_pow2) || (h->scale_mode == 0 && h->mxfp4))
        return MOE_ERR_BAD_SCALE;
    const bool bs = h->mxfp4 || h->scale_mode == 1 || (h->scale_mode == 2 && h->weights_pow2);
    // automatic combine: inside the FFN kernel for an output written in place into pinned host
    // memory by the block-scaled kernel, whose epilogue warps have slack; the fp32-scale kernel's
    // epilogue is its critical path, so there the combine kernel writes the output in place
    const int fused = h->combine_mode == 2 ? ((out_is_host && bs) ? 1 : 0) : h->combine_mode;
    CallArgs c{T, x, x_sf, topk_idx, topk_w, out, h->timeout_ns, h->debug_skip_barrier, bs ? 1 : 0, fused};
    if (h->S > 0) {
        // shared experts: each token's route gains slots K_routed.. naming expert E_routed + s
        // with weight 1, written by one small kernel ahead of the routing kernel
        c.idx = h->ext_idx;
        c.w = h->ext_w;
    }
    cudaEvent_t *ev = nullptr;
    if (h->profile && (h->prof_seen++ % h->prof_every) == 0) {
        if (h->prof_calls < PROF_MAX_CALLS)
            ev = &h->events[static_cast<size_t>(h->prof_calls++) * 4];
        else
            ++h->prof_dropped;
    }
    auto mark = [&](int i) { return ev ? cudaEventRecord(ev[i], s) : cudaSuccess; };
    // MXFP4: the weight-tile maps of the E2M1 tiles
    FfnMaps maps4 = h->maps;
    if (h->mxfp4) {
        maps4.b1 = h->b41;
        maps4.b2 = h->b42;
    }
    if (mark(0) != cudaSuccess ||
        (h->S > 0 && launch_extend_route(topk_idx, topk_w, h->ext_idx, h->ext_w, T, h->K_routed, h->S, h->E_routed,
                                         h->num_sms, s) != cudaSuccess) ||
        launch_dispatch(h->d, h->ws, c, h->num_sms, s) != cudaSuccess ||
        mark(1) != cudaSuccess ||
        (bs ? launch_ffn_bs(maps4, h->d, h->ws, c, h->mxfp4 ? h->sfb41 : h->sfb1, h->mxfp4 ? h->sfb42 : h->sfb2,
                            wave_blocks(h), h->num_sms, h->mxfp4, s)
            : launch_ffn(h->maps, h->d, h->ws, c, h->s1, h->s2, wave_blocks(h), h->num_sms, s)) !=
            cudaSuccess ||
        mark(2) != cudaSuccess || (!c.fused_combine && launch_combine(h->d, h->ws, c, h->num_sms, s) != cudaSuccess) ||
        mark(3) != cudaSuccess)
        return MOE_ERR_CUDA;
    h->last_stream = s;
    h->have_last = true;
    h->last_T = T;
    return MOE_OK;
}

int moe_forward(moe_handle_t h, int T, const uint8_t *x, const float *x_sf, const int64_t *topk_idx,
                const float *topk_w, uint16_t *out, void *stream)
{
    return forward_impl(h, T, x, x_sf, topk_idx, topk_w, out, stream, false);
}

// Device address of a host buffer the GPU can access in place (pinned, mapped into the
// device's address space), or nullptr (pageable memory: it goes through a copy).
static void *mapped_host(const void *p)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// Shared body of the host-buffer entry points.  Asynchronous calls with pinned inputs copy
// them with the copy engines on a side stream into one of two staging sets, so the copies of
// call i+1 overlap the kernels of call i (the forward waits for its copies by an event, and
// a set is refilled only after the forward that read it).  Otherwise pinned inputs are read
// in place by one staging kernel (16-byte aligned buffers) and pageable ones copied on the
// forward's stream.  The output is written in place when it is pinned and 16-byte aligned (by
// the block-scaled FFN kernel in the automatic combine mode, else by the combine kernel), else
// copied back from the staging buffer.
static int forward_host_impl(moe_handle_t h, int T, const uint8_t *host_x, const float *host_x_sf,
                             const int64_t *host_topk_idx, const float *host_topk_w, uint16_t *host_out,
                             void *stream, bool wait)
{
    if (!h || T < 0)
        return MOE_ERR_INVALID_ARG;
    if (!h->reserved)
        return MOE_ERR_NOT_RESERVED;
    if (T > h->ws.max_tokens)
        return MOE_ERR_CAPACITY;
    if (T == 0)
        return MOE_OK;
    if (!host_x || !host_x_sf || !host_topk_idx || !host_topk_w || !host_out)
        return MOE_ERR_INVALID_ARG;
    if (T % h->d.R != 0)
        return MOE_ERR_INVALID_ARG;
    CK(cudaSetDevice(h->dev));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Dims &d = h->d;
    const void *src[4] = {host_x, host_x_sf, host_topk_idx, host_topk_w};
    const long long bytes[4] = {static_cast<long long>(T) * d.H, 4ll * T * (d.H / 128), 8ll * T * h->K_routed,
                                4ll * T * h->K_routed};
    const void *dev_src[4];
    bool pinned = true, in_place = true;
    for (int i = 0; i < 4; ++i) {
        dev_src[i] = mapped_host(src[i]);
        pinned = pinned && dev_src[i] != nullptr;
        in_place = in_place && dev_src[i] != nullptr && aligned(dev_src[i], 16);
    }
    int set = 0;
    if (!wait && pinned) {
        if (!h->copy_stream) {
            CK(cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking));
            for (int i = 0; i < 2; ++i) {
                CK(cudaEventCreateWithFlags(&h->ev_staged[i], cudaEventDisableTiming));
                CK(cudaEventCreateWithFlags(&h->ev_free[i], cudaEventDisableTiming));
            }
        }
        set = static_cast<int>(h->host_calls++ & 1u);
        void *dst[4] = {h->st_x[set], h->st_sf[set], h->st_idx[set], h->st_w[set]};
        if (h->free_recorded[set])
            CK(cudaStreamWaitEvent(h->copy_stream, h->ev_free[set], 0));
        for (int i = 0; i < 4; ++i)
            CK(cudaMemcpyAsync(dst[i], src[i], static_cast<size_t>(bytes[i]), cudaMemcpyHostToDevice,
                               h->copy_stream));
        CK(cudaEventRecord(h->ev_staged[set], h->copy_stream));
        CK(cudaStreamWaitEvent(s, h->ev_staged[set], 0));
    } else {
        // set 0: any asynchronous call that used it has been waited for by this stream order
        // (its forward ran on a stream this call follows) or by a synchronous return
        if (h->free_recorded[0])
            CK(cudaStreamWaitEvent(s, h->ev_free[0], 0));
        void *dst[4] = {h->st_x[0], h->st_sf[0], h->st_idx[0], h->st_w[0]};
        if (in_place) {
            CK(launch_stage_inputs(dev_src, dst, bytes, h->num_sms, s));
        } else {
            for (int i = 0; i < 4; ++i)
                CK(cudaMemcpyAsync(dst[i], src[i], static_cast<size_t>(bytes[i]), cudaMemcpyHostToDevice, s));
        }
    }
    uint16_t *out_dev = static_cast<uint16_t *>(mapped_host(host_out));
    const bool out_in_place = out_dev != nullptr && aligned(out_dev, 16);
    int rc = forward_impl(h, T, h->st_x[set], h->st_sf[set], h->st_idx[set], h->st_w[set],
                          out_in_place ? out_dev : h->st_out, stream, out_in_place);
    if (rc != MOE_OK)
        return rc;
    if (h->ev_free[set]) {
        CK(cudaEventRecord(h->ev_free[set], s));
        h->free_recorded[set] = true;
    }
    if (!out_in_place)
        CK(cudaMemcpyAsync(host_out, h->st_out, sizeof(uint16_t) * T * d.H, cudaMemcpyDeviceToHost, s));
    if (wait)
        CK(cudaStreamSynchronize(s));
    return MOE_OK;
}

int moe_forward_host(moe_handle_t h, int T, const uint8_t *host_x, const float *host_x_sf,
                     const int64_t *host_topk_idx, const float *host_topk_w, uint16_t *host_out,
                     void *stream)
{
    return forward_host_impl(h, T, host_x, host_x_sf, host_topk_idx, host_topk_w, host_out, stream, true);
}

int moe_forward_host_async(moe_handle_t h, int T, const uint8_t *host_x, const float *host_x_sf,
                           const int64_t *host_topk_idx, const float *host_topk_w, uint16_t *host_out,
                           void *stream)
{
    return forward_host_impl(h, T, host_x, host_x_sf, host_topk_idx, host_topk_w, host_out, stream, false);
}

int moe_get_error(moe_handle_t h, int *device_status)
{
    if (!h || !device_status)
        return MOE_ERR_INVALID_ARG;
    *device_status = MOE_OK;
    if (!h->small_mem)
        return MOE_OK;
    CK(cudaSetDevice(h->dev));
    if (sync_last(h) != MOE_OK)
        return MOE_ERR_CUDA;
    uint32_t hdr[HDR_WORDS];
    CK(cudaMemcpy(hdr, h->ws.hdr, sizeof(hdr), cudaMemcpyDeviceToHost));
    const uint32_t st = hdr[HDR_ERR_STICKY] ? hdr[HDR_ERR_STICKY] : hdr[HDR_ERR_CALL];
    if (st != 0) {
        CK(cudaMemset(h->ws.hdr, 0, sizeof(uint32_t) * HDR_WORDS));
        CK(cudaMemset(h->ws.send, 0, sizeof(unsigned long long) * h->d.R * h->d.E));
        if (h->reserved) {
            CK(cudaMemset(h->ws.arrive, 0, sizeof(uint32_t) * h->ws.max_blocks));
            CK(cudaMemset(h->ws.l1_done, 0, sizeof(uint32_t) * h->ws.max_blocks));
            CK(cudaMemset(h->ws.tok_cnt, 0,
                          sizeof(uint32_t) * static_cast<size_t>(h->ws.max_tokens) * ((h->d.H + BN - 1) / BN)));
        }
        CK(cudaDeviceSynchronize());
    }
    *device_status = static_cast<int>(st);
    return MOE_OK;
}

int moe_debug_routing(moe_handle_t h, uint32_t *counts, uint32_t *recv, int32_t *block_offset,
                      uint32_t *meta, int *P, int *block_m)
{
    if (!h)
        return MOE_ERR_INVALID_ARG;
    if (!h->reserved)
        return MOE_ERR_NOT_RESERVED;
    CK(cudaSetDevice(h->dev));
    if (sync_last(h) != MOE_OK)
        return MOE_ERR_CUDA;
    const Dims &d = h->d;
    int32_t off_last = 0;
    CK(cudaMemcpy(&off_last, h->ws.blk_off + d.E, sizeof(int32_t), cudaMemcpyDeviceToHost));
    if (off_last < 0 || off_last > h->ws.max_blocks)
        return MOE_ERR_CUDA;
    if (counts)
        CK(cudaMemcpy(counts, h->ws.counts, sizeof(uint32_t) * d.E, cudaMemcpyDeviceToHost));
    if (recv)
        CK(cudaMemcpy(recv, h->ws.recv, sizeof(uint32_t) * d.E * d.R, cudaMemcpyDeviceToHost));
    if (block_offset)
        CK(cudaMemcpy(block_offset, h->ws.blk_off, sizeof(int32_t) * (d.E + 1), cudaMemcpyDeviceToHost));
    if (meta && off_last > 0)
        CK(cudaMemcpy(meta, h->ws.meta, sizeof(uint32_t) * 3 * static_cast<size_t>(off_last) * BM,
                      cudaMemcpyDeviceToHost));
    if (P)
        *P = off_last * BM;
    if (block_m)
        *block_m = BM;
    return MOE_OK;
}

int moe_cumulative_expert_rows(moe_handle_t h, uint64_t *rows)
{
    if (!h || !rows)
        return MOE_ERR_INVALID_ARG;
    if (!h->small_mem) {
        std::memset(rows, 0, sizeof(uint64_t) * h->d.E);
        return MOE_OK;
    }
    CK(cudaSetDevice(h->dev));
    if (sync_last(h) != MOE_OK)
        return MOE_ERR_CUDA;
    CK(cudaMemcpy(rows, h->ws.cum_rows, sizeof(uint64_t) * h->d.E, cudaMemcpyDeviceToHost));
    return MOE_OK;
}

int moe_debug_buffer(moe_handle_t h, int which, void *host_dst, uint64_t bytes)
{
    if (!h || !host_dst)
        return MOE_ERR_INVALID_ARG;
    if (!h->reserved)
        return MOE_ERR_NOT_RESERVED;
    const Dims &d = h->d;
    const Workspace &ws = h->ws;
    const void *src = nullptr;
    uint64_t need = 0;
    switch (which) {
    case MOE_BUF_POOL_X: src = ws.pool_x; need = static_cast<uint64_t>(ws.P) * d.H; break;
    case MOE_BUF_POOL_SF: src = ws.pool_sf; need = 4ull * ws.P * (d.H / 128); break;
    case MOE_BUF_ACT: src = ws.act; need = static_cast<uint64_t>(ws.P) * d.I; break;
    case MOE_BUF_ACT_SF: src = ws.act_sf; need = 4ull * ws.P * (d.I / 128); break;
    case MOE_BUF_COMBINE: src = ws.combine; need = 2ull * d.K * ws.max_tokens * d.H; break;
    case MOE_BUF_TABLE: src = ws.table; need = 4ull * d.E * d.R * ws.tsrc_cap; break;
    default: return MOE_ERR_INVALID_ARG;
    }
    if (bytes != need)
        return MOE_ERR_INVALID_ARG;
    CK(cudaSetDevice(h->dev));
    if (sync_last(h) != MOE_OK)
        return MOE_ERR_CUDA;
    CK(cudaMemcpy(host_dst, src, bytes, cudaMemcpyDeviceToHost));
    return MOE_OK;
}

int moe_get_info(moe_handle_t h, moe_info *info)
{
    if (!h || !info)
        return MOE_ERR_INVALID_ARG;
    info->E = h->d.E;
    info->H = h->d.H;
    info->I = h->d.I;
    info->topk = h->d.K;
    info->R = h->d.R;
    info->max_tokens = h->reserved ? h->ws.max_tokens : 0;
    info->pool_rows = h->reserved ? h->ws.P : 0;
    info->block_m = BM;
    info->block_n = BN;
    info->num_sms = h->num_sms;
    info->workspace_bytes = h->small_bytes + h->big_bytes;
    info->weight_bytes = h->w_bytes + h->w4_bytes;
    info->n_shared = h->S;
    info->weight_format = h->fmt_routed;
    return MOE_OK;
}

int moe_set_option(moe_handle_t h, int option, int64_t value)
{
    if (!h)
        return MOE_ERR_INVALID_ARG;
    switch (option) {
    case MOE_OPT_TIMEOUT_NS:
        if (value < 1000000 || value > 600000000000LL)
            return MOE_ERR_INVALID_ARG;
        h->timeout_ns = value;
        return MOE_OK;
    case MOE_OPT_DEBUG_SKIP_BARRIER:
        h->debug_skip_barrier = value != 0;
        return MOE_OK;
    case MOE_OPT_FFN_MODE:
        if (value < 0 || value > 1)
            return MOE_ERR_INVALID_ARG;
        h->ffn_mode = static_cast<int>(value);
        return MOE_OK;
    case MOE_OPT_SCALE_MODE:
        if (value < 0 || value > 2)
            return MOE_ERR_INVALID_ARG;
        h->scale_mode = static_cast<int>(value);
        return MOE_OK;
    case MOE_OPT_COMBINE_MODE:
        if (value < 0 || value > 2)
            return MOE_ERR_INVALID_ARG;
        h->combine_mode = static_cast<int>(value);
        return MOE_OK;
    default:
        return MOE_ERR_INVALID_ARG;
    }
}

int moe_profile_enable(moe_handle_t h, int enable)
{
    if (!h || enable < 0)
        return MOE_ERR_INVALID_ARG;
    CK(cudaSetDevice(h->dev));
    if (enable && h->events.empty()) {
        h->events.resize(static_cast<size_t>(PROF_MAX_CALLS) * 4);
        for (auto &e : h->events)
            CK(cudaEventCreate(&e));
    }
    h->profile = enable != 0;
    h->prof_every = enable > 0 ? enable : 1;
    h->prof_seen = 0;
    h->prof_calls = 0;
    h->prof_dropped = 0;
    return MOE_OK;
}

int moe_profile_read(moe_handle_t h, double *stage_ms, int *calls, int *dropped)
{
    if (!h || !stage_ms)
        return MOE_ERR_INVALID_ARG;
    CK(cudaSetDevice(h->dev));
    if (sync_last(h) != MOE_OK)
        return MOE_ERR_CUDA;
    for (int j = 0; j < 3; ++j)
        stage_ms[j] = 0.0;
    for (int i = 0; i < h->prof_calls; ++i) {
        for (int j = 0; j < 3; ++j) {
            float ms = 0.0f;
            CK(cudaEventElapsedTime(&ms, h->events[static_cast<size_t>(i) * 4 + j],
                                    h->events[static_cast<size_t>(i) * 4 + j + 1]));
            stage_ms[j] += ms;
        }
    }
    if (calls)
        *calls = h->prof_calls;
    if (dropped)
        *dropped = h->prof_dropped;
    h->prof_calls = 0;
    h->prof_dropped = 0;
    return MOE_OK;
}

int moe_destroy(moe_handle_t h)
{
    if (!h)
        return MOE_ERR_INVALID_ARG;
    cudaSetDevice(h->dev);
    sync_last(h);
    for (auto &e : h->events)
        cudaEventDestroy(e);
    free_big(h);
    for (int i = 0; i < 2; ++i) {
        if (h->ev_staged[i])
            cudaEventDestroy(h->ev_staged[i]);
        if (h->ev_free[i])
            cudaEventDestroy(h->ev_free[i]);
    }
    if (h->copy_stream)
        cudaStreamDestroy(h->copy_stream);
    if (h->small_mem)
        cudaFree(h->small_mem);
    if (h->w_mem)
        cudaFree(h->w_mem);
    if (h->w4_mem)
        cudaFree(h->w4_mem);
    delete h;
    return MOE_OK;
}

#ifdef CPW_TRACE
// Development builds only (-DCPW_TRACE): stamps of the FFN kernel's trace buffer.
int moe_trace_read(void *dst, uint64_t bytes)
{
    return cpw::trace_read(dst, bytes) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
int moe_trace_clear(void) { return cpw::trace_clear() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }
#endif

}  // extern "C"
