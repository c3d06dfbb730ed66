// tc_gemm.cu -- the projections of the gated multi-scale retention layer as tcgen05 GEMMs.
//
// [RN2] "Transformer取代者登場！…RetNet…（2）", section "門控多尺度 Retention": the layer
// projects X with W_Q, W_K, W_V (per head) and W_G, runs retention per head, normalises and
// gates, and projects the result with W_O.  Every projection is C = A W with
//   A: [M][K] bf16 row-major (the token rows), W: [K][Nc] bf16 row-major (the weights as the
//   layer applies them: x W), fp32 accumulation,
// and an epilogue that writes C either row-major (fp32 or bf16) or as head-major rows
// [b][H][Nseq][d] (bf16) -- the layout the retention calls read -- optionally rotating the
// coordinate pairs of each head by xPos, [RN2] "Retention" eqs.(2)-(3): the pair (2j, 2j+1)
// of position p as a complex number times e^{i p theta_j}.
//
// Kernel: persistent (one CTA per SM), warp-specialised.
//   warp 0      TMA producer: a 4-stage ring of {A: 128 rows x 64 K (16 KB), W: 64 K rows x
//               256 columns (4 boxes of 64 columns, 32 KB)}
//   warp 1      tensor-memory allocation (512 columns) and the MMA issuer: per stage four
//               tcgen05.mma of M=128, N=256, K=16 (A K-major, W MN-major, both 128B-swizzled),
//               into one of two 256-column fp32 accumulators
//   warps 2-9   epilogue: two warps per TMEM lane quarter (128 columns each), 32 columns at
//               a time: optional rotation, then coalesced stores (8-lane transposes: every
//               store instruction writes four whole 128-byte segments)
// The two accumulators let the epilogue of one tile overlap the MMAs of the next.  Tiles
// are 128 rows x 256 columns, walked in bands of 16 row tiles, the row index fastest inside
// a band: the ~148 tiles in flight at one time then cover about 16 row panels of A and 9
// column panels of W (~35 MB at K = 4096), which stay in L2 while they are reused, instead
// of all of W (the row-major order's working set).  Every wait is bounded
// (2 s); a wait that gives up sets the device error word and the CTA unwinds.
//
// xPos phase: p * theta_j / (2 pi) turns, reduced exactly as 64-bit fixed point:
// T_j = round(2^64 * frac(theta_j / (2 pi))) is prepared on the host; the low 64 bits of
// p * T_j are the fraction of a turn, whose top 32 bits read as a signed integer give the
// angle in [-pi, pi) without any loss for large positions.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"
#include "gemm.cuh"

namespace ret {
namespace {

__device__ unsigned g_err_gemm;

using namespace tc;

constexpr int kThreads = 320;
constexpr int kStages = 4;
constexpr int kTileM = 128, kTileN = 256, kTileK = 64;
constexpr int kABytes = kTileM * 128;            // 16 KB
constexpr int kWBox = kTileK * 128;              // 8 KB: 64 K rows x 64 columns
constexpr int kStageBytes = kABytes + 4 * kWBox; // 48 KB
constexpr int kSmemBytes = kStages * kStageBytes;
constexpr uint32_t kEpiArrivals = 8;

struct Bars {
    uint64_t full[kStages], empty[kStages];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t drain;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}

constexpr int kBand = 16;          // row tiles per band of the tile order

// Tile t of the order above -> its first row and column.
__device__ __forceinline__ void tile_origin(int t, int mtiles, int ntiles, int& m0, int& n0) {
    const int band = t / (kBand * ntiles);
    const int first = band * kBand;
    const int rows = min(kBand, mtiles - first);
    const int r = t - band * kBand * ntiles;
    m0 = (first + r % rows) * kTileM;
    n0 = (r / rows) * kTileN;
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mw,
            int M, int Nc, int K, const __grid_constant__ GemmEpilogue ep) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ Bars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_p = &abort_flag;
    const int mtiles = (M + kTileM - 1) / kTileM, ntiles = Nc / kTileN;
    const int tiles = mtiles * ntiles;
    const int ksteps = K / kTileK;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < kStages; ++s) { mbar_init(&bars.full[s], 1); mbar_init(&bars.empty[s], 1); }
        for (int b = 0; b < 2; ++b) { mbar_init(&bars.acc_full[b], 1); mbar_init(&bars.acc_empty[b], kEpiArrivals); }
        mbar_init(&bars.drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) { tmem_alloc(&tmem_slot, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    auto fail = [&]() { *abort_p = 1; atomicOr(&g_err_gemm, 1u); };

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&ma); tma_prefetch_desc(&mw);
            uint32_t it = 0;                 // stage uses so far (ring position and parity)
            uint32_t issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                int m0, n0;
                tile_origin(t, mtiles, ntiles, m0, n0);
                for (int ks = 0; ks < ksteps; ++ks, ++it) {
                    const uint32_t s = it % kStages, use = it / kStages;
                    if (use > 0 && !mbar_wait(&bars.empty[s], (use - 1) & 1, abort_p)) {
                        ok = false; fail(); break;
                    }
                    uint8_t* st = sm + s * kStageBytes;
                    mbar_arrive_expect_tx(&bars.full[s], kStageBytes);
                    tma_load_2d(st, &ma, ks * kTileK, m0, &bars.full[s]);
#pragma unroll
                    for (int nb = 0; nb < 4; ++nb)
                        tma_load_2d(st + kABytes + nb * kWBox, &mw, n0 + 64 * nb, ks * kTileK, &bars.full[s]);
                    ++issued;
                }
            }
            if (!ok && issued) {
                // let the loads in flight land before the CTA unwinds
                const uint32_t last = issued - 1;
                for (uint32_t i = (issued > kStages ? issued - kStages : 0); i <= last; ++i)
                    mbar_wait(&bars.full[i % kStages], (i / kStages) & 1, nullptr, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kTileM, kTileN, 0, 1);   // A K-major, W MN-major
            const uint64_t d0 = sdesc_sw128(smem_u32(sm), 16, 1024);
            uint32_t it = 0, tl = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++tl) {
                const uint32_t buf = tl & 1, use = tl >> 1;
                if (use > 0 && !mbar_wait(&bars.acc_empty[buf], (use - 1) & 1, abort_p)) {
                    ok = false; fail(); break;
                }
                tc_fence_after();
                const uint32_t acc = tmem + 256 * buf;
                for (int ks = 0; ks < ksteps; ++ks, ++it) {
                    const uint32_t s = it % kStages, su = it / kStages;
                    if (!mbar_wait(&bars.full[s], su & 1, abort_p)) { ok = false; fail(); break; }
                    tc_fence_after();
                    const uint32_t base = (uint32_t)(s * kStageBytes);
                    // W: MN-major, 64-column blocks 8 KB apart (LBO), 8-row groups 1 KB (SBO)
                    const uint64_t dw = sdesc_sw128(smem_u32(sm) + base + kABytes, kWBox, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = d0 + (uint64_t)((base + kk * 32) >> 4);
                        const uint64_t w = dw + (uint64_t)((kk * 2048) >> 4);
                        mma_bf16(acc, a, w, idesc, (ks | kk) != 0);
                    }
                    mma_commit(&bars.empty[s]);
                }
                if (!ok) break;
                mma_commit(&bars.acc_full[buf]);
            }
            mma_commit(&bars.drain);
            mbar_wait(&bars.drain, 0, nullptr, 200000000ull);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int q4 = warp & 3;
        const int half = (warp - 2) >> 2;            // columns 128*half .. +127 of the tile
        const uint32_t lrow = (uint32_t)(32 * q4) << 16;
        const int p8 = lane & 7;
        uint32_t tl = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++tl) {
            int m0, n0;
            tile_origin(t, mtiles, ntiles, m0, n0);
            const uint32_t buf = tl & 1, use = tl >> 1;
            const bool got = __all_sync(0xffffffffu, mbar_wait(&bars.acc_full[buf], use & 1, abort_p));
            if (!got) { ok = false; if (lane == 0) fail(); break; }
            tc_fence_after();
            const int m = m0 + 32 * q4 + lane;       // this thread's row
            // xPos position of this row (head-major outputs only)
            const unsigned long long pos =
                (unsigned long long)ep.pos0 + (unsigned long long)(ep.mode == 1 ? m % ep.nseq : 0);
            const uint32_t pos_lo = (uint32_t)pos, pos_hi = (uint32_t)(pos >> 32);
#pragma unroll 1
            for (int sg = 0; sg < 4; ++sg) {
                const int c0 = n0 + 128 * half + 32 * sg;    // first column of the segment
                float x[32];
                tmem_ld32(tmem + lrow + 256 * buf + 128 * half + 32 * sg, x);
                tmem_wait_ld();
                if (sg == 3) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.acc_empty[buf]);
                }
                if (ep.mode == 1 && ep.xpos) {
                    const int j0 = (c0 % ep.d) >> 1;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint32_t tlo = ep.turns_lo[j0 + e], thi = ep.turns_hi[j0 + e];
                        // top 32 bits of the low 64 bits of pos * T_j
                        const uint32_t f = __umulhi(pos_lo, tlo) + pos_lo * thi + pos_hi * tlo;
                        float sn, cs;
                        __sincosf((float)(int)f * 1.46291807926715968e-9f, &sn, &cs);   // 2 pi / 2^32
                        const float a = x[2 * e], b = x[2 * e + 1];
                        x[2 * e] = a * cs - b * sn;
                        x[2 * e + 1] = a * sn + b * cs;
                    }
                }
                if (ep.out_bf16) {
                    // 32 bf16 columns = 64 bytes = 4 items of 16 bytes per row, transposed
                    // within 4-lane groups: each store instruction writes eight 64-byte
                    // row pieces
                    uint32_t a[4][4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int w = 0; w < 4; ++w) a[k][w] = pack_bf16(x[8 * k + 2 * w], x[8 * k + 2 * w + 1]);
                    const int p4 = lane & 3;
                    transpose4x4(a, p4);
                    const int m4 = m - p4;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int r = m4 + k;
                        if (r < M) {
                            uint4* dst = reinterpret_cast<uint4*>(gemm_out_addr(ep, r, c0, 2)) + p4;
                            *dst = make_uint4(a[k][0], a[k][1], a[k][2], a[k][3]);
                        }
                    }
                } else {
                    uint32_t a[8][4];
#pragma unroll
                    for (int k = 0; k < 8; ++k)
#pragma unroll
                        for (int w = 0; w < 4; ++w) a[k][w] = __float_as_uint(x[4 * k + w]);
                    transpose8x8(a, p8);
                    // rows of this 8-lane group: m - p8 .. m - p8 + 7
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int r = m - p8 + k;
                        if (r < M) {
                            uint4* dst = reinterpret_cast<uint4*>(gemm_out_addr(ep, r, c0, 4)) + p8;
                            *dst = make_uint4(a[k][0], a[k][1], a[k][2], a[k][3]);
                        }
                    }
                }
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_gemm_bf16(const void* a, const void* w, int M, int Nc, int K,
                             const GemmEpilogue& ep, cudaStream_t s) {
    if (M <= 0 || Nc <= 0 || K <= 0) return cudaSuccess;
    if (Nc % kTileN != 0 || K % kTileK != 0) return cudaErrorNotSupported;
    if (ep.mode == 1 && (ep.d % 64 != 0 || ep.nseq <= 0 || ep.H <= 0 || Nc != ep.H * ep.d))
        return cudaErrorNotSupported;
    if (ep.mode == 1 && ep.xpos && ep.d > 2 * kGemmMaxPairs) return cudaErrorNotSupported;
    CUtensorMap ma, mw;
    if (!make_map_bf16(&ma, a, (uint64_t)M, (uint64_t)K, kTileM) ||
        !make_map_bf16(&mw, w, (uint64_t)K, (uint64_t)Nc, kTileK))
        return cudaErrorInvalidValue;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long tiles = (long long)((M + kTileM - 1) / kTileM) * (Nc / kTileN);
    const int grid = (int)(tiles < sms ? tiles : sms);
    const int smem = kSmemBytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gemm_kernel<<<grid, kThreads, smem, s>>>(ma, mw, M, Nc, K, ep);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launch(RET_KERNEL_GEMM_TC);
    return e;
}

unsigned read_clear_error_gemm(cudaStream_t s) {
    unsigned h = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_err_gemm, sizeof(h), 0, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_err_gemm, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return h;
}

}  // namespace ret
