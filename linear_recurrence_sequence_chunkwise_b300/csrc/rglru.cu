// rglru.cu -- RG-LRU scan, the diagonal gated linear recurrence of the Griffin page
// ("Griffin ：將門控線性循環與局部注意力混合以實現高效的語言模型", section
// "實門線性循環單元 (RG-LRU)"):
//   r_t = sigmoid(gate_a_t), i_t = sigmoid(gate_x_t), a = sigmoid(lambda),
//   a_t = a^(c r_t),  h_t = a_t h_{t-1} + sqrt(1 - a_t^2) (i_t x_t),  y_t = h_t.
// Every operation is elementwise over channels; only t is sequential.  a_t is taken
// in log space, as the page prescribes: log2 a_t = c r_t log2 sigmoid(lambda), and
// 1 - a_t^2 = -expm1(2 ln a_t), so that a_t close to 1 keeps its precision.
//
// Memory-bound: per step and channel three inputs are read and one output written,
// each exactly once.  The sequential dependence on t is split the chunkwise way:
// a CTA owns 64 channels of one batch row (a warp lane owns two adjacent ones) and
// walks t in tiles of 8 segments; warp w scans segment w of the tile from a zero state,
// keeping each step's local output y_loc and decay product P (= prod of a_s since the
// segment start) in registers, and publishes the segment's (prod a, h_end) through
// shared memory.  Each warp then folds the published pairs of the segments before its
// own into the state entering its segment, c, and writes y_t = y_loc_t + P_t c.  The
// last warp carries the tile's final state to the next tile.
//
// bf16 inputs (rglru_tma_kernel): the tiles of x, gate_a and gate_x stream into shared
// memory through TMA, two tiles in flight per CTA, so the loads of the next tile run
// while the current one is computed; the gate arithmetic is rearranged to share work
// (see rglru_step_fast).  fp32 inputs (rglru_scan_kernel): each warp loads its whole
// segment (3 x SEG rows of 256 contiguous bytes) into registers before computing it.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace ret {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void store2(float* p, float a, float b) {
    __stcs(reinterpret_cast<float2*>(p), make_float2(a, b));
}
__device__ __forceinline__ void store2(__nv_bfloat16* p, float a, float b) {
    __stcs(reinterpret_cast<__nv_bfloat162*>(p), __floats2bfloat162_rn(a, b));
}

// Two arithmetic variants.  Accurate (fp32 inputs, 1e-4 relative tolerance): IEEE
// reciprocal and square root, exp2f.  Fast (bf16 inputs): one hardware instruction each
// for tanh, 2^x and the square root; sigmoid(z) = 1/2 + tanh(z/2)/2, whose error (below
// 2.5e-4 absolute) sits far under the bf16 inputs' own rounding.  Both give exactly 0
// for a gate driven to -inf (tanh saturates at -1, 1/inf = 0).
__device__ __forceinline__ float tanh_hw(float v) {
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float ex2_hw(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float sqrt_hw(float v) {
    float r;
    asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float sigm(float z) { return __frcp_rn(1.0f + __expf(-z)); }

// 1 - 2^v for v <= 0: with u = v ln 2, the Taylor series -(u + u^2/2 + u^3/6 + u^4/24)
// where |u| < 1/16 (its next term is below 2^-24 relative there), else 1 - 2^v directly.
__device__ __forceinline__ float one_minus_pow2(float v) {
    const float u = v * 0.69314718055994531f;
    if (u > -0.0625f) return -u * fmaf(u, fmaf(u, fmaf(u, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f), 1.0f);
    return 1.0f - exp2f(v);
}

// One accurate step for one channel; la2 = log2 sigmoid(lambda).  Returns h_t, and a_t
// in at.
__device__ __forceinline__ float rglru_step(float h, float x, float ga, float gx, float la2,
                                            float c, float& at) {
    const float r = sigm(ga);
    const float l2 = (r > 0.0f) ? c * r * la2 : 0.0f;        // log2 a_t (a^0 = 1, also for a = 0)
    at = exp2f(l2);
    const float om = one_minus_pow2(2.0f * l2);               // 1 - a_t^2
    return fmaf(at, h, sqrtf(om) * (sigm(gx) * x));
}

constexpr int kWarps = 8;        // segments per tile
constexpr int kLanes = 32;       // a lane owns channels 2*lane, 2*lane+1 of the CTA's 64

template <typename TO, int SEG>
__global__ void __launch_bounds__(kThreads, 2)
rglru_scan_kernel(const float* __restrict__ x, const float* __restrict__ ga,
                  const float* __restrict__ gx, const float* __restrict__ lam,
                  const float* __restrict__ h0, TO* __restrict__ y, float* __restrict__ h_last,
                  int b, int T, int D, float c) {
    __shared__ float2 segA[kWarps][kLanes];   // prod of a_t over the segment, per channel
    __shared__ float2 segH[kWarps][kLanes];   // segment's final state from a zero start
    __shared__ float2 carry[kLanes];          // state entering the current tile
    const int blocks_per_row = D / (2 * kLanes);
    const int bi = blockIdx.x / blocks_per_row;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int d = (blockIdx.x % blocks_per_row) * (2 * kLanes) + 2 * lane;
    // log2 sigmoid(lambda) = -log2(1 + e^-lambda): -inf for a = 0, 0 for a = 1
    const float la0 = -log1pf(expf(-lam[d])) * 1.4426950408889634f;
    const float la1 = -log1pf(expf(-lam[d + 1])) * 1.4426950408889634f;
    if (w == 0) {
        float2 s0 = make_float2(0.f, 0.f);
        if (h0) s0 = make_float2(h0[(size_t)bi * D + d], h0[(size_t)bi * D + d + 1]);
        carry[lane] = s0;
    }
    const size_t base = (size_t)bi * T * D + d;
    const float* xp = x + base;
    const float* ap = ga + base;
    const float* gp = gx + base;
    TO* yp = y + base;
    for (int t0 = 0; t0 < T; t0 += kWarps * SEG) {
        const int ts = t0 + w * SEG;          // this warp's segment
        float2 bx[SEG], ba[SEG], bg[SEG];
#pragma unroll
        for (int u = 0; u < SEG; ++u) {
            if (ts + u < T) {
                bx[u] = __ldg(reinterpret_cast<const float2*>(xp + (size_t)(ts + u) * D));
                ba[u] = __ldg(reinterpret_cast<const float2*>(ap + (size_t)(ts + u) * D));
                bg[u] = __ldg(reinterpret_cast<const float2*>(gp + (size_t)(ts + u) * D));
            }
        }
        float yl0[SEG], yl1[SEG], p0[SEG], p1[SEG];
        float hl0 = 0.f, hl1 = 0.f, pa0 = 1.f, pa1 = 1.f;
#pragma unroll
        for (int u = 0; u < SEG; ++u) {
            if (ts + u < T) {
                const float2 xv = bx[u], av = ba[u], gv = bg[u];
                float at;
                hl0 = rglru_step(hl0, xv.x, av.x, gv.x, la0, c, at);
                pa0 *= at;
                hl1 = rglru_step(hl1, xv.y, av.y, gv.y, la1, c, at);
                pa1 *= at;
            }
            yl0[u] = hl0; yl1[u] = hl1; p0[u] = pa0; p1[u] = pa1;
        }
        segA[w][lane] = make_float2(pa0, pa1);
        segH[w][lane] = make_float2(hl0, hl1);
        __syncthreads();
        float2 cs = carry[lane];              // state entering the tile
        for (int k = 0; k < w; ++k) {         // ... then entering this warp's segment
            const float2 A = segA[k][lane], Hk = segH[k][lane];
            cs.x = fmaf(A.x, cs.x, Hk.x);
            cs.y = fmaf(A.y, cs.y, Hk.y);
        }
        __syncthreads();                      // every warp has read carry and the pairs
        if (w == kWarps - 1)
            carry[lane] = make_float2(fmaf(pa0, cs.x, hl0), fmaf(pa1, cs.y, hl1));
#pragma unroll
        for (int u = 0; u < SEG; ++u)
            if (ts + u < T)
                store2(yp + (size_t)(ts + u) * D, fmaf(p0[u], cs.x, yl0[u]),
                       fmaf(p1[u], cs.y, yl1[u]));
    }
    __syncthreads();
    if (h_last && w == 0) {
        h_last[(size_t)bi * D + d] = carry[lane].x;
        h_last[(size_t)bi * D + d + 1] = carry[lane].y;
    }
}

// One step of the bf16-input path for one channel, with the constants of the channel
// folded: hcla = c * log2(a) / 2 (finite: -1e30 stands for a = 0).  ga_h, gx_h, x_h are
// half the gate pre-activations and half the input (halved exactly in bf16).
//   r = (1 + tanh(ga/2)) / 2  ->  log2 a_t = c r log2 a = hcla + hcla tanh(ga/2)
//   (exactly 0 for ga = -inf, so a_t = 1),  a_t = 2^(log2 a_t),
//   1 - a_t^2 = -expm1(u) with u = 2 ln(a_t): a cubic Taylor polynomial for |u| < 1/16
//   (next term below 2^-24 relative), else 1 - a_t a_t (no cancellation there),
//   i_t x_t sqrt(1 - a_t^2) = p + p tanh(gx/2) with p = sqrt(1 - a_t^2) x / 2.
__device__ __forceinline__ float rglru_step_fast(float h, float x_h, float ga_h, float gx_h,
                                                 float hcla, float& at) {
    const float l2 = fmaf(hcla, tanh_hw(ga_h), hcla);
    at = ex2_hw(l2);
    const float u = l2 * 1.3862943611198906f;
    const float tay = -u * fmaf(u, fmaf(u, fmaf(u, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f), 1.0f);
    const float om = (u > -0.0625f) ? tay : fmaf(-at, at, 1.0f);
    const float p = sqrt_hw(om) * x_h;
    return fmaf(at, h, fmaf(p, tanh_hw(gx_h), p));
}

__device__ unsigned g_err_rglru;

constexpr int kTmaSeg = 8;                    // steps per segment (warp) in a tile
constexpr int kTileRows = kWarps * kTmaSeg;   // 64 steps per tile
constexpr int kRowBytes = 128;                // 64 bf16 channels
constexpr int kInBytes = kTileRows * kRowBytes;   // one input's tile: 8 KB
constexpr int kStageBytes = 3 * kInBytes;
constexpr int kStages = 2;

template <typename TO>
__global__ void __launch_bounds__(kThreads, 4)
rglru_tma_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap ma,
                 const __grid_constant__ CUtensorMap mg, const float* __restrict__ lam,
                 const float* __restrict__ h0, TO* __restrict__ y, float* __restrict__ h_last,
                 int T, int D, float c, uint64_t wait_ns) {
    extern __shared__ __align__(128) uint8_t tiles[];   // kStages x {x, gate_a, gate_x}
    __shared__ uint64_t full[kStages];
    __shared__ float2 segA[kWarps][kLanes];
    __shared__ float2 segH[kWarps][kLanes];
    __shared__ float2 carry[kLanes];
    __shared__ int abort_flag;
    const int blocks_per_row = D / (2 * kLanes);
    const int bi = blockIdx.x / blocks_per_row;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int d0 = (blockIdx.x % blocks_per_row) * (2 * kLanes);
    const int d = d0 + 2 * lane;
    const int ntiles = (T + kTileRows - 1) / kTileRows;
    auto issue = [&](int tile) {       // one thread: the three boxes of a tile
        uint8_t* st = tiles + (tile % kStages) * kStageBytes;
        uint64_t* bar = &full[tile % kStages];
        tc::mbar_arrive_expect_tx(bar, kStageBytes);
        tc::tma_load_3d(st, &mx, d0, tile * kTileRows, bi, bar);
        tc::tma_load_3d(st + kInBytes, &ma, d0, tile * kTileRows, bi, bar);
        tc::tma_load_3d(st + 2 * kInBytes, &mg, d0, tile * kTileRows, bi, bar);
    };
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < kStages; ++i) tc::mbar_init(&full[i], 1);
        tc::fence_barrier_init();
    }
    // c log2(a) / 2 per channel, with -1e30 standing for log2(0)
    auto hc = [&](float l) {
        const float la2 = -log1pf(expf(-l)) * 1.4426950408889634f;
        return 0.5f * c * fmaxf(la2, -1e30f);
    };
    const float hc0 = hc(lam[d]), hc1 = hc(lam[d + 1]);
    if (w == 0) {
        float2 s0 = make_float2(0.f, 0.f);
        if (h0) s0 = make_float2(h0[(size_t)bi * D + d], h0[(size_t)bi * D + d + 1]);
        carry[lane] = s0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        tc::tma_prefetch_desc(&mx); tc::tma_prefetch_desc(&ma); tc::tma_prefetch_desc(&mg);
        for (int i = 0; i < kStages && i < ntiles; ++i) issue(i);
    }
    const __nv_bfloat162 half2 = __float2bfloat162_rn(0.5f);
    TO* yp = y + (size_t)bi * T * D + d;
    int t = 0;
    for (; t < ntiles; ++t) {
        const int t0 = t * kTileRows;
        const int ts = t0 + w * kTmaSeg;           // this warp's segment
        const uint8_t* st = tiles + (t % kStages) * kStageBytes + (w * kTmaSeg) * kRowBytes + 4 * lane;
        const bool got = tc::mbar_wait(&full[t % kStages], (uint32_t)(t / kStages) & 1u,
                                       &abort_flag, wait_ns);
        if (!got) abort_flag = 1;
        float yl0[kTmaSeg], yl1[kTmaSeg], p0[kTmaSeg], p1[kTmaSeg];
        float hl0 = 0.f, hl1 = 0.f, pa0 = 1.f, pa1 = 1.f;
        if (got) {
#pragma unroll
            for (int u = 0; u < kTmaSeg; ++u) {
                if (ts + u < T) {
                    // x/2, gate_a/2, gate_x/2 of this lane's two channels (exact in bf16)
                    const float2 xv = __bfloat1622float2(
                        __hmul2(*reinterpret_cast<const __nv_bfloat162*>(st + u * kRowBytes), half2));
                    const float2 av = __bfloat1622float2(__hmul2(
                        *reinterpret_cast<const __nv_bfloat162*>(st + kInBytes + u * kRowBytes), half2));
                    const float2 gv = __bfloat1622float2(__hmul2(
                        *reinterpret_cast<const __nv_bfloat162*>(st + 2 * kInBytes + u * kRowBytes), half2));
                    float at;
                    hl0 = rglru_step_fast(hl0, xv.x, av.x, gv.x, hc0, at);
                    pa0 *= at;
                    hl1 = rglru_step_fast(hl1, xv.y, av.y, gv.y, hc1, at);
                    pa1 *= at;
                }
                yl0[u] = hl0; yl1[u] = hl1; p0[u] = pa0; p1[u] = pa1;
            }
        }
        segA[w][lane] = make_float2(pa0, pa1);
        segH[w][lane] = make_float2(hl0, hl1);
        __syncthreads();                       // every warp has read the stage and published
        if (abort_flag) break;                 // uniform: set only before this barrier
        if (threadIdx.x == 0 && t + kStages < ntiles) issue(t + kStages);   // the stage is free
        float2 cs = carry[lane];               // state entering the tile
        for (int k = 0; k < w; ++k) {          // ... then entering this warp's segment
            const float2 A = segA[k][lane], Hk = segH[k][lane];
            cs.x = fmaf(A.x, cs.x, Hk.x);
            cs.y = fmaf(A.y, cs.y, Hk.y);
        }
        __syncthreads();                       // every warp has read carry and the pairs
        if (w == kWarps - 1)
            carry[lane] = make_float2(fmaf(pa0, cs.x, hl0), fmaf(pa1, cs.y, hl1));
#pragma unroll
        for (int u = 0; u < kTmaSeg; ++u)
            if (ts + u < T)
                store2(yp + (size_t)(ts + u) * D, fmaf(p0[u], cs.x, yl0[u]),
                       fmaf(p1[u], cs.y, yl1[u]));
    }
    if (t < ntiles) {
        // a wait gave up: record it, and let the loads still in flight land before exit
        if (threadIdx.x == 0) {
            atomicOr(&g_err_rglru, 1u);
            for (int i = t; i < ntiles && i < t + kStages; ++i)
                tc::mbar_wait(&full[i % kStages], (uint32_t)(i / kStages) & 1u, nullptr, 100000000ull);
        }
        return;
    }
    __syncthreads();
    if (h_last && w == 0) {
        h_last[(size_t)bi * D + d] = carry[lane].x;
        h_last[(size_t)bi * D + d + 1] = carry[lane].y;
    }
}

template <typename TO>
cudaError_t launch_rg(const void* x, const void* ga, const void* gx, const float* lam,
                      const float* h0, void* y, float* h_last, int b, int T, int D, float c,
                      cudaStream_t s) {
    // D % 64 == 0 is checked by the caller; one CTA per (batch row, 64 channels)
    const long long blocks = (long long)b * (D / (2 * kLanes));
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // 8 steps per segment (three fp32 inputs buffered in registers within 128 registers)
    rglru_scan_kernel<TO, 8><<<(unsigned)blocks, kThreads, 0, s>>>(
        static_cast<const float*>(x), static_cast<const float*>(ga), static_cast<const float*>(gx),
        lam, h0, static_cast<TO*>(y), h_last, b, T, D, c);
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) count_launch(RET_KERNEL_RGLRU);
    return err;
}

template <typename TO>
cudaError_t launch_rg_tma(const void* x, const void* ga, const void* gx, const float* lam,
                          const float* h0, void* y, float* h_last, int b, int T, int D, float c,
                          cudaStream_t s) {
    const long long blocks = (long long)b * (D / (2 * kLanes));
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    CUtensorMap mx, ma, mg;
    if (!tc::make_map_bf16_3d_plain(&mx, x, b, T, D, kTileRows) ||
        !tc::make_map_bf16_3d_plain(&ma, ga, b, T, D, kTileRows) ||
        !tc::make_map_bf16_3d_plain(&mg, gx, b, T, D, kTileRows))
        return cudaErrorInvalidValue;
    const int smem = kStages * kStageBytes;
    cudaError_t err = cudaFuncSetAttribute(rglru_tma_kernel<TO>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    rglru_tma_kernel<TO><<<(unsigned)blocks, kThreads, smem, s>>>(
        mx, ma, mg, lam, h0, static_cast<TO*>(y), h_last, T, D, c, 2000000000ull);
    err = cudaGetLastError();
    if (err == cudaSuccess) count_launch(RET_KERNEL_RGLRU);
    return err;
}

}  // namespace

unsigned read_clear_error_rglru(cudaStream_t s) {
    unsigned h = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_err_rglru, sizeof(h), 0, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_err_rglru, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return h;
}

cudaError_t launch_rglru_scan(const void* x, const void* ga, const void* gx, const float* lam,
                              const float* h0, void* y, float* h_last, int in_bf16, int out_bf16,
                              int b, int T, int D, float c, cudaStream_t s) {
    using bf = __nv_bfloat16;
    // bf16 inputs: the TMA-fed kernel (T < 2^31 rows of a 3-D map; D % 64 == 0 checked by
    // the caller)
    if (in_bf16)
        return out_bf16 ? launch_rg_tma<bf>(x, ga, gx, lam, h0, y, h_last, b, T, D, c, s)
                        : launch_rg_tma<float>(x, ga, gx, lam, h0, y, h_last, b, T, D, c, s);
    return out_bf16 ? launch_rg<bf>(x, ga, gx, lam, h0, y, h_last, b, T, D, c, s)
                    : launch_rg<float>(x, ga, gx, lam, h0, y, h_last, b, T, D, c, s);
}

}  // namespace ret
