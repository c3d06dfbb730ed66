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
// last warp carries the tile's final state to the next tile.  A warp loads its whole
// segment (3 x SEG rows of 128 or 256 contiguous bytes) before computing it.
#include "common.cuh"

namespace ret {
namespace {

constexpr int kThreads = 256;

template <typename T> struct Vec2;
template <> struct Vec2<float> {
    using type = float2;
    static __device__ __forceinline__ float2 load(const float* p) {
        return __ldg(reinterpret_cast<const float2*>(p));
    }
    static __device__ __forceinline__ float2 unpack(float2 v) { return v; }
};
template <> struct Vec2<__nv_bfloat16> {
    using type = __nv_bfloat162;
    static __device__ __forceinline__ __nv_bfloat162 load(const __nv_bfloat16* p) {
        return __ldg(reinterpret_cast<const __nv_bfloat162*>(p));
    }
    static __device__ __forceinline__ float2 unpack(__nv_bfloat162 v) {
        return __bfloat1622float2(v);
    }
};

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

template <bool FAST> __device__ __forceinline__ float sigm(float z) {
    if (FAST) return fmaf(0.5f, tanh_hw(0.5f * z), 0.5f);
    return __frcp_rn(1.0f + __expf(-z));
}
template <bool FAST> __device__ __forceinline__ float pow2(float v) {
    return FAST ? ex2_hw(v) : exp2f(v);
}

// 1 - 2^v for v <= 0: with u = v ln 2, the Taylor series -(u + u^2/2 + u^3/6 + u^4/24)
// where |u| < 1/16 (its next term is below 2^-24 relative there), else 1 - 2^v directly.
template <bool FAST> __device__ __forceinline__ float one_minus_pow2(float v) {
    const float u = v * 0.69314718055994531f;
    if (u > -0.0625f) return -u * fmaf(u, fmaf(u, fmaf(u, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f), 1.0f);
    return 1.0f - pow2<FAST>(v);
}

// One step for one channel; la2 = log2 sigmoid(lambda).  Returns h_t, and a_t in at.
template <bool FAST>
__device__ __forceinline__ float rglru_step(float h, float x, float ga, float gx, float la2,
                                            float c, float& at) {
    const float r = sigm<FAST>(ga);
    const float l2 = (r > 0.0f) ? c * r * la2 : 0.0f;        // log2 a_t (a^0 = 1, also for a = 0)
    at = pow2<FAST>(l2);
    const float om = one_minus_pow2<FAST>(2.0f * l2);          // 1 - a_t^2
    const float w = FAST ? sqrt_hw(om) : sqrtf(om);
    return fmaf(at, h, w * (sigm<FAST>(gx) * x));
}

constexpr int kWarps = 8;        // segments per tile
constexpr int kLanes = 32;       // a lane owns channels 2*lane, 2*lane+1 of the CTA's 64

template <typename TI, typename TO, int SEG, bool FAST>
__global__ void __launch_bounds__(kThreads, 2)
rglru_scan_kernel(const TI* __restrict__ x, const TI* __restrict__ ga, const TI* __restrict__ gx,
                  const float* __restrict__ lam, const float* __restrict__ h0,
                  TO* __restrict__ y, float* __restrict__ h_last, int b, int T, int D, float c) {
    using V = typename Vec2<TI>::type;
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
    const TI* xp = x + base;
    const TI* ap = ga + base;
    const TI* gp = gx + base;
    TO* yp = y + base;
    for (int t0 = 0; t0 < T; t0 += kWarps * SEG) {
        const int ts = t0 + w * SEG;          // this warp's segment
        V bx[SEG], ba[SEG], bg[SEG];
#pragma unroll
        for (int u = 0; u < SEG; ++u) {
            if (ts + u < T) {
                bx[u] = Vec2<TI>::load(xp + (size_t)(ts + u) * D);
                ba[u] = Vec2<TI>::load(ap + (size_t)(ts + u) * D);
                bg[u] = Vec2<TI>::load(gp + (size_t)(ts + u) * D);
            }
        }
        float yl0[SEG], yl1[SEG], p0[SEG], p1[SEG];
        float hl0 = 0.f, hl1 = 0.f, pa0 = 1.f, pa1 = 1.f;
#pragma unroll
        for (int u = 0; u < SEG; ++u) {
            if (ts + u < T) {
                const float2 xv = Vec2<TI>::unpack(bx[u]);
                const float2 av = Vec2<TI>::unpack(ba[u]);
                const float2 gv = Vec2<TI>::unpack(bg[u]);
                float at;
                hl0 = rglru_step<FAST>(hl0, xv.x, av.x, gv.x, la0, c, at);
                pa0 *= at;
                hl1 = rglru_step<FAST>(hl1, xv.y, av.y, gv.y, la1, c, at);
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

template <typename TI, typename TO>
cudaError_t launch_rg(const void* x, const void* ga, const void* gx, const float* lam,
                      const float* h0, void* y, float* h_last, int b, int T, int D, float c,
                      cudaStream_t s) {
    // D % 64 == 0 is checked by the caller; one CTA per (batch row, 64 channels)
    const long long blocks = (long long)b * (D / (2 * kLanes));
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // 12 steps per segment for 2-byte inputs, 8 for 4-byte ones (both within 128 registers)
    constexpr int SEG = sizeof(TI) == 2 ? 12 : 8;
    rglru_scan_kernel<TI, TO, SEG, sizeof(TI) == 2><<<(unsigned)blocks, kThreads, 0, s>>>(
        static_cast<const TI*>(x), static_cast<const TI*>(ga), static_cast<const TI*>(gx), lam,
        h0, static_cast<TO*>(y), h_last, b, T, D, c);
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) count_launch(RET_KERNEL_RGLRU);
    return err;
}

}  // namespace

cudaError_t launch_rglru_scan(const void* x, const void* ga, const void* gx, const float* lam,
                              const float* h0, void* y, float* h_last, int in_bf16, int out_bf16,
                              int b, int T, int D, float c, cudaStream_t s) {
    using bf = __nv_bfloat16;
    if (in_bf16)
        return out_bf16 ? launch_rg<bf, bf>(x, ga, gx, lam, h0, y, h_last, b, T, D, c, s)
                        : launch_rg<bf, float>(x, ga, gx, lam, h0, y, h_last, b, T, D, c, s);
    return out_bf16 ? launch_rg<float, bf>(x, ga, gx, lam, h0, y, h_last, b, T, D, c, s)
                    : launch_rg<float, float>(x, ga, gx, lam, h0, y, h_last, b, T, D, c, s);
}

}  // namespace ret
