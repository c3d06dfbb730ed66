// rglru.cu -- RG-LRU scan, the diagonal gated linear recurrence of the Griffin page
// ("Griffin ：將門控線性循環與局部注意力混合以實現高效的語言模型", section
// "實門線性循環單元 (RG-LRU)"):
//   r_t = sigmoid(gate_a_t), i_t = sigmoid(gate_x_t), a = sigmoid(lambda),
//   a_t = a^(c r_t),  h_t = a_t h_{t-1} + sqrt(1 - a_t^2) (i_t x_t),  y_t = h_t.
// Every operation is elementwise over channels; only t is sequential.  a_t is taken
// in log space, as the page prescribes: log2 a_t = c r_t log2 sigmoid(lambda), and
// 1 - a_t^2 = -expm1(2 ln a_t), so that a_t close to 1 keeps its precision.
//
// Memory-bound: per step and channel three inputs are read and one output written.
// One thread owns two adjacent channels of one batch row (8-byte or 4-byte vector
// accesses, a warp covers 64 consecutive channels) and scans t in blocks of P steps;
// the loads of block k+1 are issued into registers before block k is computed, so
// P steps of three inputs per thread are in flight while the recurrence runs.
#include "common.cuh"

namespace ret {
namespace {

// Small blocks: b * D / 2 threads in all (16 K for 8 x 4096 channels) spread over every SM.
constexpr int kThreads = 64;

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

__device__ __forceinline__ float sigmoidf_(float z) {
    return __frcp_rn(1.0f + __expf(-z));   // IEEE reciprocal: z -> -inf gives exactly 0
}

// 1 - e^u for u <= 0: the Taylor series -(u + u^2/2 + u^3/6 + u^4/24) where |u| is
// small (its next term is below 2^-24 relative for |u| < 1/16), else 1 - e^u directly.
__device__ __forceinline__ float one_minus_exp(float u) {
    if (u > -0.0625f) return -u * fmaf(u, fmaf(u, fmaf(u, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f), 1.0f);
    return 1.0f - __expf(u);
}

// One step for one channel; la2 = log2 sigmoid(lambda).
__device__ __forceinline__ float rglru_step(float h, float x, float ga, float gx, float la2,
                                            float c) {
    const float r = sigmoidf_(ga);
    const float l2 = (r > 0.0f) ? c * r * la2 : 0.0f;        // log2 a_t (a^0 = 1, also for a = 0)
    const float at = exp2f(l2);
    const float w = sqrtf(one_minus_exp(2.0f * 0.69314718055994531f * l2));
    return fmaf(at, h, w * (sigmoidf_(gx) * x));
}

template <typename TI, typename TO, int P>
__global__ void __launch_bounds__(kThreads)
rglru_scan_kernel(const TI* __restrict__ x, const TI* __restrict__ ga, const TI* __restrict__ gx,
                  const float* __restrict__ lam, const float* __restrict__ h0,
                  TO* __restrict__ y, float* __restrict__ h_last, int b, int T, int D, float c) {
    using V = typename Vec2<TI>::type;
    const int pairs = D >> 1;
    const long long idx = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (idx >= (long long)b * pairs) return;
    const int bi = (int)(idx / pairs);
    const int d = (int)(idx % pairs) * 2;
    // log2 sigmoid(lambda) = -log2(1 + e^-lambda): -inf for a = 0, 0 for a = 1
    const float la0 = -log1pf(expf(-lam[d])) * 1.4426950408889634f;
    const float la1 = -log1pf(expf(-lam[d + 1])) * 1.4426950408889634f;
    float h_0 = 0.f, h_1 = 0.f;
    if (h0) {
        h_0 = h0[(size_t)bi * D + d];
        h_1 = h0[(size_t)bi * D + d + 1];
    }
    const size_t base = (size_t)bi * T * D + d;
    const TI* xp = x + base;
    const TI* ap = ga + base;
    const TI* gp = gx + base;
    TO* yp = y + base;

    V bx[P], ba[P], bg[P];
#pragma unroll
    for (int u = 0; u < P; ++u) {
        if (u < T) {
            bx[u] = Vec2<TI>::load(xp + (size_t)u * D);
            ba[u] = Vec2<TI>::load(ap + (size_t)u * D);
            bg[u] = Vec2<TI>::load(gp + (size_t)u * D);
        }
    }
    for (int t0 = 0; t0 < T; t0 += P) {
        V nx[P], na[P], ng[P];
        const int tn = t0 + P;
#pragma unroll
        for (int u = 0; u < P; ++u) {
            if (tn + u < T) {
                nx[u] = Vec2<TI>::load(xp + (size_t)(tn + u) * D);
                na[u] = Vec2<TI>::load(ap + (size_t)(tn + u) * D);
                ng[u] = Vec2<TI>::load(gp + (size_t)(tn + u) * D);
            }
        }
#pragma unroll
        for (int u = 0; u < P; ++u) {
            if (t0 + u < T) {
                const float2 xv = Vec2<TI>::unpack(bx[u]);
                const float2 av = Vec2<TI>::unpack(ba[u]);
                const float2 gv = Vec2<TI>::unpack(bg[u]);
                h_0 = rglru_step(h_0, xv.x, av.x, gv.x, la0, c);
                h_1 = rglru_step(h_1, xv.y, av.y, gv.y, la1, c);
                store2(yp + (size_t)(t0 + u) * D, h_0, h_1);
            }
        }
#pragma unroll
        for (int u = 0; u < P; ++u) {
            bx[u] = nx[u];
            ba[u] = na[u];
            bg[u] = ng[u];
        }
    }
    if (h_last) {
        h_last[(size_t)bi * D + d] = h_0;
        h_last[(size_t)bi * D + d + 1] = h_1;
    }
}

template <typename TI, typename TO>
cudaError_t launch_rg(const void* x, const void* ga, const void* gx, const float* lam,
                      const float* h0, void* y, float* h_last, int b, int T, int D, float c,
                      cudaStream_t s) {
    const long long threads = (long long)b * (D / 2);
    const long long blocks = (threads + kThreads - 1) / kThreads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // 16 steps in flight for 2-byte inputs, 8 for 4-byte ones (the same bytes)
    constexpr int P = sizeof(TI) == 2 ? 16 : 8;
    rglru_scan_kernel<TI, TO, P><<<(unsigned)blocks, kThreads, 0, s>>>(
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
