// xpos.cu -- xPos rotation of Q and K, "Transformer取代者登場！…RetNet…（2）",
// "Retention", eqs.(2)-(3): Q_n e^{i n theta}, K_m e^{i m theta}, so that the score
// of eq.(4) (conjugate transpose) depends on n - m only.  For real inputs the pair of
// coordinates (2j, 2j+1) is one complex number, multiplied by e^{i p theta_j} at
// position p = pos0 + n.
//
// Memory-bound prologue (each element read and written once).  The phase depends on
// (p, j) only, so a thread owns four consecutive pairs of one position (16 bytes of a
// bf16 row, 32 of an fp32 one) and applies their rotations in every (batch, head) row,
// two rows' loads in flight before their stores; a block covers 8 consecutive positions
// of a 256-wide row, 4 KB contiguous per (batch, head).  The phase is exact to fp32: the
// fraction of turns p theta_j / (2 pi) is reduced in fp64 (one multiply, rint and a
// subtraction, exact for |p theta_j / 2pi| < 2^52), then sincospi in fp32.
#include "common.cuh"

namespace ret {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxPairs = 128;   // dk <= 256

struct Turns {
    double c[kMaxPairs];         // theta_j / (2 pi), computed on the host in fp64
};

// Eight consecutive elements as floats.
template <typename T> struct Oct;
template <> struct Oct<float> {
    static __device__ __forceinline__ void load(const float* p, float (&v)[8]) {
        const float4 a = *reinterpret_cast<const float4*>(p);
        const float4 b = *reinterpret_cast<const float4*>(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    static __device__ __forceinline__ void store(float* p, const float (&v)[8]) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
};
template <> struct Oct<__nv_bfloat16> {
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[8]) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

__device__ __forceinline__ void rotate4(float (&v)[8], const float (&cs)[4], const float (&sn)[4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float a = v[2 * u], b = v[2 * u + 1];
        v[2 * u] = a * cs[u] - b * sn[u];
        v[2 * u + 1] = a * sn[u] + b * cs[u];
    }
}

template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads)
xpos_kernel(const TI* q, const TI* k, TO* q_out, TO* k_out, int bH, int N, int d,
            long long pos0, const Turns turns) {
    const int groups = d >> 3;                      // four pairs per thread
    const long long idx = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (idx >= (long long)N * groups) return;
    const int n = (int)(idx / groups), g = (int)(idx % groups);
    float cs[4], sn[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const double t = (double)(pos0 + n) * turns.c[4 * g + u];
        const float f = (float)(t - rint(t));    // in [-1/2, 1/2] turns
        sincospif(2.0f * f, &sn[u], &cs[u]);
    }
    const size_t row = (size_t)N * d;
    const size_t off0 = (size_t)n * d + 8 * g;
    int r = 0;
    for (; r + 1 < bH; r += 2) {                    // two rows in flight
        float a[8], b[8];
        Oct<TI>::load(q + (size_t)r * row + off0, a);
        Oct<TI>::load(q + (size_t)(r + 1) * row + off0, b);
        rotate4(a, cs, sn);
        rotate4(b, cs, sn);
        Oct<TO>::store(q_out + (size_t)r * row + off0, a);
        Oct<TO>::store(q_out + (size_t)(r + 1) * row + off0, b);
        if (k) {
            Oct<TI>::load(k + (size_t)r * row + off0, a);
            Oct<TI>::load(k + (size_t)(r + 1) * row + off0, b);
            rotate4(a, cs, sn);
            rotate4(b, cs, sn);
            Oct<TO>::store(k_out + (size_t)r * row + off0, a);
            Oct<TO>::store(k_out + (size_t)(r + 1) * row + off0, b);
        }
    }
    if (r < bH) {
        float a[8];
        Oct<TI>::load(q + (size_t)r * row + off0, a);
        rotate4(a, cs, sn);
        Oct<TO>::store(q_out + (size_t)r * row + off0, a);
        if (k) {
            Oct<TI>::load(k + (size_t)r * row + off0, a);
            rotate4(a, cs, sn);
            Oct<TO>::store(k_out + (size_t)r * row + off0, a);
        }
    }
}

template <typename TI, typename TO>
cudaError_t launch_x(const void* q, const void* k, void* q_out, void* k_out, int bH, int N,
                     int d, long long pos0, const Turns& turns, cudaStream_t s) {
    const long long threads = (long long)N * (d / 8);
    const long long blocks = (threads + kThreads - 1) / kThreads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    xpos_kernel<TI, TO><<<(unsigned)blocks, kThreads, 0, s>>>(
        static_cast<const TI*>(q), static_cast<const TI*>(k), static_cast<TO*>(q_out),
        static_cast<TO*>(k_out), bH, N, d, pos0, turns);
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) count_launch(RET_KERNEL_XPOS);
    return err;
}

}  // namespace

cudaError_t launch_xpos_rotate(const void* q, const void* k, void* q_out, void* k_out,
                               int in_bf16, int out_bf16, int b, int H, int N, int d,
                               const double* theta, long long pos0, cudaStream_t s) {
    if (d / 2 > kMaxPairs) return cudaErrorInvalidValue;
    Turns turns;
    for (int j = 0; j < d / 2; ++j) turns.c[j] = theta[j] / (2.0 * M_PI);
    for (int j = d / 2; j < kMaxPairs; ++j) turns.c[j] = 0.0;
    using bf = __nv_bfloat16;
    const int bH = b * H;
    if (in_bf16)
        return out_bf16 ? launch_x<bf, bf>(q, k, q_out, k_out, bH, N, d, pos0, turns, s)
                        : launch_x<bf, float>(q, k, q_out, k_out, bH, N, d, pos0, turns, s);
    return out_bf16 ? launch_x<float, bf>(q, k, q_out, k_out, bH, N, d, pos0, turns, s)
                    : launch_x<float, float>(q, k, q_out, k_out, bH, N, d, pos0, turns, s);
}

}  // namespace ret
