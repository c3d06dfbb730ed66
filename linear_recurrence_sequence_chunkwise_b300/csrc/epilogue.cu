// epilogue.cu -- gated multi-scale retention epilogue ("Transformer取代者登場！…RetNet…（2）",
// section "門控多尺度 Retention"): GroupNorm over each head's dv outputs of one
// token (biased variance, eps inside the square root, optional per-channel
// affine), then the swish gate: out = swish(G) * GroupNorm(Y), swish(x) = x*sigmoid(x).
//
// Memory-bound: per (batch, token, head) it reads dv values of Y and of G and
// writes dv outputs.  One warp per group; lane l owns 8-element pieces
// l, l+32 of the group (16-byte vector loads for bf16, two for fp32), so a
// warp reads each group's contiguous dv values in whole 32-byte sectors.
// Layouts: y [b][H][N][dv]; g, out [b][N][H*dv]; weight, bias [H*dv].
#include "common.cuh"

namespace ret {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxPieces = 2;  // dv <= 512 = 2 pieces x 8 elements x 32 lanes

template <typename T> __device__ __forceinline__ void load8(const T* p, float* x);
template <> __device__ __forceinline__ void load8<float>(const float* p, float* x) {
    float4 a = *reinterpret_cast<const float4*>(p);
    float4 b = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <> __device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float* x) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
template <typename T> __device__ __forceinline__ void store8(T* p, const float* x);
template <> __device__ __forceinline__ void store8<float>(float* p, const float* x) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(x[4], x[5], x[6], x[7]);
}
template <> __device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, const float* x) {
    uint4 u;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 t = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&t);
    }
    u.x = w[0]; u.y = w[1]; u.z = w[2]; u.w = w[3];
    *reinterpret_cast<uint4*>(p) = u;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <typename TY, typename TG, typename TO>
__global__ void __launch_bounds__(kWarps * 32)
msr_epilogue_kernel(const TY* __restrict__ y, const TG* __restrict__ g, TO* __restrict__ out,
                    int H, int N, int dv, long long groups, float eps,
                    const float* __restrict__ weight, const float* __restrict__ bias) {
    const long long grp = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (grp >= groups) return;
    const int lane = threadIdx.x & 31;
    const int h = (int)(grp % H);
    const long long bn = grp / H;          // b * N + n
    const int n = (int)(bn % N);
    const long long bi = bn / N;
    const TY* yp = y + (((size_t)bi * H + h) * N + n) * dv;
    const size_t go = (size_t)bn * H * dv + (size_t)h * dv;
    const int pieces = dv >> 3;

    float x[kMaxPieces][8];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPieces; ++i) {
        int p = lane + 32 * i;
        if (p < pieces) {
            load8(yp + 8 * p, x[i]);
#pragma unroll
            for (int e = 0; e < 8; ++e) s += x[i][e];
        }
    }
    const float mu = warp_sum(s) / (float)dv;
    float s2 = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPieces; ++i) {
        int p = lane + 32 * i;
        if (p < pieces) {
#pragma unroll
            for (int e = 0; e < 8; ++e) { float d = x[i][e] - mu; s2 += d * d; }
        }
    }
    const float var = warp_sum(s2) / (float)dv;
    const float rstd = 1.0f / sqrtf(var + eps);
#pragma unroll
    for (int i = 0; i < kMaxPieces; ++i) {
        int p = lane + 32 * i;
        if (p < pieces) {
            float gv[8], o[8];
            load8(g + go + 8 * p, gv);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float yn = (x[i][e] - mu) * rstd;
                int ch = h * dv + 8 * p + e;
                if (weight) yn *= weight[ch];
                if (bias) yn += bias[ch];
                float sw = gv[e] / (1.0f + expf(-gv[e]));
                o[e] = sw * yn;
            }
            store8(out + go + 8 * p, o);
        }
    }
}

template <typename TY, typename TG, typename TO>
cudaError_t launch(const void* y, const void* g, void* out, int b, int H, int N, int dv,
                   float eps, const float* w, const float* bias, cudaStream_t s) {
    long long groups = (long long)b * N * H;
    long long grid = (groups + kWarps - 1) / kWarps;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    msr_epilogue_kernel<TY, TG, TO><<<(unsigned)grid, kWarps * 32, 0, s>>>(
        static_cast<const TY*>(y), static_cast<const TG*>(g), static_cast<TO*>(out), H, N, dv,
        groups, eps, w, bias);
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) count_launch(RET_KERNEL_EPILOGUE);
    return err;
}

template <typename TY, typename TG>
cudaError_t launch_o(const void* y, const void* g, void* out, int ob, int b, int H, int N,
                     int dv, float eps, const float* w, const float* bias, cudaStream_t s) {
    return ob ? launch<TY, TG, __nv_bfloat16>(y, g, out, b, H, N, dv, eps, w, bias, s)
              : launch<TY, TG, float>(y, g, out, b, H, N, dv, eps, w, bias, s);
}

template <typename TY>
cudaError_t launch_g(const void* y, const void* g, void* out, int gb, int ob, int b, int H,
                     int N, int dv, float eps, const float* w, const float* bias,
                     cudaStream_t s) {
    return gb ? launch_o<TY, __nv_bfloat16>(y, g, out, ob, b, H, N, dv, eps, w, bias, s)
              : launch_o<TY, float>(y, g, out, ob, b, H, N, dv, eps, w, bias, s);
}

}  // namespace

cudaError_t launch_msr_epilogue(const void* y, const void* g, void* out, int y_bf16,
                                int g_bf16, int out_bf16, int b, int H, int N, int dv,
                                float eps, const float* weight, const float* bias,
                                cudaStream_t s) {
    return y_bf16 ? launch_g<__nv_bfloat16>(y, g, out, g_bf16, out_bf16, b, H, N, dv, eps,
                                            weight, bias, s)
                  : launch_g<float>(y, g, out, g_bf16, out_bf16, b, H, N, dv, eps, weight,
                                    bias, s);
}

}  // namespace ret
