// decode.cu -- one step of the recurrent form (eq.6 of "Transformer取代者登場！…RetNet…（2）",
// section "Retention" 2); the "推理" paragraph uses it for O(1) decoding):
//     S <- gamma S + k^T v,   o = q S   (o reads the updated state)
//
// The step is a pure stream over the fp32 state: every element is read once
// and written once, so HBM bandwidth bounds it (2 * 4 * dk * dv bytes per
// (batch, head)).  Layout: state [b][H][dk][dv] row-major (dv contiguous).
//
// Mapping: one CTA of 256 threads per (batch*head, 128-column slice).  Lane l
// of every warp owns columns 4l..4l+3 of the slice (one float4: a warp covers
// 512 contiguous bytes of a state row); warp w owns rows w, w+8, w+16, ...
// Each thread keeps its q.S partial sums for its 4 columns in registers; the
// 8 warps' partials are added through shared memory at the end.  State loads
// and stores use the streaming cache hints (__ldcs/__stcs): the state is far
// larger than L2 and is not reused within a step.
#include "common.cuh"

namespace ret {
namespace {

constexpr int kWarps = 8;
constexpr int kCols = 128;  // columns per CTA: 32 lanes x float4
constexpr int kUnroll = 8;

template <typename TI, typename TO>
__global__ void __launch_bounds__(kWarps * 32)
recurrent_step_kernel(const TI* __restrict__ q, const TI* __restrict__ k,
                      const TI* __restrict__ v, float* __restrict__ state, TO* __restrict__ o,
                      int dk, int dv, int H, int slices, const HeadConsts hc) {
    __shared__ float qs[256], ks[256];
    __shared__ float4 red[kWarps][32];
    const int bh = blockIdx.x / slices;
    const int slice = blockIdx.x % slices;
    const int h = bh % H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < dk; i += blockDim.x) {
        qs[i] = ld(q + (size_t)bh * dk + i);
        ks[i] = ld(k + (size_t)bh * dk + i);
    }
    const int col = slice * kCols + lane * 4;
    const bool active = col < dv;  // dv is a multiple of 16, so a float4 never straddles dv
    float4 vv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active) {
        const TI* vp = v + (size_t)bh * dv + col;
        vv = make_float4(ld(vp), ld(vp + 1), ld(vp + 2), ld(vp + 3));
    }
    const float g = hc.g1[h];
    __syncthreads();

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float* base = state + (size_t)bh * dk * dv + col;
    if (active) {
        for (int a0 = warp; a0 < dk; a0 += kWarps * kUnroll) {
            float4 s[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                int a = a0 + u * kWarps;
                if (a < dk) s[u] = __ldcs(reinterpret_cast<const float4*>(base + (size_t)a * dv));
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                int a = a0 + u * kWarps;
                if (a < dk) {
                    float ka = ks[a], qa = qs[a];
                    float4 t;
                    t.x = fmaf(g, s[u].x, ka * vv.x);
                    t.y = fmaf(g, s[u].y, ka * vv.y);
                    t.z = fmaf(g, s[u].z, ka * vv.z);
                    t.w = fmaf(g, s[u].w, ka * vv.w);
                    __stcs(reinterpret_cast<float4*>(base + (size_t)a * dv), t);
                    acc.x = fmaf(qa, t.x, acc.x);
                    acc.y = fmaf(qa, t.y, acc.y);
                    acc.z = fmaf(qa, t.z, acc.z);
                    acc.w = fmaf(qa, t.w, acc.w);
                }
            }
        }
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && active) {
        float4 r = red[0][lane];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
            float4 p = red[w][lane];
            r.x += p.x; r.y += p.y; r.z += p.z; r.w += p.w;
        }
        TO* op = o + (size_t)bh * dv + col;
        st(op, r.x); st(op + 1, r.y); st(op + 2, r.z); st(op + 3, r.w);
    }
}

template <typename TI, typename TO>
cudaError_t launch(const void* q, const void* k, const void* v, float* state, void* o, int b,
                   int H, int dk, int dv, const HeadConsts& hc, cudaStream_t s) {
    int slices = (dv + kCols - 1) / kCols;
    long long grid = (long long)b * H * slices;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    recurrent_step_kernel<TI, TO><<<(unsigned)grid, kWarps * 32, 0, s>>>(
        static_cast<const TI*>(q), static_cast<const TI*>(k), static_cast<const TI*>(v), state,
        static_cast<TO*>(o), dk, dv, H, slices, hc);
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) count_launch(RET_KERNEL_DECODE);
    return err;
}

}  // namespace

cudaError_t launch_recurrent_step(const void* q, const void* k, const void* v, float* state,
                                  void* o, int in_bf16, int out_bf16, int b, int H, int dk,
                                  int dv, const HeadConsts& hc, cudaStream_t s) {
    using bf = __nv_bfloat16;
    if (in_bf16) {
        return out_bf16 ? launch<bf, bf>(q, k, v, state, o, b, H, dk, dv, hc, s)
                        : launch<bf, float>(q, k, v, state, o, b, H, dk, dv, hc, s);
    }
    return out_bf16 ? launch<float, bf>(q, k, v, state, o, b, H, dk, dv, hc, s)
                    : launch<float, float>(q, k, v, state, o, b, H, dk, dv, hc, s);
}

}  // namespace ret
