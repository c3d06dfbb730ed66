// simt_forms.cu -- CUDA-core (fp32 FMA) kernels of the parallel and chunkwise forms.
//
// They serve fp32 inputs (whose 1e-4 relative tolerance is below what tf32
// tensor-core products deliver) and every supported shape the tensor-core
// kernels do not take.  Plain shared-memory tiling, fp32 accumulation.
//
// Parallel form: "Transformer取代者登場！…RetNet…（2）", section "Retention" 1), eq.(5), with
// the three factors of "Retention Score 歸一化".  Chunkwise form: same page,
// "Retention" 3), eq.(7).
#include "common.cuh"

namespace ret {
namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------------------
// Parallel form.  CTA = (batch*head, 32-row query tile).  Key tiles of 32 up to
// the diagonal: S = Q K^T (one 32x32 tile in shared memory), scaled, decayed
// and masked into R, accumulated into the row sums, then O += R V.
// ---------------------------------------------------------------------------
constexpr int PQ = 32;  // query rows per CTA
constexpr int PK = 32;  // keys per tile

template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads)
parallel_simt_kernel(const TI* __restrict__ q, const TI* __restrict__ k,
                     const TI* __restrict__ v, TO* __restrict__ o, int H, int N, int dk, int dv,
                     int qtiles, unsigned flags, const HeadConsts hc) {
    extern __shared__ float smem[];
    const int ldk = dk + 1;
    float* Qs = smem;                 // [PQ][ldk]
    float* Ks = Qs + PQ * ldk;        // [PK][ldk]
    float* Vs = Ks + PK * ldk;        // [PK][dv]
    float* Ps = Vs + PK * dv;         // [PQ][PK+1]
    float* rsum = Ps + PQ * (PK + 1); // [PQ]

    const int bh = blockIdx.x / qtiles;
    const int qt = blockIdx.x % qtiles;
    const int h = bh % H;
    const int q0 = qt * PQ;
    const int t = threadIdx.x;
    const float l2g = hc.l2g[h];
    const float scale = (flags & RET_NORM_SCALE) ? rsqrtf((float)dk) : 1.0f;
    const TI* qb = q + (size_t)bh * N * dk;
    const TI* kb = k + (size_t)bh * N * dk;
    const TI* vb = v + (size_t)bh * N * dv;

    for (int e = t; e < PQ * dk; e += kThreads) {
        int r = e / dk, a = e % dk;
        Qs[r * ldk + a] = (q0 + r < N) ? ld(qb + (size_t)(q0 + r) * dk + a) : 0.f;
    }
    if (t < PQ) rsum[t] = 0.f;

    float acc[PQ][2];
#pragma unroll
    for (int r = 0; r < PQ; ++r) { acc[r][0] = 0.f; acc[r][1] = 0.f; }

    const int last_key = min(N, q0 + PQ) - 1;
    for (int k0 = 0; k0 <= last_key; k0 += PK) {
        __syncthreads();
        for (int e = t; e < PK * dk; e += kThreads) {
            int r = e / dk, a = e % dk;
            Ks[r * ldk + a] = (k0 + r < N) ? ld(kb + (size_t)(k0 + r) * dk + a) : 0.f;
        }
        for (int e = t; e < PK * dv; e += kThreads) {
            int r = e / dv, c = e % dv;
            Vs[r * dv + c] = (k0 + r < N) ? ld(vb + (size_t)(k0 + r) * dv + c) : 0.f;
        }
        __syncthreads();
        {   // scores: thread t -> row r = t/8, keys m = t%8 + 8j
            const int r = t >> 3, n = q0 + r;
            float part = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int m = (t & 7) + 8 * j, mm = k0 + m;
                float p = 0.f;
                if (n < N && mm <= n) {
                    float s = 0.f;
                    for (int a = 0; a < dk; ++a) s = fmaf(Qs[r * ldk + a], Ks[m * ldk + a], s);
                    float d = decay_pow(l2g, (float)(n - mm));
                    if (flags & RET_NORM_DECAY)
                        d *= rsqrtf(decay_rowsum(hc.lng[h], hc.omg[h], n));
                    p = s * scale * d;
                }
                Ps[r * (PK + 1) + m] = p;
                part += p;
            }
            // the 8 threads of row r are consecutive lanes of one warp
#pragma unroll
            for (int off = 4; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            if ((t & 7) == 0) rsum[r] += part;
        }
        __syncthreads();
        for (int m = 0; m < PK; ++m) {
            float v0 = (t < dv) ? Vs[m * dv + t] : 0.f;
            float v1 = (t + kThreads < dv) ? Vs[m * dv + t + kThreads] : 0.f;
#pragma unroll
            for (int r = 0; r < PQ; ++r) {
                float p = Ps[r * (PK + 1) + m];
                acc[r][0] = fmaf(p, v0, acc[r][0]);
                acc[r][1] = fmaf(p, v1, acc[r][1]);
            }
        }
    }
    __syncthreads();
    TO* ob = o + (size_t)bh * N * dv;
#pragma unroll
    for (int r = 0; r < PQ; ++r) {
        const int n = q0 + r;
        if (n >= N) break;
        float den = 1.f;
        if (flags & RET_NORM_ROWSUM) den = fmaxf(fabsf(rsum[r]), 1.0f);
        if (t < dv) st(ob + (size_t)n * dv + t, acc[r][0] / den);
        if (t + kThreads < dv) st(ob + (size_t)n * dv + t + kThreads, acc[r][1] / den);
    }
}

// ---------------------------------------------------------------------------
// Chunkwise form.  CTA = (batch*head, 64-column slice of dv); the fp32 state
// R[dk][64] of that slice stays in shared memory for the whole sequence.  For
// each chunk, 16-row query tiles take the intra-chunk part (key tiles of 16 up
// to the diagonal) and the cross-chunk part gamma^(j+1) q_j R; then
// R <- gamma^B R + sum_r gamma^(B-1-r) k_r^T v_r.
// ---------------------------------------------------------------------------
constexpr int CT = 16;  // rows per query / key tile
constexpr int CS = 64;  // dv columns per CTA

template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads)
chunkwise_simt_kernel(const TI* __restrict__ q, const TI* __restrict__ k,
                      const TI* __restrict__ v, TO* __restrict__ o, int H, int N, int dk, int dv,
                      int B, int slices, const HeadConsts hc, const float* __restrict__ state_in,
                      float* __restrict__ state_out) {
    extern __shared__ float smem[];
    const int ldk = dk + 1;
    float* Rs = smem;                // [dk][CS]
    float* Qs = Rs + dk * CS;        // [CT][ldk]
    float* Ks = Qs + CT * ldk;       // [CT][ldk]
    float* Vs = Ks + CT * ldk;       // [CT][CS]
    float* Ps = Vs + CT * CS;        // [CT][CT+1]

    const int bh = blockIdx.x / slices;
    const int c0 = (blockIdx.x % slices) * CS;
    const int ncol = min(CS, dv - c0);
    const int h = bh % H;
    const int t = threadIdx.x;
    const float l2g = hc.l2g[h];
    const float gB = hc.gB[h];
    const TI* qb = q + (size_t)bh * N * dk;
    const TI* kb = k + (size_t)bh * N * dk;
    const TI* vb = v + (size_t)bh * N * dv;
    TO* ob = o + (size_t)bh * N * dv;

    for (int e = t; e < dk * CS; e += kThreads) {
        int a = e / CS, c = e % CS;
        Rs[e] = (state_in && c < ncol) ? state_in[((size_t)bh * dk + a) * dv + c0 + c] : 0.f;
    }

    // output mapping of the 16x64 tile: row r = t/16, columns c = t%16 + 16j
    const int orow = t >> 4;
    for (int i0 = 0; i0 < N; i0 += B) {
        for (int j0 = 0; j0 < B; j0 += CT) {       // query tile rows i0+j0 .. +15
            __syncthreads();
            for (int e = t; e < CT * dk; e += kThreads) {
                int r = e / dk, a = e % dk;
                Qs[r * ldk + a] = ld(qb + (size_t)(i0 + j0 + r) * dk + a);
            }
            __syncthreads();
            float acc[4];
            const float xi = decay_pow(l2g, (float)(j0 + orow + 1));
#pragma unroll
            for (int j = 0; j < 4; ++j) {       // cross-chunk part from R_{i-1}
                const int c = (t & 15) + 16 * j;
                float s = 0.f;
                for (int a = 0; a < dk; ++a) s = fmaf(Qs[orow * ldk + a], Rs[a * CS + c], s);
                acc[j] = xi * s;
            }
            for (int r0 = 0; r0 <= j0; r0 += CT) {  // intra-chunk key tiles
                __syncthreads();
                for (int e = t; e < CT * dk; e += kThreads) {
                    int r = e / dk, a = e % dk;
                    Ks[r * ldk + a] = ld(kb + (size_t)(i0 + r0 + r) * dk + a);
                }
                for (int e = t; e < CT * CS; e += kThreads) {
                    int r = e / CS, c = e % CS;
                    Vs[e] = (c < ncol) ? ld(vb + (size_t)(i0 + r0 + r) * dv + c0 + c) : 0.f;
                }
                __syncthreads();
                {   // P[jr][m] = (q.k) gamma^(j-r), r <= j, one entry per thread
                    const int jr = t >> 4, m = t & 15;
                    const int jj = j0 + jr, rr = r0 + m;
                    float p = 0.f;
                    if (rr <= jj) {
                        float s = 0.f;
                        for (int a = 0; a < dk; ++a) s = fmaf(Qs[jr * ldk + a], Ks[m * ldk + a], s);
                        p = s * decay_pow(l2g, (float)(jj - rr));
                    }
                    Ps[jr * (CT + 1) + m] = p;
                }
                __syncthreads();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = (t & 15) + 16 * j;
                    float s = 0.f;
                    for (int m = 0; m < CT; ++m) s = fmaf(Ps[orow * (CT + 1) + m], Vs[m * CS + c], s);
                    acc[j] += s;
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = (t & 15) + 16 * j;
                if (c < ncol) st(ob + (size_t)(i0 + j0 + orow) * dv + c0 + c, acc[j]);
            }
        }
        // state update: R <- gamma^B R + sum_r zeta_r k_r^T v_r
        __syncthreads();
        for (int e = t; e < dk * CS; e += kThreads) Rs[e] *= gB;
        for (int r0 = 0; r0 < B; r0 += CT) {
            __syncthreads();
            for (int e = t; e < CT * dk; e += kThreads) {
                int r = e / dk, a = e % dk;
                Ks[r * ldk + a] = ld(kb + (size_t)(i0 + r0 + r) * dk + a)
                                  * decay_pow(l2g, (float)(B - 1 - r0 - r));
            }
            for (int e = t; e < CT * CS; e += kThreads) {
                int r = e / CS, c = e % CS;
                Vs[e] = (c < ncol) ? ld(vb + (size_t)(i0 + r0 + r) * dv + c0 + c) : 0.f;
            }
            __syncthreads();
            for (int e = t; e < dk * CS; e += kThreads) {
                int a = e / CS, c = e % CS;
                float s = Rs[e];
                for (int r = 0; r < CT; ++r) s = fmaf(Ks[r * ldk + a], Vs[r * CS + c], s);
                Rs[e] = s;
            }
        }
    }
    __syncthreads();
    if (state_out) {
        for (int e = t; e < dk * CS; e += kThreads) {
            int a = e / CS, c = e % CS;
            if (c < ncol) state_out[((size_t)bh * dk + a) * dv + c0 + c] = Rs[e];
        }
    }
}

template <typename TI, typename TO>
cudaError_t launch_par(const void* q, const void* k, const void* v, void* o, int b, int H, int N,
                       int dk, int dv, const HeadConsts& hc, unsigned flags, cudaStream_t s) {
    const int ldk = dk + 1;
    size_t smem = sizeof(float) * ((size_t)PQ * ldk + (size_t)PK * ldk + (size_t)PK * dv +
                                   PQ * (PK + 1) + PQ);
    auto kern = parallel_simt_kernel<TI, TO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int qtiles = (N + PQ - 1) / PQ;
    long long grid = (long long)b * H * qtiles;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, kThreads, smem, s>>>(static_cast<const TI*>(q), static_cast<const TI*>(k),
                                               static_cast<const TI*>(v), static_cast<TO*>(o), H, N,
                                               dk, dv, qtiles, flags, hc);
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) count_launch(RET_KERNEL_PARALLEL_SIMT);
    return err;
}

template <typename TI, typename TO>
cudaError_t launch_chk(const void* q, const void* k, const void* v, void* o, int b, int H, int N,
                       int dk, int dv, int B, const HeadConsts& hc, const float* si, float* so,
                       cudaStream_t s) {
    const int ldk = dk + 1;
    size_t smem = sizeof(float) * ((size_t)dk * CS + 2 * (size_t)CT * ldk + CT * CS +
                                   CT * (CT + 1));
    auto kern = chunkwise_simt_kernel<TI, TO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int slices = (dv + CS - 1) / CS;
    long long grid = (long long)b * H * slices;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, kThreads, smem, s>>>(static_cast<const TI*>(q), static_cast<const TI*>(k),
                                               static_cast<const TI*>(v), static_cast<TO*>(o), H, N,
                                               dk, dv, B, slices, hc, si, so);
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) count_launch(RET_KERNEL_CHUNKWISE_SIMT);
    return err;
}

}  // namespace

cudaError_t launch_parallel_simt(const void* q, const void* k, const void* v, void* o,
                                 int in_bf16, int out_bf16, int b, int H, int N, int dk, int dv,
                                 const HeadConsts& hc, unsigned flags, cudaStream_t s) {
    using bf = __nv_bfloat16;
    if (in_bf16)
        return out_bf16 ? launch_par<bf, bf>(q, k, v, o, b, H, N, dk, dv, hc, flags, s)
                        : launch_par<bf, float>(q, k, v, o, b, H, N, dk, dv, hc, flags, s);
    return out_bf16 ? launch_par<float, bf>(q, k, v, o, b, H, N, dk, dv, hc, flags, s)
                    : launch_par<float, float>(q, k, v, o, b, H, N, dk, dv, hc, flags, s);
}

cudaError_t launch_chunkwise_simt(const void* q, const void* k, const void* v, void* o,
                                  int in_bf16, int out_bf16, int b, int H, int N, int dk,
                                  int dv, int chunk, const HeadConsts& hc,
                                  const float* state_in, float* state_out, cudaStream_t s) {
    using bf = __nv_bfloat16;
    if (in_bf16)
        return out_bf16
                   ? launch_chk<bf, bf>(q, k, v, o, b, H, N, dk, dv, chunk, hc, state_in, state_out, s)
                   : launch_chk<bf, float>(q, k, v, o, b, H, N, dk, dv, chunk, hc, state_in, state_out, s);
    return out_bf16
               ? launch_chk<float, bf>(q, k, v, o, b, H, N, dk, dv, chunk, hc, state_in, state_out, s)
               : launch_chk<float, float>(q, k, v, o, b, H, N, dk, dv, chunk, hc, state_in, state_out, s);
}

}  // namespace ret
