// simt_backward.cu -- gradient of the chunkwise form on CUDA cores (fp32 FMA).
//
// "Transformer取代者登場！…RetNet…（2）", "訓練/推理": training runs the parallel and
// chunkwise forms.  The page prints no backward pass; what follows is the exact
// derivative of eq.(7) ("Retention" 3)).  With S0 the incoming state, o_n =
// gamma^(n+1) q_n S0 + sum_{m<=n} gamma^(n-m) (q_n.k_m) v_m and the loss
// L = sum_n dout_n.o_n + <dS_final, S_final>:
//
//   dq_n = sum_{m<=n} gamma^(n-m) (dout_n.v_m) k_m + gamma^(n+1) dout_n S0^T
//        -- the forward chunkwise scan itself with (q, k, v) -> (dout, v, k) and the
//           state R^T: R^T_i = gamma^B R^T_{i-1} + sum_r gamma^(B-1-r) v_r^T k_r.
//   G_n  = dL/dS_n = sum_{m>=n} gamma^(m-n) q_m^T dout_m + gamma^(N-1-n) dS_final
//   dv_n = k_n G_n,   dk_n = G_n v_n^T,   dS0 = gamma G_0
//        -- a scan backwards in time.  Per chunk i (rows iB+j), with the carry
//           T_i = gamma G_{(i+1)B} (T = dS_final for the last chunk):
//             dv_j = sum_{r>=j} gamma^(r-j) (k_j.q_r) dout_r + gamma^(B-1-j) k_j T_i
//             dk_j = sum_{r>=j} gamma^(r-j) (v_j.dout_r) q_r + gamma^(B-1-j) v_j T_i^T
//             T_{i-1} = gamma^B T_i + sum_r gamma^(r+1) q_r^T dout_r,   dS0 = T_{-1}.
//
// All three are one generic scan over (x, y, z) with a carried state St[dx][dz]:
//   forward: out_j = sum_{r<=j} gamma^(j-r) (x_j.y_r) z_r + gamma^(j+1) x_j St,
//            St <- gamma^B St + sum_r gamma^(B-1-r) y_r^T z_r;
//   reverse: chunks last to first,
//            out_j = sum_{r>=j} gamma^(r-j) (x_j.y_r) z_r + gamma^(B-1-j) x_j St,
//            St <- gamma^B St + sum_r gamma^(r+1) y_r^T z_r.
//   dq: forward, x = dout, y = v,    z = k, St = S0^T      (dx = dv, dz = dk)
//   dv: reverse, x = k,    y = q,    z = dout, St = dS_final   (dx = dk, dz = dv)
//   dk: reverse, x = v,    y = dout, z = q, St = dS_final^T  (dx = dv, dz = dk)
// One launch runs the three roles side by side: CTA = (role, batch*head, 64-column
// slice of dz), its fp32 state slice St[dx][64] resident in shared memory.
#include "common.cuh"

namespace ret {
namespace {

constexpr int kThreads = 256;
constexpr int CT = 16;  // rows per query / key tile
constexpr int CS = 64;  // output columns per CTA

struct ScanRole {
    const void* x;          // [bh][N][dx]
    const void* y;          // [bh][N][dx]
    const void* z;          // [bh][N][dz]
    void* out;              // [bh][N][dz]
    const float* st_in;     // [bh][dx][dz], or [bh][dz][dx] when st_in_t; NULL = zero
    float* st_out;          // [bh][dx][dz] after the last chunk, or NULL
    int dx, dz;
    int st_in_t;
    int rev;
    int slices;             // ceil(dz / CS)
    int cta0;               // first CTA of this role in the grid
};

struct ScanArgs {
    ScanRole role[3];
    int nroles;
};

template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads)
chunkwise_backward_simt_kernel(const ScanArgs args, int H, int N, int B, const HeadConsts hc) {
    extern __shared__ float smem[];
    int ri = 0;
    while (ri + 1 < args.nroles && (int)blockIdx.x >= args.role[ri + 1].cta0) ++ri;
    const ScanRole& R = args.role[ri];
    const int dx = R.dx, dz = R.dz, ldx = dx + 1;
    const bool rev = R.rev != 0;
    float* St = smem;                // [dx][CS]
    float* Xs = St + dx * CS;        // [CT][ldx]
    float* Ys = Xs + CT * ldx;       // [CT][ldx]
    float* Zs = Ys + CT * ldx;       // [CT][CS]
    float* Ps = Zs + CT * CS;        // [CT][CT+1]

    const int local = blockIdx.x - R.cta0;
    const int bh = local / R.slices;
    const int c0 = (local % R.slices) * CS;
    const int ncol = min(CS, dz - c0);
    const int h = bh % H;
    const int t = threadIdx.x;
    const float l2g = hc.l2g[h];
    const float gB = hc.gB[h];
    const TI* xb = static_cast<const TI*>(R.x) + (size_t)bh * N * dx;
    const TI* yb = static_cast<const TI*>(R.y) + (size_t)bh * N * dx;
    const TI* zb = static_cast<const TI*>(R.z) + (size_t)bh * N * dz;
    TO* ob = static_cast<TO*>(R.out) + (size_t)bh * N * dz;

    for (int e = t; e < dx * CS; e += kThreads) {
        const int a = e / CS, c = e % CS;
        float s = 0.f;
        if (R.st_in && c < ncol)
            s = R.st_in_t ? R.st_in[((size_t)bh * dz + c0 + c) * dx + a]
                          : R.st_in[((size_t)bh * dx + a) * dz + c0 + c];
        St[e] = s;
    }

    // output mapping of the 16x64 tile: row orow = t/16, columns (t%16) + 16j
    const int orow = t >> 4;
    const int nch = N / B;
    for (int ii = 0; ii < nch; ++ii) {
        const int i0 = (rev ? nch - 1 - ii : ii) * B;
        for (int j0 = 0; j0 < B; j0 += CT) {  // query tile rows i0+j0 .. +15
            __syncthreads();
            for (int e = t; e < CT * dx; e += kThreads) {
                const int r = e / dx, a = e % dx;
                Xs[r * ldx + a] = ld(xb + (size_t)(i0 + j0 + r) * dx + a);
            }
            __syncthreads();
            float acc[4];
            const int jrow = j0 + orow;
            const float cf = decay_pow(l2g, (float)(rev ? B - 1 - jrow : jrow + 1));
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // cross-chunk part from the carried state
                const int c = (t & 15) + 16 * j;
                float s = 0.f;
                for (int a = 0; a < dx; ++a) s = fmaf(Xs[orow * ldx + a], St[a * CS + c], s);
                acc[j] = cf * s;
            }
            // key tiles on the causal side of the query tile (diagonal tile included)
            const int rbeg = rev ? j0 : 0;
            const int rend = rev ? B : j0 + CT;
            for (int r0 = rbeg; r0 < rend; r0 += CT) {
                __syncthreads();
                for (int e = t; e < CT * dx; e += kThreads) {
                    const int r = e / dx, a = e % dx;
                    Ys[r * ldx + a] = ld(yb + (size_t)(i0 + r0 + r) * dx + a);
                }
                for (int e = t; e < CT * CS; e += kThreads) {
                    const int r = e / CS, c = e % CS;
                    Zs[e] = (c < ncol) ? ld(zb + (size_t)(i0 + r0 + r) * dz + c0 + c) : 0.f;
                }
                __syncthreads();
                {   // P[jr][m] = (x_j.y_r) gamma^|j-r| on the causal side, one entry per thread
                    const int jr = t >> 4, m = t & 15;
                    const int jj = j0 + jr, rr = r0 + m;
                    const int ex = rev ? rr - jj : jj - rr;
                    float p = 0.f;
                    if (ex >= 0) {
                        float s = 0.f;
                        for (int a = 0; a < dx; ++a) s = fmaf(Xs[jr * ldx + a], Ys[m * ldx + a], s);
                        p = s * decay_pow(l2g, (float)ex);
                    }
                    Ps[jr * (CT + 1) + m] = p;
                }
                __syncthreads();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = (t & 15) + 16 * j;
                    float s = 0.f;
                    for (int m = 0; m < CT; ++m) s = fmaf(Ps[orow * (CT + 1) + m], Zs[m * CS + c], s);
                    acc[j] += s;
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = (t & 15) + 16 * j;
                if (c < ncol) st(ob + (size_t)(i0 + jrow) * dz + c0 + c, acc[j]);
            }
        }
        // carried state: St <- gamma^B St + sum_r w_r y_r^T z_r
        __syncthreads();
        for (int e = t; e < dx * CS; e += kThreads) St[e] *= gB;
        for (int r0 = 0; r0 < B; r0 += CT) {
            __syncthreads();
            for (int e = t; e < CT * dx; e += kThreads) {
                const int r = e / dx, a = e % dx;
                const int rr = r0 + r;
                Ys[r * ldx + a] = ld(yb + (size_t)(i0 + rr) * dx + a) *
                                  decay_pow(l2g, (float)(rev ? rr + 1 : B - 1 - rr));
            }
            for (int e = t; e < CT * CS; e += kThreads) {
                const int r = e / CS, c = e % CS;
                Zs[e] = (c < ncol) ? ld(zb + (size_t)(i0 + r0 + r) * dz + c0 + c) : 0.f;
            }
            __syncthreads();
            for (int e = t; e < dx * CS; e += kThreads) {
                const int a = e / CS, c = e % CS;
                float s = St[e];
                for (int r = 0; r < CT; ++r) s = fmaf(Ys[r * ldx + a], Zs[r * CS + c], s);
                St[e] = s;
            }
        }
    }
    __syncthreads();
    if (R.st_out) {
        for (int e = t; e < dx * CS; e += kThreads) {
            const int a = e / CS, c = e % CS;
            if (c < ncol) R.st_out[((size_t)bh * dx + a) * dz + c0 + c] = St[e];
        }
    }
}

// ---------------------------------------------------------------------------
// Register-blocked variant for N a multiple of 64.  The gradient is the same
// function for every chunk length, so this kernel scans in chunks of BT = 64 tokens
// whatever chunk the caller validated.  Per chunk and 64-column slice the work is
// four small products, each thread owning a 4x4 micro-tile (rows 4ty.., columns
// 4tx..) and every operand staged k-major in shared memory so that one 16-byte
// load feeds four FMAs:
//   S  = X Y^T                       64 x 64, over dx in slabs of KS
//   O  = X St                        64 x 64, same slabs (state as it entered the chunk)
//   O  = cf (.) O + (S (.) decay) Z  decay and causal side applied in registers
//   St = gamma^BT St + Y^T (w (.) Z) 64-row blocks of St
// Global loads of the next slab / block go to registers before the current one is
// computed.
// ---------------------------------------------------------------------------
constexpr int BT = 64;   // internal chunk length
constexpr int KS = 16;   // slab width over dx
constexpr int LP = 68;   // padded row length of the k-major tiles (16-byte aligned rows)

template <typename TO> __device__ __forceinline__ void st4(TO* p, float4 v);
template <> __device__ __forceinline__ void st4<float>(float* p, float4 v) {
    *reinterpret_cast<float4*>(p) = v;
}
template <> __device__ __forceinline__ void st4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ float comp(const float4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads)
chunkwise_backward_blocked_kernel(const ScanArgs args, int H, int N, const HeadConsts hc) {
    extern __shared__ __align__(16) float smem[];
    int ri = 0;
    while (ri + 1 < args.nroles && (int)blockIdx.x >= args.role[ri + 1].cta0) ++ri;
    const ScanRole& R = args.role[ri];
    const int dx = R.dx, dz = R.dz;
    const bool rev = R.rev != 0;
    float* St = smem;                 // [dx][CS]   carried state slice
    float* Zs = St + dx * CS;         // [BT][CS]   z rows of the chunk
    float* Zw = Zs + BT * CS;         // [BT][CS]   the same rows times w_r
    float* XT = Zw + BT * CS;         // [KS][LP]   x slab, k-major
    float* YT = XT + KS * LP;         // [KS][LP]   y slab, k-major
    float* PT = YT + KS * LP;         // [BT][LP]   decayed scores, key-major; then y block

    const int local = blockIdx.x - R.cta0;
    const int bh = local / R.slices;
    const int c0 = (local % R.slices) * CS;
    const int ncol = min(CS, dz - c0);
    const int h = bh % H;
    const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
    const float l2g = hc.l2g[h];
    const float gB = hc.gB[h];        // gamma^BT
    const TI* xb = static_cast<const TI*>(R.x) + (size_t)bh * N * dx;
    const TI* yb = static_cast<const TI*>(R.y) + (size_t)bh * N * dx;
    const TI* zb = static_cast<const TI*>(R.z) + (size_t)bh * N * dz;
    TO* ob = static_cast<TO*>(R.out) + (size_t)bh * N * dz;

    for (int e = t; e < dx * CS; e += kThreads) {
        const int a = e / CS, c = e % CS;
        float s = 0.f;
        if (R.st_in && c < ncol)
            s = R.st_in_t ? R.st_in[((size_t)bh * dz + c0 + c) * dx + a]
                          : R.st_in[((size_t)bh * dx + a) * dz + c0 + c];
        St[e] = s;
    }

    const int nch = N / BT;
    const int nslab = dx / KS;
    const int nblk = (dx + BT - 1) / BT;
    for (int ii = 0; ii < nch; ++ii) {
        const int i0 = (rev ? nch - 1 - ii : ii) * BT;
        const TI* xc = xb + (size_t)i0 * dx;
        const TI* yc = yb + (size_t)i0 * dx;
        // previous chunk's readers of Zs / Zw / St are done
        __syncthreads();
        for (int u = 0; u < (BT * CS) / kThreads; ++u) {
            const int e = t + kThreads * u, r = e >> 6, c = e & 63;
            const float zv = (c < ncol) ? ld(zb + (size_t)(i0 + r) * dz + c0 + c) : 0.f;
            Zs[e] = zv;
            Zw[e] = zv * decay_pow(l2g, (float)(rev ? r + 1 : BT - 1 - r));
        }
        float S[4][4], O[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) S[i][j] = O[i][j] = 0.f;
        // slab element u of this thread: row (t + 256u) / KS, column (t + 256u) % KS
        float px[4], py[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = t + kThreads * u, r = e >> 4, k = e & 15;
            px[u] = ld(xc + (size_t)r * dx + k);
            py[u] = ld(yc + (size_t)r * dx + k);
        }
        for (int sl = 0; sl < nslab; ++sl) {
            __syncthreads();   // readers of the previous slab are done
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = t + kThreads * u, r = e >> 4, k = e & 15;
                XT[k * LP + r] = px[u];
                YT[k * LP + r] = py[u];
            }
            __syncthreads();
            if (sl + 1 < nslab) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int e = t + kThreads * u, r = e >> 4, k = e & 15;
                    px[u] = ld(xc + (size_t)r * dx + (sl + 1) * KS + k);
                    py[u] = ld(yc + (size_t)r * dx + (sl + 1) * KS + k);
                }
            }
            const float* st_slab = St + (size_t)sl * KS * CS;
#pragma unroll 4
            for (int k = 0; k < KS; ++k) {
                const float4 xa = *reinterpret_cast<const float4*>(XT + k * LP + 4 * ty);
                const float4 yv = *reinterpret_cast<const float4*>(YT + k * LP + 4 * tx);
                const float4 sv = *reinterpret_cast<const float4*>(st_slab + k * CS + 4 * tx);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float xi = comp(xa, i);
                    S[i][0] = fmaf(xi, yv.x, S[i][0]); S[i][1] = fmaf(xi, yv.y, S[i][1]);
                    S[i][2] = fmaf(xi, yv.z, S[i][2]); S[i][3] = fmaf(xi, yv.w, S[i][3]);
                    O[i][0] = fmaf(xi, sv.x, O[i][0]); O[i][1] = fmaf(xi, sv.y, O[i][1]);
                    O[i][2] = fmaf(xi, sv.z, O[i][2]); O[i][3] = fmaf(xi, sv.w, O[i][3]);
                }
            }
        }
        // decayed scores on the causal side, stored key-major
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int r = 4 * tx + jj;
            float4 p;
            float* pp = &p.x;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 4 * ty + i;
                const int ex = rev ? r - j : j - r;
                pp[i] = ex >= 0 ? S[i][jj] * decay_pow(l2g, (float)ex) : 0.f;
            }
            *reinterpret_cast<float4*>(PT + r * LP + 4 * ty) = p;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = 4 * ty + i;
            const float cf = decay_pow(l2g, (float)(rev ? BT - 1 - j : j + 1));
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) O[i][jj] *= cf;
        }
#pragma unroll 4
        for (int r = 0; r < BT; ++r) {
            const float4 pa = *reinterpret_cast<const float4*>(PT + r * LP + 4 * ty);
            const float4 zv = *reinterpret_cast<const float4*>(Zs + r * CS + 4 * tx);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float pi = comp(pa, i);
                O[i][0] = fmaf(pi, zv.x, O[i][0]); O[i][1] = fmaf(pi, zv.y, O[i][1]);
                O[i][2] = fmaf(pi, zv.z, O[i][2]); O[i][3] = fmaf(pi, zv.w, O[i][3]);
            }
        }
        if (4 * tx < ncol) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                st4<TO>(ob + (size_t)(i0 + 4 * ty + i) * dz + c0 + 4 * tx,
                        make_float4(O[i][0], O[i][1], O[i][2], O[i][3]));
        }
        // carried state, 64 rows at a time: St = gamma^BT St + Y^T Zw
        float py16[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int e = t + kThreads * u, r = e >> 6, al = e & 63;
            py16[u] = (al < dx) ? ld(yc + (size_t)r * dx + al) : 0.f;
        }
        for (int ab = 0; ab < nblk; ++ab) {
            __syncthreads();   // PT (scores, or the previous y block) is no longer read
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int e = t + kThreads * u, r = e >> 6, al = e & 63;
                PT[r * LP + al] = py16[u];
            }
            __syncthreads();
            if (ab + 1 < nblk) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int e = t + kThreads * u, r = e >> 6, al = e & 63;
                    const int a = (ab + 1) * BT + al;
                    py16[u] = (a < dx) ? ld(yc + (size_t)r * dx + a) : 0.f;
                }
            }
            const int a0 = ab * BT + 4 * ty;
            if (a0 < dx) {
                float A[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) A[i][j] = 0.f;
#pragma unroll 4
                for (int r = 0; r < BT; ++r) {
                    const float4 ya = *reinterpret_cast<const float4*>(PT + r * LP + 4 * ty);
                    const float4 zv = *reinterpret_cast<const float4*>(Zw + r * CS + 4 * tx);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float yi = comp(ya, i);
                        A[i][0] = fmaf(yi, zv.x, A[i][0]); A[i][1] = fmaf(yi, zv.y, A[i][1]);
                        A[i][2] = fmaf(yi, zv.z, A[i][2]); A[i][3] = fmaf(yi, zv.w, A[i][3]);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float4* sp = reinterpret_cast<float4*>(St + (size_t)(a0 + i) * CS + 4 * tx);
                    float4 sv = *sp;
                    sv.x = fmaf(gB, sv.x, A[i][0]); sv.y = fmaf(gB, sv.y, A[i][1]);
                    sv.z = fmaf(gB, sv.z, A[i][2]); sv.w = fmaf(gB, sv.w, A[i][3]);
                    *sp = sv;
                }
            }
        }
    }
    __syncthreads();
    if (R.st_out) {
        for (int e = t; e < dx * CS; e += kThreads) {
            const int a = e / CS, c = e % CS;
            if (c < ncol) R.st_out[((size_t)bh * dx + a) * dz + c0 + c] = St[e];
        }
    }
}

template <typename TI, typename TO>
cudaError_t launch_bwd(ScanArgs& args, int bH, int H, int N, int chunk, const HeadConsts& hc,
                       cudaStream_t s) {
    int dxmax = 0;
    long long grid = 0;
    for (int i = 0; i < args.nroles; ++i) {
        ScanRole& r = args.role[i];
        r.slices = (r.dz + CS - 1) / CS;
        r.cta0 = (int)grid;
        grid += (long long)bH * r.slices;
        if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        dxmax = r.dx > dxmax ? r.dx : dxmax;
    }
    cudaError_t e;
    if (chunk == BT) {   // register-blocked kernel (the caller passes BT when N % BT == 0)
        const size_t smem = sizeof(float) * ((size_t)dxmax * CS + 2 * (size_t)BT * CS +
                                             2 * (size_t)KS * LP + (size_t)BT * LP);
        auto kern = chunkwise_backward_blocked_kernel<TI, TO>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)grid, kThreads, smem, s>>>(args, H, N, hc);
    } else {
        const size_t smem = sizeof(float) * ((size_t)dxmax * CS + 2 * (size_t)CT * (dxmax + 1) +
                                             CT * CS + CT * (CT + 1));
        auto kern = chunkwise_backward_simt_kernel<TI, TO>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)grid, kThreads, smem, s>>>(args, H, N, chunk, hc);
    }
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) count_launch(RET_KERNEL_CHUNKWISE_BACKWARD_SIMT);
    return err;
}

}  // namespace

cudaError_t launch_chunkwise_backward_simt(const void* q, const void* k, const void* v,
                                           const void* dout, void* dq, void* dk, void* dv,
                                           int in_bf16, int out_bf16, int b, int H, int N,
                                           int dkk, int dvv, int chunk, const HeadConsts& hc,
                                           const float* state_in, const float* dstate_out,
                                           float* dstate_in, cudaStream_t s) {
    ScanArgs a{};
    a.nroles = 3;
    //            x     y     z     out  st_in       st_out     dx   dz   st_in_t rev
    a.role[0] = {dout, v,    k,    dq,  state_in,   nullptr,   dvv, dkk, 1,      0, 0, 0};
    a.role[1] = {k,    q,    dout, dv,  dstate_out, dstate_in, dkk, dvv, 0,      1, 0, 0};
    a.role[2] = {v,    dout, q,    dk,  dstate_out, nullptr,   dvv, dkk, 1,      1, 0, 0};
    using bf = __nv_bfloat16;
    const int bH = b * H;
    if (in_bf16)
        return out_bf16 ? launch_bwd<bf, bf>(a, bH, H, N, chunk, hc, s)
                        : launch_bwd<bf, float>(a, bH, H, N, chunk, hc, s);
    return out_bf16 ? launch_bwd<float, bf>(a, bH, H, N, chunk, hc, s)
                    : launch_bwd<float, float>(a, bH, H, N, chunk, hc, s);
}

}  // namespace ret
