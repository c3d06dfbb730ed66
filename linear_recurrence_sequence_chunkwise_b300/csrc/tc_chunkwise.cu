// tc_chunkwise.cu -- chunkwise recurrent retention on sm_103a tensor cores (tcgen05 + TMA).
//
// Computes eq.(7) of "Transformer取代者登場！…RetNet…（2）", section "Retention" 3): inside
// each chunk of B tokens the parallel form, across chunks the recurrent state
//     O[iB+j] = sum_{r<=j} (q_j.k_r) g^(j-r) v_r + g^(j+1) (q_j R_{i-1})
//     R_i     = sum_r g^(B-1-r) k_r^T v_r + g^B R_{i-1}
// for bf16 Q/K/V, fp32 accumulation, fp32 state, B in {128, 256}, dk in {128, 256},
// dv a multiple of 64.
//
// Work split: one CTA per (batch*head, 64-column block of dv).  State columns
// are independent (R = K^T V and q R both separate over dv), so each CTA owns
// R[:, 64 cols] in tensor memory for the whole sequence and scans the chunks in
// order.  The intra-chunk score tile Q K^T does not depend on dv and is
// recomputed by each of the dv/64 CTAs of a head.
//
// Inside a chunk, rows and keys go in 128-blocks (rb = row block, cb = key
// block, cb <= rb).  Decay factors are folded so that no per-element power is
// needed:
//   * V block cb is scaled in shared memory by g^(127-r') (r' = row in block):
//     Vt = g^(127-r') v.
//   * Score tile (rb, cb) then needs one factor per ROW j':
//     P'[j'][r'] = (q.k) g^(128(rb-cb) + j' - 127), masked to r' <= j' on the
//     diagonal, so that P' Vt = sum (q.k) g^(j-r) v exactly.
//   * The state update becomes R <- g^128 R; R += K_cb^T Vt_cb, once per key
//     block, which expands to g^B R_{i-1} + sum_r g^(B-1-r) k_r^T v_r.
//   * The cross-chunk read uses xi_j = g^(128 rb + j' + 1), applied per row.
// The folded factors stay inside fp32/bf16 range when g^127 >= 2^-64
// (g >= 0.7071); other decays go to the CUDA-core kernel.
//
// Roles (192 threads): warp 0 issues TMA loads, warp 1 owns tensor memory and
// issues tcgen05.mma, warps 2-5 (one per 32-lane TMEM quarter) convert scores,
// rescale the state, scale V and write outputs.  Every wait is bounded; a
// wait that gives up sets the device error word and the CTA unwinds.
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [  0,128) R: state, dk rows 0-127 (cols 0-63) and 128-255 (cols 64-127)
//   [128,384) S: two 128-column score buffers
//   [384,448) O: intra-chunk output accumulator of the current row block
//   [448,512) C: cross-chunk accumulator q R_{i-1} of the current row block
// Shared memory (1024-aligned, 224 KB):
//   4 ring stages x 32 KB (one stage = 128 rows x 128 columns of Q or K,
//   two 64-column 128B-swizzled atoms), 2 x 16 KB scaled V blocks, 32 KB bf16
//   copy of R_{i-1} (B operand of q R), 32 KB bf16 score tile P'.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace ret {
namespace {

__device__ unsigned g_err_chunkwise;

using namespace tc;

constexpr int kStages = 4;
constexpr int kAtom = 128 * 128;          // 128 rows x 64 bf16
constexpr int kStage = 2 * kAtom;         // 128 rows x 128 bf16
constexpr int kRingBytes = kStages * kStage;
constexpr int kVtOff = kRingBytes;        // 2 x kAtom
constexpr int kRbOff = kVtOff + 2 * kAtom;
constexpr int kPOff = kRbOff + 2 * kAtom;
constexpr int kSmemBytes = kPOff + 2 * kAtom;   // 229376
constexpr int kThreads = 192;

constexpr uint32_t kTR = 0, kTS = 128, kTO = 384, kTC = 448;

struct Decay {
    float l2g[kMaxHeads];   // log2(gamma)
    float g128[kMaxHeads];  // gamma^128
};

struct Bars {
    uint64_t full[kStages], empty[kStages];
    uint64_t vfull[2], vempty[2], vt_ready[2];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full, p_empty;
    uint64_t o_full, o_free, c_full, c_free;
    uint64_t r_done, rb_ready, r_scaled;
    uint64_t drain;
};

__device__ __forceinline__ void fail(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_err_chunkwise, 1u);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
chunkwise_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, void* __restrict__ out,
                    const float* __restrict__ state_in, float* __restrict__ state_out, int N,
                    int B, int H, int dk, int dv, const Decay dc) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* ring = sm;
    uint8_t* vt = sm + kVtOff;
    uint8_t* rbuf = sm + kRbOff;
    uint8_t* pbuf = sm + kPOff;
    __shared__ Bars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nblk = dv / 64;
    const int bh = blockIdx.x / nblk, blk = blockIdx.x % nblk;
    const int head = bh % H;
    const int nrb = B / 128, nh = dk / 128, nchunks = N / B;
    volatile int* abort_p = &abort_flag;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < kStages; ++s) { mbar_init(&bars.full[s], 1); mbar_init(&bars.empty[s], 1); }
        for (int c = 0; c < 2; ++c) {
            mbar_init(&bars.vfull[c], 1); mbar_init(&bars.vempty[c], 1);
            mbar_init(&bars.vt_ready[c], 128);
            mbar_init(&bars.s_full[c], 1); mbar_init(&bars.s_free[c], 128);
        }
        mbar_init(&bars.p_full, 128); mbar_init(&bars.p_empty, 1);
        mbar_init(&bars.o_full, 1); mbar_init(&bars.o_free, 128);
        mbar_init(&bars.c_full, 1); mbar_init(&bars.c_free, 128);
        mbar_init(&bars.r_done, 1); mbar_init(&bars.rb_ready, 128);
        mbar_init(&bars.r_scaled, 128); mbar_init(&bars.drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) { tmem_alloc(&tmem_slot, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&mq); tma_prefetch_desc(&mk); tma_prefetch_desc(&mv);
            uint32_t fill = 0, vuse[2] = {0, 0};
            bool ok = true;
            for (int i = 0; i < nchunks && ok; ++i) {
                for (int rb = 0; rb < nrb && ok; ++rb) {
                    const int row0 = bh * N + i * B + 128 * rb;
                    for (int which = 0; which < 2 && ok; ++which) {
                        const CUtensorMap* m = which ? &mk : &mq;
                        for (int hh = 0; hh < nh; ++hh) {
                            const int s = fill % kStages;
                            if (!mbar_wait(&bars.empty[s], ((fill / kStages) & 1) ^ 1, abort_p)) { ok = false; break; }
                            mbar_arrive_expect_tx(&bars.full[s], kStage);
                            tma_load_2d(ring + s * kStage, m, hh * 128, row0, &bars.full[s]);
                            tma_load_2d(ring + s * kStage + kAtom, m, hh * 128 + 64, row0, &bars.full[s]);
                            ++fill;
                        }
                    }
                    if (!ok) break;
                    if (!mbar_wait(&bars.vempty[rb], (vuse[rb] & 1) ^ 1, abort_p)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bars.vfull[rb], kAtom);
                    tma_load_2d(vt + rb * kAtom, &mv, blk * 64, row0, &bars.vfull[rb]);
                    ++vuse[rb];
                }
            }
            if (!ok) {
                fail(abort_p);
                // let loads already in flight land before the CTA unwinds
                for (uint32_t f = fill > kStages ? fill - kStages : 0; f < fill; ++f)
                    mbar_wait(&bars.full[f % kStages], (f / kStages) & 1, nullptr, 100000000ull);
                for (int c = 0; c < nrb; ++c)
                    if (vuse[c]) mbar_wait(&bars.vfull[c], (vuse[c] - 1) & 1, nullptr, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, 128, 0, 0);
            const uint32_t id_c = idesc_bf16(128, 64, 0, 1);
            const uint32_t id_pv = idesc_bf16(128, 64, 0, 1);
            const uint32_t id_r = idesc_bf16(128, 64, 1, 1);
            const uint32_t ring_a = smem_u32(ring), vt_a = smem_u32(vt);
            const uint32_t rb_a = smem_u32(rbuf), p_a = smem_u32(pbuf);
            uint32_t s_use[2] = {0, 0}, sbuf = 0, c_use = 0, o_use = 0, p_use = 0, rsc = 0;
            bool ok = true;
            auto wait = [&](uint64_t* bar, uint32_t par) {
                if (ok && !mbar_wait(bar, par, abort_p)) { ok = false; fail(abort_p); }
                return ok;
            };
            auto stage_addr = [&](uint32_t f) { return ring_a + (f % kStages) * kStage; };
            for (int i = 0; i < nchunks && ok; ++i) {
                const uint32_t base = (uint32_t)i * nrb * 2 * nh;
                for (int rb = 0; rb < nrb && ok; ++rb) {
                    const uint32_t qf = base + rb * 2 * nh;
                    for (int hh = 0; hh < nh; ++hh)
                        wait(&bars.full[(qf + hh) % kStages], ((qf + hh) / kStages) & 1);
                    for (int cb = 0; cb <= rb && ok; ++cb) {
                        const uint32_t kf = base + cb * 2 * nh + nh;
                        if (cb == rb)
                            for (int hh = 0; hh < nh; ++hh)
                                wait(&bars.full[(kf + hh) % kStages], ((kf + hh) / kStages) & 1);
                        // S(rb, cb) = Q_rb K_cb^T  (M=128, N=128, K=dk)
                        if (!wait(&bars.s_free[sbuf], (s_use[sbuf] & 1) ^ 1)) break;
                        tc_fence_after();
                        const uint32_t ts = tmem + kTS + 128 * sbuf;
                        for (int k0 = 0; k0 < dk; k0 += 16) {
                            const uint32_t off = ((k0 % 128) / 64) * kAtom + (k0 % 64) * 2;
                            uint64_t ad = sdesc_sw128(stage_addr(qf + k0 / 128) + off, 16, 1024);
                            uint64_t bd = sdesc_sw128(stage_addr(kf + k0 / 128) + off, 16, 1024);
                            mma_bf16(ts, ad, bd, id_s, k0 > 0);
                        }
                        mma_commit(&bars.s_full[sbuf]);
                        ++s_use[sbuf];
                        sbuf ^= 1;
                        if (rb == nrb - 1) {
                            // state update with key block cb: R += K_cb^T Vt_cb (after R <- g^128 R)
                            wait(&bars.vt_ready[cb], i & 1);
                            if (!wait(&bars.r_scaled, rsc & 1)) break;
                            ++rsc;
                            tc_fence_after();
                            for (int hh = 0; hh < nh; ++hh)
                                for (int t0 = 0; t0 < 128; t0 += 16) {
                                    uint64_t ad = sdesc_sw128(stage_addr(kf + hh) + t0 * 128, kAtom, 1024);
                                    uint64_t bd = sdesc_sw128(vt_a + cb * kAtom + t0 * 128, kAtom, 1024);
                                    mma_bf16(tmem + kTR + 64 * hh, ad, bd, id_r, 1);
                                }
                            mma_commit(&bars.r_done);
                            for (int hh = 0; hh < nh; ++hh) mma_commit(&bars.empty[(kf + hh) % kStages]);
                        }
                    }
                    if (!ok) break;
                    // C_rb = Q_rb R_{i-1}  (M=128, N=64, K=dk)
                    if (rb == 0) wait(&bars.rb_ready, i & 1);
                    if (!wait(&bars.c_free, (c_use & 1) ^ 1)) break;
                    ++c_use;
                    tc_fence_after();
                    for (int k0 = 0; k0 < dk; k0 += 16) {
                        const uint32_t off = ((k0 % 128) / 64) * kAtom + (k0 % 64) * 2;
                        uint64_t ad = sdesc_sw128(stage_addr(qf + k0 / 128) + off, 16, 1024);
                        uint64_t bd = sdesc_sw128(rb_a + k0 * 128, kAtom, 1024);
                        mma_bf16(tmem + kTC, ad, bd, id_c, k0 > 0);
                    }
                    mma_commit(&bars.c_full);
                    for (int hh = 0; hh < nh; ++hh) mma_commit(&bars.empty[(qf + hh) % kStages]);
                    // O_rb = sum_cb P'(rb, cb) Vt_cb  (M=128, N=64, K=128 per key block)
                    if (!wait(&bars.o_free, (o_use & 1) ^ 1)) break;
                    ++o_use;
                    for (int cb = 0; cb <= rb && ok; ++cb) {
                        if (!wait(&bars.p_full, p_use & 1)) break;
                        ++p_use;
                        tc_fence_after();
                        for (int t0 = 0; t0 < 128; t0 += 16) {
                            uint64_t ad = sdesc_sw128(p_a + (t0 / 64) * kAtom + (t0 % 64) * 2, 16, 1024);
                            uint64_t bd = sdesc_sw128(vt_a + cb * kAtom + t0 * 128, kAtom, 1024);
                            mma_bf16(tmem + kTO, ad, bd, id_pv, (cb | t0) != 0);
                        }
                        mma_commit(&bars.p_empty);
                        if (rb == nrb - 1) mma_commit(&bars.vempty[cb]);
                    }
                    mma_commit(&bars.o_full);
                }
            }
            // every issued MMA must finish before tensor memory is released
            mma_commit(&bars.drain);
            mbar_wait(&bars.drain, 0, nullptr, 200000000ull);
        }
    } else {
        // ------------------------------------------------------------ transform warps
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane;              // TMEM lane = tile row
        const uint32_t lrow = (uint32_t)(32 * q4) << 16;
        const float l2g = dc.l2g[head];
        const float g128 = dc.g128[head];
        uint32_t rdone = 0, s_cnt[2] = {0, 0}, sbuf = 0, p_cnt = 0, o_cnt = 0;
        bool ok = true;
        // the warp's tcgen05 loads/stores are warp-collective: keep the outcome
        // of every wait uniform across the warp
        auto wait = [&](uint64_t* bar, uint32_t par) {
            if (!ok) return false;
            const bool got = __all_sync(0xffffffffu, mbar_wait(bar, par, abort_p));
            if (!got) { ok = false; if (lane == 0) fail(abort_p); }
            return ok;
        };
        // R <- g^128 R, reading and writing the TMEM state in place
        auto rescale = [&]() {
            for (int hh = 0; hh < nh; ++hh)
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    float x[32];
                    tmem_ld32(tmem + lrow + kTR + 64 * hh + c0, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] *= g128;
                    tmem_st32(tmem + lrow + kTR + 64 * hh + c0, x);
                }
            tmem_wait_st();
        };
        for (int i = 0; i < nchunks && ok; ++i) {
            // ---- R_{i-1}: bf16 copy for q R, then R <- g^128 R
            if (i > 0) {
                if (!wait(&bars.r_done, rdone & 1)) break;
                ++rdone;
                tc_fence_after();
            }
            for (int hh = 0; hh < nh; ++hh) {
                const int a = 128 * hh + row;          // dk row
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    float x[32];
                    if (i == 0) {
                        if (state_in) {
                            const float4* src = reinterpret_cast<const float4*>(
                                state_in + ((size_t)bh * dk + a) * dv + blk * 64 + c0);
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                float4 f = src[j];
                                x[4 * j] = f.x; x[4 * j + 1] = f.y; x[4 * j + 2] = f.z; x[4 * j + 3] = f.w;
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) x[j] = 0.f;
                        }
                    } else {
                        tmem_ld32(tmem + lrow + kTR + 64 * hh + c0, x);
                        tmem_wait_ld();
                    }
                    // 32 values = 4 chunks of 8 bf16 in the 128B-swizzled row a
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int chunk = (c0 / 8) + cc;
                        uint4 u;
                        u.x = pack_bf16(x[8 * cc + 0], x[8 * cc + 1]);
                        u.y = pack_bf16(x[8 * cc + 2], x[8 * cc + 3]);
                        u.z = pack_bf16(x[8 * cc + 4], x[8 * cc + 5]);
                        u.w = pack_bf16(x[8 * cc + 6], x[8 * cc + 7]);
                        *reinterpret_cast<uint4*>(rbuf + a * 128 + ((chunk ^ (a & 7)) << 4)) = u;
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] *= g128;
                    tmem_st32(tmem + lrow + kTR + 64 * hh + c0, x);
                }
            }
            tmem_wait_st();
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(&bars.rb_ready);
            mbar_arrive(&bars.r_scaled);

            for (int rb = 0; rb < nrb && ok; ++rb) {
                // ---- scale V block rb: row r' times g^(127-r')
                if (!wait(&bars.vfull[rb], i & 1)) break;
                {
                    const float f = exp2f(l2g * (float)(127 - row));
                    uint4* vp = reinterpret_cast<uint4*>(vt + rb * kAtom + row * 128);
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        uint4 u = vp[cc];
                        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float lo = __uint_as_float(w[e] << 16) * f;
                            float hi = __uint_as_float(w[e] & 0xffff0000u) * f;
                            w[e] = pack_bf16(lo, hi);
                        }
                        vp[cc] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                fence_proxy_async();
                mbar_arrive(&bars.vt_ready[rb]);

                for (int cb = 0; cb <= rb && ok; ++cb) {
                    if (rb == nrb - 1 && cb >= 1) {
                        if (!wait(&bars.r_done, rdone & 1)) break;
                        ++rdone;
                        tc_fence_after();
                        rescale();
                        tc_fence_before();
                        mbar_arrive(&bars.r_scaled);
                    }
                    // ---- P'(rb, cb) = S * g^(128(rb-cb) + j' - 127), causal on the diagonal
                    if (!wait(&bars.s_full[sbuf], s_cnt[sbuf] & 1)) break;
                    ++s_cnt[sbuf];
                    if (!wait(&bars.p_empty, (p_cnt & 1) ^ 1)) break;
                    ++p_cnt;
                    tc_fence_after();
                    const float f = exp2f(l2g * (float)(128 * (rb - cb) + row - 127));
                    const uint32_t ts = tmem + lrow + kTS + 128 * sbuf;
                    for (int c0 = 0; c0 < 128; c0 += 32) {
                        float x[32];
                        tmem_ld32(ts + c0, x);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const bool keep = (rb != cb) || (c0 + j <= row);
                            x[j] = keep ? x[j] * f : 0.f;
                        }
                        uint8_t* prow = pbuf + (c0 / 64) * kAtom + row * 128;
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            const int chunk = ((c0 % 64) / 8) + cc;
                            uint4 u;
                            u.x = pack_bf16(x[8 * cc + 0], x[8 * cc + 1]);
                            u.y = pack_bf16(x[8 * cc + 2], x[8 * cc + 3]);
                            u.z = pack_bf16(x[8 * cc + 4], x[8 * cc + 5]);
                            u.w = pack_bf16(x[8 * cc + 6], x[8 * cc + 7]);
                            *reinterpret_cast<uint4*>(prow + ((chunk ^ (row & 7)) << 4)) = u;
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(&bars.s_free[sbuf]);
                    sbuf ^= 1;
                    fence_proxy_async();
                    mbar_arrive(&bars.p_full);
                }
                if (!ok) break;
                // ---- output rows of block rb: O + xi C
                if (!wait(&bars.o_full, o_cnt & 1)) break;
                if (!wait(&bars.c_full, o_cnt & 1)) break;
                ++o_cnt;
                tc_fence_after();
                const float xi = exp2f(l2g * (float)(128 * rb + row + 1));
                const size_t orow = (size_t)bh * N + (size_t)i * B + 128 * rb + row;
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    float o[32], c[32];
                    tmem_ld32(tmem + lrow + kTO + c0, o);
                    tmem_ld32(tmem + lrow + kTC + c0, c);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = fmaf(xi, c[j], o[j]);
                    if (OUT_BF16) {
                        uint4* dst = reinterpret_cast<uint4*>(
                            static_cast<__nv_bfloat16*>(out) + orow * dv + blk * 64 + c0);
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc)
                            dst[cc] = make_uint4(pack_bf16(o[8 * cc], o[8 * cc + 1]),
                                                 pack_bf16(o[8 * cc + 2], o[8 * cc + 3]),
                                                 pack_bf16(o[8 * cc + 4], o[8 * cc + 5]),
                                                 pack_bf16(o[8 * cc + 6], o[8 * cc + 7]));
                    } else {
                        float4* dst = reinterpret_cast<float4*>(
                            static_cast<float*>(out) + orow * dv + blk * 64 + c0);
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc)
                            dst[cc] = make_float4(o[4 * cc], o[4 * cc + 1], o[4 * cc + 2], o[4 * cc + 3]);
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars.o_free);
                mbar_arrive(&bars.c_free);
            }
        }
        // ---- final state
        if (ok && state_out) {
            if (wait(&bars.r_done, rdone & 1)) {
                ++rdone;
                tc_fence_after();
                for (int hh = 0; hh < nh; ++hh) {
                    const int a = 128 * hh + row;
                    for (int c0 = 0; c0 < 64; c0 += 32) {
                        float x[32];
                        tmem_ld32(tmem + lrow + kTR + 64 * hh + c0, x);
                        tmem_wait_ld();
                        float4* dst = reinterpret_cast<float4*>(
                            state_out + ((size_t)bh * dk + a) * dv + blk * 64 + c0);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
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

cudaError_t launch_chunkwise_tc(const void* q, const void* k, const void* v, void* o,
                                int out_bf16, int b, int H, int N, int dk, int dv, int chunk,
                                const HeadConsts& hc, const float* state_in, float* state_out,
                                cudaStream_t s) {
    if (!(dk == 128 || dk == 256) || dv % 64 != 0 || !(chunk == 128 || chunk == 256))
        return cudaErrorNotSupported;
    Decay dc;
    for (int h = 0; h < H; ++h) {
        // folded decay factors need g^127 >= 2^-64; g = 0 goes elsewhere too
        if (!(hc.l2g[h] >= -0.5f)) return cudaErrorNotSupported;
        dc.l2g[h] = hc.l2g[h];
        dc.g128[h] = hc.g128[h];
    }
    const long long rows = (long long)b * H * N;
    if (rows >= (1LL << 31)) return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv;
    if (!make_map_bf16(&mq, q, rows, dk, 128) || !make_map_bf16(&mk, k, rows, dk, 128) ||
        !make_map_bf16(&mv, v, rows, dv, 128))
        return cudaErrorInvalidValue;
    const long long grid = (long long)b * H * (dv / 64);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int smem = kSmemBytes + 1024;
    auto kern = out_bf16 ? chunkwise_tc_kernel<true> : chunkwise_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, kThreads, smem, s>>>(mq, mk, mv, o, state_in, state_out, N, chunk, H,
                                               dk, dv, dc);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launch(RET_KERNEL_CHUNKWISE_TC);
    return e;
}

unsigned read_clear_error_tc_chunkwise(cudaStream_t s) {
    unsigned h = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_err_chunkwise, sizeof(h), 0, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_err_chunkwise, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return h;
}

}  // namespace ret
