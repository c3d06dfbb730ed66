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
// are independent (R = K^T V and q R both separate over dv), so each CTA keeps
// R[:, 64 cols] in tensor memory for the whole sequence and scans the chunks in
// order.  The intra-chunk score tile Q K^T does not depend on dv and is
// recomputed by each of the dv/64 CTAs of a head (their Q/K tiles hit in L2).
//
// Decay folding (no per-element power anywhere):
//   * V rows are scaled in shared memory by zeta_r = g^(B-1-r):  Vz = zeta (.) V.
//   * Then sum_{r<=j} S_jr g^(j-r) v_r = g^(j+1) * g^(-B) * sum_{r<=j} S_jr Vz_r, so the
//     score tile only needs the causal mask and one constant: P = g^(-B) (S (.) M).
//   * The cross-chunk read shares the row factor g^(j+1) = xi_j, so one fp32
//     accumulator per row block collects  P Vz + Q R_{i-1}  and the epilogue
//     multiplies each row by xi_j.
//   * The state update is R <- g^B R (one TMEM pass per chunk), then R += K^T Vz.
//   The folded factors stay in range when g^(-B) <= 2^64; smaller decays go to
//   the CUDA-core kernel.
// Precision: both low-precision operands that carry accumulated quantities are
// split into two bf16 parts, x = hi + lo with hi = bf16(x), lo = bf16(x - hi),
// each part feeding its own MMA into the same fp32 accumulator: the state copy
// (q R = q R_hi + q R_lo) and the scores (P Vz = P_hi Vz + P_lo Vz).  A single
// bf16 copy of either kept the error of the long-sequence workload at the 2e-2
// tolerance instead of well inside it.
//
// Roles (320 threads): warp 0 issues TMA loads (plus L2 prefetches one chunk
// ahead), warp 1 owns tensor memory and issues tcgen05.mma, warps 2-5 turn
// scores into P, warps 6-9 copy and rescale the state, scale V and write the
// outputs.  In each group, warp w reaches TMEM lanes 32*(w%4)..+31 (rows).  Every
// wait is bounded; a wait that gives up sets the device error word and the CTA
// unwinds.
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [  0,128) R: state, dk rows 0-127 (cols 0-63) and 128-255 (cols 64-127)
//   [128,256) O: two 64-column accumulators (row blocks of a 256-chunk, or
//             alternating chunks when B = 128)
//   [256,512) S: two 128-column score buffers.  P is written in place as bf16 pairs,
//             per 32 keys (32 columns of S): hi pairs in the first 16 columns, lo
//             pairs in the next 16; the P.V MMAs read it as their A operand.
// Shared memory (1024-aligned, 224 KB): 4 ring stages x 32 KB (one piece = 128 rows
//   x 128 columns of Q or K, two 64-column 128B-swizzled atoms), 2 x 16 KB scaled V
//   blocks, 2 x 32 KB bf16 hi/lo copies of R_{i-1} (B operand of q R).
//
// MMA order inside a 256-chunk (row blocks 0/1, key blocks 0/1), chosen so that a
// ring piece is released as early as possible and every TMA load or transform it
// waits for is covered by about 1500 cycles of other tensor work:
//   S00, Q0.R, P00.Vz0, K0^T Vz0, S10 (frees K0), Q1.R, P10.Vz0, S11 (frees Q1),
//   K1^T Vz1 (frees K1 per dk half), P11.Vz1.
// For B = 128: S00, Q0.R (frees Q0), K0^T Vz0 (frees K0 per dk half), P00.Vz0.
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
constexpr int kVzOff = kRingBytes;        // 2 x kAtom
constexpr int kRhiOff = kVzOff + 2 * kAtom;
constexpr int kRloOff = kRhiOff + 2 * kAtom;
constexpr int kSmemBytes = kRloOff + 2 * kAtom;   // 229376
constexpr int kThreads = 320;
constexpr int kGroupWarps = 4;

constexpr uint32_t kTR = 0, kTO = 128, kTS = 256;

struct Decay {
    float l2g[kMaxHeads];   // log2(gamma)
    float gB[kMaxHeads];    // gamma^B
    float cP[kMaxHeads];    // gamma^(-B)
};

struct Bars {
    uint64_t full[kStages], empty[kStages];
    uint64_t vfull[2], vempty[2], vz_ready[2];
    uint64_t s_full[2], p_ready[2], pv_done[2];
    uint64_t o_full[2], o_free[2];
    uint64_t rcopy, r_done;
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
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// hi/lo bf16 pairs of two values: hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16(x0, x1);
    lo = pack_bf16(x0 - bf16_lo(hi), x1 - bf16_hi(hi));
}

// Ring pieces of one chunk, in load order: for each row block rb, Q pieces
// (one per 128 dk columns) then K pieces.
__device__ __forceinline__ uint32_t piece_index(int which_k, int rb, int hh, int nh) {
    return (uint32_t)((2 * rb + which_k) * nh + hh);
}

template <int NH, int NRB, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
chunkwise_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, void* __restrict__ out,
                    const float* __restrict__ state_in, float* __restrict__ state_out, int N,
                    int B, int H, int dk, int dv, const Decay dc) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* ring = sm;
    uint8_t* vz = sm + kVzOff;
    uint8_t* rhi = sm + kRhiOff;
    uint8_t* rlo = sm + kRloOff;
    __shared__ Bars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nblk = dv / 64;
    const int bh = blockIdx.x / nblk, blk = blockIdx.x % nblk;
    const int head = bh % H;
    constexpr int nrb = NRB, nh = NH;
    const int nchunks = N / B;
    const uint32_t per_chunk = (uint32_t)(2 * nrb * nh);   // ring pieces per chunk
    volatile int* abort_p = &abort_flag;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < kStages; ++s) { mbar_init(&bars.full[s], 1); mbar_init(&bars.empty[s], 1); }
        for (int c = 0; c < 2; ++c) {
            mbar_init(&bars.vfull[c], 1); mbar_init(&bars.vempty[c], 1);
            mbar_init(&bars.vz_ready[c], kGroupWarps);
            mbar_init(&bars.s_full[c], 1); mbar_init(&bars.p_ready[c], kGroupWarps);
            mbar_init(&bars.pv_done[c], 1);
            mbar_init(&bars.o_full[c], 1); mbar_init(&bars.o_free[c], kGroupWarps);
        }
        mbar_init(&bars.rcopy, kGroupWarps); mbar_init(&bars.r_done, 1);
        mbar_init(&bars.drain, 1);
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
            auto load_piece = [&](const CUtensorMap* m, int row0, int hh) {
                const int s = fill % kStages;
                if (!mbar_wait(&bars.empty[s], ((fill / kStages) & 1) ^ 1, abort_p)) return false;
                mbar_arrive_expect_tx(&bars.full[s], kStage);
                tma_load_2d(ring + s * kStage, m, hh * 128, row0, &bars.full[s]);
                tma_load_2d(ring + s * kStage + kAtom, m, hh * 128 + 64, row0, &bars.full[s]);
                ++fill;
                return true;
            };
            auto load_v = [&](int vb, int row0) {
                if (!mbar_wait(&bars.vempty[vb], (vuse[vb] & 1) ^ 1, abort_p)) return false;
                mbar_arrive_expect_tx(&bars.vfull[vb], kAtom);
                tma_load_2d(vz + vb * kAtom, &mv, blk * 64, row0, &bars.vfull[vb]);
                ++vuse[vb];
                return true;
            };
            // the CTAs of one head share Q/K: each prefetches every nblk-th box of the
            // next chunk into L2, and its own V block
            auto prefetch_chunk = [&](int i) {
                if (i >= nchunks) return;
                const int rowc = bh * N + i * B;
                int box = 0;
                for (int rb = 0; rb < nrb; ++rb)
                    for (int which = 0; which < 2; ++which)
                        for (int c = 0; c < dk; c += 64, ++box)
                            if (box % nblk == blk)
                                tma_prefetch_l2(which ? &mk : &mq, c, rowc + 128 * rb);
                for (int rb = 0; rb < nrb; ++rb) tma_prefetch_l2(&mv, blk * 64, rowc + 128 * rb);
            };
            prefetch_chunk(0);
            for (int i = 0; i < nchunks && ok; ++i) {
                prefetch_chunk(i + 1);
                const int rowc = bh * N + i * B;
                for (int rb = 0; rb < nrb && ok; ++rb) {
                    const int row0 = rowc + 128 * rb;
                    for (int hh = 0; hh < nh && ok; ++hh) ok = load_piece(&mq, row0, hh);
                    for (int hh = 0; hh < nh && ok; ++hh) ok = load_piece(&mk, row0, hh);
                    if (ok) ok = load_v(nrb == 1 ? (i & 1) : rb, row0);
                }
            }
            if (!ok) {
                fail(abort_p);
                // let loads already in flight land before the CTA unwinds
                for (uint32_t f = fill > kStages ? fill - kStages : 0; f < fill; ++f)
                    mbar_wait(&bars.full[f % kStages], (f / kStages) & 1, nullptr, 100000000ull);
                for (int c = 0; c < 2; ++c)
                    if (vuse[c]) mbar_wait(&bars.vfull[c], (vuse[c] - 1) & 1, nullptr, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, 128, 0, 0);   // Q K^T: both K-major
            const uint32_t id_q = idesc_bf16(128, 64, 0, 1);    // Q R: B (state) MN-major
            const uint32_t id_p = idesc_bf16(128, 64, 0, 1);    // P Vz: A in TMEM, B MN-major
            const uint32_t id_r = idesc_bf16(128, 64, 1, 1);    // K^T Vz: both MN-major
            const uint32_t ring_a = smem_u32(ring), vz_a = smem_u32(vz);
            const uint32_t rhi_a = smem_u32(rhi), rlo_a = smem_u32(rlo);
            uint32_t s_use0 = 0, s_use1 = 0, pv_use0 = 0, pv_use1 = 0, o_use0 = 0, o_use1 = 0;
            bool ok = true;
            auto wait = [&](uint64_t* bar, uint32_t par) {
                if (ok && !mbar_wait(bar, par, abort_p)) { ok = false; fail(abort_p); }
                return ok;
            };
            // Descriptors are linear in the start-address field (address >> 4, low 14 bits),
            // so every operand descriptor is a base descriptor plus a byte offset / 16.
            const uint64_t dK = sdesc_sw128(ring_a, 16, 1024);      // K-major, ring base
            const uint64_t dMN = sdesc_sw128(ring_a, kAtom, 1024);  // MN-major, ring base
            const uint64_t dVz = sdesc_sw128(vz_a, kAtom, 1024);
            const uint64_t dRhi = sdesc_sw128(rhi_a, kAtom, 1024);
            const uint64_t dRlo = sdesc_sw128(rlo_a, kAtom, 1024);
            auto slot_off = [&](uint32_t f) { return (uint64_t)(((f % kStages) * kStage) >> 4); };
            auto wait_piece = [&](uint32_t f) { return wait(&bars.full[f % kStages], (f / kStages) & 1); };
            auto release_piece = [&](uint32_t f) { mma_commit(&bars.empty[f % kStages]); };
            // S(sb) = Q_rb K_cb^T  (M=128, N=128, K=dk), waiting for each dk half's pieces
            // just before its k-steps.
            auto mma_s = [&](uint32_t base, int rb, int cb, int sb) {
                uint32_t& su = sb ? s_use1 : s_use0;
                // the buffer's previous P.V (issued earlier by this thread) reads it before
                // this MMA writes it: tcgen05.mma operations of one thread run in issue order
                const uint32_t ts = tmem + kTS + 128 * sb;
                for (int hh = 0; hh < nh && ok; ++hh) {
                    wait_piece(base + piece_index(0, rb, hh, nh));
                    wait_piece(base + piece_index(1, cb, hh, nh));
                    if (!ok) return;
                    tc_fence_after();
                    const uint64_t da = dK + slot_off(base + piece_index(0, rb, hh, nh));
                    const uint64_t db = dK + slot_off(base + piece_index(1, cb, hh, nh));
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t off = (uint64_t)((((kk * 16) / 64) * kAtom + ((kk * 16) % 64) * 2) >> 4);
                        mma_bf16(ts, da + off, db + off, id_s, (hh | kk) != 0);
                    }
                }
                mma_commit(&bars.s_full[sb]);
                ++su;
            };
            // O_acc(ob) = Q_rb (R_hi + R_lo); the first MMA overwrites the accumulator.
            auto mma_qr = [&](uint32_t base, int rb, int ob) {
                uint32_t& ou = ob ? o_use1 : o_use0;
                if (ou > 0) wait(&bars.o_free[ob], (ou - 1) & 1);
                if (!ok) return;
                tc_fence_after();
                const uint32_t to = tmem + kTO + 64 * ob;
#pragma unroll 1
                for (int hh = 0; hh < nh; ++hh) {
                    const uint64_t da = dK + slot_off(base + piece_index(0, rb, hh, nh));
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = da + (uint64_t)((((kk * 16) / 64) * kAtom + ((kk * 16) % 64) * 2) >> 4);
                        const uint64_t rof = (uint64_t)(hh * ((128 * 128) >> 4) + ((16 * kk * 128) >> 4));
                        mma_bf16(to, ad, dRhi + rof, id_q, (hh | kk) != 0);
                        mma_bf16(to, ad, dRlo + rof, id_q, 1);
                    }
                }
                ++ou;
            };
            // O_acc(ob) += (P_hi + P_lo)(sb) Vz_vb  (M=128, N=64, K=128 keys; A from TMEM)
            auto mma_pv = [&](int sb, int vb, int ob) {
                uint32_t& pu = sb ? pv_use1 : pv_use0;
                if (!wait(&bars.p_ready[sb], pu & 1)) return;
                tc_fence_after();
                const uint32_t ts = tmem + kTS + 128 * sb;
                const uint64_t dv0 = dVz + (uint64_t)((vb * kAtom) >> 4);
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const uint32_t a_hi = ts + 32 * (t / 2) + 8 * (t % 2);
                    const uint64_t bd = dv0 + (uint64_t)((16 * t * 128) >> 4);
                    mma_ts(tmem + kTO + 64 * ob, a_hi, bd, id_p, 1);
                    mma_ts(tmem + kTO + 64 * ob, a_hi + 16, bd, id_p, 1);
                }
                mma_commit(&bars.pv_done[sb]);
                ++pu;
            };
            // R += K_cb^T Vz_vb  (M=128 per dk half, N=64, K=128 keys), releasing each K
            // piece as soon as its half is issued when `release` is set.
            auto mma_kv = [&](uint32_t base, int cb, int vb, bool release) {
                tc_fence_after();
                const uint64_t dv0 = dVz + (uint64_t)((vb * kAtom) >> 4);
#pragma unroll 1
                for (int hh = 0; hh < nh; ++hh) {
                    const uint32_t f = base + piece_index(1, cb, hh, nh);
                    const uint64_t da = dMN + slot_off(f);
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const uint64_t off = (uint64_t)((16 * t * 128) >> 4);
                        mma_bf16(tmem + kTR + 64 * hh, da + off, dv0 + off, id_r, 1);
                    }
                    if (release) release_piece(f);
                }
            };
            auto release_q = [&](uint32_t base, int rb) {
                for (int hh = 0; hh < nh; ++hh) release_piece(base + piece_index(0, rb, hh, nh));
            };
            auto release_k = [&](uint32_t base, int cb) {
                for (int hh = 0; hh < nh; ++hh) release_piece(base + piece_index(1, cb, hh, nh));
            };
            for (int i = 0; i < nchunks && ok; ++i) {
                const uint32_t base = (uint32_t)i * per_chunk;
                if (nrb == 1) {
                    const int sb = i & 1, ob = i & 1, vb = i & 1;
                    mma_s(base, 0, 0, sb);
                    wait(&bars.rcopy, i & 1);                    // R_{i-1} copied, R scaled
                    mma_qr(base, 0, ob);
                    release_q(base, 0);
                    wait(&bars.vz_ready[vb], (i >> 1) & 1);
                    if (!ok) break;
                    mma_kv(base, 0, vb, true);
                    mma_commit(&bars.r_done);
                    mma_pv(sb, vb, ob);
                    mma_commit(&bars.o_full[ob]);
                    mma_commit(&bars.vempty[vb]);
                } else {
                    const int sa = i & 1, sbb = sa ^ 1;
                    mma_s(base, 0, 0, sa);                         // S00
                    wait(&bars.rcopy, i & 1);
                    mma_qr(base, 0, 0);                            // O0 = Q0 R
                    release_q(base, 0);
                    wait(&bars.vz_ready[0], i & 1);
                    mma_pv(sa, 0, 0);                              // O0 += P00 Vz0
                    mma_commit(&bars.o_full[0]);
                    if (!ok) break;
                    mma_kv(base, 0, 0, false);                     // R += K0^T Vz0
                    mma_s(base, 1, 0, sbb);                        // S10
                    release_k(base, 0);
                    mma_qr(base, 1, 1);                            // O1 = Q1 R
                    mma_pv(sbb, 0, 1);                             // O1 += P10 Vz0
                    mma_commit(&bars.vempty[0]);
                    mma_s(base, 1, 1, sa);                         // S11 (after P00 read)
                    release_q(base, 1);
                    wait(&bars.vz_ready[1], i & 1);
                    if (!ok) break;
                    mma_kv(base, 1, 1, true);                      // R += K1^T Vz1
                    mma_commit(&bars.r_done);
                    mma_pv(sa, 1, 1);                              // O1 += P11 Vz1
                    mma_commit(&bars.o_full[1]);
                    mma_commit(&bars.vempty[1]);
                }
            }
            // every issued MMA must finish before tensor memory is released
            mma_commit(&bars.drain);
            mbar_wait(&bars.drain, 0, nullptr, 200000000ull);
        }
    } else {
        // ------------------------------------------------------------ transform warps
        const bool pwarp = warp < 6;                 // warps 2-5: scores; 6-9: state/V/out
        const int q4 = warp & 3;                     // TMEM lane quarter of this warp
        const int row = 32 * q4 + lane;              // TMEM lane = tile row
        const uint32_t lrow = (uint32_t)(32 * q4) << 16;
        const float l2g = dc.l2g[head];
        const float gB = dc.gB[head];
        const float cP = dc.cP[head];
        bool ok = true;
        // tcgen05.ld/st are warp-collective: keep the outcome of every wait uniform
        auto wait = [&](uint64_t* bar, uint32_t par) {
            if (!ok) return false;
            const bool got = __all_sync(0xffffffffu, mbar_wait(bar, par, abort_p));
            if (!got) { ok = false; if (lane == 0) fail(abort_p); }
            return ok;
        };
        auto arrive = [&](uint64_t* bar) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        };
        if (pwarp) {
            uint32_t s_cnt0 = 0, s_cnt1 = 0;
            // P = g^(-B) S, causal mask on diagonal tiles, as hi/lo bf16 pairs in place.
            auto do_p = [&](int sb, bool diag) {
                uint32_t& sc = sb ? s_cnt1 : s_cnt0;
                if (!wait(&bars.s_full[sb], sc & 1)) return;
                ++sc;
                tc_fence_after();
                const uint32_t ts = tmem + lrow + kTS + 128 * sb;
                // quarter qq of the keys (32 columns of S) becomes 16 hi and 16 lo columns
                // in the same 32 columns: read all of it before writing any of it
#pragma unroll 1
                for (int qq = 0; qq < 4; ++qq) {
                    float x[32];
                    tmem_ld32(ts + 32 * qq, x);
                    tmem_wait_ld();
                    uint32_t pp[32];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int kc = 32 * qq + 2 * e;
                        float x0 = x[2 * e] * cP, x1 = x[2 * e + 1] * cP;
                        if (diag) {
                            if (kc > row) x0 = 0.f;
                            if (kc + 1 > row) x1 = 0.f;
                        }
                        split2(x0, x1, pp[e], pp[16 + e]);
                    }
                    tmem_st32(ts + 32 * qq, reinterpret_cast<const float*>(pp));
                }
                tmem_wait_st();
                tc_fence_before();
                arrive(&bars.p_ready[sb]);
            };
            for (int i = 0; i < nchunks && ok; ++i) {
                if (nrb == 1) {
                    do_p(i & 1, true);
                } else {
                    const int sa = i & 1, sbb = sa ^ 1;
                    do_p(sa, true);                       // P00
                    do_p(sbb, false);                     // P10
                    do_p(sa, true);                       // P11
                }
            }
        } else {
            uint32_t o_cnt0 = 0, o_cnt1 = 0;
            // state: hi/lo bf16 copies of R_{i-1} for q R, then R <- g^B R in TMEM.
            auto do_state = [&](int i) {
                if (i > 0) {
                    if (!wait(&bars.r_done, (i - 1) & 1)) return;
                    tc_fence_after();
                }
                for (int hh = 0; hh < nh; ++hh) {
                    const int a = 128 * hh + row;          // dk row
#pragma unroll 1
                    for (int c0 = 0; c0 < 64; c0 += 32) {
                        const uint32_t tcol = tmem + lrow + kTR + 64 * hh + c0;
                        float x[32];
                        if (i == 0) {
                            if (state_in) {
                                const float4* src = reinterpret_cast<const float4*>(
                                    state_in + ((size_t)bh * dk + a) * dv + blk * 64 + c0);
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    const float4 f = src[j];
                                    x[4 * j] = f.x; x[4 * j + 1] = f.y; x[4 * j + 2] = f.z; x[4 * j + 3] = f.w;
                                }
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j) x[j] = 0.f;
                            }
                        } else {
                            tmem_ld32(tcol, x);
                            tmem_wait_ld();
                        }
                        // 32 values = 4 chunks of 8 bf16 in the 128B-swizzled row a
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            uint32_t h[4], l[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                split2(x[8 * cc + 2 * e], x[8 * cc + 2 * e + 1], h[e], l[e]);
                            const uint32_t off = a * 128 + ((((uint32_t)(c0 / 8 + cc)) ^ (a & 7)) << 4);
                            *reinterpret_cast<uint4*>(rhi + off) = make_uint4(h[0], h[1], h[2], h[3]);
                            *reinterpret_cast<uint4*>(rlo + off) = make_uint4(l[0], l[1], l[2], l[3]);
                        }
#pragma unroll
                        for (int j = 0; j < 32; ++j) x[j] *= gB;
                        tmem_st32(tcol, x);
                    }
                }
                tmem_wait_st();
                fence_proxy_async();
                tc_fence_before();
                arrive(&bars.rcopy);
            };
            // V block vb (keys 128*cb.. of chunk i): key row kr scaled by g^(B-1-(128 cb + kr)).
            auto do_v = [&](int vb, uint32_t phase, int cb) {
                if (!wait(&bars.vfull[vb], phase)) return;
                const float f = exp2f(l2g * (float)(B - 1 - (128 * cb + row)));
                uint8_t* vrow = vz + vb * kAtom + row * 128;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    uint4* p = reinterpret_cast<uint4*>(vrow + (((uint32_t)cc ^ (row & 7)) << 4));
                    uint4 u = *p;
                    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) w[e] = pack_bf16(bf16_lo(w[e]) * f, bf16_hi(w[e]) * f);
                    *p = make_uint4(w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async();
                arrive(&bars.vz_ready[vb]);
            };
            // output rows of one accumulator: xi_j * O_acc, j = 128 rb + row
            auto do_out = [&](int i, int rb, int ob) {
                uint32_t& oc = ob ? o_cnt1 : o_cnt0;
                if (!wait(&bars.o_full[ob], oc & 1)) return;
                ++oc;
                tc_fence_after();
                const float xi = exp2f(l2g * (float)(128 * rb + row + 1));
                float o[64];
                tmem_ld32(tmem + lrow + kTO + 64 * ob, o);
                tmem_ld32(tmem + lrow + kTO + 64 * ob + 32, o + 32);
                tmem_wait_ld();
                tc_fence_before();
                arrive(&bars.o_free[ob]);
                const size_t orow = (size_t)bh * N + (size_t)i * B + 128 * rb + row;
                const size_t col = (size_t)blk * 64;
                if (OUT_BF16) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + orow * dv + col);
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc)
                        dst[cc] = make_uint4(pack_bf16(xi * o[8 * cc], xi * o[8 * cc + 1]),
                                             pack_bf16(xi * o[8 * cc + 2], xi * o[8 * cc + 3]),
                                             pack_bf16(xi * o[8 * cc + 4], xi * o[8 * cc + 5]),
                                             pack_bf16(xi * o[8 * cc + 6], xi * o[8 * cc + 7]));
                } else {
                    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + orow * dv + col);
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc)
                        dst[cc] = make_float4(xi * o[4 * cc], xi * o[4 * cc + 1], xi * o[4 * cc + 2],
                                              xi * o[4 * cc + 3]);
                }
            };
            for (int i = 0; i < nchunks && ok; ++i) {
                do_state(i);
                if (nrb == 1) {
                    do_v(i & 1, (i >> 1) & 1, 0);
                    if (i > 0) do_out(i - 1, 0, (i - 1) & 1);
                } else {
                    do_v(0, i & 1, 0);
                    if (i > 0) do_out(i - 1, 1, 1);
                    do_v(1, i & 1, 1);
                    do_out(i, 0, 0);
                }
            }
            if (ok && nchunks > 0) {
                if (nrb == 1) do_out(nchunks - 1, 0, (nchunks - 1) & 1);
                else do_out(nchunks - 1, 1, 1);
            }
            // ---- final state R_{N/B-1}
            if (ok && state_out && nchunks > 0) {
                if (wait(&bars.r_done, (nchunks - 1) & 1)) {
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
        // folded factors: g^(-B) must stay <= 2^64 (g = 0 goes elsewhere too)
        if (!(hc.l2g[h] * (float)chunk >= -64.0f)) return cudaErrorNotSupported;
        dc.l2g[h] = hc.l2g[h];
        dc.gB[h] = hc.gB[h];
        dc.cP[h] = hc.ginvB[h];
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
    void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, void*, const float*,
                 float*, int, int, int, int, int, const Decay);
    const int sel = (dk == 256 ? 4 : 0) + (chunk == 256 ? 2 : 0) + (out_bf16 ? 1 : 0);
    switch (sel) {
        case 0: kern = chunkwise_tc_kernel<1, 1, false>; break;
        case 1: kern = chunkwise_tc_kernel<1, 1, true>; break;
        case 2: kern = chunkwise_tc_kernel<1, 2, false>; break;
        case 3: kern = chunkwise_tc_kernel<1, 2, true>; break;
        case 4: kern = chunkwise_tc_kernel<2, 1, false>; break;
        case 5: kern = chunkwise_tc_kernel<2, 1, true>; break;
        case 6: kern = chunkwise_tc_kernel<2, 2, false>; break;
        default: kern = chunkwise_tc_kernel<2, 2, true>; break;
    }
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
