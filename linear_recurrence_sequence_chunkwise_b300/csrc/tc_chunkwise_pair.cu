// tc_chunkwise_pair.cu -- chunkwise recurrent retention on pairs of SMs (tcgen05 cta_group::2).
//
// Computes eq.(7) of "Transformer取代者登場！…RetNet…（2）", section "Retention" 3), the same
// function as tc_chunkwise.cu:
//     O[iB+j] = sum_{r<=j} (q_j.k_r) g^(j-r) v_r + g^(j+1) (q_j R_{i-1})
//     R_i     = sum_r g^(B-1-r) k_r^T v_r + g^B R_{i-1}
// for bf16 Q/K/V, fp32 accumulation and state, chunk B = 256, dk = 256, dv a multiple of
// 128.  Decay folding and the hi/lo bf16 split of the state copy and of the scores are
// those of tc_chunkwise.cu (Vz = zeta (.) V, P = g^(-B) S (.) M, xi_j applied to the
// output rows, R <- g^B R then R += K^T Vz).
//
// Work split: one cluster of two CTAs (the two SMs of a pair) per (batch*head, 128-column
// block of dv); the even CTA issues every MMA as a pair MMA (M = 256, 128 rows per SM):
//   S  = Q K^T        M = 256 query rows of the chunk (CTA r: rows 128r..), N = 256 keys
//                     (B operand split: CTA r holds keys 128r..), K = dk
//   O  = Q R_{i-1}    N = 128 value columns (B split: CTA r holds the bf16 hi/lo copy of
//                     R[:, 64r..64r+63]), K = dk, as two MMAs (hi, lo)
//   R += K^T Vz       M = 256 dk rows (CTA r: dk 128r..; the state lives in tensor memory,
//                     split by dk), N = 128 value columns, K = 256 keys
//   O += P Vz         A = P from tensor memory (hi and lo), N = 128, K = 256 keys
// Every MMA has N >= 128 per SM, and each SM reads only its half of each B operand, so
// the tensor pipe runs at full rate with half the shared-memory operand traffic of the
// one-SM split into 64-column blocks, and the score tile of a head is computed by dv/128
// pairs instead of dv/64 CTAs.  The pair costs one duplicated quarter of the score tile
// (the even CTA's rows against keys 128-255, all masked) and of P.V.
//
// Roles (576 threads = 18 warps per CTA).  The transform work of a chunk is spread over
// sixteen warps in two groups that run side by side, so that no group has more than one
// task on the path between two MMAs:
//   warp 0      TMA loads of this CTA (Q, K and the K^T operand complete on the even CTA's
//               barriers, V on a local one) and L2 prefetches one chunk ahead
//   warp 1      tensor-memory allocation (both CTAs, collectively); in the even CTA the
//               MMA issuer
//   warps 2-9   scores -> P (two warps per TMEM lane quarter, one per 128-key half), then
//               the chunk's output rows (one per 64-column half), coalesced stores
//   warps 10-17 state copy (two warps per lane quarter: this CTA's own 64 value columns
//               into its own shared memory, the peer's 64 into the peer's, 64-byte row
//               pieces), the rescale
//               R <- g^B R, then V -> Vz (one key row per thread)
// Warp w reaches TMEM lanes 32*(w%4)..+31.  Every wait is bounded; a wait that gives up
// sets the device error word and both CTAs' abort flags, and the CTAs unwind, meet at a
// final cluster barrier and free their tensor memory.
//
// Tensor memory per CTA (512 columns x 128 lanes, fp32):
//   [  0,256) S: this CTA's 128 query rows x 256 keys; P written in place as bf16 pairs
//             (per 32 keys: 16 columns of hi pairs, then 16 of lo pairs)
//   [256,384) O: this CTA's 128 query rows x 128 value columns
//   [384,512) R: this CTA's 128 dk rows of the state x 128 value columns
// Shared memory per CTA (1024-aligned, 224 KB), each box 128 rows x 64 bf16, 128B swizzle:
//   Q   64 KB  own 128 query rows x 4 dk boxes
//   K   64 KB  own 128 keys x 4 dk boxes (S); after S the K^T operand of the state update:
//              key block j (keys 128j..) x own 128 dk columns in boxes 2j, 2j+1.  The own
//              key block's boxes stay from S; the peer key block is loaded into the two
//              boxes S no longer needs (the same offsets in both CTAs)
//   V   32 KB  256 keys x own 64 value columns (scaled in place to Vz)
//   Rhi 32 KB, Rlo 32 KB  bf16 copy of R_{i-1}: 256 dk rows x own 64 columns
// MMA order in a chunk: S (dk boxes 0-1, then 2-3), Q.R, K^T.Vz (key block 0, then 1),
// P.Vz.  Commits between the halves free shared memory early: after S's first half the
// odd CTA loads its peer key block (boxes 0-1), after its second half the even CTA
// (boxes 2-3); after K^T.Vz's first half the next chunk's keys load into boxes 0-1.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace ret {
namespace {

__device__ unsigned g_err_chunkwise_pair;

using namespace tc;

constexpr int kThreads = 576;
constexpr int kB = 256;                        // chunk length
constexpr int kDk = 256;
constexpr int kBox = 128 * 128;                // 128 rows x 64 bf16
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + 4 * kBox;
constexpr int kVOff = kKOff + 4 * kBox;
constexpr int kRhiOff = kVOff + 2 * kBox;
constexpr int kRloOff = kRhiOff + 2 * kBox;
constexpr int kSmemBytes = kRloOff + 2 * kBox;  // 229376
constexpr uint32_t kTS = 0, kTO = 256, kTR = 384;
constexpr uint32_t kPairArrivals = 16;         // 8 warps in each CTA
constexpr uint16_t kBoth = 3;                  // multicast mask: both CTAs of the pair
constexpr int kFirstP = 2, kFirstR = 10;       // first warp of each transform group

struct Decay {
    float l2g[kMaxHeads];   // log2(gamma)
    float gB[kMaxHeads];    // gamma^B
    float cP[kMaxHeads];    // gamma^(-B)
};

struct Bars {
    // the even CTA's copies count both CTAs' work
    uint64_t q_full, k_full0, k_full1;             // pair loads: Q; K dk boxes 0-1 / 2-3
    uint64_t kt_full0, kt_full1;                   // peer key block of K^T in boxes 0-1 / 2-3
    uint64_t vz_ready, p_ready, rcopy, o_free;     // warp arrivals of both CTAs

    // each CTA's own copy, arrived on by the MMA commits (multicast)
    uint64_t q_empty;                              // Q.R done: Q area free
    uint64_t s_half, s_full;                       // S done with dk boxes 0-1 / all of S
    uint64_t kt_empty0, kt_empty1;                 // K^T.Vz done with boxes 0-1 / 2-3
    uint64_t v_empty, o_full, r_done;              // P.Vz done (V free, O complete); K^T.Vz done
    uint64_t v_full;                               // local V load
    uint64_t drain;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16(x0, x1);
    lo = pack_bf16(x0 - bf16_lo(hi), x1 - bf16_hi(hi));
}

template <bool OUT_BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
chunkwise_pair_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                      const __grid_constant__ CUtensorMap mv,
                      void* __restrict__ out_base, const float* __restrict__ state_in,
                      float* __restrict__ state_out, int N,
                      int H, int dv, const Decay dc) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sq = sm + kQOff;
    uint8_t* sk = sm + kKOff;
    uint8_t* sv = sm + kVOff;
    uint8_t* rhi = sm + kRhiOff;
    uint8_t* rlo = sm + kRloOff;
    __shared__ Bars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int nblk = dv / 128;
    const int pair = (int)(blockIdx.x >> 1);
    const int bh = pair / nblk, blk = pair % nblk;
    const int head = bh % H;
    const int nchunks = N / kB;
    volatile int* abort_p = &abort_flag;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bars.q_full, 1); mbar_init(&bars.k_full0, 1); mbar_init(&bars.k_full1, 1);
        mbar_init(&bars.kt_full0, 1); mbar_init(&bars.kt_full1, 1);
        mbar_init(&bars.vz_ready, kPairArrivals); mbar_init(&bars.p_ready, kPairArrivals);
        mbar_init(&bars.rcopy, kPairArrivals); mbar_init(&bars.o_free, kPairArrivals);
        mbar_init(&bars.q_empty, 1); mbar_init(&bars.s_half, 1); mbar_init(&bars.s_full, 1);
        mbar_init(&bars.kt_empty0, 1); mbar_init(&bars.kt_empty1, 1);
        mbar_init(&bars.v_empty, 1); mbar_init(&bars.o_full, 1); mbar_init(&bars.r_done, 1);
        mbar_init(&bars.v_full, 1); mbar_init(&bars.drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) { tmem_alloc_pair(&tmem_slot, 512); tmem_relinquish_pair(); }
    tc_fence_before();
    cluster_sync_all();     // both CTAs' barriers exist before any remote arrive or pair load
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t peer_abort = map_peer(&abort_flag, peer);
    auto fail = [&]() {
        *abort_p = 1;
        st_cluster_s32(peer_abort, 1);
        atomicOr(&g_err_chunkwise_pair, 1u);
    };
    auto lead = [&](uint64_t* b) { return map_peer(b, 0); };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&mq); tma_prefetch_desc(&mk); tma_prefetch_desc(&mv);
            const uint32_t qf = lead(&bars.q_full), kf0 = lead(&bars.k_full0),
                           kf1 = lead(&bars.k_full1);
            const uint32_t ktf = lead(rank == 0 ? &bars.kt_full1 : &bars.kt_full0);
            const int rowbase = bh * N;
            const int own = 128 * (int)rank, other = 128 * (int)peer;
            const int vcol = blk * 128 + 64 * (int)rank;
            uint32_t armed_q = 0, armed_k = 0, armed_kt = 0, v_loads = 0;
            bool ok = true;
            auto w = [&](uint64_t* bar, uint32_t par) {
                if (ok && !mbar_wait(bar, par, abort_p)) { ok = false; fail(); }
                return ok;
            };
            // the pairs of one head share Q and K: pull the next chunk's boxes into L2
            auto prefetch = [&](int c) {
                if (c >= nchunks) return;
                const int r0 = rowbase + c * kB;
                for (int a = 0; a < 4; ++a) {
                    tma_prefetch_l2(&mq, 64 * a, r0 + own);
                    tma_prefetch_l2(&mk, 64 * a, r0 + own);
                }
                for (int m = 0; m < 2; ++m) tma_prefetch_l2(&mk, 64 * (2 * (int)rank + m), r0 + other);
                for (int j = 0; j < 2; ++j) tma_prefetch_l2(&mv, vcol, r0 + 128 * j);
            };
            prefetch(0);
            for (int c = 0; c < nchunks && ok; ++c) {
                const uint32_t pp = (uint32_t)(c - 1) & 1u;
                const int r0 = rowbase + c * kB;
                // Q: own query rows, all dk (after the previous chunk's Q.R)
                if (c > 0 && !w(&bars.q_empty, pp)) break;
                if (rank == 0) { mbar_arrive_expect_tx(&bars.q_full, 2 * 4 * kBox); ++armed_q; }
                for (int a = 0; a < 4; ++a) tma_load_2d_pair(sq + a * kBox, &mq, 64 * a, r0 + own, qf);
                // K: own keys; dk boxes 0-1 once K^T.Vz has read key block 0, boxes 2-3 once
                // it has read key block 1
                if (c > 0 && !w(&bars.kt_empty0, pp)) break;
                if (rank == 0) {
                    mbar_arrive_expect_tx(&bars.k_full0, 2 * 2 * kBox);
                    mbar_arrive_expect_tx(&bars.k_full1, 2 * 2 * kBox);
                    ++armed_k;
                }
                for (int a = 0; a < 2; ++a) tma_load_2d_pair(sk + a * kBox, &mk, 64 * a, r0 + own, kf0);
                if (c > 0 && !w(&bars.kt_empty1, pp)) break;
                for (int a = 2; a < 4; ++a) tma_load_2d_pair(sk + a * kBox, &mk, 64 * a, r0 + own, kf1);
                // V: all keys of the chunk, own 64 value columns (after the previous P.Vz)
                if (c > 0 && !w(&bars.v_empty, pp)) break;
                mbar_arrive_expect_tx(&bars.v_full, 2 * kBox);
                for (int j = 0; j < 2; ++j) tma_load_2d(sv + j * kBox, &mv, vcol, r0 + 128 * j, &bars.v_full);
                ++v_loads;
                // K^T operand of the state update: the peer key block x own dk half goes
                // into boxes 2*peer, 2*peer+1 once S has read them (the odd CTA's after S's
                // first half, the even CTA's after all of S)
                if (!w(rank == 1 ? &bars.s_half : &bars.s_full, (uint32_t)c & 1u)) break;
                if (rank == 0) {
                    mbar_arrive_expect_tx(&bars.kt_full0, 2 * kBox);
                    mbar_arrive_expect_tx(&bars.kt_full1, 2 * kBox);
                    ++armed_kt;
                }
                for (int m = 0; m < 2; ++m)
                    tma_load_2d_pair(sk + (2 * (int)peer + m) * kBox, &mk, 64 * (2 * (int)rank + m),
                                     r0 + other, ktf);
                // the next chunk's boxes into L2, behind this chunk's loads in the TMA queue
                prefetch(c + 1);
            }
            if (!ok) {
                // let loads in flight land before the CTAs unwind
                if (v_loads) mbar_wait(&bars.v_full, (v_loads - 1) & 1, nullptr, 100000000ull);
                if (rank == 0) {
                    if (armed_q) mbar_wait(&bars.q_full, (armed_q - 1) & 1, nullptr, 100000000ull);
                    if (armed_k) {
                        mbar_wait(&bars.k_full0, (armed_k - 1) & 1, nullptr, 100000000ull);
                        mbar_wait(&bars.k_full1, (armed_k - 1) & 1, nullptr, 100000000ull);
                    }
                    if (armed_kt) {
                        mbar_wait(&bars.kt_full0, (armed_kt - 1) & 1, nullptr, 100000000ull);
                        mbar_wait(&bars.kt_full1, (armed_kt - 1) & 1, nullptr, 100000000ull);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        if (rank == 0 && lane == 0) {
            const uint32_t id_s = idesc_bf16(256, 256, 0, 0);    // Q K^T: both K-major
            const uint32_t id_q = idesc_bf16(256, 128, 0, 1);    // Q R: B MN-major
            const uint32_t id_r = idesc_bf16(256, 128, 1, 1);    // K^T Vz: both MN-major
            const uint32_t id_p = idesc_bf16(256, 128, 0, 1);    // P Vz: A in TMEM, B MN-major
            // descriptors are linear in the start address: base descriptor + offset / 16
            const uint64_t dQ = sdesc_sw128(smem_u32(sq), 16, 1024);
            const uint64_t dK = sdesc_sw128(smem_u32(sk), 16, 1024);
            const uint64_t dKT = sdesc_sw128(smem_u32(sk), kBox, 1024);   // dk boxes 16 KB apart
            const uint64_t dV = sdesc_sw128(smem_u32(sv), 2 * kBox, 1024);
            const uint64_t dRhi = sdesc_sw128(smem_u32(rhi), 2 * kBox, 1024);
            const uint64_t dRlo = sdesc_sw128(smem_u32(rlo), 2 * kBox, 1024);
            bool ok = true;
            auto w = [&](uint64_t* bar, uint32_t par) {
                if (ok && !mbar_wait_cl(bar, par, abort_p)) { ok = false; fail(); }
                return ok;
            };
            auto s_boxes = [&](int a0) {
#pragma unroll 1
                for (int a = a0; a < a0 + 2; ++a)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t off = (uint64_t)((a * kBox + kk * 32) >> 4);
                        mma_pair(tmem + kTS, dQ + off, dK + off, id_s, (a | kk) != 0);
                    }
            };
            auto kv_block = [&](int j) {
#pragma unroll
                for (int t = 8 * j; t < 8 * j + 8; ++t) {
                    const uint64_t ka = (uint64_t)(((t >> 3) * 2 * kBox + (t & 7) * 2048) >> 4);
                    const uint64_t off = (uint64_t)((t * 2048) >> 4);
                    mma_pair(tmem + kTR, dKT + ka, dV + off, id_r, 1);
                }
            };
            for (int c = 0; c < nchunks && ok; ++c) {
                const uint32_t ph = (uint32_t)c & 1u;
                // S = Q K^T (the previous P.Vz, issued earlier, reads the S columns first:
                // tcgen05.mma operations of one thread run in issue order)
                if (!w(&bars.q_full, ph) || !w(&bars.k_full0, ph)) break;
                tc_fence_after();
                s_boxes(0);
                mma_commit_pair(&bars.s_half, kBoth);
                if (!w(&bars.k_full1, ph)) break;
                tc_fence_after();
                s_boxes(2);
                mma_commit_pair(&bars.s_full, kBoth);
                // O = Q (R_hi + R_lo); the first MMA overwrites the accumulator
                if (!w(&bars.rcopy, ph)) break;
                if (c > 0 && !w(&bars.o_free, (c - 1) & 1)) break;
                tc_fence_after();
#pragma unroll 1
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t qa = dQ + (uint64_t)((a * kBox + kk * 32) >> 4);
                        const uint64_t ro = (uint64_t)(((4 * a + kk) * 2048) >> 4);
                        mma_pair(tmem + kTO, qa, dRhi + ro, id_q, (a | kk) != 0);
                        mma_pair(tmem + kTO, qa, dRlo + ro, id_q, 1);
                    }
                mma_commit_pair(&bars.q_empty, kBoth);
                // R += K^T Vz (R was rescaled by g^B with the copy), key block 0 then 1
                if (!w(&bars.vz_ready, ph) || !w(&bars.kt_full0, ph)) break;
                tc_fence_after();
                kv_block(0);
                mma_commit_pair(&bars.kt_empty0, kBoth);
                if (!w(&bars.kt_full1, ph)) break;
                tc_fence_after();
                kv_block(1);
                mma_commit_pair(&bars.kt_empty1, kBoth);
                mma_commit_pair(&bars.r_done, kBoth);
                // O += (P_hi + P_lo) Vz
                if (!w(&bars.p_ready, ph)) break;
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const uint32_t a_hi = tmem + kTS + 32 * (t >> 1) + 8 * (t & 1);
                    const uint64_t bd = dV + (uint64_t)((t * 2048) >> 4);
                    mma_pair_ts(tmem + kTO, a_hi, bd, id_p, 1);
                    mma_pair_ts(tmem + kTO, a_hi + 16, bd, id_p, 1);
                }
                mma_commit_pair(&bars.o_full, kBoth);
                mma_commit_pair(&bars.v_empty, kBoth);
            }
            // every issued MMA completes before tensor memory is released
            mma_commit_pair(&bars.drain, 1);
            mbar_wait(&bars.drain, 0, nullptr, 200000000ull);
        }
    } else {
        // ------------------------------------------------------------ transform warps
        const int q4 = warp & 3;                     // TMEM lane quarter of this warp
        const int row = 32 * q4 + lane;              // TMEM lane
        const uint32_t lrow = (uint32_t)(32 * q4) << 16;
        const int j = 128 * (int)rank + row;         // query row in the chunk / dk row of R
        const float l2g = dc.l2g[head];
        bool ok = true;
        // tcgen05.ld/st are warp-collective: keep the outcome of every wait uniform
        auto wait = [&](uint64_t* bar, uint32_t par) {
            if (!ok) return false;
            const bool got = __all_sync(0xffffffffu, mbar_wait(bar, par, abort_p));
            if (!got) { ok = false; if (lane == 0) fail(); }
            return ok;
        };
        // Every signal below publishes tensor memory (after tcgen05.fence::before_thread_sync)
        // or shared memory that a proxy fence has made visible to the tensor cores that read
        // it, so a CTA-scope release is enough; a cluster-scope one would also wait for the
        // output warps' global stores to be acknowledged, which costs ~2 k cycles per chunk.
        auto arrive_lead = [&](uint64_t* bar) {
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(lead(bar));
        };
        if (warp < kFirstR) {
            // -------------------------------------------------- scores -> P, then output
            const int half = (warp - kFirstP) >> 2;  // key half (P) / 64-column half (O)
            const float cP = dc.cP[head];
            // P = g^(-B) S with the causal mask (key > j is zero), as hi/lo bf16 pairs in place.
            // Key quarter qq (32 keys) is below this warp's rows for qq < dq, holds their
            // diagonal for qq = dq and lies after them for qq > dq (all zero): warp-uniform.
            const int dq = 4 * (int)rank + q4;
            auto convert = [&](const float* x, int qq, uint32_t* pp) {
                if (qq < dq) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) split2(x[2 * e] * cP, x[2 * e + 1] * cP, pp[e], pp[16 + e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int kc = 32 * qq + 2 * e;
                        const float x0 = kc > j ? 0.f : x[2 * e] * cP;
                        const float x1 = kc + 1 > j ? 0.f : x[2 * e + 1] * cP;
                        split2(x0, x1, pp[e], pp[16 + e]);
                    }
                }
            };
            // output rows of chunk c: xi_j * O for this warp's 64 columns, straight from
            // registers.  Each 128-byte row segment (32 fp32 or 64 bf16 columns = 8 items of
            // 16 bytes) is transposed within 8-lane groups (8 consecutive rows), so that every
            // store instruction writes four whole 128-byte segments.  The last TMEM read
            // releases O for the next Q.R.
            const float xi = exp2f(l2g * (float)(j + 1));
            auto do_out = [&](int c) {
                if (!wait(&bars.o_full, (uint32_t)c & 1u)) return;
                tc_fence_after();
                const int p8 = lane & 7;
                const size_t row0 = (size_t)bh * N + (size_t)c * kB + (size_t)(j - p8);
                constexpr int kSegs = OUT_BF16 ? 1 : 2;           // 128-byte segments per 64 columns
                constexpr int kSegCols = OUT_BF16 ? 64 : 32;
#pragma unroll 1
                for (int sg = 0; sg < kSegs; ++sg) {
                    uint32_t a[8][4];
                    const uint32_t tc0 = tmem + lrow + kTO + 64 * half + kSegCols * sg;
                    if (OUT_BF16) {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            float o[32];
                            tmem_ld32(tc0 + 32 * hh, o);
                            tmem_wait_ld();
                            if (hh == 1) { tc_fence_before(); arrive_lead(&bars.o_free); }
#pragma unroll
                            for (int k = 0; k < 4; ++k)
#pragma unroll
                                for (int w = 0; w < 4; ++w)
                                    a[4 * hh + k][w] =
                                        pack_bf16(xi * o[8 * k + 2 * w], xi * o[8 * k + 2 * w + 1]);
                        }
                    } else {
                        float o[32];
                        tmem_ld32(tc0, o);
                        tmem_wait_ld();
                        if (sg == kSegs - 1) { tc_fence_before(); arrive_lead(&bars.o_free); }
#pragma unroll
                        for (int k = 0; k < 8; ++k)
#pragma unroll
                            for (int w = 0; w < 4; ++w) a[k][w] = __float_as_uint(xi * o[4 * k + w]);
                    }
                    transpose8x8(a, p8);
                    const size_t col = (size_t)blk * 128 + (size_t)(64 * half + kSegCols * sg);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        uint4* dst;
                        if (OUT_BF16)
                            dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out_base) +
                                                           (row0 + k) * dv + col) + p8;
                        else
                            dst = reinterpret_cast<uint4*>(static_cast<float*>(out_base) +
                                                           (row0 + k) * dv + col) + p8;
                        *dst = make_uint4(a[k][0], a[k][1], a[k][2], a[k][3]);
                    }
                }
            };
            for (int c = 0; c < nchunks && ok; ++c) {
                if (!wait(&bars.s_full, (uint32_t)c & 1u)) break;
                tc_fence_after();
#pragma unroll 1
                for (int qq = 4 * half; qq < 4 * half + 4; ++qq) {
                    const uint32_t ts = tmem + lrow + kTS + 32 * qq;
                    uint32_t pp[32];
                    if (qq <= dq) {
                        float x[32];
                        tmem_ld32(ts, x);
                        tmem_wait_ld();
                        convert(x, qq, pp);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) pp[e] = 0u;
                    }
                    tmem_st32(ts, reinterpret_cast<const float*>(pp));
                }
                tmem_wait_st();
                tc_fence_before();
                arrive_lead(&bars.p_ready);
                // while the chunk's P.Vz runs nothing is left to do; then its output
                do_out(c);
            }
        } else {
            // -------------------------------------------------- state copy, then V -> Vz
            const int g = warp - kFirstR;            // 0..7
            const bool remote = g >= 4;              // peer's 64 columns (else this CTA's own)
            const uint32_t cbase = 64u * (remote ? peer : rank);   // TMEM column of the 64
            const float gB = dc.gB[head];
            const uint32_t hi_peer = map_peer(rhi, peer);
            const uint32_t lo_peer = map_peer(rlo, peer);
            // State copy for chunk c: the hi/lo bf16 copy of R_{i-1} (this CTA's dk row j,
            // 64 value columns) into the B operand of Q.R, and R <- g^B R in TMEM, in two
            // halves of 32 columns (4 items of 16 bytes per row).  Own columns go to this
            // CTA's copy; the peer's columns are transposed within 4-lane groups so that
            // each remote store writes 64 contiguous bytes of a row of the peer's copy.
            // R_{-1} comes from state_in (zero without it).
            const int p4 = lane & 3;
            const uint32_t j0 = (uint32_t)(j - p4);
            auto do_state = [&](int c) {
                if (c > 0) {
                    if (!wait(&bars.r_done, (uint32_t)(c - 1) & 1u)) return;
                    tc_fence_after();
                }
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t tcol = tmem + lrow + kTR + cbase + 32 * hh;
                    float x[32];
                    if (c == 0) {
                        if (state_in) {
                            const float4* src = reinterpret_cast<const float4*>(
                                state_in + ((size_t)bh * kDk + j) * dv + blk * 128 + cbase + 32 * hh);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float4 f = src[e];
                                x[4 * e] = f.x; x[4 * e + 1] = f.y; x[4 * e + 2] = f.z; x[4 * e + 3] = f.w;
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) x[e] = 0.f;
                        }
                    } else {
                        tmem_ld32(tcol, x);
                        tmem_wait_ld();
                    }
                    uint32_t h[4][4], l[4][4];      // 16-byte items k = 8 columns each
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            split2(x[8 * k + 2 * e], x[8 * k + 2 * e + 1], h[k][e], l[k][e]);
                            x[8 * k + 2 * e] *= gB;
                            x[8 * k + 2 * e + 1] *= gB;
                        }
                    // the rescaled state goes back now (asynchronous until tcgen05.wait::st)
                    tmem_st32(tcol, x);
                    if (remote) {
                        // lane p of a 4-lane group then holds item 4hh+p of row j0 + k in slot k
                        transpose4x4(h, p4);
                        transpose4x4(l, p4);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t r = j0 + (uint32_t)k;
                            const uint32_t off =
                                r * 128u + ((((uint32_t)(4 * hh + p4)) ^ (r & 7u)) << 4);
                            st_cluster_v4(hi_peer + off, h[k][0], h[k][1], h[k][2], h[k][3]);
                            st_cluster_v4(lo_peer + off, l[k][0], l[k][1], l[k][2], l[k][3]);
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t off = (uint32_t)j * 128u +
                                                 ((((uint32_t)(4 * hh + k)) ^ ((uint32_t)j & 7u)) << 4);
                            *reinterpret_cast<uint4*>(rhi + off) = make_uint4(h[k][0], h[k][1], h[k][2], h[k][3]);
                            *reinterpret_cast<uint4*>(rlo + off) = make_uint4(l[k][0], l[k][1], l[k][2], l[k][3]);
                        }
                    }
                }
                tmem_wait_st();
                if (remote) fence_proxy_async_cluster(); else fence_proxy_async();
                tc_fence_before();
                arrive_lead(&bars.rcopy);
            };
            // V row kr of chunk c scaled in place by g^(B-1-kr); the block lands after the
            // previous P.Vz, while this group copies the state
            const int kr = 32 * g + lane;
            const float fz = exp2f(l2g * (float)(kB - 1 - kr));
            auto do_v = [&](int c) {
                if (!wait(&bars.v_full, (uint32_t)c & 1u)) return;
                uint8_t* vrow = sv + kr * 128;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    uint4* pv = reinterpret_cast<uint4*>(vrow + (((uint32_t)cc ^ ((uint32_t)kr & 7u)) << 4));
                    uint4 u = *pv;
                    uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) wv[e] = pack_bf16(bf16_lo(wv[e]) * fz, bf16_hi(wv[e]) * fz);
                    *pv = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
                fence_proxy_async();
                arrive_lead(&bars.vz_ready);
            };
            for (int c = 0; c < nchunks && ok; ++c) {
                do_state(c);
                do_v(c);
            }
            // ---- final state: this CTA's dk rows of R_{N/B-1}, this warp's 64 columns
            if (ok && state_out && nchunks > 0) {
                if (wait(&bars.r_done, (uint32_t)(nchunks - 1) & 1u)) {
                    tc_fence_after();
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        float x[32];
                        tmem_ld32(tmem + lrow + kTR + cbase + 32 * hh, x);
                        tmem_wait_ld();
                        float4* dst = reinterpret_cast<float4*>(
                            state_out + ((size_t)bh * kDk + j) * dv + blk * 128 + cbase + 32 * hh);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = make_float4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]);
                    }
                }
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();     // no MMA in flight, no remote access pending
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

}  // namespace

bool chunkwise_pair_supported(int dk, int dv, int chunk, const HeadConsts& hc, int H) {
    if (dk != kDk || chunk != kB || dv % 128 != 0) return false;
    for (int h = 0; h < H; ++h)
        if (!(hc.l2g[h] * (float)chunk >= -64.0f)) return false;   // g^(-B) <= 2^64
    return true;
}

cudaError_t launch_chunkwise_tc_pair(const void* q, const void* k, const void* v, void* o,
                                     int out_bf16, int b, int H, int N, int dk, int dv, int chunk,
                                     const HeadConsts& hc, const float* state_in, float* state_out,
                                     cudaStream_t s) {
    if (!chunkwise_pair_supported(dk, dv, chunk, hc, H)) return cudaErrorNotSupported;
    Decay dc;
    for (int h = 0; h < H; ++h) {
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
    const long long grid = 2LL * b * H * (dv / 128);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int smem = kSmemBytes + 1024;
    auto kern = out_bf16 ? chunkwise_pair_kernel<true> : chunkwise_pair_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, kThreads, smem, s>>>(mq, mk, mv, o, state_in, state_out, N, H, dv, dc);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launch(RET_KERNEL_CHUNKWISE_TC_PAIR);
    return e;
}

unsigned read_clear_error_tc_chunkwise_pair(cudaStream_t s) {
    unsigned h = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_err_chunkwise_pair, sizeof(h), 0, cudaMemcpyDeviceToHost,
                                  s) != cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_err_chunkwise_pair, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return h;
}

}  // namespace ret
