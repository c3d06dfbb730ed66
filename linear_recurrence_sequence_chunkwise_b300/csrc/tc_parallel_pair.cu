// tc_parallel_pair.cu -- parallel retention on pairs of SMs (tcgen05 cta_group::2).
//
// Computes eq.(5) of "Transformer取代者登場！…RetNet…（2）", section "Retention" 1) (Fig.3a),
// with the optional factors of "Retention Score 歸一化" and, optionally, the gated GroupNorm
// epilogue of "門控多尺度 Retention" -- the same function as tc_parallel.cu:
//     R[n][m] = (q_n . k_m) [/ sqrt(dk)] * g^(n-m) [/ sqrt(s_n)]   for m <= n, else 0
//     O[n]    = sum_m R[n][m] v_m  [/ max(|sum_m R[n][m]|, 1)]
// for bf16 Q/K/V, dk = 256, dv a multiple of 256, N a multiple of 256.
//
// Work split: one cluster of two CTAs (the two SMs of a pair) per (batch*head, 256-row
// query block, 256 value columns); CTA r owns query rows 128r.. of the block.  The even
// CTA issues every MMA as a pair MMA (M = 256, 128 rows per SM), and the B operands are
// split by N between the SMs, so that each SM loads half of every key and value tile:
//   S  = Q K_t^T     N = 128 keys of tile t (B: CTA r holds keys 64r..64r+63 x all dk)
//   O += P V_t       N = 256 value columns (B: CTA r holds columns 128r..128r+127),
//                    A = P from tensor memory
// Per key tile each SM receives 64 KB (32 KB of K, 32 KB of V) where a single-SM tile
// needs 128 KB.  The even CTA's rows never see the query block's last key tile (it is all
// masked for them); they compute it with the pair and P zeroes it.
//
// Operand format.  P and V enter P.V as fp16 (11 significant bits; one MMA per K step):
// the transform warps round P to fp16 and convert each landed V piece to fp16 in place.
// A unit whose P or V leaves fp16's range, or whose largest |v| is below 2^-6 (typical
// values then near fp16's subnormals), is recomputed in the same launch (second pass)
// with P as a hi/lo pair of bf16 values against the bf16 V, two MMAs per K step -- the
// format tc_parallel.cu uses throughout; the re-run decision is taken for the whole
// cluster.  S = Q K^T takes the loaded bf16 operands (exact products).
//
// With the fused epilogue the two value blocks of a query block (dv = 512) form one
// cluster of four CTAs (two pairs) that exchange per-row GroupNorm statistics; CTA rank
// 2 vb + r holds rows 128r.. of value block vb.
//
// Roles (320 threads): warp 0 TMA -- lane 0 Q (once per pass), the K pieces (three slots,
// completing on the even CTA's barriers) and the gate tiles, lane 1 the V pieces (two
// slots, each CTA's own barrier), so that a K load never waits behind a V slot; warp 1
// tensor memory and, in the even CTA, the MMA issuer; warps 2-9 scores -> P, V -> fp16 and
// the epilogue.  Tensor memory per CTA: [0,256) O (this CTA's 128 rows x 256 value
// columns), [256,384) and [384,512) S (this CTA's 128 rows x the tile's 128 keys, double-
// buffered).  Shared memory: Q 64 KB + 3 K slots + 2 V slots of 32 KB = 224 KB.  Every
// wait is bounded; a wait that gives up sets the device error word and the CTAs unwind.
#include <type_traits>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace ret {
namespace {

__device__ unsigned g_err_parallel_pair;
__device__ unsigned g_reruns_parallel_pair;   // units re-run in the hi/lo bf16 format

using namespace tc;

constexpr int kKRing = 3;                 // K pieces in flight
constexpr int kVRing = 2;                 // V pieces in flight
constexpr int kAtom = 128 * 128;          // 128 rows x 64 bf16 (16 KB)
constexpr int kKBox = 64 * 128;           // 64 keys x 64 bf16 (8 KB)
constexpr int kPiece = 2 * kAtom;         // 32 KB ring slot
constexpr int kQBytes = 4 * kAtom;        // 128 rows x 256 dk
constexpr float kF16Max = 65504.0f;
// fp16 V keeps 11 significant bits only above 2^-14; a unit whose largest |v| is below
// 2^-6 (typical values then near fp16's subnormals) takes the hi/lo format
constexpr float kF16VMin = 0.015625f;
constexpr int kThreads = 320;
constexpr int kXWarps = 8;
constexpr int kW = 256;                   // value columns of a pair (128 per CTA for P.V's B)
constexpr uint32_t kTO = 0, kTS = 256;
constexpr int kHeadGroup = 8;
constexpr int kMaxVb = 4;                 // value blocks in one cluster (8 CTAs)

struct ParConsts {
    float l2g[kMaxHeads];
    float lng[kMaxHeads];
    float omg[kMaxHeads];
};

struct EpiArgs {
    void* out;              // [b][H][N][dv] (EPI = 0) or [b][N][H*dv]
    const void* g;          // [b][N][H*dv], fp32 or bf16 (template EPI); read through a TMA map
    const float* weight;    // [H*dv] or NULL
    const float* bias;      // [H*dv] or NULL
    float eps;
};

struct Bars {
    // the even CTA's copies count both CTAs' loads and warps
    uint64_t q_full;
    uint64_t k_full[kKRing];
    uint64_t p_ready[2], v_ready[kVRing];
    // each CTA's own copy, arrived on by the MMA commits (multicast)
    uint64_t k_empty[kKRing], v_empty[kVRing];
    uint64_t s_full[2];
    uint64_t o_full;
    uint64_t q_free;
    uint64_t drain;
    // each CTA's own loads
    uint64_t v_full[kVRing];
    uint64_t g_full[2], g_pre;
};

__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}

// 3-D tiled load into this CTA's shared memory, completion counted on the barrier at
// cluster address bar_cl (the even CTA's barrier for pair operands).
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map, int c0, int c1,
                                                 int c2, uint32_t bar_cl) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar_cl)
        : "memory");
}

template <bool OUT_BF16, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
parallel_pair_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                     const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mg,
                     int N, int H, int dv, int bH, int nvb, unsigned flags, const ParConsts pc,
                     const EpiArgs ea, uint64_t wait_ns) {
    constexpr int kCols = kW / 2;                        // value columns of a transform group
    constexpr int kEpiChunks = kCols / 64;               // 64-column chunks per group
    // bf16 gate tiles of both groups fit where Q was: load them while the last P.V runs
    constexpr bool kGPrefetch = (EPI == 2);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* qarea = sm;
    uint8_t* ring = sm + kQBytes;                  // K ring then V ring (the epilogue's scratch)
    uint8_t* kring = ring;
    uint8_t* vring = ring + kKRing * kPiece;
    __shared__ Bars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    // epilogue scratch in the ring once every MMA of the pair has completed (after o_full)
    float (*rs_part)[128] = reinterpret_cast<float (*)[128]>(ring);
    float (*st_part)[128] = reinterpret_cast<float (*)[128]>(ring + 1024);
    float2 (*peer_stats)[128] = reinterpret_cast<float2 (*)[128]>(ring + 2048);
    __shared__ __align__(16) float colf[128];     // g^(-j), j = key column in a tile

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const uint32_t rank = crank & 1u;              // position in the pair
    const uint32_t lead_rank = crank & ~1u;        // the pair's even CTA
    const uint16_t pair_mask = (uint16_t)(3u << lead_rank);
    // unit = (head group, heavy query blocks first, head, value block); two CTAs each
    const int nqb = N / 256;
    const int unit = (int)(blockIdx.x >> 1);
    const int full_grp = kHeadGroup * nqb * nvb;
    const int gi = unit / full_grp;
    const int gheads = min(kHeadGroup, bH - gi * kHeadGroup);
    const int r_in = unit % full_grp;
    const int qb = nqb - 1 - r_in / (gheads * nvb);
    const int rest = r_in % (gheads * nvb);
    const int bh = gi * kHeadGroup + rest / nvb, vb = rest % nvb;
    const int head = bh % H;
    const int n0 = 256 * qb + 128 * (int)rank;     // first query row of this CTA
    const int T = 2 * qb + 2;                      // key tiles under the mask for the pair
    volatile int* abort_p = &abort_flag;
    float stat_mean = 0.f, stat_m2 = 0.f, row_inv = 1.f;

    const int csize = EPI != 0 ? 2 * nvb : 2;       // CTAs in the cluster
    __shared__ int range_flag;                      // an fp16 conversion left fp16's range
    __shared__ unsigned vmax_bits;                  // largest |v| of the fp16 pass (as bits)

    if (threadIdx.x == 0) {
        abort_flag = 0;
        range_flag = 0;
        vmax_bits = 0u;
        mbar_init(&bars.q_full, 1);
        for (int s = 0; s < kKRing; ++s) { mbar_init(&bars.k_full[s], 1); mbar_init(&bars.k_empty[s], 1); }
        for (int s = 0; s < kVRing; ++s) {
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.v_ready[s], 2 * kXWarps);
            mbar_init(&bars.v_empty[s], 1);
        }
        for (int c = 0; c < 2; ++c) {
            mbar_init(&bars.s_full[c], 1);
            mbar_init(&bars.p_ready[c], 2 * kXWarps);
        }
        mbar_init(&bars.o_full, 1);
        mbar_init(&bars.q_free, 1);
        mbar_init(&bars.g_full[0], 1); mbar_init(&bars.g_full[1], 1);
        mbar_init(&bars.g_pre, 1);
        mbar_init(&bars.drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) { tmem_alloc_pair(&tmem_slot, 512); tmem_relinquish_pair(); }
    tc_fence_before();
    cluster_sync_all();     // every CTA's barriers exist before any remote arrive or pair load
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t peer_abort = map_peer(&abort_flag, crank ^ 1u);
    volatile int* range_p = &range_flag;
    auto fail = [&]() {
        *abort_p = 1;
        st_cluster_s32(peer_abort, 1);
        atomicOr(&g_err_parallel_pair, 1u);
    };
    auto lead = [&](uint64_t* b) { return map_peer(b, lead_rank); };
    // an fp16 conversion met a magnitude outside fp16's range (or V too small for it): every
    // CTA of the cluster re-runs its unit with the hi/lo bf16 format
    auto out_of_range = [&]() {
        for (int r = 0; r < csize; ++r) st_cluster_s32(map_peer(&range_flag, (uint32_t)r), 1);
    };

    // transform warps' state that outlives a pass
    const int grp = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;
    const uint32_t lrow = (uint32_t)(32 * q4) << 16;
    const int n = n0 + row;
    const float l2g = pc.l2g[head];
    float rowc = (flags & RET_NORM_SCALE) ? rsqrtf(256.0f) : 1.0f;
    if (warp >= 2 && (flags & RET_NORM_DECAY)) rowc *= rsqrtf(decay_rowsum(pc.lng[head], pc.omg[head], n));
    const bool want_rs = (flags & RET_NORM_ROWSUM) != 0;
    // g^(n-m) = g^(n-m0) * g^(-(m-m0)): one exp2 per row and tile, times a column factor
    // from a table; a g with g^(-127) > 2^64 takes one exp2 per element.
    const bool factored = l2g >= -0.5f;
    if (warp >= 2 && grp == 0) colf[row] = factored ? exp2f(-l2g * (float)row) : 0.f;
    if (warp >= 2) named_bar(1, kXWarps * 32);
    float rs = 0.f;
    bool tok = true;                                // transform warps: no wait gave up
    int passes = 0;

    // Pass 0 uses fp16 P and V (one P.V MMA per K step); pass 1 runs only if pass 0 left
    // fp16's range somewhere in the cluster and recomputes the unit with hi/lo bf16 P.
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const bool f16 = pass == 0;
        const uint32_t tb = (uint32_t)(pass * T);   // global index of this pass's tile 0
        passes = pass + 1;
        if (warp == 0) {
            // -------------------------------------------------------- TMA producers
            // lane 0: Q, the K pieces and the gate tiles; lane 1: the V pieces.  Two threads,
            // so that a K load never queues behind a wait for a V slot (V slots free only
            // after their P.V, K slots after their score MMA).
            if (lane == 0) {
                bool ok = !*abort_p;
                if (pass == 0) {
                    tma_prefetch_desc(&mq); tma_prefetch_desc(&mk); tma_prefetch_desc(&mv);
                    if (EPI != 0) tma_prefetch_desc(&mg);
                } else if (ok) {
                    // Q's area: the last score MMA of pass 0 has read it, and the gate tiles
                    // loaded into it have landed
                    if (!mbar_wait(&bars.q_free, 0, abort_p, wait_ns)) { ok = false; fail(); }
                    if (ok && kGPrefetch && !mbar_wait(&bars.g_pre, 0, abort_p, wait_ns)) { ok = false; fail(); }
                }
                bool q_issued = false;
                if (ok) {
                    if (rank == 0) mbar_arrive_expect_tx(&bars.q_full, 2 * kQBytes);
                    for (int a = 0; a < 4; ++a)
                        tma_load_3d_pair(qarea + a * kAtom, &mq, 64 * a, n0, bh, lead(&bars.q_full));
                    q_issued = true;
                }
                int kf = 0;
                for (int t = 0; t < T && ok; ++t) {
                    const uint32_t g = tb + (uint32_t)t;
                    // K half of tile t: keys 128t + 64 rank .. +63, all dk (four 8 KB boxes)
                    const int ks = (int)(g % kKRing);
                    if (!mbar_wait(&bars.k_empty[ks], ((g / kKRing) & 1) ^ 1, abort_p, wait_ns)) {
                        ok = false; fail(); break;
                    }
                    if (rank == 0) mbar_arrive_expect_tx(&bars.k_full[ks], 2 * kPiece);
                    for (int a = 0; a < 4; ++a)
                        tma_load_3d_pair(kring + ks * kPiece + a * kKBox, &mk, 64 * a,
                                         128 * t + 64 * (int)rank, bh, lead(&bars.k_full[ks]));
                    ++kf;
                }
                bool g_issued = false;
                if (kGPrefetch && ok) {
                    // the last score MMA of the pass has read Q: its area takes the gate tiles
                    if (!mbar_wait(&bars.q_free, (uint32_t)pass, abort_p, wait_ns)) {
                        ok = false;
                        fail();
                    } else {
                        mbar_arrive_expect_tx(&bars.g_pre, 2 * kEpiChunks * 16384);
                        for (int gg = 0; gg < 2; ++gg)
                            for (int ch = 0; ch < kEpiChunks; ++ch)
                                tma_load_3d(qarea + (gg * kEpiChunks + ch) * 16384, &mg,
                                            head * dv + kW * vb + kCols * gg + 64 * ch, n0, bh / H,
                                            &bars.g_pre);
                        g_issued = true;
                    }
                }
                if (!ok) {
                    // let the loads in flight land before the CTAs unwind (the even CTA waits
                    // for the pair's K and Q loads, each CTA for its own gate loads)
                    for (int i = kf > kKRing ? kf - kKRing : 0; i < kf && rank == 0; ++i) {
                        const uint32_t g = tb + (uint32_t)i;
                        mbar_wait(&bars.k_full[g % kKRing], (g / kKRing) & 1, nullptr, 100000000ull);
                    }
                    if (q_issued && rank == 0) mbar_wait(&bars.q_full, (uint32_t)pass, nullptr, 100000000ull);
                    if (g_issued) mbar_wait(&bars.g_pre, (uint32_t)pass, nullptr, 100000000ull);
                }
            } else if (lane == 1) {
                bool ok = !*abort_p;
                int vf = 0;
                for (int t = 0; t < T && ok; ++t) {
                    const uint32_t g = tb + (uint32_t)t;
                    // V half of tile t: its 128 keys x value columns kW vb + 128 rank .. +127,
                    // completing on this CTA's barrier (the transform warps convert it)
                    const int vs = (int)(g % kVRing);
                    if (!mbar_wait(&bars.v_empty[vs], ((g / kVRing) & 1) ^ 1, abort_p, wait_ns)) {
                        ok = false; fail(); break;
                    }
                    mbar_arrive_expect_tx(&bars.v_full[vs], kPiece);
                    for (int a = 0; a < 2; ++a)
                        tma_load_3d(vring + vs * kPiece + a * kAtom, &mv, kW * vb + 128 * (int)rank + 64 * a,
                                    128 * t, bh, &bars.v_full[vs]);
                    ++vf;
                }
                if (!ok) {
                    for (int i = vf > kVRing ? vf - kVRing : 0; i < vf; ++i) {
                        const uint32_t g = tb + (uint32_t)i;
                        mbar_wait(&bars.v_full[g % kVRing], (g / kVRing) & 1, nullptr, 100000000ull);
                    }
                }
            }
        } else if (warp == 1) {
            // -------------------------------------------------------- MMA issuer (even CTA)
            if (rank == 0 && lane == 0) {
                const uint32_t id_s = idesc_bf16(256, 128, 0, 0);          // Q K^T: both K-major
                const uint32_t id_p = idesc_f16(256, kW, 0, 1, f16 ? 0 : 1); // P V: A in TMEM
                const uint64_t dQ = sdesc_sw128(smem_u32(qarea), 16, 1024);
                const uint64_t dK = sdesc_sw128(smem_u32(kring), 16, 1024);
                const uint64_t dV = sdesc_sw128(smem_u32(vring), kAtom, 1024);
                bool ok = !*abort_p;
                auto wait = [&](uint64_t* bar, uint32_t par) {
                    if (ok && !mbar_wait_cl(bar, par, abort_p, wait_ns)) { ok = false; fail(); }
                    return ok;
                };
                wait(&bars.q_full, (uint32_t)pass);
                for (int st = 0; st <= T && ok; ++st) {
                    if (st < T) {
                        const uint32_t g = tb + (uint32_t)st;
                        const int ks = (int)(g % kKRing);
                        // S(g) overwrites the buffer P(g-2) was read from: tcgen05.mma operations
                        // of one thread execute in issue order, so P(g-2).V has read it first.
                        const uint32_t ts = tmem + kTS + 128 * (g & 1);
                        if (!wait(&bars.k_full[ks], (g / kKRing) & 1)) break;
                        tc_fence_after();
                        const uint64_t db = dK + (uint64_t)((ks * kPiece) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk) {
                            // dk box kk/4 (Q: 16 KB boxes; K: 8 KB boxes), 16 dk values per step
                            const uint64_t qa = dQ + (uint64_t)(((kk / 4) * kAtom + (kk % 4) * 32) >> 4);
                            const uint64_t kb = db + (uint64_t)(((kk / 4) * kKBox + (kk % 4) * 32) >> 4);
                            mma_pair(ts, qa, kb, id_s, kk != 0);
                        }
                        mma_commit_pair(&bars.k_empty[ks], pair_mask);
                        mma_commit_pair(&bars.s_full[g & 1], pair_mask);
                        if (st == T - 1) mma_commit_pair(&bars.q_free, pair_mask);
                    }
                    if (st >= 1) {
                        const int t = st - 1;
                        const uint32_t g = tb + (uint32_t)t;
                        const int vs = (int)(g % kVRing);
                        if (!wait(&bars.p_ready[g & 1], (g >> 1) & 1)) break;
                        if (!wait(&bars.v_ready[vs], (g / kVRing) & 1)) break;
                        tc_fence_after();
                        const uint32_t ts = tmem + kTS + 128 * (g & 1);
                        const uint64_t db = dV + (uint64_t)((vs * kPiece) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t a_t = ts + 32 * (kk / 2) + 8 * (kk % 2);
                            const uint64_t bd = db + (uint64_t)((16 * kk * 128) >> 4);
                            mma_pair_ts(tmem + kTO, a_t, bd, id_p, (t | kk) != 0);
                            if (!f16) mma_pair_ts(tmem + kTO, a_t + 16, bd, id_p, 1);
                        }
                        mma_commit_pair(&bars.v_empty[vs], pair_mask);
                    }
                }
                mma_commit_pair(&bars.o_full, pair_mask);
                // every issued MMA completes before the next pass or the release of TMEM
                mma_commit_pair(&bars.drain, (uint16_t)(1u << lead_rank));
                mbar_wait(&bars.drain, (uint32_t)pass, nullptr, 200000000ull);
            }
        } else {
            // -------------------------------------------------------- transform warps
            auto wait = [&](uint64_t* bar, uint32_t par) {
                if (!tok) return false;
                const bool got = __all_sync(0xffffffffu, mbar_wait(bar, par, abort_p, wait_ns));
                if (!got) { tok = false; if (lane == 0) fail(); }
                return tok;
            };
            tok = !*abort_p;
            rs = 0.f;
            __half2 pmax2 = __float2half2_rn(0.f);      // largest |P| rounded to fp16
            float vmax = 0.f;                            // largest |v| converted to fp16
            // P for this warp's 64 keys of tile t, 32 at a time, specialised at compile time
            // for the format (fp16 / hi-lo bf16), the factored decay and the diagonal tile
            // (the only one that needs the causal mask; tiles after it hold no key of these
            // rows).  fp16: 16 columns of pairs per 32 keys; hi/lo: hi pairs, then lo pairs.
            const int kc0 = 64 * grp;
            const int tdiag = n0 / 128;
            auto convert = [&](uint32_t ts, int t, float a, auto fmt, auto fac, auto diag) {
                constexpr bool F16 = decltype(fmt)::value;
                constexpr bool FAC = decltype(fac)::value, DIAG = decltype(diag)::value;
                const int m0 = 128 * t + kc0;               // first key of this warp's 64
#pragma unroll 1
                for (int c32 = 0; c32 < 2; ++c32) {
                    float x[32];
                    tmem_ld32(ts + kc0 + 32 * c32, x);
                    tmem_wait_ld();
                    uint32_t pk[F16 ? 16 : 32];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int j = 32 * c32 + 2 * e;
                        float w0, w1;
                        if (FAC) {
                            const float2 cf = *reinterpret_cast<const float2*>(colf + kc0 + j);
                            w0 = a * cf.x;
                            w1 = a * cf.y;
                        } else {
                            w0 = rowc * decay_pow(l2g, (float)(n - m0 - j));
                            w1 = rowc * decay_pow(l2g, (float)(n - m0 - j - 1));
                        }
                        float p0 = x[2 * e] * w0, p1 = x[2 * e + 1] * w1;
                        if (DIAG) {
                            if (m0 + j > n) p0 = 0.f;
                            if (m0 + j + 1 > n) p1 = 0.f;
                        }
                        if (want_rs) rs += p0 + p1;
                        if (F16) {
                            __half2 h = __floats2half2_rn(p0, p1);
                            pmax2 = __hmax2_nan(pmax2, __habs2(h));
                            pk[e] = *reinterpret_cast<uint32_t*>(&h);
                        } else {
                            pk[e] = pack_bf16(p0, p1);
                            pk[(16 + e) % (F16 ? 16 : 32)] =
                                pack_bf16(p0 - __uint_as_float(pk[e] << 16),
                                          p1 - __uint_as_float(pk[e] & 0xffff0000u));
                        }
                    }
                    if (F16) tmem_st16(ts + kc0 + 32 * c32, pk);
                    else tmem_st32(ts + kc0 + 32 * c32, reinterpret_cast<const float*>(pk));
                }
            };
            auto tile = [&](uint32_t ts, int t, auto fmt) {
                if (t > tdiag) {
                    // the pair's last tile lies after every row of the even CTA: P = 0
                    float z[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) z[e] = 0.f;
                    tmem_st32(ts + kc0, z);
                    tmem_st32(ts + kc0 + 32, z);
                    return;
                }
                const float a = rowc * (factored ? decay_pow(l2g, (float)(n - 128 * t)) : 1.0f);
                if (factored) {
                    if (t == tdiag) convert(ts, t, a, fmt, std::true_type{}, std::true_type{});
                    else convert(ts, t, a, fmt, std::true_type{}, std::false_type{});
                } else {
                    if (t == tdiag) convert(ts, t, a, fmt, std::false_type{}, std::true_type{});
                    else convert(ts, t, a, fmt, std::false_type{}, std::false_type{});
                }
            };
            // this CTA's V piece in slot vs -> fp16 in place: thread i takes row i % 128 of
            // 64-column box i / 128, its 16-byte items in swizzled order (conflict-free)
            const int vt = threadIdx.x - 64;
            auto convert_v = [&](int vs) {
                const int vrow = vt & 127;
                uint8_t* vr = vring + vs * kPiece + (vt >> 7) * kAtom + vrow * 128;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    uint4* pv = reinterpret_cast<uint4*>(vr + ((((uint32_t)cc) ^ ((uint32_t)vrow & 7u)) << 4));
                    const uint4 u = *pv;
                    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float y0 = __uint_as_float(wv[e] << 16), y1 = __uint_as_float(wv[e] & 0xffff0000u);
                        vmax = fmaxf(vmax, fmaxf(fabsf(y0), fabsf(y1)));
                        __half2 h = __floats2half2_rn(y0, y1);
                        o[e] = *reinterpret_cast<uint32_t*>(&h);
                    }
                    *pv = make_uint4(o[0], o[1], o[2], o[3]);
                }
            };
            for (int t = 0; t < T && tok; ++t) {
                const uint32_t g = tb + (uint32_t)t;
                if (!wait(&bars.s_full[g & 1], (g >> 1) & 1)) break;
                tc_fence_after();
                const uint32_t ts = tmem + lrow + kTS + 128 * (g & 1);
                if (f16) tile(ts, t, std::true_type{});
                else tile(ts, t, std::false_type{});
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(lead(&bars.p_ready[g & 1]));
                // V of the tile (loaded about two tiles ahead): fp16 for this pass's P.V
                const int vs = (int)(g % kVRing);
                if (!wait(&bars.v_full[vs], (g / kVRing) & 1)) break;
                if (f16) {
                    convert_v(vs);
                    fence_proxy_async();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(lead(&bars.v_ready[vs]));
            }
            if (f16) {
                const float pm = fmaxf(__low2float(pmax2), __high2float(pmax2));
                if (tok && (!(pm < kF16Max) || !(vmax < kF16Max))) out_of_range();
                // the largest |v| of this CTA's V pieces, over all its transform threads
                atomicMax(&vmax_bits, __float_as_uint(vmax));
                named_bar(2, kXWarps * 32);
                if (tok && vt == 0 && __uint_as_float(vmax_bits) < kF16VMin) out_of_range();
            }
        }
        // ---------------------------------------------------------- end of the pass
        __syncwarp();
        tc_fence_before();
        cluster_sync_all();     // every MMA of the pass was issued and drained; flags are set
        tc_fence_after();
        if (pass == 1 || *abort_p || !*range_p) break;
        if (threadIdx.x == 0 && crank == 0) atomicAdd(&g_reruns_parallel_pair, 1u);
    }
    if (warp >= 2) {
        // ---- output: O / max(|row sum|, 1)
        auto wait = [&](uint64_t* bar, uint32_t par) {
            if (!tok) return false;
            const bool got = __all_sync(0xffffffffu, mbar_wait(bar, par, abort_p, wait_ns));
            if (!got) { tok = false; if (lane == 0) fail(); }
            return tok;
        };
        const uint32_t ocol = tmem + lrow + kTO + kCols * grp;
        const bool have_o = tok && wait(&bars.o_full, (uint32_t)(passes - 1));
        if (have_o) tc_fence_after();
        rs_part[grp][row] = rs;
        named_bar(2, kXWarps * 32);
        float den = 1.f;
        if (want_rs) den = fmaxf(fabsf(rs_part[0][row] + rs_part[1][row]), 1.0f);
        const float inv = 1.0f / den;
        if (EPI != 0) {
            // mean, then sum of squared deviations, of this CTA's 256 values of the row
            float s1 = 0.f;
            if (have_o) {
#pragma unroll 1
                for (int c0 = 0; c0 < kCols; c0 += 32) {
                    float o[32];
                    tmem_ld32(ocol + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) s1 += o[j] * inv;
                }
            }
            st_part[grp][row] = s1;
            named_bar(3, kXWarps * 32);
            const float mean_b = (st_part[0][row] + st_part[1][row]) / (float)kW;
            named_bar(4, kXWarps * 32);
            float s2 = 0.f;
            if (have_o) {
#pragma unroll 1
                for (int c0 = 0; c0 < kCols; c0 += 32) {
                    float o[32];
                    tmem_ld32(ocol + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) { const float d = o[j] * inv - mean_b; s2 += d * d; }
                }
            }
            st_part[grp][row] = s2;
            named_bar(5, kXWarps * 32);
            if (grp == 0) {
                stat_mean = mean_b;
                stat_m2 = st_part[0][row] + st_part[1][row];
            }
        }
        row_inv = inv;
    }
    if (EPI != 0) {
        // 1st cluster barrier: every CTA is past its last MMA, so its ring may receive the
        // statistics of the CTAs holding the same rows in the other value blocks; 2nd: all
        // statistics have arrived.
        __syncwarp();
        tc_fence_before();
        cluster_sync_all();
        tc_fence_after();
        if (warp >= 2 && warp < 6) {
            const int row = 32 * (warp & 3) + (threadIdx.x & 31);
            for (int r = 0; r < nvb; ++r)
                st_cluster_f32x2(map_peer(&peer_stats[vb][row], (uint32_t)(2 * r) + rank), stat_mean,
                                 stat_m2);
        }
        __syncwarp();
        cluster_sync_all();
    }
    // ---- output: per transform group, 64-column chunks of the group's 128 columns, stored
    // from registers as whole 128-byte row segments (8-lane transposes).  Without the gate
    // prefetch (fp32 gate), the ring takes a gate tile per chunk.
    if (warp >= 2) {
        const int grp = (warp - 2) >> 2;
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane;
        const uint32_t lrow = (uint32_t)(32 * q4) << 16;
        const bool issuer = (threadIdx.x == (unsigned)(64 + 128 * grp));   // lane 0 of warp 2 / 6
        constexpr int kGAtoms = (EPI == 2) ? 1 : 2;
        const float inv = row_inv;
        float mean = 0.f, rstd = 1.f;
        if (EPI != 0) {
            for (int r = 0; r < nvb; ++r) mean += peer_stats[r][row].x;
            mean /= (float)nvb;
            float m2 = 0.f;
            for (int r = 0; r < nvb; ++r) {
                const float d = peer_stats[r][row].x - mean;
                m2 += peer_stats[r][row].y + (float)kW * d * d;
            }
            rstd = rsqrtf(m2 / (float)dv + ea.eps);
        }
        const int bi = bh / H;
        const bool live = __all_sync(0xffffffffu, abort_flag == 0);
        if (live) tc_fence_after();
        auto swz = [&](int c16) { return (uint32_t)(row * 128 + ((((uint32_t)c16) ^ (row & 7)) << 4)); };
        const int p8 = lane & 7;
        const int r0 = row - p8;
        const size_t row_elems = (EPI != 0) ? (size_t)H * dv : (size_t)dv;
        const size_t row_base = (EPI != 0) ? (size_t)bi * N : (size_t)bh * N;
#pragma unroll 1
        for (int ch = 0; ch < kEpiChunks; ++ch) {
            const int col = kW * vb + kCols * grp + 64 * ch;          // first value column
            const int gcol = (EPI != 0) ? head * dv + col : col;
            const int plane = (EPI != 0) ? bi : bh;
            uint8_t* gst = kGPrefetch ? qarea + (grp * kEpiChunks + ch) * 16384
                                      : ring + 8192 + grp * 65536;
            if (issuer && EPI != 0 && !kGPrefetch && live) {
                mbar_arrive_expect_tx(&bars.g_full[grp], kGAtoms * 16384);
                for (int a2 = 0; a2 < kGAtoms; ++a2)
                    tma_load_3d(gst + a2 * 16384, &mg, gcol + a2 * (EPI == 2 ? 64 : 32), n0, plane,
                                &bars.g_full[grp]);
            }
            bool got_g = true;
            if (EPI != 0 && live) {
                got_g = kGPrefetch
                            ? __all_sync(0xffffffffu, mbar_wait(&bars.g_pre, (uint32_t)(passes - 1), abort_p, wait_ns))
                            : __all_sync(0xffffffffu, mbar_wait(&bars.g_full[grp], ch & 1, abort_p, wait_ns));
                if (!got_g && lane == 0) fail();
            }
            if (live && got_g) {
                uint32_t a[8][4];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float o[32];
                    tmem_ld32(tmem + lrow + kTO + kCols * grp + 64 * ch + 32 * hf, o);
                    float gv[32];
                    if (EPI == 2) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint4 u = *reinterpret_cast<const uint4*>(gst + swz(4 * hf + c));
                            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                gv[8 * c + 2 * e] = __uint_as_float(w4[e] << 16);
                                gv[8 * c + 2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
                            }
                        }
                    } else if (EPI == 1) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const float4 f = *reinterpret_cast<const float4*>(gst + hf * 16384 + swz(c));
                            gv[4 * c] = f.x; gv[4 * c + 1] = f.y; gv[4 * c + 2] = f.z; gv[4 * c + 3] = f.w;
                        }
                    }
                    tmem_wait_ld();
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        if (EPI == 0) {
                            o[jj] = o[jj] * inv;
                        } else {
                            float yn = (o[jj] * inv - mean) * rstd;
                            const int ch_ = head * dv + col + 32 * hf + jj;
                            if (ea.weight) yn *= ea.weight[ch_];
                            if (ea.bias) yn += ea.bias[ch_];
                            // swish(g) = h (1 + tanh(h)), h = g / 2
                            const float hg = 0.5f * gv[jj];
                            o[jj] = fmaf(hg, tanh_approx(hg), hg) * yn;
                        }
                    }
                    if (OUT_BF16) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
#pragma unroll
                            for (int w = 0; w < 4; ++w)
                                a[4 * hf + k][w] = pack_bf16(o[8 * k + 2 * w], o[8 * k + 2 * w + 1]);
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k)
#pragma unroll
                            for (int w = 0; w < 4; ++w) a[k][w] = __float_as_uint(o[4 * k + w]);
                    }
                    if (!OUT_BF16 || hf == 1) {
                        transpose8x8(a, p8);
                        const int c0 = gcol + (OUT_BF16 ? 0 : 32 * hf);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const size_t e0 = (row_base + (size_t)(n0 + r0 + k)) * row_elems + (size_t)c0;
                            uint4* dst = OUT_BF16
                                ? reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(ea.out) + e0) + p8
                                : reinterpret_cast<uint4*>(static_cast<float*>(ea.out) + e0) + p8;
                            *dst = make_uint4(a[k][0], a[k][1], a[k][2], a[k][3]);
                        }
                    }
                }
            }
            // every warp of the group is done with this chunk's gate tile
            if (!kGPrefetch && EPI != 0) named_bar(6 + grp, 128);
        }
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();     // no tensor-memory access pending in any CTA of the pair
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

using PairKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap,
                            const CUtensorMap, int, int, int, int, int, unsigned, const ParConsts,
                            const EpiArgs, uint64_t);

template <int EPI>
PairKernel pick(int out_bf16) {
    return out_bf16 ? parallel_pair_kernel<true, EPI> : parallel_pair_kernel<false, EPI>;
}

}  // namespace

// Every wait of the kernel gives up after this long (wall time).
constexpr uint64_t kPairWaitNs = 2000000000ull;

// epi: 0 plain output, 1 gated with fp32 G, 2 gated with bf16 G
cudaError_t launch_parallel_pair(const void* q, const void* k, const void* v, const void* g,
                                 void* out, int out_bf16, int epi, int b, int H, int N, int dk,
                                 int dv, const HeadConsts& hc, unsigned flags, float eps,
                                 const float* weight, const float* bias, cudaStream_t s) {
    if (dk != 256 || dv % kW != 0 || N < 256 || N % 256 != 0) return cudaErrorNotSupported;
    const int nvb = dv / kW;
    if (epi != 0 && nvb > kMaxVb) return cudaErrorNotSupported;
    ParConsts pc;
    for (int h = 0; h < H; ++h) {
        pc.l2g[h] = hc.l2g[h];
        pc.lng[h] = hc.lng[h];
        pc.omg[h] = hc.omg[h];
    }
    const long long bH = (long long)b * H;
    if (bH >= (1LL << 31) || N >= (1 << 30)) return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv, mg;
    if (!tc::make_map_bf16_3d(&mq, q, bH, N, dk, 128) || !tc::make_map_bf16_3d(&mk, k, bH, N, dk, 64) ||
        !tc::make_map_bf16_3d(&mv, v, bH, N, dv, 128))
        return cudaErrorInvalidValue;
    if (epi == 0) {
        mg = mq;
    } else if (!tc::make_map_3d_128b(&mg, g, epi == 2, b, N, (uint64_t)H * dv, 128)) {
        return cudaErrorInvalidValue;
    }
    const long long grid = 2LL * (N / 256) * bH * nvb;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int smem = kQBytes + (kKRing + kVRing) * kPiece + 1024;
    PairKernel kern = epi == 0 ? pick<0>(out_bf16) : epi == 1 ? pick<1>(out_bf16) : pick<2>(out_bf16);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    EpiArgs ea;
    ea.out = out;
    ea.g = g;
    ea.weight = weight;
    ea.bias = bias;
    ea.eps = eps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)(epi != 0 ? 2 * nvb : 2);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mg, N, H, dv, (int)bH, nvb, flags, pc, ea,
                           kPairWaitNs);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess)
        count_launch(epi == 0 ? RET_KERNEL_PARALLEL_TC_PAIR : RET_KERNEL_PARALLEL_GATED_TC_PAIR);
    return e;
}

unsigned read_clear_reruns_parallel_pair(cudaStream_t s) {
    unsigned h = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_reruns_parallel_pair, sizeof(h), 0, cudaMemcpyDeviceToHost,
                                  s) != cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_reruns_parallel_pair, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return h;
}

unsigned read_clear_error_parallel_pair(cudaStream_t s) {
    unsigned h = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_err_parallel_pair, sizeof(h), 0, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_err_parallel_pair, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return h;
}

}  // namespace ret
