// attention_fwd.cu - attention forward on sm_103a:  O = softmax(scale * Q K^T [causal]) V.
//
// The FlashAttention kernel of the aikraft.ru TileLang tutorial survey ("TileLang: создание
// высокопроизводительных GPU-ядер", section 6 "FlashAttention: Слияние внимания"): tiles of
// queries, keys and values, no materialised score matrix, online softmax (running row
// maxima, normalisation sums, rescaling factors), causal masking, copies pipelined with the
// matrix products.  Its thread roles follow "TileLang异步协作终极指南" (producers load K/V, one
// role computes QK^T, another the softmax and the output), rebuilt on tcgen05:
//
//  * one CTA per (128-query tile, batch x head); 320 threads: warp 0 issues TMA copies (Q
//    once, then K_j and V_j into a 2-stage ring), warp 1 issues every MMA from one lane,
//    warps 2-9 run the softmax in two groups of four warps: each query row (TMEM lane) has
//    one thread in each group, and each thread owns half of the row's keys and half of its
//    output columns.  Per tile the threads of a row combine their partial maxima with a
//    shared-memory atomicMax (three rotating slots; the block-wide vote that ends a failed
//    wait doubles as the barrier), then each exponentiates its keys (packed f32x2 arithmetic,
//    ex2.approx) and merges its columns; the partial row sums are added once at the end;
//  * S_j = Q K_j^T (M 128 queries, N 128 keys, K = head_dim) accumulates in TMEM, two
//    buffers, so S_{j+1} is computed while the softmax reads S_j;
//  * the softmax reads its S row twice from TMEM (max, then exponentials), writes P_j in
//    fp16 to 128-byte-swizzled shared memory, and keeps the running max m, sum l and the
//    output row O in fp32 registers;
//  * PV_j = P_j V_j (K = 128 keys, N = head_dim, V read as an MN-major operand) lands in a
//    second pair of TMEM buffers; the softmax merges it as O = alpha_j O + PV_j with
//    alpha_j = exp2(m_{j-1} - m_j), and at the end divides by l.
// All waits are bounded (device_common.cuh); nothing traps.
#include <atomic>

#include "device_common.cuh"
#include "kernels.h"

namespace gsr {
namespace {

template <int D_, int G_>
struct AttnCfg {
    static constexpr int D = D_;                      // head dim: 64 or 128
    static constexpr int BQ = 128, BKV = 128;
    static constexpr int DCH = D / 64;                // 64-column (128-byte) chunks per row
    static constexpr int CHUNK_BYTES = 128 * 128;     // one 128-row chunk: 16 KB
    static constexpr int Q_BYTES = BQ * D * 2;
    static constexpr int KV_BYTES = BKV * D * 2;
    static constexpr int P_BYTES = BQ * BKV * 2;      // 32 KB: two 64-key chunks
    static constexpr int G = G_;                      // softmax warp groups per query row
    static constexpr int SM_THREADS = 128 * G;        // softmax threads
    static constexpr int NUM_THREADS = 64 + SM_THREADS;
    static constexpr int KEYS_PER_G = BKV / G;        // keys of a row each group owns
    static constexpr int DCOLS_PER_G = D / G;         // output columns each group accumulates
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;
    static constexpr int OFF_P = OFF_V + 2 * KV_BYTES;
    static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
    static constexpr int NUM_BARS = 1 + 9 * 2 + 1;
    // three rotating slots of 128 row maxima, order-encoded as int for shared atomicMax
    static constexpr int MAX_SLOTS = 3;
    static constexpr int OFF_MAXP = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_MISC = OFF_MAXP + MAX_SLOTS * BQ * 4;
    // no alignment slack: the window is declared 1024-byte aligned and the kernel checks it
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int TMEM_COLS = 512;             // S 2 x 128, PV 2 x D
    static constexpr uint32_t T_S = 0, T_PV = 256;
    static constexpr uint32_t IDESC_S = idesc_f16_f32(BQ, BKV, false, false);   // Q, K both K-major
    static constexpr uint32_t IDESC_PV = idesc_f16_f32(BQ, D, false, true);     // P K-major, V MN-major

    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static_assert(G == 2 || G == 4, "two or four softmax groups");
    static_assert(KEYS_PER_G % 32 == 0 && DCOLS_PER_G % 16 == 0, "TMEM load widths");
    static_assert((G - 1) * BQ * 4 <= 2 * P_BYTES, "row-sum exchange lives in the P buffers");
    static_assert(SMEM_BYTES <= 232448, "exceeds the per-CTA shared-memory limit");
    static_assert(T_PV + 2 * D <= TMEM_COLS, "TMEM budget");
};

// Order-preserving map of fp32 to int (a < b as floats <=> enc(a) < enc(b) as ints, NaN
// aside), so that shared-memory atomicMax takes the maximum of floats; it is its own inverse.
__device__ __forceinline__ int ord_enc(float f) {
    const int i = __float_as_int(f);
    return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float ord_dec(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff); }

// Loads 32 consecutive TMEM columns of this warp's 32 lanes into r[at .. at+31] (or 16).
template <int W, int N>
__device__ __forceinline__ void tmem_ld_at(uint32_t taddr, uint32_t (&r)[N], int at) {
    static_assert(W == 32 || W == 16, "load width");
    if constexpr (W == 32)
        tmem_ld_32x32b_x32(taddr, *reinterpret_cast<uint32_t(*)[32]>(r + at));
    else
        tmem_ld_32x32b_x16(taddr, *reinterpret_cast<uint32_t(*)[16]>(r + at));
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
    gsr_attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    constexpr int D = Cfg::D;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {                // the 128-byte-swizzled operands need it
        if (threadIdx.x == 0) atomicCAS(p.err, 0, kDevErrKernelAttention | kDevErrLayout);
        return;
    }
    uint8_t* smem = smem_raw;
    const uint32_t sb = smem_u32(smem);

    // barriers: 0 qfull | 1+s kfull | 3+s kempty | 5+s vfull | 7+s vempty | 9+s sfull |
    //           11+s sempty | 13+s pfull | 15+s pvfull | 17+s pvempty | 19 drain
    auto bar = [&](int i) { return sb + Cfg::OFF_BAR + 8u * i; };
    const uint32_t qfull = bar(0), drain = bar(19);
    auto kfull = [&](int s) { return bar(1 + s); };
    auto kempty = [&](int s) { return bar(3 + s); };
    auto vfull = [&](int s) { return bar(5 + s); };
    auto vempty = [&](int s) { return bar(7 + s); };
    auto sfull = [&](int s) { return bar(9 + s); };
    auto sempty = [&](int s) { return bar(11 + s); };
    auto pfull = [&](int s) { return bar(13 + s); };
    auto pvfull = [&](int s) { return bar(15 + s); };
    auto pvempty = [&](int s) { return bar(17 + s); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_qt = (p.Sq + Cfg::BQ - 1) / Cfg::BQ;
    const int qt = blockIdx.x % n_qt;
    const int bh = blockIdx.x / n_qt;
    const int q0 = qt * Cfg::BQ;
    // key tiles this query tile needs (causal: keys k <= q + offset only)
    int kv_end = p.Skv;
    if (p.causal) kv_end = min(p.Skv, q0 + Cfg::BQ + p.causal_offset);
    const int nkv = kv_end > 0 ? (kv_end + Cfg::BKV - 1) / Cfg::BKV : 0;

    if (threadIdx.x == 0) {
        mbar_init(qfull, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(kfull(s), 1);
            mbar_init(kempty(s), 1);
            mbar_init(vfull(s), 1);
            mbar_init(vempty(s), 1);
            mbar_init(sfull(s), 1);
            mbar_init(sempty(s), Cfg::SM_THREADS);
            mbar_init(pfull(s), Cfg::SM_THREADS);
            mbar_init(pvfull(s), 1);
            mbar_init(pvempty(s), Cfg::SM_THREADS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0u;
        fence_mbarrier_init();
    }
    for (int i = threadIdx.x; i < Cfg::MAX_SLOTS * Cfg::BQ; i += Cfg::NUM_THREADS)
        reinterpret_cast<int*>(smem + Cfg::OFF_MAXP)[i] = ord_enc(-INFINITY);
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish_alloc_permit();
    }
    tcgen05_fence_before();
    __syncthreads();
    tcgen05_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Waiter w{p.err, p.timeout_ns, abort_flag, kDevErrKernelAttention};

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && nkv > 0) {
            const uint64_t pol = l2_policy_evict_last();   // K and V are read by every query tile
            uint32_t armed = 0, armed_parity = 0;          // bit 0 Q, bits 1-2 K, bits 3-4 V
            const bool drop_q = (p.test_flags & kTestDropFirstLoad) && blockIdx.x == 0;
            if (!drop_q) {
                mbar_arrive_expect_tx(qfull, Cfg::Q_BYTES);
#pragma unroll
                for (int c = 0; c < Cfg::DCH; ++c)
                    tma_load_3d(sb + Cfg::OFF_Q + c * Cfg::CHUNK_BYTES, &tmQ, qfull, c * 64, q0, bh, pol);
                armed |= 1u;
            }
            for (int j = 0; j < nkv; ++j) {
                const int s = j & 1;
                const uint32_t ph = (j >> 1) & 1u;
                if (!w.wait(kempty(s), ph ^ 1u, kDevErrProducerEmpty)) break;
                mbar_arrive_expect_tx(kfull(s), Cfg::KV_BYTES);
#pragma unroll
                for (int c = 0; c < Cfg::DCH; ++c)
                    tma_load_3d(sb + Cfg::OFF_K + s * Cfg::KV_BYTES + c * Cfg::CHUNK_BYTES, &tmK, kfull(s),
                                c * 64, j * Cfg::BKV, bh, pol);
                armed |= 2u << s;
                armed_parity = (armed_parity & ~(2u << s)) | (ph << (1 + s));
                if (!w.wait(vempty(s), ph ^ 1u, kDevErrProducerEmpty)) break;
                mbar_arrive_expect_tx(vfull(s), Cfg::KV_BYTES);
#pragma unroll
                for (int c = 0; c < Cfg::DCH; ++c)
                    tma_load_3d(sb + Cfg::OFF_V + s * Cfg::KV_BYTES + c * Cfg::CHUNK_BYTES, &tmV, vfull(s),
                                c * 64, j * Cfg::BKV, bh, pol);
                armed |= 8u << s;
                armed_parity = (armed_parity & ~(8u << s)) | (ph << (3 + s));
            }
            // every copy started must land before the CTA may exit
            if (armed & 1u) w.drain(qfull, 0);
            for (int s = 0; s < 2; ++s) {
                if (armed & (2u << s)) w.drain(kfull(s), (armed_parity >> (1 + s)) & 1u);
                if (armed & (8u << s)) w.drain(vfull(s), (armed_parity >> (3 + s)) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && nkv > 0) {
            bool ok = w.wait(qfull, 0, kDevErrMmaFull);
            for (int j = 0; ok && j <= nkv; ++j) {
                if (j < nkv) {
                    // S_j = Q K_j^T into S buffer j & 1
                    const int s = j & 1;
                    const uint32_t ph = (j >> 1) & 1u;
                    if (!w.wait(kfull(s), ph, kDevErrMmaFull) ||
                        !w.wait(sempty(s), ph ^ 1u, kDevErrMmaAccEmpty)) {
                        ok = false;
                        break;
                    }
                    tcgen05_fence_after();
                    const uint32_t q_s = sb + Cfg::OFF_Q;
                    const uint32_t k_s = sb + Cfg::OFF_K + s * Cfg::KV_BYTES;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = (k >> 2) * Cfg::CHUNK_BYTES + (k & 3) * 32;
                        mma_f16_ss(tmem_base + Cfg::T_S + s * 128, smem_desc_sw128(q_s + off, 16, 1024),
                                   smem_desc_sw128(k_s + off, 16, 1024), Cfg::IDESC_S, k > 0 ? 1u : 0u);
                    }
                    mma_commit(kempty(s));
                    mma_commit(sfull(s));
                }
                if (j >= 1) {
                    // PV_{j-1} = P_{j-1} V_{j-1} into PV buffer (j-1) & 1
                    const int t = j - 1, s = t & 1;
                    const uint32_t ph = (t >> 1) & 1u;
                    if (!w.wait(pfull(s), ph, kDevErrMmaFull) || !w.wait(vfull(s), ph, kDevErrMmaFull) ||
                        !w.wait(pvempty(s), ph ^ 1u, kDevErrMmaAccEmpty)) {
                        ok = false;
                        break;
                    }
                    tcgen05_fence_after();
                    const uint32_t p_s = sb + Cfg::OFF_P + s * Cfg::P_BYTES;
                    const uint32_t v_s = sb + Cfg::OFF_V + s * Cfg::KV_BYTES;
#pragma unroll
                    for (int k = 0; k < Cfg::BKV / 16; ++k) {
                        // P: K-major, keys contiguous; V: MN-major, 64-column chunks 16 KB apart,
                        // 16 key rows = 2048 bytes per k step
                        const uint64_t ad =
                            smem_desc_sw128(p_s + (k >> 2) * Cfg::CHUNK_BYTES + (k & 3) * 32, 16, 1024);
                        const uint64_t bd = smem_desc_sw128(v_s + k * 2048, Cfg::CHUNK_BYTES, 1024);
                        mma_f16_ss(tmem_base + Cfg::T_PV + s * D, ad, bd, Cfg::IDESC_PV, k > 0 ? 1u : 0u);
                    }
                    mma_commit(vempty(s));
                    mma_commit(pvfull(s));
                }
            }
            mma_commit(drain);
            w.drain(drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + output (warps 2..)
        constexpr int G = Cfg::G;
        constexpr int KG = Cfg::KEYS_PER_G;
        constexpr int DG = Cfg::DCOLS_PER_G;
        constexpr int LDW = DG % 32 == 0 ? 32 : 16;  // TMEM load width of the PV merge
        const int quad = warp & 3;
        const int g = (warp - 2) >> 2;               // softmax group
        const int r = quad * 32 + lane;              // query row in the tile == TMEM lane
        const int qi = q0 + r;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
        const bool scale_pos = p.scale_log2 >= 0.0f;
        const float sl2 = p.scale_log2;
        float o[DG];
#pragma unroll
        for (int d = 0; d < DG; ++d) o[d] = 0.0f;
        float m = -INFINITY, l = 0.0f, a_prev = 1.0f;
        bool ok = true;

        // O (this group's columns) = a_prev O + PV_t.  A warp vote keeps the TMEM loads
        // warp-uniform; a failed wait is carried into the next block-wide vote, so every
        // softmax thread takes the same number of barrier-1 steps and leaves the loop together.
        auto merge_pv = [&](int t) -> bool {
            const int s = t & 1;
            const bool got = __all_sync(0xffffffffu, w.wait(pvfull(s), (t >> 1) & 1u, kDevErrEpilogueFull));
            if (!got) return false;
            tcgen05_fence_after();
            uint32_t rr[DG];
#pragma unroll
            for (int c = 0; c < DG / LDW; ++c)
                tmem_ld_at<LDW>(lane_base + Cfg::T_PV + s * D + g * DG + c * LDW, rr, c * LDW);
            tmem_ld_wait(rr);
#pragma unroll
            for (int i = 0; i < DG; i += 2)
                ffma2(o[i], o[i + 1], o[i], o[i + 1], a_prev, a_prev, __uint_as_float(rr[i]),
                      __uint_as_float(rr[i + 1]));
            tcgen05_fence_before();
            mbar_arrive(pvempty(s));
            return true;
        };

        int* maxp = reinterpret_cast<int*>(smem + Cfg::OFF_MAXP);
        int slot = 0;                                // this tile's row-maximum slot: j % 3
        for (int j = 0; j < nkv; ++j) {
            const int s = j & 1;
            const int next_slot = slot == Cfg::MAX_SLOTS - 1 ? 0 : slot + 1;
            const bool got = __all_sync(0xffffffffu, w.wait(sfull(s), (j >> 1) & 1u, kDevErrEpilogueFull));
            tcgen05_fence_after();
            const uint32_t s_col = lane_base + Cfg::T_S + s * 128 + g * KG;
            const int k0 = j * Cfg::BKV + g * KG;        // first key this thread owns
            const int k_lim = p.causal ? min(p.Skv, qi + p.causal_offset + 1) : p.Skv;   // keys < k_lim
            const bool masked = k0 + KG > k_lim;         // only the diagonal / last tile of a row
            // pass 1: maximum of this thread's KG scores (scaled, masked, log2 units); pass 2
            // reads them again from TMEM, which is cheaper than holding them in registers over
            // the exchange.  `masked` differs between rows of one warp on a diagonal tile, so
            // the TMEM loads (.sync.aligned) stay outside the branch.
            uint32_t sv[KG];
            float mt = -INFINITY;
            if (got) {
#pragma unroll
                for (int c = 0; c < KG / 32; ++c) tmem_ld_at<32>(s_col + c * 32, sv, c * 32);
                tmem_ld_wait(sv);
                if (!masked) {
                    float e0 = scale_pos ? -INFINITY : INFINITY, e1 = e0, e2 = e0, e3 = e0;
                    if (scale_pos) {
#pragma unroll
                        for (int i = 0; i < KG; i += 8) {
                            e0 = max3f(e0, __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]));
                            e1 = max3f(e1, __uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3]));
                            e2 = max3f(e2, __uint_as_float(sv[i + 4]), __uint_as_float(sv[i + 5]));
                            e3 = max3f(e3, __uint_as_float(sv[i + 6]), __uint_as_float(sv[i + 7]));
                        }
                        mt = max3f(fmaxf(e0, e1), e2, e3) * sl2;
                    } else {
#pragma unroll
                        for (int i = 0; i < KG; i += 8) {
                            e0 = min3f(e0, __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]));
                            e1 = min3f(e1, __uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3]));
                            e2 = min3f(e2, __uint_as_float(sv[i + 4]), __uint_as_float(sv[i + 5]));
                            e3 = min3f(e3, __uint_as_float(sv[i + 6]), __uint_as_float(sv[i + 7]));
                        }
                        mt = min3f(fminf(e0, e1), e2, e3) * sl2;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < KG; ++i)
                        if (k0 + i < k_lim) mt = fmaxf(mt, __uint_as_float(sv[i]) * sl2);
                }
            }
            // row maximum over the groups: shared atomicMax into this tile's slot.  Slot j%3 was
            // last read at tile j-3 (before barrier j-2) and is reset by group 0 at tile j-1,
            // i.e. after barrier j-2 and before barrier j-1, so neither the reset nor the
            // maxima of tile j can meet an older reader or writer.
            if (g == 0) maxp[next_slot * Cfg::BQ + r] = ord_enc(-INFINITY);
            atomicMax(&maxp[slot * Cfg::BQ + r], ord_enc(mt));
            if (!named_bar_and(1, Cfg::SM_THREADS, got && ok)) {
                ok = false;
                break;
            }
            mt = ord_dec(maxp[slot * Cfg::BQ + r]);
            slot = next_slot;
            const float m_new = fmaxf(m, mt);
            const float alpha = (m_new == -INFINITY) ? 1.0f : ex2_approx(m - m_new);
            const float neg_m = (m_new == -INFINITY) ? 0.0f : -m_new;
            // pass 2: P = 2^(x - m_new) in fp16 into shared memory, 128-byte-swizzled K-major
            uint8_t* prow = smem + Cfg::OFF_P + s * Cfg::P_BYTES + r * 128;
            float ls0 = 0.0f, ls1 = 0.0f;
#pragma unroll
            for (int c = 0; c < KG / 32; ++c) {
                const int kc = g * KG + c * 32;          // first key of this 32-key slice in the tile
                uint32_t sr[32];
                tmem_ld_at<32>(s_col + c * 32, sr, 0);
                tmem_ld_wait(sr);
                uint32_t packed[16];
                if (!masked) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float x0, x1;
                        ffma2(x0, x1, __uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]),
                              sl2, sl2, neg_m, neg_m);
                        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        fadd2(ls0, ls1, p0, p1);
                        __half2 h = __floats2half2_rn(p0, p1);
                        packed[i] = *reinterpret_cast<uint32_t*>(&h);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int kk = k0 + c * 32 + 2 * i;
                        float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * i]), sl2, neg_m));
                        float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * i + 1]), sl2, neg_m));
                        if (kk >= k_lim || m_new == -INFINITY) p0 = 0.0f;
                        if (kk + 1 >= k_lim || m_new == -INFINITY) p1 = 0.0f;
                        ls0 += p0;
                        ls1 += p1;
                        __half2 h = __floats2half2_rn(p0, p1);
                        packed[i] = *reinterpret_cast<uint32_t*>(&h);
                    }
                }
                // keys kc .. kc+31: 64-key chunk kc/64, 16-byte pieces ((kc%64)/8) .. +3, swizzled by row
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int piece = ((kc & 63) >> 3) + t;
                    uint4 v;
                    v.x = packed[4 * t];
                    v.y = packed[4 * t + 1];
                    v.z = packed[4 * t + 2];
                    v.w = packed[4 * t + 3];
                    *reinterpret_cast<uint4*>(prow + (kc >> 6) * Cfg::CHUNK_BYTES + ((piece ^ (r & 7)) << 4)) = v;
                }
            }
            tcgen05_fence_before();
            mbar_arrive(sempty(s));          // S buffer free for S_{j+2}
            fence_proxy_async_smem();
            mbar_arrive(pfull(s));           // P_j ready for the MMA
            l = l * alpha + (ls0 + ls1);     // this group's part of the row sum
            m = m_new;
            if (j >= 1 && !merge_pv(j - 1)) ok = false;
            a_prev = alpha;
        }
        if (ok && nkv > 0) ok = merge_pv(nkv - 1);
        // the row sum: group 0 adds the other groups' parts (one exchange per kernel) in the P
        // buffers, idle once the last PV product has completed (every thread waited for it)
        float* lpart = reinterpret_cast<float*>(smem + Cfg::OFF_P);
        if (g > 0) lpart[(g - 1) * Cfg::BQ + r] = l;
        named_bar_sync(2, Cfg::SM_THREADS);
        if (g == 0) {
            float total = l;
#pragma unroll
            for (int gg = 1; gg < G; ++gg) total += lpart[(gg - 1) * Cfg::BQ + r];
            lpart[r] = total;                // publish the full sum back
        }
        named_bar_sync(2, Cfg::SM_THREADS);
        l = lpart[r];
        // epilogue: this group's output columns, O / l in fp16, and the log-sum-exp
        if (ok && qi < p.Sq) {
            const float inv = l > 0.0f ? 1.0f / l : 0.0f;
            uint4* dst = reinterpret_cast<uint4*>(p.O + ((size_t)bh * p.Sq + qi) * D + g * DG);
#pragma unroll
            for (int c = 0; c < DG / 8; ++c) {
                uint32_t h[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    __half2 v = __floats2half2_rn(o[8 * c + 2 * i] * inv, o[8 * c + 2 * i + 1] * inv);
                    h[i] = *reinterpret_cast<uint32_t*>(&v);
                }
                dst[c] = make_uint4(h[0], h[1], h[2], h[3]);
            }
            if (p.lse && g == 0)
                p.lse[(size_t)bh * p.Sq + qi] = l > 0.0f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
    }

    tcgen05_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tcgen05_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

// O = 0 and lse = -inf for every row (no keys at all).
__global__ void gsr_attention_empty_kernel(__half* O, float* lse, long long rows, int D) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < rows * D) O[i] = __float2half_rn(0.0f);
    if (lse && i < rows) lse[i] = -INFINITY;
}

template <class Cfg>
cudaError_t launch_cfg(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const AttnParams& p, cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(gsr_attention_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    const long long blocks = (long long)((p.Sq + Cfg::BQ - 1) / Cfg::BQ) * p.BH;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    gsr_attention_kernel<Cfg><<<(unsigned)blocks, Cfg::NUM_THREADS, Cfg::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

// Softmax warp groups per query tile for each head size.  Four groups measured slower than
// two at both sizes: at 576 threads a thread gets 96 registers and the per-tile fixed costs
// (TMEM load waits, the exchange) do not shrink with the work per thread.
constexpr int kGroupsD64 = 2;
constexpr int kGroupsD128 = 2;

}  // namespace

cudaError_t launch_attention(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const AttnParams& p, int D, cudaStream_t stream) {
    if (D == 64) return launch_cfg<AttnCfg<64, kGroupsD64>>(tmQ, tmK, tmV, p, stream);
    if (D == 128) return launch_cfg<AttnCfg<128, kGroupsD128>>(tmQ, tmK, tmV, p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attention_empty(__half* O, float* lse, long long rows, int D, cudaStream_t stream) {
    const long long n = rows * D > rows ? rows * D : rows;
    const long long blocks = (n + 255) / 256;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    gsr_attention_empty_kernel<<<(unsigned)blocks, 256, 0, stream>>>(O, lse, rows, D);
    return cudaGetLastError();
}

}  // namespace gsr
