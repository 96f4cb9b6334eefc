// attention_fwd.cu - attention forward on sm_103a:  O = softmax(scale * Q K^T [causal]) V.
//
// The FlashAttention kernel of the aikraft.ru TileLang tutorial survey ("TileLang: создание
// высокопроизводительных GPU-ядер", section 6 "FlashAttention: Слияние внимания"): tiles of
// queries, keys and values, no materialised score matrix, online softmax (running row
// maxima, normalisation sums, rescaling factors), causal masking, copies pipelined with the
// matrix products.  Its thread roles follow "TileLang异步协作终极指南" (producers load K/V, one
// role computes QK^T, another the softmax and the output), rebuilt on tcgen05:
//
//  * one CTA per (two 128-query tiles, batch x head); 320 threads: warp 0 issues TMA copies
//    (both Q tiles once, then K_j with V_{j-1} into a 2-entry ring, one barrier per entry, so
//    the MMA issuer waits once per key tile for both), warp 1 issues every MMA from
//    one lane, warps 2-5 run the softmax of query tile 0 and warps 6-9 that of tile 1, one
//    thread per query row (= TMEM lane) over all 128 keys of a key tile;
//  * per query tile q, S_q(j) = Q_q K_j^T (M 128, N 128 keys, K = head_dim) lands in a
//    128-column TMEM region; the softmax writes P_q(j) in fp16 over the last 64 columns of
//    that same region (tcgen05.st), and PV_q(j) = P_q(j) V_j reads P from TMEM (A operand)
//    and V from shared memory (MN-major B operand), accumulating O_q in TMEM;
//  * the MMA issue order PV_q(j-1), S_q(j) keeps each query tile's stream ordered: when
//    S_q(j) completes, PV_q(j-1) has too, so O_q is final for a rescale and P_q(j-1) has been
//    read before S_q(j) overwrites it.  The two query tiles alternate on the tensor core:
//    while one softmax group exponentiates, the other tile's products run;
//  * the running maximum m used for the exponentials moves only when a tile's maximum
//    exceeds it by more than 2^8 (then O_q and l are rescaled by 2^(m_old - m_new) first), so
//    P <= 256 in fp16 and O / l is unchanged: P and l use the same m.  lse = m + log2 l.
// All waits are bounded (device_common.cuh); nothing traps.
#include <atomic>

#include "device_common.cuh"
#include "attention.h"
#include "kernels.h"

namespace gsr {
namespace {

template <int D_>
struct AttnCfg {
    static constexpr int D = D_;                      // head dim: 64 or 128
    static constexpr int BQ = 128, BKV = 128;         // rows of a query tile / keys of a key tile
    static constexpr int NQ = 2;                      // query tiles per CTA
    static constexpr int DCH = D / 64;                // 64-column (128-byte) chunks per row
    static constexpr int CHUNK_BYTES = 128 * 128;     // one 128-row chunk: 16 KB
    static constexpr int Q_BYTES = BQ * D * 2;
    static constexpr int KV_BYTES = BKV * D * 2;
    static constexpr int SM_THREADS = 128 * NQ;       // softmax threads
    static constexpr int NUM_THREADS = 64 + SM_THREADS;
    // Q buffers: at D = 64 a second set (32 KB) fits, so the next item's Q loads while the
    // current item still reads its own; at D = 128 there is no room (one set, reloaded once the
    // last Q K^T products of an item have read it)
    static constexpr int QBUF = D == 64 ? 2 : 1;
    // ring of 2 entries; entry e holds K_e and V_{e-1}, the two tiles step e consumes
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + QBUF * NQ * Q_BYTES;
    static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;
    static constexpr int OFF_BAR = OFF_V + 2 * KV_BYTES;
    static constexpr int NUM_BARS = 17 + 2 * (QBUF - 1);
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    // no alignment slack: the window is declared 1024-byte aligned and the kernel checks it
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int TMEM_COLS = 512;
    // TMEM columns: S_q / P_q at 128 q, O_q at 256 + D q
    static constexpr uint32_t T_S = 0, T_O = 256;
    static constexpr uint32_t P_COL = 64;             // P_q: upper 64 columns of the S_q region
    static constexpr uint32_t IDESC_S = idesc_f16_f32(BQ, BKV, false, false);   // Q, K both K-major
    static constexpr uint32_t IDESC_PV = idesc_f16_f32(BQ, D, false, true);     // P (TMEM), V MN-major
    // the exponent base moves only when a tile's maximum is more than this above it (log2 units)
    static constexpr float RESCALE_LOG2 = 8.0f;

    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static_assert(SMEM_BYTES <= 232448, "exceeds the per-CTA shared-memory limit");
    static_assert(T_O + NQ * D <= TMEM_COLS, "TMEM budget");
};

template <class Cfg>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
    gsr_attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    constexpr int D = Cfg::D;
    constexpr int NQ = Cfg::NQ;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {                // the 128-byte-swizzled operands need it
        if (threadIdx.x == 0) atomicCAS(p.err, 0, kDevErrKernelAttention | kDevErrLayout);
        return;
    }
    uint8_t* smem = smem_raw;
    const uint32_t sb = smem_u32(smem);

    // barriers: 0 qfull | 1 qfree | 2+s full | 4+s empty | 6+q sfull | 8+q pfull | 10+q odone |
    // 12+i item published | 14+i item read | 16 drain | 17 qfull, 18 qfree of the second Q set
    auto bar = [&](int i) { return sb + Cfg::OFF_BAR + 8u * i; };
    const uint32_t drain = bar(16);
    auto qfull = [&](int b) { return bar(b == 0 ? 0 : 17); };
    auto qfree = [&](int b) { return bar(b == 0 ? 1 : 18); };
    auto full = [&](int s) { return bar(2 + s); };
    auto empty = [&](int s) { return bar(4 + s); };
    auto sfull = [&](int q) { return bar(6 + q); };
    auto pfull = [&](int q) { return bar(8 + q); };
    auto odone = [&](int q) { return bar(10 + q); };
    auto item_pub = [&](int i) { return bar(12 + i); };
    auto item_read = [&](int i) { return bar(14 + i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_MISC + 4);
    volatile int* item_box = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 8);   // 2 slots

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_qb = (p.Sq + NQ * Cfg::BQ - 1) / (NQ * Cfg::BQ);

    // Work item -> (query block, batch x head) and the key tiles each query tile needs.  The
    // (batch x head) slices are taken in groups of head_group; within a group the latest query
    // blocks of all its heads (the most keys under a causal mask) come first, then the ones
    // before them, so the items fetched last are the shortest and the CTAs drain together,
    // while the group's K and V stay in L2.  head_group = 1 walks one head at a time.
    struct Item {
        int bh, q_base, nkv[NQ], nkv_max;
    };
    auto decode = [&](int item) {
        Item it;
        const int per_group = p.head_group * n_qb;
        const int grp = item / per_group;
        const int r_in = item - grp * per_group;
        const int gsz = min(p.BH - grp * p.head_group, p.head_group);   // the last group may be smaller
        const int qb = n_qb - 1 - r_in / gsz;
        it.bh = grp * p.head_group + r_in % gsz;
        it.q_base = qb * NQ * Cfg::BQ;
        // key tiles each query tile needs (causal: keys k <= q + offset only); nkv[0] <= nkv[1]
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            int kv_end = p.Skv;
            if (p.causal) kv_end = min(p.Skv, it.q_base + (q + 1) * Cfg::BQ + p.causal_offset);
            it.nkv[q] = kv_end > 0 ? (kv_end + Cfg::BKV - 1) / Cfg::BKV : 0;
        }
        it.nkv_max = it.nkv[NQ - 1];
        return it;
    };

    if (threadIdx.x == 0) {
        for (int b = 0; b < Cfg::QBUF; ++b) {
            mbar_init(qfull(b), 1);
            mbar_init(qfree(b), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
            mbar_init(item_pub(s), 1);
            mbar_init(item_read(s), 1 + Cfg::SM_THREADS / 32);   // the MMA lane and every softmax warp
        }
        for (int q = 0; q < NQ; ++q) {
            mbar_init(sfull(q), 1);
            mbar_init(pfull(q), 128);
            mbar_init(odone(q), 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0u;
        fence_mbarrier_init();
    }
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
        // ------------------------------------------------------------ work fetch + TMA producer
        // Takes the next work item from the launch's counter and publishes it to the other roles
        // (a 2-slot box, so it can run one item ahead), then loads the item's Q tiles (once the
        // previous item's last Q K^T products have read theirs) and its ring entries, which
        // continue from the previous item's: entry e of an item holds K_e and V_{e-1}.
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();   // K and V are read by every query block
            uint32_t n_pub = 0, n_q = 0, g = 0;            // items published, Q loads, ring entries
            int last_q0 = -1, last_q1 = -1;                 // Q load number last armed, per set
            uint32_t ring_armed = 0, ring_parity = 0;
            bool drop_q = (p.test_flags & kTestDropFirstLoad) && blockIdx.x == 0;
            while (true) {
                int item = atomicAdd(p.work, 1);
                if (item >= p.num_items) item = -1;
                const uint32_t box = n_pub & 1u;
                // the box's previous item has been read by every role
                if (!w.wait(item_read(box), ((n_pub >> 1) & 1u) ^ 1u, kDevErrProducerEmpty)) break;
                item_box[box] = item;
                mbar_arrive(item_pub(box));          // release: the consumers read the box after
                ++n_pub;
                if (item < 0) break;
                const Item it = decode(item);
                if (it.nkv_max == 0) continue;       // no keys: O = 0 needs no copies
                // Q set n_q % QBUF: free once the item that last used it has read it
                const int qb = (int)(n_q % Cfg::QBUF);
                if (n_q >= (uint32_t)Cfg::QBUF &&
                    !w.wait(qfree(qb), ((n_q - Cfg::QBUF) / Cfg::QBUF) & 1u, kDevErrProducerEmpty))
                    break;
                if (drop_q) {
                    drop_q = false;                  // test hook: this Q is never loaded
                } else {
                    const uint32_t qbase = sb + Cfg::OFF_Q + qb * NQ * Cfg::Q_BYTES;
                    mbar_arrive_expect_tx(qfull(qb), NQ * Cfg::Q_BYTES);
#pragma unroll
                    for (int q = 0; q < NQ; ++q)
#pragma unroll
                        for (int c = 0; c < Cfg::DCH; ++c)
                            tma_load_3d(qbase + q * Cfg::Q_BYTES + c * Cfg::CHUNK_BYTES, &tmQ, qfull(qb),
                                        c * 64, it.q_base + q * Cfg::BQ, it.bh, pol);
                    (qb == 0 ? last_q0 : last_q1) = (int)n_q;
                }
                ++n_q;
                bool ok = true;
                // entry e: K_e (e < nkv_max) and V_{e-1} (e >= 1); the last entry holds only V
                for (int e = 0; e <= it.nkv_max; ++e, ++g) {
                    const int s = (int)(g & 1u);
                    const uint32_t ph = (g >> 1) & 1u;
                    if (!w.wait(empty(s), ph ^ 1u, kDevErrProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const bool has_k = e < it.nkv_max, has_v = e >= 1;
                    mbar_arrive_expect_tx(full(s), (has_k ? Cfg::KV_BYTES : 0) + (has_v ? Cfg::KV_BYTES : 0));
                    if (has_k) {
#pragma unroll
                        for (int c = 0; c < Cfg::DCH; ++c)
                            tma_load_3d(sb + Cfg::OFF_K + s * Cfg::KV_BYTES + c * Cfg::CHUNK_BYTES, &tmK, full(s),
                                        c * 64, e * Cfg::BKV, it.bh, pol);
                    }
                    if (has_v) {
#pragma unroll
                        for (int c = 0; c < Cfg::DCH; ++c)
                            tma_load_3d(sb + Cfg::OFF_V + s * Cfg::KV_BYTES + c * Cfg::CHUNK_BYTES, &tmV, full(s),
                                        c * 64, (e - 1) * Cfg::BKV, it.bh, pol);
                    }
                    ring_armed |= 1u << s;
                    ring_parity = (ring_parity & ~(1u << s)) | (ph << s);
                }
                if (!ok) break;
            }
            // The launch's fetch counter: this CTA takes no more items.  The last CTA to get here
            // (after every other one has taken its last item) resets the counter for the next
            // launch on the stream.
            __threadfence();
            if (atomicAdd(p.work + 1, 1) == (int)gridDim.x - 1) {
                atomicExch(p.work, 0);
                atomicExch(p.work + 1, 0);
            }
            // every copy started must land before the CTA may exit
            if (last_q0 >= 0) w.drain(qfull(0), (uint32_t)(last_q0 / Cfg::QBUF) & 1u);
            if (last_q1 >= 0) w.drain(qfull(1), (uint32_t)(last_q1 / Cfg::QBUF) & 1u);
            for (int s = 0; s < 2; ++s)
                if (ring_armed & (1u << s)) w.drain(full(s), (ring_parity >> s) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t n_item = 0, n_q = 0, g = 0;      // items taken, items with keys, ring entries
            uint32_t pv_n0 = 0u, pv_n1 = 0u;          // pfull phases waited for, per query tile
            bool ok = true;
            while (ok) {
                const uint32_t box = n_item & 1u;
                if (!w.wait(item_pub(box), (n_item >> 1) & 1u, kDevErrMmaFull)) break;
                const int item = item_box[box];
                mbar_arrive(item_read(box));
                ++n_item;
                if (item < 0) break;
                const Item it = decode(item);
                if (it.nkv_max == 0) continue;
                const int qb = (int)(n_q % Cfg::QBUF);      // this item's Q set (as the producer's)
                if (!w.wait(qfull(qb), (n_q / Cfg::QBUF) & 1u, kDevErrMmaFull)) break;
                ++n_q;
                tcgen05_fence_after();
                // PV_q(t) = P_q(t) V_t accumulated into O_q; V_t sits in the ring slot `s` the
                // caller has waited for.  After its last key tile, O_q is published to the softmax.
                auto issue_pv = [&](int q, int t, int s) -> bool {
                    uint32_t& pv_n = q == 0 ? pv_n0 : pv_n1;
                    if (!w.wait(pfull(q), pv_n & 1u, kDevErrMmaFull)) return false;
                    ++pv_n;
                    tcgen05_fence_after();
                    const uint32_t v_s = sb + Cfg::OFF_V + s * Cfg::KV_BYTES;
                    const uint32_t p_t = tmem_base + Cfg::T_S + q * 128 + Cfg::P_COL;
#pragma unroll
                    for (int k = 0; k < Cfg::BKV / 16; ++k) {
                        // P: 16 keys = 8 TMEM columns per step; V: MN-major, 64-column chunks 16 KB
                        // apart, 16 key rows = 2048 bytes per step
                        const uint64_t bd = smem_desc_sw128(v_s + k * 2048, Cfg::CHUNK_BYTES, 1024);
                        mma_f16_ts(tmem_base + Cfg::T_O + q * D, p_t + k * 8, bd, Cfg::IDESC_PV,
                                   (t > 0 || k > 0) ? 1u : 0u);
                    }
                    if (t == (q == 0 ? it.nkv[0] : it.nkv[NQ - 1]) - 1) mma_commit(odone(q));
                    return true;
                };
                for (int j = 0; ok && j < it.nkv_max; ++j, ++g) {
                    const int s = (int)(g & 1u);
                    if (!w.wait(full(s), (g >> 1) & 1u, kDevErrMmaFull)) {   // K_j and V_{j-1}
                        ok = false;
                        break;
                    }
                    tcgen05_fence_after();
                    const uint32_t k_s = sb + Cfg::OFF_K + s * Cfg::KV_BYTES;
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        if (j > 0 && j <= it.nkv[q] && !(ok = issue_pv(q, j - 1, s))) break;
                        if (j < it.nkv[q]) {
                            // S_q(j) = Q_q K_j^T, over P_q(j-1) (read by the PV just issued, or by
                            // the previous item's last PV_q: one thread's products complete in order)
                            const uint32_t q_s = sb + Cfg::OFF_Q + (qb * NQ + q) * Cfg::Q_BYTES;
#pragma unroll
                            for (int k = 0; k < D / 16; ++k) {
                                const uint32_t off = (k >> 2) * Cfg::CHUNK_BYTES + (k & 3) * 32;
                                mma_f16_ss(tmem_base + Cfg::T_S + q * 128, smem_desc_sw128(q_s + off, 16, 1024),
                                           smem_desc_sw128(k_s + off, 16, 1024), Cfg::IDESC_S, k > 0 ? 1u : 0u);
                            }
                            mma_commit(sfull(q));
                        }
                    }
                    if (!ok) break;
                    // every Q K^T product of the item is issued: Q may be replaced once they finish
                    if (j == it.nkv_max - 1) mma_commit(qfree(qb));
                    mma_commit(empty(s));
                }
                if (!ok) break;
                // last entry: V_{nkv_max-1} for the final products of the tiles that need it
                {
                    const int s = (int)(g & 1u);
                    if (!w.wait(full(s), (g >> 1) & 1u, kDevErrMmaFull)) break;
                    tcgen05_fence_after();
#pragma unroll
                    for (int q = 0; q < NQ; ++q)
                        if (ok && it.nkv[q] == it.nkv_max) ok = issue_pv(q, it.nkv_max - 1, s);
                    if (!ok) break;
                    mma_commit(empty(s));
                    ++g;
                }
            }
            mma_commit(drain);
            w.drain(drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + output (warps 2-9)
        const int q = (warp - 2) >> 2;               // query tile of this group
        const int quad = warp & 3;
        const int r = quad * 32 + lane;              // query row in the tile == TMEM lane
        const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
        const uint32_t s_col = lane_base + Cfg::T_S + q * 128;
        const uint32_t o_col = lane_base + Cfg::T_O + q * D;
        const bool scale_pos = p.scale_log2 >= 0.0f;
        const float sl2 = p.scale_log2;
        uint32_t n_item = 0, s_n = 0, o_n = 0;       // items taken; sfull / odone phases waited for
        bool ok = true;
        while (ok) {
            const uint32_t box = n_item & 1u;
            if (!__all_sync(0xffffffffu, w.wait(item_pub(box), (n_item >> 1) & 1u, kDevErrEpilogueFull))) break;
            const int item = item_box[box];
            __syncwarp();
            if (lane == 0) mbar_arrive(item_read(box));
            ++n_item;
            if (item < 0) break;
            const Item it = decode(item);
            const int qi = it.q_base + q * Cfg::BQ + r;
            const int k_lim = p.causal ? min(p.Skv, qi + p.causal_offset + 1) : p.Skv;   // keys < k_lim
            const int nkv_q = q == 0 ? it.nkv[0] : it.nkv[NQ - 1];
            float m = -INFINITY, l = 0.0f;

            for (int j = 0; j < nkv_q; ++j) {
                // the warp agrees before any .sync.aligned TMEM access
                if (!__all_sync(0xffffffffu, w.wait(sfull(q), s_n & 1u, kDevErrEpilogueFull))) {
                    ok = false;
                    break;
                }
                ++s_n;
                tcgen05_fence_after();
                const int k0 = j * Cfg::BKV;
                const bool masked = k0 + Cfg::BKV > k_lim;   // only the diagonal / last tile of a row
                // The row's 128 scores are four 32-column chunks c0..c3, all four loaded before
                // one wait.  `masked` differs between rows of one warp on a diagonal tile, so every TMEM
                // access stays outside the branches.
                float e0 = scale_pos ? -INFINITY : INFINITY, e1 = e0, e2 = e0, e3 = e0;
                float mt = -INFINITY;                        // masked tiles: running max, scaled
                auto chunk_max = [&](const uint32_t (&rr)[32], int c) {
                    if (!masked) {
                        if (scale_pos) {
#pragma unroll
                            for (int i = 0; i < 32; i += 8) {
                                e0 = max3f(e0, __uint_as_float(rr[i]), __uint_as_float(rr[i + 1]));
                                e1 = max3f(e1, __uint_as_float(rr[i + 2]), __uint_as_float(rr[i + 3]));
                                e2 = max3f(e2, __uint_as_float(rr[i + 4]), __uint_as_float(rr[i + 5]));
                                e3 = max3f(e3, __uint_as_float(rr[i + 6]), __uint_as_float(rr[i + 7]));
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; i += 8) {
                                e0 = min3f(e0, __uint_as_float(rr[i]), __uint_as_float(rr[i + 1]));
                                e1 = min3f(e1, __uint_as_float(rr[i + 2]), __uint_as_float(rr[i + 3]));
                                e2 = min3f(e2, __uint_as_float(rr[i + 4]), __uint_as_float(rr[i + 5]));
                                e3 = min3f(e3, __uint_as_float(rr[i + 6]), __uint_as_float(rr[i + 7]));
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (k0 + c * 32 + i < k_lim) mt = fmaxf(mt, __uint_as_float(rr[i]) * sl2);
                    }
                };
                // pass 1: maximum of the scaled, masked scores of the row, in log2 units.  The whole
                // row (128 scores) comes into registers with one wait and stays there for pass 2.
                uint32_t sc0[32], sc1[32], sc2[32], sc3[32];
                tmem_ld_32x32b_x32(s_col + 0, sc0);
                tmem_ld_32x32b_x32(s_col + 32, sc1);
                tmem_ld_32x32b_x32(s_col + 64, sc2);
                tmem_ld_32x32b_x32(s_col + 96, sc3);
                tmem_ld_wait(sc0);
                reg_tie(sc1);
                reg_tie(sc2);
                reg_tie(sc3);
                chunk_max(sc0, 0);
                chunk_max(sc1, 1);
                chunk_max(sc2, 2);
                chunk_max(sc3, 3);
                if (!masked)
                    mt = (scale_pos ? max3f(fmaxf(e0, e1), e2, e3) : min3f(fminf(e0, e1), e2, e3)) * sl2;
                // lazy move of the exponent base: only by more than 2^RESCALE_LOG2 (always from -inf)
                float factor = 1.0f;
                const bool bump = mt > m + Cfg::RESCALE_LOG2;
                if (bump) {
                    factor = (m == -INFINITY) ? 0.0f : ex2_approx(m - mt);
                    m = mt;
                }
                l *= factor;
                const float neg_m = (m == -INFINITY) ? 0.0f : -m;
                // pass 2: P = 2^(x - m) in fp16, two keys per column, chunk c to columns
                // 64 + 16c .. +15 of the S region (free: every score is in registers)
                float ls0 = 0.0f, ls1 = 0.0f;
                auto chunk_p = [&](const uint32_t (&rr)[32], int c) {
                    uint32_t packed[16];
                    if (!masked) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float x0, x1;
                            ffma2(x0, x1, __uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1]), sl2, sl2,
                                  neg_m, neg_m);
                            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                            fadd2(ls0, ls1, p0, p1);
                            __half2 h = __floats2half2_rn(p0, p1);
                            packed[i] = *reinterpret_cast<uint32_t*>(&h);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int kk = k0 + c * 32 + 2 * i;
                            float p0 = ex2_approx(fmaf(__uint_as_float(rr[2 * i]), sl2, neg_m));
                            float p1 = ex2_approx(fmaf(__uint_as_float(rr[2 * i + 1]), sl2, neg_m));
                            if (kk >= k_lim || m == -INFINITY) p0 = 0.0f;
                            if (kk + 1 >= k_lim || m == -INFINITY) p1 = 0.0f;
                            ls0 += p0;
                            ls1 += p1;
                            __half2 h = __floats2half2_rn(p0, p1);
                            packed[i] = *reinterpret_cast<uint32_t*>(&h);
                        }
                    }
                    tmem_st_32x32b_x16(s_col + Cfg::P_COL + c * 16, packed);
                };
                chunk_p(sc0, 0);
                chunk_p(sc1, 1);
                chunk_p(sc2, 2);
                chunk_p(sc3, 3);
                if (j > 0 && __any_sync(0xffffffffu, bump)) {
                    // O_q (this warp's rows) *= factor: PV_q(j-1) completed before S_q(j) did, and
                    // PV_q(j) waits for the arrival below; done after pass 2, when the scores are dead
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t rr[32];
                        tmem_ld_32x32b_x32(o_col + c * 32, rr);
                        tmem_ld_wait(rr);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            float y0, y1;
                            fmul2(y0, y1, __uint_as_float(rr[i]), __uint_as_float(rr[i + 1]), factor, factor);
                            rr[i] = __float_as_uint(y0);
                            rr[i + 1] = __float_as_uint(y1);
                        }
                        tmem_st_32x32b_x32(o_col + c * 32, rr);
                    }
                }
                tmem_st_wait();
                tcgen05_fence_before();
                mbar_arrive(pfull(q));           // P_q(j) (and a rescaled O_q) ready for the MMA
                l += ls0 + ls1;
            }
            // output: O_q / l in fp16, and the log-sum-exp.  The next item's first PV_q, which
            // overwrites O_q, waits for this group's next P, issued only after these loads.
            if (ok && nkv_q > 0) {
                ok = __all_sync(0xffffffffu, w.wait(odone(q), o_n & 1u, kDevErrEpilogueFull));
                ++o_n;
                tcgen05_fence_after();
            }
            if (!ok) break;
            const float inv = l > 0.0f ? 1.0f / l : 0.0f;
            uint4* dst = reinterpret_cast<uint4*>(p.O + ((size_t)it.bh * p.Sq + qi) * D);
            if constexpr (D == 64) {
                // the whole row (two 32-column chunks) with one wait: +0.8 % at D = 64; at
                // D = 128 the same, or two chunks per wait, cost 1-3 % (register allocation of
                // the softmax loop), so D = 128 keeps one chunk per wait
                uint32_t ra[32], rb[32];
                if (nkv_q > 0) {
                    tmem_ld_32x32b_x32(o_col, ra);
                    tmem_ld_32x32b_x32(o_col + 32, rb);
                    tmem_ld_wait(ra);
                    reg_tie(rb);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        ra[i] = 0u;
                        rb[i] = 0u;
                    }
                }
                if (qi < p.Sq) {
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const uint32_t* rr = t < 4 ? ra : rb;
                        uint32_t h[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int b = 8 * (t & 3) + 2 * i;
                            __half2 v = __floats2half2_rn(__uint_as_float(rr[b]) * inv, __uint_as_float(rr[b + 1]) * inv);
                            h[i] = *reinterpret_cast<uint32_t*>(&v);
                        }
                        dst[t] = make_uint4(h[0], h[1], h[2], h[3]);
                    }
                }
            } else {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t rr[32];
                    if (nkv_q > 0) {
                        tmem_ld_32x32b_x32(o_col + c * 32, rr);
                        tmem_ld_wait(rr);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) rr[i] = 0u;
                    }
                    if (qi < p.Sq) {
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            uint32_t h[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                __half2 v = __floats2half2_rn(__uint_as_float(rr[8 * t + 2 * i]) * inv,
                                                              __uint_as_float(rr[8 * t + 2 * i + 1]) * inv);
                                h[i] = *reinterpret_cast<uint32_t*>(&v);
                            }
                            dst[c * 4 + t] = make_uint4(h[0], h[1], h[2], h[3]);
                        }
                    }
                }
            }
            if (p.lse && qi < p.Sq)
                p.lse[(size_t)it.bh * p.Sq + qi] = l > 0.0f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
            tcgen05_fence_before();
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
                       const AttnParams& p, int grid, cudaStream_t stream) {
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
    if (grid <= 0 || grid > p.num_items) return cudaErrorInvalidValue;
    gsr_attention_kernel<Cfg><<<(unsigned)grid, Cfg::NUM_THREADS, Cfg::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const AttnParams& p, int D, int grid, cudaStream_t stream) {
    if (D == 64) return launch_cfg<AttnCfg<64>>(tmQ, tmK, tmV, p, grid, stream);
    if (D == 128) return launch_cfg<AttnCfg<128>>(tmQ, tmK, tmV, p, grid, stream);
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
