// gemm_pair.cu - tiled path of C = ReLU(alpha * A.B) on CTA pairs (sm_103a, cta_group::2).
//
// Same operator and epilogue as gemm_tiled.cu ("Tutorial14: 使用TileLang语言编写attention算子",
// section 2 kernel and section 3 formula / tiling / fused epilogue); what changes is how a
// 256 x 256 output tile is shared by the two CTAs (two SMs) of a cluster:
//  * CTA r of the pair loads rows [m0 + 128r, +128) of A and columns [n0 + 128r, +128) of B
//    into its own shared memory, at the same offsets in both CTAs;
//  * one thread of the leader CTA (rank 0) issues tcgen05.mma.cta_group::2 with M = 256,
//    N = 256: the tensor cores of both SMs read both CTAs' A rows and B columns, and each
//    CTA's TMEM receives its 128 rows x 256 columns of the accumulator;
//  * both CTAs' TMA loads count their bytes on the leader's "full" barrier (the leader
//    arms it with the pair's total); the MMA's commits arrive on the "empty" and
//    "accumulator full" barriers of both CTAs at once (multicast); both CTAs' epilogue
//    warps arrive on the leader's "accumulator empty" barrier.
// Each SM thus moves half of B through its shared memory instead of all of it: per k-block
// an SM stages 32 KB (not 48 KB) and its tensor core reads 32 KB (not 48 KB) of operands
// for the same 128 x 256 x 64 of work, which is what limited the single-CTA kernel.
// The persistent pairs walk work units: whole tiles, then, when the last wave would keep at
// most half of the pairs busy, that wave's tiles as two 256 x 128 halves each (an N = 128
// MMA over one 64-column chunk of B per CTA), so that twice as many pairs finish it sooner.
#include <atomic>

#include "device_common.cuh"
#include "kernels.h"

namespace gsr {
namespace {

// 64-wide K sub-blocks per pipeline stage (1 or 2)
constexpr int kPairKsub = 2;

// BN: width of the pair's tile (256, or 128 where 256-wide tiles leave a wave badly filled)
template <int BN_>
struct PairCfg {
    // BK = 64 is one TMA box of K (128 bytes); a stage holds KSUB such sub-blocks, so that the
    // MMA issuer waits once per KSUB * 4 MMAs
    static constexpr int BM = 256, BN = BN_, BK = 64, KSUB = kPairKsub;
    static constexpr int HALF_M = 128, HALF_N = BN / 2;       // per CTA
    static constexpr int NUM_THREADS = 192;
    static constexpr int A_SUB_BYTES = HALF_M * BK * 2;       // 16 KB: one 64-wide K sub-block
    static constexpr int B_CHUNK_BYTES = BK * 64 * 2;         // 8 KB box (64 columns)
    static constexpr int B_SUB_BYTES = BK * HALF_N * 2;       // 16 KB (BN 256) or 8 KB
    static constexpr int A_STAGE_BYTES = KSUB * A_SUB_BYTES;
    static constexpr int B_STAGE_BYTES = KSUB * B_SUB_BYTES;
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;   // per CTA
    static constexpr int C_BUF_BYTES = HALF_M * 64 * 2;       // 16 KB staging chunk
    static constexpr int C_BUFS = 2;
    // as many stages as fit beside the staging buffers (3 x 64 KB at BN 256, 4 x 48 KB at 128)
    static constexpr int STAGES = (232448 - 1024 - 256 - C_BUFS * C_BUF_BYTES) / STAGE_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;                  // two accumulators of BN columns
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE_BYTES;
    static constexpr int OFF_C = OFF_B + STAGES * B_STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_C + C_BUFS * C_BUF_BYTES;
    // full/empty per stage, two accumulator full/empty pairs, the MMA drain, the exit handshake
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 2;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // TMEM base, abort flag, peer's slots
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr uint32_t IDESC = idesc_f16_f32(BM, BN, /*a_mn=*/false, /*b_mn=*/true);
    static constexpr uint32_t IDESC_HALF = idesc_f16_f32(BM, BN / 2, false, true);   // half-width units
    static constexpr uint32_t TEMPTY_ARRIVALS = 8;            // 4 epilogue warps x 2 CTAs
    static constexpr uint32_t SLOT_DROPPED = 0x80000000u;     // handshake word: peer skipped slot 0

    static_assert(BN == 256 || BN == 128, "pair tile width");
    static_assert(STAGES >= 3, "pipeline depth");
    static_assert(SMEM_BYTES <= 232448, "exceeds the per-CTA shared-memory limit");
};

// Work unit u -> tile (mb, nb) and which half of its columns (-1: the whole tile).  Units
// below num_full are whole tiles; each later tile is split into two half-width units.
__device__ __forceinline__ void pair_unit(int u, const TiledParams& p, int& mb, int& nb, int& half) {
    int t = u;
    half = -1;
    if (u >= p.num_full) {
        const int v = u - p.num_full;
        t = p.num_full + (v >> 1);
        half = v & 1;
    }
    raster_tile_coords(t, p.num_m_blocks, p.num_n_blocks, p.group_m, mb, nb);
}

// KIND_SPLIT: the epilogue's chunk loop is compiled once per epilogue kind (no branch on the kind
// per group of values: about half the cycles per chunk, 232 registers instead of 124).  Launches
// of at most two waves of units take it, where the last units' epilogues are not hidden behind
// MMAs; longer ones keep the single copy, whose slower epilogue still hides behind the next
// tile's MMAs and draws less power (under the power cap the split copy lost 0.5-1.7 %).
template <class Cfg, bool KIND_SPLIT>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
    gsr_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const TiledParams p) {
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);

    auto full_bar = [&](int s) { return sb + Cfg::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sb + Cfg::OFF_BAR + 8u * (S + s); };
    auto tfull_bar = [&](int a) { return sb + Cfg::OFF_BAR + 8u * (2 * S + a); };
    auto tempty_bar = [&](int a) { return sb + Cfg::OFF_BAR + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = sb + Cfg::OFF_BAR + 8u * (2 * S + 4);
    const uint32_t exit_bar = sb + Cfg::OFF_BAR + 8u * (2 * S + 5);    // leader's: peer's slot count
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_MISC + 4);
    volatile uint32_t* peer_slots = reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_MISC + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();          // 0: leader, 1: peer
    const int cluster = (int)cluster_id_x();
    const int nclusters = (int)cluster_count_x();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);                // leader: its arrive.expect_tx (pair bytes)
            mbar_init(empty_bar(s), 1);               // multicast commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);               // multicast commit
            mbar_init(tempty_bar(a), Cfg::TEMPTY_ARRIVALS);
        }
        mbar_init(drain_bar, 1);
        mbar_init(exit_bar, 1);                       // the peer producer's remote arrive
        *abort_flag = 0u;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish_alloc_permit_pair();
    }
    // Within the CTA, the thread barrier publishes the TMEM address and the abort flag; across
    // the pair, the cluster barrier only has to order the barrier initialisation, which thread 0
    // released with fence.mbarrier_init before arriving, so its arrive can be relaxed (~800
    // cycles less than a release arrive, per launch).
    tcgen05_fence_before();
    __syncthreads();
    cluster_sync_relaxed();                           // barriers of both CTAs exist from here on
    tcgen05_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Waiter w{p.err, p.timeout_ns, abort_flag, kDevErrKernelTiled};

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (both CTAs)
        // One thread issues every copy: per stage, this CTA's 128 A rows and its 128 B
        // columns (one 3-D box when B is described as 64-column chunks, else two 2-D boxes).
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            const uint64_t pol_b = (p.test_flags & kTestBEvictFirst) ? l2_policy_evict_first()
                                 : (p.test_flags & kTestBEvictNormal) ? l2_policy_evict_normal() : pol;
            uint32_t stage = 0, phase = 0;
            uint32_t slots = 0;           // stage slots taken, in order: slot j is stage j % S
            bool dropped0 = false;        // test hook: slot 0 was taken but never filled
            bool drop_first = ((p.test_flags & kTestDropFirstLoad) && blockIdx.x == 0) ||
                              ((p.test_flags & kTestDropFirstLoadPeer) && blockIdx.x == 1);
            bool ok = true;
            // Serpentine K order: odd waves of units walk K from the end.  A wave's tiles share
            // their A panels with the next wave's (same raster group); read forward twice, the
            // panels (4 MiB each at K = 8192) are gone from L2 before the next wave reaches
            // them, while read back to front the next wave starts on the k-blocks the last one
            // touched most recently (8192^3: DRAM reads 1283 -> 819 MB per launch).  The MMA
            // issuer takes the stages as they come; only the summation order changes.
            const bool serpentine = (p.test_flags & kTestKForward) == 0;
            uint32_t wave = 0;
            for (int u = cluster; ok && u < p.num_units; u += nclusters, ++wave) {
                int mb, nb, half;
                pair_unit(u, p, mb, nb, half);
                const bool backwards = serpentine && (wave & 1u);
                // this CTA's B columns: half of the unit's width (128 or, for a half unit, 64)
                const int cta_cols = half < 0 ? Cfg::HALF_N : Cfg::HALF_N / 2;
                const int chunks = cta_cols / 64;
                const int m_row = mb * Cfg::BM + (int)rank * Cfg::HALF_M;
                const int n_col = nb * Cfg::BN + (half < 0 ? 0 : half * (Cfg::BN / 2)) + (int)rank * cta_cols;
                const uint32_t pair_bytes = 2u * Cfg::KSUB * (Cfg::A_SUB_BYTES + chunks * Cfg::B_CHUNK_BYTES);
                const int n_stages = (p.num_k_blocks + Cfg::KSUB - 1) / Cfg::KSUB;
                for (int kb = 0; kb < n_stages; ++kb) {
                    if (!w.wait(empty_bar(stage), phase ^ 1u, kDevErrProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    if (drop_first) {
                        drop_first = false;   // test hook: this stage is never filled
                        dropped0 = true;
                    } else {
                        const uint32_t leader_full = map_to_cta(full_bar(stage), 0);
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), pair_bytes);
#pragma unroll
                        for (int h = 0; h < Cfg::KSUB; ++h) {
                            // sub-block h: K columns [(KSUB kb + h) 64, +64); past K, TMA fills zeros
                            const int kbs = backwards ? n_stages - 1 - kb : kb;
                            const int k0 = (kbs * Cfg::KSUB + h) * Cfg::BK;
                            tma_load_2d_pair(sb + Cfg::OFF_A + stage * Cfg::A_STAGE_BYTES + h * Cfg::A_SUB_BYTES,
                                             &tmA, leader_full, k0, m_row, pol);
                            const uint32_t b_dst = sb + Cfg::OFF_B + stage * Cfg::B_STAGE_BYTES + h * Cfg::B_SUB_BYTES;
                            if (p.b_chunked) {
                                // boxes of b_box_chunks 64-column chunks (1 when half units exist)
                                for (int j = 0; j < chunks; j += p.b_box_chunks)
                                    tma_load_3d_pair(b_dst + j * Cfg::B_CHUNK_BYTES, &tmB, leader_full, 0, k0,
                                                     n_col / 64 + j, pol_b);
                            } else {
                                for (int j = 0; j < chunks; ++j)
                                    tma_load_2d_pair(b_dst + j * Cfg::B_CHUNK_BYTES, &tmB, leader_full,
                                                     n_col + j * 64, k0, pol_b);
                            }
                        }
                    }
                    ++slots;
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            // Exit handshake.  The peer's copies count on the leader's full barriers, so only
            // the leader can see them land: the peer reports how many slots it took, and the
            // leader settles every stage's last phase before the pair may leave (after an
            // abort the two producers may have stopped at different slots).
            if (rank == 1) {
                st_shared_cluster_u32(map_to_cta(smem_u32((const void*)peer_slots), 0),
                                      slots | (dropped0 ? Cfg::SLOT_DROPPED : 0u));
                mbar_arrive_cluster(map_to_cta(exit_bar, 0));
            } else if (w.drain_cluster(exit_bar, 0)) {
                const uint32_t word = *peer_slots;
                const uint32_t pslots = word & ~Cfg::SLOT_DROPPED;
                const bool pdropped0 = (word & Cfg::SLOT_DROPPED) != 0;
                const int n_stages = (p.num_k_blocks + Cfg::KSUB - 1) / Cfg::KSUB;
                // one CTA's bytes of slot j (both CTAs' shares are equal): whole units stage
                // HALF_N columns of B per CTA, half units half of that
                auto share = [&](uint32_t j) -> uint32_t {
                    const int u = cluster + (int)(j / (uint32_t)n_stages) * nclusters;
                    const int chunks = (Cfg::BN == 256 && u >= p.num_full) ? Cfg::HALF_N / 128 : Cfg::HALF_N / 64;
                    return (uint32_t)(Cfg::KSUB * (Cfg::A_SUB_BYTES + chunks * Cfg::B_CHUNK_BYTES));
                };
                // fills of stage s among the first n slots, less a skipped slot 0
                auto fills = [&](uint32_t n, int s, bool skipped0) -> uint32_t {
                    const uint32_t f = n > (uint32_t)s ? (n - 1u - (uint32_t)s) / (uint32_t)S + 1u : 0u;
                    return f - ((s == 0 && skipped0) ? 1u : 0u);
                };
                for (int s = 0; s < S; ++s) {
                    // phases [0, A) of full_bar(s) were armed by the leader, [0, P) received
                    // the peer's copies; a slot is only taken once the one S slots earlier
                    // has completed, so A and P differ by at most one.
                    const uint32_t A = fills(slots, s, dropped0), P = fills(pslots, s, pdropped0);
                    const uint32_t last = A > P ? A : P;
                    if (last == 0) continue;
                    if (P == A + 1) {
                        // the peer filled a phase the leader never armed: arm it for the
                        // peer's bytes alone (the phase before it has completed)
                        mbar_arrive_expect_tx(full_bar(s), share(A * S + s));
                    } else if (A == P + 1) {
                        // the leader armed a phase the peer never filled: count the peer's
                        // share as arrived, so the phase completes once the leader's bytes land
                        mbar_complete_tx(full_bar(s), share(P * S + s));
                    } else if (A != P) {
                        atomicCAS(p.err, 0, kDevErrKernelTiled | kDevErrTeardown);
                        continue;
                    }
                    w.drain(full_bar(s), (last - 1u) & 1u);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader)
        // One thread, no warp-wide synchronisation per k-block: the tensor pipe must never
        // wait on the issuing loop.
        if (rank == 0 && lane == 0) {
            uint32_t stage = 0, phase = 0, it = 0;
            bool ok = true;
            // Descriptors of stage 0, advanced by adding (byte offset >> 4) to their start-address
            // field (bits 0-13): every operand lies below 232448 bytes, so the field cannot carry.
            const uint64_t a_desc0 = smem_desc_sw128(sb + Cfg::OFF_A, 16, 1024);
            const uint64_t b_desc0 = smem_desc_sw128(sb + Cfg::OFF_B, Cfg::B_CHUNK_BYTES, 1024);
            for (int u = cluster; ok && u < p.num_units; u += nclusters, ++it) {
                const uint32_t acc = it & 1u, acc_parity = (it >> 1) & 1u;
                if (!w.wait(tempty_bar(acc), acc_parity ^ 1u, kDevErrMmaAccEmpty)) break;
                tcgen05_fence_after();
                const uint32_t d_tmem = tmem_base + acc * Cfg::BN;
                const uint32_t idesc = u < p.num_full ? Cfg::IDESC : Cfg::IDESC_HALF;
                const int n_stages = (p.num_k_blocks + Cfg::KSUB - 1) / Cfg::KSUB;
                for (int kb = 0; kb < n_stages; ++kb) {
                    if (!w.wait(full_bar(stage), phase, kDevErrMmaFull)) { ok = false; break; }
                    tcgen05_fence_after();
                    const uint64_t ad_s = a_desc0 + (uint64_t)((stage * Cfg::A_STAGE_BYTES) >> 4);
                    const uint64_t bd_s = b_desc0 + (uint64_t)((stage * Cfg::B_STAGE_BYTES) >> 4);
#pragma unroll
                    for (int k = 0; k < Cfg::KSUB * Cfg::BK / 16; ++k) {
                        const uint32_t hs = (uint32_t)(k >> 2), kk = (uint32_t)(k & 3);
                        mma_f16_ss_pair(d_tmem, ad_s + (uint64_t)((hs * Cfg::A_SUB_BYTES + kk * 32) >> 4),
                                        bd_s + (uint64_t)((hs * Cfg::B_SUB_BYTES + kk * 2048) >> 4), idesc,
                                        (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit_pair(empty_bar(stage), 0x3);
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair(tfull_bar(acc), 0x3);
            }
            mma_commit_pair(drain_bar, 0x1);
            w.drain(drain_bar, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int et = threadIdx.x - 64;
        // C is written once and never read here: its lines go first when L2 needs room, so
        // they do not push out A and B panels still in use
        const bool store_first = (p.test_flags & kTestStoreNoHint) == 0;
        const uint64_t pol_c = l2_policy_evict_first();
        uint32_t it = 0, cidx = 0;
        for (int u = cluster; u < p.num_units; u += nclusters, ++it) {
            const uint32_t acc = it & 1u, acc_parity = (it >> 1) & 1u;
            const bool got = w.wait(tfull_bar(acc), acc_parity, kDevErrEpilogueFull);
            if (!named_bar_and(1, 128, got)) break;
            tcgen05_fence_after();
            int mb, nb, half;
            pair_unit(u, p, mb, nb, half);
            const int m0 = mb * Cfg::BM + (int)rank * Cfg::HALF_M;   // this CTA's rows
            const int n0 = nb * Cfg::BN + (half < 0 ? 0 : half * (Cfg::BN / 2));
            // columns of C in this unit (a second half unit may lie wholly past N)
            const int ncols = min(half < 0 ? Cfg::BN : Cfg::BN / 2, p.N - n0);
            const int nchunks = (m0 < p.M && ncols > 0) ? (ncols + 63) / 64 : 0;
            const uint32_t t_row = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * Cfg::BN;
            const uint32_t leader_tempty = map_to_cta(tempty_bar(acc), 0);
            if (nchunks == 0) {
                // nothing of this half-tile lies inside C; still release the accumulator
                tcgen05_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(leader_tempty);
            }
            for (int c = 0; c < nchunks; ++c) {
                uint32_t r0[32], r1[32];
                tmem_ld_32x32b_x32(t_row + c * 64, r0);
                tmem_ld_32x32b_x32(t_row + c * 64 + 32, r1);
                tmem_ld_wait(r0);
                tmem_ld_wait(r1);
                if (c == nchunks - 1) {
                    tcgen05_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(leader_tempty);
                }
                const uint32_t buf = cidx & 1u;
                uint8_t* const cbuf = smem + Cfg::OFF_C + buf * Cfg::C_BUF_BYTES;
                const uint32_t cbuf_s = sb + Cfg::OFF_C + buf * Cfg::C_BUF_BYTES;
                if constexpr (KIND_SPLIT) {
                    if (p.epi == kEpiScaleRelu)
                        epilogue_store_chunk<kEpiScaleRelu>(r0, r1, cbuf, cbuf_s, row, et, p, n0 + c * 64, m0,
                                                            &tmC, store_first, pol_c);
                    else if (p.epi == kEpiScale)
                        epilogue_store_chunk<kEpiScale>(r0, r1, cbuf, cbuf_s, row, et, p, n0 + c * 64, m0,
                                                        &tmC, store_first, pol_c);
                    else
                        epilogue_store_chunk<kEpiBiasGelu>(r0, r1, cbuf, cbuf_s, row, et, p, n0 + c * 64, m0,
                                                           &tmC, store_first, pol_c);
                } else {
                    epilogue_store_chunk(r0, r1, cbuf, cbuf_s, row, et, p, n0 + c * 64, m0, &tmC, store_first,
                                         pol_c);
                }
                ++cidx;
            }
        }
        if (et == 0) bulk_wait_group<0>();
    }

    // Neither CTA may leave (or free TMEM) while the pair still uses its shared memory,
    // barriers or tensor memory.
    tcgen05_fence_before();
    cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tcgen05_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace

namespace {

template <class Cfg>
cudaLaunchConfig_t pair_launch_config(int clusters, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(Cfg::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Largest number of co-resident CTA pairs, per device (0 if the query fails).
template <class Cfg>
int max_clusters() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaFuncSetAttribute(gsr_pair_kernel<Cfg, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM_BYTES) != cudaSuccess)
        return 0;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_launch_config<Cfg>(1, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gsr_pair_kernel<Cfg, false>, &cfg) != cudaSuccess) return 0;
    cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

template <class Cfg, bool KIND_SPLIT>
cudaError_t launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                   const TiledParams& p, int clusters, cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(gsr_pair_kernel<Cfg, KIND_SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_launch_config<Cfg>(clusters, stream, attr);
    return cudaLaunchKernelEx(&cfg, gsr_pair_kernel<Cfg, KIND_SPLIT>, tmA, tmB, tmC, p);
}

// At most this many waves of work units per launch take the kernel copy with one epilogue
// loop per kind.
constexpr int kKindSplitMaxWaves = 2;

template <class Cfg>
cudaError_t launch_any(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                       const TiledParams& p, int clusters, cudaStream_t stream) {
    if ((long long)p.num_units <= (long long)kKindSplitMaxWaves * clusters)
        return launch<Cfg, true>(tmA, tmB, tmC, p, clusters, stream);
    return launch<Cfg, false>(tmA, tmB, tmC, p, clusters, stream);
}

}  // namespace

int pair_smem_bytes(int bn) { return bn == 128 ? PairCfg<128>::SMEM_BYTES : PairCfg<256>::SMEM_BYTES; }

int pair_max_active_clusters(int bn) { return bn == 128 ? max_clusters<PairCfg<128>>() : max_clusters<PairCfg<256>>(); }

cudaError_t launch_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                        const TiledParams& p, int bn, int clusters, cudaStream_t stream) {
    if (bn == 256) return launch_any<PairCfg<256>>(tmA, tmB, tmC, p, clusters, stream);
    if (bn == 128) return launch_any<PairCfg<128>>(tmA, tmB, tmC, p, clusters, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gsr
