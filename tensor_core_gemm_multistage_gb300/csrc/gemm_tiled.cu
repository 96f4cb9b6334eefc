// gemm_tiled.cu - tiled path of C = ReLU(alpha * A.B) on sm_103a.
//
// Follows the operator of "Tutorial14: 使用TileLang语言编写attention算子": section 2 (the
// gemm_fused kernel: a grid of output tiles, a K loop pipelined through shared memory,
// a tensor-core GEMM into a float accumulator, then scale, max with 0 and an fp16
// store) and section 3 (分块与流水线: tiles plus a multi-stage prefetch pipeline; 融合
// Epilogue: scale and ReLU applied on chip before the single write-back).
//
// The GB300 design keeps those steps and changes how each one is carried out:
//  * tile 128 x BN (BN = 256, 128 or 64) with K in 64-wide sub-blocks, one or two per
//    pipeline stage, instead of 64 x 64 x 32, because one tcgen05 MMA covers 128 x BN x 16;
//  * a persistent grid (one CTA per SM) walks the tiles in grouped-M order so
//    neighbouring CTAs share A and B panels in L2;
//  * warp roles: warp 0 issues TMA loads into a STAGES-deep shared-memory ring
//    (full/empty mbarriers, expect-tx byte counts), warp 1 allocates tensor memory and
//    issues tcgen05.mma from one thread, warps 2-5 run the epilogue;
//  * the accumulator lives in tensor memory, double-buffered (2 x BN columns) so the
//    epilogue of one tile overlaps the MMAs of the next;
//  * epilogue: tcgen05.ld -> y = max(alpha * acc, 0) -> fp16 (round to nearest even)
//    -> 128-byte-swizzled shared staging -> TMA store (clipped at the M/N edges).
// A is K-major (row-major M x K); B is MN-major (row-major K x N), described to the MMA
// as such, so neither operand is transposed in memory.
#include <atomic>

#include "device_common.cuh"
#include "kernels.h"

namespace gsr {
namespace {

// BK = 64 is one TMA box of K (128 bytes); a stage holds KSUB such sub-blocks.  With the copies
// taken out, the MMA issuer's loop took ~570 cycles per stage of 4 MMAs whatever N was (64, 128
// or 256) and ~790 per stage of 8: at N = 64 or 128 (128 or 256 cycles of tensor work per
// sub-block) one sub-block per stage leaves the tensor pipe idle most of the time, so those tiles
// take two sub-blocks per stage (8 MMAs per wait and commit).  At N = 256 one sub-block is 512
// cycles of tensor work, and two would leave room for only two stages (10 % slower).
template <int BN_, int STAGES_, int KSUB_>
struct TiledCfg {
    static constexpr int BM = 128, BN = BN_, BK = 64, STAGES = STAGES_, KSUB = KSUB_;
    static constexpr int NUM_THREADS = 192;                  // 6 warps
    static constexpr int A_SUB_BYTES = BM * BK * 2;          // 16 KB: one 64-wide K sub-block
    static constexpr int B_CHUNK_BYTES = BK * 64 * 2;        // one 64-column TMA box: 8 KB
    static constexpr int B_SUB_BYTES = BK * BN * 2;
    static constexpr int A_STAGE_BYTES = KSUB * A_SUB_BYTES;
    static constexpr int B_STAGE_BYTES = KSUB * B_SUB_BYTES;
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
    static constexpr int C_CHUNK_COLS = 64;
    static constexpr int C_BUF_BYTES = BM * C_CHUNK_COLS * 2;  // 16 KB
    static constexpr int C_BUFS = 2;
    static constexpr int TMEM_COLS = 2 * BN;                 // two accumulators
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE_BYTES;
    static constexpr int OFF_C = OFF_B + STAGES * B_STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_C + C_BUFS * C_BUF_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 1;      // full, empty, tfull x2, tempty x2, drain
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;  // TMEM base, abort flag, stats
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1024-byte alignment
    static constexpr uint32_t IDESC = idesc_f16_f32(BM, BN, /*a_mn=*/false, /*b_mn=*/true);

    static_assert(SMEM_BYTES <= 232448, "exceeds the per-CTA shared-memory limit");
    static_assert(TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512,
                  "TMEM allocation must be a power of two");
    static_assert(BN % 64 == 0 && BN <= 256, "BN must be a multiple of 64, at most 256");
};

template <class Cfg>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
    gsr_tiled_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
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
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);      // producer's arrive.expect_tx
            mbar_init(empty_bar(s), 1);     // tcgen05.commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);     // tcgen05.commit at the end of a tile
            mbar_init(tempty_bar(a), 128);  // every epilogue thread
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish_alloc_permit();
    }
    tcgen05_fence_before();
    __syncthreads();
    tcgen05_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Waiter w{p.err, p.timeout_ns, abort_flag, kDevErrKernelTiled};
    bool tmem_freed = false;                      // warp 1: released before the teardown

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // One lane issues everything, with no warp-wide synchronisation per stage.
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint32_t armed_mask = 0, armed_parity = 0;   // last phase each stage was filled in
            bool drop_first = (p.test_flags & kTestDropFirstLoad) && blockIdx.x == 0;
            bool ok = true;
            const int n_stages = (p.num_k_blocks + Cfg::KSUB - 1) / Cfg::KSUB;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                int mb, nb;
                raster_tile_coords(tile, p.num_m_blocks, p.num_n_blocks, p.group_m, mb, nb);
                for (int kb = 0; kb < n_stages; ++kb) {
                    if (!w.wait(empty_bar(stage), phase ^ 1u, kDevErrProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    if (drop_first) {
                        drop_first = false;   // test hook: this stage is never filled
                    } else {
                        const uint32_t fb = full_bar(stage);
                        mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
#pragma unroll
                        for (int h = 0; h < Cfg::KSUB; ++h) {
                            // sub-block h: K columns [(KSUB kb + h) 64, +64); past K, TMA fills
                            // zeros (and still counts the whole box), which add nothing
                            const int k0 = (kb * Cfg::KSUB + h) * Cfg::BK;
                            tma_load_2d(sb + Cfg::OFF_A + stage * Cfg::A_STAGE_BYTES + h * Cfg::A_SUB_BYTES, &tmA,
                                        fb, k0, mb * Cfg::BM);
#pragma unroll
                            for (int j = 0; j < Cfg::BN / 64; ++j)
                                tma_load_2d(sb + Cfg::OFF_B + stage * Cfg::B_STAGE_BYTES + h * Cfg::B_SUB_BYTES +
                                                j * Cfg::B_CHUNK_BYTES,
                                            &tmB, fb, nb * Cfg::BN + j * 64, k0);
                        }
                        armed_mask |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            // Every copy this CTA started must land before the CTA may exit.
            for (int s = 0; s < S; ++s)
                if (armed_mask & (1u << s)) w.drain(full_bar(s), (armed_parity >> s) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // One lane issues every MMA and commit; the tensor pipe must never wait on the loop.
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, it = 0;
            bool ok = true;
            // Descriptors of stage 0, advanced by adding (byte offset >> 4) to their start-address
            // field (bits 0-13): every operand lies below 232448 bytes, so the field cannot carry.
            // Building each from scratch cost ~10 cycles per MMA in the issuing thread.
            // A: K-major, 16 elements (32 bytes) per MMA inside the 128-byte swizzle row.
            // B: MN-major, 16 K rows (2048 bytes) per MMA; 64-column chunks 8 KB apart.
            const uint64_t a_desc0 = smem_desc_sw128(sb + Cfg::OFF_A, 16, 1024);
            const uint64_t b_desc0 = smem_desc_sw128(sb + Cfg::OFF_B, Cfg::B_CHUNK_BYTES, 1024);
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++it) {
                const uint32_t acc = it & 1u, acc_parity = (it >> 1) & 1u;
                if (!w.wait(tempty_bar(acc), acc_parity ^ 1u, kDevErrMmaAccEmpty)) break;
                tcgen05_fence_after();
                const uint32_t d_tmem = tmem_base + acc * Cfg::BN;
                const int n_stages = (p.num_k_blocks + Cfg::KSUB - 1) / Cfg::KSUB;
                for (int kb = 0; kb < n_stages; ++kb) {
                    if (!w.wait(full_bar(stage), phase, kDevErrMmaFull)) {
                        ok = false;
                        break;
                    }
                    tcgen05_fence_after();
                    const uint64_t ad_s = a_desc0 + (uint64_t)((stage * Cfg::A_STAGE_BYTES) >> 4);
                    const uint64_t bd_s = b_desc0 + (uint64_t)((stage * Cfg::B_STAGE_BYTES) >> 4);
#pragma unroll
                    for (int k = 0; k < Cfg::KSUB * Cfg::BK / 16; ++k) {
                        const uint32_t hs = (uint32_t)(k >> 2), kk = (uint32_t)(k & 3);
                        const uint64_t ad = ad_s + (uint64_t)((hs * Cfg::A_SUB_BYTES + kk * 32) >> 4);
                        const uint64_t bd = bd_s + (uint64_t)((hs * Cfg::B_SUB_BYTES + kk * 2048) >> 4);
                        mma_f16_ss(d_tmem, ad, bd, Cfg::IDESC, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(empty_bar(stage));   // frees the stage once these MMAs have read it
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(tfull_bar(acc));   // accumulator ready for the epilogue
            }
            // Every MMA this thread issued must finish before tensor memory is released.
            mma_commit(drain_bar);
            w.drain(drain_bar, 0);
            // Tensor memory goes back as soon as the epilogue has read the last accumulator
            // (its arrival on tempty), while it still writes that tile out: the release takes
            // about a microsecond, which at the end of the kernel would add to every launch.
            if (ok && it > 0) {
                const uint32_t last = it - 1;
                tmem_freed = w.wait(tempty_bar(last & 1u), (last >> 1) & 1u, kDevErrMmaAccEmpty);
            }
        }
        tmem_freed = __shfl_sync(0xffffffffu, tmem_freed, 0);
        if (tmem_freed) {
            tcgen05_fence_after();
            tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (warps 2-5)
        const int quad = warp & 3;                 // TMEM lane quadrant this warp may read
        const int row = quad * 32 + lane;          // tile row == TMEM lane
        const int et = threadIdx.x - 64;           // 0..127
        uint32_t it = 0, cidx = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
            const uint32_t acc = it & 1u, acc_parity = (it >> 1) & 1u;
            const bool got = w.wait(tfull_bar(acc), acc_parity, kDevErrEpilogueFull);
            if (!named_bar_and(1, 128, got)) break;
            tcgen05_fence_after();
            int mb, nb;
            raster_tile_coords(tile, p.num_m_blocks, p.num_n_blocks, p.group_m, mb, nb);
            const int m0 = mb * Cfg::BM, n0 = nb * Cfg::BN;
            const int nchunks = (min(Cfg::BN, p.N - n0) + 63) / 64;   // skip columns past N
            const uint32_t t_row = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * Cfg::BN;
            for (int c = 0; c < nchunks; ++c) {
                uint32_t r0[32], r1[32];
                tmem_ld_32x32b_x32(t_row + c * 64, r0);
                tmem_ld_32x32b_x32(t_row + c * 64 + 32, r1);
                tmem_ld_wait(r0);
                tmem_ld_wait(r1);
                if (c == nchunks - 1) {
                    tcgen05_fence_before();
                    mbar_arrive(tempty_bar(acc));   // MMA may now overwrite this accumulator
                }
                const uint32_t buf = cidx & 1u;
                uint8_t* const cbuf = smem + Cfg::OFF_C + buf * Cfg::C_BUF_BYTES;
                const uint32_t cbuf_s = sb + Cfg::OFF_C + buf * Cfg::C_BUF_BYTES;
                // one copy of the chunk's code per epilogue kind (the kind is the same for every
                // chunk of the launch): the values of a chunk then convert without a branch
                if (p.epi == kEpiScaleRelu)
                    epilogue_store_chunk<kEpiScaleRelu>(r0, r1, cbuf, cbuf_s, row, et, p, n0 + c * 64, m0, &tmC, false, 0);
                else if (p.epi == kEpiScale)
                    epilogue_store_chunk<kEpiScale>(r0, r1, cbuf, cbuf_s, row, et, p, n0 + c * 64, m0, &tmC, false, 0);
                else
                    epilogue_store_chunk<kEpiBiasGelu>(r0, r1, cbuf, cbuf_s, row, et, p, n0 + c * 64, m0, &tmC, false, 0);
                ++cidx;
            }
        }
        if (et == 0) bulk_wait_group<0>();
    }

    tcgen05_fence_before();
    __syncthreads();
    if (warp == 1 && !tmem_freed) {   // an aborted run releases it here, after every role stopped
        __syncwarp();
        tcgen05_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

using Cfg256 = TiledCfg<256, 4, 1>;
using Cfg128 = TiledCfg<128, 3, 2>;
using Cfg64 = TiledCfg<64, 4, 2>;

template <class Cfg>
cudaError_t launch_cfg(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                       const TiledParams& p, int grid, cudaStream_t stream) {
    // The shared-memory opt-in is per device; do it once for each.
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(gsr_tiled_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    gsr_tiled_kernel<Cfg><<<grid, Cfg::NUM_THREADS, Cfg::SMEM_BYTES, stream>>>(tmA, tmB, tmC, p);
    return cudaGetLastError();
}

// One thread per output element; only used when K == 0.
__global__ void gsr_fill_bias_gelu_kernel(__half* C, const __half* bias, int M, int N) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)M * N) return;
    C[i] = __float2half_rn(gelu_tanh(__half2float(bias[i % N])));
}

}  // namespace

cudaError_t launch_fill_bias_gelu(__half* C, const __half* bias, int M, int N, cudaStream_t stream) {
    const long long total = (long long)M * N;
    const long long blocks = (total + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    gsr_fill_bias_gelu_kernel<<<(unsigned)blocks, 256, 0, stream>>>(C, bias, M, N);
    return cudaGetLastError();
}

int tiled_smem_bytes(int bn) {
    return bn == 256 ? Cfg256::SMEM_BYTES : bn == 128 ? Cfg128::SMEM_BYTES : Cfg64::SMEM_BYTES;
}

cudaError_t launch_tiled(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                         const TiledParams& p, int bn, int grid, cudaStream_t stream) {
    if (bn == 256) return launch_cfg<Cfg256>(tmA, tmB, tmC, p, grid, stream);
    if (bn == 128) return launch_cfg<Cfg128>(tmA, tmB, tmC, p, grid, stream);
    if (bn == 64) return launch_cfg<Cfg64>(tmA, tmB, tmC, p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gsr
