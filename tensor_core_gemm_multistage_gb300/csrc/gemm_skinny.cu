// gemm_skinny.cu - small-M path of C = ReLU(alpha * A.B) on sm_103a (M <= 64; up to 256 when forced).
//
// Same operator as the tiled path ("Tutorial14: 使用TileLang语言编写attention算子",
// section 3 formula; section 2 kernel: float accumulator, scale, max with 0, fp16 out).
// When M is a handful of rows the work is streaming B (K x N) from HBM once; a 128-row
// M tile would leave most of each MMA empty and only ceil(N/BN) CTAs busy.  So:
//  * swap A and B: the MMA computes C^T (N x M) = B^T (N x K) . A^T (K x M), with
//    128 columns of C per tile as the MMA's M and M (rounded up to MP = 16/32/64, or
//    128/256 when the path is forced for 65 to 256 rows) as its N.  B^T is read straight
//    from row-major B as an MN-major operand and A^T from row-major A as a K-major
//    operand: nothing is transposed in memory;
//  * split K into S equal slabs per tile (S = #SMs / #tiles, at least 1): work item w =
//    (slab w / T, tile w % T) for T tiles, so the CTAs running at one time work on the
//    same slab and walk through the same rows of B in step, as one streaming pass (DRAM
//    pages are read whole); with S == 1 each item is a whole tile and is stored directly.
//    With S > 1 each item writes an fp32 partial tile into its own slot (tile, slab) of
//    the workspace and takes a ticket; the CTA that takes the S-th ticket sums the S
//    partials in slab order (deterministic), applies the epilogue and resets the ticket to
//    0 for the next launch.  Nobody waits on another CTA, so nothing can deadlock across
//    CTAs.
#include <atomic>

#include "device_common.cuh"
#include "kernels.h"

namespace gsr {
namespace {

template <int MP_, int STAGES_>
struct SkinnyCfg {
    static constexpr int TN = 128;          // columns of C per tile (MMA M)
    static constexpr int BK = 64;
    static constexpr int MP = MP_;          // MMA N: M rounded up to a multiple of 16
    static constexpr int STAGES = STAGES_;
    static constexpr int NUM_THREADS = 192;
    static constexpr int BT_CHUNK_BYTES = BK * 64 * 2;   // one 64-column box of B: 8 KB
    static constexpr int BT_STAGE_BYTES = BK * TN * 2;   // 16 KB
    static constexpr int AT_STAGE_BYTES = MP * BK * 2;   // MP rows of A, 128 bytes each
    static constexpr int STAGE_BYTES = BT_STAGE_BYTES + AT_STAGE_BYTES;
    static constexpr int TMEM_COLS = (2 * MP <= 32) ? 32 : (2 * MP <= 64 ? 64 : (2 * MP <= 128 ? 128 : (2 * MP <= 256 ? 256 : 512)));
    static constexpr int OFF_BT = 0;
    static constexpr int OFF_AT = OFF_BT + STAGES * BT_STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_AT + STAGES * AT_STAGE_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // TMEM base, abort flag, ticket result
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr uint32_t IDESC = idesc_f16_f32(TN, MP, /*a_mn=*/true, /*b_mn=*/false);

    static_assert(MP % 16 == 0 && MP >= 16 && (MP <= 64 || MP == 128 || MP == 256),
                  "MP must be 16, 32, 48, 64, 128 or 256");
    static_assert(AT_STAGE_BYTES % 1024 == 0, "A^T stage must keep 1024-byte alignment");
    static_assert(SMEM_BYTES <= 232448, "exceeds the per-CTA shared-memory limit");
};

template <class Cfg>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
    gsr_skinny_kernel(const __grid_constant__ CUtensorMap tmBt, const __grid_constant__ CUtensorMap tmAt,
                      const SkinnyParams p) {
    constexpr int NS = Cfg::STAGES;
    constexpr int MP = Cfg::MP;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);

    auto full_bar = [&](int s) { return sb + Cfg::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sb + Cfg::OFF_BAR + 8u * (NS + s); };
    auto tfull_bar = [&](int a) { return sb + Cfg::OFF_BAR + 8u * (2 * NS + a); };
    auto tempty_bar = [&](int a) { return sb + Cfg::OFF_BAR + 8u * (2 * NS + 2 + a); };
    const uint32_t drain_bar = sb + Cfg::OFF_BAR + 8u * (2 * NS + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_MISC + 4);
    volatile int* s_last = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kbpt = p.num_k_blocks;
    const int n_tiles = p.num_n_tiles;
    const int S = p.num_slabs;
    const int W = n_tiles * S;                 // work items, slab-major

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 128);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmBt);
        tma_prefetch_desc(&tmAt);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish_alloc_permit();
    }
    tcgen05_fence_before();
    __syncthreads();
    tcgen05_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Waiter w{p.err, p.timeout_ns, abort_flag, kDevErrKernelSkinny};

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // One lane issues everything, with no warp-wide synchronisation per stage.
        if (lane == 0) {
            const uint64_t pol_stream = l2_policy_evict_first();   // B: every byte read once
            const uint64_t pol_keep = l2_policy_evict_last();      // A: read by every CTA
            uint32_t stage = 0, phase = 0;
            uint32_t armed_mask = 0, armed_parity = 0;
            bool drop_first = (p.test_flags & kTestDropFirstLoad) && blockIdx.x == 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < W; item += gridDim.x) {
                const int tile = item % n_tiles, slab = item / n_tiles;
                const int kb0 = slab * kbpt / S, kb1 = (slab + 1) * kbpt / S;
                const int n0 = tile * Cfg::TN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!w.wait(empty_bar(stage), phase ^ 1u, kDevErrProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    if (drop_first) {
                        drop_first = false;
                    } else {
                        const uint32_t fb = full_bar(stage);
                        const uint32_t bt = sb + Cfg::OFF_BT + stage * Cfg::BT_STAGE_BYTES;
                        mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
                        tma_load_2d_hint(bt, &tmBt, fb, n0, kb * Cfg::BK, pol_stream);
                        tma_load_2d_hint(bt + Cfg::BT_CHUNK_BYTES, &tmBt, fb, n0 + 64, kb * Cfg::BK,
                                         pol_stream);
                        tma_load_2d_hint(sb + Cfg::OFF_AT + stage * Cfg::AT_STAGE_BYTES, &tmAt, fb,
                                         kb * Cfg::BK, 0, pol_keep);
                        armed_mask |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == NS) { stage = 0; phase ^= 1u; }
                }
            }
            for (int s = 0; s < NS; ++s)
                if (armed_mask & (1u << s)) w.drain(full_bar(s), (armed_parity >> s) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, it = 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < W; item += gridDim.x, ++it) {
                const int slab = item / n_tiles;
                const int kb0 = slab * kbpt / S, kb1 = (slab + 1) * kbpt / S;
                const uint32_t acc = it & 1u, acc_parity = (it >> 1) & 1u;
                if (!w.wait(tempty_bar(acc), acc_parity ^ 1u, kDevErrMmaAccEmpty)) break;
                tcgen05_fence_after();
                const uint32_t d_tmem = tmem_base + acc * MP;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!w.wait(full_bar(stage), phase, kDevErrMmaFull)) {
                        ok = false;
                        break;
                    }
                    tcgen05_fence_after();
                    const uint32_t bt = sb + Cfg::OFF_BT + stage * Cfg::BT_STAGE_BYTES;
                    const uint32_t at = sb + Cfg::OFF_AT + stage * Cfg::AT_STAGE_BYTES;
#pragma unroll
                    for (int k = 0; k < Cfg::BK / 16; ++k) {
                        // MMA A = B^T: MN-major, 16 K rows = 2048 bytes per step, 64-col chunks 8 KB apart.
                        const uint64_t ad = smem_desc_sw128(bt + k * 2048, Cfg::BT_CHUNK_BYTES, 1024);
                        // MMA B = A^T: K-major, 16 elements = 32 bytes per step.
                        const uint64_t bd = smem_desc_sw128(at + k * 32, 16, 1024);
                        mma_f16_ss(d_tmem, ad, bd, Cfg::IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(empty_bar(stage));
                    if (++stage == NS) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(tfull_bar(acc));
            }
            mma_commit(drain_bar);
            w.drain(drain_bar, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (warps 2-5)
        const int quad = warp & 3;
        const int nl = quad * 32 + lane;     // column of C inside the tile == TMEM lane
        const int et = threadIdx.x - 64;
        uint32_t it = 0;
        bool live = true;
        for (int item = blockIdx.x; item < W; item += gridDim.x, ++it) {
            const int tile = item % n_tiles, slab = item / n_tiles;
            const uint32_t acc = it & 1u, acc_parity = (it >> 1) & 1u;
            if (live) {
                const bool got = w.wait(tfull_bar(acc), acc_parity, kDevErrEpilogueFull);
                live = named_bar_and(1, 128, got);
            }
            if (!live) {
                // This CTA gave up on a wait.  It still takes its ticket for each slab it was
                // given, so that every tile's counter sees exactly S takers in this launch and
                // ends it at 0 (the S-th taker resets it), whatever the other CTAs did: the
                // next launch starts clean without the host having to intervene.  The tiles
                // concerned are left unspecified (the timeout is reported).
                if (S > 1 && et == 0) {
                    const int old = atomicAdd(p.tickets + tile, 1);
                    if (old + 1 == S) p.tickets[tile] = 0;
                }
                continue;
            }
            tcgen05_fence_after();

            if constexpr (MP <= 64) {
                float v[MP];
                {
                    const uint32_t t_row = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * MP;
#pragma unroll
                    for (int c = 0; c < MP / 16; ++c) {
                        uint32_t r[16];
                        tmem_ld_32x32b_x16(t_row + c * 16, r);
                        tmem_ld_wait(r);
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[c * 16 + i] = __uint_as_float(r[i]);
                    }
                }
                tcgen05_fence_before();
                mbar_arrive(tempty_bar(acc));

                const int n = tile * Cfg::TN + nl;
                bool store = true;
                if (S > 1) {
                    // One slab of a tile: publish the partial, take a ticket.
                    float* mine = p.partials + ((size_t)tile * S + slab) * (MP * Cfg::TN);
#pragma unroll
                    for (int m = 0; m < MP; ++m) mine[m * Cfg::TN + nl] = v[m];
                    __threadfence();
                    named_bar_sync(1, 128);
                    if (et == 0) {
                        const int old = atomicAdd(p.tickets + tile, 1);
                        *s_last = (old + 1 == S) ? 1 : 0;
                    }
                    named_bar_sync(1, 128);
                    store = (*s_last != 0);
                    if (store) {
                        // Last slab to finish: sum the tile's partials in slab order.
                        __threadfence();
                        float sum[MP];
#pragma unroll
                        for (int m = 0; m < MP; ++m) sum[m] = 0.0f;
                        for (int q = 0; q < S; ++q) {
                            if (q == slab) {
#pragma unroll
                                for (int m = 0; m < MP; ++m) sum[m] += v[m];
                            } else {
                                const float* src = p.partials + ((size_t)tile * S + q) * (MP * Cfg::TN);
#pragma unroll
                                for (int m = 0; m < MP; ++m) sum[m] += __ldcg(src + m * Cfg::TN + nl);
                            }
                        }
#pragma unroll
                        for (int m = 0; m < MP; ++m) v[m] = sum[m];
                        if (et == 0) p.tickets[tile] = 0;   // ready for the next launch
                    }
                }
                if (store && n < p.N) {
                    const float b = (p.epi == kEpiBiasGelu) ? __half2float(p.bias[n]) : 0.0f;
#pragma unroll
                    for (int m = 0; m < MP; ++m)
                        if (m < p.M)
                            p.C[(size_t)m * p.N + n] = __float2half_rn(epilogue_value(v[m], p.alpha, b, p.epi));
                }
            } else {
                // MMA N of 128 or 256: a whole row of the accumulator would not fit in registers,
                // so every step walks it in chunks of 32 columns (rows m of C), reading them from
                // tensor memory again where it needs them, and gives the accumulator back only
                // after the last read.
                constexpr int CH = 32;
                const uint32_t t_row = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * MP;
                const int n = tile * Cfg::TN + nl;
                bool store = true;
                if (S > 1) {
                    // One slab of a tile: publish the partial, take a ticket.
                    float* mine = p.partials + ((size_t)tile * S + slab) * (MP * Cfg::TN);
                    for (int c = 0; c < MP / CH; ++c) {
                        uint32_t r[CH];
                        tmem_ld_32x32b_x32(t_row + c * CH, r);
                        tmem_ld_wait(r);
#pragma unroll
                        for (int i = 0; i < CH; ++i) mine[(c * CH + i) * Cfg::TN + nl] = __uint_as_float(r[i]);
                    }
                    __threadfence();
                    named_bar_sync(1, 128);
                    if (et == 0) {
                        const int old = atomicAdd(p.tickets + tile, 1);
                        *s_last = (old + 1 == S) ? 1 : 0;
                    }
                    named_bar_sync(1, 128);
                    store = (*s_last != 0);
                    if (store) __threadfence();
                }
                if (store) {
                    // (the last slab to finish sums the tile's partials in slab order, its own
                    // from tensor memory, then applies the epilogue)
                    const float b = (p.epi == kEpiBiasGelu && n < p.N) ? __half2float(p.bias[n]) : 0.0f;
                    for (int c = 0; c < MP / CH; ++c) {
                        uint32_t r[CH];
                        tmem_ld_32x32b_x32(t_row + c * CH, r);
                        tmem_ld_wait(r);
                        float v[CH];
#pragma unroll
                        for (int i = 0; i < CH; ++i) v[i] = __uint_as_float(r[i]);
                        if (S > 1) {
                            float sum[CH];
#pragma unroll
                            for (int i = 0; i < CH; ++i) sum[i] = 0.0f;
                            for (int q = 0; q < S; ++q) {
                                if (q == slab) {
#pragma unroll
                                    for (int i = 0; i < CH; ++i) sum[i] += v[i];
                                } else {
                                    const float* src = p.partials + ((size_t)tile * S + q) * (MP * Cfg::TN);
#pragma unroll
                                    for (int i = 0; i < CH; ++i) sum[i] += __ldcg(src + (c * CH + i) * Cfg::TN + nl);
                                }
                            }
#pragma unroll
                            for (int i = 0; i < CH; ++i) v[i] = sum[i];
                        }
                        if (n < p.N) {
#pragma unroll
                            for (int i = 0; i < CH; ++i) {
                                const int m = c * CH + i;
                                if (m < p.M)
                                    p.C[(size_t)m * p.N + n] =
                                        __float2half_rn(epilogue_value(v[i], p.alpha, b, p.epi));
                            }
                        }
                    }
                    if (S > 1 && et == 0) p.tickets[tile] = 0;   // ready for the next launch
                }
                tcgen05_fence_before();
                mbar_arrive(tempty_bar(acc));
            }
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

using Sk16 = SkinnyCfg<16, 11>;
using Sk32 = SkinnyCfg<32, 10>;
using Sk64 = SkinnyCfg<64, 8>;
using Sk128 = SkinnyCfg<128, 6>;
using Sk256 = SkinnyCfg<256, 4>;

template <class Cfg>
cudaError_t launch_cfg(const CUtensorMap& tmBt, const CUtensorMap& tmAt, const SkinnyParams& p,
                       cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(gsr_skinny_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    gsr_skinny_kernel<Cfg><<<p.num_ctas, Cfg::NUM_THREADS, Cfg::SMEM_BYTES, stream>>>(tmBt, tmAt, p);
    return cudaGetLastError();
}

}  // namespace

int skinny_smem_bytes(int mp) {
    return mp <= 16 ? Sk16::SMEM_BYTES
                    : (mp <= 32 ? Sk32::SMEM_BYTES
                                : (mp <= 64 ? Sk64::SMEM_BYTES : (mp <= 128 ? Sk128::SMEM_BYTES : Sk256::SMEM_BYTES)));
}

cudaError_t launch_skinny(const CUtensorMap& tmBt, const CUtensorMap& tmAt, const SkinnyParams& p,
                          int mp, cudaStream_t stream) {
    if (mp == 16) return launch_cfg<Sk16>(tmBt, tmAt, p, stream);
    if (mp == 32) return launch_cfg<Sk32>(tmBt, tmAt, p, stream);
    if (mp == 64) return launch_cfg<Sk64>(tmBt, tmAt, p, stream);
    if (mp == 128) return launch_cfg<Sk128>(tmBt, tmAt, p, stream);
    if (mp == 256) return launch_cfg<Sk256>(tmBt, tmAt, p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gsr

// ---------------------------------------------------------------------------
// Allocation-free variant of the small-M launch.
//
// Some callers cannot let a library call cudaMalloc: a serving runtime that plans all of
// its device memory at start-up and forbids allocations afterwards, or a latency-critical
// loop where the implicit synchronisation of a first-time cudaMalloc is not acceptable.
// For them, gemm_scale_relu_noalloc runs the same small-M kernel with its scratch (error
// word, per-tile tickets, split-K partial tiles) carved out of the fixed array below
// instead of a library-allocated workspace.  The array is a module global, so every GPU
// that loads this library holds its 12 MiB until the process exits.
//
// Every call on a device shares the one array and it keeps whatever the last call left in
// it: the error word and the tickets, which must start at zero, are cleared on the stream
// at the start of each call; the partial tiles are always written before they are read.
// Two calls whose kernels overlap on the GPU (different streams, no ordering between them)
// race on the array and give wrong results.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {
constexpr size_t kNoAllocScratchBytes = (size_t)12 << 20;
constexpr int kNoAllocMaxDevices = 64;
}  // namespace

static __device__ __align__(256) unsigned char g_gsr_noalloc_scratch[kNoAllocScratchBytes];

namespace gsr {

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

// Byte layout inside the array: [0, 256) error word, [256, 256 + tickets) tickets rounded up
// to 256 bytes, then the partial tiles.
size_t noalloc_scratch_need(int n_tiles, int slabs, int mp) {
    const size_t tickets = ((size_t)n_tiles * sizeof(int) + 255) / 256 * 256;
    const size_t slots = slabs > 1 ? (size_t)n_tiles * slabs : 0;
    return 256 + tickets + slots * mp * 128 * sizeof(float);
}

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_base[kNoAllocMaxDevices] = {};

// Shared-memory attribute of one variant, set once per device (as launch_cfg does); under
// CUDA's lazy loading this is also what places the kernel's code on the device.
template <class Cfg>
cudaError_t noalloc_prepare_cfg() {
    return cudaFuncSetAttribute(gsr_skinny_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg::SMEM_BYTES);
}

// Set-up, once per device and with that device current: the device address of the array (in
// host code the array's name is only a host-side stand-in), and every kernel variant the
// entry point can launch made resident, so that no later call makes the driver place
// anything on the device.
cudaError_t noalloc_base(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_base[dev]) {
        void* ptr = nullptr;
        if ((e = cudaGetSymbolAddress(&ptr, g_gsr_noalloc_scratch)) != cudaSuccess) return e;
        if ((e = noalloc_prepare_cfg<Sk16>()) != cudaSuccess ||
            (e = noalloc_prepare_cfg<Sk32>()) != cudaSuccess ||
            (e = noalloc_prepare_cfg<Sk64>()) != cudaSuccess)
            return e;
        g_noalloc_base[dev] = ptr;
    }
    *out = g_noalloc_base[dev];
    return cudaSuccess;
}
}  // namespace

cudaError_t launch_skinny_noalloc(const CUtensorMap& tmBt, const CUtensorMap& tmAt, SkinnyParams p,
                                  int mp, cudaStream_t stream) {
    void* base = nullptr;
    cudaError_t e = noalloc_base(&base);
    if (e != cudaSuccess) return e;
    if (noalloc_scratch_need(p.num_n_tiles, p.num_slabs, mp) > kNoAllocScratchBytes)
        return cudaErrorInvalidValue;
    unsigned char* b = static_cast<unsigned char*>(base);
    const size_t tickets = ((size_t)p.num_n_tiles * sizeof(int) + 255) / 256 * 256;
    p.err = reinterpret_cast<int*>(b);
    p.tickets = reinterpret_cast<int*>(b + 256);
    p.partials = reinterpret_cast<float*>(b + 256 + tickets);
    e = cudaMemsetAsync(b, 0, 256 + tickets, stream);   // error word and tickets start at 0
    if (e != cudaSuccess) return e;
    if (mp == 16) return launch_cfg<Sk16>(tmBt, tmAt, p, stream);
    if (mp == 32) return launch_cfg<Sk32>(tmBt, tmAt, p, stream);
    if (mp == 64) return launch_cfg<Sk64>(tmBt, tmAt, p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t noalloc_take_error(cudaStream_t stream, int* code) {
    *code = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaSuccess;
    void* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        base = g_noalloc_base[dev];
    }
    if (!base) return cudaSuccess;   // the entry point never ran on this device
    int h = 0;
    if ((e = cudaMemcpyAsync(&h, base, sizeof(int), cudaMemcpyDeviceToHost, stream)) != cudaSuccess ||
        (e = cudaStreamSynchronize(stream)) != cudaSuccess)
        return e;
    if (h != 0) {
        if ((e = cudaMemsetAsync(base, 0, sizeof(int), stream)) != cudaSuccess ||
            (e = cudaStreamSynchronize(stream)) != cudaSuccess)
            return e;
    }
    *code = h;
    return cudaSuccess;
}

}  // namespace gsr
