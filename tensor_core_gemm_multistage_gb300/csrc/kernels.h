// kernels.h - internal interface between the C-ABI layer (gsr_api.cu) and the GEMM kernel
// translation units (gemm_tiled.cu, gemm_pair.cu, gemm_skinny.cu), plus the device error codes
// and test flags every kernel shares.  Not installed; not part of the ABI.  The attention
// kernel's parameters are in attention.h.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace gsr {

// Device-side error codes written (first one wins) into the per-device error word.
// The low byte says which wait gave up, the next byte which kernel.
enum DeviceError : int {
    kDevErrNone = 0,
    kDevErrProducerEmpty = 1,   // producer: no free shared-memory stage
    kDevErrMmaFull = 2,         // MMA issuer: stage never filled by TMA
    kDevErrMmaAccEmpty = 3,     // MMA issuer: accumulator never released by the epilogue
    kDevErrEpilogueFull = 4,    // epilogue: accumulator never committed by the MMA issuer
    kDevErrTeardown = 5,        // teardown: in-flight copies or MMAs did not drain
    kDevErrLayout = 6,          // dynamic shared memory not 1024-byte aligned (kernel did nothing)
    kDevErrKernelTiled = 0x100,
    kDevErrKernelSkinny = 0x200,
    kDevErrKernelAttention = 0x300,
};

// Test-only flags (gsr_set_test_flags).
enum TestFlags : uint32_t {
    kTestDropFirstLoad = 1u,    // CTA 0's producer skips its first stage fill
    kTestNoChunkedB = 2u,       // host: copy B as separate 64-column boxes even when N % 64 == 0
    kTestKForward = 4u,         // pair kernel: every wave walks K forward (no serpentine order)
    kTestStoreNoHint = 8u,      // pair kernel: C stores without the L2 evict-first hint
    kTestDropFirstLoadPeer = 16u,   // pair kernel: CTA 1 (the first pair's peer) skips its first fill
    kTestBEvictFirst = 32u,     // pair kernel: B copies with an L2 evict-first hint (not evict-last)
    kTestBEvictNormal = 64u,    // pair kernel: B copies with an L2 evict-normal hint
    kTestAttnHeadMajor = 128u,  // attention: one head's query blocks at a time, even when causal
};

// What the epilogue applies to the fp32 accumulator before the fp16 store.
enum Epilogue : int {
    kEpiScaleRelu = 0,   // max(alpha * acc, 0)
    kEpiScale = 1,       // alpha * acc (alpha = 1: plain GEMM)
    kEpiBiasGelu = 2,    // GELU(acc + bias[n]), tanh approximation
};

struct TiledParams {
    int M, N, K;
    float alpha;
    int num_m_blocks, num_n_blocks, num_k_blocks, num_tiles, group_m;
    // CTA-pair kernel at BN 256: work units [0, num_full) are whole tiles; every tile after
    // them is two half-width units (256 x 128), so a last wave that would leave most pairs
    // idle is spread over twice as many.  num_units = num_full + 2 (num_tiles - num_full).
    // Other kernels: num_full = num_units = num_tiles.
    int num_full, num_units;
    int b_box_chunks;       // 64-column chunks per 3-D copy of B (b_chunked only)
    int* err;               // device error word
    uint64_t timeout_ns;    // bound on every mbarrier wait
    uint32_t test_flags;
    int b_chunked;          // tmB is the 3-D view {64, K, N/64} of B (N % 64 == 0)
    int epi;                // Epilogue
    const __half* bias;     // kEpiBiasGelu: N values, 16-byte aligned
};

struct SkinnyParams {
    int M, N, K;
    float alpha;
    int num_n_tiles;        // ceil(N / 128)
    int num_k_blocks;       // ceil(K / 64) per tile
    int num_slabs;          // S: each tile's k blocks are split into S equal slabs
    int num_ctas;           // grid: min(num_n_tiles * S, #SMs), items strided by the grid
    float* partials;        // S > 1: [num_n_tiles][S][MP][128] fp32 partial tiles
    int* tickets;           // [num_n_tiles], zero between launches
    __half* C;              // (M, N) row-major output
    int* err;
    uint64_t timeout_ns;
    uint32_t test_flags;
    int epi;                // Epilogue
    const __half* bias;     // kEpiBiasGelu: N values
};

// Split of the small-M work: S slabs per tile so that n_tiles * S fills the SMs once (each
// slab at least one k block), grid = min(n_tiles * S, sms).
inline void skinny_split(int n_tiles, int k_blocks, int sms, int* slabs, int* ctas) {
    int S = n_tiles >= sms ? 1 : sms / n_tiles;
    if (S > k_blocks) S = k_blocks;
    if (S < 1) S = 1;
    const long long items = (long long)n_tiles * S;
    *slabs = S;
    *ctas = (int)(items < sms ? items : sms);
}



// Tiled path: persistent, one 128 x BN output tile per CTA iteration.
// bn is 128 or 256.  grid = min(num_tiles, num_sms).
cudaError_t launch_tiled(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                         const TiledParams& p, int bn, int grid, cudaStream_t stream);

// Paired tiled path: clusters of 2 CTAs, 256 x bn tiles (bn 256 or 128), cta_group::2 MMA.
// tmB's 3-D box (when p.b_chunked) holds bn / 128 chunks of 64 columns.
// grid = 2 * clusters, clusters <= pair_max_active_clusters(bn).
cudaError_t launch_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                        const TiledParams& p, int bn, int clusters, cudaStream_t stream);
int pair_max_active_clusters(int bn);
int pair_smem_bytes(int bn);

// Skinny path (M <= 64): C^T = B^T A^T on 128-row tiles of N, K split into slabs.
// mp is the MMA N (16, 32 or 64; 128 or 256 when forced for 65 to 256 rows).
cudaError_t launch_skinny(const CUtensorMap& tmBt, const CUtensorMap& tmAt, const SkinnyParams& p,
                          int mp, cudaStream_t stream);

// Allocation-free small-M launch: scratch comes from a fixed module array of
// noalloc_scratch_bytes() bytes (see gemm_skinny.cu); p.partials, p.tickets and p.err are
// filled in by the call.  noalloc_scratch_need() is the byte count a launch uses.
cudaError_t launch_skinny_noalloc(const CUtensorMap& tmBt, const CUtensorMap& tmAt, SkinnyParams p,
                                  int mp, cudaStream_t stream);
size_t noalloc_scratch_bytes();
size_t noalloc_scratch_need(int n_tiles, int slabs, int mp);
// Reads (after `stream`'s earlier work) and clears the error word of the fixed array on the
// current device; *code = 0 when the allocation-free entry point never ran there.
cudaError_t noalloc_take_error(cudaStream_t stream, int* code);

// C[m, n] = GELU(bias[n]) for every m: the bias-GELU epilogue of an empty (K == 0) sum.
cudaError_t launch_fill_bias_gelu(__half* C, const __half* bias, int M, int N, cudaStream_t stream);

// Shared-memory bytes a launch needs (for the one-time attribute set-up).
int tiled_smem_bytes(int bn);
int skinny_smem_bytes(int mp);

}  // namespace gsr
