// device_common.cuh - bounded mbarrier waits, the raster order of the tiled kernels, and the
// epilogue arithmetic, shared by the kernels.
//
// Every wait in the kernels is bounded: after `timeout_ns` of %globaltimer time the
// waiting thread records an error code in the per-device error word, raises the CTA's
// abort flag (so the other roles stop waiting too) and returns false.  Nothing traps;
// the kernel drains its in-flight copies and MMAs, frees its tensor memory and exits,
// and the host reads the code with gsr_device_status().
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace gsr {

struct Waiter {
    int* err;                       // device error word (first code wins)
    uint64_t timeout_ns;
    volatile uint32_t* abort_flag;  // shared memory, one per CTA
    int kernel_code;                // kDevErrKernelTiled / kDevErrKernelSkinny

    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, int code) const {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t spin = 1;; ++spin) {
            if (mbar_try_wait(bar, parity)) return true;
            if ((spin & 63u) == 0u) {
                if (*abort_flag) return false;
                if (globaltimer_ns() - t0 > timeout_ns) {
                    *abort_flag = 1u;
                    atomicCAS(err, 0, kernel_code | code);
                    return false;
                }
            }
        }
    }

    // Teardown variant: ignores the abort flag (it must really drain), still bounded.
    __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t spin = 1;; ++spin) {
            if (mbar_try_wait(bar, parity)) return true;
            if ((spin & 63u) == 0u && globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1u;
                atomicCAS(err, 0, kernel_code | kDevErrTeardown);
                return false;
            }
        }
    }

    // Teardown wait on a barrier a thread of the peer CTA arrives on (release at cluster
    // scope): what that thread wrote before its arrive is visible after a true return.
    __device__ __forceinline__ bool drain_cluster(uint32_t bar, uint32_t parity) const {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t spin = 1;; ++spin) {
            if (mbar_try_wait_cluster(bar, parity)) return true;
            if ((spin & 63u) == 0u && globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1u;
                atomicCAS(err, 0, kernel_code | kDevErrTeardown);
                return false;
            }
        }
    }

    __device__ __forceinline__ bool aborted() const { return *abort_flag != 0u; }
};

// ---------------------------------------------------------------------------
// Tile scheduling shared by the one-CTA and CTA-pair tiled kernels
// ---------------------------------------------------------------------------
// Tile t -> (m block, n block), grouped along M: `group_m` consecutive M blocks share each
// N block before the walk moves to the next N block (the last group may be shorter), so
// the tiles running at one time reuse the same A panels (and each B panel) from L2.
__device__ __forceinline__ void raster_tile_coords(int t, int num_m_blocks, int num_n_blocks,
                                                   int group_m, int& mb, int& nb) {
    const int per_group = group_m * num_n_blocks;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int gsz = min(num_m_blocks - first_m, group_m);
    const int r = t - g * per_group;
    mb = first_m + r % gsz;
    nb = r / gsz;
}

// ---------------------------------------------------------------------------
// Epilogue functions on the fp32 accumulator
// ---------------------------------------------------------------------------
// GELU, tanh approximation: 0.5 x (1 + tanh(u)), u = sqrt(2/pi) (x + 0.044715 x^3).
// Since 0.5 (1 + tanh(u)) = 1 / (1 + e^(-2u)), it is evaluated as x / (1 + 2^(-w)) with
// w = 2 u log2(e): one exp2 and one reciprocal on the special-function unit (~8 instructions
// against ~25 for tanhf, which matters because the epilogue warp of TMEM lanes 32-63 shares
// its scheduler with the MMA issuer), and no cancellation for large negative x, where
// 1 + tanh(u) would lose its digits.  2^(-w) is capped at 2^64, where x / (1 + 2^64) is
// already far below the smallest fp16 subnormal for any accumulator value.
__device__ __forceinline__ float gelu_tanh(float x) {
    constexpr float kC1 = 2.0f * 0.7978845608028654f * 1.4426950408889634f;
    constexpr float kC3 = kC1 * 0.044715f;
    const float w = x * fmaf(kC3, x * x, kC1);
    return __fdividef(x, 1.0f + ex2_approx(fminf(-w, 64.0f)));
}

__device__ __forceinline__ float epilogue_value(float acc, float alpha, float bias, int epi) {
    if (epi == kEpiScaleRelu) return fmaxf(acc * alpha, 0.0f);
    if (epi == kEpiScale) return acc * alpha;
    return gelu_tanh(acc + bias);
}

// Eight consecutive accumulator columns (fp32 bit patterns) -> eight fp16 in a uint4.
// `col0` is the first column's index in C (a multiple of 8); its bias values are read
// only when the columns lie inside C (N is a multiple of 8, so all eight or none do).
__device__ __forceinline__ uint4 epilogue_8(const uint32_t* src, float alpha, int epi,
                                            const __half* bias, int col0, int N) {
    uint4 v;
    if (epi == kEpiScaleRelu) {
        v.x = scale_relu_pack(src[0], src[1], alpha);
        v.y = scale_relu_pack(src[2], src[3], alpha);
        v.z = scale_relu_pack(src[4], src[5], alpha);
        v.w = scale_relu_pack(src[6], src[7], alpha);
        return v;
    }
    float b[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (epi == kEpiBiasGelu && col0 < N) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(bias + col0));
        const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(h[i]);
            b[2 * i] = f.x;
            b[2 * i + 1] = f.y;
        }
    }
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = epilogue_value(__uint_as_float(src[2 * i]), alpha, b[2 * i], epi);
        const float hi = epilogue_value(__uint_as_float(src[2 * i + 1]), alpha, b[2 * i + 1], epi);
        __half2 h2 = __floats2half2_rn(lo, hi);
        out[i] = *reinterpret_cast<uint32_t*>(&h2);
    }
    v.x = out[0];
    v.y = out[1];
    v.z = out[2];
    v.w = out[3];
    return v;
}

// One 64-column chunk of a 128-row output tile, from the four epilogue warps' registers (thread
// = tile row `row`, r0/r1 = the chunk's two 32-column halves of fp32 accumulators) to C: wait
// until the previous store from staging buffer `buf` has read it, write the row's 64 outputs
// into the buffer in the 128-byte-swizzled layout of the tensor map (16-byte chunk j of row r
// at j ^ (r & 7): conflict-free), and hand the buffer to one TMA store of the box at (col0, m0),
// which clips whatever lies outside C.  Named barrier 1 spans the 128 epilogue threads; `et`
// is the thread's index among them.  `pol`, when `hinted`, is the L2 policy of the written lines.
// KIND >= 0 fixes the epilogue kind at compile time (p.epi must equal it), so that the eight
// groups of values carry no branch on it; KIND = -1 reads p.epi.
template <int KIND = -1>
__device__ __forceinline__ void epilogue_store_chunk(const uint32_t (&r0)[32], const uint32_t (&r1)[32],
                                                     uint8_t* buf, uint32_t buf_saddr, int row, int et,
                                                     const TiledParams& p, int col0, int m0,
                                                     const CUtensorMap* tmC, bool hinted, uint64_t pol) {
    const int epi = KIND >= 0 ? KIND : p.epi;
    if (et == 0) bulk_wait_group_read<1>();   // the store from this buffer is done reading it
    named_bar_sync(1, 128);
    uint8_t* crow = buf + row * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t* src = (j < 4) ? (r0 + 8 * j) : (r1 + 8 * (j - 4));
        const uint4 v = epilogue_8(src, p.alpha, epi, p.bias, col0 + 8 * j, p.N);
        *reinterpret_cast<uint4*>(crow + ((j ^ (row & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 128);
    if (et == 0) {
        if (hinted)
            tma_store_2d_hint(tmC, buf_saddr, col0, m0, pol);
        else
            tma_store_2d(tmC, buf_saddr, col0, m0);
        bulk_commit_group();
    }
}

}  // namespace gsr
