// gsr_api.cu - the C ABI of libgsr: argument checks, path choice, tensor-map encoding,
// per-(device, stream) state, and the launches.  See include/gsr.h for the contract.
//
// Nothing here computes any part of the operator; every step of C = ReLU(alpha * A.B)
// runs in the kernels of gemm_tiled.cu, gemm_pair.cu and gemm_skinny.cu (attention in
// attention_fwd.cu).  The one exception is K == 0, where the empty sum makes every output
// ReLU(alpha * 0) = 0 and C is cleared with cudaMemsetAsync (GELU(bias) by a fill kernel).
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "gsr.h"
#include "attention.h"
#include "kernels.h"

namespace {

thread_local int t_last_cuda_error = 0;
std::atomic<int> g_path_override{0};
std::atomic<uint64_t> g_timeout_ns{1000000000ull};
std::atomic<uint32_t> g_test_flags{0};
std::atomic<int> g_raster_group{0};   // 0: each kernel's default grouping
std::atomic<int> g_split_k{0};        // 0: the small-M kernel's own slab count

constexpr int kSkinnyMaxM = 64;
// Up to 64 rows with B under 16 MiB the launch is latency-bound and one-CTA tiles finish first:
// L2 flushed between calls, mean of 50: 64 x 1024 x 2048 13.1 us on 128 x 64 tiles against 22.5
// on the small-M kernel, 32 x 2048 x 512 9.5 against 13.8, 64 x 5488 x 416 10.3 against 14.5,
// 16 x 1024 x 2048 12.9 against 16.4, 16 x 4096 x 1024 12.3 against 12.6; at 32 MiB the two
// are within ~10 % either way (16 x 4096 x 4096 18.2 on the small-M kernel against 20.5,
// 48 x 8192 x 2048 18.3 against 16.4), and from there on B's streaming favours the small-M one.
constexpr double kSkinnyMinBBytes = 16.0 * (1 << 20);
// The small-M kernel also runs up to 256 rows (MMA N of 128 or 256) when forced.
constexpr int kSkinnyMaxForcedM = 256;
constexpr int kGroupM = 16;

// Device words per (device, stream): [0] the error word of kernels on the stream, [1] and [2]
// the attention kernel's work counter and done count (zero between launches).
constexpr int kStreamWords = 4;

struct StreamState {
    int* err = nullptr;          // kStreamWords device words, the error word first
    float* partials = nullptr;   // small-M split-K partial tiles
    size_t partial_floats = 0;
    int* tickets = nullptr;      // small-M per-tile ticket counters (zero between launches)
    size_t ticket_count = 0;
};

struct DeviceInfo {
    int cc_major = 0, cc_minor = 0, num_sms = 0;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
std::map<std::pair<int, CUstream_st*>, StreamState> g_streams;

// Copy streams and events of the pipelined host entry point, one set per device (created on
// first use, released by gsr_shutdown).  `m` keeps one call's enqueue sequence together.
// Events: start, done, one per row chunk of A, one per column block of B, one per block of C.
constexpr int kHostMaxChunks = 8;      // row chunks of A and C
constexpr int kHostMaxColBlocks = 4;   // column blocks of B and C
constexpr int kHostEvents = 2 + kHostMaxChunks + kHostMaxColBlocks + kHostMaxChunks * kHostMaxColBlocks;
struct HostPipe {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev[kHostEvents] = {};
    std::mutex m;
};
std::map<int, HostPipe*> g_pipes;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

gsr_status cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return GSR_ERR_CUDA;
}

gsr_status load_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess && fn)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else if (g_encode_err == cudaSuccess)
            g_encode_err = cudaErrorSymbolNotFound;
    });
    if (!g_encode) return cuda_fail(g_encode_err);
    return GSR_OK;
}

// Row-major fp16 matrix of `rows` x `cols` (cols contiguous, `ld` elements from one row to the
// next; 0: dense, ld = cols) seen as a 2-D tensor map with a box of box_cols x box_rows, 128-byte
// swizzle, zero fill outside the matrix (so a block of a wider matrix is clipped at its own edge).
gsr_status encode_fp16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                          uint32_t box_cols, uint32_t box_rows, uint64_t ld = 0) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {(ld ? ld : cols) * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return GSR_ERR_CUDA;
    }
    return GSR_OK;
}

// Row-major fp16 B (K x N, N % 64 == 0) seen as 64-column chunks: a 3-D tensor map
// {64 columns, K rows, N/64 chunks} whose box {64, box_k, box_chunks} lands box_chunks
// consecutive chunks one after the other in shared memory, each box_k rows of 128 bytes
// (the same layout as box_chunks separate 64 x box_k boxes), in one copy instruction.
gsr_status encode_fp16_chunked(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                               uint32_t box_rows, uint32_t box_chunks, uint64_t ld = 0) {
    cuuint64_t dims[3] = {64, rows, cols / 64};
    cuuint64_t strides[2] = {(ld ? ld : cols) * 2, 128};
    cuuint32_t box[3] = {64, box_rows, box_chunks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return GSR_ERR_CUDA;
    }
    return GSR_OK;
}

// (batch*heads, seq, D) fp16 as a 3-D tensor map {D, seq, BH}, box {64, 128, 1}: tiles never
// cross heads and rows past `seq` are zero-filled.
gsr_status encode_fp16_bsd(CUtensorMap* map, const void* base, uint64_t bh, uint64_t seq, uint64_t d) {
    cuuint64_t dims[3] = {d, seq, bh};
    cuuint64_t strides[2] = {d * 2, seq * d * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return GSR_ERR_CUDA;
    }
    return GSR_OK;
}

bool overlaps(const void* a, uint64_t an, const void* b, uint64_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a && b && an && bn && a0 < b0 + bn && b0 < a0 + an;
}

// Checks that need no GPU: sizes, null pointers, alignment, aliasing.  `*nothing` is set
// when there is no output to produce.
gsr_status validate(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
                    bool* nothing) {
    *nothing = false;
    if (M < 0 || N < 0 || K < 0) return GSR_ERR_INVALID_ARG;
    if (M > INT_MAX || N > INT_MAX || K > INT_MAX) return GSR_ERR_INVALID_ARG;
    if (M == 0 || N == 0) {
        *nothing = true;
        return GSR_OK;
    }
    if (!C) return GSR_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B)) return GSR_ERR_INVALID_ARG;
    // tile counts must fit the kernels' int arithmetic
    const uint64_t m_blocks = ((uint64_t)M + 127) / 128, n_blocks = ((uint64_t)N + 127) / 128;
    if (m_blocks * n_blocks > (uint64_t)INT_MAX) return GSR_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(C) & 15u) || (N & 7)) return GSR_ERR_ALIGNMENT;
    if (K > 0) {
        if ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u) ||
            (K & 7))
            return GSR_ERR_ALIGNMENT;
        const uintptr_t c0 = reinterpret_cast<uintptr_t>(C), c1 = c0 + (uint64_t)M * N * 2;
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(A), a1 = a0 + (uint64_t)M * K * 2;
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(B), b1 = b0 + (uint64_t)K * N * 2;
        if ((c0 < a1 && a0 < c1) || (c0 < b1 && b0 < c1)) return GSR_ERR_ALIAS;
    }
    return GSR_OK;
}

gsr_status device_info(int* dev_out, DeviceInfo* info) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_devices.find(dev);
    if (it == g_devices.end()) {
        DeviceInfo d;
        if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) !=
                cudaSuccess)
            return cuda_fail(e);
        it = g_devices.emplace(dev, d).first;
    }
    *dev_out = dev;
    *info = it->second;
    if (info->cc_major != 10 || info->cc_minor != 3) return GSR_ERR_UNSUPPORTED_DEVICE;
    return GSR_OK;
}

// Per-(device, stream) state: the error word always, the small-M workspace on demand.
// Returns a copy of the state (pointers stay valid until gsr_shutdown or regrowth).
gsr_status stream_state(int dev, cudaStream_t stream, size_t need_partials, size_t need_tickets,
                        StreamState* out) {
    std::lock_guard<std::mutex> lock(g_mu);
    StreamState& s = g_streams[{dev, stream}];
    cudaError_t e;
    if (!s.err) {
        if ((e = cudaMalloc(&s.err, kStreamWords * sizeof(int))) != cudaSuccess) {
            s.err = nullptr;
            return cuda_fail(e);
        }
        if ((e = cudaMemsetAsync(s.err, 0, kStreamWords * sizeof(int), stream)) != cudaSuccess)
            return cuda_fail(e);
    }
    if (need_partials > s.partial_floats || need_tickets > s.ticket_count) {
        // Earlier launches on this stream may still use the old buffers.
        if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e);
        if (need_partials > s.partial_floats) {
            cudaFree(s.partials);
            s.partials = nullptr;
            s.partial_floats = 0;
            if ((e = cudaMalloc(&s.partials, need_partials * sizeof(float))) != cudaSuccess) {
                s.partials = nullptr;
                return cuda_fail(e);
            }
            s.partial_floats = need_partials;
        }
        if (need_tickets > s.ticket_count) {
            cudaFree(s.tickets);
            s.tickets = nullptr;
            s.ticket_count = 0;
            if ((e = cudaMalloc(&s.tickets, need_tickets * sizeof(int))) != cudaSuccess) {
                s.tickets = nullptr;
                return cuda_fail(e);
            }
            s.ticket_count = need_tickets;
            if ((e = cudaMemsetAsync(s.tickets, 0, need_tickets * sizeof(int), stream)) !=
                cudaSuccess)
                return cuda_fail(e);
        }
    }
    *out = s;
    return GSR_OK;
}

// Whole 256 x 256 tiles of a pair launch: all of them, unless the last wave would keep at
// most half of the pairs busy; then that wave's tiles run as two 256 x 128 halves each, on
// twice as many pairs (a half costs ~0.6-0.7 of a tile: half the MMAs, at N = 128, and 3/4
// of the copies).
int pair_full_tiles(int num_tiles, int clusters, int bn) {
    if (bn != 256 || clusters <= 0) return num_tiles;
    const int rem = num_tiles % clusters;
    return (rem > 0 && 2 * rem <= clusters) ? num_tiles - rem : num_tiles;
}

// 0: tiled, one CTA per 128 x BN tile; 1: small-M; 2: tiled on CTA pairs (256 x 256 tiles),
// taken above 128 rows and K = 384 when there are at least as many pair tiles as half the SMs
// (one full wave of pairs), or below that for a long K where the one-CTA kernel would take
// 128 x 256 tiles (choose_path).
// Pair tiles 256 wide (with a last wave of half tiles where that helps), or 128 wide where
// that is estimated to be faster: time ~ waves x tile cost, a wave of 256 x 128 tiles or half
// units costing kHalfTileCost of a wave of 256 x 256 tiles (half the MMAs plus the fixed
// per-tile part), and the narrower tiles must win by 5 %.  Measured per wave on GB300 (same
// process, interleaved): 0.61 (4096 x 1280 x 4096), 0.68 (6144^2 x 2048), 0.70 (16384 x 640 x
// 4096).  At 0.56 the model sent 16384 x 384 and 16384 x 640 (K 4096) to the narrow tiles,
// 4.7 % and 17 % slower than 256 x 256; now only N <= 128-like shapes, where a 256-wide tile is
// half empty, take them.
constexpr double kHalfTileCost = 0.68;

int pair_path(int64_t M, int64_t N, int num_sms) {
    const long long mb = (M + 255) / 256, clusters = num_sms / 2 > 0 ? num_sms / 2 : 1;
    const long long t256 = mb * ((N + 255) / 256);
    const long long full = pair_full_tiles((int)t256, (int)clusters, 256);
    const double w256 =
        (double)(full / clusters) + (full < t256 ? kHalfTileCost : (t256 % clusters ? 1.0 : 0.0));
    const long long w128 = (mb * ((N + 127) / 128) + clusters - 1) / clusters;
    return kHalfTileCost * (double)w128 < 0.95 * w256 ? 3 : 2;
}

// Tile width of the one-CTA-per-tile kernel: whichever finishes first when a wave of
// 128 x 256 tiles costs kWideTileCost waves of 128 x 128 tiles (an N = 256 MMA does twice the
// work of an N = 128 one in ~1.45x the time, and its tile stages 1.5x the bytes per k-block).
// L2 flushed, median of 5 x 100 calls, 128-wide tiles at 8 MMAs per stage: 2048^3 with 128
// tiles of 128 x 256 18.8 us against 20.9 with 256 of 128 x 128, 1536 x 2048 x 2048 with 96
// tiles 17.6 against 20.7, while below half a wave the narrow tiles win (64 tiles: 1024 x 2048
// x 1024 12.6 against 11.2).  Counting waves, not tiles, also keeps N = 128 on 128-wide tiles,
// where a 256-wide one is half empty (16384 x 128 x 4096: 27.1 against 31.1 us).
constexpr double kWideTileCost = 1.45;

// 128 x 64 tiles: a wave of them costs kNarrowTileCost waves of 128 x 128 tiles (a stage of
// 48 KB instead of 64 KB per SM, and half the epilogue), so they are taken when they still fit
// in one wave.  L2 flushed, median of 5 x 100 calls: 1024^3 10.7 us against 11.3, 1000 x 1000 x
// 200 9.1 against 10.1, 1024 x 1024 x 4096, 512 x 2048 x 4096 and 768 x 1536 x 2048 within 1 %;
// at two waves they lose (1024 x 2048 x 1024: 14.7 against 12.4).
constexpr double kNarrowTileCost = 0.9;

int tiled_width(long long mb, int64_t N, int num_sms) {
    const long long sms = num_sms > 0 ? num_sms : 1;
    const long long t256 = mb * ((N + 255) / 256), t128 = mb * ((N + 127) / 128), t64 = mb * ((N + 63) / 64);
    const double w256 = kWideTileCost * (double)((t256 + sms - 1) / sms);
    const double w128 = (double)((t128 + sms - 1) / sms);
    const double w64 = kNarrowTileCost * (double)((t64 + sms - 1) / sms);
    if (w64 < w128 && w64 < w256) return 64;
    return w256 < w128 ? 256 : 128;
}

// Below a full wave of 256 x 256 pair tiles the one-CTA kernel is taken, except where it would
// run 128 x 256 tiles (two SMs per 256 x 256 of C, as a pair tile) over a long K.  Per 64-wide K
// sub-block a pair's SM spends ~500 cycles (N = 256 MMAs), a single tile's ~660 (its 48 KB
// stage is copy-bound), which from K of about 6000 on repays the pair's larger cost per launch
// (its first cluster barrier and paired TMEM release, and a slower start).  L2 flushed where A
// and B fit in it, median of 5 rounds: K = 4096, single tiles 1-3 % faster (256 x 16384,
// 4096 x 1024, 8192 x 384); K = 8192, pairs 1.5-4.7 % faster (256 x 16384, 2048 x 2048,
// 1024 x 4096, 4096 x 1024, 512 x 8192); K = 16384, pairs 3.3-6.5 % (256 x 16384, 2048 x 2048).
constexpr int64_t kPairMinK = 6144;
constexpr int64_t kPairMaxShortK = 384;

// 65 to 128 rows: the small-M kernel with an MMA N of 128 where B is large enough for the call to
// stream it from HBM and the one-CTA kernel's tiles would keep under two thirds of the SMs busy:
// its K slabs then use them all.  Back to back, median of 5 x 20 calls: 65, 96 and 128 x 4096 x
// 14336 (B 117 MB, 64 tiles of 128 x 64) 32.8-32.9 us against 43.3-43.9, 128 x 4096 x 16384 37.0
// against 49.3, 80 x 3072 x 16384 38.9 against 56.5, 100 x 6144 x 8192 (96 tiles) 34.0 against
// 39.3, 128 x 4096 x 8192 (B 64 MiB) 31.3 against 34.1.  Where the tiles fill more SMs it
// loses 2-7 % (x 8192 x 8192, x 14336 x 4096) or wins little (x 16384 x 16384: 2-4 %, 128 tiles);
// with a small B (17-34 MB, L2 flushed between calls) its split-K sums cost more than the idle
// SMs (128 x 2048 x 4096 33.1 against 18.9, 128 x 4096 x 4096 26.7 against 21.0); and with 129 to
// 256 rows (MMA N 256) it lost to the tiled kernels on all four large shapes.
constexpr int kSkinnyWideMaxM = 128;
constexpr double kSkinnyWideMinBBytes = 64.0 * (1 << 20);

int choose_path(int64_t M, int64_t N, int64_t K, int num_sms) {
    const int o = g_path_override.load(std::memory_order_relaxed);
    if (o == 1 || o == 3 || o == 4 || o == 7) return 0;
    if (o == 5) return 2;
    if (o == 6) return 3;
    if (o == 2 && M <= kSkinnyMaxForcedM) return 1;
    if (M <= kSkinnyMaxM) return 2.0 * (double)K * (double)N < kSkinnyMinBBytes ? 0 : 1;
    // At 128 rows or fewer a pair tile (256 rows) is at least half empty: one-CTA tiles
    // (128 rows) do the same work in one wave of half the size.  Back to back: 100 x 28672 x
    // 8192 72.0 us on 112 tiles of 128 x 256 against 91.9 on 112 pair tiles, 80 x 32768 x 4096
    // 43.0 against 56.0, 128 x 16384 x 16384 87.6 against 98.9.
    // With a few k-blocks a tile is mostly its epilogue, and the pair's costs per tile and per
    // launch outweigh its faster K loop: L2 flushed, 4096 x 16384 x K on 128 x 256 tiles against
    // 256 x 256 pairs: K = 64 33.0 against 45.3 us, 256 39.2 against 47.4, 320 41.7 against 48.0,
    // but 512 56.1 against 50.2; 8192 x 8192 x 256 39.0 against 47.4, 1496 x 18912 x 112 19.7
    // against 25.0.  Up to K = 384 the one-CTA kernel is taken.
    const long long pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
    if (M > 128 && K > kPairMaxShortK) {
        if (pair_tiles >= num_sms / 2) return pair_path(M, N, num_sms);
        if (K >= kPairMinK && tiled_width((M + 127) / 128, N, num_sms) == 256) return pair_path(M, N, num_sms);
    }
    if (M <= kSkinnyWideMaxM && 2.0 * (double)K * (double)N >= kSkinnyWideMinBBytes) {
        const int bn = tiled_width(1, N, num_sms);
        if (3 * ((N + bn - 1) / bn) < 2 * (int64_t)num_sms) return 1;
    }
    return 0;
}

constexpr int kDefaultSms = 152;   // for gsr_select_path before any device is touched

// Which epilogue a call applies, and its bias vector (kEpiBiasGelu only).
struct Epi {
    int kind;
    const __half* bias;
};

// ldb, ldc: row strides (elements) of B and C when they are column blocks of wider matrices;
// 0 for dense ones.
gsr_status run_tiled(const void* A, const void* B, void* C, int M, int N, int K, float alpha,
                     const Epi& ep, cudaStream_t stream, int dev, const DeviceInfo& info,
                     int64_t ldb = 0, int64_t ldc = 0) {
    StreamState st;
    gsr_status s = stream_state(dev, stream, 0, 0, &st);
    if (s != GSR_OK) return s;

    const int mb = (M + 127) / 128;
    const int o = g_path_override.load(std::memory_order_relaxed);
    int bn = tiled_width(mb, N, info.num_sms);
    if (o == 3) bn = 256;
    if (o == 4) bn = 128;
    if (o == 7) bn = 64;
    const int nb = (N + bn - 1) / bn;
    const int kb = (K + 63) / 64;

    CUtensorMap tmA, tmB, tmC;
    if ((s = encode_fp16_2d(&tmA, A, M, K, 64, 128)) != GSR_OK) return s;
    if ((s = encode_fp16_2d(&tmB, B, K, N, 64, 64, ldb)) != GSR_OK) return s;
    if ((s = encode_fp16_2d(&tmC, C, M, N, 64, 128, ldc)) != GSR_OK) return s;

    gsr::TiledParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.num_m_blocks = mb;
    p.num_n_blocks = nb;
    p.num_k_blocks = kb;
    p.num_tiles = mb * nb;
    p.num_full = p.num_units = p.num_tiles;
    p.b_box_chunks = 1;
    p.group_m = kGroupM;
    if (const int g = g_raster_group.load(std::memory_order_relaxed)) p.group_m = g;
    p.b_chunked = 0;
    p.err = st.err;
    p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    p.test_flags = g_test_flags.load(std::memory_order_relaxed);
    p.epi = ep.kind;
    p.bias = ep.bias;
    const int grid = p.num_tiles < info.num_sms ? p.num_tiles : info.num_sms;
    cudaError_t e = gsr::launch_tiled(tmA, tmB, tmC, p, bn, grid, stream);
    return e == cudaSuccess ? GSR_OK : cuda_fail(e);
}

gsr_status run_pair(int bn, const void* A, const void* B, void* C, int M, int N, int K, float alpha,
                    const Epi& ep, cudaStream_t stream, int dev, const DeviceInfo& info,
                    int64_t ldb = 0, int64_t ldc = 0) {
    StreamState st;
    gsr_status s = stream_state(dev, stream, 0, 0, &st);
    if (s != GSR_OK) return s;
    CUtensorMap tmA, tmB, tmC;
    const bool chunked = (N % 64) == 0 &&
                         !(g_test_flags.load(std::memory_order_relaxed) & gsr::kTestNoChunkedB);
    const int num_tiles = ((M + 255) / 256) * ((N + bn - 1) / bn);
    int clusters = gsr::pair_max_active_clusters(bn);
    if (clusters <= 0) clusters = info.num_sms / 2;
    const int num_full = pair_full_tiles(num_tiles, clusters, bn);   // before capping at the units
    const int box_chunks = (bn == 256 && num_full == num_tiles) ? 2 : 1;
    if ((s = encode_fp16_2d(&tmA, A, M, K, 64, 128)) != GSR_OK) return s;
    if (chunked) {
        if ((s = encode_fp16_chunked(&tmB, B, K, N, 64, box_chunks, ldb)) != GSR_OK) return s;
    } else if ((s = encode_fp16_2d(&tmB, B, K, N, 64, 64, ldb)) != GSR_OK) {
        return s;
    }
    if ((s = encode_fp16_2d(&tmC, C, M, N, 64, 128, ldc)) != GSR_OK) return s;
    gsr::TiledParams p;
    p.b_chunked = chunked ? 1 : 0;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.num_m_blocks = (M + 255) / 256;
    p.num_n_blocks = (N + bn - 1) / bn;
    p.num_k_blocks = (K + 63) / 64;
    p.num_tiles = num_tiles;
    p.num_full = num_full;
    p.num_units = num_full + 2 * (num_tiles - num_full);
    p.b_box_chunks = box_chunks;
    // 16 row blocks of 256 per raster group: under the power cap of long back-to-back runs it
    // beat 8 by 0.6 % on 8192^3 and 2.8 % on 16384 x 14336 x 4096, while 4 and 32 lost ~3 %
    // (the group size moves DRAM traffic, not SM cycles, so it shows only when power binds)
    p.group_m = kGroupM;
    if (const int g = g_raster_group.load(std::memory_order_relaxed)) p.group_m = g;
    p.err = st.err;
    p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    p.test_flags = g_test_flags.load(std::memory_order_relaxed);
    p.epi = ep.kind;
    p.bias = ep.bias;
    if (clusters > p.num_units) clusters = p.num_units;
    cudaError_t e = gsr::launch_pair(tmA, tmB, tmC, p, bn, clusters, stream);
    return e == cudaSuccess ? GSR_OK : cuda_fail(e);
}

gsr_status run_skinny(const void* A, const void* B, void* C, int M, int N, int K, float alpha,
                    const Epi& ep,
                      cudaStream_t stream, int dev, const DeviceInfo& info) {
    const int mp = M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : (M <= 128 ? 128 : 256)));
    const int n_tiles = (N + 127) / 128;
    const int kbpt = (K + 63) / 64;
    int S = 1, P = 1;
    gsr::skinny_split(n_tiles, kbpt, info.num_sms, &S, &P);
    if (const int o = g_split_k.load(std::memory_order_relaxed)) {   // every slab keeps a k-block
        S = o < kbpt ? o : kbpt;
        const long long items = (long long)n_tiles * S;
        P = (int)(items < info.num_sms ? items : info.num_sms);
    }

    StreamState st;
    const size_t partial_floats = S > 1 ? (size_t)n_tiles * S * mp * 128 : 0;
    gsr_status s = stream_state(dev, stream, partial_floats, (size_t)n_tiles, &st);
    if (s != GSR_OK) return s;

    CUtensorMap tmBt, tmAt;
    if ((s = encode_fp16_2d(&tmBt, B, K, N, 64, 64)) != GSR_OK) return s;
    if ((s = encode_fp16_2d(&tmAt, A, M, K, 64, mp)) != GSR_OK) return s;

    gsr::SkinnyParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.num_n_tiles = n_tiles;
    p.num_k_blocks = kbpt;
    p.num_slabs = S;
    p.num_ctas = P;
    p.partials = st.partials;
    p.tickets = st.tickets;
    p.C = static_cast<__half*>(C);
    p.err = st.err;
    p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    p.test_flags = g_test_flags.load(std::memory_order_relaxed);
    p.epi = ep.kind;
    p.bias = ep.bias;
    cudaError_t e = gsr::launch_skinny(tmBt, tmAt, p, mp, stream);
    return e == cudaSuccess ? GSR_OK : cuda_fail(e);
}

// Every entry point that runs the GEMM: validation, K == 0, path choice, launch.
gsr_status gemm_impl(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                     float alpha, const Epi& ep, CUstream_st* stream) {
    bool nothing = false;
    gsr_status s = validate(A, B, C, M, N, K, &nothing);
    if (s != GSR_OK || nothing) return s;
    int dev = 0;
    DeviceInfo info;
    if ((s = device_info(&dev, &info)) != GSR_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) {   // empty sum: every output is the epilogue applied to 0
        cudaError_t e = (ep.kind == gsr::kEpiBiasGelu)
                            ? gsr::launch_fill_bias_gelu(static_cast<__half*>(C), ep.bias, (int)M, (int)N, st)
                            : cudaMemsetAsync(C, 0, (size_t)M * N * 2, st);
        return e == cudaSuccess ? GSR_OK : cuda_fail(e);
    }
    if ((s = load_encoder()) != GSR_OK) return s;
    const int path = choose_path(M, N, K, info.num_sms);
    if (path == 1) return run_skinny(A, B, C, (int)M, (int)N, (int)K, alpha, ep, st, dev, info);
    if (path == 2 || path == 3)
        return run_pair(path == 3 ? 128 : 256, A, B, C, (int)M, (int)N, (int)K, alpha, ep, st, dev, info);
    return run_tiled(A, B, C, (int)M, (int)N, (int)K, alpha, ep, st, dev, info);
}

// One block of the pipelined host path: M rows of A (dense, K wide) times N columns of B into
// the same columns of C, B and C keeping the row strides ldb and ldc of the whole matrices
// (validated whole by the caller).  A block always has more than 64 rows: the small-M kernel,
// which writes C without a tensor map, never runs one.
gsr_status gemm_block(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                      int64_t ldb, int64_t ldc, float alpha, CUstream_st* stream) {
    int dev = 0;
    DeviceInfo info;
    gsr_status s = device_info(&dev, &info);
    if (s != GSR_OK) return s;
    if ((s = load_encoder()) != GSR_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const Epi ep{gsr::kEpiScaleRelu, nullptr};
    // (the small-M kernel cannot write column blocks of C: where it would be chosen, forced or for
    // a block of 65-128 rows, one-CTA tiles run instead)
    const int path = choose_path(M, N, K, info.num_sms);
    if (path == 2 || path == 3)
        return run_pair(path == 3 ? 128 : 256, A, B, C, (int)M, (int)N, (int)K, alpha, ep, st, dev, info,
                        ldb, ldc);
    return run_tiled(A, B, C, (int)M, (int)N, (int)K, alpha, ep, st, dev, info, ldb, ldc);
}

}  // namespace

extern "C" {

gsr_status gemm_scale_relu(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                           float alpha, CUstream_st* stream) {
    return gemm_impl(A, B, C, M, N, K, alpha, Epi{gsr::kEpiScaleRelu, nullptr}, stream);
}

gsr_status gemm_scale(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                      float alpha, CUstream_st* stream) {
    return gemm_impl(A, B, C, M, N, K, alpha, Epi{gsr::kEpiScale, nullptr}, stream);
}

gsr_status gemm_bias_gelu(const void* A, const void* B, const void* bias, void* C, int64_t M,
                          int64_t N, int64_t K, CUstream_st* stream) {
    // the bias vector: present, 16-byte aligned, not overlapping C (sizes are checked later)
    if (M > 0 && N > 0 && M <= INT_MAX && N <= INT_MAX && C) {
        if (!bias) return GSR_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(bias) & 15u) return GSR_ERR_ALIGNMENT;
        const uintptr_t c0 = reinterpret_cast<uintptr_t>(C), c1 = c0 + (uint64_t)M * N * 2;
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(bias), b1 = b0 + (uint64_t)N * 2;
        if (c0 < b1 && b0 < c1) return GSR_ERR_ALIAS;
    }
    return gemm_impl(A, B, C, M, N, K, 1.0f, Epi{gsr::kEpiBiasGelu, static_cast<const __half*>(bias)},
                     stream);
}

}  // extern "C"

namespace {

// Row chunks of the pipelined host path: none below 2^33 flop (~8.6 GFLOP) or 1024 rows
// (the copies of a small problem take microseconds and each extra launch costs several),
// else one chunk per 2^33 flop, 2..8 of them, each a multiple of 256 rows (whole CTA-pair
// tiles).  Measured end to end: 8192^3 1.65 ms in 8 chunks against 2.59 ms in one piece,
// 2000 x 3000 x 1000 145 us in 2 against 149 us.
int host_chunk_rows(int64_t M, int64_t N, int64_t K) {
    const double flops = 2.0 * (double)M * (double)N * (double)K;
    if (K == 0 || M < 1024 || flops < 8589934592.0) return 0;
    int64_t r = (int64_t)(flops / 8589934592.0);
    r = r < 2 ? 2 : (r > kHostMaxChunks ? kHostMaxChunks : r);
    const int64_t rows = ((M + r - 1) / r + 255) / 256 * 256;
    return (int)rows;
}

// Columns per block of B and C when they are split into j blocks: whole 256-column pair tiles.
int64_t host_block_cols(int64_t N, int j) { return ((N + j - 1) / j + 255) / 256 * 256; }

// Column blocks of the pipelined host path.  Where C (copied back) outweighs A and B (copied
// in), the copy back bounds the call, and with B sent whole it cannot start before all of B and
// the first rows of A have landed (0.65 of 3.3 ms on 16384 x 14336 x 4096).  Split into column
// blocks, the first block of C goes back once the first rows of A and the first block of B are
// in.  Each block keeps at least a wave of 256 x 256 pair tiles per row chunk (fewer would leave
// SMs idle in every block's product); at most kHostMaxColBlocks blocks.
int host_col_blocks(int64_t M, int64_t N, int64_t K, int rows, int num_sms) {
    if (rows == 0 || M * N <= M * K + K * N) return 1;
    int best = 1;
    for (int j = 2; j <= kHostMaxColBlocks; ++j) {
        const int64_t cols = host_block_cols(N, j);
        if ((N + cols - 1) / cols != j) continue;
        if (((rows + 255) / 256) * (cols / 256) >= num_sms / 2) best = j;
    }
    return best;
}

gsr_status host_pipe(int dev, HostPipe** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    HostPipe*& hp = g_pipes[dev];
    if (!hp) {
        HostPipe* fresh = new HostPipe();
        cudaError_t e = cudaStreamCreateWithFlags(&fresh->h2d, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&fresh->d2h, cudaStreamNonBlocking);
        for (int i = 0; e == cudaSuccess && i < kHostEvents; ++i)
            e = cudaEventCreateWithFlags(&fresh->ev[i], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            for (cudaEvent_t ev : fresh->ev)
                if (ev) cudaEventDestroy(ev);
            if (fresh->h2d) cudaStreamDestroy(fresh->h2d);
            if (fresh->d2h) cudaStreamDestroy(fresh->d2h);
            delete fresh;
            return cuda_fail(e);
        }
        hp = fresh;
    }
    *out = hp;
    return GSR_OK;
}

}  // namespace

extern "C" {

// The host path overlaps its three parts.  A goes over in row chunks and B whole, or, where C
// is the larger transfer, in column blocks (host_col_blocks); the product of each (row chunk,
// column block) runs as soon as both have landed, and that block of C goes back (a strided
// copy when there are column blocks) while later ones are copied in and multiplied.  Copies in
// each direction run on a library stream of their own (host->device and device->host use
// separate copy engines), the products on the caller's stream, joined by events: the whole
// call still behaves as one operation on `stream`.  Small problems run the three parts one
// after the other.
gsr_status gemm_scale_relu_host(const void* hA, const void* hB, void* hC, void* dA, void* dB,
                                void* dC, int64_t M, int64_t N, int64_t K, float alpha,
                                CUstream_st* stream) {
    bool nothing = false;
    gsr_status s = validate(dA, dB, dC, M, N, K, &nothing);
    if (s != GSR_OK || nothing) return s;
    if (!hC || (K > 0 && (!hA || !hB))) return GSR_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    const int rows = host_chunk_rows(M, N, K);
    if (rows == 0) {
        if (K > 0) {
            if ((e = cudaMemcpyAsync(dA, hA, (size_t)M * K * 2, cudaMemcpyHostToDevice, st)) != cudaSuccess)
                return cuda_fail(e);
            if ((e = cudaMemcpyAsync(dB, hB, (size_t)K * N * 2, cudaMemcpyHostToDevice, st)) != cudaSuccess)
                return cuda_fail(e);
        }
        if ((s = gemm_scale_relu(dA, dB, dC, M, N, K, alpha, stream)) != GSR_OK) return s;
        if ((e = cudaMemcpyAsync(hC, dC, (size_t)M * N * 2, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
            return cuda_fail(e);
        return GSR_OK;
    }
    int dev = 0;
    DeviceInfo info;
    if ((s = device_info(&dev, &info)) != GSR_OK) return s;
    HostPipe* hp = nullptr;
    if ((s = host_pipe(dev, &hp)) != GSR_OK) return s;
    std::lock_guard<std::mutex> lock(hp->m);
    // Row chunks [m0[r], m0[r + 1]) (a last one of 64 rows or fewer joins the one before it, so
    // no product is a small-M one) and column blocks of `cols` columns of B and C.
    int64_t m0[kHostMaxChunks + 1];
    int nch = 0;
    for (int64_t m = 0; m < M && nch < kHostMaxChunks; m += rows) m0[nch++] = m;
    if (nch > 1 && M - m0[nch - 1] <= 64) --nch;
    m0[nch] = M;
    const int nblk = host_col_blocks(M, N, K, rows, info.num_sms);
    const int64_t cols = nblk > 1 ? host_block_cols(N, nblk) : N;
    cudaEvent_t start = hp->ev[0], done = hp->ev[1];
    auto ev_a = [&](int r) { return hp->ev[2 + r]; };
    auto ev_b = [&](int j) { return hp->ev[2 + kHostMaxChunks + j]; };
    auto ev_c = [&](int r, int j) { return hp->ev[2 + kHostMaxChunks + kHostMaxColBlocks + r * kHostMaxColBlocks + j]; };
    const char* a_h = static_cast<const char*>(hA);
    const char* b_h = static_cast<const char*>(hB);
    char* a_d = static_cast<char*>(dA);
    char* b_d = static_cast<char*>(dB);
    char* c_h = static_cast<char*>(hC);
    char* c_d = static_cast<char*>(dC);
    const size_t row_b = (size_t)N * 2;   // bytes from one row of B or C to the next
    auto copy_a = [&](int r) {
        const size_t off = (size_t)m0[r] * K * 2, bytes = (size_t)(m0[r + 1] - m0[r]) * K * 2;
        cudaError_t err = cudaMemcpyAsync(a_d + off, a_h + off, bytes, cudaMemcpyHostToDevice, hp->h2d);
        return err == cudaSuccess ? cudaEventRecord(ev_a(r), hp->h2d) : err;
    };
    auto copy_b = [&](int j) {
        const int64_t n0 = j * cols, nj = (N - n0 < cols) ? N - n0 : cols;
        cudaError_t err = nblk == 1 ? cudaMemcpyAsync(b_d, b_h, (size_t)K * row_b, cudaMemcpyHostToDevice, hp->h2d)
                                    : cudaMemcpy2DAsync(b_d + n0 * 2, row_b, b_h + n0 * 2, row_b, (size_t)nj * 2,
                                                        (size_t)K, cudaMemcpyHostToDevice, hp->h2d);
        return err == cudaSuccess ? cudaEventRecord(ev_b(j), hp->h2d) : err;
    };
    // host -> device, after everything already queued on the caller's stream: the first rows of
    // A and the first block of B, then the other rows of A (each one lets a block of the first
    // column go), then the other blocks of B
    gsr_status result = GSR_OK;
    if ((e = cudaEventRecord(start, st)) != cudaSuccess) return cuda_fail(e);   // nothing queued yet
    if ((e = cudaStreamWaitEvent(hp->h2d, start, 0)) != cudaSuccess || (e = copy_a(0)) != cudaSuccess ||
        (e = copy_b(0)) != cudaSuccess)
        result = cuda_fail(e);
    for (int r = 1; r < nch && result == GSR_OK; ++r)
        if ((e = copy_a(r)) != cudaSuccess) result = cuda_fail(e);
    for (int j = 1; j < nblk && result == GSR_OK; ++j)
        if ((e = copy_b(j)) != cudaSuccess) result = cuda_fail(e);
    // the products on the caller's stream, block column by block column, each block of C going
    // back on the copy stream as soon as it is written
    for (int j = 0; j < nblk && result == GSR_OK; ++j) {
        const int64_t n0 = j * cols, nj = (N - n0 < cols) ? N - n0 : cols;
        if ((e = cudaStreamWaitEvent(st, ev_b(j), 0)) != cudaSuccess) {
            result = cuda_fail(e);
            break;
        }
        for (int r = 0; r < nch && result == GSR_OK; ++r) {
            const int64_t mr = m0[r + 1] - m0[r];
            const size_t c_off = (size_t)m0[r] * row_b + (size_t)n0 * 2;
            if (j == 0 && (e = cudaStreamWaitEvent(st, ev_a(r), 0)) != cudaSuccess) {
                result = cuda_fail(e);
                break;
            }
            if ((result = gemm_block(a_d + (size_t)m0[r] * K * 2, b_d + n0 * 2, c_d + c_off, mr, nj, K, N, N,
                                     alpha, stream)) != GSR_OK)
                break;
            if ((e = cudaEventRecord(ev_c(r, j), st)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(hp->d2h, ev_c(r, j), 0)) != cudaSuccess ||
                (e = nblk == 1 ? cudaMemcpyAsync(c_h + c_off, c_d + c_off, (size_t)mr * row_b, cudaMemcpyDeviceToHost,
                                                 hp->d2h)
                               : cudaMemcpy2DAsync(c_h + c_off, row_b, c_d + c_off, row_b, (size_t)nj * 2,
                                                   (size_t)mr, cudaMemcpyDeviceToHost, hp->d2h)) != cudaSuccess)
                result = cuda_fail(e);
        }
    }
    // The caller's stream continues only after both copy streams (the last copy back, and on a
    // failure whatever copies in were queued), so nothing of this call is left running unordered.
    if ((e = cudaEventRecord(done, hp->h2d)) != cudaSuccess || (e = cudaStreamWaitEvent(hp->d2h, done, 0)) != cudaSuccess ||
        (e = cudaEventRecord(done, hp->d2h)) != cudaSuccess || (e = cudaStreamWaitEvent(st, done, 0)) != cudaSuccess)
        return result != GSR_OK ? result : cuda_fail(e);
    return result;
}

// No device-memory allocation anywhere on this path: plain attribute queries instead of
// the cached device table, the small-M kernel with its scratch in the library's fixed
// array (gemm_skinny.cu).
gsr_status gemm_scale_relu_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N,
                                   int64_t K, float alpha, CUstream_st* stream) {
    bool nothing = false;
    gsr_status s = validate(A, B, C, M, N, K, &nothing);
    if (s != GSR_OK || nothing) return s;
    if (M > kSkinnyMaxM) return GSR_ERR_INVALID_ARG;
    const int mp = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    const int n_tiles = (int)((N + 127) / 128);
    const int kbpt = (int)((K + 63) / 64);
    // The tickets alone (every tile one slab) must fit whatever the device: checked before any
    // CUDA call.  A K == 0 call needs no scratch.
    if (K > 0 && gsr::noalloc_scratch_need(n_tiles, 1, mp) > gsr::noalloc_scratch_bytes())
        return GSR_ERR_SCRATCH_LIMIT;
    int dev = 0, major = 0, minor = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail(e);
    if (major != 10 || minor != 3) return GSR_ERR_UNSUPPORTED_DEVICE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) {
        e = cudaMemsetAsync(C, 0, (size_t)M * N * 2, st);
        return e == cudaSuccess ? GSR_OK : cuda_fail(e);
    }
    int S = 1, P = 1;
    gsr::skinny_split(n_tiles, kbpt, sms, &S, &P);
    if (gsr::noalloc_scratch_need(n_tiles, S, mp) > gsr::noalloc_scratch_bytes())
        return GSR_ERR_SCRATCH_LIMIT;
    if ((s = load_encoder()) != GSR_OK) return s;
    CUtensorMap tmBt, tmAt;
    if ((s = encode_fp16_2d(&tmBt, B, K, N, 64, 64)) != GSR_OK) return s;
    if ((s = encode_fp16_2d(&tmAt, A, M, K, 64, mp)) != GSR_OK) return s;
    gsr::SkinnyParams p;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.alpha = alpha;
    p.num_n_tiles = n_tiles;
    p.num_k_blocks = kbpt;
    p.num_slabs = S;
    p.num_ctas = P;
    p.partials = nullptr;   // filled from the fixed array by the launch
    p.tickets = nullptr;
    p.err = nullptr;
    p.C = static_cast<__half*>(C);
    p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    p.test_flags = g_test_flags.load(std::memory_order_relaxed);
    p.epi = gsr::kEpiScaleRelu;
    p.bias = nullptr;
    e = gsr::launch_skinny_noalloc(tmBt, tmAt, p, mp, st);
    return e == cudaSuccess ? GSR_OK : cuda_fail(e);
}

gsr_status flash_attention_fwd(const void* Q, const void* K, const void* V, void* O, float* lse,
                               int64_t batch, int64_t heads, int64_t seq_q, int64_t seq_kv,
                               int64_t head_dim, float softmax_scale, int causal,
                               CUstream_st* stream) {
    if (batch < 0 || heads < 0 || seq_q < 0 || seq_kv < 0) return GSR_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return GSR_ERR_INVALID_ARG;
    if (batch > INT_MAX || heads > INT_MAX || seq_q > INT_MAX || seq_kv > INT_MAX ||
        batch * heads > INT_MAX)
        return GSR_ERR_INVALID_ARG;
    const int64_t BH = batch * heads;
    if (BH == 0 || seq_q == 0) return GSR_OK;
    if (!O || (seq_kv > 0 && (!Q || !K || !V)) || (seq_kv == 0 && !Q)) return GSR_ERR_INVALID_ARG;
    auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (misaligned(O) || (Q && misaligned(Q)) || (K && misaligned(K)) || (V && misaligned(V)) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return GSR_ERR_ALIGNMENT;
    const uint64_t q_bytes = (uint64_t)BH * seq_q * head_dim * 2;
    const uint64_t kv_bytes = (uint64_t)BH * seq_kv * head_dim * 2;
    const uint64_t lse_bytes = lse ? (uint64_t)BH * seq_q * 4 : 0;
    if (overlaps(O, q_bytes, Q, q_bytes) || overlaps(O, q_bytes, K, kv_bytes) ||
        overlaps(O, q_bytes, V, kv_bytes) || overlaps(lse, lse_bytes, O, q_bytes) ||
        overlaps(lse, lse_bytes, Q, q_bytes) || overlaps(lse, lse_bytes, K, kv_bytes) ||
        overlaps(lse, lse_bytes, V, kv_bytes))
        return GSR_ERR_ALIAS;
    int dev = 0;
    DeviceInfo info;
    gsr_status s;
    if ((s = device_info(&dev, &info)) != GSR_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (seq_kv == 0) {   // no keys at all: every row is empty
        e = gsr::launch_attention_empty(static_cast<__half*>(O), lse, BH * seq_q, (int)head_dim, st);
        return e == cudaSuccess ? GSR_OK : cuda_fail(e);
    }
    StreamState ss;
    if ((s = stream_state(dev, st, 0, 0, &ss)) != GSR_OK) return s;
    if ((s = load_encoder()) != GSR_OK) return s;
    CUtensorMap tmQ, tmK, tmV;
    if ((s = encode_fp16_bsd(&tmQ, Q, BH, seq_q, head_dim)) != GSR_OK) return s;
    if ((s = encode_fp16_bsd(&tmK, K, BH, seq_kv, head_dim)) != GSR_OK) return s;
    if ((s = encode_fp16_bsd(&tmV, V, BH, seq_kv, head_dim)) != GSR_OK) return s;
    const double scale = softmax_scale != 0.0f ? (double)softmax_scale : 1.0 / std::sqrt((double)head_dim);
    gsr::AttnParams p;
    p.BH = (int)BH;
    p.Sq = (int)seq_q;
    p.Skv = (int)seq_kv;
    p.causal = causal ? 1 : 0;
    p.causal_offset = (int)(seq_kv - seq_q);
    p.scale_log2 = (float)(scale * 1.4426950408889634);
    // Causal blocks differ in length (the latest query blocks see the most keys): launch them
    // longest first across as many heads as keep their K and V (seq_kv x head_dim x 4 bytes
    // each) within ~48 MiB of L2; without a mask every block is equally long and one head's
    // blocks run together.
    {
        const uint64_t kv_head = (uint64_t)seq_kv * (uint64_t)head_dim * 4u;
        const bool head_major = (g_test_flags.load(std::memory_order_relaxed) & gsr::kTestAttnHeadMajor) != 0;
        uint64_t g = (causal && !head_major) ? ((uint64_t)48 << 20) / (kv_head ? kv_head : 1) : 1;
        if (g < 1) g = 1;
        if (g > (uint64_t)BH) g = (uint64_t)BH;
        p.head_group = (int)g;
    }
    const int64_t items = (seq_q + 255) / 256 * BH;
    if (items > INT_MAX) return GSR_ERR_INVALID_ARG;
    p.num_items = (int)items;
    p.work = ss.err + 1;
    p.O = static_cast<__half*>(O);
    p.lse = lse;
    p.err = ss.err;
    p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    p.test_flags = g_test_flags.load(std::memory_order_relaxed);
    const int grid = items < info.num_sms ? (int)items : info.num_sms;   // one CTA per SM
    e = gsr::launch_attention(tmQ, tmK, tmV, p, (int)head_dim, grid, st);
    return e == cudaSuccess ? GSR_OK : cuda_fail(e);
}

gsr_status gsr_device_status(CUstream_st* stream, int* code) {
    if (code) *code = 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
    // the allocation-free entry point's error word (one per device; its calls run in order)
    int h_fixed = 0;
    if ((e = gsr::noalloc_take_error(st, &h_fixed)) != cudaSuccess) return cuda_fail(e);
    StreamState s;
    bool have = false;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_streams.find({dev, stream});
        if (it != g_streams.end() && it->second.err) {
            s = it->second;
            have = true;
        }
    }
    int h = 0;
    if (have && (e = cudaMemcpy(&h, s.err, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e);
    if (h == 0) h = h_fixed;
    if (code) *code = h;
    if (h == 0) return GSR_OK;
    if (have) {
        if ((e = cudaMemset(s.err, 0, sizeof(int))) != cudaSuccess) return cuda_fail(e);
        // The small-M kernel leaves its tickets at zero even when it gives up; clearing them
        // here as well costs nothing and does not depend on it.
        if (s.tickets && (e = cudaMemset(s.tickets, 0, s.ticket_count * sizeof(int))) != cudaSuccess)
            return cuda_fail(e);
    }
    return GSR_ERR_DEVICE_TIMEOUT;
}

gsr_status gsr_release_stream(CUstream_st* stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    StreamState s;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_streams.find({dev, stream});
        if (it == g_streams.end()) return GSR_OK;
        s = it->second;
        g_streams.erase(it);
    }
    // Kernels queued earlier on the stream may still use the memory.
    e = cudaStreamSynchronize(st);
    cudaError_t e1 = cudaFree(s.err), e2 = cudaFree(s.partials), e3 = cudaFree(s.tickets);
    if (e == cudaSuccess) e = e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3);
    return e == cudaSuccess ? GSR_OK : cuda_fail(e);
}

int gsr_select_path(int64_t M, int64_t N, int64_t K) {
    int sms = kDefaultSms;
    int dev = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (cudaGetDevice(&dev) == cudaSuccess) {
            auto it = g_devices.find(dev);
            if (it != g_devices.end()) sms = it->second.num_sms;
        }
    }
    return choose_path(M, N, K, sms);
}

void gsr_set_path_override(int path) { g_path_override.store(path, std::memory_order_relaxed); }

void gsr_set_wait_timeout_ns(uint64_t ns) {
    g_timeout_ns.store(ns ? ns : 1, std::memory_order_relaxed);
}

void gsr_set_raster_group(int group) { g_raster_group.store(group > 0 ? group : 0, std::memory_order_relaxed); }

void gsr_set_split_k(int slabs) { g_split_k.store(slabs > 0 ? slabs : 0, std::memory_order_relaxed); }

void gsr_set_test_flags(uint32_t flags) { g_test_flags.store(flags, std::memory_order_relaxed); }

int gsr_last_cuda_error(void) { return t_last_cuda_error; }

const char* gsr_status_string(gsr_status s) {
    switch (s) {
        case GSR_OK: return "GSR_OK";
        case GSR_ERR_INVALID_ARG: return "GSR_ERR_INVALID_ARG";
        case GSR_ERR_ALIGNMENT: return "GSR_ERR_ALIGNMENT";
        case GSR_ERR_ALIAS: return "GSR_ERR_ALIAS";
        case GSR_ERR_CUDA: return "GSR_ERR_CUDA";
        case GSR_ERR_DEVICE_TIMEOUT: return "GSR_ERR_DEVICE_TIMEOUT";
        case GSR_ERR_UNSUPPORTED_DEVICE: return "GSR_ERR_UNSUPPORTED_DEVICE";
        case GSR_ERR_SCRATCH_LIMIT: return "GSR_ERR_SCRATCH_LIMIT";
    }
    return "GSR_ERR_UNKNOWN";
}

const char* gsr_version(void) { return "gsr 0.1.0 sm_103a"; }

gsr_status gsr_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = -1;
    cudaGetDevice(&cur);
    gsr_status result = GSR_OK;
    for (auto& kv : g_streams) {
        if (cudaSetDevice(kv.first.first) != cudaSuccess) continue;
        StreamState& s = kv.second;
        cudaError_t e1 = cudaFree(s.err), e2 = cudaFree(s.partials), e3 = cudaFree(s.tickets);
        if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess) {
            result = cuda_fail(e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3));
        }
    }
    g_streams.clear();
    for (auto& kv : g_pipes) {
        if (cudaSetDevice(kv.first) != cudaSuccess) continue;
        HostPipe* hp = kv.second;
        cudaStreamSynchronize(hp->h2d);
        cudaStreamSynchronize(hp->d2h);
        for (cudaEvent_t ev : hp->ev) cudaEventDestroy(ev);
        cudaStreamDestroy(hp->h2d);
        cudaStreamDestroy(hp->d2h);
        delete hp;
    }
    g_pipes.clear();
    if (cur >= 0) cudaSetDevice(cur);
    return result;
}

}  // extern "C"
