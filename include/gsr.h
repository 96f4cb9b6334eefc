/*
 * gsr.h - fused GEMM + scale + ReLU on GB300 (sm_103a):
 *
 *     C[m,n] = ReLU( alpha * sum_{k=0}^{K-1} A[m,k] * B[k,n] )
 *
 * Operator definition: "Tutorial14: 使用TileLang语言编写attention算子" (PKUHPC
 * scow-tutorial), section 3 (算子介绍) gives the formula and ReLU(x) = max(x, 0);
 * section 2 (编写算子), the gemm_fused kernel, fixes the data types (A, B, C
 * float16, accumulator float32, scale float32) and the order of the epilogue
 * (multiply by the scale first, then the max with 0, then the fp16 store).
 *
 * Plain C ABI: pointers and sizes only.  Every entry point returns a
 * gsr_status and never aborts the process.  Entry points that launch work are
 * asynchronous on the given stream: returning GSR_OK means the work was
 * queued, not that it finished.  A NULL stream is the legacy default stream.
 * Thread-safety: the entry points may be called from several host threads.
 */
#ifndef GSR_H_
#define GSR_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; declared here so this header needs no
 * CUDA header. */
struct CUstream_st;

typedef enum gsr_status {
    GSR_OK = 0,
    /* A negative size, a size above 2^31 - 1, a NULL pointer where data is
     * needed, or a NULL stream pointer argument where one is required. */
    GSR_ERR_INVALID_ARG = 1,
    /* A, B or C not 16-byte aligned, or N or K not a multiple of 8 (the tensor
     * copy engine needs every row pitch to be a multiple of 16 bytes). */
    GSR_ERR_ALIGNMENT = 2,
    /* C overlaps A or B. */
    GSR_ERR_ALIAS = 3,
    /* A CUDA runtime call failed; gsr_last_cuda_error() has its code. */
    GSR_ERR_CUDA = 4,
    /* A kernel gave up on a bounded wait (reported by gsr_device_status). */
    GSR_ERR_DEVICE_TIMEOUT = 5,
    /* The current device is not compute capability 10.3 (GB300). */
    GSR_ERR_UNSUPPORTED_DEVICE = 6,
    /* gemm_scale_relu_noalloc: these sizes need more scratch than its fixed
     * array holds. */
    GSR_ERR_SCRATCH_LIMIT = 7
} gsr_status;

/*
 * C = ReLU(alpha * A.B).
 *
 *   A      device pointer, M x K float16, row-major (row stride K elements).
 *   B      device pointer, K x N float16, row-major (row stride N elements).
 *   C      device pointer, M x N float16, row-major (row stride N elements);
 *          written, never read.  Must not overlap A or B.
 *   M,N,K  sizes, 0 <= M, N, K <= 2^31 - 1; N and K multiples of 8.
 *   alpha  float32 scale, applied to the float32 sum before the ReLU.
 *   stream CUDA stream the work is queued on (NULL: legacy default stream).
 *
 * All three buffers are owned by the caller and must stay valid until the
 * work on `stream` has finished.  Results: the sum is carried in float32 on
 * the tensor cores and rounded once to float16 (nearest, ties to even).
 * ReLU of -0 or NaN gives 0.  M == 0 or N == 0: nothing to do, GSR_OK.
 * K == 0: C is filled with zeros (ReLU(alpha * 0)).
 *
 * Paths: M <= 64 runs the small-M kernel (B streamed once, K split across
 * SMs) when B holds at least 16 MiB, and so do 65 to 128 rows when B is large and
 * the tiles below would leave SMs idle; larger M runs a tiled kernel, on CTA pairs with 256 x 256 tiles when
 * there are enough of them to fill the GPU (or K is long), else one CTA per
 * 128-row tile (gsr_select_path gives the rules).
 *
 * Device memory the library owns: on the first call on each (device, stream)
 * pair it allocates 16 bytes for that stream (the kernels' error word and the
 * attention kernel's work counters), and the small-M kernel keeps fp32 partial
 * tiles and per-tile ticket counters in a workspace allocated (or grown) on the
 * first small-M call on the pair.  Both stay until gsr_release_stream() for that
 * stream or gsr_shutdown().  Calls on different streams never share them; such a
 * first call synchronises its stream and so should not be made during stream
 * capture.  Once a stream has seen a call of the same kind (and size, for the
 * small-M workspace), further calls on it only encode tensor maps on the host
 * and launch, so they can be captured into a CUDA graph and replayed; a
 * replay reads whatever the captured buffers hold then.  A captured call keeps
 * using the capture stream's library memory (error word, attention work
 * counters, small-M workspace): replays must not run at the same time as each
 * other or as other library calls on that stream.
 */
gsr_status gemm_scale_relu(const void* A, const void* B, void* C, int64_t M, int64_t N,
                           int64_t K, float alpha, struct CUstream_st* stream);

/*
 * C = alpha * A.B, the same GEMM without the ReLU; alpha = 1 gives the plain
 * tiled matrix product.  ("TileLang: создание высокопроизводительных GPU-ядер"
 * survey page, section 2 "Тилированное умножение матриц": make_matmul, the plain
 * tiled tensor-core GEMM the fused operator extends.)  Arguments, layout,
 * ownership, paths and errors as for gemm_scale_relu; K == 0 gives zeros.
 */
gsr_status gemm_scale(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                      float alpha, struct CUstream_st* stream);

/*
 * C[m,n] = GELU( sum_k A[m,k] * B[k,n] + bias[n] ), GELU in its tanh form
 * 0.5 x (1 + tanh( sqrt(2/pi) (x + 0.044715 x^3) )), computed in fp32 on the
 * accumulator before the fp16 store.  (Same survey page, section 4 "Слияние
 * эпиколов: GEMM + Bias + GELU": make_matmul_bias_gelu adds the bias and applies
 * an exponential-formula GELU approximation in registers.)
 *
 *   bias   device pointer to N float16 values, 16-byte aligned, must not
 *          overlap C; read, never written.
 * Other arguments, paths and errors as for gemm_scale_relu.  K == 0 gives
 * C[m,n] = GELU(bias[n]).
 */
gsr_status gemm_bias_gelu(const void* A, const void* B, const void* bias, void* C, int64_t M,
                          int64_t N, int64_t K, struct CUstream_st* stream);

/*
 * Attention forward, FlashAttention style:
 *
 *     O = softmax( softmax_scale * Q K^T  [causal mask] ) V        per batch and head
 *
 * (aikraft.ru TileLang tutorial survey "TileLang: создание высокопроизводительных
 * GPU-ядер", section 6 "FlashAttention: Слияние внимания": online softmax with running
 * maxima, normalisation sums and rescaling factors, causal masks, pipelined copies.)
 *
 *   Q      device pointer, (batch, heads, seq_q, head_dim) float16, row-major.
 *   K, V   device pointers, (batch, heads, seq_kv, head_dim) float16, row-major.
 *   O      device pointer, (batch, heads, seq_q, head_dim) float16; written.
 *   lse    optional device pointer (NULL: not written), (batch, heads, seq_q) float32:
 *          the natural-log log-sum-exp of each query's scaled, masked scores.
 *   head_dim        64 or 128.
 *   softmax_scale   0 selects 1/sqrt(head_dim).
 *   causal          nonzero: query i keeps key j only when j <= i + (seq_kv - seq_q)
 *                   (lower triangle aligned to the bottom-right corner).
 * Scores and softmax in fp32, P rounded to fp16 for the second product, output rounded
 * once to fp16.  A query with no key left (causal with seq_q > seq_kv, or seq_kv == 0)
 * gets O = 0 and lse = -inf.  All pointers 16-byte aligned (lse 4-byte); O and lse must
 * not overlap the inputs or each other.  Caller-owned buffers; asynchronous on `stream`;
 * errors as for gemm_scale_relu.
 */
gsr_status flash_attention_fwd(const void* Q, const void* K, const void* V, void* O, float* lse,
                               int64_t batch, int64_t heads, int64_t seq_q, int64_t seq_kv,
                               int64_t head_dim, float softmax_scale, int causal,
                               struct CUstream_st* stream);

/*
 * gemm_scale_relu with the operands in host memory: copies A and B host ->
 * device into the caller's device buffers dA and dB, runs gemm_scale_relu
 * into dC and copies C back device -> host, all ordered on `stream`: the call
 * starts after the work already queued there, and work queued after it sees hC
 * complete.  The host buffers should be page-locked (cudaHostAlloc / pinned) for
 * the copies to be asynchronous.  Sizes, alignment and errors as for
 * gemm_scale_relu; dC must not overlap dA or dB.
 * From 2^33 flop (~8.6 GFLOP) and 1024 rows up the three parts overlap: A is copied
 * in 2..8 chunks of rows, and B whole or, where C has more elements than A and B
 * together, in 2..4 blocks of columns (each a multiple of 256 columns, wide enough
 * for a full wave of the CTA-pair kernel); the product of each chunk of rows and
 * block of columns runs on `stream` as soon as both have landed, and that block of
 * C goes back (a strided copy) while later ones are copied in.  dB and dC then
 * hold the whole matrices as for gemm_scale_relu; only the order in which their
 * parts are written changes.  The copies run on two library-owned streams per device (one
 * per direction, joined to `stream` by library-owned events; created on first
 * use, released by gsr_shutdown), and concurrent calls on one device queue their
 * copies one call after the other.
 */
gsr_status gemm_scale_relu_host(const void* hA, const void* hB, void* hC, void* dA, void* dB,
                                void* dC, int64_t M, int64_t N, int64_t K, float alpha,
                                struct CUstream_st* stream);

/*
 * gemm_scale_relu without any device-memory allocation, for callers that cannot
 * let a library allocate: for example a serving runtime that plans all of its
 * device memory at start-up and forbids allocations afterwards, or a
 * latency-critical loop that cannot take the implicit synchronisation of a
 * first-time cudaMalloc.  (No counterpart on the pages: they allocate through
 * the TileLang JIT and PyTorch.)
 *
 * Arguments, layout, ownership and result are those of gemm_scale_relu, for
 * the small-M kernel only: 1 <= M <= 64 (M > 64 returns GSR_ERR_INVALID_ARG;
 * M == 0 or N == 0 is a no-op and K == 0 clears C, as there).  The small-M kernel
 * has no raster order to set: gsr_set_raster_group does not apply to it.  The caller
 * passes A, B and C; the kernel's scratch (error word, per-tile tickets and
 * split-K partial tiles) lives in one fixed 12 MiB array inside the library,
 * which every GPU that loads the library holds until the process exits.
 * Sizes whose scratch would not fit return GSR_ERR_SCRATCH_LIMIT before any
 * work is queued; on a 152-SM GB300 that happens only for N above about 4.0e8
 * (sizes whose per-tile tickets alone cannot fit are refused before any CUDA
 * call).  The call never runs cudaMalloc, cudaFree or any other allocating
 * routine.
 *
 * Set-up: the first call on each device, with that device current, looks up the
 * array's device address and makes the kernel variants resident.  Under CUDA's
 * default lazy module loading, that is when the driver places the array and the
 * kernels' code on the device: an allocation by the driver, which can also
 * synchronise.  A caller with a fixed memory plan should therefore make one call
 * on each device during start-up.  Later calls place nothing.
 *
 * Every call shares the array and it keeps the last call's contents; each call
 * clears the parts that must start at zero, on `stream`, before its kernel.
 * Calls whose work overlaps on the GPU (for example on two streams with no
 * ordering between them) race on the array and produce wrong results: order
 * them on one stream.  If a bounded wait inside the kernel runs out, C is left
 * unspecified; gsr_device_status reports GSR_ERR_DEVICE_TIMEOUT for the most
 * recent call of this entry point on the current device, until it has been read
 * once or the next call starts.  It reads the word after the work of the stream it
 * is given: pass the stream the call was queued on (or one ordered after it).
 */
gsr_status gemm_scale_relu_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N,
                                   int64_t K, float alpha, struct CUstream_st* stream);

/*
 * Waits for `stream`, then reads and clears the error word of the (current
 * device, stream) pair, and that of gemm_scale_relu_noalloc on the current device.
 * Returns GSR_ERR_DEVICE_TIMEOUT if a kernel queued on that stream since the last
 * call (or the latest gemm_scale_relu_noalloc call on the device) gave up on a
 * bounded wait, GSR_ERR_CUDA if the stream reported an error, else GSR_OK.  The
 * output of the call that gave up is unspecified; later calls are correct
 * whether or not this function is called (the small-M kernel leaves its ticket
 * counters at zero even when it gives up).  `code` (may be NULL) receives the raw
 * device error code, 0 if none: low byte = which wait gave up (1 producer
 * waiting for a free stage, 2 MMA issuer waiting for loaded data, 3 MMA issuer
 * waiting for a free accumulator, 4 epilogue waiting for a finished
 * accumulator, 5 teardown drain, 6 shared-memory window not 1024-byte aligned:
 * the kernel returned at once), 0x100 = tiled kernel, 0x200 = small-M,
 * 0x300 = attention.
 */
gsr_status gsr_device_status(struct CUstream_st* stream, int* code);

/*
 * Releases the library's state for the (current device, stream) pair: the
 * stream's 16 bytes of words and, if a small-M call ran on it, its workspace.
 * Waits for the stream first (queued kernels may still use them).  For callers
 * that create and destroy streams: call it before destroying a stream the
 * library was used on, from no other thread launching on that stream at the same
 * time.  A later call on the stream allocates afresh.  GSR_OK if the pair holds
 * nothing; GSR_ERR_CUDA if the wait or a free failed.
 */
gsr_status gsr_release_stream(struct CUstream_st* stream);

/* Kernel the library would run for these sizes on the current device: 0 = tiled
 * (one CTA per 128-row tile, 128 x 256, 128 x 128 or 128 x 64 tiles, whichever
 * needs fewer waves with a wave of 256-wide tiles counted as 1.45 and one of 64-wide
 * tiles as 0.9 of a wave of 128-wide ones), 1 = small-M (M <= 64 with B of at
 * least 16 MiB, and 65 to 128
 * rows when B holds at least 64 MiB and those one-CTA tiles would keep under two
 * thirds of the SMs busy),
 * 2 = tiled on CTA pairs with 256 x 256 tiles (for more than 128 rows and K above
 * 384, where a tile is more than its epilogue, chosen when
 * there is at least one full wave of such tiles, or when K >= 6144 and 0 would use
 * 128 x 256 tiles: the pair's faster K loop then repays its larger cost per launch;
 * at 128 rows or fewer a pair tile would be at least half empty), 3 = tiled on CTA
 * pairs with 256 x 128 tiles (instead
 * of 2 where a wave of them, counted as 0.68 of a wide wave, finishes the work at
 * least 5 % sooner: in practice N of about 128, where a 256-wide tile is half
 * empty).  The constants come from measured sweeps on GB300. */
int gsr_select_path(int64_t M, int64_t N, int64_t K);

/* Forces a path for later calls (process-wide): 0 = automatic (default),
 * 1 = tiled with automatic tile width, 2 = small-M (only honoured when
 * M <= 256: 65 to 256 rows run with an MMA N of 128 or 256, which the automatic
 * choice takes only for the 65-128-row case above; the host-buffer entry point's
 * blocks ignore it),
 * 3 = tiled with 128 x 256 tiles, 4 = tiled with 128 x 128 tiles,
 * 5 = tiled on CTA pairs with 256 x 256 tiles, 6 = tiled on CTA pairs with
 * 256 x 128 tiles, 7 = tiled with 128 x 64 tiles.
 * For tests and measurements. */
void gsr_set_path_override(int path);

/* Raster grouping of the tiled kernels (process-wide): `group` consecutive tile rows
 * (M blocks) share each tile column before moving on, so that concurrently running
 * CTAs reuse the same A and B panels from L2 -- the "L2 swizzle" knob of the aikraft.ru
 * TileLang tutorial survey's "Knobs" section (3).  0 restores the default, 16 row
 * blocks per group (128-row blocks for one CTA per tile, 256-row blocks for CTA pairs).
 * The small-M kernel walks K slabs, not a raster, and ignores it.  For tuning and
 * measurements. */
void gsr_set_raster_group(int group);

/* Split-K of the small-M kernel (process-wide): each 128-column tile's K is cut
 * into `slabs` slabs of whole 64-wide k-blocks (at most one slab per k-block), run
 * as separate work items and summed in slab order (deterministic for a given
 * `slabs`).  0 restores the default, as many slabs as fill the SMs once.  The
 * split-K knob of the aikraft.ru TileLang tutorial survey's "Knobs" section (3);
 * for tuning and measurements.  gemm_scale_relu_noalloc ignores it (its fixed
 * scratch is sized for the default split). */
void gsr_set_split_k(int slabs);

/* Upper bound, in nanoseconds, on every wait inside the kernels (default 1 s).
 * A wait that runs out records an error (see gsr_device_status) and the kernel
 * exits early, leaving C incomplete. */
void gsr_set_wait_timeout_ns(uint64_t ns);

/* Test-only switches, 0 in normal use.  Bit 0: the first CTA's producer skips
 * its first shared-memory fill, so that CTA's waits run out (exercises the
 * bounded-wait path without faulting the GPU).  Bit 1: the tiled kernels copy B
 * as separate 64-column boxes even where one 3-D copy per stage would do.
 * Bits 2-7 switch off or swap what the CTA-pair and attention kernels normally
 * do, for measurements: bit 2 every wave of pair tiles walks K forward (no
 * serpentine order); bit 3 C stores without the L2 evict-first hint; bit 4 the
 * first pair's second CTA skips its first fill (like bit 0, on the other CTA);
 * bit 5 / bit 6 B copies with an L2 evict-first / evict-normal hint instead of
 * evict-last; bit 7 causal attention launches one head's query blocks at a time. */
void gsr_set_test_flags(uint32_t flags);

/* CUDA error code of the last failing CUDA call on this host thread (0: none). */
int gsr_last_cuda_error(void);

/* Static, human-readable name of a status. */
const char* gsr_status_string(gsr_status s);

/* Library version string, e.g. "gsr 0.1.0 sm_103a". */
const char* gsr_version(void);

/* Frees every workspace and error word the library holds, on every device.
 * Must not run while work queued by the library is still executing. */
gsr_status gsr_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* GSR_H_ */
