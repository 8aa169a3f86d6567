/*
 * tk_cast.h -- C ABI of the GB300 per-token group-wise activation cast.
 *
 * The operation (TileKernels README, section "Features": "per-token ...
 * FP8/FP4 casting ... with fused SwiGLU+quantization"; aiwiki "TileKernels",
 * section "Quantization": scale-factor groups of 16, 32, 64 or 128 channels,
 * power-of-two rounding of scale factors, packed UE8M0 scale factors, and
 * per-token scale factors "in DeepGEMM's layout"):
 *
 *   for every row m (a token) and every group j of `group` consecutive
 *   channels of that row:
 *     amax  = max |x[m, k]| over the group           (fp32, exact)
 *     r     = max(amax, 1e-4f) / fmt_max              (one IEEE fp32 division)
 *     scale = r                      (TK_SCALE_FP32)
 *           = 2^ceil(log2 r)         (TK_SCALE_FP32_POW2, TK_SCALE_UE8M0_PACKED)
 *     code  = round-to-nearest-even(saturate(x / scale, +-fmt_max))
 *             with x / scale one IEEE fp32 division (for a power-of-two scale
 *             the exact product by 2^-k, which is the same number)
 *   fmt_max = 448 for FP8 E4M3 (OCP E4M3FN), 6 for FP4 E2M1 (OCP MX).
 *   The sign of x is kept on every code, zeros included.
 *
 * Conventions shared by every entry point:
 *  - All data pointers are DEVICE pointers (global memory of the current
 *    CUDA device), except the x, codes and scales of the two *_host entry
 *    points.  The caller allocates and owns every buffer; the library
 *    allocates nothing and keeps no pointer after the call returns.
 *  - Calls are asynchronous: they validate on the host, enqueue their work
 *    on `stream` (a cudaStream_t passed as void*, NULL = legacy default
 *    stream; one kernel, except tk_per_channel_cast) and return.  Outputs
 *    are ready once the stream reaches that point.  Input and outputs must
 *    not overlap.
 *  - Inputs must be finite; NaN/Inf inputs give unspecified codes/scales.
 *  - Errors are returned, never raised: nothing aborts or throws across
 *    the ABI, and nothing is launched when a check fails.
 *  - Alignment (TK_ERR_MISALIGNED otherwise; there is no scalar fallback):
 *    x and codes 16-byte aligned; row strides ld_x * 2 bytes and ld_codes
 *    bytes multiples of 16; scales 4-byte aligned; for the transposed layout
 *    ld_scales a multiple of 4 (16-byte aligned scale rows).
 *  - Entries of the scale tensor outside the written region (row-major
 *    columns past the last word, transposed columns m >= M) are left
 *    untouched, as are code bytes past each row's K (or K/2) bytes.
 *  - M == 0 is a no-op that returns TK_OK without looking at the pointers.
 *  - Limits: 0 <= M <= 2^30, K (or N) <= 2^28 (TK_ERR_UNSUPPORTED beyond).
 */
#ifndef TK_CAST_H
#define TK_CAST_H

#include <stddef.h>
#include <stdint.h>

/* Exported from the shared library even when it is built with hidden
 * default visibility. */
#if defined(__GNUC__)
#define TK_API __attribute__((visibility("default")))
#else
#define TK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TK_OK = 0,
    TK_ERR_INVALID_ARG = 1,  /* bad enum, group, shape, stride or null ptr */
    TK_ERR_UNSUPPORTED = 2,  /* a size beyond the stated limits */
    TK_ERR_MISALIGNED = 3,   /* pointer or stride breaks the alignment rule */
    TK_ERR_CUDA = 4          /* the launch failed (see tk_last_cuda_error) */
} tk_status;

typedef enum {
    TK_FMT_E4M3 = 0,  /* FP8 E4M3FN, 1 byte per code */
    TK_FMT_E2M1 = 1   /* FP4 E2M1, 2 codes per byte, element 2i in bits 3:0 */
} tk_format;

typedef enum {
    TK_SCALE_FP32 = 0,         /* fp32 scale r */
    TK_SCALE_FP32_POW2 = 1,    /* fp32 scale 2^k, the smallest power of two >= r */
    TK_SCALE_UE8M0_PACKED = 2  /* the byte 127 + k, four per int32 word:
                                  group 4w+b in byte b of word w (little endian);
                                  unused bytes of a partial last word are 0 */
} tk_scale_mode;

typedef enum {
    /* [M][ld_scales] words: ld_scales >= G (fp32) or ceil(G/4) (packed). */
    TK_SCALE_ROW_MAJOR = 0,
    /* DeepGEMM's per-token layout: [G or ceil(G/4)][ld_scales] words with
     * ld_scales >= M and a multiple of 4 (M padded, e.g. M_pad = ceil(M/4)*4).
     * Word (j, m) holds row m's scale of group j (packed: groups 4j..4j+3). */
    TK_SCALE_TRANSPOSED_PADDED = 1
} tk_scale_layout;

typedef enum {
    TK_OUT_BF16 = 0,  /* dequantized values rounded to BF16 (nearest even) */
    TK_OUT_FP32 = 1   /* dequantized values as fp32 */
} tk_out_dtype;

/*
 * tk_per_token_cast -- per-token group-wise cast of a BF16 matrix.
 *
 *   x         BF16 [M][ld_x] row-major, K values used per row.
 *   M, K      rows (tokens) and channels; K % group == 0.
 *   ld_x      input row stride in elements, >= K.
 *   group     channels per scale: 16, 32, 64 or 128.
 *   fmt       tk_format.  mode: tk_scale_mode.  layout: tk_scale_layout.
 *   codes     uint8 [M][ld_codes]: K bytes (E4M3) or K/2 bytes (E2M1) per row.
 *   ld_codes  code row stride in bytes, >= the row's code bytes.
 *   scales    fp32 or int32 words laid out per `layout`, G = K / group.
 *   ld_scales scale row stride in 4-byte words (see tk_scale_layout).
 *   stream    cudaStream_t as void*.
 */
TK_API tk_status tk_per_token_cast(const void *x, int64_t M, int64_t K, int64_t ld_x,
                            int group, int fmt, int mode, int layout,
                            void *codes, int64_t ld_codes, void *scales,
                            int64_t ld_scales, void *stream);

/*
 * tk_swiglu_per_token_cast -- fused SwiGLU + per-token cast (TileKernels
 * README, "Features": "fused SwiGLU+quantization ops"; the activation and the
 * narrowing happen in one pass with no intermediate tensor in memory).
 *
 *   x         BF16 [M][ld_x], row m = [gate (N values) | up (N values)].
 *   y[m, k] = silu(gate[m, k]) * up[m, k] = gate*up / (1 + e^-gate), in fp32,
 *   then cast exactly as tk_per_token_cast casts a row of K = N values.
 *   ld_x >= 2N.  Other arguments as for tk_per_token_cast with K = N.
 *   Scales: each group's amax is taken from products re-evaluated to about
 *   2^-44 relative, so scales equal those of the correctly rounded product
 *   except (rarely) by one fp32 ulp.  Codes: computed from the fp32 product
 *   (expf and one IEEE division, within a few ulps), so a small fraction of
 *   codes can differ by one step from a cast of the correctly rounded one.
 *   gate * up must be finite in fp32 (|gate * up| < 2^128).
 */
TK_API tk_status tk_swiglu_per_token_cast(const void *x, int64_t M, int64_t N,
                                   int64_t ld_x, int group, int fmt, int mode,
                                   int layout, void *codes, int64_t ld_codes,
                                   void *scales, int64_t ld_scales,
                                   void *stream);

/*
 * Host-buffer forms of tk_per_token_cast and tk_swiglu_per_token_cast: the
 * same operation on rows that live in HOST memory, with codes and scales
 * delivered to host memory.  These are the only entry points that take
 * host pointers and the only ones that block: they return once the
 * outputs are in host memory (or after a failure, once everything they
 * enqueued has finished).
 *
 *   x, codes, scales   HOST buffers with the layouts, strides and
 *             arguments of tk_per_token_cast (tk_swiglu_per_token_cast: x
 *             holds [gate | up], K = N).  No alignment rule applies to
 *             them; page-locked (pinned) memory lets the copies run
 *             asynchronously and overlap.  Scale entries outside the
 *             written region and code bytes past each row's K (K/2) bytes
 *             are left untouched, as on the device.
 *   scratch   DEVICE memory of at least tk_host_scratch_bytes(...) bytes
 *             (same M, K, group, fmt, mode, layout; swiglu 1 for the SwiGLU
 *             form), 16-byte aligned, owned by the caller and not in use by
 *             pending work on either stream; nothing is read from it.
 *   chunk_rows   rows per chunk (rounded down to a multiple of 4, at least
 *             4); 0 splits M into about 4 chunks of at least 4 MiB of input
 *             each (rounded up to a multiple of 4 rows).
 *   streams, n_streams   an array of 1 to 64 cudaStream_t (as void*; NULL
 *             entries mean the legacy default stream); chunk i goes to
 *             streams[i % n_streams].  Each chunk's upload, cast and download
 *             run in order on its stream, so uploads overlap earlier chunks'
 *             casts and downloads; an upload waits only for the download of
 *             the chunk n_streams places earlier, so 3 or 4 distinct streams
 *             keep the upload engine busy.  Entries may repeat (one stream:
 *             the chunks run one after another).
 *   Errors as for tk_per_token_cast, plus TK_ERR_INVALID_ARG for a scratch
 *   smaller than required, chunk_rows < 0, or a bad stream array,
 *   TK_ERR_MISALIGNED for an unaligned scratch, and TK_ERR_CUDA for a
 *   failed copy or wait.
 */
TK_API size_t tk_host_scratch_bytes(int64_t M, int64_t K, int group, int fmt,
                                    int mode, int layout, int swiglu);

TK_API tk_status tk_per_token_cast_host(const void *x, int64_t M, int64_t K,
                                        int64_t ld_x, int group, int fmt,
                                        int mode, int layout, void *codes,
                                        int64_t ld_codes, void *scales,
                                        int64_t ld_scales, void *scratch,
                                        size_t scratch_bytes,
                                        int64_t chunk_rows,
                                        void *const *streams, int n_streams);

TK_API tk_status tk_swiglu_per_token_cast_host(const void *x, int64_t M,
                                               int64_t N, int64_t ld_x,
                                               int group, int fmt, int mode,
                                               int layout, void *codes,
                                               int64_t ld_codes, void *scales,
                                               int64_t ld_scales,
                                               void *scratch,
                                               size_t scratch_bytes,
                                               int64_t chunk_rows,
                                               void *const *streams,
                                               int n_streams);

/*
 * tk_per_token_dequant -- per-token dequantization (TileKernels README,
 * "Features": "FP8/FP4 casting and dequantization"): the inverse of the cast.
 *
 *   y[m, k] = value(code[m, k]) * scale(m, k / group)
 *   one IEEE fp32 multiply; value() decodes E4M3FN / E2M1 exactly; the scale
 *   is read from a tensor laid out as tk_per_token_cast writes it (fp32, or
 *   packed UE8M0 byte e giving 2^(e-127)).  Output fp32, or rounded to BF16
 *   with round-to-nearest-even (out_dtype, tk_out_dtype).
 *
 *   codes     uint8 [M][ld_codes] (K or K/2 bytes used per row), 16-byte
 *             aligned, ld_codes a multiple of 16.  For E2M1 with K not a
 *             multiple of 32, the kernel reads each row up to the next
 *             16-byte boundary: the buffer must span M * ld_codes bytes.
 *   scales    as for tk_per_token_cast with the same mode/layout/ld_scales.
 *   y         [M][ld_y] elements of out_dtype, 16-byte aligned,
 *             ld_y * sizeof(element) a multiple of 16, ld_y >= K.
 *   Codes that the cast never writes still decode: the E4M3 NaN pattern
 *   gives NaN, and a product beyond the output range gives +-inf.
 */
TK_API tk_status tk_per_token_dequant(const void *codes, int64_t ld_codes,
                                      const void *scales, int64_t ld_scales,
                                      int64_t M, int64_t K, int group, int fmt,
                                      int mode, int layout, void *y,
                                      int64_t ld_y, int out_dtype,
                                      void *stream);

/*
 * tk_per_token_cast_back -- per-token cast-and-cast-back (aiwiki
 * "TileKernels", section "Version 2.0.0": "per-token cast-and-cast-back"):
 * each row is cast exactly as tk_per_token_cast casts it, and the codes are
 * dequantized again in the same pass (as tk_per_token_dequant with BF16
 * output), so y holds the BF16 values the quantized tensor represents.
 * Neither codes nor scales are written.
 *
 *   x    BF16 [M][ld_x] as for tk_per_token_cast.
 *   y    BF16 [M][ld_y], 16-byte aligned, ld_y * 2 a multiple of 16, ld_y >= K.
 *   group, fmt, mode: as for tk_per_token_cast (no scale layout: no scales).
 */
TK_API tk_status tk_per_token_cast_back(const void *x, int64_t M, int64_t K,
                                        int64_t ld_x, int group, int fmt,
                                        int mode, void *y, int64_t ld_y,
                                        void *stream);

/*
 * tk_rmsnorm_per_token_cast -- RMSNorm with a fused per-token cast (aiwiki
 * "TileKernels", section "Version 2.0.0": "RMSNorm forward ... with an
 * optional fused FP8 cast").  RMSNorm by its published definition (Zhang
 * and Sennrich, "Root Mean Square Layer Normalization", 2019):
 *   y[m, k] = w[k] * x[m, k] / sqrt(eps + (1/K) * sum_j x[m, j]^2)
 * then y is cast exactly as tk_per_token_cast casts a row (no BF16
 * intermediate).  The kernel works in fp32: the sum of squares by fused
 * multiply-adds in a fixed order, rstd = rsqrtf(sum * RN(1/K) + eps), and
 * y = RN((x * w) * rstd), where x * w is exact.  Against y formed exactly,
 * y is within about 25 fp32 ulps (K <= 8192), so fp32 scales can differ
 * from an exact evaluation by that many ulps (power-of-two scales only
 * next to a power of two), and a code by one step where the exact quotient
 * lies that close to a rounding midpoint.
 *
 *   x         BF16 [M][ld_x], K values per row; K <= 8192 (one row per
 *             pipeline stage; TK_ERR_UNSUPPORTED beyond).
 *   w         BF16 [K], the per-channel gain; 16-byte aligned.
 *   eps       finite and >= 0 (TK_ERR_INVALID_ARG otherwise); a row of
 *             zeros needs eps > 0 (0/0 otherwise: unspecified codes).
 *   Other arguments as for tk_per_token_cast; y must be finite.
 */
TK_API tk_status tk_rmsnorm_per_token_cast(const void *x, const void *w,
                                           int64_t M, int64_t K, int64_t ld_x,
                                           float eps, int group, int fmt,
                                           int mode, int layout, void *codes,
                                           int64_t ld_codes, void *scales,
                                           int64_t ld_scales, void *stream);

/* Block edge of tk_per_block_cast (square blocks of rows x channels), and
 * the channel granularity of tk_per_channel_cast's workspace. */
#define TK_BLOCK 128

/*
 * tk_per_block_cast -- per-block cast (TileKernels README, "Features":
 * "per-block ... FP8/FP4 casting"; the pages give no block shape, and this
 * library uses square TK_BLOCK x TK_BLOCK blocks of rows x channels).
 *
 *   Block (i, j) is rows [128 i, 128 i + 128) x channels [128 j, 128 j + 128),
 *   clipped to the matrix (the last block row and column may be partial).
 *   Its elements share one scale, computed as in tk_per_token_cast from the
 *   amax over the whole block; codes as tk_per_token_cast writes them.
 *
 *   x         BF16 [M][ld_x], K values used per row; K % 16 == 0, ld_x >= K.
 *   codes     uint8 [M][ld_codes]: K bytes (E4M3) or K/2 bytes (E2M1) per row.
 *   scales    4-byte words, [ceil(M/128)][ld_scales]: block (i, j) is fp32
 *             word j of row i, or, for TK_SCALE_UE8M0_PACKED, byte j of row
 *             i's packed words (byte j % 4 of word j / 4; the unused bytes of
 *             a row's last word are set to 0).  ld_scales >= ceil(K/128)
 *             (fp32 modes) or >= ceil(ceil(K/128) / 4) (packed).
 *   fmt, mode tk_format, tk_scale_mode; scales are always row-major.
 */
TK_API tk_status tk_per_block_cast(const void *x, int64_t M, int64_t K,
                                   int64_t ld_x, int fmt, int mode,
                                   void *codes, int64_t ld_codes,
                                   void *scales, int64_t ld_scales,
                                   void *stream);

/* Bytes of workspace tk_per_channel_cast needs for K channels: 4 per
 * channel with K rounded up to a multiple of TK_BLOCK, plus 4 per TK_BLOCK
 * channels rounded up to 16 (0 if K is out of range). */
TK_API size_t tk_per_channel_workspace_bytes(int64_t K);

/*
 * tk_per_channel_cast -- per-channel cast (TileKernels README, "Features":
 * "per-channel ... FP8/FP4 casting"): channel k (column k) shares one scale
 * over all M rows, computed as in tk_per_token_cast from the column's amax;
 * codes as tk_per_token_cast writes them.
 *
 *   x, codes  as for tk_per_block_cast (K % 16 == 0).
 *   scales    a vector: K fp32 words, or ceil(K/4) int32 words of packed
 *             UE8M0 bytes (channel k in byte k % 4 of word k / 4).  4-byte
 *             aligned.
 *   workspace device memory of at least tk_per_channel_workspace_bytes(K)
 *             bytes, 16-byte aligned, owned by the caller, ZERO-FILLED
 *             before its first use (e.g. one cudaMemset).  It holds the
 *             column maxima and per-strip counters during the call, and
 *             every call that completes leaves it zero-filled again, so one
 *             workspace serves any sequence of calls on one stream.  Calls
 *             that may run at the same time (other streams) must not share
 *             a workspace.  If tk_get_device_fault reports a fault, zero it
 *             again before the next call.
 *   Enqueues two kernels on `stream` (column amax, then the cast, which
 *   derives each column's scale from its maximum); x is read twice.
 *   M == 0 writes nothing (no element to take a scale from).
 */
TK_API tk_status tk_per_channel_cast(const void *x, int64_t M, int64_t K,
                                     int64_t ld_x, int fmt, int mode,
                                     void *codes, int64_t ld_codes,
                                     void *scales, void *workspace,
                                     size_t workspace_bytes, void *stream);

/*
 * tk_per_block_dequant, tk_per_channel_dequant -- dequantization of the
 * per-block / per-channel casts' output (TileKernels README, "Features":
 * "per-block, and per-channel FP8/FP4 casting and dequantization"):
 *   y[m, k] = value(code[m, k]) * scale(block of (m, k), or channel k)
 * as tk_per_token_dequant computes it (exact decode, one IEEE fp32
 * multiply, BF16 nearest-even or fp32 out; a UE8M0 byte e is 2^(e-127)).
 *
 *   codes     uint8 [M][ld_codes] as the casts write them (K % 16 == 0),
 *             16-byte aligned, ld_codes a multiple of 16.  Per-block E2M1
 *             codes are read up to the next 16-byte boundary of each row
 *             (as tk_per_token_dequant does): the buffer spans M * ld_codes.
 *   scales    per-block: as tk_per_block_cast writes them, with its
 *             ld_scales (4-byte aligned); per-channel: the scale vector,
 *             16-byte aligned.
 *   y         [M][ld_y] elements of out_dtype (tk_out_dtype), 16-byte
 *             aligned, ld_y * sizeof(element) a multiple of 16, ld_y >= K.
 */
TK_API tk_status tk_per_block_dequant(const void *codes, int64_t ld_codes,
                                      const void *scales, int64_t ld_scales,
                                      int64_t M, int64_t K, int fmt, int mode,
                                      void *y, int64_t ld_y, int out_dtype,
                                      void *stream);

TK_API tk_status tk_per_channel_dequant(const void *codes, int64_t ld_codes,
                                        const void *scales, int64_t M,
                                        int64_t K, int fmt, int mode, void *y,
                                        int64_t ld_y, int out_dtype,
                                        void *stream);

/*
 * tk_per_channel_cast_noalloc -- tk_per_channel_cast without a caller
 * workspace.  The pages have no counterpart: it is an interface for
 * callers that cannot allocate device memory where they call the cast (a
 * C host without a caching allocator, where cudaMalloc and cudaFree
 * synchronise the device; a serving loop that allows no allocation after
 * warm-up).  The workspace is a fixed array in the library's static device
 * memory, one per device.
 *
 *   Arguments and results as for tk_per_channel_cast, with K <= 65536
 *   (TK_ERR_UNSUPPORTED beyond: the array holds the workspace of 65,536
 *   channels, 264,192 bytes).
 *   The first call on each device finds the array (cudaGetSymbolAddress)
 *   and clears it with a synchronous cudaMemset; make that first call
 *   outside any stream capture.
 *   All calls on one device share the array: calls that may overlap in
 *   time (other streams, other host threads) race on it and give wrong
 *   results; the caller must order them (one stream, or events).
 */
TK_API tk_status tk_per_channel_cast_noalloc(const void *x, int64_t M,
                                             int64_t K, int64_t ld_x,
                                             int fmt, int mode, void *codes,
                                             int64_t ld_codes, void *scales,
                                             void *stream);

/*
 * tk_get_device_fault -- read (and optionally clear) the library's device
 * fault words on the current device (the OR of the per-token kernels' word
 * and the per-block / per-channel kernels' word).  Every wait inside the kernels is
 * bounded in time (1 s); a wait that runs out makes the kernel stop, let its
 * own in-flight copies land and return, OR-ing a code into this word:
 *   1 = a consumer waited too long for a tile, 2 = the producer waited too
 *   long for a free stage, 4 = in-flight copies did not land in time.
 * 0 means no kernel has given up.  Synchronous (device-to-host copy of one
 * word); TK_ERR_INVALID_ARG for a null pointer, TK_ERR_CUDA if the copy fails.
 */
TK_API tk_status tk_get_device_fault(unsigned int *fault, int clear);

/* Static string naming a status value ("TK_OK", ...). */
TK_API const char *tk_status_string(int status);

/* Text of the CUDA error behind the calling thread's most recent
 * TK_ERR_CUDA, or "" if there was none.  Static or thread-local storage. */
TK_API const char *tk_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TK_CAST_H */
