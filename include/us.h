/*
 * us.h -- C ABI of libus, a GB300 (sm_103a) library for unstructured-sparse
 * weight matrices stored as bitmap tiles, multiplied by tall-skinny
 * activations:  Y = W . X.
 *
 * Sources.  The stored format is the Index-Efficient Bitmap Encoding of
 * "UnionSparse: An Index-Efficient Sparsity Framework for Low-Bit Sparse LLM
 * Inference on Edge" (section V-A: Union Bitmaps, Union Value Offsets,
 * Compressed Values, Fig. 7) with one area per tile (Q = 1), in its row-major
 * scan or in the column-major tile scan of the Tiled-CBC format of "Unified
 * Static-Dynamic Pruning for Efficient LLM Inference" (section 4.1), with the
 * 16-byte value padding of that page's section 4.2.3.  The products follow
 * UnionSparse Fig. 2 (INT4 x INT4 -> INT32 -> dequantised FP16) and SPDP
 * section 2 / 4.2 (static mask W (.) M, dynamic mask W (.) M(x), spMspV).
 *
 * ---------------------------------------------------------------- format --
 * Parameters: M x K weights, tiles TM x TK with TM in {64,128,256},
 * TK in {16,32,64,128}, M % TM == 0, K % TK == 0, M*K < 2^32.
 * nTM = M/TM, nTK = K/TK, nT = nTM*nTK; tile t = tm*nTK + tk covers rows
 * [tm*TM, tm*TM+TM) and columns [tk*TK, tk*TK+TK).
 * Scan position p inside a tile:  US_ORDER_ROW  p = i*TK + j
 *                                 US_ORDER_COL  p = j*TM + i
 * bitmap:   uint64[nT * TM*TK/64]; tile t owns words [t*TM*TK/64, ...);
 *           bit (p % 64) of word p/64 is set iff W[tm*TM+i][tk*TK+j] != 0
 *           (fp16: +0 and -0 are zero; NaN is stored).  Earlier position =
 *           less significant bit.
 * tile_off: uint32[nT+1], in ELEMENTS; tile_off[0] = 0,
 *           tile_off[t+1] = tile_off[t] + roundup(P_t, E) where P_t is the
 *           popcount of tile t's words and E = 8 (fp16) or 32 (int4), i.e.
 *           every tile's run is padded with zeros to 16 bytes.
 * values:   the nonzeros of tile t in increasing p, starting at element
 *           tile_off[t] (o_t + rho, rho = set positions scanned before p).
 *           fp16: 2 bytes little-endian.  int4: element e in byte e>>1,
 *           even e in the low nibble, two's complement in [-8, 7].
 *
 * ------------------------------------------------------------ conventions --
 * All pointers are DEVICE pointers unless marked "host".  Every device
 * pointer must be 16-byte aligned.  The caller allocates and owns every
 * buffer; the library never allocates, never synchronises the device (except
 * us_get_last_device_status) and never throws: every entry point returns a
 * us_status.  `stream` is a cudaStream_t (NULL = legacy default stream).
 * Argument errors are detected on the host before anything is enqueued.
 * Kernels guard every access with the offsets they read; a run that does not
 * fit its tile, or a tile_off beyond values_bytes, is not read: the tile is
 * treated as empty and US_ERR_CORRUPT is recorded in the device status word
 * (us_get_last_device_status).
 *
 * Workspace: query its size with us_workspace_bytes / us_encode_sizes.  It
 * must be zero-filled once before its first use; every call leaves it
 * zero-filled again where the next call needs zeros (split-K arrival
 * counters).  One workspace serves one call at a time: two calls in flight
 * at once on different streams must not share it.
 */
#ifndef US_H_
#define US_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    US_OK = 0,
    US_ERR_INVALID_ARG = 1,   /* bad shape, null or misaligned pointer, bad enum */
    US_ERR_UNSUPPORTED = 2,   /* valid format, but no kernel for this combination */
    US_ERR_TOO_LARGE = 3,     /* M*K >= 2^32 or another size limit */
    US_ERR_WORKSPACE = 4,     /* workspace (or values capacity) too small */
    US_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    US_ERR_TIMEOUT = 6,       /* a device-side wait hit its iteration limit */
    US_ERR_CORRUPT = 7        /* inconsistent format detected (host or device) */
} us_status;

/* Element types of the value stream: fp16; int4 (two per byte, even element in
 * the low nibble, two's complement in [-8, 7]); int2 for W2A4 (four per byte,
 * the earlier element in the lower bits, two's complement in [-2, 1]: the
 * pages name W2A4 in UnionSparse Fig. 11 without its layout, so this is the
 * plain reading).  Runs are padded to 16 bytes: 8 / 32 / 64 elements. */
typedef enum { US_F16 = 0, US_I4 = 1, US_I2 = 2 } us_elem;
typedef enum { US_ORDER_ROW = 0, US_ORDER_COL = 1 } us_order;
typedef enum {
    US_OP_ENCODE = 0,
    US_OP_SPMM_W4A4 = 1,
    US_OP_SPMM_F16 = 2,
    US_OP_SPMSPV_F16 = 3
} us_op;

/* A view of an encoded matrix.  Plain data, copied by value into kernel
 * parameters; the caller owns the three arrays.  values_bytes is the
 * readable length of `values` (at least tile_off[nT] * bits / 8).
 * flags: 0, or US_BITMAP_STATIC.  US_BITMAP_STATIC promises that no work
 * enqueued earlier on the same stream writes bitmap, tile_off or values, nor,
 * in us_spmm_w4a4, the row scales s_w (the usual case for inference weights).
 * Kernels then start fetching and decoding them before the preceding kernel
 * has finished (programmatic dependent launch); the activations, their scales
 * and the outputs are still touched only after it has.  Leave it 0 when the
 * matrix may still be in the making, e.g. right after us_encode. */
#define US_BITMAP_STATIC 1u
typedef struct {
    int32_t M, K, TM, TK;
    int32_t elem;             /* us_elem */
    int32_t order;            /* us_order */
    const uint64_t* bitmap;
    const uint32_t* tile_off;
    const void* values;
    uint64_t values_bytes;
    uint32_t flags;
    uint32_t reserved;        /* must be 0 */
} us_bitmap;

/* Sizes of the encoder's outputs and workspace (all host out-params).
 * values_cap_bytes is the worst case (every position nonzero). */
us_status us_encode_sizes(int M, int K, int TM, int TK, us_elem elem,
                          size_t* bitmap_bytes, size_t* tile_off_bytes,
                          size_t* values_cap_bytes, size_t* ws_bytes);

/* Dense -> bitmap tiles on the GPU (UnionSparse V-A, Q = 1; SPDP 4.1 for
 * US_ORDER_COL).  W: M x K row-major with leading dimension ldw (elements):
 * fp16 bit patterns (US_F16) or int8 codes in [-8, 7] (US_I4).  Writes
 * bitmap, tile_off (nT+1 entries; tile_off[nT] is the used length in
 * elements) and values (capacity values_cap bytes).  An int4 code outside
 * [-8, 7] records US_ERR_INVALID_ARG and a run beyond values_cap records
 * US_ERR_WORKSPACE in the device status word (that tile's run is not
 * written).  Output bytes are identical to those of a sequential encoder. */
us_status us_encode(const void* W, int64_t ldw, int M, int K, int TM, int TK,
                    us_elem elem, us_order order, uint64_t* bitmap,
                    uint32_t* tile_off, void* values, size_t values_cap,
                    void* ws, size_t ws_bytes, void* stream);

/* W4A4 SpMM (UnionSparse Fig. 2):  Yacc[n][m] = sum_k Wq[m][k] * Xq[n][k]
 * (exact int32) and, if Y != NULL,
 * Y[n][m] = fp16_rn((fp32(Yacc) * s_w[m]) * s_x[n]).
 * W: elem US_I4, order US_ORDER_ROW.  Xq: N x K int4 codes, token-major,
 * packed like `values` (element n*K + k); requires K % 32 == 0.
 * s_w: M fp16 bit patterns, s_x: N fp16.  Yacc: N x M int32, Y: N x M fp16.
 * 1 <= N <= 2048.  split_k: 0 = automatic, else K tiles are split into that
 * many slices (1..nTK).  Results do not depend on split_k.  With 64 x 64 tiles
 * and 1 <= N <= 32 the automatic choice slices nothing: the tile sequence is
 * spread evenly over the SMs, and a band shared by several CTAs is finished by
 * the CTA holding its first tile from the others' posted {value, tag} words
 * (the workspace, left zeroed after every call). */
us_status us_spmm_w4a4(const us_bitmap* W, const uint8_t* Xq, const uint16_t* s_w,
                       const uint16_t* s_x, int N, int32_t* Yacc, uint16_t* Y,
                       void* ws, size_t ws_bytes, int split_k, void* stream);

/* fp16 SpMM (UnionSparse Fig. 2 with fp16 operands; SPDP section 4 for the
 * prefill shapes):  Y[n][m] = fp16(sum_k W[m][k] * X[n][k]) with fp32
 * accumulation.  W: elem US_F16, order US_ORDER_ROW or US_ORDER_COL (the
 * spMspV layout serves this product too).  X: N x K fp16 token-major,
 * Y: N x M fp16, 1 <= N <= 2048.  split_k as above.  With 64 x 64 tiles,
 * N >= 64 and M % 128 == 0 the product runs on the tensor cores (tcgen05);
 * there K is cut into at most 8 slices (a larger split_k is lowered to 8):
 * the slices of an output tile form one thread-block cluster and reduce in
 * its shared memory, so that path uses no workspace.  1-63 tokens on ROW
 * tiles run on the mma.sync decode kernel; every other case on the generic
 * CUDA-core kernel.  The fp32 partial sums are reduced in fixed slice order,
 * so repeated calls with the same arguments give bitwise identical results;
 * calls that take different kernels may differ in the last bits. */
us_status us_spmm_f16(const us_bitmap* W, const uint16_t* X, int N, uint16_t* Y,
                      void* ws, size_t ws_bytes, int split_k, void* stream);

/* fp16 SpMM with no workspace argument and no allocation.  (No counterpart on
 * the pages: this is a convenience of this library.)  For callers that cannot
 * allocate device memory where they multiply - fixed-arena allocators that
 * hand out no extra buffers, embedders that own every allocation, code paths
 * that must not enter the CUDA allocator - the split-K scratch comes from a
 * device array inside the library, US_NOALLOC_SCRATCH_BYTES (8 MiB), which
 * every GPU that loads the library keeps until the process exits.
 * Same arguments and results as us_spmm_f16 without ws/ws_bytes.  With
 * split_k = 0 the automatic split is lowered to 1 if its scratch would not
 * fit; an explicit split_k whose scratch exceeds the array returns
 * US_ERR_TOO_LARGE before anything is enqueued.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress), so make that
 * first call before any stream capture.  Each call off the tensor-core path
 * clears the split-K counters with cudaMemsetAsync on `stream` (no
 * allocation); the tensor-core path needs no scratch.  All calls share
 * the one array: calls that may run at the same time on the GPU (different
 * streams, overlapping graph branches) race and must not be issued. */
#define US_NOALLOC_SCRATCH_BYTES (8u << 20)
us_status us_spmm_f16_noalloc(const us_bitmap* W, const uint16_t* X, int N, uint16_t* Y,
                              int split_k, void* stream);

/* fp16 spMspV (SPDP section 4.2):  y[m] = fp16(sum over k with |x_k| > tau of
 * W[m][k] * x[k]), fp32 accumulation.  Columns whose activation fails the
 * test are skipped: their bitmap words are read, their values are not.
 * W: elem US_F16, order US_ORDER_COL.  x: K fp16, y: M fp16, tau >= 0. */
us_status us_spmspv_f16(const us_bitmap* W, const uint16_t* x, float tau, uint16_t* y,
                        void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * IE-BME with areas ("UnionSparse: An Index-Efficient Sparsity Framework for
 * Low-Bit Sparse LLM Inference on Edge", section V-A with Q = RA*CA > 1,
 * Fig. 7, and the bitmap-aware row reordering of section V-B).
 *
 * A TM x TK tile is the page's local tile.  Its rows are first permuted by
 * perm (row p of the reordered tile is row perm[t*TM + p] of the original
 * tile; NULL = identity).  The reordered tile is cut into RA row partitions
 * and CA column partitions: area q = a*CA + c holds rows a*LM .. a*LM+LM-1
 * and columns c*LK .. c*LK+LK-1, with LM = TM/RA and LK = TK/CA.
 *
 * One union mask per tile: logical position (i, j), scanned row-major
 * (p = i*LK + j, bit p%64 of word p/64, earlier = less significant), is set
 * iff some area holds a nonzero there.  TM*TK/(64*Q) words per tile,
 * tile-major.
 *
 * Values: each set position emits one value per area, zeros included, at
 * CV[tile_off[t] + q*P_t + rho], rho = set positions before it.  The run of
 * Q*P_t values is zero-padded to 16 bytes:
 * tile_off[t+1] = tile_off[t] + roundup(Q*P_t).
 *
 * Shapes: TM in {16, 64, 128, 256}; TK in {16, 32, 64, 128}; RA, CA in
 * {1, 2, 4}; RA*CA <= 4; (TM/RA)*(TK/CA) a multiple of 128 (whole 16-byte
 * bitmap runs); M % TM == K % TK == 0.  Scan order is ROW.
 * ------------------------------------------------------------------------- */
typedef struct {
    us_bitmap W;              /* W.order = US_ORDER_ROW; W.bitmap holds the union masks */
    int32_t RA, CA;           /* row and column partitions, Q = RA * CA */
    const uint8_t* perm;      /* device, TM bytes per tile (tile-major), or NULL */
} us_bitmap_ie;

/* Buffer sizes of us_encode_ie (bitmap M*K/(8*Q), offsets, worst-case values,
 * workspace). */
us_status us_encode_ie_sizes(int M, int K, int TM, int TK, int RA, int CA, us_elem elem, size_t* bitmap_bytes,
                             size_t* tile_off_bytes, size_t* values_cap_bytes, size_t* ws_bytes);

/* Dense -> IE-BME with areas, on the GPU (same dense input as us_encode, ROW
 * scan).  perm: device, TM bytes per tile or NULL; each tile's entries must be
 * a permutation of 0..TM-1 (an entry >= TM or a repeated row records
 * US_ERR_INVALID_ARG in the device status).  ws: us_encode_ie_sizes' ws_bytes. */
us_status us_encode_ie(const void* W, int64_t ldw, int M, int K, int TM, int TK, int RA, int CA, us_elem elem,
                       const uint8_t* perm, uint64_t* bitmap, uint32_t* tile_off, void* values, size_t values_cap,
                       void* ws, size_t ws_bytes, void* stream);

/* Bitmap-aware row reordering (UnionSparse V-B, Eq. 3-5, Algorithm 1), offline
 * on the host: for every TM x TK tile of the HOST matrix W, the exact minimum
 * of active union-mask positions over all groupings of its rows into groups of
 * RA, canonicalised (rows ascending inside a group, groups lexicographic) and
 * laid out partition-wise.  perm: HOST, TM bytes per tile, tile-major, ready
 * for us_encode_ie.  The search is exponential in TM: TM <= 20
 * (US_ERR_UNSUPPORTED otherwise).  nthreads host threads share the tiles. */
us_status us_reorder_rows(const void* W, int64_t ldw, int M, int K, int TM, int TK, int RA, int CA, us_elem elem,
                          uint8_t* perm, int nthreads);

/* W4A4 SpMM on IE-BME with areas: the results of us_spmm_w4a4 (int32
 * accumulators, optional fp16 epilogue) for the matrix W encodes, outputs in
 * the original row order.  W->W.elem must be US_I4.  Workspace: query
 * us_workspace_bytes_ie, zero it once.  split_k as in us_spmm_w4a4. */
us_status us_spmm_w4a4_ie(const us_bitmap_ie* W, const uint8_t* Xq, const uint16_t* s_w, const uint16_t* s_x, int N,
                          int32_t* Yacc, uint16_t* Y, void* ws, size_t ws_bytes, int split_k, void* stream);
us_status us_workspace_bytes_ie(const us_bitmap_ie* W, int N, int split_k, size_t* bytes);

/* The split_k the automatic rule picks for us_spmm_w4a4_ie on W with N tokens:
 * 0 when the balanced kernel serves the call (16 x 64 local tiles, RA in
 * {1, 2, 4}, CA in {1, 2}, M a multiple of 64, 1..32 tokens: four local tiles
 * along M make one 64 x 64 tile of the even partition that us_spmm_w4a4
 * uses), else the K slices of the generic kernel.  W's pointers are not read
 * beyond the null checks. */
us_status us_pick_split_k_ie(const us_bitmap_ie* W, int N, int* split_k);

/* ColInfo of a COL-order matrix ("Unified Static-Dynamic Pruning for
 * Efficient LLM Inference", section 4.1, Tiled-CBC storage structure): one
 * uint32 per column of every tile, tile-major (colinfo[t * TK + j] for tile t,
 * column j), holding (offset << 16) | nnz: nnz is the number of nonzeros of
 * the column, offset the number of nonzeros of the columns before it in the
 * same tile, i.e. where the column's values start in the tile's value run.
 * Derived from the bitmap alone, for either element type.  colinfo: device,
 * nT * TK * 4 bytes, 16-byte aligned, written in full.  W->order must be
 * US_ORDER_COL (US_ERR_UNSUPPORTED otherwise). */
us_status us_colinfo(const us_bitmap* W, uint32_t* colinfo, void* stream);

/* Batched fp16 spMspV with column metadata (SPDP section 4.2, dynamic pruning
 * per token):  Y[n][m] = fp16(sum over k with |X[n][k]| > tau of
 * W[m][k] * X[n][k]), fp32 accumulation.  A column is fetched only if some
 * token keeps its activation; it is found through colinfo (us_colinfo of the
 * same W), so an inactive column costs 4 bytes of metadata and neither bitmap
 * words nor values.  W: elem US_F16, order US_ORDER_COL.  X: N x K fp16
 * token-major, Y: N x M fp16 token-major, N >= 1, tau >= 0.  ws may be NULL
 * (us_workspace_bytes for US_OP_SPMSPV_F16 gives the size, currently 0).
 * colinfo that disagrees with the bitmap or overruns a tile's run records
 * US_ERR_CORRUPT (us_get_last_device_status); such a column contributes only
 * the values inside its run. */
us_status us_spmspv_f16_ci(const us_bitmap* W, const uint32_t* colinfo, const uint16_t* X, int N, float tau,
                           uint16_t* Y, void* ws, size_t ws_bytes, void* stream);

/* Per-token int4 quantisation of fp16 activations (UnionSparse Fig. 2, the
 * "Quant" step from FP16 X to INT4 X with a per-token scale; the page does not
 * fix the rounding, this is the plain symmetric reading):
 *   s_x[n]   = fp16_rn(max_k |X[n][k]| / 7)   (fp32 division), 1 if that is 0
 *   Xq[n][k] = clamp(rint(X[n][k] / s_x[n]), -8, 7)   (fp32 division, ties to even)
 * X: N x K fp16 token-major.  Xq: N x K int4 packed like us_spmm_w4a4's Xq
 * (element n*K + k in byte (n*K + k) >> 1, even elements in the low nibble).
 * s_x: N fp16.  1 <= N, K % 32 == 0.  NaN does not take part in the maximum and
 * gives code 0.  One pass over X: its output feeds us_spmm_w4a4 directly. */
us_status us_quantize_x(const uint16_t* X, int N, int K, uint8_t* Xq, uint16_t* s_x, void* stream);

/* Workspace bytes for `op` on W with N tokens and the given split_k
 * (0 = the automatic choice).  For US_OP_ENCODE only W->M, K, TM, TK are read. */
us_status us_workspace_bytes(us_op op, const us_bitmap* W, int N, int split_k, size_t* bytes);

/* The split_k the automatic rule picks for (op, W, N) on the current device:
 * the smallest of {1,2,4,8,16} whose grid fills every SM, while each slice
 * keeps at least 4 K tiles (split-K rule of "Realizable N:M Sparse
 * Transformer Inference via Search-Kernel Co-Design", section 4.3); 0 when the
 * automatic choice spreads the tiles evenly instead (see us_spmm_w4a4). */
us_status us_pick_split_k(us_op op, const us_bitmap* W, int N, int* split_k);

/* Host-side check of an encoded matrix.  W's three pointers are HOST
 * pointers here.  Returns US_OK, US_ERR_INVALID_ARG (bad parameters) or
 * US_ERR_CORRUPT (offsets not monotone, a run shorter than its popcount or
 * not padded to 16 bytes, nonzero padding, values_bytes too small). */
us_status us_validate(const us_bitmap* W);

/* Waits for `stream`, then returns and clears the device status word that
 * kernels set on device-side errors (US_ERR_TIMEOUT, US_ERR_CORRUPT,
 * US_ERR_INVALID_ARG, US_ERR_WORKSPACE; US_OK if none). */
us_status us_get_last_device_status(void* stream);

/* Self-test of the device-side timeout path.  (No counterpart on the pages:
 * every wait of every kernel here is bounded, and this entry point shows that
 * a wait that runs out ends the kernel with a status instead of a hang.)
 * Launches one thread that waits, through the same bounded mbarrier wait the
 * kernels use, on a barrier that nothing completes, with no copy or other
 * asynchronous operation in flight.  After limit_ns the wait gives up and
 * records US_ERR_TIMEOUT in the device status word; the kernel then returns
 * and the context stays usable.  limit_ns: 1000 .. 1000000000 (else
 * US_ERR_INVALID_ARG).  elapsed_ns: device, 8-byte aligned, nullable; receives
 * the nanoseconds the wait took before giving up (0 if it completed). */
us_status us_selftest_wait_timeout(uint64_t limit_ns, uint64_t* elapsed_ns, void* stream);

/* Static description of a status code. */
const char* us_status_string(us_status s);

/* Library version, major*10000 + minor*100 + patch. */
int us_version(void);

#ifdef __cplusplus
}
#endif
#endif /* US_H_ */
