/*
 * lw.h -- C ABI of liblw: LLM weights kept losslessly entropy-coded in HBM and
 * decoded on demand inside the batch-1 / small-batch matrix products of token
 * generation, so that HBM moves only coded bytes.
 *
 * Sources (page title, then section / figure / equation):
 *  [LW]  "LazyWeights: Decode-on-Demand Edge LLMs" -- TL;DR and Fig. 1 (codes
 *        decoded on demand so DRAM moves only coded bytes); "2 . Code them"
 *        and Fig. 3(a) (one 11-bit length-limited Huffman table per matrix,
 *        4-bit codes coded in pairs, a 64x256 tile = 32 lanes of two rows,
 *        lanes' 32-bit words interleaved, per-tile lane offsets, scales and
 *        minimums kept as stored); "3 . Decode on demand" and Fig. 3(b)
 *        (11-bit peek compared with per-length limits, plus the length's
 *        offset into a symbol table; no 2048-entry table); the runtime
 *        paragraph after Fig. 3 (software decode fused with GEMV, and the
 *        decode-free fixed-width "twin").
 *  [UW]  "Unweight: Compressing LLM Weights for Faster Inference" --
 *        "Understanding BF16 weight structure" (sign 1 / exponent 8 /
 *        mantissa 7), "The exponent's exploitable redundancy" (Huffman on the
 *        exponent byte over a top-16 palette, sign+mantissa raw, a row of 64
 *        with an out-of-palette exponent stored verbatim), "Four approaches
 *        to using compressed weights" and "How reconstructive matmul works"
 *        (full decode vs. reconstruction in shared memory feeding tensor
 *        cores).
 *  [SDB] "Software-Defined Bandwidth Expansion" -- eq. (1) (dense-equivalent
 *        effective bandwidth), section IV.A (b + 16/G storage cost).
 *
 * Shapes.  W is N x K (rows = outputs, as nn.Linear.weight); y = W x.  Every
 * call requires N % 64 == 0 and K % 256 == 0 (else LW_ERR_SHAPE).  Tile t =
 * (r/64) * (K/256) + (k/256) covers 64 rows x 256 columns.  Lane l of a tile
 * carries rows 2l and 2l+1 (row 2l first), columns ascending.
 *
 * Ownership.  Host bundles (lw_bundle) belong to the library: free them with
 * lw_bundle_free.  Device memory and streams belong to the caller: the
 * library never allocates or frees device memory and never synchronises a
 * stream.  Device calls are asynchronous on `stream` (a cudaStream_t passed
 * as void*; NULL = the legacy default stream) and deterministic: a fixed
 * reduction order, no floating-point atomics.  Kernels are launched with
 * programmatic stream serialisation: a call may be scheduled while the
 * previous library kernel on the stream drains and then reads only the
 * bundle's sections until that kernel has completed (activations, the
 * workspace, outputs and *d_status are touched after it).  So bundle
 * sections must not be written by a kernel that allows early launch of its
 * successor and runs immediately before the call; ordinary kernels and
 * copies (and every library call) are waited for in full.
 *
 * Errors.  Argument, shape and format checks run on the host before any
 * launch and return a status; a failed launch returns LW_ERR_CUDA.  A kernel
 * that finds a corrupt stream never traps and never reads outside its tile:
 * it writes a nonzero LW_DEV_* code into *d_status (first writer wins) and
 * finishes.  The caller zeroes *d_status before the call and reads it after
 * synchronising.  lw_last_error() returns a thread-local text for the last
 * failing host call.
 */
#ifndef LW_H_
#define LW_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LW_OK = 0,
  LW_ERR_INVALID_ARG = 1,
  LW_ERR_SHAPE = 2,
  LW_ERR_UNSUPPORTED = 3,
  LW_ERR_ALLOC = 4,       /* host allocation failed */
  LW_ERR_CORRUPT = 5,     /* malformed bundle or table detected on the host */
  LW_ERR_CUDA = 6,        /* launch or CUDA runtime error */
  LW_ERR_IO = 7           /* a bundle file could not be opened, read or written */
} lw_status;

/* device-side error codes written to *d_status */
enum {
  LW_DEV_OK = 0,
  LW_DEV_LANE_LENGTH = 1,   /* a lane (or its first row) ended at a bit count
                               other than lane_bits (lane_mid) */
  LW_DEV_BAD_CODE = 2,      /* a peek matched no codeword (incomplete table) */
  LW_DEV_TILE_SIZE = 3,     /* a tile is longer than max_tile_rows */
  LW_DEV_TIMEOUT = 4,       /* a bounded wait on an asynchronous copy ran out */
  LW_DEV_BAD_TABLE = 5,     /* the device table fails its in-kernel checks, or
                               its length span exceeds what the launch expects */
  LW_DEV_BAD_STRIPS = 6     /* a strip-list entry is outside the matrix or not
                               above the entry before it (its tiles skipped) */
};

typedef enum {
  LW_FMT_Q4_PAIR = 1,  /* 4-bit codes, coded in pairs (8-bit symbols) [LW] */
  LW_FMT_Q6 = 2,       /* 6-bit codes, one symbol each (Q6_K-like)      [LW] */
  LW_FMT_BF16_EXP = 3  /* BF16: exponent byte coded over a top-16 palette [UW] */
} lw_format;

#define LW_MAX_CODE_LEN 11

/* What to build.  twin = 1 builds the decode-free fixed-width "twin" of the
   same tiles, lanes and interleave [LW]: 4-bit codes at 4 bits, 6-bit codes at
   6 bits, BF16 exponents as a 4-bit palette index ([UW] "direct palette"). */
typedef struct {
  int32_t fmt;    /* lw_format */
  int32_t twin;   /* 0: Huffman-coded, 1: fixed-width twin */
  int64_t rows;   /* N, multiple of 64 */
  int64_t cols;   /* K, multiple of 256 */
} lw_desc;

/*
 * Decoder table, one per matrix (device-ready, 1024 bytes, byte-copyable).
 * Canonical code: lengths come from code_len; codes are assigned shortest
 * first, ties by ascending symbol value (the RFC 1951 section 3.2.2 rule).
 * The comparator rule [LW "3 . Decode on demand"]: for a 32-bit window whose
 * first stream bit is the MSB, L = lmin + #{ j < lmax - lmin :
 * window > lim_m1[j] }, where lim_m1[j] = (limit(lmin+j) << 21) - 1 and
 * limit(L) = (first_code(L) + count(L)) << (11 - L); then the symbol is
 * sym[(window >> (32 - L)) + off[L - lmin]].
 */
typedef struct {
  int32_t fmt;
  int32_t alpha;          /* 256 (Q4 pairs), 64 (Q6), 16 (BF16 palette idx) */
  int32_t n_sym;          /* symbols that have a code */
  int32_t lmin, lmax;     /* shortest and longest code length */
  int32_t n_palette;      /* BF16 only: entries of palette[] in use */
  int32_t phantom;        /* 1 if the table was completed with a phantom code
                             (a lone symbol of length 1) */
  int32_t reserved0;
  uint32_t lim_m1[12];    /* see above; unused entries 0xFFFFFFFF */
  int32_t off[12];        /* base(L) - first_code(L), index L - lmin */
  uint16_t sym[256];      /* symbols in canonical order (+ phantom) */
  uint8_t code_len[256];  /* code length per symbol, 0 = no code */
  uint8_t palette[16];    /* BF16: exponent byte of each palette index,
                             ascending */
  uint8_t reserved1[112];
} lw_table;

/* Opaque host bundle. */
typedef struct lw_bundle lw_bundle;

/* Sections of a bundle, in the order of lw_sections.ptr[] */
enum {
  LW_SEC_WORDS = 0,   /* uint32: coded (or fixed-width) lane words.  Word j of
                         lane l of tile t is words[(tile_off[t] + j)*32 + l]:
                         one aligned 128-byte row holds the next word of every
                         lane [LW Fig. 3(a)].  Codes MSB-first: stream bit p
                         is bit 31 - p%32 of word p/32.  Lanes are zero-padded
                         to the tile's longest lane (W_t words). */
  LW_SEC_TILE_OFF,    /* uint32 [n_tiles + 1]: start of each tile's words in
                         128-byte rows (prefix sum of W_t) -- the per-tile
                         offsets that let any tile start on its own. */
  LW_SEC_LANE_BITS,   /* uint16 [n_tiles][32]: bits in each lane (checked at
                         the end of every lane). */
  LW_SEC_TABLE,       /* lw_table (1024 bytes). */
  LW_SEC_QPARAMS,     /* Q4: per tile, per row of the tile (64), the fp16
                         scale then the fp16 min of the row's 256-weight
                         super-block: [n_tiles][64][2] uint16.
                         Q6: per tile, per 16-byte chunk q (0..3), per lane
                         l: 8 fp16 scales; lane l's 32 scales (row 2l groups
                         0..15, then row 2l+1) are chunks 0..3:
                         [n_tiles][4][32][8] uint16.  BF16: empty. */
  LW_SEC_SIGNMAN,     /* BF16: sign+mantissa bytes, sm = sign<<7 | mantissa,
                         every weight.  Tile-major, 16-byte chunks
                         interleaved over lanes: byte q (0..511) of lane l of
                         tile t is at t*16384 + ((q/16)*32 + l)*16 + q%16;
                         a lane's bytes follow its lane order. */
  LW_SEC_VFLAGS,      /* BF16: uint32 [N][GW], GW = ceil(K/64/32): bit g%32
                         of word g/32 of row r is set iff the 64-column group
                         g of row r is stored verbatim. */
  LW_SEC_VROW_OFF,    /* BF16: uint32 [N + 1]: verbatim groups before row r. */
  LW_SEC_VEXP,        /* BF16: uint8 [n_verbatim][64]: raw exponent bytes of
                         each verbatim group, ordered by row, then group. */
  LW_SEC_LANE_MID,    /* uint16 [n_tiles][32]: bit offset in each lane where
                         its second row (2l+1) starts, so a decoder can run the
                         lane's two rows as independent streams (coded bundles
                         only; an extension of the per-tile lane offsets). */
  LW_NUM_SECTIONS
};

typedef struct {
  const void* ptr[LW_NUM_SECTIONS];   /* host pointers, owned by the bundle */
  uint64_t bytes[LW_NUM_SECTIONS];    /* 0 = section absent */
  uint64_t coded_bytes;     /* all sections a product reads (its HBM bytes,
                               activations and outputs excluded) */
  uint64_t n_tiles;
  int64_t n_verbatim;       /* BF16 verbatim groups */
  int32_t max_tile_rows;    /* max W_t over the tiles */
  int32_t max_len;          /* longest code length (lmax) */
  int32_t min_len;          /* shortest code length (lmin) */
  int32_t palette_size;     /* BF16 */
  double bits_per_weight;   /* 8 * coded_bytes / (N*K) */
  int32_t lut_entries;      /* coded bundles: entries of the compact decode
                               table (index max(peek >> s, peek - C), s and
                               C chosen per table, 128 bytes each in shared
                               memory); 0 for twins */
  int32_t reserved;
} lw_sections;

/*
 * Device view of an uploaded bundle: raw device pointers into caller-owned
 * buffers holding byte-for-byte copies of the host sections (NULL where a
 * section is absent).  Filled by the caller; the library only reads it on the
 * host at call time.  words, lane_bits, table, qparams, signman and lane_mid
 * must be 16-byte aligned (the kernels copy them with the bulk-copy engine);
 * calls refuse other addresses with LW_ERR_INVALID_ARG.
 */
typedef struct {
  int32_t fmt;
  int32_t twin;
  int64_t rows;
  int64_t cols;
  int32_t max_tile_rows;    /* from lw_sections; bounds shared-memory staging */
  int32_t lmin, lmax;       /* from lw_sections: code-length span of the table
                               (selects the kernel variant; checked on device) */
  int32_t lut_entries;      /* from lw_sections: entries of the compact decode
                               table of the table-driven product kernel
                               (4-/6-bit, and BF16 up to 4 activation rows
                               per pass).  1..512 selects that kernel (the device
                               rebuilds the table from the bundle's lw_table
                               and reports LW_DEV_BAD_TABLE if it needs more);
                               0 selects the comparator kernel (any table).
                               Ignored for twins and BF16. */
  const uint32_t* words;
  const uint32_t* tile_off;
  const uint16_t* lane_bits;
  const lw_table* table;
  const void* qparams;
  const uint8_t* signman;
  const uint32_t* vflags;
  const uint32_t* vrow_off;
  const uint8_t* vexp;
  const uint16_t* lane_mid;
} lw_dev_bundle;

/*
 * Build a bundle on the host [LW "2 . Code them"; UW "The exponent's
 * exploitable redundancy"].
 *  payload: Q4 / Q6: uint8 codes [N][K] (values < 16 / < 64);
 *           BF16: uint16 bf16 bit patterns [N][K].
 *  scales:  Q4: fp16 bits [N][K/256]; Q6: fp16 bits [N][K/16]; BF16: NULL.
 *  mins:    Q4: fp16 bits [N][K/256]; otherwise NULL.
 * One length-limited (<= 11 bits) optimal Huffman table per matrix over the
 * symbols actually coded.  On success *out owns copies of everything.
 * Errors: LW_ERR_INVALID_ARG (NULL pointers, code values out of range),
 * LW_ERR_SHAPE, LW_ERR_UNSUPPORTED (fmt), LW_ERR_ALLOC.
 */
lw_status lw_encode_bundle(const lw_desc* desc, const void* payload,
                           const uint16_t* scales, const uint16_t* mins,
                           lw_bundle** out);

/* Section pointers and sizes of a bundle (valid until lw_bundle_free). */
lw_status lw_bundle_sections(const lw_bundle* b, lw_sections* out);

/* Free a bundle and every section it owns (NULL is allowed); pointers
   obtained from lw_bundle_sections become invalid. */
void lw_bundle_free(lw_bundle* b);

/* Format, twin flag and shape of a bundle (e.g. one just loaded). */
lw_status lw_bundle_desc(const lw_bundle* b, lw_desc* out);

/*
 * Bundle files [UW "One Format, Two Purposes"]: the coded bundle is the
 * distribution format -- shipped as a byte string, loaded back, then
 * uploaded (or transcoded to the twin, lw_transcode_twin) at load time.
 * The string: a 192-byte little-endian header ("LWBUNDLE", version 1, fmt,
 * twin, rows, cols, max_tile_rows, section count, n_verbatim, the byte size
 * of every section in lw_sections order), the sections in that order each
 * at a multiple of 64 bytes, then a 64-bit FNV-1a checksum of everything
 * before it.  lw_bundle_serialized_bytes: its length (0 for NULL).
 * lw_bundle_serialize writes it into buf (cap >= that length; the caller
 * owns buf).  lw_bundle_deserialize builds a new bundle (free with
 * lw_bundle_free) after checking the header, the checksum, every section
 * size against the shape and format, and everything lw_validate_sections
 * checks; errors: LW_ERR_CORRUPT (any mismatch), LW_ERR_UNSUPPORTED (another
 * version, a big-endian host), LW_ERR_ALLOC, LW_ERR_INVALID_ARG.
 * lw_bundle_save / lw_bundle_load do the same through a file (LW_ERR_IO when
 * it cannot be opened, read or written).
 */
size_t lw_bundle_serialized_bytes(const lw_bundle* b);
lw_status lw_bundle_serialize(const lw_bundle* b, void* buf, size_t cap);
lw_status lw_bundle_deserialize(const void* buf, size_t bytes, lw_bundle** out);
lw_status lw_bundle_save(const lw_bundle* b, const char* path);
lw_status lw_bundle_load(const char* path, lw_bundle** out);

/*
 * Fill an lw_table from per-symbol code lengths (for bundles built or stored
 * elsewhere).  code_len[alpha]: lengths 0..11.  palette: BF16 exponent bytes
 * (n_palette <= 16, ascending), NULL otherwise.  The code must be complete
 * (Kraft sum exactly 1) unless a single symbol has a code, which gets a
 * phantom partner.  Errors: LW_ERR_CORRUPT (length > 11, over- or
 * under-full code), LW_ERR_INVALID_ARG.
 */
lw_status lw_table_from_lengths(int32_t fmt, const uint8_t* code_len,
                                int32_t alpha, const uint8_t* palette,
                                int32_t n_palette, lw_table* out);

/*
 * Check the host sections of a bundle for consistency (tile offsets
 * non-decreasing and within the word count, lane bit counts within W_t*32,
 * the table equal to the one its code lengths define -- for a twin, its
 * alphabet and, for BF16, an ascending palette of 1..16 entries -- BF16
 * verbatim offsets consistent).  Returns LW_OK or LW_ERR_CORRUPT with the
 * reason in lw_last_error().
 */
lw_status lw_validate_sections(const lw_desc* desc, const lw_sections* s);

/* Bytes of device workspace a product call on this bundle needs for
   `batch` activation rows: the per-strip counters (N/64 uint32, padded to
   256 bytes; zeroed by the caller before first use and left at zero by
   every call that completes), then the split-K partial sums (fp32
   [K/256][8][N]: room for a full CUDA-core pass of 8 rows whatever
   `batch`, or the tensor-core path's K-split partials where that path is
   taken and they are larger).  lw_decode takes no workspace.  0 for a NULL
   view, batch < 1 or a non-positive shape. */
size_t lw_workspace_bytes(const lw_dev_bundle* b, int32_t batch);

/*
 * Decode only: restore the fixed-width weights into `out` (device)
 * [LW "3 . Decode on demand"; UW "Four approaches": full decode].
 *  Q4: packed bytes [N][K/2], low nibble = even column (the pair symbol);
 *  Q6: uint8 [N][K];  BF16: uint16 bf16 bits [N][K].
 * Works on coded bundles and on twins.
 */
lw_status lw_decode(const lw_dev_bundle* b, void* out, int32_t* d_status,
                    void* stream);

/*
 * Fused decode + matrix-vector product, batch 1: y[r] = sum_k W[r][k] x[k]
 * [LW runtime paragraph: software decode fused with GEMV; UW "How
 * reconstructive matmul works"].  x: fp32 [K] (Q4, Q6) or bf16 [K] (BF16);
 * y: fp32 [N].  ws: device workspace of at least lw_workspace_bytes(b, 1).
 * Dequantisation: Q4 w = scale*c + min per 256-weight super-block; Q6 w =
 * scale*(c - 32) per 16 weights; BF16 the value itself.
 * Reduction order (fixed): within a lane and row, two fp32 accumulators
 * (even, odd column) over the tile's columns ascending; Q4 folds the
 * super-block scale and min once per tile row; Q6 folds each 16-weight group
 * into the row sum as it ends; the per-tile partial sums of a row are added
 * in ascending tile order.
 */
lw_status lw_decode_gemv(const lw_dev_bundle* b, const void* x, float* y,
                         void* ws, size_t ws_bytes, int32_t* d_status,
                         void* stream);

/*
 * Fused decode + small-batch product: Y[b][r] = sum_k W[r][k] X[b][k],
 * X [batch][K] row-major (fp32, or bf16 for BF16), Y fp32 [batch][N],
 * batch 1..256.  Passes (each decodes the matrix once):
 *  - 4-/6-bit, up to 5 rows (up to 8 for matrices too small to fill the
 *    device's tensor-core CTAs): CUDA cores, each row in the order of
 *    lw_decode_gemv (bitwise equal to it and to the twin);
 *  - 4-/6-bit, otherwise up to 32 rows: tensor cores -- each weight
 *    dequantised in fp32
 *    and split exactly into a BF16 high part plus a BF16-rounded remainder,
 *    each activation likewise; tcgen05.mma accumulates hi*x_hi + hi*x_lo +
 *    lo*x_hi in FP32 tensor memory (relative error ~2^-16 per product);
 *  - BF16, fewer than 16 rows: CUDA cores, passes of up to 8;
 *  - BF16, 16..64 rows: tensor cores on the rebuilt BF16 weights
 *    (tcgen05.mma, BF16 x BF16 -> FP32 in tensor memory), [UW] "How
 *    reconstructive matmul works".
 * Batches beyond one pass take as many passes as needed (the largest pass
 * first).  On the tensor cores the order within an MMA is the hardware's;
 * a row block's K range may be cut among several CTAs (contiguous tile
 * ranges; the cut follows the device's SM count), whose partial sums are
 * added in ascending order -- deterministic on a given device, but not
 * bitwise equal to the CUDA-core path.  The workspace must hold
 * lw_workspace_bytes(b, batch) bytes.
 */
lw_status lw_decode_gemm(const lw_dev_bundle* b, const void* X, int32_t batch,
                         float* Y, void* ws, size_t ws_bytes,
                         int32_t* d_status, void* stream);

/*
 * The decode-free fixed-width twin [LW: its measured time stands in for the
 * decode unit's]: same product, same order, read from a twin bundle
 * (desc.twin = 1).  Same arguments as lw_decode_gemv.
 */
lw_status lw_twin_gemv(const lw_dev_bundle* twin, const void* x, float* y,
                       void* ws, size_t ws_bytes, int32_t* d_status,
                       void* stream);

/* Twin product for a batch of activation rows (same contract and passes
   as lw_decode_gemm; a BF16 twin of 16..64 rows per pass takes the tensor
   cores with the palette's exponents -- [UW] "Four different execution
   pipelines", direct palette -- and gives bitwise what lw_decode_gemm gives
   on the coded bundle). */
lw_status lw_twin_gemm(const lw_dev_bundle* twin, const void* X, int32_t batch,
                       float* Y, void* ws, size_t ws_bytes, int32_t* d_status,
                       void* stream);

/*
 * Fused decode + GEMV of n (1..LW_MAX_GROUP) independent coded matrices of one
 * 4-/6-bit format in ONE launch: y[i] = W_i x[i] for every i (e.g. a layer's
 * q, k and v projections; the x[i] may alias).  [LW] runtime paragraph after
 * Fig. 3: the decode work of a step fused into as few passes as possible.  A
 * matrix with few tiles leaves most of the GPU idle when launched alone; the
 * group's tiles are decoded by one grid.  Each y[i] is bitwise what
 * lw_decode_gemv(b[i], x[i], y[i], ...) gives.  b, x, y: host arrays of n
 * pointers (bundles, device activations fp32 [K_i], device outputs fp32
 * [N_i]).  ws: one workspace of lw_workspace_bytes_group(b, n) bytes, zeroed
 * before first use (the matrices' counters and partial sums in consecutive
 * 256-byte-aligned slices).  Errors: LW_ERR_INVALID_ARG for n outside
 * 1..LW_MAX_GROUP, NULL pointers, twins, mixed formats; LW_ERR_UNSUPPORTED for
 * BF16 bundles.
 */
#define LW_MAX_GROUP 8
lw_status lw_decode_gemv_group(const lw_dev_bundle* const* b, int32_t n, const void* const* x,
                               float* const* y, void* ws, size_t ws_bytes, int32_t* d_status,
                               void* stream);
size_t lw_workspace_bytes_group(const lw_dev_bundle* const* b, int32_t n);

/*
 * The fixed-width twin of lw_decode_gemv_group: n (1..LW_MAX_GROUP) twin
 * bundles of one 4-/6-bit format in one launch ([LW] runtime paragraph after
 * Fig. 3, the decode-free comparison), each y[i] bitwise what
 * lw_twin_gemv(b[i], x[i], y[i], ...) gives.  Same arguments, workspace
 * (lw_workspace_bytes_group) and errors, with every b[i] a twin (coded
 * bundles are rejected with LW_ERR_INVALID_ARG).
 */
lw_status lw_twin_gemv_group(const lw_dev_bundle* const* b, int32_t n, const void* const* x,
                             float* const* y, void* ws, size_t ws_bytes, int32_t* d_status,
                             void* stream);

/*
 * The grouped launches for small batches: Y[i] = X[i] W_i^T for `batch` = 1..8
 * activation rows (X[i] fp32 [batch][K_i], Y[i] fp32 [batch][N_i]) on the
 * CUDA cores, one launch for the group; each Y[i] is bitwise what
 * lw_decode_gemm / lw_twin_gemm gives for that matrix when its pass stays on
 * the CUDA cores (below 6 rows always; a larger pass on a matrix that fills
 * the device takes the tensor cores in lw_decode_gemm).  Same workspace
 * (lw_workspace_bytes_group) and errors as lw_decode_gemv_group, plus
 * LW_ERR_INVALID_ARG for a batch outside 1..8.
 */
lw_status lw_decode_gemm_group(const lw_dev_bundle* const* b, int32_t n, const void* const* X,
                               int32_t batch, float* const* Y, void* ws, size_t ws_bytes,
                               int32_t* d_status, void* stream);
lw_status lw_twin_gemm_group(const lw_dev_bundle* const* b, int32_t n, const void* const* X,
                             int32_t batch, float* const* Y, void* ws, size_t ws_bytes,
                             int32_t* d_status, void* stream);

/*
 * Tile-skip launch list ["Software-Defined Bandwidth Expansion" §IV.C: an
 * inactive tile is absent from a smaller launch grid, so it moves no
 * weight bytes]: Y = W X for the n_strips 64-row strips listed in `strips`
 * (device int32 array, strictly ascending strip indices in [0, N/64)),
 * every row of every other strip of Y left as it was.  One launch per pass
 * of up to 8 activation rows over the listed strips' tiles only (CUDA
 * cores; 4-/6-bit coded bundles).  The list is read on the device after
 * the previous kernel on `stream` has completed (it may be computed there).
 * Same X, Y and workspace (lw_workspace_bytes(b, batch) suffices) as
 * lw_decode_gemm, and the order of summation of its CUDA-core passes: the
 * listed rows are bitwise what lw_decode_gemm gives on X in slices of up to
 * 8 rows that stay on the CUDA cores (a pass it sends to the tensor cores
 * sums in another order).  n_strips = 0 launches nothing.  A bad entry is
 * reported as LW_DEV_BAD_STRIPS and its tiles are skipped.  Errors:
 * LW_ERR_INVALID_ARG (NULL list with n_strips > 0, n_strips > N/64,
 * alignment, workspace size), LW_ERR_UNSUPPORTED (BF16, twins).
 */
lw_status lw_decode_gemm_strips(const lw_dev_bundle* b, const int32_t* strips, int32_t n_strips,
                                const void* X, int32_t batch, float* Y, void* ws, size_t ws_bytes,
                                int32_t* d_status, void* stream);

/*
 * Load-time transcode [UW "Four approaches to using compressed weights" (the
 * palette pipelines), "One Format, Two Purposes"]: decode a coded bundle on
 * the device into its fixed-width twin ([LW] runtime paragraph after Fig. 3),
 * bit-exact with lw_encode_bundle(twin = 1) of the same weights.  Writes the
 * twin's words, tile offsets and lane bit counts; every other twin section
 * (table, qparams; BF16 signman, vflags, vrow_off, vexp) equals the coded
 * bundle's and may point at the same device buffers.  `twin`: a view with
 * twin = 1, the coded bundle's fmt, rows and cols, max_tile_rows =
 * lw_twin_tile_rows(fmt), and caller-owned device buffers words
 * (n_tiles * max_tile_rows * 128 bytes, 16-byte aligned, not overlapping the
 * coded bundle), tile_off ((n_tiles + 1) uint32) and lane_bits
 * (n_tiles * 32 uint16).  Runs in plain stream order and is followed by an
 * empty plain-order kernel, so the next call on `stream` (whose kernels read
 * bundle sections before waiting on their predecessor) sees the complete
 * twin.  Device status as lw_decode (a corrupt stream is reported, the
 * twin is then undefined).  Errors: LW_ERR_INVALID_ARG (views, shapes,
 * alignment, overlap), LW_ERR_UNSUPPORTED, LW_ERR_CUDA.
 */
lw_status lw_transcode_twin(const lw_dev_bundle* coded, const lw_dev_bundle* twin,
                            int32_t* d_status, void* stream);
/* 128-byte word rows per tile of a format's twin: 64 (4-bit codes, BF16
   palette index), 96 (6-bit codes); 0 for an unknown format. */
int32_t lw_twin_tile_rows(int32_t fmt);

/*
 * lw_decode_gemv without a caller workspace, for callers that cannot allocate
 * device memory: code running under CUDA-graph capture, engines whose pool
 * allocator owns all device memory, latency-critical paths that cannot afford
 * cudaMalloc's implicit synchronisation, foreign-language callers without a
 * device allocator.  The pages have no counterpart; this is an interface
 * convenience.  Same product, order and arguments as lw_decode_gemv minus
 * `ws`/`ws_bytes`.  Scratch comes from a fixed array in device memory of
 * lw_noalloc_scratch_bytes() bytes (16 MiB), held on every GPU that loads
 * the library until the process exits; a matrix whose
 * lw_workspace_bytes(b, 1) exceeds it is rejected with LW_ERR_UNSUPPORTED
 * (that figure counts partial sums for a pass of 8 activation rows,
 * (K/256)*8*N*4 bytes, of which a batch-1 call writes an eighth: both
 * entry points accept the same matrices).  Outside stream capture every
 * call looks up the array's device address; under capture the address the
 * last call outside capture found on the device is used, so make one call
 * on the device before capturing.  After its argument checks every call
 * clears the array's counters on `stream` (they protect against an earlier
 * call that ended early, e.g. a refused or aborted launch); then it runs
 * lw_decode_gemv.  All calls share the array: calls that overlap on the GPU
 * race and must be serialised by the caller.  Allocates nothing.
 */
lw_status lw_decode_gemv_noalloc(const lw_dev_bundle* b, const void* x, float* y,
                                 int32_t* d_status, void* stream);
size_t lw_noalloc_scratch_bytes(void);

/*
 * Testing hook for the bounded waits (not for production use): the next
 * launch of the table-driven 4-/6-bit product kernel in this process (the
 * CUDA-core path of lw_decode_gemv, lw_decode_gemm, lw_twin_gemv,
 * lw_twin_gemm and their group and strip forms, whichever runs first)
 * arms the first stage of its first CTA for copies it never issues, and
 * limits every wait of that launch to `wait_us` microseconds instead of
 * about a second.  The consumer of that stage gives up, writes
 * LW_DEV_TIMEOUT into *d_status, and the launch finishes with no copy in
 * flight; its outputs are void, and every workspace counter still ends at
 * zero, so the workspace serves the next call.  One launch only; a later
 * request replaces a pending one, and wait_us = 0 withdraws it.  Errors:
 * LW_ERR_INVALID_ARG (wait_us outside 0..1000000).
 */
lw_status lw_test_stall_next(int32_t wait_us);

/* Entries of the compact decode table that the table-driven product
   kernel builds from this decoder table (the value lw_sections and
   lw_dev_bundle carry as lut_entries); 0 for a NULL table.  Host only; for
   tables built by lw_table_from_lengths. */
int32_t lw_table_lut_entries(const lw_table* t);

/* The status's name ("LW_OK", "LW_ERR_SHAPE", ...; "unknown lw_status" for
   other values): a static string, never NULL, not to be freed. */
const char* lw_status_string(lw_status s);
/* The calling thread's text for its last failing host call (the reason a
   status was returned; calls that succeed may leave it unchanged).  Owned
   by the library, valid until the thread's next library call. */
const char* lw_last_error(void);

/*
 * Step graphs: the library calls of a decode step captured once on a
 * stream and replayed as one CUDA graph ([LW] runtime: each pass captured in
 * CUDA graphs; the programmatic launch dependencies between the library's
 * kernels become graph edges).  lw_graph_begin starts a thread-local capture
 * on `stream` (a created stream; the default stream cannot be captured);
 * every library call on that stream until lw_graph_end is recorded, not run;
 * lw_graph_end ends the capture and instantiates the graph (*out, owned by
 * the caller, freed with lw_graph_free).  lw_graph_launch replays it on
 * `stream` (asynchronous, like the calls it holds).  The buffers the calls
 * named must stay allocated while the graph is used.  Errors:
 * LW_ERR_INVALID_ARG, LW_ERR_CUDA (capture or launch refused, with the
 * runtime's reason), LW_ERR_ALLOC.
 */
typedef struct lw_graph lw_graph;
lw_status lw_graph_begin(void* stream);
lw_status lw_graph_end(void* stream, lw_graph** out);
lw_status lw_graph_launch(const lw_graph* g, void* stream);
void lw_graph_free(lw_graph* g);

/* ABI revision of this header: 4 (3 + lw_sections.lut_entries and
   lw_dev_bundle.lut_entries, which selects the table-driven product
   kernel; 3 added grouped launches, strip lists, the load-time
   transcode, bundle files, step graphs, LW_ERR_IO, LW_DEV_BAD_STRIPS).  The
   bundle file format carries its own version. */
int32_t lw_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LW_H_ */
