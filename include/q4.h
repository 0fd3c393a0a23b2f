/*
 * q4.h -- C ABI of the GGUF Q4_0 weight-only-quantized linear layer on NVIDIA
 * B300 (sm_103a).  Library: bit_weight_quantized_03_b300/libq4.so.
 *
 * What it computes.  The GeekNews write-up of the Rust/Burn port of Voxtral
 * Mini 4B Realtime (es.news.hada.io/topic?id=26595) describes a quantized
 * inference path whose weights are GGUF Q4_0, multiplied by custom GPU shaders
 * (section "Arquitectura"), and an embedding table kept as Q4 rows that are
 * looked up per token (section "Soluciones técnicas").  The model shapes come
 * from the same section: a 26-layer decoder with hidden size 3072 and GQA
 * 32Q/8KV, and a 32-layer, 1280-wide causal audio encoder.  The calls below are
 * that layer's operations: quantize, decode, the batch-1 decode product, the
 * prefill/encoder product and the embedding-row gather.
 *
 * Block format (GGUF Q4_0; the pages name it but do not print it):
 *   32 weights in 18 bytes.  Bytes [0,2): scale d, IEEE binary16, little-endian.
 *   Bytes [2,18): qs[16]; weight j (0..15) is the low nibble of qs[j], weight
 *   j+16 the high nibble.  Decoded weight: w = (q - 8) * d, one exact fp32
 *   multiply (so code 8 with a negative d decodes to -0.0).
 *   A matrix W with n outputs and reduction length k (k % 32 == 0) is n rows of
 *   k/32 blocks, rows contiguous: row stride 18*k/32 bytes, "row-major blocks".
 *
 * Conventions shared by every call.
 *   - Pointers are DEVICE pointers owned by the caller, unless a call says
 *     otherwise.  Scratch space is passed in as `workspace`; the one
 *     exception is q4_gemv_noalloc, whose scratch is a fixed array of
 *     Q4_GEMV_NOALLOC_SCRATCH_BYTES that the library holds in device memory
 *     of every GPU that loads it.  The library allocates nothing else.
 *   - Every call is asynchronous on stream `s` (NULL = the legacy default
 *     stream) and never synchronizes the host.
 *   - Errors the host can see (null pointer, bad size, k % 32 != 0, broken
 *     alignment, too little workspace) return at once and launch nothing.
 *   - Errors found on the device are written to the caller's int32 status word
 *     `status_dev` (device memory, may be NULL): the first error wins (an
 *     atomic compare-and-swap from Q4_OK), so the caller clears it to 0 before
 *     the call and reads it after synchronizing.
 *   - Launch or runtime failures return Q4_ERR_CUDA.
 *   - Leading dimensions are in elements.
 *   - Flag Q4_FLAG_PDL lets the kernel be launched as a programmatic dependent
 *     launch: it may start while the previous kernel on the stream is still
 *     running and read W early; everything else it reads or writes waits for
 *     that kernel.  Only set it when the previous kernel does not write W.
 *   - Workspaces (q4_gemv, q4_gemm, q4_linear) hold split-K partial sums and
 *     arrival counters.  Zero-fill a workspace once before its first use; every
 *     call that ends without a device error leaves it zero-filled again.  Calls
 *     that may run concurrently need separate workspaces.
 *   - Flag Q4_FLAG_TEST_STALL is for tests only: one bounded wait inside the
 *     kernel is made to run out, so the call reports Q4_ERR_TIMEOUT in
 *     status_dev after about a second, part of y is left unwritten, and the
 *     workspace must be zero-filled again.
 */
#ifndef Q4_H
#define Q4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* q4_stream_t; /* the same type as cudaStream_t */

typedef enum q4_status {
  Q4_OK = 0,
  Q4_ERR_INVALID_ARG = 1,       /* null pointer, size <= 0, bad leading dimension or dtype */
  Q4_ERR_MISALIGNED = 2,        /* a pointer or leading dimension breaks the call's alignment rule */
  Q4_ERR_UNSUPPORTED_SHAPE = 3, /* k % 32 != 0, or a size beyond the call's stated limit */
  Q4_ERR_NONFINITE = 4,         /* device: NaN/Inf input or a binary16 scale overflow in quantize */
  Q4_ERR_ID_OUT_OF_RANGE = 5,   /* device: a gather id outside [0, vocab) */
  Q4_ERR_TIMEOUT = 6,           /* device: a bounded wait inside a kernel ran out */
  Q4_ERR_CUDA = 7,              /* a CUDA runtime call or kernel launch failed */
  Q4_ERR_WORKSPACE = 8          /* workspace missing or smaller than the *_workspace_bytes() figure */
} q4_status;

typedef enum q4_dtype { Q4_F32 = 0, Q4_BF16 = 1 } q4_dtype;

#define Q4_BLOCK_ELEMS 32
#define Q4_BLOCK_BYTES 18
#define Q4_FLAG_PDL 1u
#define Q4_FLAG_TEST_STALL (1u << 30)
#define Q4_GEMV_MAX_M 16 /* largest batch the fp32 GEMV takes */

/* Quantize fp32 weights to Q4_0 blocks.
 * The pages give no quantizer ("Arquitectura" names only the GGUF Q4_0
 * format); the rule implemented is: m = first element of largest |x| in the
 * block; d = binary16(m / -8), round to nearest even (+0 when m = +-0);
 * dd = float(d); code q = clamp(floor(x/dd + 8.5), 0, 15), every code 8 when
 * dd == 0; byte j = q[j] | q[j+16] << 4.  Division and add are IEEE fp32.
 *   w          [n][k] fp32, row-major contiguous, 16-byte aligned.
 *   blocks     output, n*k/32*18 bytes, 16-byte aligned.
 *   status_dev a block holding NaN/Inf, or whose d rounds to Inf, is written as
 *              d = +0 with all codes 8 and sets Q4_ERR_NONFINITE.
 * n >= 1, k >= 32, k % 32 == 0. */
q4_status q4_quantize(const float* w, int64_t n, int64_t k, void* blocks,
                      int32_t* status_dev, q4_stream_t s);

/* Decode rows [row0, row0 + n_rows) of a Q4_0 matrix to fp32 (bit-exact
 * (q - 8) * d) or bf16 (that fp32 value rounded to nearest even).
 *   blocks  the matrix base (row 0), 16-byte aligned.
 *   out     [n_rows][k] contiguous, 16-byte aligned. */
q4_status q4_dequant_rows(const void* blocks, int64_t row0, int64_t n_rows, int64_t k, void* out,
                          q4_dtype out_dtype, q4_stream_t s);

/* Batch-1 (and small-batch) decode product, fp32 in and out:
 *   y[i][r] = sum_j w^[r][j] * x[i][j]   for r < n, i < m
 * with w^ the decoded weights, accumulated in fp32 (per-element error within
 * 1e-4 * sum_j |w^[r][j] x[i][j]|).  The decoder's linears (hidden 3072, GQA
 * 32Q/8KV, "Arquitectura") run through this at one token per step.
 *   W   [n rows of k/32 blocks], 16-byte aligned.
 *   x   [m][ldx] fp32, 16-byte aligned, ldx >= k, ldx % 4 == 0.
 *   y   [m][ldy] fp32, 4-byte aligned, ldy >= n; must not overlap x or W.
 *   1 <= m <= Q4_GEMV_MAX_M.  The workspace holds split-K partial sums:
 *   pass at least q4_gemv_workspace_bytes(n, k, m) bytes, 16-byte aligned
 *   (NULL is fine when that figure is 0).  Results do not depend on timing:
 *   the partial sums are added in a fixed order.
 *   With k % 256 == 0 the call makes one launch per group of up to 4 rows of
 *   x (each weight tile is decoded once for the rows of its launch), so the
 *   weights are streamed ceil(m / 4) times; from m = 5 on the tensor-core
 *   q4_gemm is the faster path (q4_linear_crossover_m).
 *   status_dev (may be NULL) receives Q4_ERR_TIMEOUT if a bounded wait ran out. */
q4_status q4_gemv(const void* W, int64_t n, int64_t k, const float* x, int64_t m, int64_t ldx,
                  float* y, int64_t ldy, void* workspace, size_t ws_bytes, int32_t* status_dev,
                  uint32_t flags, q4_stream_t s);
size_t q4_gemv_workspace_bytes(int64_t n, int64_t k, int64_t m);

/* q4_gemv that also prefetches a region of device memory into L2 while it
 * runs: in a decode step, the weights of the next product.  Each product of
 * the step waits on the one before it (programmatic dependent launch), and
 * the part of a product's weights that its early ring fill does not cover
 * would otherwise stream from HBM only after that wait; prefetched, it comes
 * from L2 while HBM works through the hand-offs.  The arithmetic and the
 * result are exactly q4_gemv's.  The pages do not describe this; it is
 * scheduling only.
 *   prefetch        the region (16-byte aligned), read-only, never written by
 *                   the call; NULL with prefetch_bytes == 0 is plain q4_gemv.
 *   prefetch_bytes  a multiple of 16 (a Q4 matrix with k % 256 == 0 is).
 * Taken by the batch-1 path (m == 1, k % 256 == 0); ignored otherwise.  The
 * region should not be written by the kernel before this one on the stream
 * when Q4_FLAG_PDL is set (it is read as W is: early).  Other arguments,
 * errors and the workspace as for q4_gemv. */
q4_status q4_gemv_prefetch(const void* W, int64_t n, int64_t k, const float* x, int64_t m,
                           int64_t ldx, float* y, int64_t ldy, void* workspace, size_t ws_bytes,
                           int32_t* status_dev, uint32_t flags, const void* prefetch,
                           size_t prefetch_bytes, q4_stream_t s);

/* q4_gemv for callers that cannot allocate device memory (a host that embeds
 * the library in a fixed memory pool where cudaMalloc is forbidden, a
 * real-time loop that must not allocate once streaming has started, a plugin
 * that is handed only its input and output buffers).  The pages have no
 * counterpart: it is a packaging choice of this library.
 * Same arguments, result and error behaviour as q4_gemv, minus the workspace:
 * the split-K scratch is one array of Q4_GEMV_NOALLOC_SCRATCH_BYTES inside the
 * library, in device memory of every GPU that loads it, held until exit.  A
 * call whose q4_gemv_workspace_bytes(n, k, m) exceeds that size returns
 * Q4_ERR_UNSUPPORTED_SHAPE and launches nothing (on a 148-SM B300 every
 * m <= 8 with n <= 2^20 fits).  The call allocates nothing; it clears the
 * part of the array it uses on stream `s` (cudaMemsetAsync) and then runs
 * the q4_gemv kernels.  The first call on each device looks up the array's
 * device address with that device current: make it before any stream
 * capture.  All calls share the array, so calls that may overlap on the GPU
 * (other streams, other host threads) race and give wrong results; serialise
 * them on one stream.  The address is cached per CUDA context, so the first
 * call in a new context (after cudaDeviceReset, say) looks it up again and
 * must also come before any capture. */
#define Q4_GEMV_NOALLOC_SCRATCH_BYTES 4194304 /* 4 MiB */
q4_status q4_gemv_noalloc(const void* W, int64_t n, int64_t k, const float* x, int64_t m,
                          int64_t ldx, float* y, int64_t ldy, int32_t* status_dev,
                          uint32_t flags, q4_stream_t s);

/* One link of a chain of batch-1 products (q4_gemv_chain). */
typedef struct q4_gemv_stage {
  const void* W;  /* [n rows of k/32 blocks], 16-byte aligned */
  int64_t n;      /* rows; n % 4 == 0 */
  int64_t k;      /* k % 256 == 0, k <= the kernel's shared-memory limit (15872) */
  const float* x; /* [k] fp32, 16-byte aligned; may point into the previous link's y */
  float* y;       /* [n] fp32, 4-byte aligned */
} q4_gemv_stage;

#define Q4_CHAIN_MAX_STAGES 128

/* A decode step's chain of dependent batch-1 products in one launch:
 *   for s = 0 .. n_stages-1 in order:  y_s[r] = sum_j w^_s[r][j] * x_s[j]
 * with the results of running the links one after another: x_s may be (a
 * slice of) any earlier y_t, and buffers may be reused by later links.  The
 * decoder of the Voxtral Mini 4B Realtime port ("Arquitectura": 26 layers,
 * hidden 3072, GQA 32Q/8KV) runs its per-token linears as such a chain, each
 * reading the previous one's output.  Each y_s is within 1e-4 * sum_j |w^ x|
 * of the exact product of the x_s it read, with a fixed summation order.
 *   stages     host array of n_stages links (1 <= n_stages <= 128); read during
 *              the call only.  An x_s that overlaps y_{s-1} must lie inside it
 *              and start on a multiple of 4 floats (else Q4_ERR_INVALID_ARG).
 *   workspace  q4_gemv_chain_workspace_bytes() bytes, 256-byte aligned, zero
 *              before the first call; every call that ends without a device
 *              error leaves its counter at zero again.
 * The launch is cooperative (one CTA per SM, all resident); it fails with
 * Q4_ERR_CUDA if the GPU cannot hold every CTA at once.  A row count so
 * large that a link would give one SM more than 8 x 32-row groups returns
 * Q4_ERR_UNSUPPORTED_SHAPE. */
q4_status q4_gemv_chain(const q4_gemv_stage* stages, int32_t n_stages, void* workspace,
                        size_t ws_bytes, int32_t* status_dev, uint32_t flags, q4_stream_t s);
size_t q4_gemv_chain_workspace_bytes(const q4_gemv_stage* stages, int32_t n_stages);

/* Prefill / audio-encoder product on the tensor cores:
 *   Y[i][r] = sum_j bf16(w^[r][j]) * X[i][j]   (fp32 accumulation)
 * for the 32-layer, 1280-wide encoder and prefill ("Arquitectura"); error within
 * 8e-3 * sum_j |w^[r][j] X[i][j]|.
 *   W  as for q4_gemv; k % 256 == 0.
 *   X  [m][ldx] bf16, 16-byte aligned, ldx % 8 == 0, ldx >= k.
 *   Y  [m][ldy] fp32 or bf16, aligned to its element size.
 *   m >= 1.  workspace as for q4_gemv with q4_gemm_workspace_bytes(). */
q4_status q4_gemm(const void* W, int64_t n, int64_t k, const void* X, int64_t m, int64_t ldx,
                  void* Y, q4_dtype y_dtype, int64_t ldy, void* workspace, size_t ws_bytes,
                  int32_t* status_dev, uint32_t flags, q4_stream_t s);
size_t q4_gemm_workspace_bytes(int64_t n, int64_t k, int64_t m);

/* Q4 embedding-row gather ("Soluciones técnicas": the 1.5 GiB table is kept as
 * Q4 rows and rows are looked up per token; here the lookup runs on the GPU):
 *   out[b][:] = decode(table row ids[b])  (fp32, bit-exact)
 *   table  [vocab rows of k/32 blocks], 16-byte aligned.
 *   ids    [n_ids] int32 (device).  An id outside [0, vocab) gives a row of
 *          +0.0 and sets Q4_ERR_ID_OUT_OF_RANGE in status_dev.
 *   out    [n_ids][k] fp32, 16-byte aligned. */
q4_status q4_embed_gather(const void* table, int64_t vocab, int64_t k, const int32_t* ids,
                          int64_t n_ids, float* out, int32_t* status_dev, q4_stream_t s);

/* Batch-1 product on the integer path: y = W x with x quantized per 32
 * elements to int8 (GGUF Q4_0's usual companion; the pages, "Arquitectura",
 * name only the weight format, so the reading is this library's): per block
 * amax = max |x_j|, d_x = amax / 127 (fp32, IEEE division), q_x = x / d_x
 * rounded to nearest with halves away from zero (IEEE division); amax == 0
 * gives d_x = +0 and codes 0, a NaN or infinity in the block gives d_x = NaN
 * (so every output is NaN).  Each block adds d_w * d_x * sum (q_w - 8) q_x
 * with the integer sum exact; y is within 1e-4 * sum_b |block term| of the fp64
 * value of that sum, and within sum_j |w^_j| d_x,b(j) / 2 more of the product
 * with the unquantized x.
 *   W  GGUF Q4_0 [n rows of k/32 blocks], 16-byte aligned; k % 32 == 0,
 *      k <= 12288 (else Q4_ERR_UNSUPPORTED_SHAPE).
 *   x  fp32 [k], 4-byte aligned;  y  fp32 [n], 4-byte aligned.
 * No workspace; results do not depend on timing. */
q4_status q4_gemv_q8(const void* W, int64_t n, int64_t k, const float* x, float* y,
                     q4_stream_t s);

/* ---------------------------------------------------------------------------
 * Repacked layout and the decode-step chain.
 *
 * q4_repack copies a GGUF Q4_0 matrix into this library's GPU layout (the pages
 * name only the GGUF format, "Arquitectura"; the layout below is a packaging
 * choice, every block's bytes are kept): rows in groups of 16, k in slices of
 * 256 (8 blocks); tile (G, t) = rows 16G..16G+15 x blocks 8t..8t+7 is 2304
 * bytes at (G * k/256 + t) * 2304.  Inside it, for g = 0..7 and hr = 0 (row
 * 16G + g) or 1 (row 16G + g + 8):
 *   scales: the binary16 d of block 8t + b of that row at byte 32g + 4b + 2hr;
 *   codes: column c = 16s + i of the tile (step s = 0..15) belongs to lane
 *   L = 4g + (i % 8) / 2 of step s, whose little-endian 32-bit word at
 *   256 + 512 (s / 4) + 16L + 4 (s % 4) holds the code in its nibble
 *   m = hr + 2 (i / 8) + 4 (i % 2) (bits 4m..4m+3).
 * That is the operand order of a 16 x 16 row-major tensor-core A fragment:
 * one word per lane and step, four steps per 16-byte load.
 * Rows past n in the last group are d = +0 with every code 8.  Each tile is
 * one contiguous 16-byte-aligned run.
 *   W  GGUF Q4_0 [n rows of k/32 blocks], 16-byte aligned; k % 256 == 0.
 *   R  output, q4_repack_bytes(n, k) bytes, 16-byte aligned, must not overlap W.
 * q4_repack_bytes returns 0 for a shape it does not take. */
size_t q4_repack_bytes(int64_t n, int64_t k);
q4_status q4_repack(const void* W, int64_t n, int64_t k, void* R, q4_stream_t s);

/* Where a chain link reads a vector: the output of an earlier link of the same
 * chain (link >= 0; elements [offset, offset + len) of that output), or fp32
 * device memory (link < 0; ptr 16-byte aligned, read when the link starts).
 * offset is a multiple of 4 elements. */
typedef struct q4_chain_src {
  const float* ptr;
  int32_t link;
  int32_t offset;
} q4_chain_src;

/* Q4_OP_SWIGLU: the gated FFN unit in the epilogue of the w1/w3 product.  The
 * link's n rows (n % 16 == 0) come in 16-row groups of 8 gate rows followed by
 * the 8 matching up rows (w1 and w3 interleaved 8 rows at a time), and its
 * output has n/2 elements: out[8g + j] = a * sigmoid(a) * b with a = row
 * 16g + j and b = row 16g + 8 + j (j < 8).  Not combined with the others. */
#define Q4_OP_SWIGLU 1u
#define Q4_OP_RESIDUAL 2u /* y = W x + residual */
#define Q4_OP_ARGMAX 4u   /* argmax[0] = index of the largest y, argmax[1] = its bits */

/* One batch-1 product of a chain: y = W x (+ residual), fp32. */
typedef struct q4_chain_link {
  const void* R;           /* q4_repack layout, n rows, k columns, k % 256 == 0, k <= 12288 */
  int64_t n, k;
  q4_chain_src x;          /* k elements */
  q4_chain_src residual;   /* Q4_OP_RESIDUAL: n elements (from memory: n % 4 == 0) */
  float* y;                /* output (n fp32, n/2 with Q4_OP_SWIGLU), 4-byte aligned, or NULL */
  int32_t* argmax;         /* Q4_OP_ARGMAX: [2] int32, 4-byte aligned */
  uint32_t ops;            /* Q4_OP_* */
  uint32_t reserved;
} q4_chain_link;

#define Q4_CHAIN_MAX_LINKS 128

/* A decode step's chain of dependent batch-1 products in one launch.  The
 * decoder of the Voxtral Mini 4B Realtime port ("Arquitectura": 26 layers,
 * hidden 3072, GQA 32Q/8KV) runs per token qkv, wo, the gated FFN pair and w2
 * per layer, each reading an earlier product's output, and its output head,
 * whose largest logit is the next token.  Links run as if one after another:
 *   p_s[r] = sum_j w^_s[r][j] x_s[j],  x_s = src(x)
 *   y_s = p_s (+ src(residual)), or the gated pairs of p_s with Q4_OP_SWIGLU
 * Each p_s is within 1e-4 * (sum_j |w^ x_s| + |residual|) of the exact value
 * for the x_s it read, x_s finite.  The products run on the tensor cores:
 * each 256-element slice of x_s is scaled by a power of two that puts its
 * largest magnitude in [2^14, 2^15) and carried as a binary16 pair hi + lo
 * (relative error below 2^-22), so an element more than ~2^38 below its
 * slice's largest magnitude, or in a slice whose largest magnitude is below
 * 2^-112, may count as zero; a non-finite element of x_s makes outputs
 * non-finite.  Sums over split work are added in a fixed order, so
 * results do not depend on timing, and a y_s written to memory is bitwise the
 * value later links read.  Q4_OP_ARGMAX writes the index of the largest y
 * (lowest index among equal values; NaN never wins; -1 if every y is NaN) and
 * its value, whether or not y itself is written.  Sigmoid: fp32 exp.
 *   links      host array of n_links (1..Q4_CHAIN_MAX_LINKS), read during the
 *              call only.
 *   workspace  q4_chain_workspace_bytes() bytes, 256-byte aligned, zero-filled
 *              before its first use and after any call that reported a device
 *              error; otherwise passed unchanged from call to call (it carries
 *              a launch counter and the hand-off slots).  Calls that may run
 *              concurrently need separate workspaces; a chain of a new shape
 *              is fine on a used workspace (its first call is a little slower).
 * The launch is cooperative (one CTA per SM, all resident): Q4_ERR_CUDA if the
 * GPU cannot hold them.  A shape whose per-SM bookkeeping would not fit the
 * kernel's shared memory returns Q4_ERR_UNSUPPORTED_SHAPE (at k = 3072, n up
 * to about 260 thousand rows fits, the 131072-row output head included; with
 * a residual, about 150 thousand). */
size_t q4_chain_workspace_bytes(const q4_chain_link* links, int32_t n_links);
q4_status q4_chain(const q4_chain_link* links, int32_t n_links, void* workspace, size_t ws_bytes,
                   int32_t* status_dev, uint32_t flags, q4_stream_t s);

/* Batch-1 product y = W x on a repacked matrix (a one-link q4_chain): the
 * per-token product of the decoder linears and the output head
 * ("Arquitectura").  Same error bound, workspace rules and x alignment as
 * q4_chain; y [n] fp32, 4-byte aligned.  A one-link chain is an ordinary
 * launch (each CTA takes whole 16-row groups); with Q4_FLAG_PDL it is a
 * programmatic dependent launch in a half-size CTA shape, so that two calls'
 * CTAs share an SM and a call fills its weight ring while the previous kernel
 * ends (x is read after that kernel). */
size_t q4_gemv_r_workspace_bytes(int64_t n, int64_t k);
q4_status q4_gemv_r(const void* R, int64_t n, int64_t k, const float* x, float* y,
                    void* workspace, size_t ws_bytes, int32_t* status_dev, uint32_t flags,
                    q4_stream_t s);

/* Linear layer with the batch-size crossover: m <= q4_linear_crossover_m(n, k)
 * and fp32 X run q4_gemv; otherwise q4_gemm (fp32 X is first rounded to bf16
 * into the workspace).  Y is fp32 [m][ldy].  X dtype Q4_F32 needs ldx % 4 == 0,
 * Q4_BF16 needs ldx % 8 == 0.  workspace >= q4_linear_workspace_bytes(). */
q4_status q4_linear(const void* W, int64_t n, int64_t k, const void* X, q4_dtype x_dtype, int64_t m,
                    int64_t ldx, float* Y, int64_t ldy, void* workspace, size_t ws_bytes,
                    int32_t* status_dev, uint32_t flags, q4_stream_t s);
size_t q4_linear_workspace_bytes(int64_t n, int64_t k, int64_t m, q4_dtype x_dtype);
/* The largest m that q4_linear sends to the fp32 GEMV: a table measured on
 * B300 for the decoder shapes (4096x3072, 1024x3072, 3072x4096, 9216x3072,
 * 3072x9216) and the encoder shapes (3840x1280, 1280x1280, 5120x1280,
 * 1280x5120); another shape takes the entry nearest to it in weight count;
 * k % 256 != 0 (no tensor-core path) gives Q4_GEMV_MAX_M. */
int64_t q4_linear_crossover_m(int64_t n, int64_t k);

/* Static strings; never NULL. */
const char* q4_status_string(q4_status st);
const char* q4_version(void);

#ifdef __cplusplus
}
#endif
#endif /* Q4_H */
