/*
 * w12.h — C ABI of the W12 library for one NVIDIA GB300 (sm_103a).
 *
 * W12 is the lossless 12-bit weight format of "SpecPilot: Autonomous Algorithm Discovery and
 * Systems Optimization for Speculative Decoding" (arXiv 2611.02501), §4.1 "W12: A Lossless
 * 12-bit Weight Format" and Fig. 5: a BF16 weight is kept as three nibbles (A: its sign and
 * three highest mantissa bits; E: its exponent relative to the channel's 16-binade window
 * [E_n-15, E_n]; B: its four lowest mantissa bits); a weight the nibbles cannot hold (exponent
 * out of the window, zero, subnormal, Inf, NaN) is kept bit for bit in an escape list; 12 KB
 * records hold 128x64 weight tiles, the 8-bit A+E view first and plane B last.
 *
 * Conventions for every call
 *   - Memory: every data pointer is a DEVICE pointer owned by the caller. The library never
 *     allocates or frees device memory and keeps no pointer after a call returns.
 *   - Matrices are row-major and dense: W is bf16 [N, K] (row n = output channel), x is bf16
 *     [M, K], y is [M, N]. bf16 values are passed as their raw 16-bit patterns (uint16_t).
 *   - Execution: calls enqueue work on `stream` and return without waiting, except where a call
 *     says it synchronises. Argument errors are detected on the host and returned before any
 *     work is enqueued.
 *   - Shapes: N >= 1, K >= 8 with K % 8 == 0 (rows must be 16-byte aligned for the tensor-memory
 *     copies); N and K need not be multiples of the 128x64 tile. GEMM rows: 1 <= M <= 384.
 *   - Device: the current device must be a compute capability 10.3 GPU (GB300);
 *     otherwise W12_ERR_DEVICE.
 *   - Determinism: for a given device, shape and input, every output is bitwise reproducible.
 *   - Thread safety: calls may run concurrently on different streams only with separate
 *     workspaces/scratch buffers.
 */
#ifndef W12_H
#define W12_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *w12_stream_t; /* the same type as cudaStream_t; NULL = legacy stream */

typedef enum {
    W12_OK = 0,
    W12_ERR_INVALID_ARG = 1,       /* null pointer, bad size, misaligned pointer, bad enum */
    W12_ERR_UNSUPPORTED_SHAPE = 2, /* K % 8 != 0, M outside [1, 384], ... */
    W12_ERR_WORKSPACE = 3,         /* workspace or scratch smaller than the size query says */
    W12_ERR_CUDA = 4,              /* a CUDA runtime call failed (launch, copy, sync) */
    W12_ERR_MISMATCH = 5,          /* w12_verify found decoded weights that differ */
    W12_ERR_TIMEOUT = 6,           /* a kernel gave up a bounded wait; its outputs are invalid */
    W12_ERR_DEVICE = 7             /* the current device is not compute capability 10.3 */
} w12_status;

enum {
    W12_TILE_N = 128,        /* output channels per record */
    W12_TILE_K = 64,         /* reduction elements per record */
    W12_RECORD_BYTES = 12288,
    W12_VIEW_BYTES = 8192,   /* the nested 8-bit A+E view: the first two thirds of a record */
    W12_MAX_M = 384
};

enum { W12_OUT_F32 = 0, W12_OUT_BF16 = 1 };          /* y element type */
enum { W12_LAUNCH_OVERLAP = 1, W12_LAUNCH_TEST_STALL = 2, W12_LAUNCH_ACCUMULATE = 4 };  /* w12_gemm_ex flags */
enum { W12_OP_GEMM = 0, W12_OP_QVIEW_GEMM = 1, W12_OP_ARGMAX = 2, W12_OP_QVIEW_ARGMAX = 3 };

/*
 * An encoded tensor. The caller allocates every buffer with the sizes given below (n_esc and
 * n_rec_esc come from w12_encode_sizes) and fills in the fields before w12_encode.
 *   records      uint8  [n_tiles * k_tiles * 12288]  record r = nt * k_tiles + kt
 *   base_exp     uint8  [n_tiles * 128]              E_n per channel (padding channels: 16)
 *   esc_off      uint32 [N + 1]                      canonical per-channel escape list (CSR) ...
 *   esc_k        uint32 [n_esc]                      ... k of each escape, increasing per channel
 *   esc_bits     uint16 [n_esc]                      ... its exact bf16 pattern
 *   rec_esc_off  uint32 [n_tiles * k_tiles + 1]      per-record index, offsets in 32-bit words
 *   rec_esc      uint32 [n_rec_esc]                  per record with escapes: 4 header words (word q
 *                                                    = entries with n_l < 32*(q+1)), then entries
 *                                                    pos | bits << 16 (pos = 64*n_l + k_l, increasing),
 *                                                    padded to a multiple of 4 words with 0xFFFFFFFF
 * n_tiles = ceil(N / 128), k_tiles = ceil(K / 64). Buffers must be 16-byte aligned.
 */
typedef struct {
    int32_t N, K;
    int32_t n_tiles, k_tiles;
    uint8_t *records;
    uint8_t *base_exp;
    uint32_t *esc_off;
    uint32_t *esc_k;
    uint16_t *esc_bits;
    uint32_t *rec_esc_off;
    uint32_t *rec_esc;
    int64_t n_esc;
    int64_t n_rec_esc;
} w12_tensor;

/* Human-readable name of a status code (static storage). */
const char *w12_status_str(w12_status status);

/* Fills t->n_tiles and t->k_tiles for a shape and returns the byte sizes of its fixed-size
 * buffers (records, base_exp). Host only. */
w12_status w12_tensor_shape(int N, int K, w12_tensor *t, size_t *records_bytes,
                            size_t *base_exp_bytes);

/* ---- a1: encode (SpecPilot §4.1, Fig. 5a) ----------------------------------------------- */

/* Scratch bytes that w12_encode_sizes / w12_encode need for an [N, K] weight matrix. Host only. */
w12_status w12_encode_scratch_size(int N, int K, size_t *bytes);

/* Runs the window and counting passes on w (device bf16 [N, K]) and returns the number of
 * escapes (n_esc) and of per-record index entries including padding (n_rec_esc).
 * SYNCHRONISES `stream` to read the two counts back. */
w12_status w12_encode_sizes(const uint16_t *w, int N, int K, void *scratch, size_t scratch_bytes,
                            int64_t *n_esc, int64_t *n_rec_esc, w12_stream_t stream);

/* Encodes w (device bf16 [N, K]) into the caller's buffers in *t (t->N, t->K, t->n_esc and
 * t->n_rec_esc must match w12_encode_sizes). `scratch` must be the buffer that
 * w12_encode_sizes filled for this same w, N and K, unchanged since. This call reuses the window
 * bases, escape counts and offsets left there and runs only the writing pass. Writes never exceed
 * the stated buffer sizes. SYNCHRONISES `stream` and returns W12_ERR_INVALID_ARG if the counts
 * written differ from t's. */
w12_status w12_encode(const uint16_t *w, int N, int K, void *scratch, size_t scratch_bytes,
                      const w12_tensor *t, w12_stream_t stream);

/* ---- a2: load-time check (SpecPilot §4.1; Table A2 caption: the decoded weights are compared
 *          bit for bit with the checkpoint when the model loads) ------------------------------ */

/* Decodes the whole tensor into w_out (device bf16 [N, K]) from records, base_exp and the
 * per-record escape index. Asynchronous. */
w12_status w12_decode(const w12_tensor *t, uint16_t *w_out, w12_stream_t stream);

/* Scratch bytes for w12_verify (host only). */
w12_status w12_verify_scratch_size(size_t *bytes);

/* Decodes every weight and compares it bit for bit with w_ref (device bf16 [N, K]); also checks
 * each canonical (CSR) escape entry and that both escape lists hold the same number of entries.
 * *n_mismatch receives the number of differing weights/entries. SYNCHRONISES `stream`.
 * Returns W12_ERR_MISMATCH when *n_mismatch > 0. */
w12_status w12_verify(const w12_tensor *t, const uint16_t *w_ref, void *scratch,
                      size_t scratch_bytes, uint64_t *n_mismatch, w12_stream_t stream);

/* ---- a3-a5: the skinny GEMMs ------------------------------------------------------------- */

/* Workspace bytes for one of the W12_OP_* operations at M rows on the current device (host
 * only). The workspace must be zero-filled once before its first use; every successful call
 * leaves it zeroed again. Calls that share a workspace must not overlap on the GPU. */
w12_status w12_workspace_size(const w12_tensor *t, int M, int op, size_t *bytes);

/* a3 (SpecPilot §4.1 and Fig. 5b; §6.3): y[m, n] = sum_k x[m, k] * w[n, k] with every weight
 * decoded exactly in registers and fp32 accumulation; y is fp32 or bf16 (round to nearest even)
 * [M, N] by y_dtype. x: device bf16 [M, K], 16-byte aligned. When the k range is split
 * between blocks, their parts are added in one fixed order (run-to-run identical). Asynchronous. */
w12_status w12_gemm(const w12_tensor *t, const uint16_t *x, int M, void *y, int y_dtype,
                    void *workspace, size_t workspace_bytes, w12_stream_t stream);

/* a5 (SpecPilot §4.3 "Zero-copy Q pass", Fig. 7): the same GEMM over the nested 8-bit view only
 * (first 8192 bytes of each record): low mantissa bits := 1000b, escapes not patched.
 * Asynchronous. */
w12_status w12_qview_gemm(const w12_tensor *t, const uint16_t *x, int M, void *y, int y_dtype,
                          void *workspace, size_t workspace_bytes, w12_stream_t stream);

/* a4 (SpecPilot §2.1 greedy acceptance of the target argmax; §4.1 and App. E, the LM head): the
 * GEMM fused with a per-row argmax; y is never written. Per row m: idx[m] = smallest n with the
 * largest y[m, n]; val[m] = that value; gap[m] = val[m] - the largest y[m, n'] over n' != idx[m]
 * (0 on an exact tie, +inf when N == 1). qview != 0 runs it over the 8-bit view as in
 * w12_qview_gemm. NaN logits are not ranked. idx/val/gap: device arrays of M elements.
 * Asynchronous. */
w12_status w12_lmhead_argmax(const w12_tensor *t, const uint16_t *x, int M, int32_t *idx,
                             float *val, float *gap, int qview, void *workspace,
                             size_t workspace_bytes, w12_stream_t stream);

/* The GEMM family with launch options (the paper has no counterpart of the options).
 * op is one of W12_OP_*. The GEMM ops write y (y_dtype) and take idx, val and gap as NULL. The
 * argmax ops write idx, val and gap and take y as NULL. Any other argument combination returns
 * W12_ERR_INVALID_ARG.
 * flags = 0 behaves exactly as w12_gemm, w12_qview_gemm or w12_lmhead_argmax.
 * flags = W12_LAUNCH_OVERLAP uses a programmatic dependent launch: the kernel may start while the
 * kernel before it on `stream` is still finishing, and meanwhile fetches and decodes its
 * weights. It reads x, reads and writes the workspace, and writes its outputs only after that
 * kernel has completed and its memory is visible.
 * Contract for the overlap: nothing the preceding kernel does may write t's buffers (records,
 * base_exp, rec_esc_off, rec_esc). They must already hold their final contents when the
 * preceding kernel starts, as they do for weights loaded once and reused.
 * This launch also lets the next kernel on the stream start early. That next kernel must itself
 * wait for this one before using its results, as kernels launched with this flag do.
 * The kernel's bounded waits give up after about a second, so the preceding kernel must not run
 * much longer than that after this launch begins.
 * flags with W12_LAUNCH_ACCUMULATE (GEMM ops with fp32 y only, else W12_ERR_INVALID_ARG): y += the
 * result instead of y = the result, one fp32 addition per element (a residual add fused into the
 * GEMM); deterministic like the plain GEMM. It combines with W12_LAUNCH_OVERLAP (y is read only
 * after the preceding kernel has completed).
 * flags = W12_LAUNCH_TEST_STALL is a test hook for the failure path. Each block's producer fills
 * only its first pipeline slot, so the block's bounded waits run out after about a second. Every
 * block then stops, the call's outputs are invalid, and w12_check reports W12_ERR_TIMEOUT; the
 * workspace must then be zero-filled again. Nothing else in the library sets it.
 * Asynchronous. */
w12_status w12_gemm_ex(const w12_tensor *t, const uint16_t *x, int M, int op, void *y, int y_dtype,
                       int32_t *idx, float *val, float *gap, unsigned flags, void *workspace,
                       size_t workspace_bytes, w12_stream_t stream);

/* w12_gemm_ex with activation rows ldx elements apart (the paper has no counterpart): x is row m
 * at x + m * ldx, K elements each, so a column range of a wider bf16 output (say the q part of
 * a concatenated q|k|v projection) feeds the next GEMM without a copy. ldx >= K and ldx % 8 == 0
 * (16-byte rows); otherwise W12_ERR_INVALID_ARG. Everything else as w12_gemm_ex. Asynchronous. */
w12_status w12_gemm_strided(const w12_tensor *t, const uint16_t *x, int ldx, int M, int op, void *y, int y_dtype,
                            int32_t *idx, float *val, float *gap, unsigned flags, void *workspace,
                            size_t workspace_bytes, w12_stream_t stream);

/* The paper has no counterpart of this call. It is w12_gemm for callers that cannot allocate
 * device memory: a plug-in whose host framework owns all device memory and hands none out, or a
 * serving loop that must not call cudaMalloc because cudaMalloc can synchronise the device. The
 * workspace lives in a fixed array of about 8.5 MB inside the library; every GPU that loads the
 * library holds it until the process exits. The caller still passes x and y (device pointers,
 * laid out as for w12_gemm).
 * Limits: 1 <= M <= 32, at most 4096 tiles of 128 output channels (N <= 524288) and at most 256
 * thread blocks; larger problems return W12_ERR_UNSUPPORTED_SHAPE. The call allocates nothing:
 * it clears the array's counters and error word with cudaMemsetAsync on `stream`, then launches
 * the GEMM kernel. Every call looks up the array's device address on the current device
 * (cudaGetSymbolAddress); the first call on a device may also load the library's device code
 * there, so make that first call before any stream capture. All calls on a device share the one
 * array, so calls that overlap on the GPU race:
 * order them (one stream, or events). A kernel that gives up one of its bounded waits is not
 * reported by this call (use w12_gemm with w12_check where that matters). Asynchronous. */
w12_status w12_gemm_noalloc(const w12_tensor *t, const uint16_t *x, int M, void *y, int y_dtype,
                            w12_stream_t stream);

/* ---- glue of the synthetic layer stream (the pages give no layer dataflow) ---------------
 * The synthetic 64-layer stream carries M rows from layer to layer (the reading taken here): h fp32
 * [M, K]; x = bf16(h / rms(h)); a = bf16(x Wq^T); h += a Wo^T (W12_LAUNCH_ACCUMULATE);
 * x2 = bf16(h / rms(h)); p = bf16((x2 Wg^T) * (x2 Wu^T)); h += p Wd^T. These two calls are its
 * steps between the GEMMs. flags: 0 or W12_LAUNCH_OVERLAP (the kernel may start while the
 * previous kernel on the stream finishes and reads its input only after that kernel has
 * completed). Both let the next kernel start early; a GEMM launched with W12_LAUNCH_OVERLAP
 * waits for their completion before it reads x. M in [1, W12_MAX_M]. Asynchronous. */

/* x[m, k] = h[m, k] / sqrt(mean_k h[m, k]^2) rounded to bf16 (nearest even), the quotient
 * evaluated to about 2^-40 relative accuracy before that one rounding (so x can differ from the
 * correctly rounded quotient only where the quotient lies that close to a rounding boundary);
 * zeros for an all-zero row. h: device fp32 [M, K], finite, 16-byte aligned; x: device bf16
 * [M, K], 8-byte aligned. K % 4 != 0 returns W12_ERR_UNSUPPORTED_SHAPE. */
w12_status w12_rms_bf16(const float *h, int M, int K, uint16_t *x, unsigned flags, w12_stream_t stream);

/* p[m, n] = bf16(g[m*ld + n] * u[m*ld + n]) for n < N: the fp32 product rounded to nearest even.
 * g, u: device fp32 with row stride ld >= N (g and u may be two halves of one [M, 2N] GEMM output,
 * ld = 2N); p: device bf16 [M, N]. */
w12_status w12_mul_bf16(const float *g, const float *u, int M, int N, int ld, uint16_t *p, unsigned flags,
                        w12_stream_t stream);

/* ---- f3: the persistent cross-GEMM kernel of the layer stream (SpecPilot App. F and Table
 *      A7: one persistent kernel over a sequence of W12 GEMMs) -----------------------------------
 * One cooperative launch runs a whole decoding step of the synthetic layer stream above, every
 * GEMM and every glue step of n_layers layers, then the final row normalisation:
 *   per layer  x = rms_bf16(h); qkv = bf16(x Wqkv^T); h += qkv[:, :n_q] Wo^T;
 *              x2 = rms_bf16(h); p = bf16((x2 Wg^T) * (x2 Wu^T)); h += p Wd^T
 *   then       x_out = rms_bf16(h)
 * with the arithmetic of the separate calls (w12_gemm with the same work split, w12_rms_bf16,
 * w12_mul_bf16, W12_LAUNCH_ACCUMULATE), so it gives the rows that chain of launches gives.
 * Weights stream continuously from one GEMM to the next: a GEMM's records are fetched and
 * decoded while the phase before it finishes, and only its activation copies wait for that
 * phase to complete on every block. The kernel uses every SM (one block each; a cooperative
 * launch, so it fails with W12_ERR_CUDA rather than starting when the GPU cannot hold them all). */
enum { W12_STREAM_MAX_LAYERS = 80, W12_STREAM_MAX_M = 32 };

/* The four encoded linears of one layer. All layers must have the same shapes:
 *   qkv      [n_qkv, hidden]: q in its first n_q rows, then k and v (their outputs are dropped)
 *   o        [hidden, n_q]
 *   gate_up  [2 * ffn, hidden]: rows 128 i .. 128 i + 63 are gate rows 64 i .., rows
 *            128 i + 64 .. 128 i + 127 the matching up rows (w12_stream_interleave builds it)
 *   down     [hidden, ffn]
 * hidden, ffn and n_q must be multiples of 64 and n_qkv a multiple of 8, else
 * W12_ERR_UNSUPPORTED_SHAPE. */
typedef struct {
    w12_tensor qkv, o, gate_up, down;
} w12_stream_layer;

/* Workspace bytes of w12_stream_step (host only). The workspace must be zero-filled once before
 * its first use; every completed step leaves its counters zeroed. It also holds the step's
 * intermediate activations. 1 <= n_layers <= W12_STREAM_MAX_LAYERS, 1 <= M <= W12_STREAM_MAX_M. */
w12_status w12_stream_workspace_size(const w12_stream_layer *layers, int n_layers, int M, int n_q, size_t *bytes);

/* Byte offsets inside the workspace of the last layer's intermediates after a step (host only,
 * for inspection and tests): offsets[0] x (bf16 [M, hidden]), [1] the q|k|v output (bf16
 * [M, n_qkv]), [2] x2 (bf16 [M, hidden]), [3] p (bf16 [M, ffn]). */
w12_status w12_stream_buffers(const w12_stream_layer *layers, int n_layers, int M, int n_q, size_t offsets[4]);

/* One decoding step over n_layers layers (layers: a HOST array of n_layers descriptors whose
 * buffers are device memory). h: device fp32 [M, hidden], 16-byte aligned, the rows carried in
 * (updated in place); x_out: device bf16 [M, hidden], 8-byte aligned, receives rms_bf16 of the
 * final h (the LM head's input). workspace: device, 256-byte aligned, w12_stream_workspace_size
 * bytes. Asynchronous on `stream`. Every wait inside the kernel is bounded (about a second); a
 * block that gives up sets the workspace's error word (w12_check reports W12_ERR_TIMEOUT). */
w12_status w12_stream_step(const w12_stream_layer *layers, int n_layers, int M, int n_q, float *h, uint16_t *x_out,
                           void *workspace, size_t workspace_bytes, w12_stream_t stream);

/* w12_stream_step with launch flags: 0, or W12_LAUNCH_TEST_STALL, a test hook for the failure
 * path: each block's activation producer issues the copies of its first slot only, so the
 * block's bounded waits run out after about a second. Every block then stops, h and x_out are
 * invalid, w12_check reports W12_ERR_TIMEOUT, and the workspace must be zero-filled again.
 * Nothing else in the library sets it. Other flags: W12_ERR_INVALID_ARG. */
w12_status w12_stream_step_ex(const w12_stream_layer *layers, int n_layers, int M, int n_q, float *h,
                              uint16_t *x_out, void *workspace, size_t workspace_bytes, unsigned flags,
                              w12_stream_t stream);

/* The gate|up layout w12_stream_step reads, from gate and up (device bf16 [ffn, hidden] each,
 * row-major; ffn % 64 == 0): gate_up (device bf16 [2 * ffn, hidden]) gets gate rows 64 i .. 64 i
 * + 63 at rows 128 i .., and up rows 64 i .. at rows 128 i + 64 ... Two strided device copies on
 * `stream`; asynchronous. */
w12_status w12_stream_interleave(const uint16_t *gate, const uint16_t *up, int ffn, int hidden, uint16_t *gate_up,
                                 w12_stream_t stream);

/* SYNCHRONISES `stream`, then reports W12_ERR_TIMEOUT if a GEMM kernel that used this
 * workspace gave up one of its bounded waits (its outputs are then invalid and the workspace
 * must be zero-filled again); W12_OK otherwise. Clears the flag. */
w12_status w12_check(void *workspace, size_t workspace_bytes, w12_stream_t stream);

/* Kernel configuration a GEMM call would use (for reports): grid size, pipeline stages,
 * dynamic shared memory bytes. Host only. */
w12_status w12_gemm_config(const w12_tensor *t, int M, int op, int *grid, int *stages,
                           int *smem_bytes);

/* ---- certified LM head (SpecPilot §4.1 "Certified LM head") ------------------------------
 * The head is also kept as INT8 codes with a bound per row (Cauchy-Schwarz on the quantisation
 * residual); a token whose upper bound falls below another token's lower bound cannot win and is
 * dropped, the tokens left are scored again from the W12 head, and a row that keeps too many
 * falls back to the full W12 argmax. The argmax and the top-1/top-2
 * gap are those of the whole head.
 *
 * The copy, per output row n of the bf16 head W [N, K] (the readings the pages leave open):
 *   scale[n] = max_k |W[n,k]| / 127 rounded to fp32 (0 for an all-zero row, a padding row, or a
 *              row holding Inf or NaN)
 *   q[n,k]   = W[n,k] / scale[n] rounded to the nearest integer (ties to even), clamped to +-127,
 *              stored as a sign-magnitude byte (bit 7 sign, bits 0-6 |q|) in 128 x 64 records of
 *              8192 bytes laid out like the W12 record's 8-bit view: record r = nt * k_tiles + kt,
 *              byte 2048 * (k_l >> 4) + 16 * n_l + (k_l & 15)
 *   bound[n] = an fp32 upper bound on ||W[n,:] - scale[n] q[n,:]||_2 plus the fp32 evaluation
 *              margin of scale[n] (x . q[n,:]); +inf for a row holding Inf or NaN
 * For a row x the certified logit interval is scale[n] (x . q[n,:]) -+ ||x||_2 bound[n].
 */
typedef struct {
    int32_t N, K;
    int32_t n_tiles, k_tiles;
    uint8_t *codes;  /* [n_tiles * k_tiles * 8192] */
    float *scale;    /* [n_tiles * 128] */
    float *bound;    /* [n_tiles * 128] */
} w12_q8_head;

enum { W12_Q8_RECORD_BYTES = 8192, W12_Q8_MAX_SURVIVORS = 4096 };

/* Fills h->N, K, n_tiles, k_tiles and returns the byte sizes of codes and of scale / bound.
 * Host only. */
w12_status w12_q8_shape(int N, int K, w12_q8_head *h, size_t *codes_bytes, size_t *row_bytes);

/* Builds the copy from the bf16 head w [h->N, h->K] (device, row-major, 16-byte aligned) into
 * the caller's buffers. Asynchronous on `stream`. */
w12_status w12_q8_build(const uint16_t *w, const w12_q8_head *h, w12_stream_t stream);

/* Workspace bytes of w12_lmhead_certified for t (the W12 head), h and M rows. The workspace
 * must be zero-filled once; every call leaves it zeroed. Host only. */
w12_status w12_certified_workspace_size(const w12_tensor *t, const w12_q8_head *h, int M, size_t *bytes);

/* idx / val / gap (device, [M]) as w12_lmhead_argmax returns them, through the certified head;
 * survivors (device, [M], may be NULL) receives each row's survivor count. t and h must
 * describe the same head (same N, K). w_bf16 (device, may be NULL) is the head in bf16,
 * row-major [N, K] with K % 8 == 0 and 16-byte alignment: when given, survivors are rescored
 * from its contiguous rows, otherwise from t's records and escapes (a gather of 16-byte pieces,
 * no extra memory). M in [1, W12_MAX_M]. If a row has more than
 * W12_Q8_MAX_SURVIVORS survivors, the full W12 argmax produces every row's result.
 * Asynchronous on `stream`: four kernels, then the full argmax, which does nothing unless a row
 * overflowed. */
w12_status w12_lmhead_certified(const w12_tensor *t, const w12_q8_head *h, const uint16_t *w_bf16,
                                const uint16_t *x, int M,
                                int32_t *idx, float *val, float *gap, int32_t *survivors, void *workspace,
                                size_t workspace_bytes, w12_stream_t stream);

/* The Q pass over the separate INT8 copy (SpecPilot §5.3 and App. C: an INT6/INT8 Q-pass
 * copy next to the nested view): idx / val / gap of each row's argmax of
 * scale[n] (x . q[n,:]), computed like w12_lmhead_argmax (fp32 accumulation, ties to the
 * smaller index). flags: 0 or W12_LAUNCH_OVERLAP. The workspace must be zero-filled once; every
 * call leaves it zeroed. Asynchronous. */
w12_status w12_q8_argmax_workspace_size(const w12_q8_head *h, int M, size_t *bytes);
w12_status w12_q8_argmax(const w12_q8_head *h, const uint16_t *x, int M, int32_t *idx, float *val, float *gap,
                         unsigned flags, void *workspace, size_t workspace_bytes, w12_stream_t stream);

/* ---- INT6 Q-pass copy (SpecPilot §5.3 "Generality Through Memory": the INT6 copy added for
 *      the Q pass, and the INT6/INT8 Q-pass copy; App. C: the Q pass reads the nested 8-bit
 *      view or a separate low-precision copy) -------------------------------------------------
 * A separate 6-bit copy of a weight matrix for the low-precision Q pass: 0.75 bytes per weight
 * against the nested view's 1.0 and W12's 1.5. The pages give no formulas; the copy here is
 * the INT8 copy's per-row symmetric quantisation with 6-bit codes. Per output row n of the bf16
 * matrix W [N, K]:
 *   scale[n] = max_k |W[n,k]| / 31 rounded to fp32 (0 for an all-zero row, a padding row, or a
 *              row holding Inf or NaN; that row's codes are 0)
 *   c[n,k]   = W[n,k] / scale[n] rounded to the nearest integer (ties to even), clamped to +-31
 * and the Q pass computes yq[m,n] = scale[n] * sum_k x[m,k] c[n,k] with fp32 accumulation.
 * Records: one per 128 x 64 tile (record r = nt * k_tiles + kt), 6144 bytes, holding u = c + 32
 * (padding rows and columns hold u = 32) in 32-bit little-endian words. For local row n_l and
 * k_l = 16 g + 2 j + h (group g 0..3, pair j 0..7, half h 0..1):
 *   plane L, bytes [0, 4096): the low four bits of u, in row word i = 2 g + (j >> 2) at bits
 *     4 (j & 3) + 16 h; row words 0-3 lie at byte 16 n_l + 4 i, words 4-7 at 2048 + 16 n_l + 4 (i - 4)
 *   plane T, bytes [4096, 6144): the top two bits of u, in row word g at byte 4096 + 16 n_l + 4 g,
 *     bits 2 j + 16 h
 */
typedef struct {
    int32_t N, K;
    int32_t n_tiles, k_tiles;
    uint8_t *codes;  /* [n_tiles * k_tiles * 6144] */
    float *scale;    /* [n_tiles * 128] */
} w12_q6_copy;

enum { W12_Q6_RECORD_BYTES = 6144 };

/* Fills c->N, K, n_tiles, k_tiles and returns the byte sizes of codes and of scale. Host only. */
w12_status w12_q6_shape(int N, int K, w12_q6_copy *c, size_t *codes_bytes, size_t *scale_bytes);

/* Builds the copy from the bf16 matrix w [c->N, c->K] (device, row-major, 16-byte aligned) into
 * the caller's buffers. Asynchronous. */
w12_status w12_q6_build(const uint16_t *w, const w12_q6_copy *c, w12_stream_t stream);

/* Workspace bytes of w12_q6_gemm (argmax = 0) or w12_q6_argmax (argmax != 0) at M rows. The
 * workspace must be zero-filled once before its first use; every call leaves it zeroed. Calls
 * that share a workspace must not overlap on the GPU. Host only. */
w12_status w12_q6_workspace_size(const w12_q6_copy *c, int M, int argmax, size_t *bytes);

/* yq = x . (scale * c)^T as above: x device bf16 [M, K] (16-byte aligned), y [M, N] fp32 or
 * bf16 (round to nearest even) by y_dtype. flags: 0 or W12_LAUNCH_OVERLAP (as for w12_gemm_ex:
 * the copy's buffers must hold their final contents when the preceding kernel starts).
 * Asynchronous. */
w12_status w12_q6_gemm(const w12_q6_copy *c, const uint16_t *x, int M, void *y, int y_dtype, unsigned flags,
                       void *workspace, size_t workspace_bytes, w12_stream_t stream);

/* The Q pass's row argmax over the copy: idx / val / gap (device, [M]) of each row of yq,
 * computed like w12_lmhead_argmax (ties to the smaller index, NaN not ranked). flags: 0 or
 * W12_LAUNCH_OVERLAP. Asynchronous. */
w12_status w12_q6_argmax(const w12_q6_copy *c, const uint16_t *x, int M, int32_t *idx, float *val, float *gap,
                         unsigned flags, void *workspace, size_t workspace_bytes, w12_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* W12_H */
