/*
 * h3q.h -- C ABI of the fused NVFP4 activation producers (GB300, sm_103a).
 *
 * Producers that turn bf16 activations into NVFP4 GEMM inputs with the
 * quantize fused into the kernel that produces them: RMSNorm + AdaLN, SwiGLU
 * and the standalone (attention-output) quantize; the residual fold before the
 * norm and the SwiGLU of a packed projection with its bias; abs-max passes for
 * dynamic and calibrated global scales.  Beside them, the QKV epilogue (bias,
 * per-head RMSNorm and rotate-half RoPE, bf16 outputs) and a dequantize used
 * for checking.  Every NVFP4 producer writes:
 *
 *   codes   uint8 [rows, cols/2]: E2M1 codes, two per byte, the even column in
 *           the low nibble (FastVideo compare "fasth3-spark-exact-perf",
 *           minimax_h3_swiglu_quant.cuh, fp4_pair).  Row pitch cols/2 bytes.
 *   scales  uint8 [h3q_padded_rows(rows), cols/16]: one E4M3 block scale per
 *           16 elements, in the 128x4 swizzled layout; the byte of (row r,
 *           scale column g) is at
 *             ((r/128)*(cols/64) + g/4)*512 + (r%32)*16 + ((r/32)%4)*4 + g%4.
 *           Padding rows rows..h3q_padded_rows(rows)-1 are written as zero.
 *           (FastVideo API page fastvideo.models.vaes.minimax_h3_nvfp4_fused:
 *           introduction -- "E4M3 block scales, layout_128x4 swizzle, zeroed
 *           padding rows" -- and new_quantized; the index is written out in
 *           quant_probe of the FastVideo compare page.)
 *
 * Block quantize (16 consecutive elements y of one row, global scale gsf):
 *   sf = E4M3_rn_satfinite(fl(gsf * fl(amax/6))), dec = fl(E4M3value(sf)/gsf),
 *   inv = dec != 0 ? fl(1/dec) : 0, code_i = E2M1_rn_satfinite(fl(y_i * inv)).
 * This is quant_probe of the FastVideo compare page with every approximate
 * reciprocal replaced by a correctly rounded division.
 *
 * Common conventions
 * ------------------
 * Memory    All pointers are DEVICE pointers into memory owned by the caller
 *           (the host-buffer call also takes host pointers).  No call allocates
 *           device or host memory, frees, or keeps a caller's pointer after it
 *           returns.  Buffers must stay alive until the work queued on `stream`
 *           has finished.  The one thing the library creates is the pair of
 *           streams and 11 events of h3q_rmsnorm_adaln_nvfp4_host, once per CUDA
 *           context on that call's first use in it, kept until the process ends
 *           (see there).
 * Stream    `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *           default stream).  Every call is asynchronous: it validates its
 *           arguments on the host, launches its kernel on `stream` (the
 *           dynamic-scale quantize launches three, in order) and returns.
 *           No call synchronises.  The device is the calling thread's current
 *           CUDA device.
 * Global    `global_scale` points to one fp32 on the device: the static
 *   scale   per-tensor scale gsf (finite, > 0; not checked, reading it would
 *           need a synchronisation).  It is read by the kernel, so it may be
 *           updated on the stream between calls and captured in a graph.
 * Shapes    rows >= 0 (rows == 0 is a successful no-op); cols > 0, a multiple
 *           of 64 (four scale columns form one swizzle atom), at most 2^24.
 *           ld_* is the row stride of an input in ELEMENTS: >= cols and a
 *           multiple of 16.  Indexing is 64-bit throughout: inputs larger
 *           than 2^31 elements are supported (FastVideo commit log, branch
 *           vae-parallel-decode, the int64 program-id fix).
 * Alignment bf16 inputs and fp32 outputs: 32-byte aligned.  codes, scales and
 *           the QKV epilogue's bf16 outputs: 16-byte aligned.  row_frame,
 *           global_scale, amax, row_rstd: 4-byte.
 * Aliasing  Outputs must not overlap inputs or each other.
 * Errors    H3Q_OK (0) on success.  H3Q_ERR_INVALID_ARGUMENT (1): an argument
 *           broke a rule above; nothing was launched and no output was
 *           touched.  H3Q_ERR_CUDA (2): the CUDA runtime reported an error
 *           (no device, launch failure, or a sticky error from earlier work).
 *           h3q_last_error() returns a message for the calling thread's most
 *           recent failure.  No call aborts, traps or prints.
 * Threads   The calls keep two kinds of state between calls, both per CUDA
 *           context (keyed on the context's unique id, so a context destroyed
 *           and re-created, e.g. by cudaDeviceReset, starts afresh): a cache of
 *           launch sizes (occupancy, and the raised shared-memory limit of the
 *           kernels that need one), and the host-buffer call's streams and
 *           events.  They are safe to call from several threads.  The one
 *           exception is h3q_quantize_nvfp4_dynamic, whose abs-max partials live
 *           in a device array inside the library: calls of it that overlap on
 *           one device race (see there).
 */
#ifndef H3Q_H
#define H3Q_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define H3Q_OK 0
#define H3Q_ERR_INVALID_ARGUMENT 1
#define H3Q_ERR_CUDA 2

#define H3Q_ABI_VERSION 4

/* Rows of the scale matrix: rows rounded up to a multiple of 128. */
static inline int64_t h3q_padded_rows(int64_t rows) { return (rows + 127) / 128 * 128; }
/* Bytes of the swizzled scale matrix. */
static inline int64_t h3q_scale_bytes(int64_t rows, int64_t cols)
{
    return h3q_padded_rows(rows) * (cols / 16);
}
/* n rounded up to a multiple of 256 bytes. */
static inline int64_t h3q_align256(int64_t n) { return (n + 255) / 256 * 256; }
/* Device workspace of h3q_rmsnorm_adaln_nvfp4_host: three staging slots of
 * chunk_rows rows, each an x chunk, a code chunk and a scale chunk (each part
 * rounded up to 256 bytes, in that order), then -- when the frames come from
 * rows_per_frame (with_frames != 0) -- the rows' frame indices, rows int32. */
static inline int64_t h3q_host_workspace_bytes(int64_t chunk_rows, int64_t cols, int64_t rows,
                                               int with_frames)
{
    int64_t slot = h3q_align256(chunk_rows * cols * 2) + h3q_align256(chunk_rows * cols / 2) +
                   h3q_align256(chunk_rows * cols / 16);
    return 3 * slot + (with_frames ? h3q_align256(rows * 4) : 0);
}
/* Bytes of the packed code matrix. */
static inline int64_t h3q_code_bytes(int64_t rows, int64_t cols) { return rows * (cols / 2); }
/* Byte offset, in the scale matrix, of the scales of row `row0` onwards when
 * row0 is a multiple of 128: the 512-byte atoms are laid out row-tile major, so
 * the scales of rows [row0, row0 + n) with n a multiple of 128 (or the tensor's
 * last rows) form one contiguous range starting here.  A call on those rows
 * writes exactly that range, which lets a large tensor be processed in
 * 128-row-aligned pieces. */
static inline int64_t h3q_scale_offset_of_row_tile(int64_t row0, int64_t cols)
{
    return row0 / 128 * (cols / 64) * 512;
}

/*
 * Standalone NVFP4 quantize, e.g. of the attention output viewed as
 * [tokens, heads*head_dim].  (TensorRT-LLM PR #21483 "Fuse the MiniMax-H3
 * NVFP4 activation quantize into the AdaLN, SwiGLU and attention-output
 * producers", commit "...quantize it with a bandwidth-bound kernel";
 * FastVideo API page, quantize.)
 *
 *   x             bf16 [rows, cols], row stride ld_x elements.
 *   global_scale  device fp32 gsf.
 *   codes         out, rows*cols/2 bytes.    scales  out, h3q_scale_bytes.
 */
int h3q_quantize_nvfp4(const void *x, int64_t ld_x, int64_t rows, int64_t cols,
                       const float *global_scale, uint8_t *codes, uint8_t *scales,
                       void *stream);

/*
 * RMSNorm with fp32 statistics, AdaLN modulation, NVFP4.  (TensorRT-LLM
 * PR #21483, summary and commit "...SwiGLU producers": the AdaLN RMSNorm +
 * modulation kernel emits packed E2M1 codes and swizzled E4M3 scales
 * directly; FastVideo API page, introduction: fp32 statistics, sequential
 * FMA per thread, no contraction of products that eager rounds.)
 *
 * Per row r with frame t:
 *   ss   = sum of x^2 in the canonical order: 8-element chunk c goes to lane
 *          c % 128; each lane keeps 8 fp32 partials, element e of its chunks
 *          (chunks in increasing order) is fused-multiply-added into partial e;
 *          lane total ((p0+p1)+(p2+p3))+((p4+p5)+(p6+p7)); within each group of
 *          32 lanes a butterfly over xor-distances 16,8,4,2,1 gives the group
 *          total T_w; ss = (T_0+T_1)+(T_2+T_3).
 *   rstd = fl(1 / fl(sqrt(fl(fl(ss / cols) + eps))))
 *   y    = bf16(fl(fl(fl(fl(x * rstd) * gamma) * fl(1 + scale[t])) + shift[t]))
 * then y is block-quantized.
 *
 *   x               bf16 [rows, cols], row stride ld_x elements.
 *   gamma           bf16 [cols].
 *   mod_table       bf16 [num_frames, 2, cols], contiguous: [t][0] is the shift,
 *                   [t][1] the scale.
 *   row_frame       int32 [rows] frame of each row, or NULL.  Entries must lie in
 *                   [0, num_frames) (the index contract of the FastVideo commit
 *                   log's modulation wrappers).  They are not checked on the
 *                   host (that would need a synchronisation); the kernel clamps
 *                   them into range so memory stays safe, and the output of a
 *                   row with an out-of-range entry is unspecified.
 *   rows_per_frame  used when row_frame is NULL: frame = row / rows_per_frame;
 *                   must be >= 1 with (rows-1)/rows_per_frame < num_frames.
 *   eps             finite, >= 0.  With eps = 0 a row whose sum of squares is 0 has
 *                   rstd = 1/0 = +inf and NaN values (0 * inf); its codes and scales
 *                   are then unspecified, like those of NaN or infinite inputs.
 *   row_rstd        optional out fp32 [rows]: rstd of each row, or NULL.
 */
int h3q_rmsnorm_adaln_nvfp4(const void *x, int64_t ld_x, const void *gamma,
                            const void *mod_table, int64_t num_frames, const int32_t *row_frame,
                            int64_t rows_per_frame, float eps, int64_t rows, int64_t cols,
                            const float *global_scale, uint8_t *codes, uint8_t *scales,
                            float *row_rstd, void *stream);

/*
 * SwiGLU producer: y = bf16(fl(fl(g * sigma) * u)) with
 * sigma = fl(1 / fl(1 + exp_c(-g))), then NVFP4.  (FastVideo compare page,
 * minimax_h3_swiglu_quant.cuh, swiglu_bf16: value * silu(gate) rounded to
 * bf16; TensorRT-LLM PR #21483, SiLU-and-mul producer.)  exp_c is a fixed
 * sequence of binary32 operations: Cody-Waite reduction by a two-part ln 2
 * applied with FMAs and a degree-7 Taylor polynomial in Horner form.
 *
 *   gate, up  bf16 [rows, cols], row strides ld_gate, ld_up elements (a
 *             gate/up pair packed in one [rows, 2*cols] projection is two views
 *             with ld = 2*cols).
 */
int h3q_swiglu_nvfp4(const void *gate, int64_t ld_gate, const void *up, int64_t ld_up,
                     int64_t rows, int64_t cols, const float *global_scale, uint8_t *codes,
                     uint8_t *scales, void *stream);

/*
 * SwiGLU of a value-first packed projection with its bias (FastVideo API page,
 * swiglu_quantize: o [M, 2F], value first, gate second, bias not yet added).
 * Each half gets its bias in binary32 and is rounded to bf16,
 *   v = bf16(fl(o[:, j] + bias[j])),  g = bf16(fl(o[:, F + j] + bias[F + j])),
 * then as h3q_swiglu_nvfp4: y = bf16(fl(fl(g * sigma(g)) * v)), quantized.
 *
 *   o       bf16 [rows, 2F], row stride ld_o (>= 2F, a multiple of 16), 32-byte aligned.
 *   bias    bf16 [2F] (value biases, then gate biases), 32-byte aligned, or NULL.
 *   f       F, a multiple of 64; codes [rows, F/2] and scales [pad128(rows), F/16].
 */
int h3q_swiglu_packed_nvfp4(const void *o, int64_t ld_o, const void *bias, int64_t rows,
                            int64_t f, const float *global_scale, uint8_t *codes, uint8_t *scales,
                            void *stream);

/*
 * Dequantize (checking path): out[r][j] = fl((E2M1value(c) * E4M3value(sf)) / gsf),
 * the value a block-scaled NVFP4 GEMM with alpha = 1/gsf sees for the element.
 * No page defines it; it is the inverse the producers' consumers apply.
 *
 *   codes, scales  as written by the producers (scales in the swizzled layout).
 *   out            fp32 [rows, cols], contiguous.
 */
int h3q_dequantize_nvfp4(const uint8_t *codes, const uint8_t *scales, int64_t rows, int64_t cols,
                         const float *global_scale, float *out, void *stream);

/*
 * Residual fold + RMSNorm + AdaLN -> NVFP4 (the residual add folded into the
 * next norm).  TensorRT-LLM PR #21483, commit "...norm1 ... from a second
 * table": a block folds its MLP residual into the next block's norm1 kernel,
 * reading the gate from its own AdaLN table while the scale and shift come from
 * the next block's.  FastVideo API page, residual_norm_quantize: in place
 * h += bf16(o + bias) * scale on a contiguous fp32 residual, then NVFP4 of the
 * normed h.  Per row r with frame t:
 *   u   = bf16(fl(o + bias))           (u = o when bias is NULL)
 *   h'  = fl(h + fl(u * gate[t]))      written back to h
 *   then h3q_rmsnorm_adaln_nvfp4's arithmetic on the fp32 values h' (same
 *   canonical reduction order, squares of fp32 values) and the NVFP4 quantize.
 *
 *   h           fp32 [rows, cols], row stride ld_h (>= cols, a multiple of 8),
 *               32-byte aligned; read and overwritten with h'.
 *   o           bf16 [rows, cols], row stride ld_o, as x of the other producers.
 *   bias        bf16 [cols] or NULL.
 *   gate_table  bf16 [num_frames, cols]: the gate of each frame (this block's).
 *   gamma, mod_table, num_frames, row_frame, rows_per_frame, eps, global_scale,
 *   codes, scales, row_rstd: as h3q_rmsnorm_adaln_nvfp4 (the next block's
 *               modulation table; the frame of a row indexes both tables).
 * Limits: cols <= 8,192.  h, codes, scales and row_rstd must not overlap an
 * input or each other.  Status codes as the other producers.
 */
int h3q_residual_rmsnorm_adaln_nvfp4(float *h, int64_t ld_h, const void *o, int64_t ld_o,
                                     const void *bias, const void *gate_table, const void *gamma,
                                     const void *mod_table, int64_t num_frames,
                                     const int32_t *row_frame, int64_t rows_per_frame, float eps,
                                     int64_t rows, int64_t cols, const float *global_scale,
                                     uint8_t *codes, uint8_t *scales, float *row_rstd,
                                     void *stream);

/*
 * Dynamic and calibrated global scales.
 *
 * FastVideo API page, NVFP4DecoderLinear: a dynamic layer scales each call by
 * the abs-max of its input, and a calibrating layer folds each call's abs-max
 * into a persistent running maximum (input_amax).  FlashRT PR #142, commit
 * "...amax pipeline": the abs-max is taken on the device in a pass of its own
 * and read by the quantize pass with no host synchronisation.
 *
 * The three abs-max passes compute the producer's bf16 output y exactly as the
 * producer does (same arguments, same arithmetic) without storing it, and fold
 * max |y| into *amax: *amax = max(*amax, max |y|).  Zero *amax first for a
 * per-call abs-max; keep it across calls for a running maximum.
 *
 *   amax  device fp32 scalar, 4-byte aligned, holding a value >= 0 (+0.0, not
 *         -0.0) on entry; updated with an atomic maximum, so several passes
 *         may fold into it, on one stream or several.
 *
 * Then h3q_global_scale_from_amax writes *global_scale = fl(2688 / *amax) on the
 * device (2688 = 448 * 6), with two readings where that has no finite positive
 * value: amax = 0 gives 1, and +inf (a producer output that overflowed bf16) is
 * clamped to the largest finite binary32 first.  The producer then reads it.
 * Nothing synchronises; the calls are ordered by the stream.
 *
 * Preconditions and status codes are those of the matching producer (shapes,
 * alignment, ld, frames), plus: amax not NULL and not overlapping an input.
 *
 * h3q_rmsnorm_adaln_amax also writes each row's rstd to row_rstd when it is not
 * NULL (fp32 [rows], 4-byte aligned, overlapping neither an input nor amax): the
 * pass forms the row statistics anyway, in the producer's canonical order, so
 * h3q_rmsnorm_adaln_nvfp4_from_rstd can then quantize without forming them again.
 */
int h3q_amax_bf16(const void *x, int64_t ld_x, int64_t rows, int64_t cols, float *amax,
                  void *stream);

int h3q_rmsnorm_adaln_amax(const void *x, int64_t ld_x, const void *gamma,
                           const void *mod_table, int64_t num_frames, const int32_t *row_frame,
                           int64_t rows_per_frame, float eps, int64_t rows, int64_t cols,
                           float *amax, float *row_rstd, void *stream);

/*
 * The RMSNorm + AdaLN producer with each row's rstd given: the second pass of a
 * dynamic scale, after h3q_rmsnorm_adaln_amax wrote row_rstd.  y and its NVFP4 are
 * those of h3q_rmsnorm_adaln_nvfp4 with rstd = row_rstd[r] in place of the row's
 * own statistics (so, with the abs-max pass's row_rstd, byte for byte the same
 * output); eps has no role.  Arguments as h3q_rmsnorm_adaln_nvfp4, plus:
 *
 *   row_rstd  fp32 [rows] on the device, 4-byte aligned, not NULL, overlapping no
 *             output.
 */
int h3q_rmsnorm_adaln_nvfp4_from_rstd(const void *x, int64_t ld_x, const void *gamma,
                                      const void *mod_table, int64_t num_frames,
                                      const int32_t *row_frame, int64_t rows_per_frame,
                                      const float *row_rstd, int64_t rows, int64_t cols,
                                      const float *global_scale, uint8_t *codes, uint8_t *scales,
                                      void *stream);

int h3q_swiglu_amax(const void *gate, int64_t ld_gate, const void *up, int64_t ld_up,
                    int64_t rows, int64_t cols, float *amax, void *stream);

int h3q_global_scale_from_amax(const float *amax, float *global_scale, void *stream);

/*
 * Dynamic quantize that needs no scratch from the caller and allocates nothing.
 * No page has a counterpart: it is this library's convenience form of the
 * dynamic scale above for the standalone quantize.  On the stream it runs an
 * abs-max pass over x whose CTAs write their partial maxima into a fixed
 * device array inside the library (a file-scope __device__ array of 4,096
 * floats, one per CUDA context, its address looked up in the current context
 * on every call: a lookup, not an allocation); then the quantize, launched as a
 * programmatic dependent of that pass, reduces them into the global scale
 * fl(2688 / max |x|) (0 -> 1, +inf clamped) in each of its CTAs and quantizes x
 * as h3q_quantize_nvfp4 does with that scale.  Outputs: codes, scales and the
 * global scale used (a device fp32 scalar written here).
 *
 * Limit: a shape whose abs-max pass needs more than 4,096 partial maxima (CTAs)
 * is rejected with H3Q_ERR_INVALID_ARGUMENT; on one GPU the pass launches at
 * most its occupancy times the SM count (1,216 CTAs on a 152-SM GB300).
 * Calls that overlap on one device (different streams, or threads without
 * ordering between them) share the array and race; order them on one stream.
 * Other preconditions and status codes as h3q_quantize_nvfp4.
 */
int h3q_quantize_nvfp4_dynamic(const void *x, int64_t ld_x, int64_t rows, int64_t cols,
                               float *global_scale, uint8_t *codes, uint8_t *scales,
                               void *stream);

/*
 * QKV epilogue: bias + per-head RMSNorm + partial rotate-half RoPE on q and k,
 * bias only on v (the step after the QKV projection GEMM; bf16 out, no
 * quantize).  FastVideo API page, qkv_epilogue: projected q/k/v [M, H*HD] bf16
 * with the bias not yet added -> roped q, k and biased v, each [M, H, HD];
 * cos/sin bf16 [M, ROT] (the eager path's cos.to(query.dtype)); an eps and no
 * norm weights.  FastVideo commit log (the q/k norm + partial RoPE kernel):
 * offsets are 64-bit, so M * H * HD may exceed 2^31.  Per row and head, with
 * x' = bf16(fl(x + b)) for each of the HD values:
 *   v:     out = x'
 *   q, k:  ss = the head's sum of squares of x' (eight fmaf partials per chunk
 *          of 8 values, the chunk total ((p0+p1)+(p2+p3))+((p4+p5)+(p6+p7)),
 *          a butterfly over the head's HD/8 chunk totals);
 *          rstd = fl(1 / fl(sqrt(fl(fl(ss / HD) + eps)))), n = bf16(fl(x' * rstd));
 *          out_i = bf16(fl(bf16(fl(n_i * cos_i)) + bf16(fl(r_i * sin_i)))) for
 *          i < ROT, r_i = -n_{i+ROT/2} (i < ROT/2) or n_{i-ROT/2} (rotate-half
 *          pairs), or with `interleaved` r_{2j} = -n_{2j+1}, r_{2j+1} = n_{2j}
 *          (FlashRT PR #142 page, the fused RMSNorm + RoPE kernel: interleaved
 *          RoPE on the [B, S, H, D] layout); out_i = n_i for i >= ROT.
 *
 *   q, k, v        bf16 [rows, heads * head_dim], row strides ld_q, ld_k, ld_v
 *                  (>= heads * head_dim, multiples of 16), 32-byte aligned.
 *   bias_q/k/v     bf16 [heads * head_dim], 32-byte aligned, not NULL.
 *   cos, sin       bf16 [rows, rot] contiguous, 16-byte aligned; NULL when rot = 0.
 *   rot            ROT, a multiple of 16 with 0 <= rot <= head_dim.
 *   interleaved    0: rotate-half pairs (i, i + ROT/2); 1: pairs (2j, 2j + 1).
 *   heads          H >= 1; head_dim HD in {64, 128, 256}; heads * head_dim <= 2^24.
 *   eps            finite, >= 0 (with eps = 0 an all-zero head gives NaN values, whose
 *                  bit patterns are unspecified).
 *   q_out, k_out, v_out  bf16 [rows, heads, head_dim] contiguous, 16-byte
 *                  aligned, caller-owned; they must not overlap an input or
 *                  each other.
 * rows = 0 returns H3Q_OK with no launch.  Status codes as the other calls.
 */
int h3q_qkv_epilogue(const void *q, int64_t ld_q, const void *k, int64_t ld_k, const void *v,
                     int64_t ld_v, const void *bias_q, const void *bias_k, const void *bias_v,
                     const void *cos, const void *sin, int64_t rot, int interleaved, int64_t rows,
                     int64_t heads, int64_t head_dim, float eps, void *q_out, void *k_out,
                     void *v_out, void *stream);

/*
 * The FFN-up projection as a block-scaled NVFP4 GEMM on the tensor cores, with
 * the SwiGLU and the NVFP4 quantize of its output in the epilogue.  (FastVideo
 * compare "fasth3-spark-exact-perf", minimax_h3_swiglu_gemm.cu:
 * launch_gemm_swiglu -- NVFP4 A and B, value/gate-paired weight columns, alpha
 * and the global scale as device pointers -- and h3_epilogue::Store -- value =
 * bf16(alpha * acc), gate = bf16(alpha * acc), SwiGLU, block quantize.)
 *
 *   acc[i][j] = sum over k of A[i][k] * B[j][k]        (fp32, tensor-core order)
 *   u = bf16(fl(alpha * acc[i][2j])),  g = bf16(fl(alpha * acc[i][2j + 1]))
 *   y[i][j] = bf16(fl(fl(g * sigma(g)) * u))           (as h3q_swiglu_nvfp4)
 * then y [m, n/2] is block-quantized with global_scale.  A element =
 * E2M1value(code) * E4M3value(scale); the products are exact and the sum is
 * accumulated in binary32 by the tensor cores in their own order (it
 * approximates the exact sum; everything after acc is bit-exact arithmetic).
 *
 *   a_codes   uint8 [m, k/2] contiguous: the activation's E2M1 codes (as the
 *             producers write them).  16-byte aligned.
 *   a_scales  uint8 [h3q_padded_rows(m), k/16] in the 128x4 layout (as the
 *             producers write them).  16-byte aligned.
 *   b_codes   uint8 [n, k/2] contiguous, b_scales uint8 [n, k/16] in the 128x4
 *             layout: the weight, row 2j the value and row 2j+1 the gate of
 *             output j.  16-byte aligned.
 *   m         rows of A, 0 <= m <= 2^31 - 128 (m = 0 is a no-op).
 *   k         a multiple of 256, at most 2^24.   n  a multiple of 256, at most 2^24.
 *   alpha     device fp32: the dequantization factor of the product (for
 *             operands quantized with global scales g_A and g_B,
 *             fl(1 / fl(g_A * g_B))).
 *   global_scale  device fp32 gsf of the output quantize.
 *   codes     out, [m, n/4].   scales  out, h3q_scale_bytes(m, n/2).
 *   y         optional out, bf16 [m, n/2] (NULL: not written).
 *   acc       optional out, fp32 [m, n]: the accumulator before alpha (NULL:
 *             not written; for checking).
 * Alignment: codes, scales, y and acc 16-byte aligned.  Outputs must not
 * overlap an input or each other.  Status codes as the other calls.  The
 * kernel keeps one CTA per SM with all 512 TMEM columns of it; its waits are
 * bounded (2 s): if one runs out the kernel stops early, the outputs are
 * unspecified, and h3q_kernel_error_flag reports it.
 */
int h3q_gemm_swiglu_nvfp4(const uint8_t *a_codes, const uint8_t *a_scales, int64_t m, int64_t k,
                          const uint8_t *b_codes, const uint8_t *b_scales, int64_t n,
                          const float *alpha, const float *global_scale, uint8_t *codes,
                          uint8_t *scales, void *y, float *acc, void *stream);

/*
 * *flag = 1 if a kernel launched since the last call had one of its bounded
 * waits run out, else 0; the flag is cleared.  The kernel that waits on
 * mbarriers (the GEMM of h3q_gemm_swiglu_nvfp4) bounds every wait (2 s) and then
 * stops early, leaving that call's outputs unspecified.  Synchronous: it waits
 * for the device.  Not on any page; a diagnostic of this library.
 */
int h3q_kernel_error_flag(int *flag);

/*
 * h3q_rmsnorm_adaln_nvfp4 on HOST buffers: x read from host memory, codes and
 * scales written to host memory, the copies inside the call.  The rows are cut
 * into chunks of chunk_rows rows (a multiple of 128); the producer runs on the
 * caller's stream on chunk i while a library stream copies chunk i+1 in and
 * another copies chunk i-1's codes and scales out (the scales of a 128-row tile
 * are one contiguous range, h3q_scale_offset_of_row_tile).  The outputs equal
 * h3q_rmsnorm_adaln_nvfp4's byte for byte.
 *
 *   x_host          bf16 [rows, cols], contiguous, in host memory (page-locked
 *                   for the copies to run asynchronously and overlap).
 *   codes_host      out, host uint8 [rows, cols/2], contiguous.
 *   scales_host     out, host uint8 [h3q_padded_rows(rows), cols/16], contiguous.
 *   gamma, mod_table, num_frames, row_frame, rows_per_frame, eps, global_scale:
 *                   as h3q_rmsnorm_adaln_nvfp4, in device memory (row_frame
 *                   int32 [rows] or NULL).
 *   workspace       device memory of at least h3q_host_workspace_bytes(chunk_rows,
 *                   cols, rows, row_frame == NULL) bytes, 256-byte aligned, owned
 *                   by the caller and not touched by other work until the stream
 *                   has passed this call.
 *   chunk_rows      a positive multiple of 128.
 * Ordering: the call runs after the work queued on `stream` before it, and work
 * queued on `stream` after it starts after its last copy back, so the host
 * outputs may be read once `stream` has been synchronised.  On its first call on
 * a device the library creates two non-blocking streams and a few events for
 * that device and keeps them; it allocates no memory.  Calls on one device are
 * enqueued one at a time (a lock), and stay asynchronous.  Status codes as the
 * other calls; a failure after the first copy was queued leaves the outputs
 * unspecified.  The streams and events belong to the CUDA context current at the
 * call (2 streams, 11 events per context, never destroyed: a context that the
 * caller destroys takes them with it).  At most 64 contexts over the process's
 * life can use this call; the 65th gets H3Q_ERR_CUDA (cudaErrorNotSupported).
 */
int h3q_rmsnorm_adaln_nvfp4_host(const void *x_host, int64_t rows, int64_t cols, const void *gamma,
                                 const void *mod_table, int64_t num_frames, const int32_t *row_frame,
                                 int64_t rows_per_frame, float eps, const float *global_scale,
                                 uint8_t *codes_host, uint8_t *scales_host, void *workspace,
                                 int64_t workspace_bytes, int64_t chunk_rows, void *stream);

/* Message for the calling thread's most recent failed call ("" if none). */
const char *h3q_last_error(void);

/* H3Q_ABI_VERSION of the loaded library. */
int h3q_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* H3Q_H */
