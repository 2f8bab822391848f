/*
 * h3attn -- packed varlen non-causal attention for the MiniMax-H3 DiT block,
 * with its fused q/k prologue, on GB300 (sm_103a).
 *
 * What is computed (per DiT block, per head):
 *   1. prologue on every q and k row: per-head RMSNorm with a gain, then the
 *      3D (t, h, w) rotary embedding on head dims 0..95 (dims 96..127 pass
 *      through);
 *   2. attention that is bidirectional inside each cu_seqlens document of the
 *      packed sequence and never crosses a document boundary.
 *
 * Pages defining it (page title, then section):
 *   [PR26]  vllm.cpp PR #26 "feat(minimax-h3): port the MiniMax-H3 omni-modal
 *           video+audio DiT" -- PR description (packed varlen NON-CAUSAL
 *           attention with the per-document contract of a cu_seqlens varlen
 *           flash-attention call, causal=false; the fp64 position grid gated
 *           bit-exact, i*step + start), "The device-resident forward (W2b)"
 *           (rotary = plain NeoX rotate_half with angles off the fp64 grid
 *           through a per-row cos/sin cache; q/k RMSNorm), the encoder text
 *           tower commit (per-head q/k RMSNorm);
 *   [SPARK] "h3-spark" model card, "What this config does" (Q RMSNorm, then
 *           rot96 RoPE, fused; byte-exact on default and non-default streams;
 *           step-invariant rope caches).
 *
 * Conventions for every call:
 *   - Tensors q, k, v, o are bf16, token-major "thd" packing: element
 *     (token s, head h, dim d) sits at base + s*row_stride + h*128 + d
 *     (strides in elements).  row_stride >= num_heads*128 lets q, k and v be
 *     read straight out of a fused-qkv GEMM output [S, 3*H*128].
 *   - All device pointers are caller-owned (the library never frees them)
 *     and must be 16-byte aligned; row strides must be multiples of 8
 *     elements.  Host pointers are caller-owned too.
 *   - All compute calls are asynchronous on the given CUDA stream
 *     (a cudaStream_t passed as void*; NULL = the legacy default stream) and
 *     may be issued on any stream.  The library allocates no device memory on
 *     the compute path; only h3attn_plan_create allocates, and
 *     h3attn_plan_destroy frees.
 *   - Functions never throw across the boundary.  Arguments are validated
 *     before anything is launched; on failure nothing is launched, the
 *     status says why, and h3attn_last_error() holds a message.
 *   - A plan is used from one host thread at a time, and the calls that use
 *     one plan must not overlap on the GPU: every forward issued with a plan
 *     writes its partial-result buffers (the pieces of a split last wave) and
 *     its device error word, so two forwards with the same plan running at
 *     once on two streams race on them.  Issue them on one stream, order the
 *     streams with events, or give each concurrent stream its own plan.
 */
#ifndef H3ATTN_H_
#define H3ATTN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  H3ATTN_OK = 0,
  H3ATTN_EINVAL = 1,        /* bad argument: null, misaligned, empty, out of range */
  H3ATTN_EUNSUPPORTED = 2,  /* valid but not built: head_dim != 128, rope_dims != 96, not sm_103 */
  H3ATTN_ENOMEM = 3,        /* device or host allocation failed (plan creation only) */
  H3ATTN_ECUDA = 4,         /* a CUDA runtime/driver call failed; message has the CUDA error */
  H3ATTN_ETIMEOUT = 5       /* a bounded device-side wait ran out (see h3attn_get_device_error) */
} h3attn_status;

/* Opaque plan: the packed layout of one request, built once and reused by
 * every block and step ([SPARK] step-invariant rope caches). */
typedef struct h3attn_plan* h3attn_plan_t;

/* A grid of n_t x n_h x n_w tokens, ordered t-major then h, w fastest.  The
 * position of token (i_t, i_h, i_w) on axis a is i_a*step[a] + start[a],
 * evaluated in fp64 as one rounded product followed by one rounded sum
 * ([PR26] PR description: numpy linspace(endpoint=False) order).  A 1D run
 * (audio) is n_h = n_w = 1 with step {1, 0, 0}. */
typedef struct {
  int32_t n_t, n_h, n_w;
  double start[3];
  double step[3];
} h3attn_span;

/* A document: its spans concatenated in order.  Documents are packed back to
 * back; cu_seqlens are the prefix sums of their lengths. */
typedef struct {
  const h3attn_span* spans;
  int32_t n_spans;
} h3attn_doc;

typedef struct {
  int32_t num_heads;   /* H >= 1 */
  int32_t head_dim;    /* must be 128 */
  int32_t rope_dims;   /* must be 96: 32 dims per axis (t, h, w), NeoX pairs j <-> j+48 */
  double rope_base;    /* > 1; per-axis frequencies base^(-2k/32), k = 0..15 */
} h3attn_plan_opts;

/* Builds the plan on the host -- cu_seqlens (int32 [n_docs+1]), the fp64
 * position grid [S,3], the fp32 cos/sin table [S,48] (angles in fp64) and the
 * attention work list -- and uploads it to the current device on cuda_stream
 * (the call synchronises that stream before returning).
 * Errors: EINVAL for null docs/out, n_docs < 1, a document with no tokens, a
 * span with a non-positive extent, non-finite start/step, S >= 2^31, H < 1;
 * EUNSUPPORTED for head_dim != 128, rope_dims != 96 or a device that is not
 * compute capability 10.3; ENOMEM / ECUDA from allocation or upload.
 * On success *out owns device memory until h3attn_plan_destroy. */
h3attn_status h3attn_plan_create(const h3attn_doc* docs, int32_t n_docs,
                                 const h3attn_plan_opts* opts, void* cuda_stream,
                                 h3attn_plan_t* out);

/* Frees the plan's device and host memory (synchronises the device first).
 * NULL is accepted and ignored. */
h3attn_status h3attn_plan_destroy(h3attn_plan_t plan);

/* Sizes of a plan; any output pointer may be NULL. */
h3attn_status h3attn_plan_info(h3attn_plan_t plan, int64_t* total_tokens, int32_t* n_docs,
                               int32_t* max_seqlen, int32_t* num_heads);

/* Host copies of the plan's layout, for checking it: cu_seqlens into
 * host_out[n_docs+1]; positions into host_out[S*3] (fp64, row-major [S,3],
 * bit-exact); the rotary table into host_out[S*48*2] as (cos, sin) pairs of
 * fp32, angle index a*16 + k for axis a in (t, h, w). */
h3attn_status h3attn_plan_copy_cu_seqlens(h3attn_plan_t plan, int32_t* host_out);
h3attn_status h3attn_plan_copy_positions(h3attn_plan_t plan, double* host_out);
h3attn_status h3attn_plan_copy_rope_table(h3attn_plan_t plan, float* host_out);

/* The q/k prologue ([SPARK] fused Q RMSNorm + rot96 RoPE; [PR26] W2b per-head
 * RMSNorm and NeoX rotate_half from the per-row cos/sin cache).  For every
 * token s, head h and tensor x in {q, k}:
 *     r    = 1 / sqrt(mean_d x_d^2 + eps)
 *     y_d  = x_d * r * gain[h*gain_head_stride + d]
 *     j < 48:  out_j    = y_j cos(th_j) - y_{j+48} sin(th_j)
 *              out_j+48 = y_{j+48} cos(th_j) + y_j sin(th_j)
 *     d >= 96: out_d    = y_d
 * with th from the plan's grid; fp32 arithmetic, one rounding to bf16.
 * q_in/k_in: bf16 [S,H,128] with in_row_stride; q_out/k_out: bf16 with
 * out_row_stride (in place is allowed when the pointers and strides are
 * equal; partial overlap is not).  gain_q/gain_k: fp32 device arrays, [128]
 * shared by all heads when gain_head_stride == 0, else [H, gain_head_stride].
 * q_in and q_out may both be NULL: then only k is processed (gain_q is
 * ignored), for use with h3attn_forward_fused_q, which applies the same
 * arithmetic to q itself.
 * Errors: EINVAL for null/misaligned pointers (or only one of q_in/q_out
 * NULL), strides < H*128 or not multiples of 8, eps < 0 or not finite,
 * partial overlap. */
h3attn_status h3attn_qk_prologue(h3attn_plan_t plan, const void* q_in, const void* k_in,
                                 int64_t in_row_stride, void* q_out, void* k_out,
                                 int64_t out_row_stride, const float* gain_q,
                                 const float* gain_k, int64_t gain_head_stride, float eps,
                                 void* cuda_stream);

/* Packed varlen non-causal attention ([PR26] PR description: per-document
 * bidirectional attention, exactly a cu_seqlens varlen flash-attention call
 * with causal=false).  For each head and each query token i of document
 * [a, b):
 *     s_ij = softmax_scale * <q_i, k_j>,   j in [a, b)
 *     o_i  = sum_j softmax_j(s_ij) v_j     (bf16 out, fp32 accumulation)
 *     lse[h*S + i] = ln sum_j exp(s_ij)    (only if lse_out != NULL)
 * q, k, v: bf16 [S,H,128] with qkv_row_stride (the prologue's outputs, or a
 * fused buffer); o: bf16 with o_row_stride, must not overlap q/k/v;
 * lse_out: fp32 [H, S] device array or NULL.  Tensor-core kernel: TMA tiles,
 * tcgen05 MMAs with TMEM accumulators, online softmax, a persistent grid over
 * the plan's work list that never visits a cross-document tile.
 * Errors: EINVAL for null/misaligned pointers, bad strides, o overlapping
 * q/k/v, softmax_scale not finite or <= 0. */
h3attn_status h3attn_forward(h3attn_plan_t plan, const void* q, const void* k, const void* v,
                             int64_t qkv_row_stride, void* o, int64_t o_row_stride,
                             float softmax_scale, float* lse_out, void* cuda_stream);

/* The same attention with the Q half of the prologue fused in ([SPARK] "What
 * this config does": Q RMSNorm + rot96 RoPE fused into one kernel).  q_raw
 * holds the raw queries (bf16 [S,H,128], qkv_row_stride); each query tile is
 * normalised with gain_q (layout as in h3attn_qk_prologue) and eps and
 * rotated with the plan's table in shared memory, with arithmetic identical
 * to h3attn_qk_prologue's (the q̂ values, and so o and lse, are bit-identical
 * to h3attn_qk_prologue followed by h3attn_forward).  q_raw is only read (it
 * may be the q part of a fused qkv buffer); k must already be k̂ (e.g.
 * h3attn_qk_prologue with q_in = q_out = NULL).  Other arguments and errors as
 * h3attn_forward, plus EINVAL for a NULL or misaligned gain_q, a bad
 * gain_head_stride, or eps < 0 or not finite. */
h3attn_status h3attn_forward_fused_q(h3attn_plan_t plan, const void* q_raw, const void* k, const void* v,
                                     int64_t qkv_row_stride, void* o, int64_t o_row_stride,
                                     const float* gain_q, int64_t gain_head_stride, float eps,
                                     float softmax_scale, float* lse_out, void* cuda_stream);

/* FP8 (e4m3) quantisation for h3attn_forward_fp8 ([PR26], [SPARK] "What this
 * config does": a SageAttention2++-style low-precision attention; the pages
 * give no scheme, this one is the plainest that runs both products on FP8
 * tensor cores).  From q-hat, k-hat, v (bf16 [S,H,128], qkv_row_stride):
 *   q8  [S,H,128] e4m3, scale sq [H,S] per (token, head) row;
 *   k8  [S,H,128] e4m3, scale sk [H,S] per (head, 128-key tile of a document,
 *       i.e. tokens [a + 128j, min(a + 128j + 128, b)) of document [a, b)),
 *       stored for every token of the tile;
 *   v8t [H,128,V] e4m3, channel-major with keys contiguous; document d's
 *       keys start at key sum_{d'<d} ceil(L_d'/16)*16 (a 16-key boundary, the
 *       gaps zero), V = that sum over all documents (h3attn_plan_fp8_v_keys);
 *       scale sv [H,128] per (head, channel) over all tokens.
 * scale = amax / 448 and r = 448 / amax (both 1 for an all-zero row, tile or
 * channel), each one correctly rounded fp32 division; code = e4m3(x * r), one
 * correctly rounded fp32 product, then round to nearest even with saturation
 * to +-448.  All outputs are device buffers owned by the
 * caller, 16-byte aligned, not overlapping the inputs or each other.
 * Errors: EINVAL for null/misaligned pointers, a bad stride, overlaps. */
h3attn_status h3attn_fp8_quantize(h3attn_plan_t plan, const void* q_hat, const void* k_hat, const void* v,
                                  int64_t qkv_row_stride, void* q8, void* k8, void* v8t, float* sq, float* sk,
                                  float* sv, void* cuda_stream);

/* The q/k prologue and the FP8 quantisation in one call, for the FP8 step
 * ([SPARK] "What this config does": the fused Q RMSNorm + rot96 kernel also
 * quantises Q for the low-precision attention; here q and k, to e4m3):
 * the same codes and scales as h3attn_qk_prologue (gains and eps as there)
 * followed by h3attn_fp8_quantize on its bf16 outputs and on v, without
 * q-hat and k-hat ever being written.  q_in, k_in, v: bf16 [S,H,128] with
 * qkv_row_stride (a fused-qkv buffer works); q8, k8, v8t, sq, sk, sv: as
 * h3attn_fp8_quantize writes them.  One kernel normalises, rotates, rounds
 * to bf16 and quantises q per row and k per document key tile (one block per
 * key tile and head, the tile's k rows held on chip until its amax is
 * known); v takes the two passes of h3attn_fp8_quantize.  All buffers are
 * caller-owned device memory, 16-byte aligned; no output may overlap an input
 * or another output.  Errors: EINVAL for null/misaligned pointers, a bad
 * stride, gain_head_stride or eps, and overlaps. */
h3attn_status h3attn_qk_prologue_fp8(h3attn_plan_t plan, const void* q_in, const void* k_in, const void* v,
                                     int64_t qkv_row_stride, const float* gain_q, const float* gain_k,
                                     int64_t gain_head_stride, float eps, void* q8, void* k8, void* v8t, float* sq,
                                     float* sk, float* sv, void* cuda_stream);

/* Kernels one h3attn_forward call launches with this plan: 1, or 2 when the
 * last round of work units is split along the keys and merged. */
h3attn_status h3attn_plan_forward_kernels(h3attn_plan_t plan, int32_t* n_kernels);

/* The forward's work list for a packed layout, built on the host alone (no
 * device and no CUDA call is needed): the list h3attn_plan_create builds for
 * n_pairs concurrent CTA pairs (a GB300 runs 76).  It schedules the
 * per-document attention of h3attn_forward ([PR26] PR description: the
 * cu_seqlens varlen contract) so that only tiles inside a document are ever
 * visited, and places the work longest-processing-time first.
 *
 * A unit is up to 512 query rows of one head inside one document [b, e), over
 * that document's 128-key tiles [tile_lo, tile_hi) (counted from b).  Units
 * are listed longest document first, then head, then query rows; each is
 * placed on the CTA pair with the least estimated load so far (ties to the
 * lower pair), a segment's estimate being its key tiles plus one.  The units
 * of the last partial round (U mod n_pairs of them, U the unit count) are
 * split along their key tiles into about n_pairs pieces, which are placed the
 * same way after the whole units; their partial results are merged by the
 * forward.
 *
 * Outputs (host memory owned by the caller; pass units = NULL to get the
 * sizes first):
 *   *n_units       segments in the list;
 *   *n_pairs_used  pairs with work (pairs 0 .. *n_pairs_used - 1; the others
 *                  get none);
 *   units          [*n_units][8] int32, grouped by pair: first query row, b,
 *                  e, head, tile_lo, tile_hi, partial slot (-1: the segment
 *                  writes the output itself), the document's first key in the
 *                  FP8 transposed V;
 *   unit_off       [*n_pairs_used + 1] int32: pair p runs units
 *                  [unit_off[p], unit_off[p + 1]) in that order.
 * units_cap is the capacity of units in segments.  Errors: EINVAL for a NULL
 * cu_seqlens or output count, n_docs < 1, num_heads < 1, n_pairs outside
 * [1, 1024], cu_seqlens[0] != 0, an empty document, or units_cap too small. */
h3attn_status h3attn_work_list_host(const int32_t* cu_seqlens, int32_t n_docs, int32_t num_heads,
                                    int32_t n_pairs, int32_t* units, int64_t units_cap, int32_t* unit_off,
                                    int64_t* n_units, int32_t* n_pairs_used);

/* Keys per row of the FP8 transposed V of this plan (see h3attn_fp8_quantize). */
h3attn_status h3attn_plan_fp8_v_keys(h3attn_plan_t plan, int64_t* v_keys);

/* The FP8 variant of h3attn_forward on h3attn_fp8_quantize's outputs: for
 * each head and query i of document [a, b),
 *     s_ij = softmax_scale * sq_i * sk_j * <q8_i, k8_j>   (fp32 accumulation)
 *     o_i  = sum_j P_ij (v8_j * sv) / sum_j p_ij
 * where p_ij = exp(s_ij - m) with the kernel's reference max m (at most 2^8
 * below the row max, so p <= 2^8) and P_ij is p_ij rounded to e4m3 for the
 * FP8 PV product; lse as h3attn_forward.  The result approximates exact
 * attention on the dequantised inputs within 2^-4 sum_j w_ij |v~_jc| +
 * 2^-10 sum_j |v~_jc| (+ bf16 rounding of o), w the exact softmax weights.
 * q8, k8: [S,H,128] e4m3; v8t, sq, sk, sv as h3attn_fp8_quantize writes them;
 * o: bf16 with o_row_stride, must not overlap the inputs; lse_out as
 * h3attn_forward.  Errors: EINVAL for null/misaligned pointers, a bad stride,
 * o overlapping an input, softmax_scale not finite or <= 0. */
h3attn_status h3attn_forward_fp8(h3attn_plan_t plan, const void* q8, const void* k8, const void* v8t,
                                 const float* sq, const float* sk, const float* sv, void* o, int64_t o_row_stride,
                                 float softmax_scale, float* lse_out, void* cuda_stream);

/* Allocation-free forward.  The pages have no counterpart: this entry point
 * exists for callers that may not allocate device memory -- code whose device
 * memory is owned by a host framework's pool or arena (an engine plugin, a
 * serving runtime that reserves all memory at start-up), or a latency-bound
 * loop where a cudaMalloc would synchronise the device.  h3attn_plan_create
 * allocates, so such callers cannot use h3attn_forward.
 * Same computation and kernel as h3attn_forward, without a plan: cu_seqlens
 * is a HOST int32 array [n_docs+1] (cu_seqlens[0] = 0, strictly increasing);
 * the work list is built on the host and, with the kernel's error word, kept
 * in one static device array of 1 MiB + 4 KiB + 16 B that every GPU loading the
 * library holds until the process exits.  At most 32768 work units (a unit is
 * up to 512 query rows of one head in one document, so sum over documents of
 * ceil(len/512) * num_heads <= 32768); larger layouts get EINVAL with a
 * message.  q, k, v, o, lse_out and their rules are those of h3attn_forward,
 * except that o must not share any byte range with q, k or v.
 * Calls no cudaMalloc/cudaFree or other allocating routine.  The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current.  All calls share the array and it keeps the last call's contents: the work list
 * is rewritten and the error word cleared on every call.  Calls from several
 * host threads on one stream are safe: each call enqueues its copy of the
 * work list and its kernel under one lock, so they run in that order.  Calls
 * that overlap on the GPU (on two streams at once) race on the array.  A
 * bounded-wait timeout inside the kernel invalidates the output but is not
 * reported here (there is no plan to hold it); use h3attn_forward where that
 * matters.  Unlike h3attn_forward, this path never splits the last round of
 * work units along the keys (that needs partial buffers), so its output can
 * differ from h3attn_forward's in the last bits while both stay within the
 * same tolerance of exact attention. */
h3attn_status h3attn_forward_noalloc(const int32_t* cu_seqlens, int32_t n_docs, int32_t num_heads,
                                     const void* q, const void* k, const void* v,
                                     int64_t qkv_row_stride, void* o, int64_t o_row_stride,
                                     float softmax_scale, float* lse_out, void* cuda_stream);

/* Synchronises cuda_stream, then reads and clears the plan's device error
 * word.  Returns OK, or ETIMEOUT if a kernel's bounded wait ran out since the
 * last call (the kernel then stopped early and its outputs are invalid), or
 * ECUDA if the stream reports an error. */
h3attn_status h3attn_get_device_error(h3attn_plan_t plan, void* cuda_stream);

/* Launches one CTA that waits on a shared-memory barrier nothing arrives on,
 * through the same bounded wait the kernels use, with the given limit in
 * nanoseconds (1e3 .. 1e10).  The kernel records the timeout and returns; the
 * call synchronises and returns ETIMEOUT when the wait ran out as designed
 * (OK would mean the bound is broken).  Exercises failure detection without
 * faulting or hanging the GPU. */
h3attn_status h3attn_selftest_bounded_wait(uint64_t timeout_ns, void* cuda_stream);

/* Message for the last failing call on this host thread ("" if none). */
const char* h3attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* H3ATTN_H_ */
