/*
 * cp_attn.h -- C ABI of the GB300 (sm_103a) context-parallel causal
 * ring-attention step.
 *
 * What it computes. One ring-attention step is block-causal flash attention
 * of a query chunk against one visiting KV chunk, followed by the
 * log-sum-exp merge of partial outputs ("Context Parallelism for Scalable
 * Million-Token Inference", section "Ring Attention Algorithms"; "Announcing
 * Long-Context Training on TPUs with MaxText Context Parallelism", sections
 * "Context Parallelism in MaxText" (P2P) and "Built on a fast attention
 * kernel"). The ring of R context-parallel ranks is emulated on one GPU:
 * rank r owns rows [r*n, (r+1)*n) of each tensor ("rank-major" order), and
 * a ring step is one launch that computes every pair (q_owner, kv_owner)
 * active at that step.
 *
 * Conventions (all entry points):
 *  - Tensors are caller-owned DEVICE memory unless stated otherwise. The
 *    library never allocates on a compute call; plans allocate their own
 *    device tables (and a buffer for an fp16 copy of V) at creation time.
 *  - Q, K, V, O, dO are bf16, row-major [tokens, heads, head_dim] with
 *    head_dim contiguous, in rank-major token order (see
 *    cp_attn_layout_apply). Base addresses must be 16-byte aligned.
 *  - LSE and delta are fp32 [heads, tokens] (natural log, softmax scale
 *    applied). Gradients and partial outputs are [tokens, heads, head_dim],
 *    fp32 unless the plan asks for bf16 (cp_attn_plan_desc.grad_dtype,
 *    partial_dtype).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Compute calls are asynchronous on that stream; argument errors
 *    are detected on the host before anything is enqueued.
 *  - Every call returns a cp_attn_status; on failure cp_attn_last_error()
 *    returns a thread-local message. Device-side failures (a pipeline wait
 *    that exceeded its time limit) are recorded in the plan's device status
 *    word and reported by cp_attn_sync_status().
 *  - Supported: head_dim 64 or 128; n_q_heads a multiple of n_kv_heads;
 *    every chunk a multiple of 128 tokens.
 */
#ifndef CP_ATTN_H
#define CP_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cp_attn_status {
  CP_ATTN_OK = 0,
  CP_ATTN_ERR_INVALID_ARG = 1, /* null pointer, misaligned pointer, bad enum */
  CP_ATTN_ERR_SHAPE = 2,       /* sizes that violate the plan's rules */
  CP_ATTN_ERR_UNSUPPORTED = 3, /* valid but not implemented (e.g. head_dim 96) */
  CP_ATTN_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  CP_ATTN_ERR_OOM = 5,         /* plan table allocation failed */
  CP_ATTN_ERR_TIMEOUT = 6,     /* a kernel pipeline wait ran out of time */
  CP_ATTN_ERR_RANGE = 7        /* an input value outside the supported range */
} cp_attn_status;

/* Chunk layout ("Load Balancing in CP"): ZIGZAG cuts the sequence into 2R
 * chunks and gives rank r chunks r and 2R-1-r (in that order); CONTIGUOUS
 * gives rank r the r-th of R equal chunks (no compute balancing).
 * USP ("A2A + P2P (USP)" in the MaxText post): D = a2a * R devices each hold
 * their zigzag pair of 2D chunks; an all-to-all inside each group of a2a
 * consecutive devices pools the group's tokens (and splits its heads, see
 * cp_attn_head_a2a), so ring rank r holds the chunks of devices
 * r*a2a .. r*a2a + a2a - 1, kept in ascending position order, and the ring
 * has R steps of a2a-times longer chunks. On one GPU the token half of that
 * all-to-all is part of the plan's layout permutation (cp_attn_layout_apply
 * goes straight from natural order to the pooled order). With R = 1 this is pure Ulysses ("All-to-All
 * (Ulysses)"): one rank holds the whole sequence for its heads. A USP plan
 * describes the ring of one head group (n_q_heads and n_kv_heads are the
 * heads each device keeps after the all-to-all). */
typedef enum cp_attn_layout {
  CP_ATTN_LAYOUT_CONTIGUOUS = 0,
  CP_ATTN_LAYOUT_ZIGZAG = 1,
  CP_ATTN_LAYOUT_USP = 2
} cp_attn_layout;

/* Ring ordering ("Ring Attention Algorithms"): PASS_KV keeps Q on its rank
 * and moves KV (at step t rank r holds the KV of rank (r-t) mod R);
 * PASS_Q keeps KV and moves Q (at step t rank r holds the Q of rank
 * (r-t) mod R), then returns partial outputs to their owners and merges.
 * VARIANT_AUTO (plan descriptors only) picks one of the two at plan time
 * with cp_attn_select_variant; cp_attn_plan_info reports the choice. */
typedef enum cp_attn_variant {
  CP_ATTN_PASS_KV = 0,
  CP_ATTN_PASS_Q = 1,
  CP_ATTN_VARIANT_AUTO = 2
} cp_attn_variant;

/* Epilogue of cp_attn_step_fwd.
 * WRITE_PARTIAL: the partial (O_t, LSE_t) of pair (q_owner, kv_owner) is
 *   written to slot kv_owner: element kv_owner*T_q*Hq*d of o_part (fp32, or
 *   bf16 when the plan's partial_dtype is BF16) and lse_part +
 *   kv_owner*Hq*T_q (fp32), at the q_owner's rows. Rows that see no key in
 *   this step get O = 0, LSE = -inf. (Storing by kv_owner is the
 *   permutation back to order that Pass Q needs before its merge.)
 * ACCUMULATE: the running merge "as it goes" of the P2P ring. o_part is an
 *   fp32 accumulator [T_q, Hq, d] and lse_part an fp32 [Hq, T_q]
 *   accumulator; step 0 initialises them, later steps merge into them. */
typedef enum cp_attn_merge_mode {
  CP_ATTN_WRITE_PARTIAL = 0,
  CP_ATTN_ACCUMULATE = 1
} cp_attn_merge_mode;

typedef enum cp_attn_op {
  CP_ATTN_OP_FORWARD = 0,
  CP_ATTN_OP_BACKWARD = 1
} cp_attn_op;

typedef enum cp_attn_tensor_kind {
  CP_ATTN_TENSOR_Q = 0,  /* query-side tensors: Q, O, dO, dQ (T_q rows) */
  CP_ATTN_TENSOR_KV = 1  /* key-side tensors: K, V, dK, dV (T_kv rows) */
} cp_attn_tensor_kind;

typedef enum cp_attn_direction {
  CP_ATTN_TO_RANK_MAJOR = 0, /* natural token order -> rank-major order */
  CP_ATTN_TO_NATURAL = 1     /* rank-major order -> natural token order */
} cp_attn_direction;

typedef struct cp_attn_plan_s* cp_attn_plan_t;

/* Element type of the partial outputs and of the gradients a plan hands out. */
typedef enum cp_attn_dtype {
  CP_ATTN_F32 = 0,
  CP_ATTN_BF16 = 1
} cp_attn_dtype;

/* Full description of a plan. Zero-initialise and set the fields. */
typedef struct cp_attn_plan_desc {
  int64_t seq_len;        /* new (query) tokens N, > 0 */
  int64_t kv_prefix_len;  /* cached tokens P before them (partial prefill;
                             "Attention Compute Patterns in Multi-Turn
                             Chat"); 0 for full prefill */
  int cp;                 /* ring size R >= 1 */
  int n_q_heads;          /* Hq */
  int n_kv_heads;         /* Hkv; Hq % Hkv == 0; query head h uses KV head
                             h / (Hq/Hkv) */
  int head_dim;           /* d: 64 or 128 */
  cp_attn_layout layout;
  cp_attn_variant variant;
  const int32_t* cu_seqlens; /* HOST pointer, n_docs+1 entries, or NULL for
                                one document. Offsets of packed documents in
                                natural positions 0..P+N: cu[0] = 0, strictly
                                increasing, cu[n_docs] = P + N. A key is
                                visible iff it is in the query's document
                                and not after it. Copied by the plan. */
  int n_docs;
  float softmax_scale;    /* 0 selects 1/sqrt(head_dim) */
  int64_t window;         /* sliding window W in tokens, 0 for none: a key k
                             is then visible to query q only if q - k < W
                             (on top of the document and causal rules). The
                             window layers of models that "mix sliding-window
                             and global layers" ("Announcing Long-Context
                             Training on TPUs with MaxText Context
                             Parallelism", section "What's next"). */
  int a2a;                /* USP layout: all-to-all group size (devices per
                             ring rank), >= 1; ignored (treated as 1) by the
                             other layouts */
  cp_attn_dtype partial_dtype; /* O partials written by WRITE_PARTIAL steps
                             (cp_attn_step_fwd's o_part) and kept by
                             cp_attn_forward for Pass Q: F32 (default) or
                             BF16, which halves the R partial slots of a
                             Pass-Q forward ("bf16 partials" for the
                             memory of the 405B-shaped Pass-Q prefill). The
                             LSE partials and the ACCUMULATE running output
                             stay fp32. */
  cp_attn_dtype grad_dtype; /* dq, dk, dv of cp_attn_backward: F32 (default)
                             or BF16, accumulated in fp32 in the workspace
                             and rounded to nearest even once at the end.
                             The step-level cp_attn_step_bwd always adds to
                             fp32 accumulators. */
  int batch;              /* B >= 1 independent sequences of kv_prefix_len +
                             seq_len tokens each (0 means 1). Each sequence is
                             sharded over the ring as described for the
                             layout; rank r holds its part of sequence 0, then
                             of sequence 1, ... Natural order is sequence-
                             major: q/dout [B*seq_len, Hq, d], k/v
                             [B*(kv_prefix_len+seq_len), Hkv, d]. Positions
                             live in one space where sequence b starts at
                             b*(kv_prefix_len+seq_len); cu_seqlens, when
                             given, covers all B*(kv_prefix_len+seq_len)
                             positions and must contain every sequence
                             start (NULL: one document per sequence). */
} cp_attn_plan_desc;

/* Build a plan: per-rank positions (zigzag or contiguous; "Context
 * Parallelism for Scalable Million-Token Inference", "Load Balancing in CP"),
 * the per-step (q_owner, kv_owner) schedule (same page, "Ring Attention
 * Algorithms"), the 128x128 block classes (fully masked blocks skipped,
 * packed sequences without padding: "Announcing Long-Context Training on
 * TPUs with MaxText Context Parallelism", "Built on a fast attention
 * kernel") and the per-step work lists, uploaded to the current CUDA device
 * if there is one (a plan made without a device serves the host-side
 * queries only). On the device the plan also holds a buffer for an fp16 copy
 * of V (T_kv * Hkv * head_dim * 2 bytes; see cp_attn_step_fwd); ERR_OOM if
 * it cannot be allocated.
 * Chunk rule: zigzag needs N and P to be multiples of 256*R; USP multiples
 * of 256*R*a2a; contiguous multiples of 128*R. Returns ERR_SHAPE otherwise. On success *out
 * owns host and device tables until cp_attn_plan_destroy. */
cp_attn_status cp_attn_plan(cp_attn_plan_t* out, int64_t seq_len, int cp,
                            int n_q_heads, int n_kv_heads, int head_dim,
                            cp_attn_layout layout, cp_attn_variant variant,
                            const int32_t* cu_seqlens, int n_docs);
cp_attn_status cp_attn_plan_ex(cp_attn_plan_t* out, const cp_attn_plan_desc* desc);

/* Pass KV or Pass Q for a prefill of n_new tokens after n_cached cached
 * ones ("Ring Attention Algorithms": Pass KV suits full prefill and partial
 * prefill with a low to medium KV-cache hit rate, Pass Q a high hit rate or
 * decode). The rule compares the per-hop ring messages: Pass Q moves the new
 * tokens' Q (n_new*Hq*d elements), Pass KV the K and V of all tokens
 * (2*(n_new+n_cached)*Hkv*d). PASS_Q iff the first is strictly smaller,
 * i.e. n_new/(n_new+n_cached) < 2*Hkv/Hq. (One page places the crossover at
 * a ~10% cache *miss* rate with the opposite direction; this library follows
 * the message-size argument and the qualitative statements, which agree.)
 * ERR_INVALID_ARG for n_new <= 0, n_cached < 0, non-positive head counts or
 * a NULL out. */
cp_attn_status cp_attn_select_variant(int64_t n_new, int64_t n_cached, int n_q_heads,
                                      int n_kv_heads, cp_attn_variant* out);
void cp_attn_plan_destroy(cp_attn_plan_t plan);

/* Sizes of a plan, written to info[0..n-1] (n <= 16):
 * 0 T_q (= R*n_q), 1 T_kv (= R*n_kv), 2 n_q (query rows per rank),
 * 3 n_kv (KV rows per rank), 4 R, 5 Hq, 6 Hkv, 7 d, 8 q tiles per rank,
 * 9 kv tiles per rank, 10 n_docs, 11 has device tables (0/1),
 * 12 ring ordering (cp_attn_variant, AUTO resolved), 13 window,
 * 14 a2a (1 unless USP), 15 batch. */
cp_attn_status cp_attn_plan_info(cp_attn_plan_t plan, int64_t* info, int n);

/* Host queries (bit-exact plan artefacts; no device needed): the layout of
 * "Load Balancing in CP" and the ring order of "Ring Attention Algorithms"
 * ("Context Parallelism for Scalable Million-Token Inference").
 * positions: global positions of rank `rank`'s query (kind Q, n_q values) or
 *   KV (kind KV, n_kv values) tokens, in local order, into a host int32 array.
 * schedule: out[(t*R + r)*2 + {0,1}] = (q_owner, kv_owner) of rank r at
 *   step t, for the plan's variant.
 * block_mask: out[((a*R + b)*nqt + i)*nkt + j] = class of q tile i of rank a
 *   against kv tile j of rank b: 0 EMPTY, 1 PARTIAL, 2 FULL.
 * visible_pairs: number of visible (query, key) pairs per query head at
 *   step `step` (or over the whole ring when step == -1). */
cp_attn_status cp_attn_plan_positions(cp_attn_plan_t plan, cp_attn_tensor_kind kind,
                                      int rank, int32_t* out);
cp_attn_status cp_attn_plan_schedule(cp_attn_plan_t plan, int32_t* out);
cp_attn_status cp_attn_plan_block_mask(cp_attn_plan_t plan, uint8_t* out);
cp_attn_status cp_attn_plan_visible_pairs(cp_attn_plan_t plan, int step, int64_t* out);

/* The compacted work list that step `step` of the forward (backward = 0) or
 * backward (backward = 1) kernel consumes (host query; block skipping of
 * "Built on a fast attention kernel" in "Announcing Long-Context Training on
 * TPUs with MaxText Context Parallelism"). Forward: one item per (q_owner,
 * q tile) of the step's pairs, with the run [lo, hi) of its non-empty kv
 * tiles of kv_owner (lo = hi = 0 when there is none). Backward: one item per
 * (kv_owner, kv tile) with a non-empty run [lo, hi) of q tiles of q_owner.
 * Items are generated pair by pair in rank order, tile by tile, then sorted
 * by run length, longest first (stable), so the heaviest tiles start in the
 * first wave. out (host, may be NULL to query the count) receives 6 int32 per
 * item: q_owner, kv_owner, tile, lo, hi, n_full (the run's FULL tiles);
 * *n_items the number of items. ERR_INVALID_ARG for a bad plan, step or
 * pointer. */
cp_attn_status cp_attn_plan_work_list(cp_attn_plan_t plan, int step, int backward, int32_t* out,
                                      int64_t* n_items);

/* Device workspace, in bytes, for cp_attn_forward (op FORWARD: the fp32
 * running output for Pass KV, or R partial slots for Pass Q, fp32 or bf16 by
 * the plan's partial_dtype, then R fp32 LSE slots) or cp_attn_backward (op
 * BACKWARD: the fp32 delta rows, then the fp16 operand copies of
 * cp_attn_half_ops_size, then, when the plan's grad_dtype is BF16, the fp32
 * accumulators of dq, dk and dv). */
cp_attn_status cp_attn_workspace_size(cp_attn_plan_t plan, cp_attn_op op, size_t* bytes);

/* One forward ring step (kernel K1): the attention kernel called once per
 * ring step on the local queries and the visiting KV chunk ("Announcing
 * Long-Context Training on TPUs with MaxText Context Parallelism", "Built on
 * a fast attention kernel"). For every pair (q_owner, kv_owner) of
 * step `step` and every query head: S = scale*Q K^T on the visible 128x128
 * tiles only (fully masked tiles are skipped, partial ones masked), online
 * softmax, O = P V, then the epilogue of `mode` (see cp_attn_merge_mode).
 * q: [T_q, Hq, d] bf16; k, v: [T_kv, Hkv, d] bf16.
 * o_final: optional bf16 [T_q, Hq, d]; when non-NULL in ACCUMULATE mode the
 *   merged result is also written there in bf16 (use on the last step).
 * Precision: S = Q K^T runs on the bf16 inputs; O += P V runs on fp16
 * operands, so P keeps 11 significant bits (bf16 keeps 8). Step 0 copies v
 * to fp16 into the plan's buffer and every step of the ring reads that copy:
 * run step 0 of a ring first, with the v of the ring, as the ring order
 * does (a later step called without it reads whatever the buffer holds), and
 * do not run two forward rings of one plan at the same time. Every bf16 value
 * of magnitude in [2^-14, 65504] converts exactly; smaller ones become fp16
 * subnormals (off by at most 2^-25); a finite value above 65504 sets
 * CP_ATTN_ERR_RANGE in the plan's status word.
 * ERR_INVALID_ARG for null/misaligned pointers or a step outside [0, R). */
cp_attn_status cp_attn_step_fwd(cp_attn_plan_t plan, int step,
                                const void* q, const void* k, const void* v,
                                void* o_part, float* lse_part,
                                cp_attn_merge_mode mode, void* o_final,
                                void* stream);

/* Chained ring steps (programmatic dependent launch). With enable = 1,
 * cp_attn_step_fwd, cp_attn_step_bwd and cp_attn_step_bwd_half launch every
 * step >= 1 so that it
 * may start on SMs left idle while the kernel before it on the stream drains;
 * the step waits for that kernel to finish before it reads or writes the
 * running output and LSE (forward, ACCUMULATE) or dK and dV (backward). Its
 * other inputs are read before that wait, so the caller promises that the
 * kernel launched just before step t >= 1 on the same stream is an earlier
 * step of the same ring on the same buffers, and that nothing written
 * between them is read by the step. cp_attn_forward and cp_attn_backward
 * always chain their own steps. enable = 0 (the default) launches every step
 * normally. The pages' ring runs one kernel per step on each rank; chaining
 * only lets consecutive steps of the emulated ring overlap at their edges.
 * Affects the head_dim 128 kernels. ERR_INVALID_ARG for a NULL plan or
 * enable outside {0, 1}. */
cp_attn_status cp_attn_plan_set_chaining(cp_attn_plan_t plan, int enable);

/* ---------------------------------------------------------------- FP8
 * The pages' benchmark model (Llama 3 405B) is quantized to FP8 throughout
 * ("Experimental Setup & Results", Model and Quantization). The format is
 * E4M3 (OCP 8-bit floating point: bias 7, three mantissa bits, largest
 * finite 448, no infinities) with one scale per tensor: with amax = max|x|,
 * x is stored as RN-even(fp32(x) * fp32(448/amax)) clamped to +-448 and
 * stands for code * fp32(amax/448) (scale 1 for an all-zero tensor). The
 * attention computed is the same as the bf16 path's, on those values.
 *
 * cp_attn_fp8_absmax: *amax (device fp32) = max |x| over n bf16 values
 *   (device, 16-byte aligned, n a multiple of 8). Overwrites *amax; NaNs
 *   are ignored.
 * cp_attn_fp8_quantize: x bf16 [rows][heads][head_dim] (device) -> out E4M3
 *   (device, 16-byte aligned), in the same layout (transpose = 0) or as
 *   [heads][head_dim][rows] (transpose = 1, rows % 64 == 0: the V^T layout
 *   the FP8 step reads), using the *amax of a preceding cp_attn_fp8_absmax;
 *   *scale (device, may be NULL) receives the descale factor amax/448.
 *   head_dim 64 or 128. ERR_SHAPE / ERR_INVALID_ARG on bad sizes, pointers
 *   or alignment.
 * cp_attn_step_fwd_fp8: cp_attn_step_fwd with E4M3 inputs, head_dim 128:
 *   q8 [T_q][Hq][128], k8 [T_kv][Hkv][128], vt8 the V^T layout
 *   [Hkv][128][T_kv], all in the plan's rank-major token order (apply
 *   cp_attn_layout_apply to the bf16 tensors before quantizing); scales a
 *   device array of three floats, the descale factors of q, k and v
 *   (16-byte aligned). P is rounded to E4M3 (after scaling by 2^4) for the
 *   P V product; the row sums, the LSE and all accumulation stay fp32.
 *   Outputs, modes and errors as cp_attn_step_fwd; ERR_UNSUPPORTED for
 *   head_dim != 128.
 * cp_attn_forward_fp8: cp_attn_forward over those inputs (same workspace).
 *   The plan's chaining flag (cp_attn_plan_set_chaining) applies to
 *   cp_attn_step_fwd_fp8 as to cp_attn_step_fwd. */
cp_attn_status cp_attn_fp8_absmax(const void* x, int64_t n, float* amax, void* stream);
cp_attn_status cp_attn_fp8_quantize(const void* x, int64_t rows, int heads, int head_dim,
                                    const float* amax, int transpose, void* out, float* scale,
                                    void* stream);
cp_attn_status cp_attn_step_fwd_fp8(cp_attn_plan_t plan, int step, const void* q8,
                                    const void* k8, const void* vt8, const float* scales,
                                    void* o_part, float* lse_part, cp_attn_merge_mode mode,
                                    void* o_final, void* stream);
cp_attn_status cp_attn_forward_fp8(cp_attn_plan_t plan, const void* q8, const void* k8,
                                   const void* vt8, const float* scales, void* o, float* lse,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of the fp16 operand copies used by the backward step: exact IEEE
 * fp16 copies of q, k, v and dout, in that order, each starting on a
 * 256-byte boundary. The backward MMAs run on fp16 operands so that the
 * probabilities P and dS they multiply keep 11 significant bits (bf16 keeps
 * 8). Domain of the copies: a bf16 value of magnitude in [2^-14, 65504]
 * converts exactly; a smaller one becomes an fp16 subnormal, off by at most
 * 2^-25 in absolute terms (values below 2^-25 become 0); a finite value
 * above 65504 is reported as CP_ATTN_ERR_RANGE. The absolute error of the
 * small values stays far below the gradients' 1e-2 tolerance (a score
 * moves by at most scale * 2^-25 * sum|other operand|). */
cp_attn_status cp_attn_half_ops_size(cp_attn_plan_t plan, size_t* bytes);

/* Backward preprocess (kernel K3; the per-step backward of "Built on a fast
 * attention kernel" needs the rows' delta): delta[h][t] = sum_d dO[t,h,:]*O[t,h,:]
 * in fp32, taking O from o_f32 (fp32 [T_q,Hq,d], e.g. the fp32 output that
 * cp_attn_forward leaves at the start of its workspace) when it is not NULL,
 * else from the bf16 o; zeroes the fp32 gradient accumulators dq
 * [T_q,Hq,d], dk and dv [T_kv,Hkv,d] (any of the three may be NULL to skip);
 * and, when half_ops is not NULL, makes the fp16 copies of q, k, v, dout
 * that cp_attn_step_bwd_half reads (half_ops: a device buffer of
 * cp_attn_half_ops_size bytes, 256-byte aligned; q, k, v may be NULL when
 * half_ops is). A finite input of magnitude above 65504 (not representable
 * in fp16) sets CP_ATTN_ERR_RANGE in the plan's status word. Using the fp32
 * O keeps the bf16 rounding of O out of delta (it otherwise moves dQ and dK
 * by up to ~6e-3 on N(0,1) inputs). */
cp_attn_status cp_attn_bwd_preprocess(cp_attn_plan_t plan, const void* q, const void* k,
                                      const void* v, const void* o, const float* o_f32,
                                      const void* dout, float* delta, void* half_ops,
                                      float* dq_acc, float* dk_acc, float* dv_acc,
                                      void* stream);

/* One backward ring step (kernel K2), with the merged (global) lse and
 * delta: P = exp(scale*Q K^T - LSE) on visible pairs, dV += P^T dO,
 * dP = dO V^T, dS = P*(dP - delta), dQ += scale*dS K, dK += scale*dS^T Q
 * ("Built on a fast attention kernel" in "Announcing Long-Context Training
 * on TPUs with MaxText Context Parallelism": the ring calls the kernel once
 * per step in the backward pass too). dK and dV are summed over the query
 * heads of each KV head.
 * q, dout: bf16 [T_q, Hq, d]; k, v: bf16 [T_kv, Hkv, d] (rank-major, 16-byte
 *   aligned); lse, delta: fp32 [Hq, T_q] (the merged forward LSE, and delta
 *   from cp_attn_bwd_preprocess); dq_acc [T_q, Hq, d], dk_acc and dv_acc
 *   [T_kv, Hkv, d]: fp32 accumulators that the step adds to (zero them
 *   before step 0, e.g. with cp_attn_bwd_preprocess).
 * workspace: device buffer of at least cp_attn_half_ops_size bytes,
 *   256-byte aligned, owned by the caller and kept across the ring's steps.
 *   The backward MMAs run on fp16 copies of the four inputs (see
 *   cp_attn_half_ops_size): step 0 makes them there, from q, k, v, dout, and
 *   steps 1..R-1 read the copies step 0 left. Run step 0 of a ring first, on
 *   the same stream and workspace, as the ring order does; a later step
 *   called without it reads whatever the workspace holds.
 * ERR_INVALID_ARG for null or misaligned pointers, a small workspace or a
 * step outside [0, R). */
cp_attn_status cp_attn_step_bwd(cp_attn_plan_t plan, int step, const void* q, const void* k,
                                const void* v, const void* dout, const float* lse,
                                const float* delta, float* dq_acc, float* dk_acc,
                                float* dv_acc, void* workspace, size_t workspace_bytes,
                                void* stream);

/* cp_attn_step_bwd on fp16 copies made beforehand by cp_attn_bwd_preprocess
 * (half_ops), for callers that make the copies once for several rings. */
cp_attn_status cp_attn_step_bwd_half(cp_attn_plan_t plan, int step, const void* half_ops,
                                     const float* lse, const float* delta, float* dq_acc,
                                     float* dk_acc, float* dv_acc, void* stream);

/* LSE merge of n_parts partial results (kernel K4; the merge "as it goes"
 * of P2P in "Context Parallelism in MaxText", and Pass Q's merge after the
 * all-to-all in "Ring Attention Algorithms" of "Context Parallelism for
 * Scalable Million-Token Inference"): for each (row, head),
 * LSE = M + ln sum_i exp(LSE_i - M) with M = max_i LSE_i, and
 * O = sum_i exp(LSE_i - LSE) * O_i. Parts with LSE_i = -inf weigh 0; a row
 * whose parts are all -inf gets O = 0, LSE = -inf.
 * o_parts: fp32, part i at o_parts + i*part_stride, each [rows, heads, d].
 * lse_parts: fp32, part i at lse_parts + i*lse_part_stride, each
 *   [heads, rows] (row stride 1, head stride `rows`).
 * o_out (bf16) and o_out_f32 may each be NULL; lse_out [heads, rows] is
 * required. head_dim must be a multiple of 4 and at most 256. */
cp_attn_status cp_attn_merge_lse(int n_parts, int64_t rows, int heads, int head_dim,
                                 const float* o_parts, int64_t part_stride,
                                 const float* lse_parts, int64_t lse_part_stride,
                                 void* o_out, float* o_out_f32, float* lse_out,
                                 void* stream);
/* cp_attn_merge_lse with the O parts in parts_dtype (F32 or BF16, e.g. the
 * bf16 partials of a plan with partial_dtype BF16); part_stride counts
 * elements. The sums are fp32 either way. With BF16 parts o_out_f32 must not
 * alias them. ERR_INVALID_ARG for another dtype. */
cp_attn_status cp_attn_merge_lse_ex(int n_parts, int64_t rows, int heads, int head_dim,
                                    cp_attn_dtype parts_dtype, const void* o_parts,
                                    int64_t part_stride, const float* lse_parts,
                                    int64_t lse_part_stride, void* o_out, float* o_out_f32,
                                    float* lse_out, void* stream);

/* Whole forward pass over the emulated ring ("Ring Attention Algorithms":
 * Pass KV and Pass Q): R step launches in step order (the first also makes
 * the fp16 copy of v, see cp_attn_step_fwd), then (Pass Q) the n-way merge
 * over kv_owner slots. o: bf16
 * [T_q,Hq,d]; lse: fp32 [Hq,T_q]. workspace: device buffer of at least
 * cp_attn_workspace_size(plan, FORWARD) bytes, 256-byte aligned. On return
 * the workspace starts with O in fp32 [T_q,Hq,d] (the unrounded result),
 * which cp_attn_backward can take as o_f32 -- except for Pass Q with bf16
 * partials, whose slots are too small for it. */
cp_attn_status cp_attn_forward(cp_attn_plan_t plan, const void* q, const void* k,
                               const void* v, void* o, float* lse,
                               void* workspace, size_t workspace_bytes,
                               void* stream);

/* Forward pass that allocates nothing (no counterpart on the pages; a
 * convenience of this library). For callers that cannot call cudaMalloc on
 * the compute path -- a plugin inside a host program that owns the whole
 * device-memory pool and gives plugins no allocator, or a serving path that
 * must never enter the allocator -- and so cannot pass the forward
 * workspace. Same result as cp_attn_forward; the workspace comes from a
 * fixed device array inside the library of cp_attn_forward_noalloc_capacity()
 * bytes (32 MiB).
 *  - The plan itself still allocates its device tables and its fp16 copy
 *    buffer for V once, when it is created (cp_attn_plan / cp_attn_plan_ex);
 *    build plans before the allocation-free phase.
 *  - A device holds the array from the moment the library's device image is
 *    loaded on it (under CUDA's lazy module loading: the first launch or
 *    symbol lookup of the library on that device) until the process exits.
 *    If that load runs out of device memory the call returns
 *    CP_ATTN_ERR_OOM.
 *  - Plans whose forward workspace (cp_attn_workspace_size, FORWARD) exceeds
 *    the capacity are rejected with CP_ATTN_ERR_SHAPE before any launch.
 *  - Every call looks up the array's device address in the current context
 *    (cudaGetSymbolAddress, which allocates nothing); the first call on a
 *    device also loads the library's device image there, so make that first
 *    call before any stream capture.
 *  - All calls share the one array, which keeps the last call's contents
 *    (nothing in it needs to start at zero: every row is written before it
 *    is read). Calls that overlap on the GPU (on different streams, or from
 *    different threads) race on it: order them on one stream.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine. */
cp_attn_status cp_attn_forward_noalloc(cp_attn_plan_t plan, const void* q, const void* k,
                                       const void* v, void* o, float* lse, void* stream);
size_t cp_attn_forward_noalloc_capacity(void);

/* Whole backward pass ("Built on a fast attention kernel": the kernel runs
 * once per ring step in the backward pass too): preprocess, then R
 * backward steps in the plan's ring order. o: bf16 [T_q,Hq,d]; o_f32: optional fp32 O used for delta
 * (see cp_attn_bwd_preprocess); dq [T_q,Hq,d]; dk, dv [T_kv,Hkv,d]
 * (overwritten), fp32 or, when the plan's grad_dtype is BF16, bf16: then
 * the fp32 sums live in the workspace and a last kernel (K6) rounds them to
 * nearest even into dq, dk, dv. workspace: at least
 * cp_attn_workspace_size(plan, BACKWARD) bytes, 256-byte aligned. */
cp_attn_status cp_attn_backward(cp_attn_plan_t plan, const void* q, const void* k,
                                const void* v, const void* o, const float* o_f32,
                                const float* lse, const void* dout, void* dq, void* dk,
                                void* dv, void* workspace, size_t workspace_bytes,
                                void* stream);

/* Reorder a [tokens, row_bytes] tensor between natural token order and the
 * plan's rank-major order (kernel K5; the sharding of "Load Balancing in CP"), for the query-side (T_q rows) or the
 * key-side (T_kv rows) token set. row_bytes = heads*head_dim*element size,
 * a multiple of 16. `in` and `out` must not overlap. */
cp_attn_status cp_attn_layout_apply(cp_attn_plan_t plan, cp_attn_tensor_kind kind,
                                    cp_attn_direction direction, const void* in,
                                    void* out, int64_t row_bytes, void* stream);

/* Sequence <-> head all-to-all of Ulysses / USP ("All-to-All (Ulysses)" and
 * "A2A + P2P (USP)" in the MaxText post), emulated on one GPU that holds
 * every device's buffer (kernel K7, a strided copy at HBM bandwidth).
 * SPLIT_HEADS (before attention): in [rows, heads, head_bytes] with rows in
 *   device order (each device's tokens, every head) -> out [a2a][rows]
 *   [heads/a2a][head_bytes]: the tensor of sub-rank u is the one every
 *   device u of a group holds after the exchange (the group's tokens for
 *   heads [u*heads/a2a, (u+1)*heads/a2a)), gathered over the groups in ring
 *   order. Each sub-rank then runs its own ring (a USP plan with heads/a2a
 *   heads) on out[u].
 * GATHER_HEADS (after attention): the inverse, out[u] -> [rows, heads, ...].
 * head_bytes: bytes of one head's row (d * element size), a multiple of 16;
 * heads must be a multiple of a2a. LSE [heads, rows] needs no exchange: the
 * rows of sub-rank u's heads are already contiguous. `in` and `out` must
 * not overlap. */
typedef enum cp_attn_a2a_direction {
  CP_ATTN_SPLIT_HEADS = 0,
  CP_ATTN_GATHER_HEADS = 1
} cp_attn_a2a_direction;
cp_attn_status cp_attn_head_a2a(int64_t rows, int heads, int64_t head_bytes, int a2a,
                                cp_attn_a2a_direction direction, const void* in, void* out,
                                void* stream);

/* One-row decode over the emulated ring (kernel K9 or K8, then the K4 merge):
 * Pass Q for decode ("Context Parallelism for Scalable Million-Token
 * Inference": "Attention Compute Patterns in Multi-Turn Chat" -- decode is a
 * single-row attention of the new token over every earlier token -- and
 * "Ring Attention Algorithms" -- for decode the KV stays on its rank, the
 * query visits each rank, and the partial outputs are merged). Each of
 * `batch` sequences has one new query row and kv_len keys (its cached tokens
 * plus its own new token, appended by the caller), all visible to that row.
 * Rank r holds keys [r*kv_len/cp, (r+1)*kv_len/cp) of every sequence; each
 * rank's shard is split further into runs of 64-512 keys so the grid fills
 * the GPU, and the merge combines every run's partial.
 * q: bf16 [batch, Hq, d]; k, v: bf16 [batch, kv_len, Hkv, d]; o: bf16
 * [batch, Hq, d]; lse: fp32 [Hq, batch] (natural log, scale applied).
 * workspace: cp_attn_decode_workspace_size bytes (fp32 partials and, for the
 * tensor-core path, one work counter per KV head that the call zeroes on
 * `stream` first), 16-byte aligned like every pointer; calls that run at the
 * same time need workspaces of their own. Supported: head_dim 64 or 128, at most 16 query
 * heads per KV head, kv_len a multiple of 64*cp. With head_dim 128 and key
 * runs that are multiples of 128 the partials come from the tensor cores
 * (S^T = K Q^T and O^T = V^T P^T with the query heads as N = 16, P in bf16);
 * otherwise from the CUDA cores in fp32. */
typedef struct cp_attn_decode_desc {
  int batch;           /* sequences, one new row each */
  int cp;              /* ring size R: ranks sharing each sequence's keys */
  int64_t kv_len;      /* keys per sequence */
  int n_q_heads;
  int n_kv_heads;
  int head_dim;
  float softmax_scale; /* 0 selects 1/sqrt(head_dim) */
} cp_attn_decode_desc;
cp_attn_status cp_attn_decode_workspace_size(const cp_attn_decode_desc* desc, size_t* bytes);
cp_attn_status cp_attn_decode(const cp_attn_decode_desc* desc, const void* q, const void* k,
                              const void* v, void* o, float* lse, void* workspace,
                              size_t workspace_bytes, void* stream);
/* Synchronise `stream`, then read and clear the decode kernels' device status
 * word (one per device: the tensor-core decode records a timed-out pipeline
 * wait there, CP_ATTN_ERR_TIMEOUT). Returns CP_ATTN_OK or that error. */
cp_attn_status cp_attn_decode_sync_status(void* stream);

/* cp_attn_decode over an E4M3 KV cache (the pages' FP8-quantized model,
 * "Experimental Setup & Results"), head_dim 128, on the tensor cores.
 * q: bf16 [batch][n_q_heads][128]; each head's row is quantized to E4M3 in the
 *   kernel with its own scale (max|row| / 448, the per-tensor rule of
 *   cp_attn_fp8_quantize applied per row).
 * k8: E4M3 [batch * kv_len][n_kv_heads][128] and vt8: E4M3 V^T
 *   [n_kv_heads][128][batch * kv_len] (cp_attn_fp8_quantize of K with
 *   transpose 0 and of V with transpose 1, rows = batch * kv_len);
 *   kv_scales: device [2] floats, their descale factors (K, V).
 * P is rounded to E4M3 (after scaling by 2^8) for P V; sums, LSE and
 * accumulation stay fp32. Outputs, workspace and errors as cp_attn_decode;
 * also ERR_UNSUPPORTED for head_dim != 128 and ERR_SHAPE unless kv_len / cp is
 * a multiple of 128 and batch * kv_len < 2^31. */
cp_attn_status cp_attn_decode_fp8(const cp_attn_decode_desc* desc, const void* q, const void* k8,
                                  const void* vt8, const float* kv_scales, void* o, float* lse,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Synchronise `stream`, then read and clear the plan's device status word.
 * Returns CP_ATTN_OK or the first device-side error (ERR_TIMEOUT). */
cp_attn_status cp_attn_sync_status(cp_attn_plan_t plan, void* stream);

/* Failure-path self test: launches one CTA whose pipeline wait has nothing
 * to wait for. After limit_ns nanoseconds (at most 2 s) the wait gives up,
 * exactly as a stalled wait in K1/K2 would, and records
 * CP_ATTN_ERR_TIMEOUT in the plan's status word (read and cleared by
 * cp_attn_sync_status). No fault, trap or hang is involved. */
cp_attn_status cp_attn_selftest_wait_timeout(cp_attn_plan_t plan, uint64_t limit_ns,
                                             void* stream);

/* Number of kernel launches the library made in this process so far. */
int64_t cp_attn_launch_count(void);

const char* cp_attn_last_error(void);
const char* cp_attn_status_string(cp_attn_status status);

#ifdef __cplusplus
}
#endif

#endif /* CP_ATTN_H */
