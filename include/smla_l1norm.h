/*
 * smla_l1norm.h -- C ABI of the GB300 Sparse-Flash-MLA Softmax-L1Norm forward.
 *
 * The operator (article "SparseFlashMlaSoftmaxL1Norm", CANN ops-transformer,
 * section 三阶段计算公式 / three-stage formula):
 *
 *   stage 1  selectedKv = Gather(K, sparse_indices[row, i]), 0 <= i < topk
 *            (or the whole K when there are no sparse indices);
 *   stage 2  P[g, i] = exp(scale * q[row, g] . selectedKv[i] - softmax_lse[row, g])
 *            for every slot that the mask keeps, 0 for the others;
 *   stage 3  out[row, i] = (sum over g < G of P[g, i]) / G,   G = N1 / N2.
 *
 * A slot is kept when its key position j lies inside the row's sequence
 * (0 <= j < Sk), its slot number is below topk_length[row] (when given), and,
 * for mask_mode 3 (rightDownCausal, the lower triangle divided at the
 * right-bottom vertex), j <= r + Sk - Sq for local query row r.  Kept slots
 * never depend on other slots; every output element is written exactly once
 * (no atomics), so results are bitwise reproducible run to run (the article's
 * constraints section states the operator is deterministic).
 *
 * Call pattern (the article's two-phase design: a metadata operator that
 * balances rows over cores, then the main operator):
 *
 *   smla_l1norm_plan_create()   once per shape: validate, build the CTA work
 *                               schedule on the host, upload it (the GB300
 *                               counterpart of SparseFlashMlaSoftmaxL1NormMetadata)
 *   smla_l1norm_run()           per call: one kernel launch on the caller's
 *                               stream; asynchronous; allocates nothing
 *   smla_l1norm_get_status()    optional: device-side warnings / timeouts
 *   smla_l1norm_plan_destroy()
 *
 * Memory ownership: the caller owns every tensor.  All tensors are dense and
 * row-major ("AutoContiguous" in the article's operator definition) with the
 * shapes below; device pointers must be 16-byte aligned.  A plan owns one
 * small device buffer (its work list and status word).  A plan is bound to the
 * device that was current when it was created; two run() calls with the same
 * plan may overlap on the GPU, but they then share the status word.
 *
 * Error codes follow the article's aclnn split between null pointers
 * (ACLNN_ERR_PARAM_NULLPTR) and invalid parameters (ACLNN_ERR_PARAM_INVALID):
 * host-side checks return before any CUDA call or launch.
 */
#ifndef SMLA_L1NORM_H_
#define SMLA_L1NORM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st *smla_stream_t;

typedef enum {
  SMLA_OK = 0,
  SMLA_ERR_NULLPTR = 1,      /* a required pointer is NULL                         */
  SMLA_ERR_INVALID = 2,      /* a shape / layout / dtype / constraint is violated  */
  SMLA_ERR_UNSUPPORTED = 3,  /* a documented feature this library does not build:
                                mask modes 1 and 2; compressed keys under the
                                causal mask in smla_l1norm_run_noalloc          */
  SMLA_ERR_CUDA = 4,         /* a CUDA runtime call failed (see get_last_cuda_error) */
  SMLA_ERR_TIMEOUT = 5,      /* a device-side wait gave up (reported by get_status) */
  SMLA_WARN_BAD_INDEX = 6,   /* a sparse index outside [-1, Sk) was seen and treated
                                as masked (reported by get_status)                 */
  SMLA_ERR_CAPACITY = 7      /* smla_l1norm_run_noalloc: the problem needs more work
                                items than its fixed scratch holds                 */
} smla_status;

typedef enum { SMLA_LAYOUT_BSND = 0, SMLA_LAYOUT_TND = 1 } smla_layout;
typedef enum { SMLA_DTYPE_F16 = 0, SMLA_DTYPE_BF16 = 1 } smla_dtype;
typedef enum { SMLA_MASK_NONE = 0, SMLA_MASK_RIGHT_DOWN_CAUSAL = 3 } smla_mask_mode;

/*
 * Operator description (article: parameter tables 参数说明 for the main
 * operator and the metadata operator; constraints 约束说明).
 *
 *   layout_q, layout_k  BSND or TND; must be equal.
 *   dtype               q and k share it (FLOAT16 or BFLOAT16).
 *   num_heads_q         N1, 1..128.   num_heads_k  N2, must be 1.   G = N1 / N2.
 *   head_dim            D, must be 512.
 *   batch_size          BSND: B (>= 0).  TND: the number of sequences (the
 *                       cu_seqlens arrays hold batch_size + 1 entries).
 *   max_seqlen_q        BSND: S1 (>= 0).  TND: ignored.
 *   max_seqlen_k        BSND: S2 (>= 0).  TND: output width of the dense form
 *                       (must be >= every sequence's key length; ignored when
 *                       topk > 0).
 *   topk                last dimension of sparse_indices; 0 = dense form.
 *   mask_mode           0 (none) or 3 (rightDownCausal).
 *   cmp_ratio           key compression ratio c, 1..128 ([SMLA] 参数说明).  With
 *                       c > 1, K holds compressed keys: key j of a sequence
 *                       stands for the original key positions j*c .. j*c+c-1
 *                       of an original sequence of L = Sk*c + cmp_residual_k
 *                       positions (Sk = the sequence's rows of K).  Under
 *                       mask_mode 3 a key is kept only when its whole block
 *                       is visible: j*c + c - 1 <= r + L - Sq (the article
 *                       leaves the rule for a partly visible block open; this
 *                       reading never shows a query a later position).  With
 *                       mask_mode 0 the ratio changes nothing.  The dense
 *                       output is as wide as K (compressed positions).
 *   softmax_scale       multiplies q.k before the exp (the article's default
 *                       is 1.0 and it recommends 1/sqrt(head_dim)).
 *   has_topk_length     1 if run() will be given topk_length.
 *   cu_seqlens_q/k      TND only: HOST arrays of batch+1 int32, cumulative
 *                       sums of the per-sequence query / key lengths,
 *                       starting at 0 and non-decreasing.  Read during
 *                       plan_create only.
 *   topk_length_hint    optional HOST array (one int32 per query token): the
 *                       expected topk_length, used only to balance the work
 *                       schedule.  NULL = estimate min(topk, visible keys).
 *   num_ctas            0 = one persistent CTA per SM of the current device;
 *                       > 0 forces a grid size (tests, multi-tenant use); the
 *                       CTA-pair launch then runs at most num_ctas / 2 pairs.
 */
typedef struct {
  int32_t layout_q;
  int32_t layout_k;
  int32_t dtype;
  int32_t num_heads_q;
  int32_t num_heads_k;
  int32_t head_dim;
  int32_t batch_size;
  int32_t max_seqlen_q;
  int32_t max_seqlen_k;
  int32_t topk;
  int32_t mask_mode;
  int32_t cmp_ratio;
  float softmax_scale;
  int32_t has_topk_length;
  const int32_t *cu_seqlens_q;
  const int32_t *cu_seqlens_k;
  const int32_t *topk_length_hint;
  int32_t num_ctas;
} smla_l1norm_desc;

typedef struct smla_plan smla_plan; /* opaque */

/* Summary of a plan's schedule (costs in the scheduler's tile units). */
typedef struct {
  int64_t num_tokens;      /* query tokens (B*S1 or T1)                          */
  int64_t num_items;       /* work items (a token, or a pack of tokens if dense) */
  int32_t num_ctas;        /* persistent grid size                               */
  int32_t rows_per_item;   /* R: query tokens packed into one MMA (dense form)   */
  int32_t mma_n;           /* N of the tensor-core instruction (R*G padded to 16) */
  int32_t stages;          /* depth of the shared-memory key ring                */
  int32_t smem_bytes;      /* dynamic shared memory per CTA                      */
  int32_t out_width;       /* last output dimension                              */
  int64_t est_tiles;       /* 128-key tiles the schedule expects                 */
  double max_cta_cost;     /* heaviest CTA                                       */
  double mean_cta_cost;    /* average CTA                                        */
  int64_t q_rows_total;    /* rows of the 2-D view of q (tokens * G)             */
  int64_t k_rows_total;    /* rows of the 2-D view of k (B*S2 or T2)             */
  int32_t host_chunks;     /* token chunks smla_l1norm_run_from_host pipelines
                              (copies of one chunk overlap the kernel of the
                              previous one); 0 = one copy, one kernel, one copy */
  int32_t mma_issuers;     /* threads issuing the L1-norm launch's MMAs: 4 when
                              the sparse form's N is at most 64 (each owns a
                              quarter of the head dimension), else 2          */
  int32_t cta_pairs;       /* 2-CTA clusters of the CTA-pair L1-norm launch
                              (sparse form, N = 128: one MMA covers both CTAs'
                              keys); 0 = the single-CTA kernel runs it        */
  int32_t split_tiles;     /* dense form: the L1-norm launch splits each token
                              pack's keys into parts of at most this many
                              128-key tiles (output slots depend on one key
                              each, so the parts are independent); 0 = one
                              part per pack                                 */
  int64_t split_items;     /* work items of that split launch (0 = no split) */
} smla_plan_info;

/*
 * Validate ``desc`` and build a plan for the current CUDA device.
 * Returns SMLA_ERR_NULLPTR / SMLA_ERR_INVALID / SMLA_ERR_UNSUPPORTED without
 * touching the GPU when the description is rejected; SMLA_ERR_CUDA if the
 * device query, allocation or upload fails.  An empty q (no query token)
 * gives a valid plan whose run() returns at once, as the article's
 * constraints section specifies for an empty q tensor.
 * Synchronous (the work list is uploaded with a blocking copy).
 *
 * Every device-side wait of the plan's launches is bounded: 2 s by default,
 * SMLA_WAIT_TIMEOUT_MS (milliseconds, > 0) as read from the environment here.
 * A wait that runs out stops the launch's CTA cleanly (copies and MMAs in
 * flight are drained, tensor memory is released) and sets the timeout flag
 * that smla_l1norm_get_status() reports; the output is then incomplete.
 * Test hook: with SMLA_DEBUG_WITHHOLD_Q=1 in the environment at plan
 * creation, every CTA of the plan's launches skips the load of the first q
 * chunk of its first work item, so a wait runs out on purpose.
 *
 * Kernel choice for the L1-norm launch (reported in smla_plan_info):
 * sparse work with exactly 128 heads whose tokens average at least 10
 * 128-key tiles runs on 2-CTA clusters (cta_pairs > 0), everything else on
 * one CTA per SM; a dense plan may split token packs along their keys
 * (split_tiles > 0).  SMLA_PAIR=0 / 1 and SMLA_SPLIT=n in the environment
 * at plan creation force these choices (SMLA_PAIR=1 still needs exactly
 * 128 heads and a grid of at least two CTAs).  Every choice computes the
 * same values to within fp32 rounding.
 */
smla_status smla_l1norm_plan_create(const smla_l1norm_desc *desc, smla_plan **plan_out);

/* Free a plan and its device buffer.  NULL is ignored.  The caller must make
 * sure no run() using the plan is still executing. */
void smla_l1norm_plan_destroy(smla_plan *plan);

/* Output shape (infershape in the article): BSND -> 4 dims (B, S1, 1, W),
 * TND -> 3 dims (T1, 1, W); W = topk when sparse, else S2 (BSND) or
 * max_seqlen_k (TND). */
smla_status smla_l1norm_output_shape(const smla_plan *plan, int64_t dims[4], int32_t *ndim);

smla_status smla_l1norm_plan_get_info(const smla_plan *plan, smla_plan_info *info);

/*
 * Compute the operator on ``stream`` (asynchronous; one kernel launch; no
 * allocation, no host synchronisation).  Device pointers, 16-byte aligned:
 *
 *   q               (B,S1,N1,512) or (T1,N1,512)  fp16/bf16  [required]
 *   k               (B,S2,1,512)  or (T2,1,512)   same dtype [required unless
 *                   there is no key row at all]
 *   softmax_lse     (B,1,S1,G)    or (1,T1,G)     fp32       [required]
 *   sparse_indices  (B,S1,1,topk) or (T1,1,topk)  int32      [required iff topk > 0]
 *                   key positions inside the row's sequence; -1 is padding
 *   topk_length     (B,S1,1)      or (T1,1)       int32      [required iff the
 *                   plan says has_topk_length]; values are clamped to [0, topk]
 *   out             output_shape()                fp32       [required]
 *
 * Every element of ``out`` is written (masked and padding slots as 0.0f), so
 * it need not be cleared.  Returns SMLA_ERR_NULLPTR for a missing required
 * pointer, SMLA_ERR_INVALID for a misaligned one, SMLA_ERR_CUDA if the
 * launch fails.  Device-side conditions (index out of range, wait timeout)
 * are recorded in the plan's status word; see smla_l1norm_get_status().
 */
smla_status smla_l1norm_run(const smla_plan *plan, const void *q, const void *k,
                            const float *softmax_lse, const int32_t *sparse_indices,
                            const int32_t *topk_length, float *out, smla_stream_t stream);

/*
 * The tensors of one call, for smla_l1norm_run_tensors().  Device pointers;
 * the first five and ``out`` as for smla_l1norm_run().  The optional inputs
 * of the article's parameter table (参数说明) that run() has no slot for:
 * seqused_q, seqused_k (below) and cmp_residual_k (see the field):
 *
 *   seqused_q   (B,) int32 or NULL: query tokens of each sequence that take
 *               part.  Sequence b's query rows r >= min(Sq_b, seqused_q[b])
 *               are written as all-zero rows.  Negative values count as 0.
 *   seqused_k   (B,) int32 or NULL: keys of each sequence that take part.
 *               Key positions j >= min(Sk_b, seqused_k[b]) are masked (0).
 *
 * With either given, mask_mode 3 places the causal diagonal on the cut
 * lengths: row r sees key j iff j <= r + Sk' - Sq', Sq' and Sk' being the
 * lengths after the cut.  B is batch_size (the number of sequences in TND).
 * The values are read on the device, so the plan's work schedule is balanced
 * on the full lengths; the cut only removes work.  An index in [Sk', Sk) is
 * masked without raising the bad-index warning.
 */
typedef struct {
  const void *q;
  const void *k;
  const float *softmax_lse;
  const int32_t *sparse_indices;
  const int32_t *topk_length;
  const int32_t *seqused_q;
  const int32_t *seqused_k;
  float *out;
  const int32_t *cmp_residual_k; /* (B,) int32: per sequence, the original key
                                    count minus Sk*cmp_ratio (the remainder of
                                    the original length // cmp_ratio), read on
                                    the device and clamped to 0..cmp_ratio-1.
                                    Required (else SMLA_ERR_NULLPTR) when the
                                    plan has cmp_ratio != 1 and mask_mode 3;
                                    ignored otherwise.  run() and
                                    run_from_host() pass NULL, so such plans
                                    run through run_tensors() and the LSE
                                    entry points.  Under seqused_k the original
                                    length is Sk'*cmp_ratio + cmp_residual_k. */
} smla_l1norm_tensors;

/* smla_l1norm_run() with every optional input; same errors (NULL ``tensors``
 * is SMLA_ERR_NULLPTR; a seqused pointer that is not 4-byte aligned is
 * SMLA_ERR_INVALID).  run() is this call with both seqused pointers NULL. */
smla_status smla_l1norm_run_tensors(const smla_plan *plan, const smla_l1norm_tensors *tensors,
                                    smla_stream_t stream);

/*
 * The forward pass's softmax_lse, computed on the GPU over the same kept
 * slots the operator uses (article "SparseFlashMlaSoftmaxL1Norm", 参数说明:
 * softmax_lse is the output of the forward attention pass; in the section
 * 三阶段计算公式, stage 2's SimpleSoftmax normalises by it):
 *
 *   lse_out[row, g] = log sum_{kept slots i} exp(scale * q[row, g] . K[j_i])
 *
 * natural logarithm, fp32, -inf for a row with no kept slot.  ``lse_out``
 * has the layout of softmax_lse: (B,1,S1,G) or (1,T1,G), i.e. token-major
 * (token, g); device pointer, 4-byte aligned.  One launch of the same
 * persistent kernel in a mode where the MMA puts the q rows on M and the
 * keys on N and each epilogue thread keeps a running maximum and sum for its
 * row.  Reads q, k, sparse_indices, topk_length and the seqused tensors of
 * ``tensors``; ignores softmax_lse and out.  Same errors as
 * smla_l1norm_run_tensors() (``lse_out`` NULL: SMLA_ERR_NULLPTR).
 */
smla_status smla_softmax_lse_run(const smla_plan *plan, const smla_l1norm_tensors *tensors,
                                 float *lse_out, smla_stream_t stream);

/*
 * Both in one launch: for each work item, a pass over its key tiles
 * computes the LSE as smla_softmax_lse_run() does and writes it to
 * ``lse_out``, then a second pass over the same tiles (the keys gathered
 * again) computes the operator with that LSE and writes ``tensors->out``.
 * The q block stays in shared memory for both passes.  Ignores
 * tensors->softmax_lse.  Each output row over its kept slots sums to 1 up
 * to rounding.
 */
smla_status smla_l1norm_run_fused_lse(const smla_plan *plan, const smla_l1norm_tensors *tensors,
                                      float *lse_out, smla_stream_t stream);

/* Host-side sizes, in bytes, of the tensors run() reads and writes. */
typedef struct {
  size_t q_bytes, k_bytes, lse_bytes, indices_bytes, topk_length_bytes, out_bytes;
} smla_io_sizes;

smla_status smla_l1norm_io_sizes(const smla_plan *plan, smla_io_sizes *sizes);

/*
 * End-to-end form for callers whose tensors live in HOST memory: copy each
 * host input into the caller's device buffer of the same role, run, and copy
 * the output back to ``h_out``.  Host buffers should be page-locked for the
 * copies to be asynchronous.  Pass NULL for tensors the plan does not use.
 * Returns as run(); the host output is valid after ``stream`` is
 * synchronised.
 *
 * When the plan has host_chunks > 0 the call is pipelined over token
 * chunks: the plan's own copy-in stream moves k, then each chunk's rows of
 * q, lse, indices and topk_length; ``stream`` runs each chunk's kernel as
 * soon as its rows have landed; the plan's copy-out stream returns each
 * chunk's output rows as soon as its kernel is done.  Both plan streams
 * start after the work already queued on ``stream``, and ``stream`` waits
 * for the last copy, so to the caller the call is ordered on ``stream`` like
 * any other.  Otherwise (small problems) it is one copy per tensor, one
 * kernel and one copy back, all on ``stream``.  The plan's streams and
 * events are shared by its calls: issue run_from_host calls of one plan from
 * one host thread at a time, and order calls that share device buffers on
 * one stream (a later call's copies may otherwise overwrite inputs an
 * earlier call's kernels still read).
 */
smla_status smla_l1norm_run_from_host(const smla_plan *plan,
                                      const void *h_q, const void *h_k, const float *h_lse,
                                      const int32_t *h_indices, const int32_t *h_topk_length,
                                      float *h_out,
                                      void *d_q, void *d_k, float *d_lse, int32_t *d_indices,
                                      int32_t *d_topk_length, float *d_out,
                                      smla_stream_t stream);

/*
 * Read and clear the plan's device status word.  Synchronises ``stream``.
 * Writes the raw flag bits to *flags (if non-NULL): bit 0 = bad index seen,
 * bit 1 = a device-side wait timed out.  Returns SMLA_ERR_TIMEOUT if bit 1 is
 * set, else SMLA_WARN_BAD_INDEX if bit 0 is set, else SMLA_OK.
 */
smla_status smla_l1norm_get_status(const smla_plan *plan, smla_stream_t stream, int32_t *flags);

/*
 * Host-only view of the scheduler, for inspection and tests: validate
 * ``desc`` and build the schedule for ``num_ctas`` CTAs without any CUDA
 * call.  ``split_tiles``: 0 = whole token packs (the schedule of every launch
 * but the dense L1-norm one); n > 0 = dense packs split into parts of at most
 * n key tiles (SMLA_ERR_INVALID for the sparse form); -1 = what a plan's
 * dense L1-norm launch runs (split or not, as the plan would choose).  If
 * ``items`` is non-NULL it receives up to ``items_capacity`` work items of 12
 * int32 each, grouped by CTA (fields: first token, tokens in the item, local
 * row of the first token, first key row of the sequence, Sq, Sk, key tiles of
 * a dense item, sequence number b, first key tile, cut_tail (1: an earlier
 * part of a split pack, which zeroes only its own key range), two reserved
 * zeros); ``cta_offsets`` (num_ctas + 1 int32) receives where each CTA's items
 * start.  ``info`` receives the summary, with the split chosen.
 */
smla_status smla_l1norm_schedule_host(const smla_l1norm_desc *desc, int32_t num_ctas,
                                      int32_t split_tiles, int32_t *items, int64_t items_capacity,
                                      int32_t *cta_offsets, smla_plan_info *info);

/*
 * Self-test of the device-side wait bound (the article has no counterpart):
 * launches one CTA whose only thread waits, with the bounded wait every
 * role of the fused kernel uses, on a barrier that nothing completes.  After
 * ``timeout_ns`` the wait gives up and records the timeout flag; the call
 * synchronises ``stream`` and returns SMLA_ERR_TIMEOUT (flags bit 1) when the
 * bound works.  Allocates and frees 4 bytes of device memory.
 */
smla_status smla_debug_wait_timeout_probe(int64_t timeout_ns, smla_stream_t stream, int32_t *flags);

/*
 * Test hook: the key gather (stage 1 of the article's three-stage formula,
 * selectedKv = Gather(K, sparse_indices)) alone, for one work item.  Runs the
 * key-producer warps of a launch mode -- the same device code the operator
 * runs -- over the work item of ``plan`` that holds query token ``token``,
 * with one warp taking the place of the tensor cores: each 16 KB ring stage
 * is copied to ``dump`` exactly as the MMA would read it, in stage order.
 *
 *   mode        0: the L1-norm launch's producers (two groups on alternate
 *               stages); 1: the forward-LSE and fused launches' (one group).
 *   dump        device buffer, 16-byte aligned, ``dump_bytes`` long.  Stage
 *               n = 8*t + c holds head-dim columns 64c .. 64c+63 of the 128
 *               key slots of key tile t: slot s of the tile (row s & 127) at
 *               byte offset 16384*n + 128*s + 16*(p ^ (s & 7)) for its 16-byte
 *               piece p (0..7) -- the 128-byte swizzle.  Stages beyond
 *               dump_bytes / 16384 are not written.  The item's key tiles
 *               are ceil(min(topk_length, topk) / 128) in the sparse form
 *               (topk when there is no topk_length; 0 when the sequence has
 *               no key), its precomputed tile count in the dense form.
 *   k, sparse_indices, topk_length   as for smla_l1norm_run().
 *
 * A slot whose key position j is in [0, Sk) holds key row j of the token's
 * sequence, bit for bit; any other slot (index -1 or out of range, slot
 * past topk_length or topk) holds zeros (nothing is read for it), and the
 * epilogue masks it to an output of 0.  Asynchronous on ``stream``; device flags go to
 * the plan's status word.  Returns SMLA_ERR_INVALID for a bad mode, token or
 * alignment, SMLA_ERR_NULLPTR for a missing pointer.
 */
smla_status smla_debug_gather(const smla_plan *plan, int32_t mode, int64_t token, const void *k,
                              const int32_t *sparse_indices, const int32_t *topk_length, void *dump,
                              int64_t dump_bytes, smla_stream_t stream);

/*
 * Allocation-free form of smla_l1norm_run() (the article has no counterpart;
 * the operator is the same).  For callers that cannot call cudaMalloc: code
 * running where a framework's caching allocator owns all device memory, a
 * plugin that is handed device pointers but no allocator, a service that
 * forbids allocation after start-up.  No plan is needed: pass the
 * description and the same tensors as smla_l1norm_run().
 *
 * Scratch: the work list and the status word live in a fixed file-scope
 * device array of 2,101,760 bytes (2 MiB of work items plus offsets and the
 * status word), which every GPU that loads this library holds until the
 * process exits.  Capacity: at most 65,536 work items (query tokens in the
 * sparse form; packs of 128/G tokens in the dense form) and 1,024 CTAs;
 * larger problems return SMLA_ERR_CAPACITY before any CUDA call.
 *
 * The call allocates nothing: no cudaMalloc / cudaFree, no allocating CUDA
 * or torch routine, no host heap.  It builds the work list in fixed host
 * staging memory, copies it into the device array with cudaMemcpyAsync on
 * ``stream`` and launches the fused kernel.  The staging memory is pageable:
 * the call returns once the copy has taken the host bytes, and the device
 * copy is ordered after earlier work on ``stream``.  The launch shape (CTAs,
 * key-ring depth, shared memory), the validation and the device-side wait
 * limit (SMLA_WAIT_TIMEOUT_MS) are the plan path's;
 * smla_debug_noalloc_config() reports the shape without a GPU.
 *
 * Set-up: the first call on each device (with that device current) looks up
 * the device address of the scratch array with cudaGetSymbolAddress and
 * caches it; make that first call before any stream capture.
 *
 * Sharing: all calls on a device use the same array, which keeps the last
 * call's contents; each call rewrites the work list and clears the status
 * word.  Calls that overlap on the GPU (issued on different streams, or from
 * several host threads) race on the array: serialise them.  Device-side flags
 * (bad index, wait timeout) are recorded in the array's status word but not
 * reported; use the plan-based path to read them.
 *
 * Returns SMLA_OK, the validation codes of smla_l1norm_plan_create /
 * smla_l1norm_run, SMLA_ERR_CAPACITY, or SMLA_ERR_CUDA.
 */
smla_status smla_l1norm_run_noalloc(const smla_l1norm_desc *desc, const void *q, const void *k,
                                    const float *softmax_lse, const int32_t *sparse_indices,
                                    const int32_t *topk_length, float *out, smla_stream_t stream);

/*
 * Host-only view of smla_l1norm_run_noalloc()'s launch shape, for tests (the
 * article has no counterpart): validates ``desc`` exactly as that call does
 * and fills ``info`` with what it would launch on a device with ``num_sms``
 * SMs and ``smem_optin`` bytes of opt-in shared memory per block: num_ctas,
 * stages (key-ring depth), smem_bytes, mma_n, rows_per_item, num_items,
 * num_tokens, out_width and the q / k row counts; the cost fields are 0.
 * No CUDA call.  Returns the validation codes, SMLA_ERR_CAPACITY for a
 * problem beyond the fixed scratch, SMLA_ERR_NULLPTR for a NULL ``info`` and
 * SMLA_ERR_INVALID for a non-positive ``num_sms`` or ``smem_optin``.
 */
smla_status smla_debug_noalloc_config(const smla_l1norm_desc *desc, int32_t num_sms, int32_t smem_optin,
                                      smla_plan_info *info);

/* Static description of a status code. */
const char *smla_status_string(smla_status status);

/* Text of the last CUDA error seen by this library on this thread ("" if none). */
const char *smla_get_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SMLA_L1NORM_H_ */
